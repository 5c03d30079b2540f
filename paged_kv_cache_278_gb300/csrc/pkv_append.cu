// pkv_append.cu -- in-place append of one decode step's K/V into the paged cache.
//
// The new token's K and V go straight into their slots of the preallocated
// pool; nothing is reallocated and no old entry is touched
// ("为什么“推理优化”不是锦上添花", sec. 3.1: append into a preallocated tensor;
// "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.3: an in-place append kernel
// instead of concatenating a new tensor every step).
//
// One thread moves one 16-byte piece of one (token, kv head) row of K or V:
// reads of k_new/v_new are fully coalesced; each row lands as a contiguous
// head_dim*2-byte run inside its (block, kv head) tile.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace {

__device__ int g_append_error;

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
    append_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                  const int64_t *__restrict__ slot_mapping, const uint4 *__restrict__ k_new,
                  const uint4 *__restrict__ v_new, int64_t pieces_per_tensor, int num_kv_heads,
                  int pieces_per_row, int block_size, int64_t num_slots) {
    int64_t idx = static_cast<int64_t>(blockIdx.x) * kAppendThreads + threadIdx.x;
    const bool is_v = idx >= pieces_per_tensor;
    if (is_v) idx -= pieces_per_tensor;
    if (idx >= pieces_per_tensor) return;
    const int piece = static_cast<int>(idx % pieces_per_row);
    const int64_t row = idx / pieces_per_row;  // = token * num_kv_heads + kv head
    const int head = static_cast<int>(row % num_kv_heads);
    const int64_t token = row / num_kv_heads;
    const int64_t slot = __ldg(slot_mapping + token);
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        pkv::record_error(&g_append_error, PKV_DEV_BAD_SLOT);
        return;
    }
    const int64_t block = slot / block_size;
    const int64_t offset = slot - block * block_size;
    const int64_t dst = ((block * num_kv_heads + head) * block_size + offset) * pieces_per_row + piece;
    if (is_v)
        v_cache[dst] = __ldg(v_new + idx);
    else
        k_cache[dst] = __ldg(k_new + idx);
}

// Int8 key cache: one warp per (token, kv head) row; lane i holds dims 4i..4i+3.  The row's
// scale max|k| / 127 comes from a warp max; codes are round-half-even(k / scale) in float32.
constexpr int kRowsPerAppendBlock = kAppendThreads / 32;

// The row's codes (4 per lane, little-endian: dim 4i in byte 0) and scale max|x| / 127.
__device__ __forceinline__ uint32_t quantize_row_part(uint2 raw, float &scale) {
    const float2 x01 = pkv::half2_bits_to_float2(raw.x);
    const float2 x23 = pkv::half2_bits_to_float2(raw.y);
    float amax = fmaxf(fmaxf(fabsf(x01.x), fabsf(x01.y)), fmaxf(fabsf(x23.x), fabsf(x23.y)));
#pragma unroll
    for (int sh = 16; sh >= 1; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(pkv::kFullMask, amax, sh));
    const float s = __fdiv_rn(amax, 127.f);
    scale = s;
    return (static_cast<uint32_t>(pkv::quantize_int8(x01.x, s)) & 0xffu) |
           ((static_cast<uint32_t>(pkv::quantize_int8(x01.y, s)) & 0xffu) << 8) |
           ((static_cast<uint32_t>(pkv::quantize_int8(x23.x, s)) & 0xffu) << 16) |
           (static_cast<uint32_t>(pkv::quantize_int8(x23.y, s)) << 24);
}

// QV: the value rows are quantised too (v_out holds int8 codes, v_scale their scales).
template <bool QV>
__global__ void __launch_bounds__(kAppendThreads)
    append_int8k_kernel(uint32_t *__restrict__ k_codes, float *__restrict__ k_scale, void *__restrict__ v_out,
                        float *__restrict__ v_scale, const int64_t *__restrict__ slot_mapping,
                        const uint2 *__restrict__ k_new, const uint2 *__restrict__ v_new, int64_t rows,
                        int num_kv_heads, int block_size, int64_t num_slots) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerAppendBlock + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;  // warp-uniform
    const int head = static_cast<int>(row % num_kv_heads);
    const int64_t token = row / num_kv_heads;
    const int64_t slot = __ldg(slot_mapping + token);
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        if (lane == 0) pkv::record_error(&g_append_error, PKV_DEV_BAD_SLOT);
        return;
    }
    const int64_t block = slot / block_size;
    const int64_t dst = (block * num_kv_heads + head) * block_size + (slot - block * block_size);
    const uint2 v_raw = __ldg(v_new + row * 32 + lane);
    if constexpr (QV) {
        float vs;
        const uint32_t vc = quantize_row_part(v_raw, vs);
        static_cast<uint32_t *>(v_out)[dst * 32 + lane] = vc;
        if (lane == 0) v_scale[dst] = vs;
    } else {
        static_cast<uint2 *>(v_out)[dst * 32 + lane] = v_raw;
    }
    float s;
    const uint32_t packed = quantize_row_part(__ldg(k_new + row * 32 + lane), s);
    k_codes[dst * 32 + lane] = packed;
    if (lane == 0) k_scale[dst] = s;
}

// fp8 (E4M3) keys and values: one warp per (token, kv head) row, lane i holds dims 4i..4i+3.
// Each row's scale is max|x| / 448 from a warp max; codes are the nearest E4M3 values of x / scale
// (float32 division), by the hardware conversion with round-to-nearest-even and clamping to 448.
__device__ __forceinline__ uint32_t quantize_row_part_e4m3(uint2 raw, float &scale) {
    const float2 x01 = pkv::half2_bits_to_float2(raw.x);
    const float2 x23 = pkv::half2_bits_to_float2(raw.y);
    float amax = fmaxf(fmaxf(fabsf(x01.x), fabsf(x01.y)), fmaxf(fabsf(x23.x), fabsf(x23.y)));
#pragma unroll
    for (int sh = 16; sh >= 1; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(pkv::kFullMask, amax, sh));
    const float s = __fdiv_rn(amax, 448.f);
    scale = s;
    return pkv::quantize_e4m3x2(x01.x, x01.y, s) | (pkv::quantize_e4m3x2(x23.x, x23.y, s) << 16);
}

__global__ void __launch_bounds__(kAppendThreads)
    append_fp8kv_kernel(uint32_t *__restrict__ k_codes, float *__restrict__ k_scale, uint32_t *__restrict__ v_codes,
                        float *__restrict__ v_scale, const int64_t *__restrict__ slot_mapping,
                        const uint2 *__restrict__ k_new, const uint2 *__restrict__ v_new, int64_t rows,
                        int num_kv_heads, int block_size, int64_t num_slots) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerAppendBlock + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;  // warp-uniform
    const int head = static_cast<int>(row % num_kv_heads);
    const int64_t token = row / num_kv_heads;
    const int64_t slot = __ldg(slot_mapping + token);
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        if (lane == 0) pkv::record_error(&g_append_error, PKV_DEV_BAD_SLOT);
        return;
    }
    const int64_t block = slot / block_size;
    const int64_t dst = (block * num_kv_heads + head) * block_size + (slot - block * block_size);
    float ks, vs;
    const uint32_t kc = quantize_row_part_e4m3(__ldg(k_new + row * 32 + lane), ks);
    const uint32_t vc = quantize_row_part_e4m3(__ldg(v_new + row * 32 + lane), vs);
    k_codes[dst * 32 + lane] = kc;
    v_codes[dst * 32 + lane] = vc;
    if (lane == 0) {
        k_scale[dst] = ks;
        v_scale[dst] = vs;
    }
}

// Whole-block copies (copy-on-write within a pool, swap between a device pool and host swap
// space): one thread per 16-byte piece of a block (all kv heads), K then V.  Plain loads and
// stores, so either side may be page-locked host memory the GPU addresses directly.
__global__ void __launch_bounds__(kAppendThreads)
    copy_blocks_kernel(uint4 *dst_k, uint4 *dst_v, int64_t dst_blocks, const uint4 *src_k, const uint4 *src_v,
                       int64_t src_blocks, const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                       int64_t pieces_per_block, int n) {
    int64_t idx = static_cast<int64_t>(blockIdx.x) * kAppendThreads + threadIdx.x;
    const int64_t per_tensor = pieces_per_block * n;
    const bool is_v = idx >= per_tensor;
    if (is_v) idx -= per_tensor;
    if (idx >= per_tensor) return;
    const int pair = static_cast<int>(idx / pieces_per_block);
    const int64_t piece = idx - pair * pieces_per_block;
    const int32_t s = src[pair], d = dst[pair];
    if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
        if (piece == 0) pkv::record_error(&g_append_error, PKV_DEV_BAD_BLOCK_ID);
        return;
    }
    (is_v ? dst_v : dst_k)[d * pieces_per_block + piece] = (is_v ? src_v : src_k)[s * pieces_per_block + piece];
}

int launch_copy_blocks(void *dst_k, void *dst_v, int64_t dst_blocks, const void *src_k, const void *src_v,
                       int64_t src_blocks, const int32_t *src, const int32_t *dst, int n, int num_kv_heads,
                       int head_dim, int block_size, pkv_stream_t stream) {
    if (!dst_k || !dst_v || !src_k || !src_v || (n > 0 && (!src || !dst))) return PKV_ERR_INVALID_ARG;
    if (n < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || dst_blocks <= 0 || src_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
    if (!pkv_internal::aligned16(dst_k) || !pkv_internal::aligned16(dst_v) || !pkv_internal::aligned16(src_k) ||
        !pkv_internal::aligned16(src_v) || (n > 0 && (!pkv_internal::aligned(src, 4) || !pkv_internal::aligned(dst, 4))))
        return PKV_ERR_INVALID_ARG;
    if (n == 0) return PKV_OK;
    const int64_t pieces = static_cast<int64_t>(num_kv_heads) * block_size * head_dim / 8;
    const int64_t blocks = (2 * pieces * n + kAppendThreads - 1) / kAppendThreads;
    if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    copy_blocks_kernel<<<static_cast<unsigned>(blocks), kAppendThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(dst_k), static_cast<uint4 *>(dst_v), dst_blocks, static_cast<const uint4 *>(src_k),
        static_cast<const uint4 *>(src_v), src_blocks, src, dst, pieces, n);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" PKV_API int pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src, const int32_t *dst, int n,
                                       int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                       pkv_stream_t stream) {
    return launch_copy_blocks(k_cache, v_cache, num_blocks, k_cache, v_cache, num_blocks, src, dst, n, num_kv_heads,
                              head_dim, block_size, stream);
}

extern "C" PKV_API int pkv_copy_blocks_between(void *dst_k, void *dst_v, int64_t dst_num_blocks, const void *src_k,
                                               const void *src_v, int64_t src_num_blocks, const int32_t *src_ids,
                                               const int32_t *dst_ids, int n, int num_kv_heads, int head_dim,
                                               int block_size, pkv_stream_t stream) {
    return launch_copy_blocks(dst_k, dst_v, dst_num_blocks, src_k, src_v, src_num_blocks, src_ids, dst_ids, n,
                              num_kv_heads, head_dim, block_size, stream);
}

extern "C" PKV_API int pkv_append_int8k(void *k_codes, float *k_scale, void *v_cache, const int64_t *slot_mapping,
                                        const void *k_new, const void *v_new, int num_tokens, int num_kv_heads,
                                        int head_dim, int block_size, int64_t num_blocks, pkv_stream_t stream) {
    if (!k_codes || !k_scale || !v_cache || (num_tokens > 0 && (!slot_mapping || !k_new || !v_new)))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != PKV_HEAD_DIM) return PKV_ERR_UNSUPPORTED;
    if (!pkv_internal::aligned16(k_codes) || !pkv_internal::aligned(k_scale, 4) || !pkv_internal::aligned16(v_cache) ||
        (num_tokens > 0 && (!pkv_internal::aligned(slot_mapping, 8) || !pkv_internal::aligned(k_new, 8) ||
                            !pkv_internal::aligned(v_new, 8))))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    const int64_t rows = static_cast<int64_t>(num_tokens) * num_kv_heads;
    const int64_t blocks = (rows + kRowsPerAppendBlock - 1) / kRowsPerAppendBlock;
    if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    append_int8k_kernel<false><<<static_cast<unsigned>(blocks), kAppendThreads, 0,
                                 reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint32_t *>(k_codes), k_scale, v_cache, nullptr, slot_mapping, static_cast<const uint2 *>(k_new),
        static_cast<const uint2 *>(v_new), rows, num_kv_heads, block_size, num_blocks * block_size);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" PKV_API int pkv_append_int8kv(void *k_codes, float *k_scale, void *v_codes, float *v_scale,
                                         const int64_t *slot_mapping, const void *k_new, const void *v_new,
                                         int num_tokens, int num_kv_heads, int head_dim, int block_size,
                                         int64_t num_blocks, pkv_stream_t stream) {
    if (!k_codes || !k_scale || !v_codes || !v_scale || (num_tokens > 0 && (!slot_mapping || !k_new || !v_new)))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != PKV_HEAD_DIM) return PKV_ERR_UNSUPPORTED;
    if (!pkv_internal::aligned16(k_codes) || !pkv_internal::aligned(k_scale, 4) || !pkv_internal::aligned16(v_codes) ||
        !pkv_internal::aligned(v_scale, 4) ||
        (num_tokens > 0 && (!pkv_internal::aligned(slot_mapping, 8) || !pkv_internal::aligned(k_new, 8) ||
                            !pkv_internal::aligned(v_new, 8))))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    const int64_t rows = static_cast<int64_t>(num_tokens) * num_kv_heads;
    const int64_t blocks = (rows + kRowsPerAppendBlock - 1) / kRowsPerAppendBlock;
    if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    append_int8k_kernel<true><<<static_cast<unsigned>(blocks), kAppendThreads, 0,
                                reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint32_t *>(k_codes), k_scale, v_codes, v_scale, slot_mapping, static_cast<const uint2 *>(k_new),
        static_cast<const uint2 *>(v_new), rows, num_kv_heads, block_size, num_blocks * block_size);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" PKV_API int pkv_append_fp8kv(void *k_codes, float *k_scale, void *v_codes, float *v_scale,
                                        const int64_t *slot_mapping, const void *k_new, const void *v_new,
                                        int num_tokens, int num_kv_heads, int head_dim, int block_size,
                                        int64_t num_blocks, pkv_stream_t stream) {
    if (!k_codes || !k_scale || !v_codes || !v_scale || (num_tokens > 0 && (!slot_mapping || !k_new || !v_new)))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != PKV_HEAD_DIM) return PKV_ERR_UNSUPPORTED;
    if (!pkv_internal::aligned16(k_codes) || !pkv_internal::aligned(k_scale, 4) || !pkv_internal::aligned16(v_codes) ||
        !pkv_internal::aligned(v_scale, 4) ||
        (num_tokens > 0 && (!pkv_internal::aligned(slot_mapping, 8) || !pkv_internal::aligned(k_new, 8) ||
                            !pkv_internal::aligned(v_new, 8))))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    const int64_t rows = static_cast<int64_t>(num_tokens) * num_kv_heads;
    const int64_t blocks = (rows + kRowsPerAppendBlock - 1) / kRowsPerAppendBlock;
    if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    append_fp8kv_kernel<<<static_cast<unsigned>(blocks), kAppendThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint32_t *>(k_codes), k_scale, static_cast<uint32_t *>(v_codes), v_scale, slot_mapping,
        static_cast<const uint2 *>(k_new), static_cast<const uint2 *>(v_new), rows, num_kv_heads, block_size,
        num_blocks * block_size);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" PKV_API int pkv_append(void *k_cache, void *v_cache, const int64_t *slot_mapping,
                                  const void *k_new, const void *v_new, int num_tokens,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int64_t num_blocks, pkv_stream_t stream) {
    if (!k_cache || !v_cache || !slot_mapping || !k_new || !v_new) return PKV_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
    if (!pkv_internal::aligned16(k_cache) || !pkv_internal::aligned16(v_cache) ||
        !pkv_internal::aligned16(k_new) || !pkv_internal::aligned16(v_new) ||
        !pkv_internal::aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    const int pieces_per_row = head_dim / 8;
    const int64_t pieces = static_cast<int64_t>(num_tokens) * num_kv_heads * pieces_per_row;
    const int64_t blocks = (2 * pieces + kAppendThreads - 1) / kAppendThreads;
    if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    append_kernel<<<static_cast<unsigned>(blocks), kAppendThreads, 0,
                    reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping,
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), pieces, num_kv_heads,
        pieces_per_row, block_size, num_blocks * block_size);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

namespace pkv_internal {

int append_take_error(int *code) {
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_append_error, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_append_error, &zero, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    }
    *code = value;
    return PKV_OK;
}

}  // namespace pkv_internal
