// pkv_prefix.cu -- decode attention for a batch whose block tables share a common prefix.
//
// Requests that start with the same system prompt reference the same KV blocks for it
// ("推理优化这件事，为什么值得反复复盘", sec. 4.2: a shared-prefix cache lets many requests use
// one copy of the prompt's KV; "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 3.2: pages
// shared across requests with the same prompt).  Attention over such a batch is computed in
// two passes and a merge that together equal softmax(scale q K^T) V over each full context:
//
//   1. prefix_kernel: for every kv head and every 128-token chunk of the shared prefix, the
//      scores of ALL requests' query rows that read this kv head (B x G rows) against the
//      chunk, their exact chunk softmax statistics and the normalised P.V, written as
//      partial slots [0, n_chunks) of the split layout.  The prefix's K/V is read once per
//      step instead of once per request.  With B x G rows the scores form a dense
//      (rows x 128 x 128) contraction, so it runs on the tensor cores: warp-level
//      m16n8k16 MMAs, fp16 operands with fp32 accumulation; P is split into fp16 hi + lo
//      parts for the P.V product so the weights keep ~22 bits.
//   2. The ordinary split decode kernel over each request's private suffix (tokens from
//      prefix_len on), writing slots n_chunks.., launched as a programmatic dependent so it
//      streams while the prefix kernel runs.
//   3. A merge launch (one CTA per request and kv head) folding all slots by log-sum-exp
//      (PKV_PREFIX_SEPARATE_MERGE; else the suffix pass's last partition merges after waiting
//      for the prefix kernel).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace {

__device__ int g_prefix_error;

constexpr int kD = PKV_HEAD_DIM;       // 128
// 128-token chunks (with 8 warps, one CTA per SM and 104 KB of shared memory) measured 5.5 % faster
// end to end than 64 (which doubles the CTAs and the prefix slots every merge reads), and 64 than 32.
#ifndef PKV_PREFIX_CHUNK
#define PKV_PREFIX_CHUNK 128
#endif
// Registers per thread of the prefix kernel: at 168 (no spills), a prefix CTA and a 4-warp
// suffix-pass CTA fit an SM's register file together, so the suffix pass streams on the prefix
// kernel's SMs too.
#ifndef PKV_PREFIX_MAXNREG
#define PKV_PREFIX_MAXNREG 168
#endif
// 1: the suffix pass writes its partials and exits; a merge kernel launched after it (one CTA per
// request and kv head) folds the prefix chunks and the suffix partitions.  0: the last suffix CTA
// of each (request, kv head) merges, waiting for the prefix kernel first, which holds a CTA slot
// while the prefix kernel runs (4 % slower on the shared-prefix step).
#ifndef PKV_PREFIX_SEPARATE_MERGE
#define PKV_PREFIX_SEPARATE_MERGE 1
#endif
// 1: the whole step is one launch of the decode kernel: its first CTAs are the prefix tiles (one
// 128-token chunk, one kv head, 64 query rows each, on the 16-row tensor-core engine), the rest the
// suffix pass, and the merge is fused where the last piece of a (request, kv head) lands.
#ifndef PKV_PREFIX_ONE_GRID
#define PKV_PREFIX_ONE_GRID 0
#endif
constexpr int kChunkTok = PKV_PREFIX_CHUNK;  // prefix tokens per CTA (a multiple of 16)
constexpr int kNT = kChunkTok / 8;           // 8-token MMA n-tiles of a chunk
static_assert(kChunkTok % 16 == 0 && kChunkTok >= 16, "chunk of whole 16-token k-steps");
// Warps per prefix CTA (16 query rows each, so 16 x warps rows per row tile).  Four (64 rows, two
// row tiles for the 128 rows of 32 requests x 4 heads: twice the CTAs, each with half the MMA work
// and the same chunk loads from L2) measured 1.5 % faster on the shared-prefix step than eight, and
// two 12 % slower.  The tcgen05 tile is 128 rows.
#ifndef PKV_PREFIX_WARPS
#ifdef PKV_PREFIX_TCGEN05
#define PKV_PREFIX_WARPS (PKV_PREFIX_TCGEN05 ? 8 : 4)
#else
#define PKV_PREFIX_WARPS 4
#endif
#endif
constexpr int kWarps = PKV_PREFIX_WARPS;  // 16 query rows per warp
constexpr int kRows = kWarps * 16;     // query rows per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kPad = kD + 8;           // halves per shared-memory row: 272 B keeps ldmatrix conflict-free
constexpr int kSmemBytes = (2 * kChunkTok + kRows) * kPad * 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct PrefixParams {
    const __half *q;
    const __half *k_cache;
    const __half *v_cache;
    const int32_t *block_tables;  // row 0 holds the shared prefix's blocks
    float *o_part;
    float *m_part;
    float *l_part;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    int prefix_len;
    int max_partitions;
    int64_t num_blocks;
    float q_scale;  // scale * log2(e)
    int overlap;    // 1: stage the prefix's K/V before the preceding kernel completes
    CUtensorMap tmap_k;  // tensor-memory kernel: the K and V caches as [NB*Hkv*bs][128] fp16, 16 x 64 boxes,
    CUtensorMap tmap_v;  //   128-byte swizzle
    CUtensorMap tmap_q;  // tensor-memory kernel: q as [B][Hq][128] fp16, (64, G, 128 / G) boxes, 128-byte swizzle
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void *p) { pkv::ldsm_x4(r, pkv::smem_addr(p)); }

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *p) {
    pkv::ldsm_x4_trans(r, pkv::smem_addr(p));
}

using pkv::mma16816;

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void cp_async16(const void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(pkv::smem_addr(smem_dst)), "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Grid (prefix chunks, kv heads, ceil(B*G / kRows)); kWarps warps, each owning 16 query rows.
__global__ void __maxnreg__(PKV_PREFIX_MAXNREG) prefix_kernel(const PrefixParams P) {  // launched with kThreads threads
    extern __shared__ __align__(128) unsigned char smem[];
    __half *sK = reinterpret_cast<__half *>(smem);      // [kChunkTok][kPad]
    __half *sV = sK + kChunkTok * kPad;                   // [kChunkTok][kPad]
    __half *sQ = sV + kChunkTok * kPad;                   // [kRows][kPad]
    // A programmatic dependent of the kernel before it on the stream: nothing is read before that
    // kernel completes, except with `overlap`, where the prefix's block ids and K/V (which the
    // caller states that kernel does not write) are staged first.  Past the wait the suffix pass
    // may launch and stream the suffixes alongside.
    auto wait_preceding = []() {
        pkv::pdl_wait_primary();
        pkv::pdl_launch_dependents();
    };
    if (!P.overlap) wait_preceding();
    const int chunk = blockIdx.x, kvh = blockIdx.y, rtile = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = P.num_q_heads, Hkv = P.num_kv_heads, G = Hq / Hkv, bs = P.block_size;
    const int rows = P.num_seqs * G;
    const int row0 = rtile * kRows;
    const int tok0 = chunk * kChunkTok;
    const int ntok = min(kChunkTok, P.prefix_len - tok0);

    // K/V chunk (zero rows past the prefix) and the CTA's query rows (zero rows past the last),
    // 16-byte asynchronous copies straight into shared memory: the block ids of the chunk first
    // (one round trip), then every row piece (a second).
    __shared__ int32_t s_ids[kChunkTok / 16];
    const int blk0 = tok0 / bs, nblk = (tok0 + ntok - 1) / bs - blk0 + 1;  // at most kChunkTok / 16
    if (static_cast<int>(threadIdx.x) < nblk) {
        int32_t id = __ldg(P.block_tables + blk0 + threadIdx.x);
        if (id < 0 || id >= P.num_blocks) {
            pkv::record_error(&g_prefix_error, PKV_DEV_BAD_BLOCK_ID);
            id = 0;
        }
        s_ids[threadIdx.x] = id;
    }
    auto stage_q = [&]() {
        for (int i = threadIdx.x; i < kRows * (kD / 8); i += kThreads) {
            const int r = i / (kD / 8), piece = i % (kD / 8);
            const int gr = row0 + r;
            __half *dst = sQ + r * kPad + piece * 8;
            if (gr < rows) {
                const int b = gr / G, hh = gr % G;
                cp_async16(dst, P.q + (static_cast<int64_t>(b) * Hq + kvh * G + hh) * kD + piece * 8);
            } else {
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
            }
        }
    };
    if (!P.overlap) stage_q();
    __syncthreads();  // s_ids
    for (int i = threadIdx.x; i < kChunkTok * (kD / 8); i += kThreads) {
        const int t = i / (kD / 8), piece = i % (kD / 8);
        __half *dk = sK + t * kPad + piece * 8;
        __half *dv = sV + t * kPad + piece * 8;
        if (t < ntok) {
            const int tok = tok0 + t;
            const int64_t src = ((static_cast<int64_t>(s_ids[tok / bs - blk0]) * Hkv + kvh) * bs + tok % bs) * kD +
                                piece * 8;
            cp_async16(dk, P.k_cache + src);
            cp_async16(dv, P.v_cache + src);
        } else {
            *reinterpret_cast<uint4 *>(dk) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(dv) = make_uint4(0, 0, 0, 0);
        }
    }
    if (P.overlap) {  // the prefix is in flight: now q, written by the preceding kernel
        wait_preceding();
        stage_q();
    }
    cp_async_wait_all();
    __syncthreads();
    if (row0 + warp * 16 >= rows) return;  // no barrier follows

    // ---- S = Q K^T for this warp's 16 rows x kChunkTok tokens (kNT n-tiles), K = 128 dims (8 k-steps)
    float s[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
        uint32_t a[4];
        ldmatrix_x4(a, sQ + (warp * 16 + (lane & 15)) * kPad + ks * 16 + (lane >> 4) * 8);
#pragma unroll
        for (int nt = 0; nt < kNT; nt += 2) {
            uint32_t bfr[4];
            ldmatrix_x4(bfr, sK + (nt * 8 + (lane & 7) + (lane >> 4) * 8) * kPad + ks * 16 + ((lane >> 3) & 1) * 8);
            mma16816(s[nt], a, bfr[0], bfr[1]);
            mma16816(s[nt + 1], a, bfr[2], bfr[3]);
        }
    }
    // ---- exact softmax over the chunk for rows g = lane/4 (regs 0,1) and g + 8 (regs 2,3)
    float m_lo = -INFINITY, m_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = nt * 8 + (lane & 3) * 2 + (e & 1);
            s[nt][e] = col < ntok ? s[nt][e] * P.q_scale : -INFINITY;
        }
        m_lo = fmaxf(m_lo, fmaxf(s[nt][0], s[nt][1]));
        m_hi = fmaxf(m_hi, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int sh = 1; sh <= 2; sh <<= 1) {
        m_lo = fmaxf(m_lo, __shfl_xor_sync(pkv::kFullMask, m_lo, sh));
        m_hi = fmaxf(m_hi, __shfl_xor_sync(pkv::kFullMask, m_hi, sh));
    }
    float l_lo = 0.f, l_hi = 0.f;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        s[nt][0] = exp2f(s[nt][0] - m_lo);
        s[nt][1] = exp2f(s[nt][1] - m_lo);
        s[nt][2] = exp2f(s[nt][2] - m_hi);
        s[nt][3] = exp2f(s[nt][3] - m_hi);
        l_lo += s[nt][0] + s[nt][1];
        l_hi += s[nt][2] + s[nt][3];
    }
#pragma unroll
    for (int sh = 1; sh <= 2; sh <<= 1) {
        l_lo += __shfl_xor_sync(pkv::kFullMask, l_lo, sh);
        l_hi += __shfl_xor_sync(pkv::kFullMask, l_hi, sh);
    }

    // ---- O = P V: 16 rows x 128 dims (16 n-tiles), K = kChunkTok tokens, P = hi + lo
    float o[16][4];
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
#pragma unroll
    for (int kt = 0; kt < kChunkTok / 16; ++kt) {
        const float src[8] = {s[2 * kt][0],     s[2 * kt][1],     s[2 * kt][2],     s[2 * kt][3],
                              s[2 * kt + 1][0], s[2 * kt + 1][1], s[2 * kt + 1][2], s[2 * kt + 1][3]};
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            // fragment r: (row g | g+8) x (tokens 16kt + {0..7} | {8..15}): C-fragment pairs
            const float x0 = src[(r >> 1) * 4 + (r & 1) * 2], x1 = src[(r >> 1) * 4 + (r & 1) * 2 + 1];
            const __half2 hi = __floats2half2_rn(x0, x1);
            const float2 hf = __half22float2(hi);
            ph[r] = *reinterpret_cast<const uint32_t *>(&hi);
            pl[r] = pack_half2(x0 - hf.x, x1 - hf.y);
        }
#pragma unroll
        for (int dt = 0; dt < 16; dt += 2) {
            uint32_t vb[4];
            ldmatrix_x4_trans(vb, sV + (kt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7)) * kPad + (dt + (lane >> 4)) * 8);
            mma16816(o[dt], ph, vb[0], vb[1]);
            mma16816(o[dt], pl, vb[0], vb[1]);
            mma16816(o[dt + 1], ph, vb[2], vb[3]);
            mma16816(o[dt + 1], pl, vb[2], vb[3]);
        }
    }

    // ---- partial slot `chunk` of each valid row: normalised o, m in natural-log units, l
    const int g = lane >> 2;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int gr = row0 + warp * 16 + g + half * 8;
        if (gr >= rows) continue;
        const int b = gr / G, hh = gr % G;
        const int64_t prow = (static_cast<int64_t>(b) * Hq + kvh * G + hh) * P.max_partitions + chunk;
        const float l = half ? l_hi : l_lo;
        const float inv = 1.f / l;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            const float2 v = make_float2(o[dt][half * 2] * inv, o[dt][half * 2 + 1] * inv);
            *reinterpret_cast<float2 *>(P.o_part + prow * kD + dt * 8 + (lane & 3) * 2) = v;
        }
        if ((lane & 3) == 0) {
            P.m_part[prow] = (half ? m_hi : m_lo) * kLn2;
            P.l_part[prow] = l;
        }
    }
}

// ---------------------------------------------------------------- tcgen05 / tensor-memory variant
// The same chunk computation as prefix_kernel on the 5th-generation tensor cores: one thread
// issues tcgen05.mma with both operands described in shared memory (128-byte swizzle) and the fp32
// accumulators in tensor memory, so the eight warps hold no accumulator registers.
//   S[128 rows x 128 tokens] = Q[128 x 128 dims] K^T          8 MMAs (M 128, N 128, K 16), TMEM cols 0-127
//   exact chunk softmax: two threads per row (64 columns each, TMEM lanes of their warp), S read
//   back with tcgen05.ld, the row's max and sum exchanged in shared memory, P = hi + lo fp16
//   O[128 rows x 128 dims] = P_hi V + P_lo V                   16 MMAs (K = tokens), TMEM cols 128-255
// Q (a 3-D tensor map over q: 128 / G requests x the G heads of one kv head), K and V arrive by
// tensor copies straight into their operand tiles, all issued by one thread before anything else;
// V enters the P.V product as it arrived (tokens x dims), an MN-major B operand.  O leaves through
// the free tiles so every global store writes a whole 512-byte row.  Tensor memory is allocated and
// freed by warp 0 on every path.  Measured on the shared-prefix step: the MMAs take 0.4 us of a
// CTA's ~7-10 us (the per-row softmax and epilogue phases dominate), and the step is 6 % slower
// than with the mma.sync tile, so the mma.sync tile is the default; this form is built and checked
// against the oracle by its own GPU test.
#ifndef PKV_PREFIX_TCGEN05
#define PKV_PREFIX_TCGEN05 0
#endif
// 1: the prefix CTAs release the suffix pass only once their tensor copies are queued.
#ifndef PKV_PREFIX_LATE_TRIGGER
#define PKV_PREFIX_LATE_TRIGGER 0
#endif
namespace tc5 {
constexpr int kTok = 128;                 // prefix tokens per CTA: N of Q K^T, K of P V
constexpr int kRowsT = 128;               // query rows per CTA: M, one tensor-memory lane each
constexpr int kThreadsT = 256;            // two threads per query row (64 columns each)
constexpr int kAtom = 128 * 128;          // one 64-element K slab of a 128-row operand tile (bytes)
constexpr int kTile = 2 * kAtom;          // 128 rows x 128 K fp16
// Q | K | V^T | barriers, TMEM slot.  P_hi and P_lo reuse the Q and K tiles once S is complete, so
// a prefix CTA (96 KB) leaves room on its SM for a suffix-pass CTA started early.
constexpr int kSmem = 3 * kTile + 64 + 2 * 2 * 128 * 4;  // + the row halves' (max, sum) exchange
constexpr uint32_t kTmemCols = 256;       // S in columns 0-127, O in 128-255
}  // namespace tc5

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// Byte offset of 16-byte chunk c (0..15 along K) of row r in a K-major 128-row operand tile.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
    return (c >> 3) * tc5::kAtom + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(tc5::kThreadsT, 1) prefix_kernel_tmem(const __grid_constant__ PrefixParams P) {
    extern __shared__ __align__(1024) unsigned char smem_tc[];
    unsigned char *smem = smem_tc;
#if !PKV_PREFIX_LATE_TRIGGER
    pkv::pdl_launch_dependents();  // the suffix pass may start streaming right away
#endif
    const uint32_t base = pkv::smem_addr(smem);
    if ((base & 1023) != 0) {  // the swizzled operand tiles need 1 KB alignment (before any allocation)
        if (threadIdx.x == 0) pkv::record_error(&g_prefix_error, PKV_DEV_SMEM_MISALIGNED);
#if PKV_PREFIX_LATE_TRIGGER
        pkv::pdl_launch_dependents();
#endif
        return;
    }
    const uint32_t sQ = base, sK = base + tc5::kTile, sV = base + 2 * tc5::kTile;
    const uint32_t sPh = sQ, sPl = sK;  // written only after the Q K^T MMAs have completed
    const uint32_t tma_bar = base + 3 * tc5::kTile, mma_bar = tma_bar + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + 3 * tc5::kTile + 16);
    int *s_ok = reinterpret_cast<int *>(smem + 3 * tc5::kTile + 20);
    float *s_max = reinterpret_cast<float *>(smem + 3 * tc5::kTile + 64);  // [2 halves][128 rows]
    float *s_sum = s_max + 2 * 128;                                        // [2 halves][128 rows]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Warp w reads tensor-memory lanes 32 (w % 4) .. + 31 (its rows) and columns 64 (w / 4) .. + 63.
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane;
    const int chunk = blockIdx.x, kvh = blockIdx.y, rtile = blockIdx.z;
    const int Hq = P.num_q_heads, Hkv = P.num_kv_heads, G = Hq / Hkv, bs = P.block_size;
    const int rows = P.num_seqs * G;
    const int row0 = rtile * tc5::kRowsT;
    const int tok0 = chunk * tc5::kTok;
    const int ntok = min(tc5::kTok, P.prefix_len - tok0);  // a multiple of 16: the prefix is whole blocks
    const int groups = ntok / 16;

    // Every operand by tensor copies on one barrier, issued before anything else: the CTA's 128 query
    // rows (the 3-D q map: 128 / G requests x the G heads of kv head kvh; rows past the batch read as
    // zeros), and per 16-token group of the chunk two 16 x 64 boxes of K and two of V into the slabs.
    if (tid == 0) {
        pkv::mbar_init(tma_bar, 1);
        pkv::mbar_init(mma_bar, 1);
        pkv::fence_mbar_init();
        pkv::mbar_arrive_expect_tx(tma_bar, 2 * tc5::kAtom + groups * 4 * 2048);
        const int rq = tc5::kRowsT / G;
        pkv::tma_load_3d(sQ, &P.tmap_q, 0, kvh * G, rtile * rq, tma_bar);
        pkv::tma_load_3d(sQ + tc5::kAtom, &P.tmap_q, 64, kvh * G, rtile * rq, tma_bar);
        int32_t ids[tc5::kTok / 16];
#pragma unroll
        for (int g = 0; g < tc5::kTok / 16; ++g) ids[g] = g < groups ? __ldg(P.block_tables + (tok0 + 16 * g) / bs) : 0;
#pragma unroll
        for (int g = 0; g < tc5::kTok / 16; ++g) {
            if (g >= groups) break;
            int32_t id = ids[g];
            if (id < 0 || id >= P.num_blocks) {
                pkv::record_error(&g_prefix_error, PKV_DEV_BAD_BLOCK_ID);
                id = 0;
            }
            const int tok = tok0 + 16 * g;
            const int y = static_cast<int>((static_cast<int64_t>(id) * Hkv + kvh) * bs + tok % bs);
            pkv::tma_load_2d(sK + g * 2048, &P.tmap_k, 0, y, tma_bar);
            pkv::tma_load_2d(sK + tc5::kAtom + g * 2048, &P.tmap_k, 64, y, tma_bar);
            pkv::tma_load_2d(sV + g * 2048, &P.tmap_v, 0, y, tma_bar);
            pkv::tma_load_2d(sV + tc5::kAtom + g * 2048, &P.tmap_v, 64, y, tma_bar);
        }
    }
    if (warp == 0) pkv::tmem_alloc(pkv::smem_addr(tmem_slot), tc5::kTmemCols);
    pkv::tmem_fence_before_sync();
    __syncthreads();
    pkv::tmem_fence_after_sync();
#if PKV_PREFIX_LATE_TRIGGER
    pkv::pdl_launch_dependents();  // the prefix's loads are queued first; the suffix pass may start now
#endif
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_s = tmem, t_o = tmem + 128;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;  // this warp's TMEM lanes

    constexpr uint32_t kIdesc = pkv::umma_idesc_f16_f32(128, 128);
    if (tid == 0) {
        const bool landed = pkv::mbar_wait_bounded(tma_bar, 0);
        if (landed) {
            pkv::tmem_fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * tc5::kAtom + (ks & 3) * 32;
                pkv::umma_f16(t_s, pkv::umma_desc_k_sw128(sQ + off), pkv::umma_desc_k_sw128(sK + off), kIdesc, ks > 0);
            }
            pkv::umma_commit(mma_bar);
        } else {
            pkv::record_error(&g_prefix_error, PKV_DEV_WAIT_TIMEOUT);
        }
        *s_ok = landed ? 1 : 0;
    }
    __syncthreads();
    bool ok = *s_ok != 0 && pkv::mbar_wait_bounded(mma_bar, 0);
    ok = __syncthreads_and(ok);
    pkv::tmem_fence_after_sync();

    // ---- exact softmax of each row over the chunk (log2 domain): this thread's 64 columns, the row's
    // max and sum exchanged with the thread holding the other half; P = hi + lo into the A tiles.
    float m = -INFINITY, l = 0.f;
    const int c_begin = 64 * half;
    uint32_t r[2][32];
    if (ok) {
        pkv::tmem_ld32(t_s + lane_base + c_begin, r[0]);
        pkv::tmem_ld32(t_s + lane_base + c_begin + 32, r[1]);
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 32; ++j)
                mx[j & 3] = fmaxf(mx[j & 3], c_begin + 32 * h + j < ntok ? __uint_as_float(r[h][j]) * P.q_scale : -INFINITY);
        s_max[half * 128 + row] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    }
    __syncthreads();
    if (ok) {
        m = fmaxf(s_max[row], s_max[128 + row]);
        float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    const int c = c_begin + 32 * h + 8 * k + j;
                    const float p0 = c < ntok ? exp2f(__uint_as_float(r[h][8 * k + j]) * P.q_scale - m) : 0.f;
                    const float p1 = c + 1 < ntok ? exp2f(__uint_as_float(r[h][8 * k + j + 1]) * P.q_scale - m) : 0.f;
                    sum[j >> 1] += p0 + p1;
                    const __half2 hh = __floats2half2_rn(p0, p1);
                    const float2 hf = __half22float2(hh);
                    hi[j / 2] = *reinterpret_cast<const uint32_t *>(&hh);
                    lo[j / 2] = pack_half2(p0 - hf.x, p1 - hf.y);
                }
                const uint32_t off = tile_off(row, (c_begin >> 3) + 4 * h + k);
                sts128(sPh + off, make_uint4(hi[0], hi[1], hi[2], hi[3]));
                sts128(sPl + off, make_uint4(lo[0], lo[1], lo[2], lo[3]));
            }
        s_sum[half * 128 + row] = (sum[0] + sum[1]) + (sum[2] + sum[3]);
    }
    pkv::fence_proxy_async_smem();
    pkv::tmem_fence_before_sync();
    __syncthreads();
    if (ok) l = s_sum[row] + s_sum[128 + row];
    if (ok && tid == 0) {
        pkv::tmem_fence_after_sync();
        // O = P V with V as it arrived (tokens x dims): the B operand MN-major, 16 tokens (two 8-row
        // groups, 1 KB apart) per K step, the dims' two 64-wide slabs one slab apart
        constexpr uint32_t kIdescPV = kIdesc | (1u << 16);
        for (int ks = 0; ks < groups; ++ks) {
            const uint32_t off = (ks >> 2) * tc5::kAtom + (ks & 3) * 32;
            const uint64_t vdesc = pkv::umma_desc_mn_sw128(sV + ks * 2048, tc5::kAtom, 1024);
            pkv::umma_f16(t_o, pkv::umma_desc_k_sw128(sPh + off), vdesc, kIdescPV, ks > 0);
        }
        for (int ks = 0; ks < groups; ++ks) {
            const uint32_t off = (ks >> 2) * tc5::kAtom + (ks & 3) * 32;
            const uint64_t vdesc = pkv::umma_desc_mn_sw128(sV + ks * 2048, tc5::kAtom, 1024);
            pkv::umma_f16(t_o, pkv::umma_desc_k_sw128(sPl + off), vdesc, kIdescPV, true);
        }
        pkv::umma_commit(mma_bar);
    }
    if (ok) {
        ok = pkv::mbar_wait_bounded(mma_bar, 1);
        if (!ok && lane == 0) pkv::record_error(&g_prefix_error, PKV_DEV_WAIT_TIMEOUT);
    }
    ok = __syncthreads_and(ok);
    pkv::tmem_fence_after_sync();
    if (ok) {
        // partial slot `chunk` of every row: normalised o, m in natural-log units, l.  Each thread's 64
        // dims go through the free operand tiles (rows padded to 528 B), then every store instruction
        // writes one 512-byte row of o_part contiguously.
        constexpr int kRowPad = kD * 4 + 16;
        const float inv = 1.f / l;
        pkv::tmem_ld32(t_o + lane_base + c_begin, r[0]);
        pkv::tmem_ld32(t_o + lane_base + c_begin + 32, r[1]);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                sts128(base + row * kRowPad + (c_begin + 32 * h + j) * 4,
                       make_uint4(__float_as_uint(__uint_as_float(r[h][j]) * inv),
                                  __float_as_uint(__uint_as_float(r[h][j + 1]) * inv),
                                  __float_as_uint(__uint_as_float(r[h][j + 2]) * inv),
                                  __float_as_uint(__uint_as_float(r[h][j + 3]) * inv)));
        const int gr = row0 + row;
        if (half == 0 && gr < rows) {
            const int64_t prow = (static_cast<int64_t>(gr / G) * Hq + kvh * G + gr % G) * P.max_partitions + chunk;
            P.m_part[prow] = m * kLn2;
            P.l_part[prow] = l;
        }
    }
    __syncthreads();
    if (ok) {
#pragma unroll 1
        for (int i = warp; i < tc5::kRowsT; i += tc5::kThreadsT / 32) {
            const int gri = row0 + i;
            if (gri >= rows) break;
            const int64_t prow = (static_cast<int64_t>(gri / G) * Hq + kvh * G + gri % G) * P.max_partitions + chunk;
            const uint4 v = pkv::lds128(base + i * (kD * 4 + 16) + lane * 16);
            *reinterpret_cast<uint4 *>(P.o_part + prow * kD + lane * 4) = v;
        }
    }
    pkv::tmem_fence_before_sync();
    __syncthreads();
    if (warp == 0) pkv::tmem_dealloc(tmem, tc5::kTmemCols);
}

constexpr int kMinSuffixPartition = 64;
constexpr int kMaxSuffixPartition = 512;
// The suffix partition is halved (from 512) until the suffix grid offers this many CTAs per
// resident CTA slot.
#ifndef PKV_SUFFIX_WAVES
#define PKV_SUFFIX_WAVES 1
#endif

struct SharedLayout {
    int n_pre, n_suf, max_parts, suffix_partition;
    size_t rows, o_bytes, m_bytes, counter_off, total;
};

// Partial-slot layout for a suffix partition size; the workspace size function uses the
// smallest partition, which bounds every layout a call can pick.
SharedLayout shared_layout(int num_seqs, int num_q_heads, int max_context, int prefix_len, int suffix_partition) {
    SharedLayout L{};
    L.suffix_partition = suffix_partition;
    L.n_pre = (prefix_len + kChunkTok - 1) / kChunkTok;
    const int rest = max_context - prefix_len;
    L.n_suf = rest > 0 ? (rest + suffix_partition - 1) / suffix_partition : 0;
    L.max_parts = L.n_pre + L.n_suf;
    L.rows = static_cast<size_t>(num_seqs) * num_q_heads * L.max_parts;
    L.o_bytes = pkv_internal::align256(L.rows * kD * sizeof(float));
    L.m_bytes = pkv_internal::align256(L.rows * sizeof(float));
    L.counter_off = L.o_bytes + 2 * L.m_bytes;
    L.total = L.counter_off + pkv_internal::align256(static_cast<size_t>(num_seqs) * num_q_heads * sizeof(int));
    return L;
}

}  // namespace

extern "C" PKV_API size_t pkv_shared_prefix_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                                           int max_context, int prefix_len) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim != kD || prefix_len <= 0 || max_context < prefix_len) return 0;
    return shared_layout(num_seqs, num_q_heads, max_context, prefix_len, kMinSuffixPartition).total;
}

extern "C" PKV_API int pkv_decode_attention_shared_prefix(
    void *out, const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    const int32_t *context_lens, int num_seqs, int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int64_t num_blocks, float scale, int prefix_len, void *workspace,
    size_t workspace_bytes, pkv_stream_t stream) {
    return pkv_internal::shared_prefix_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                              max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                                              num_blocks, scale, prefix_len, nullptr, nullptr, workspace,
                                              workspace_bytes, stream);
}

namespace pkv_internal {

int shared_prefix_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                         int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, float scale, int prefix_len, const void *k_new, const void *v_new,
                         void *workspace, size_t workspace_bytes, void *stream, bool overlap) {
    int st = check_decode_args(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                               num_q_heads, num_kv_heads, head_dim, block_size, num_blocks);
    if (st != PKV_OK) return st;
    if (!out || !pkv_internal::aligned(out, 8)) return PKV_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID_ARG;
    if (k_new && (!pkv_internal::aligned16(k_new) || !pkv_internal::aligned16(v_new))) return PKV_ERR_INVALID_ARG;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    if (prefix_len <= 0 || prefix_len % block_size != 0 || prefix_len > cap) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    const SharedLayout bound = shared_layout(num_seqs, num_q_heads, static_cast<int>(cap), prefix_len,
                                             kMinSuffixPartition);
    if (!workspace || workspace_bytes < bound.total || !pkv_internal::aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    // Suffix partition: halve from 512 tokens (down to 64) until the suffix grid offers
    // PKV_SUFFIX_WAVES CTAs per resident CTA slot (3 per SM), so short private suffixes still fill
    // the GPU.
    int dev_sm = 0;
    int suffix_part = kMaxSuffixPartition;
    {
        int d = 0;
        if (cudaGetDevice(&d) != cudaSuccess || cudaDeviceGetAttribute(&dev_sm, cudaDevAttrMultiProcessorCount, d) !=
                                                      cudaSuccess)
            return PKV_ERR_CUDA;
        const int64_t want = static_cast<int64_t>(PKV_SUFFIX_WAVES) * 3 * dev_sm;
        const int64_t rest = cap - prefix_len;
        while (suffix_part > kMinSuffixPartition &&
               static_cast<int64_t>(num_seqs) * num_kv_heads * ((rest + suffix_part - 1) / suffix_part) < want)
            suffix_part /= 2;
    }
    const SharedLayout L = shared_layout(num_seqs, num_q_heads, static_cast<int>(cap), prefix_len, suffix_part);
    const int rows = num_seqs * (num_q_heads / num_kv_heads);
    if (num_seqs > 65535 || (rows + kRows - 1) / kRows > 65535) return PKV_ERR_UNSUPPORTED;

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    PrefixParams p{};
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const __half *>(k_cache);
    p.v_cache = static_cast<const __half *>(v_cache);
    p.block_tables = block_tables;
    p.o_part = reinterpret_cast<float *>(ws);
    p.m_part = reinterpret_cast<float *>(ws + L.o_bytes);
    p.l_part = reinterpret_cast<float *>(ws + L.o_bytes + L.m_bytes);
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = block_size;
    p.prefix_len = prefix_len;
    p.max_partitions = L.max_parts;
    p.num_blocks = num_blocks;
    p.q_scale = scale * kLog2e;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev & 63);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
#if PKV_PREFIX_ONE_GRID
    static_assert(kChunkTok == 128, "the one-grid prefix tiles are 128-token chunks");
    (void)configured;
    (void)bit;
    (void)s;
#elif PKV_PREFIX_TCGEN05
    static_assert(kChunkTok == tc5::kTok && kRows == tc5::kRowsT, "partial slots are 128-token chunks of 128 rows");
    const int64_t cache_rows = num_blocks * num_kv_heads * block_size;
    if (cache_rows >= 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    if (pkv_internal::encode_fp16_cache_map(&p.tmap_k, k_cache, cache_rows) != PKV_OK ||
        pkv_internal::encode_fp16_cache_map(&p.tmap_v, v_cache, cache_rows) != PKV_OK ||
        pkv_internal::encode_q_map(&p.tmap_q, q, num_seqs, num_q_heads, num_q_heads / num_kv_heads) != PKV_OK)
        return PKV_ERR_CUDA;
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(prefix_kernel_tmem, cudaFuncAttributeMaxDynamicSharedMemorySize, tc5::kSmem) !=
            cudaSuccess)
            return PKV_ERR_CUDA;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const dim3 grid(L.n_pre, num_kv_heads, (rows + tc5::kRowsT - 1) / tc5::kRowsT);
    prefix_kernel_tmem<<<grid, tc5::kThreadsT, tc5::kSmem, s>>>(p);
#else
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        // The whole shared memory as carveout: an SM running a prefix CTA (104 KB) then still has room
        // for a suffix-pass CTA, which otherwise could not share the SM's smaller configuration.
        if (cudaFuncSetAttribute(prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
                cudaSuccess ||
            cudaFuncSetAttribute(prefix_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    p.overlap = overlap ? 1 : 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(L.n_pre, num_kv_heads, (rows + kRows - 1) / kRows);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, prefix_kernel, p) != cudaSuccess) return PKV_ERR_CUDA;
#endif
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;

    pkv_internal::SplitPass a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.partition_size = L.suffix_partition;
    a.max_partitions = L.max_parts;
    a.token_offset = prefix_len;
    a.slot_offset = L.n_pre;
    a.grid_partitions = L.n_suf > 0 ? L.n_suf : 1;
    a.o_part = p.o_part;
    a.m_part = p.m_part;
    a.l_part = p.l_part;
    a.counters = reinterpret_cast<int *>(ws + L.counter_off);
    a.k_new = k_new;
    a.v_new = v_new;
    a.separate_merge = PKV_PREFIX_SEPARATE_MERGE != 0;
#if PKV_PREFIX_ONE_GRID
    a.prefix_ctas = L.n_pre * num_kv_heads * ((rows + 63) / 64);
    a.prefix_chunks = L.n_pre;
    a.separate_merge = false;
    a.overlap = overlap;
#endif
    return pkv_internal::launch_split_pass(a, stream);
}

}  // namespace pkv_internal

namespace pkv_internal {

int prefix_take_error(int *code) {
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_prefix_error, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_prefix_error, &zero, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    }
    *code = value;
    return PKV_OK;
}

}  // namespace pkv_internal
