// pkv_decode.cu -- decode attention over a paged KV cache on sm_103a.
//
// What is computed ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.2: a decode
// step reads every cached K/V of the request, scores it, normalises with
// softmax and takes the weighted sum of V; sec. 3.2: the cache is paged and
// addressed through a page table):
//
//     out[b][h] = softmax(scale * q[b][h] . K_b^T) . V_b
//
// How (GB300 design; the pages only give the operation):
//   * One CTA owns one (request b, kv head, partition of the context; 1024 tokens by default).
//     All g = Hq/Hkv query heads that read that kv head are packed into the CTA, so every K/V
//     byte is fetched from HBM exactly once per step.
//   * The partition is cut into 16-token chunks; a chunk never straddles a block (block_size is
//     a multiple of 16).  Its K and V rows arrive by 2-D tensor copies (TMA: 16-row x 64-dim
//     boxes of the cache viewed as [rows][128], 128-byte swizzle) into shared memory, counted on
//     an mbarrier with a bounded wait.
//   * Each of the 4 warps streams its own chunks (w, w+4, w+8, ...) through a private 2-stage
//     ring: no block-wide barrier inside the main loop; 3 CTAs per SM.
//   * q . K and P . V run on the tensor cores (mma.m16n8k16, fp32 accumulation): the packed
//     heads are the 8 MMA columns, K comes from the swizzled tile by ldmatrix, P is split into
//     fp16 hi + lo parts.  Variants of the same engine serve int8 keys (codes converted to exact
//     fp16 integers in registers, row scales applied to the finished dot products), int8 keys
//     and values (value scales folded into the weights) and several new tokens per request
//     ((token, head) rows as the 8 columns, or for more than 8 rows per kv head 16 rows as the MMA's
//     M dimension with P kept in registers; causal masks per row).  A CUDA-core engine (packed
//     fp32x2 FMAs) remains behind PKV_DECODE_TC_MIN_GROUP.
//   * Online softmax in fp32 with lazy rescaling: the reference max is only raised (and the
//     accumulators rescaled) when a score exceeds it by more than 2^8; the true max is tracked
//     on the side and everything is re-referenced to it once at the end.
//   * The new token's K/V (decode step) is written by the CTA that owns its position and
//     patched into the staged tile.  At the end the 4 warps' (m, l, acc) are merged in shared
//     memory; the CTA writes the fp16 output when the request fits one partition, else fp32
//     partials, and the last partition CTA of a (request, kv head) to finish merges them by
//     log-sum-exp in the same launch (after a shared prefix, by default a separate merge launch).
//   * Indices read from memory are checked (block ids, context length) and clamped; problems
//     are recorded in the device error word.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace {

__device__ int g_decode_error;

}  // namespace

#include "pkv_engine.cuh"

namespace {

// MQ: 0 one token per request; 1 or 2 several tokens per request, with that many 8-column tiles.
// Copy stages per warp of a kernel variant.
template <int MQ>
constexpr int stages_of() {
    return MQ == 2 ? PKV_DECODE_MQ2_STAGES : kStages;
}
// New token rows a CTA of a fused step stages: one; up to 8 with one 8-column tile (then
// n_b * G <= 8); up to PKV_MAX_STEP_QUERY_LEN with 16 rows.  (Each CTA keeps 3 per SM.)
template <int MQ>
constexpr int new_rows_of() {
    return MQ == 2 ? PKV_MAX_STEP_QUERY_LEN : (MQ ? 8 : 1);
}

// One prefix tile of the one-grid shared-prefix step: CTA (chunk c, kv head kvh, row tile rt) of
// the first P.prefix_ctas.  Its eight 16-token K/V tiles of prefix tokens 128 c .. 128 c + 127 are
// copied once into the stage buffers (swizzled 2-D tensor boxes, as the decode path's; in overlap
// mode before the preceding kernel completes); each warp then runs the 16-row tensor-core engine
// over all eight for its 16 of the tile's 64 query rows (row r of the B * G rows reading kvh is
// request r / G, head r % G) and stores their partial as slot c.  The tile then counts once
// toward the merge of every request it covers; where its arrival is the last, it merges.
template <int G, class L, class Wait>
__device__ __forceinline__ void prefix_tile(const DecodeParams &P, unsigned char *smem, int warp, int lane, bool overlap,
                                         Wait wait_preceding) {
    const int Hkv = P.num_kv_heads, Hq = P.num_q_heads, bs = P.block_size;
    const int c = static_cast<int>(blockIdx.x) % P.prefix_chunks;
    const int kvh = (static_cast<int>(blockIdx.x) / P.prefix_chunks) % Hkv;
    const int rt = static_cast<int>(blockIdx.x) / (P.prefix_chunks * Hkv);
    const int rows = P.num_seqs * G;
    const int prefix_len = P.token_offset;
    const int tok0 = c * 128;
    const int nsub = min(128, prefix_len - tok0) / kChunk;  // the prefix is whole 16-token chunks
    const uint32_t bars = pkv::smem_addr(smem + L::bars);
    const uint32_t tiles = pkv::smem_addr(smem + L::stages);
    const bool smem_ok = (pkv::smem_addr(smem) & 1023) == 0;
    if (!smem_ok && threadIdx.x == 0) pkv::record_error(&g_decode_error, PKV_DEV_SMEM_MISALIGNED);
    if (threadIdx.x == 0) {
        for (int j = 0; j < nsub; ++j) pkv::mbar_init(bars + 8 * j, 1);
        pkv::fence_mbar_init();
    }
    __syncthreads();
    if (smem_ok && static_cast<int>(threadIdx.x) < nsub) {  // thread j stages tile j (cache history)
        const int j = threadIdx.x, tok = tok0 + j * kChunk;
        int32_t id = __ldg(P.block_tables + tok / bs);  // every table starts with the prefix's blocks
        if (id < 0 || id >= P.num_blocks) {
            pkv::record_error(&g_decode_error, PKV_DEV_BAD_BLOCK_ID);
            id = 0;
        }
        const int y = static_cast<int>((static_cast<int64_t>(id) * Hkv + kvh) * bs + tok % bs);
        const uint32_t dst = tiles + j * L::stage, bar = bars + 8 * j;
        pkv::mbar_arrive_expect_tx(bar, 4 * kHalfTile);
        pkv::tma_load_2d(dst, &P.tmap_k, 0, y, bar);
        pkv::tma_load_2d(dst + kHalfTile, &P.tmap_k, 64, y, bar);
        pkv::tma_load_2d(dst + L::k_tile, &P.tmap_v, 0, y, bar);
        pkv::tma_load_2d(dst + L::k_tile + kHalfTile, &P.tmap_v, 64, y, bar);
    }
    if (overlap) wait_preceding();  // q, the workspace and out from here on

    const int rg16 = rt * 4 + warp;  // this warp's 16-row group of the B * G rows
    if (smem_ok && rg16 * 16 < rows) {
        TcEngineR16<G> e;
        e.init(P, 0, 0, 0);
        e.bind(P, kvh, lane, rg16, 0, P.num_seqs, 0x3fffffff);  // requests as rows; every prefix token visible
        bool ok = true;
        for (int j = 0; j < nsub && ok; ++j) {
            ok = __all_sync(pkv::kFullMask, pkv::mbar_wait_bounded(bars + 8 * j, 0));
            if (!ok) {
                if (lane == 0) pkv::record_error(&g_decode_error, PKV_DEV_WAIT_TIMEOUT);
                break;
            }
            const uint32_t kt = tiles + j * L::stage;
            e.qk(kt, 0, kChunk, lane, nullptr, tok0 + j * kChunk);
            e.pv(kt + L::k_tile, kChunk, lane, nullptr);
        }
        e.store_partial(P, lane, rg16, rows, kvh, c);
    }
    // nothing of this CTA's copies left in flight before the stage buffers are reused (bounded)
    if (smem_ok && threadIdx.x == 0)
        for (int j = 0; j < nsub; ++j) pkv::mbar_wait_bounded(bars + 8 * j, 0);
    __syncthreads();  // every warp's partial stores before the arrivals

    // ---- arrivals: one per request of the tile.  A tile never merges: where its arrival is the
    // last piece of a (request, kv head), the count is left complete and the merge launch after the
    // grid folds that pair (a tile's requests with short suffixes would otherwise queue many merges
    // on one CTA).
    const int b_lo = rt * 64 / G, b_hi = min(rt * 64 + 64, rows) / G;
    for (int b = b_lo + static_cast<int>(threadIdx.x); b < b_hi; b += kThreads)
        pkv::atomic_add_acq_rel_gpu(P.counters + static_cast<int64_t>(b) * Hkv + kvh, 1);
    (void)Hq;
}

// SP: the shared-prefix step in one grid: the first P.prefix_ctas CTAs attend over the shared
// prefix (one 128-token chunk, one kv head, 64 query rows each), the rest are the suffix pass; the
// merge of each (request, kv head) is fused where the last of its pieces lands.
template <int G, int LPT, bool TC, int KQ, int MQ, bool SP = false>
__global__ void __launch_bounds__(kThreads, (!TC && G >= 8) ? 2 : (KQ ? PKV_DECODE_KQ_MIN_CTAS : PKV_DECODE_MIN_CTAS))
    decode_partition_kernel(const __grid_constant__ DecodeParams P) {
    static_assert(!KQ || TC, "int8 keys run on the tensor-core engine");
    static_assert(!MQ || (TC && !KQ), "several tokens per request run on the fp16 tensor-core engine");
    static_assert(!SP || (TC && !KQ && !MQ), "the one-grid shared-prefix step reads fp16 K/V, one token per request");
    constexpr int kStages = stages_of<MQ>();  // this variant's ring depth
    using L = SmemLayout<TC, KQ, MQ == 2 ? 2 : 1, kStages, new_rows_of<MQ>()>;
    using Engine = EngineFor<G, LPT, TC, KQ, MQ>;
    constexpr int kRow = L::row;
    constexpr int NC = MQ ? 8 * MQ : G;  // packed output columns per CTA

    extern __shared__ __align__(1024) unsigned char smem[];

    // Launched as a programmatic dependent of the kernel before it on the stream.  The suffix pass
    // after a shared-prefix kernel reads nothing that kernel writes until its merge.  Otherwise the
    // CTA reads nothing before the preceding kernel has completed, except with `overlap`, where it
    // first stages its cache history (tables, context lengths, K/V tiles: what the caller states the
    // preceding kernel does not write) and waits just before it touches q, the new token's rows or
    // any output.  Once past that point, the kernel after this one may start launching: it too
    // touches nothing written here before this grid completes.
    const bool suffix_pass = !SP && P.slot_offset > 0;
    const bool overlap = P.overlap != 0;          // set by the step calls only
    const bool late_q = overlap && !suffix_pass;  // q read after the wait
    auto wait_preceding = [suffix_pass]() {
        if (suffix_pass) return;
        pkv::pdl_wait_primary();
        pkv::pdl_launch_dependents();
    };
    if (!overlap) wait_preceding();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if constexpr (SP) {
        if (static_cast<int>(blockIdx.x) < P.prefix_ctas) {
            prefix_tile<G, L>(P, smem, warp, lane, overlap, wait_preceding);
            return;
        }
    }
    const int n_rg = MQ ? P.n_row_groups : 1;
    const int lin_s = SP ? static_cast<int>(blockIdx.x) - P.prefix_ctas : 0;  // one-grid step: suffix CTA index
    const int part = SP ? lin_s % P.grid_parts : (MQ ? blockIdx.x / n_rg : blockIdx.x);
    const int rg = SP ? 0 : (MQ ? blockIdx.x - part * n_rg : 0);  // row group (fastest: groups share K/V in L2)
    const int kvh = SP ? (lin_s / P.grid_parts) % P.num_kv_heads : blockIdx.y;
    const int b = SP ? lin_s / (P.grid_parts * P.num_kv_heads) : blockIdx.z;
    const int Hq = P.num_q_heads;
    const int bs = P.block_size;
    int q_len = 1;
    int64_t qs_b = b;
    if constexpr (MQ) {
        qs_b = __ldg(P.query_start + b);
        q_len = __ldg(P.query_start + b + 1) - static_cast<int>(qs_b);
        if (q_len < 0 || q_len > P.max_query_len || qs_b < 0 || qs_b + q_len > P.total_q) {
            if (part == 0 && kvh == 0 && rg == 0 && threadIdx.x == 0)
                pkv::record_error(&g_decode_error, PKV_DEV_BAD_CONTEXT);
            return;
        }
        if (rg * NC >= q_len * G) return;  // no live column (also q_len == 0: nothing this step)
    }

    // ---------------------------------------------------------------- extent
    // The block ids of this warp's first chunks and q depend only on (b, kv head, partition):
    // load them now, in parallel with the context length.
    const int cap = P.max_blocks_per_seq * bs;
    // Partition p covers [first(p), first(p + 1)) with first(p) = offset + p * partition_size, less
    // the stagger for odd p; the last partition ends at the context.
    auto part_first = [&P](int p) { return P.token_offset + p * P.partition_size - ((p & 1) ? P.stagger : 0); };
    const int start = part_first(part);
    int32_t first_ids[kStages];
#pragma unroll
    for (int k = 0; k < kStages; ++k) {
        const int tok = start + (warp + k * kWarps) * kChunk;
        first_ids[k] = (lane == 0 && tok < cap)
                           ? __ldg(P.block_tables + static_cast<int64_t>(b) * P.max_blocks_per_seq + tok / bs)
                           : 0;
    }
    Engine eng;
    if (!late_q) eng.init(P, b, kvh, lane);
    int ctx = __ldg(P.context_lens + b);
    if (ctx > cap) {
        if (part == 0 && kvh == 0 && threadIdx.x == 0) pkv::record_error(&g_decode_error, PKV_DEV_BAD_CONTEXT);
        ctx = cap;
    }
    if (ctx < 0) ctx = 0;
    const int ctx_full = ctx;  // several tokens: before the row group's cut below
    if constexpr (MQ) {
        if (ctx < q_len) {  // the new tokens must already be in the cache
            if (part == 0 && kvh == 0 && rg == 0 && threadIdx.x == 0)
                pkv::record_error(&g_decode_error, PKV_DEV_BAD_CONTEXT);
            return;
        }
        if (!late_q) eng.bind(P, kvh, lane, rg, qs_b, q_len, ctx);
        // keys past the group's last live token are visible to none of its columns
        const int last_tok = min(q_len - 1, (rg * NC + NC - 1) / G);
        ctx = ctx - q_len + last_tok + 1;
    }
    const int tok_begin = P.token_offset;  // > 0 only for the suffix pass after a shared prefix
    if (tok_begin > 0 && ctx < tok_begin) {
        if (part == 0 && kvh == 0 && threadIdx.x == 0) pkv::record_error(&g_decode_error, PKV_DEV_BAD_CONTEXT);
        ctx = tok_begin;
    }
    const int n_parts = (ctx - tok_begin + P.partition_size - 1) / P.partition_size;
    const bool direct = P.direct_single && n_parts <= 1 && P.slot_offset == 0;

    if (ctx == 0) {  // empty request: zero output (or an empty partial)
        if (part != 0) return;
        if (overlap) wait_preceding();
        for (int i = threadIdx.x; i < G * kD; i += kThreads) {
            const int hq = kvh * G + i / kD, d = i % kD;
            const int64_t row = static_cast<int64_t>(b) * Hq + hq;
            if (direct) {
                P.out[row * kD + d] = __float2half_rn(0.f);
            } else {
                P.o_part[(row * P.max_partitions) * kD + d] = 0.f;
                if (d == 0) {
                    P.m_part[row * P.max_partitions] = -INFINITY;
                    P.l_part[row * P.max_partitions] = 0.f;
                }
            }
        }
        return;
    }
    // Suffix pass whose merge is a separate launch: this CTA alone waits for the prefix kernel once
    // its own work is done, so the pass cannot complete before the prefix kernel (evaluated where
    // used, so nothing stays live through the main loop; the pass reads fp16 K/V, one token per request).
    auto waits_for_prefix = [&P]() {
        return KQ == 0 && MQ == 0 && P.slot_offset > 0 && P.counters == nullptr && blockIdx.x == 0 &&
               blockIdx.y == 0 && blockIdx.z == 0;
    };
    if (n_parts == 0) {  // shared-prefix pass: the whole context is the prefix, merge its chunks only
        if (SP) return;  // the prefix tiles' last arrival merges
        if (part == 0 && P.counters != nullptr) {
            pkv::pdl_wait_primary();  // the prefix kernel's partials
            merge_group<G, L::stage_bytes>(P, HeadRows{static_cast<int64_t>(b) * Hq + kvh * G}, P.slot_offset, smem);
        } else if (waits_for_prefix()) {
            pkv::pdl_wait_primary();
        }
        return;
    }
    if (part >= n_parts) return;

    const int n_tok = (part == n_parts - 1 ? ctx : part_first(part + 1)) - start;
    const int n_chunks = (n_tok + kChunk - 1) / kChunk;
    const int lb0 = start / bs;
    const int n_bt = (start + n_tok - 1) / bs - lb0 + 1;

    int32_t *s_table = reinterpret_cast<int32_t *>(smem + L::table(G));
    unsigned char *scratch = smem + L::probs + warp * L::probs_per_warp(G);
    // per warp: the K barriers of its stages, then (split K/V) the V barriers
    const uint32_t bar0 = pkv::smem_addr(smem + L::bars) + warp * kStages * kBarsPerStage * 8;
    const uint32_t bar_v0 = bar0 + (kSplitKV ? 8 * kStages : 0);
    const uint32_t stage0 = pkv::smem_addr(smem + L::stages) + warp * kStages * L::stage;
    const uint32_t scale0 = pkv::smem_addr(smem + L::scales) + warp * kStages * L::scale_stride;

    // The 128-byte swizzle needs 1 KB-aligned tiles.  A CTA whose shared memory is not so aligned
    // stages none of its tokens (the error is recorded) but still writes its result and takes part
    // in the split's completion counter, so the merge runs and the counter returns to zero.
    const bool smem_ok = !TC || (pkv::smem_addr(smem) & 1023) == 0;
    if (!smem_ok && threadIdx.x == 0) pkv::record_error(&g_decode_error, PKV_DEV_SMEM_MISALIGNED);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages * kBarsPerStage; ++s) pkv::mbar_init(bar0 + 8 * s, 1);
        pkv::fence_mbar_init();
    }
    const int my_chunks = smem_ok && n_chunks > warp ? (n_chunks - warp + kWarps - 1) / kWarps : 0;
    const int64_t head_stride = static_cast<int64_t>(bs) * kRowBytes;
    const int64_t block_stride = head_stride * P.num_kv_heads;

    // Stage chunk i of this warp (called by all 32 lanes): the CUDA-core engine takes the K and V
    // rows as two contiguous bulk copies, the tensor-core engine four swizzled 2-D tensor boxes.
    // The lambdas capture plain values only: the tensor maps must be read where the grid-constant
    // parameter lives, never from a local copy.
    const unsigned char *kc = P.k_cache;
    const unsigned char *vc = P.v_cache;
    const void *tmap_k = &P.tmap_k;
    const void *tmap_v = &P.tmap_v;
    const float *ksc = P.k_scale;
    const float *vsc = P.v_scale;
    const int hkv = P.num_kv_heads;
    // Logical block of a token: a shift for power-of-two block sizes (a uniform branch), so the
    // per-chunk copy issue carries no integer division.
    const int bs_shift = (bs & (bs - 1)) == 0 ? __ffs(bs) - 1 : -1;
    auto block_of = [bs, bs_shift](int tok) { return bs_shift >= 0 ? tok >> bs_shift : tok / bs; };
    // parts: 1 = K (with the int8 keys' scales), 2 = V, 3 = both.  Without split K/V both land on
    // one barrier with one expect_tx for their sum.
    auto issue_from = [=](int i, int64_t phys, int parts) {
        const int cidx = warp + i * kWarps;
        const int tok0 = start + cidx * kChunk;
        const int valid = min(kChunk, n_tok - cidx * kChunk);
        const int lb = block_of(tok0);
        const int off = tok0 - lb * bs;
        const int64_t byte_off = phys * block_stride + kvh * head_stride + static_cast<int64_t>(off) * kRowBytes;
        const uint32_t bytes = static_cast<uint32_t>(valid) * kRowBytes;
        const int st = i % kStages;
        const uint32_t bar_k = bar0 + 8 * st;
        const uint32_t bar_v = bar_v0 + 8 * st;
        const uint32_t dst = stage0 + st * L::stage;
        // TC: whole 16-row boxes (a ragged tail's extra rows stay inside the block and are masked)
        const uint32_t k_bytes = KQ ? L::k_tile + kChunk * 4 : (TC ? 2 * kHalfTile : bytes);
        const uint32_t v_bytes = KQ >= 2 ? L::v_tile + kChunk * 4 : (TC ? 2 * kHalfTile : bytes);
        if (lane != 0) return;
        if (kSplitKV) {
            if (parts & 1) pkv::mbar_arrive_expect_tx(bar_k, k_bytes);
            if (parts & 2) pkv::mbar_arrive_expect_tx(bar_v, v_bytes);
        } else {
            pkv::mbar_arrive_expect_tx(bar_k, k_bytes + v_bytes);
        }
#if PKV_WAIT_TEST
        // Test build only: the grid's first CTA arms warp 0's first stage for its bytes but issues
        // no copy, so that wait can only run out (nothing is in flight for the stage).
        if (i == 0 && warp == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) return;
#endif
        const int64_t y = (phys * hkv + kvh) * bs + off;
        if (parts & 1) {
            if constexpr (KQ) {  // one 16-row box of int8 keys and the 16 key scales (64 B)
                pkv::tma_load_2d(dst, tmap_k, 0, static_cast<int>(y), bar_k);
                pkv::bulk_copy_g2s(scale0 + st * L::scale_stride, ksc + y, kChunk * 4, bar_k);
            } else if constexpr (TC) {
                pkv::tma_load_2d(dst, tmap_k, 0, static_cast<int>(y), bar_k);
                pkv::tma_load_2d(dst + kHalfTile, tmap_k, 64, static_cast<int>(y), bar_k);
            } else {
                pkv::bulk_copy_g2s(dst, kc + byte_off, bytes, bar_k);
            }
        }
        if (parts & 2) {
            if constexpr (KQ >= 2) {  // one 16-row box of 8-bit value codes and their 16 scales
                pkv::tma_load_2d(dst + L::k_tile, tmap_v, 0, static_cast<int>(y), bar_v);
                pkv::bulk_copy_g2s(scale0 + st * L::scale_stride + kChunk * 4, vsc + y, kChunk * 4, bar_v);
            } else if constexpr (TC) {
                pkv::tma_load_2d(dst + L::k_tile, tmap_v, 0, static_cast<int>(y), bar_v);
                pkv::tma_load_2d(dst + L::k_tile + kHalfTile, tmap_v, 64, static_cast<int>(y), bar_v);
            } else {
                pkv::bulk_copy_g2s(dst + L::k_tile, vc + byte_off, bytes, bar_v);
            }
        }
    };

    auto issue = [=](int i, int parts) {
        const int tok0 = start + (warp + i * kWarps) * kChunk;
        issue_from(i, s_table[block_of(tok0) - lb0], parts);
    };

    // Start-up: each warp reads the block ids of its first chunks straight from the table and
    // issues their copies before the CTA-wide barrier, so the copy latency overlaps the
    // prologue (table slice, q, barrier).
    {
        const int pre = my_chunks < kStages ? my_chunks : kStages;
#pragma unroll
        for (int k = 0; k < kStages; ++k) {
            if (k < pre) {
                const int32_t id = __shfl_sync(pkv::kFullMask, first_ids[k], 0);
                issue_from(k, (id < 0 || id >= P.num_blocks) ? 0 : id, 3);  // bad ids: recorded by the table pass
            }
        }
    }

    {
        const int32_t *bt_row = P.block_tables + static_cast<int64_t>(b) * P.max_blocks_per_seq + lb0;
        for (int i = threadIdx.x; i < n_bt; i += kThreads) {
            int32_t id = __ldg(bt_row + i);
            if (id < 0 || id >= P.num_blocks) {
                pkv::record_error(&g_decode_error, PKV_DEV_BAD_BLOCK_ID);
                id = 0;
            }
            s_table[i] = id;
        }
        if (tok_begin > 0 && part == 0 && kvh == 0 && b > 0) {  // every table must start with the shared prefix
            const int32_t *row_b = P.block_tables + static_cast<int64_t>(b) * P.max_blocks_per_seq;
            for (int i = threadIdx.x; i < tok_begin / bs; i += kThreads)
                if (__ldg(row_b + i) != __ldg(P.block_tables + i))
                    pkv::record_error(&g_decode_error, PKV_DEV_PREFIX_MISMATCH);
        }
    }

    static_assert((kWarps * NC * (kAccStride + 3) + 2 * NC) * 4 <= L::stage_bytes, "combine area must fit the stages");

    if (late_q) {  // the history is in flight: now q and the new rows of the preceding kernel
        wait_preceding();
        eng.init(P, b, kvh, lane);
        if constexpr (MQ) eng.bind(P, kvh, lane, rg, qs_b, q_len, ctx_full);
    }

    // ---- fused append of several new tokens per request (pkv_decode_step_multi): positions
    // ctx_full - q_len .. ctx_full - 1 take rows query_start[b] .. of k_new / v_new.  Every CTA
    // whose token range holds some of them stages those rows in shared memory and patches them
    // into its tiles once the chunks have landed (whatever the copies brought); the CTA of the
    // request's last row group, whose range runs to ctx_full, also writes them to the cache.
    int new_lo = 0, new_hi = 0;
    unsigned char *s_new = smem + L::newrow(G);  // [rows][K row | V row] of the new tokens
    if constexpr (MQ) {
        if (P.k_new != nullptr) {
            new_lo = max(start, ctx_full - q_len);
            // (at most q_len <= max_query_len rows, which the host bounds by the staging's capacity)
            new_hi = min(min(start + n_tok, ctx_full), new_lo + new_rows_of<MQ>());
            const bool writer = rg == (q_len * G - 1) / NC;
            const int64_t t0 = qs_b - (ctx_full - q_len);  // k_new row of position p: t0 + p
            for (int idx = threadIdx.x; idx < (new_hi - new_lo) * 32; idx += kThreads) {
                const int p = new_lo + (idx >> 5), piece = idx & 31;
                const int64_t src = ((t0 + p) * P.num_kv_heads + kvh) * kD + (piece & 15) * 8;
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>((piece < 16 ? P.k_new : P.v_new) + src));
                *reinterpret_cast<uint4 *>(s_new + (p - new_lo) * 2 * kRowBytes + piece * 16) = v;
                if (writer) {
                    const int32_t id = __ldg(P.block_tables + static_cast<int64_t>(b) * P.max_blocks_per_seq + p / bs);
                    if (id >= 0 && id < P.num_blocks) {  // bad ids: recorded by the table pass
                        const int64_t grow = (static_cast<int64_t>(id) * P.num_kv_heads + kvh) * bs + p % bs;
                        *reinterpret_cast<uint4 *>((piece < 16 ? P.k_cache_w : P.v_cache_w) + grow * kD +
                                                   (piece & 15) * 8) = v;
                    }
                }
            }
        }
    }

    // ---- fused append: the CTA holding the request's last position writes the new token's K/V
    // row for its kv head into the cache (lanes 0-15: K, 16-31: V of warp own_warp) and patches the
    // row in its shared-memory tile once the chunk has landed, so the attention sees the new token
    // whatever the order of the global write and the bulk copy.
    const int new_pos = ctx - 1;
    const bool appends = !MQ && P.k_new != nullptr && part == n_parts - 1;
    const int own_chunk = appends ? (new_pos - start) / kChunk : -1;
    const int own_warp = own_chunk % kWarps;
    unsigned char *s_newrow = smem + L::newrow(G);  // [K row | V row] of the new token
    if (appends && warp == own_warp) {
        const int64_t src = (static_cast<int64_t>(b) * P.num_kv_heads + kvh) * kD + (lane & 15) * 8;
        const uint4 new_row = __ldg(reinterpret_cast<const uint4 *>((lane < 16 ? P.k_new : P.v_new) + src));
        const int32_t id = __ldg(P.block_tables + static_cast<int64_t>(b) * P.max_blocks_per_seq + new_pos / bs);
        const bool id_ok = id >= 0 && id < P.num_blocks;
        const int64_t grow = (static_cast<int64_t>(id) * P.num_kv_heads + kvh) * bs + new_pos % bs;
        if constexpr (KQ) {
            // Lanes 0-15 quantise the K row (8 dims each; scale from a 16-lane max), 16-31 move V
            // (or quantise it the same way).
            const uint32_t w[4] = {new_row.x, new_row.y, new_row.z, new_row.w};
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = pkv::half2_bits_to_float2(w[e]);
                f[2 * e] = x.x;
                f[2 * e + 1] = x.y;
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
            for (int sh = 8; sh >= 1; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(pkv::kFullMask, amax, sh));
            const float sc = __fdiv_rn(amax, KQ == 3 ? 448.f : 127.f);
            // this lane's 8 codes, dims in byte order
            auto encode = [&]() {
                uint32_t c[2] = {0u, 0u};
                if constexpr (KQ == 3) {
#pragma unroll
                    for (int e = 0; e < 8; e += 2) c[e >> 2] |= pkv::quantize_e4m3x2(f[e], f[e + 1], sc) << (8 * (e & 3));
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        c[e >> 2] |= (static_cast<uint32_t>(pkv::quantize_int8(f[e], sc)) & 0xffu) << (8 * (e & 3));
                }
                return make_uint2(c[0], c[1]);
            };
            if (lane < 16) {
                const uint2 codes = encode();
                *reinterpret_cast<uint2 *>(s_newrow + lane * 8) = codes;
                if (lane == 0) *reinterpret_cast<float *>(s_newrow + kD) = sc;
                if (id_ok) {
                    *reinterpret_cast<uint2 *>(reinterpret_cast<unsigned char *>(P.k_cache_w) + grow * kD + lane * 8) =
                        codes;
                    if (lane == 0) P.k_scale_w[grow] = sc;
                }
            } else if (KQ >= 2) {  // lanes 16-31 quantise the V row the same way
                const int l16 = lane & 15;
                const uint2 codes = encode();
                *reinterpret_cast<uint2 *>(s_newrow + 2 * kD + l16 * 8) = codes;
                if (l16 == 0) *reinterpret_cast<float *>(s_newrow + 3 * kD) = sc;
                if (id_ok) {
                    *reinterpret_cast<uint2 *>(reinterpret_cast<unsigned char *>(P.v_cache_w) + grow * kD + l16 * 8) =
                        codes;
                    if (l16 == 0) P.v_scale_w[grow] = sc;
                }
            } else {
                *reinterpret_cast<uint4 *>(s_newrow + lane * 16) = new_row;
                if (id_ok) *reinterpret_cast<uint4 *>(P.v_cache_w + grow * kD + (lane & 15) * 8) = new_row;
            }
        } else {
            *reinterpret_cast<uint4 *>(s_newrow + lane * 16) = new_row;
            if (id_ok) *reinterpret_cast<uint4 *>((lane < 16 ? P.k_cache_w : P.v_cache_w) + grow * kD + (lane & 15) * 8) =
                new_row;
        }
    }

    __syncthreads();  // table + barrier init visible to every warp


    // Per chunk: wait for K, patch the appended token's K row, q.K and softmax, refill the K stage
    // (split K/V), wait for V, clear a ragged tail's V rows (the MMA reads all 16), patch the V
    // row, P.V, refill the V stage.  Without split K/V one wait covers both and one refill
    // issues both.
    int consumed_k = 0, consumed_v = 0;  // chunks whose K / V wait succeeded
    int issued_k = my_chunks < kStages ? my_chunks : kStages, issued_v = issued_k;
    bool aborted = false;
    auto landed = [&](uint32_t bar, int i) {
        const bool ok = pkv::mbar_wait_bounded(bar, (i / kStages) & 1);
        if (__all_sync(pkv::kFullMask, ok)) return true;  // warp-uniform decision
        if (lane == 0) pkv::record_error(&g_decode_error, PKV_DEV_WAIT_TIMEOUT);
        aborted = true;
        return false;
    };
    for (int i = 0; i < my_chunks; ++i) {
        const int st = i % kStages;
        if (!landed(bar0 + 8 * st, i)) break;
        consumed_k = i + 1;
        if (!kSplitKV) consumed_v = i + 1;
        const int cidx = warp + i * kWarps;
        const int valid = min(kChunk, n_tok - cidx * kChunk);
        const uint32_t k_tile = stage0 + st * L::stage;
        const uint32_t v_tile = k_tile + L::k_tile;
        const uint32_t s_tile = scale0 + st * L::scale_stride;
        const bool own = cidx == own_chunk;
        const int nr_row = (new_pos - start) % kChunk;
        // several-token step: rows [r0, r1) of this chunk are new tokens staged in s_new
        const int tok0c = start + cidx * kChunk;
        const int r0 = max(new_lo - tok0c, 0), r1 = min(new_hi - tok0c, kChunk);
        auto patch_new = [&](uint32_t tile, int half) {
            for (int x = lane; x < (r1 - r0) * 16; x += 32) {
                const int r = r0 + (x >> 4), pc = x & 15;
                const uint4 nr =
                    *reinterpret_cast<const uint4 *>(s_new + (tok0c + r - new_lo) * 2 * kRowBytes + half * kRowBytes + pc * 16);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(tile + TcEngine<4>::swz(r, pc)), "r"(nr.x),
                             "r"(nr.y), "r"(nr.z), "r"(nr.w)
                             : "memory");
            }
        };
        // the appended token's V row and a ragged tail's V rows, once V has landed
        auto fix_v = [&]() {
            bool touched = false;
            // (int8 values need no clearing: codes are finite and the scaled weights of the unused
            // rows are forced to zero; fp8 codes include NaN, so their unused rows are zeroed)
            if (TC && KQ != 2 && KQ != 3 && valid < kChunk) {
                for (int x = lane; x < (kChunk - valid) * 16; x += 32)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(v_tile + TcEngine<4>::swz(valid + x / 16, x % 16)),
                                 "r"(0)
                                 : "memory");
                touched = true;
            }
            if (KQ == 3 && valid < kChunk) {
                for (int x = lane; x < (kChunk - valid) * 8; x += 32)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(v_tile + TcEngineQ<G>::swz8(valid + x / 8, x % 8)),
                                 "r"(0)
                                 : "memory");
                touched = true;
            }
            if (own) {
                if (KQ >= 2 && lane >= 16) {  // 8-bit value row (8 bytes a lane) and its scale
                    const int l16 = lane & 15;
                    const uint2 nc = *reinterpret_cast<const uint2 *>(s_newrow + 2 * kD + l16 * 8);
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(v_tile + TcEngineQ<G>::swz8(nr_row, l16 >> 1) +
                                                                     (l16 & 1) * 8),
                                 "r"(nc.x), "r"(nc.y)
                                 : "memory");
                    if (l16 == 0)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(s_tile + kChunk * 4 + nr_row * 4),
                                     "f"(*reinterpret_cast<const float *>(s_newrow + 3 * kD))
                                     : "memory");
                } else if (KQ < 2 && lane >= 16) {
                    const uint4 nr = *reinterpret_cast<const uint4 *>(s_newrow + lane * 16);
                    const uint32_t row = TC ? TcEngine<4>::swz(nr_row, lane & 15) : nr_row * kRow + (lane & 15) * 16;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(v_tile + row), "r"(nr.x), "r"(nr.y),
                                 "r"(nr.z), "r"(nr.w)
                                 : "memory");
                }
                touched = true;
            }
            if (MQ && r1 > r0) {
                patch_new(v_tile, 1);
                touched = true;
            }
            return touched;
        };
        bool touched = false;
        if (own) {  // the appended token's K row (lanes 0-15): overwrite what the copy brought
            if (lane < 16) {
                if (KQ) {
                    const uint2 nc = *reinterpret_cast<const uint2 *>(s_newrow + lane * 8);
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(k_tile + TcEngineQ<G>::swz8(nr_row, lane >> 1) +
                                                                         (lane & 1) * 8),
                                 "r"(nc.x), "r"(nc.y)
                                 : "memory");
                    if (lane == 0)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(s_tile + nr_row * 4),
                                     "f"(*reinterpret_cast<const float *>(s_newrow + kD))
                                     : "memory");
                } else {
                    const uint4 nr = *reinterpret_cast<const uint4 *>(s_newrow + lane * 16);
                    const uint32_t row = TC ? TcEngine<4>::swz(nr_row, lane & 15) : nr_row * kRow + (lane & 15) * 16;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(k_tile + row), "r"(nr.x), "r"(nr.y),
                                 "r"(nr.z), "r"(nr.w)
                                 : "memory");
                }
            }
            touched = true;
        }
        if (MQ && r1 > r0) {  // the new tokens' K rows
            patch_new(k_tile, 0);
            touched = true;
        }
        if (!kSplitKV) touched |= fix_v();
        if (touched) __syncwarp();
        eng.qk(k_tile, s_tile, valid, lane, scratch, start + cidx * kChunk);
        if (kSplitKV) {
            if (i + kStages < my_chunks) {
                pkv::fence_proxy_async_smem();
                issue(i + kStages, 1);
                ++issued_k;
            }
            if (!landed(bar_v0 + 8 * st, i)) break;
            consumed_v = i + 1;
            if (fix_v()) __syncwarp();
        }
        eng.pv(v_tile, valid, lane, scratch);
        __syncwarp();
        if (i + kStages < my_chunks) {
            pkv::fence_proxy_async_smem();
            issue(i + kStages, kSplitKV ? 2 : 3);
            if (!kSplitKV) ++issued_k;
            ++issued_v;
        }
    }
    if (aborted) {
        // Let this warp's copies still in flight land before the buffers are reused (bounded waits).
        for (int i = consumed_k; i < issued_k; ++i) pkv::mbar_wait_bounded(bar0 + 8 * (i % kStages), (i / kStages) & 1);
        if (kSplitKV)
            for (int i = consumed_v; i < issued_v; ++i)
                pkv::mbar_wait_bounded(bar_v0 + 8 * (i % kStages), (i / kStages) & 1);
    }

    // ---- merge the 4 warps in shared memory (reusing the stage buffers)
    __syncthreads();
    float *c_acc = reinterpret_cast<float *>(smem);                  // [kWarps][NC][kAccStride]
    float *c_m = c_acc + kWarps * NC * kAccStride;                   // [kWarps][NC]
    float *c_l = c_m + kWarps * NC;                                  // [kWarps][NC]
    float *c_f = c_l + kWarps * NC;                                  // [kWarps][NC] weight of each warp
    float *c_row = c_f + kWarps * NC;                                // [2][NC] row max, row sum
    eng.finish(warp, lane, c_acc, c_m, c_l);
    __syncthreads();
    // Per row, once: the max over the warps, each warp's weight 2^(m_w - M) (0 for a warp without
    // chunks; with causal masking a column can have seen no token at all) and the weighted sum of l.
    // The element pass below then has no dependent chain longer than the four warps' FMAs, so its
    // iterations overlap (one row after another, it cost ~0.35 us per row).
    if (threadIdx.x < NC) {
        const int hh = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, c_m[w * NC + hh]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float cm = c_m[w * NC + hh];
            const float f = (MQ && cm == -INFINITY) ? 0.f : exp2f(cm - M);
            c_f[w * NC + hh] = f;
            L = fmaf(c_l[w * NC + hh], f, L);
        }
        c_row[hh] = M;
        c_row[NC + hh] = L;
    }
    __syncthreads();
    const TokenRows<G, NC> token_rows{qs_b, q_len, rg, Hq, kvh};
    // Four consecutive dims per thread and iteration (16-byte shared loads and global stores):
    // with the SM's other CTAs streaming, the pass's cost is its instruction count.
    constexpr int kQuads = kD / 4;
    constexpr int kUnroll = MQ ? 1 : 4;  // the 16-row engine's kernel has no registers to spare
#pragma unroll kUnroll
    for (int idx = threadIdx.x; idx < NC * kQuads; idx += kThreads) {
        const int hh = idx / kQuads, d = 4 * (idx % kQuads);
        if (MQ && !token_rows.live(hh)) continue;
        float O[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float4 a = *reinterpret_cast<const float4 *>(c_acc + (w * NC + hh) * kAccStride + d);
            const float f = c_f[w * NC + hh];
            O[0] = fmaf(a.x, f, O[0]);
            O[1] = fmaf(a.y, f, O[1]);
            O[2] = fmaf(a.z, f, O[2]);
            O[3] = fmaf(a.w, f, O[3]);
        }
        const float L = c_row[NC + hh];
        const int64_t row = MQ ? token_rows.row(hh) : static_cast<int64_t>(b) * Hq + kvh * G + hh;
        float o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = (MQ && L == 0.f) ? 0.f : O[k] / L;
        if (direct) {
            const __half2 lo = __floats2half2_rn(o[0], o[1]), hi = __floats2half2_rn(o[2], o[3]);
            *reinterpret_cast<uint2 *>(P.out + row * kD + d) =
                make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
        } else {
            const int64_t prow = row * P.max_partitions + P.slot_offset + part;
            *reinterpret_cast<float4 *>(P.o_part + prow * kD + d) = make_float4(o[0], o[1], o[2], o[3]);
            if (d == 0) {
                P.m_part[prow] = c_row[hh] * kLn2;
                P.l_part[prow] = L;
            }
        }
    }
    if (direct || P.counters == nullptr) {
        if (waits_for_prefix()) pkv::pdl_wait_primary();
        return;
    }

    // ---- fused log-sum-exp merge: the last partition CTA of (b, kv head) to finish merges them all.
    // The CTA's partial writes are ordered before one acquire-release increment of the counter by
    // thread 0 (barrier, then atom.acq_rel.gpu); the CTA that sees the final count reads every
    // partial from L2 (ld.global.cg) after a second barrier, then returns the counter to zero.
    __shared__ int s_last;
    __syncthreads();
    int *counter = P.counters + (static_cast<int64_t>(b) * P.num_kv_heads + kvh) * n_rg + rg;
    if (threadIdx.x == 0)
        s_last = pkv::atomic_add_acq_rel_gpu(counter, 1) == n_parts + (SP ? P.prefix_chunks : 0) - 1;
    __syncthreads();
    if (!s_last) return;
    if (!SP && P.slot_offset > 0) pkv::pdl_wait_primary();  // shared-prefix pass: the prefix kernel's partials
    if constexpr (MQ)
        merge_group<NC, L::stage_bytes>(P, token_rows, P.slot_offset + n_parts, smem);
    else
        merge_group<G, L::stage_bytes>(P, HeadRows{static_cast<int64_t>(b) * Hq + kvh * G}, P.slot_offset + n_parts,
                                       smem);
    if (threadIdx.x == 0) *counter = 0;
}

// The shared-prefix merge as its own launch: one CTA per (kv head, request) runs the fused merge
// (same code, same result) over the prefix chunks and the suffix partitions, after waiting
// (griddepcontrol.wait) for the suffix pass, which completes only after the prefix kernel.
constexpr int kMergeStageBytes = 24 * 1024;
template <int G>
__global__ void __launch_bounds__(kThreads) merge_groups_kernel(const __grid_constant__ DecodeParams P) {
    __shared__ __align__(16) unsigned char smem[kMergeStageBytes];
    pkv::pdl_wait_primary();
    pkv::pdl_launch_dependents();  // the next step's first kernel touches nothing written here early
    const int kvh = blockIdx.x, b = blockIdx.y;
    // the suffix pass's partition count for this request (same clamps)
    const int cap = P.max_blocks_per_seq * P.block_size;
    int ctx = __ldg(P.context_lens + b);
    ctx = max(min(ctx, cap), P.token_offset);
    const int n_parts = (ctx - P.token_offset + P.partition_size - 1) / P.partition_size;
    int *counter = nullptr;
    if (P.prefix_ctas > 0) {  // one-grid step: only pairs whose last piece was a prefix tile remain
        counter = P.counters + static_cast<int64_t>(b) * P.num_kv_heads + kvh;
        if (__ldcg(counter) != P.prefix_chunks + n_parts) return;  // 0: merged in the grid
    }
    merge_group<G, kMergeStageBytes>(P, HeadRows{static_cast<int64_t>(b) * P.num_q_heads + kvh * G},
                                     P.slot_offset + n_parts, smem);
    if (counter && threadIdx.x == 0) *counter = 0;
}

// One CTA per (q head, request); thread d owns output dim d.  Partitions are taken in tiles
// of 128: the tile's (m, l) pairs are loaded in parallel (one per thread), the weights
// w_p = l_p exp(m_p - M) go to shared memory, then every thread issues its tile of o loads
// independently, so a tile costs a few memory round trips instead of one per partition.
__global__ void __launch_bounds__(kD) merge_kernel(__half *__restrict__ out, const float *__restrict__ o_part,
                                                   const float *__restrict__ m_part,
                                                   const float *__restrict__ l_part,
                                                   const int32_t *__restrict__ context_lens, int num_q_heads,
                                                   int partition_size, int max_partitions, int skip_single) {
    __shared__ float s_w[kD];
    __shared__ float s_red[kD / 32];
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int d = threadIdx.x;
    const int lane = d & 31, warp = d >> 5;
    int ctx = __ldg(context_lens + b);
    if (ctx < 0) ctx = 0;
    int n_parts = (ctx + partition_size - 1) / partition_size;
    if (n_parts > max_partitions) {
        if (h == 0 && d == 0) pkv::record_error(&g_decode_error, PKV_DEV_BAD_CONTEXT);
        n_parts = max_partitions;
    }
    if (skip_single && n_parts <= 1) return;  // written by the partition kernel
    const int64_t row = static_cast<int64_t>(b) * num_q_heads + h;
    if (n_parts == 0) {
        out[row * kD + d] = __float2half_rn(0.f);
        return;
    }
    const float *m = m_part + row * max_partitions;
    const float *l = l_part + row * max_partitions;
    const float *o = o_part + row * max_partitions * kD + d;

    // M = max over partitions (block reduction)
    float M = -INFINITY;
    for (int p = d; p < n_parts; p += kD) M = fmaxf(M, __ldg(m + p));
#pragma unroll
    for (int sh = 16; sh >= 1; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(pkv::kFullMask, M, sh));
    if (lane == 0) s_red[warp] = M;
    __syncthreads();
    M = s_red[0];
#pragma unroll
    for (int w = 1; w < kD / 32; ++w) M = fmaxf(M, s_red[w]);

    float wsum = 0.f, acc = 0.f;
    for (int p0 = 0; p0 < n_parts; p0 += kD) {
        const int n = min(kD, n_parts - p0);
        __syncthreads();  // previous tile's weights consumed
        if (d < n) s_w[d] = __ldg(l + p0 + d) * expf(__ldg(m + p0 + d) - M);
        __syncthreads();
        int p = 0;
        for (; p + 4 <= n; p += 4) {
            const float o0 = __ldg(o + static_cast<int64_t>(p0 + p) * kD);
            const float o1 = __ldg(o + static_cast<int64_t>(p0 + p + 1) * kD);
            const float o2 = __ldg(o + static_cast<int64_t>(p0 + p + 2) * kD);
            const float o3 = __ldg(o + static_cast<int64_t>(p0 + p + 3) * kD);
            acc = fmaf(s_w[p], o0, acc);
            acc = fmaf(s_w[p + 1], o1, acc);
            acc = fmaf(s_w[p + 2], o2, acc);
            acc = fmaf(s_w[p + 3], o3, acc);
            wsum += s_w[p] + s_w[p + 1] + s_w[p + 2] + s_w[p + 3];
        }
        for (; p < n; ++p) {
            acc = fmaf(s_w[p], __ldg(o + static_cast<int64_t>(p0 + p) * kD), acc);
            wsum += s_w[p];
        }
    }
    out[row * kD + d] = __float2half_rn(acc / wsum);
}

// ------------------------------------------------------------------ host side

template <int G>
constexpr int lanes_per_token() {
    return G >= 8 ? 16 : 8;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

// The cache as a 2-D fp16 tensor [rows][128] (rows = NB * Hkv * bs, 256-byte row stride) read in
// 16-row x 64-dim boxes with the 128-byte swizzle.
int encode_cache_map(CUtensorMap *map, const void *base, int64_t rows) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return PKV_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kChunk)};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// The int8 key codes as a 2-D byte tensor [rows][128] read in 16-row x 128-byte boxes, same swizzle.
int encode_code_map(CUtensorMap *map, const void *base, int64_t rows) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return PKV_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kChunk)};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

template <int G, int KQ, int MQ, bool SP = false>
int launch_partition(const DecodeParams &p_in, int num_seqs, cudaStream_t stream, int grid_parts) {
    constexpr int LPT = lanes_per_token<G>();
    constexpr bool TC = SP || KQ || MQ || (PKV_DECODE_TC && G >= PKV_DECODE_TC_MIN_GROUP);
    auto kernel = decode_partition_kernel<G, LPT, TC, KQ, MQ, SP>;
    DecodeParams p = p_in;
    if (TC) {
        const int64_t rows = p.num_blocks * p.num_kv_heads * p.block_size;
        if (rows >= 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // box row coordinates are signed 32-bit
        int st = KQ ? encode_code_map(&p.tmap_k, p.k_cache, rows) : encode_cache_map(&p.tmap_k, p.k_cache, rows);
        if (st == PKV_OK)
            st = KQ >= 2 ? encode_code_map(&p.tmap_v, p.v_cache, rows) : encode_cache_map(&p.tmap_v, p.v_cache, rows);
        if (st != PKV_OK) return st;
    }
    using L = SmemLayout<TC, KQ, MQ == 2 ? 2 : 1, stages_of<MQ>(), new_rows_of<MQ>()>;
    // three fp16 tensor-core CTAs per SM at the default partition (228 KB; 1 KB static and 1 KB
    // reserved per CTA)
    static_assert(!TC || KQ || 3 * (L::total(G, PKV_DEFAULT_PARTITION) + 2048) <= 228 * 1024, "3 CTAs per SM");
    const int smem = L::total(G, p.partition_size + p.stagger);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    static std::atomic<uint64_t> configured{0};  // one bit per device
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::total(G, PKV_MAX_PARTITION)) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const int64_t gx = static_cast<int64_t>(grid_parts > 0 ? grid_parts : p.max_partitions) * (MQ ? p.n_row_groups : 1);
    if (gx > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(gx), p.num_kv_heads, num_seqs);
    if (SP) {  // one dimension: the prefix tiles, then (partition, kv head, request) fastest first
        const int64_t n = p.prefix_ctas + gx * p.num_kv_heads * num_seqs;
        if (n > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
        p.grid_parts = static_cast<int>(gx);
        p.num_seqs = num_seqs;
        grid = dim3(static_cast<unsigned>(n));
    }
    // Always a programmatic dependent of the preceding kernel: its CTAs may become resident while
    // that kernel drains (the kernel waits, see above).  The suffix pass after the shared-prefix
    // kernel streams the suffixes while the prefix kernel runs; only its merges wait for the prefix.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <int G>
int launch_mode(const DecodeParams &p, int num_seqs, cudaStream_t stream, int grid_parts) {
    if (p.prefix_ctas > 0) return launch_partition<G, 0, 0, true>(p, num_seqs, stream, grid_parts);
    if (p.query_start)
        return p.mq_tiles == 2 ? launch_partition<G, 0, 2>(p, num_seqs, stream, grid_parts)
                               : launch_partition<G, 0, 1>(p, num_seqs, stream, grid_parts);
    if (p.k_scale && p.v_scale)
        return p.kv_fp8 ? launch_partition<G, 3, 0>(p, num_seqs, stream, grid_parts)
                        : launch_partition<G, 2, 0>(p, num_seqs, stream, grid_parts);
    if (p.k_scale) return launch_partition<G, 1, 0>(p, num_seqs, stream, grid_parts);
    return launch_partition<G, 0, 0>(p, num_seqs, stream, grid_parts);
}

int dispatch_partition(const DecodeParams &p, int num_seqs, int group, cudaStream_t stream, int grid_parts = 0) {
    switch (group) {
        case 1: return launch_mode<1>(p, num_seqs, stream, grid_parts);
        case 2: return launch_mode<2>(p, num_seqs, stream, grid_parts);
        case 4: return launch_mode<4>(p, num_seqs, stream, grid_parts);
        case 8: return launch_mode<8>(p, num_seqs, stream, grid_parts);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

int check_common(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
                 const int32_t *context_lens, int num_seqs, int max_blocks_per_seq, int num_q_heads,
                 int num_kv_heads, int head_dim, int block_size, int64_t num_blocks) {
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        block_size <= 0 || num_blocks <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != kD) return PKV_ERR_UNSUPPORTED;
    if (block_size % PKV_MIN_BLOCK_SIZE != 0 || block_size > PKV_MAX_BLOCK_SIZE) return PKV_ERR_UNSUPPORTED;
    if (num_blocks > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    const int g = num_q_heads / num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_UNSUPPORTED;
    if (!pkv_internal::aligned16(q) || !pkv_internal::aligned16(k_cache) || !pkv_internal::aligned16(v_cache) ||
        !pkv_internal::aligned(block_tables, 4) || !pkv_internal::aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

using pkv_internal::align256;

constexpr int kStaggerMinParts = 8;
constexpr int kStaggerMinWaves = 3;

// Split workspace layout: o_part | m_part | l_part | counters, each 256-byte aligned.
size_t counters_offset(size_t rows) {
    return align256(rows * kD * sizeof(float)) + 2 * align256(rows * sizeof(float));
}

}  // namespace

extern "C" PKV_API size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim, int max_context,
                                                    int partition_size) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context <= 0 || partition_size <= 0) return 0;
    const size_t parts = (static_cast<size_t>(max_context) + partition_size - 1) / partition_size;
    if (parts <= 1) return 0;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * parts;
    return align256(rows * head_dim * sizeof(float)) + 2 * align256(rows * sizeof(float)) +
           align256(static_cast<size_t>(num_seqs) * num_q_heads * sizeof(int));
}

extern "C" PKV_API int pkv_decode_partition(float *o_part, float *m_part, float *l_part, const void *q,
                                            const void *k_cache, const void *v_cache,
                                            const int32_t *block_tables, const int32_t *context_lens,
                                            int num_seqs, int max_blocks_per_seq, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                            float scale, int partition_size, int max_partitions,
                                            pkv_stream_t stream) {
    int st = check_common(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks);
    if (st != PKV_OK) return st;
    if (!o_part || !m_part || !l_part) return PKV_ERR_INVALID_ARG;
    if (!pkv_internal::aligned16(o_part) || !pkv_internal::aligned(m_part, 4) || !pkv_internal::aligned(l_part, 4))
        return PKV_ERR_INVALID_ARG;
    if (partition_size < kChunk || partition_size > PKV_MAX_PARTITION || partition_size % kChunk != 0)
        return PKV_ERR_UNSUPPORTED;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    if (max_partitions < (cap + partition_size - 1) / partition_size || max_partitions > 0x7fffffff)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    DecodeParams p{};
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const unsigned char *>(k_cache);
    p.v_cache = static_cast<const unsigned char *>(v_cache);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.o_part = o_part;
    p.m_part = m_part;
    p.l_part = l_part;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.q_scale = scale * kLog2e;
    p.partition_size = partition_size;
    p.max_partitions = max_partitions;
    p.direct_single = 0;
    return dispatch_partition(p, num_seqs, num_q_heads / num_kv_heads, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" PKV_API int pkv_merge(void *out, const float *o_part, const float *m_part, const float *l_part,
                                 const int32_t *context_lens, int num_seqs, int num_q_heads, int head_dim,
                                 int partition_size, int max_partitions, pkv_stream_t stream) {
    if (!out || !o_part || !m_part || !l_part || !context_lens) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || partition_size <= 0 || max_partitions <= 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != kD) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    merge_kernel<<<dim3(num_q_heads, num_seqs), kD, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<__half *>(out), o_part, m_part, l_part, context_lens, num_q_heads, partition_size,
        max_partitions, 0);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

namespace {

// pkv_decode_attention, optionally appending the new token first (k_new/v_new non-null).
// k_scale non-null: k_cache holds int8 codes with these float32 row scales (v_scale too: so does
// v_cache).  kv_fp8 (with both scales): the codes are E4M3 instead of int8.
int decode_attention_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                          int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int64_t num_blocks, float scale, const void *k_new, const void *v_new, void *workspace,
                          size_t workspace_bytes, pkv_stream_t stream, const float *k_scale = nullptr,
                          int partition_size = PKV_DEFAULT_PARTITION, const float *v_scale = nullptr,
                          unsigned flags = 0, bool kv_fp8 = false) {
    if (flags & ~PKV_STEP_OVERLAP) return PKV_ERR_INVALID_ARG;
    int st = check_common(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks);
    if (st != PKV_OK) return st;
    if (k_scale && !pkv_internal::aligned16(k_scale)) return PKV_ERR_INVALID_ARG;
    if (v_scale && (!k_scale || !pkv_internal::aligned16(v_scale))) return PKV_ERR_INVALID_ARG;
    if (kv_fp8 && !v_scale) return PKV_ERR_INVALID_ARG;
    if (!out || !pkv_internal::aligned(out, 8)) return PKV_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID_ARG;
    if (k_new && (!pkv_internal::aligned16(k_new) || !pkv_internal::aligned16(v_new))) return PKV_ERR_INVALID_ARG;
    if (partition_size < kChunk || partition_size > PKV_MAX_PARTITION || partition_size % kChunk != 0)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    const int part = partition_size;
    const int max_parts = static_cast<int>((cap + part - 1) / part);
    DecodeParams p{};
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const unsigned char *>(k_cache);
    p.v_cache = static_cast<const unsigned char *>(v_cache);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<__half *>(out);
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.q_scale = scale * kLog2e;
    p.partition_size = part;
    p.max_partitions = max_parts;
    p.direct_single = 1;
    p.k_new = static_cast<const __half *>(k_new);
    p.v_new = static_cast<const __half *>(v_new);
    p.k_cache_w = static_cast<__half *>(const_cast<void *>(k_cache));
    p.v_cache_w = static_cast<__half *>(const_cast<void *>(v_cache));
    p.k_scale = k_scale;
    p.k_scale_w = const_cast<float *>(k_scale);
    p.v_scale = v_scale;
    p.v_scale_w = const_cast<float *>(v_scale);
    p.kv_fp8 = kv_fp8 ? 1 : 0;
    p.overlap = (flags & PKV_STEP_OVERLAP) ? 1 : 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (max_parts <= 1) return dispatch_partition(p, num_seqs, num_q_heads / num_kv_heads, s);
    // Equal partitions in several waves start together and end together, and the SMs idle at every
    // wave boundary until the next wave's first copies land; partitions of alternating length
    // (P - P/4, P + P/4) end at staggered times.  Taken when a request can span kStaggerMinParts
    // partitions and the grid fills kStaggerMinWaves waves of resident CTAs: with fewer, the longer
    // partitions only lengthen the critical path.
    const int stagger = part / 4 / kChunk * kChunk;
    if (max_parts >= kStaggerMinParts && stagger > 0 && part + stagger <= PKV_MAX_PARTITION) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PKV_ERR_CUDA;
        const int64_t slots = static_cast<int64_t>(sms) * (k_scale ? PKV_DECODE_KQ_MIN_CTAS : PKV_DECODE_MIN_CTAS);
        if (static_cast<int64_t>(num_seqs) * num_kv_heads * max_parts >= kStaggerMinWaves * slots) p.stagger = stagger;
    }

    const size_t need = pkv_decode_workspace_size(num_seqs, num_q_heads, head_dim, static_cast<int>(cap), part);
    if (!workspace || workspace_bytes < need || !pkv_internal::aligned(workspace, 256)) return PKV_ERR_WORKSPACE;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_parts;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    p.o_part = reinterpret_cast<float *>(ws);
    p.m_part = reinterpret_cast<float *>(ws + align256(rows * kD * sizeof(float)));
    p.l_part = reinterpret_cast<float *>(ws + align256(rows * kD * sizeof(float)) + align256(rows * sizeof(float)));
    p.counters = reinterpret_cast<int *>(ws + counters_offset(rows));
    return dispatch_partition(p, num_seqs, num_q_heads / num_kv_heads, s);
}

}  // namespace

extern "C" PKV_API int pkv_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *block_tables, const int32_t *context_lens,
                                            int num_seqs, int max_blocks_per_seq, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                            float scale, void *workspace, size_t workspace_bytes,
                                            pkv_stream_t stream) {
    return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, nullptr, nullptr,
                                 workspace, workspace_bytes, stream);
}

extern "C" PKV_API size_t pkv_decode_step_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                                         int max_context, int prefix_len) {
    if (prefix_len > 0)
        return pkv_shared_prefix_workspace_size(num_seqs, num_q_heads, head_dim, max_context, prefix_len);
    return pkv_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context, PKV_DEFAULT_PARTITION);
}

extern "C" PKV_API int pkv_decode_step(void *out, const void *q, const void *k_new, const void *v_new,
                                       void *k_cache, void *v_cache, const int32_t *block_tables,
                                       const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                       int64_t num_blocks, float scale, int prefix_len, void *workspace,
                                       size_t workspace_bytes, unsigned flags, pkv_stream_t stream) {
    if (!k_new || !v_new || (flags & ~PKV_STEP_OVERLAP)) return PKV_ERR_INVALID_ARG;
    if (prefix_len > 0)
        return pkv_internal::shared_prefix_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                                  max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                                                  num_blocks, scale, prefix_len, k_new, v_new, workspace,
                                                  workspace_bytes, stream, (flags & PKV_STEP_OVERLAP) != 0);
    if (prefix_len < 0) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream, nullptr, PKV_DEFAULT_PARTITION, nullptr, flags);
}

extern "C" PKV_API int pkv_decode_step_partition(void *out, const void *q, const void *k_new, const void *v_new,
                                                 void *k_cache, void *v_cache, const int32_t *block_tables,
                                                 const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                                 int64_t num_blocks, float scale, int partition_size,
                                                 void *workspace, size_t workspace_bytes, unsigned flags,
                                                 pkv_stream_t stream) {
    if (!k_new || !v_new || partition_size < 0) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream, nullptr,
                                 partition_size > 0 ? partition_size : PKV_DEFAULT_PARTITION, nullptr, flags);
}

// ------------------------------------------------------------------ int8 key cache

extern "C" PKV_API int pkv_decode_attention_int8k(void *out, const void *q, const void *k_codes, const float *k_scale,
                                                  const void *v_cache, const int32_t *block_tables,
                                                  const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                                  int64_t num_blocks, float scale, void *workspace,
                                                  size_t workspace_bytes, pkv_stream_t stream) {
    if (!k_scale) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_codes, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, nullptr, nullptr,
                                 workspace, workspace_bytes, stream, k_scale);
}

extern "C" PKV_API int pkv_decode_step_int8k(void *out, const void *q, const void *k_new, const void *v_new,
                                             void *k_codes, float *k_scale, void *v_cache,
                                             const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                                             int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim,
                                             int block_size, int64_t num_blocks, float scale, void *workspace,
                                             size_t workspace_bytes, unsigned flags, pkv_stream_t stream) {
    if (!k_new || !v_new || !k_scale) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_codes, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream, k_scale, PKV_DEFAULT_PARTITION, nullptr, flags);
}

// ------------------------------------------------------------------ several new tokens per request

namespace {
// 8-column tiles per CTA: two once a request brings more than 8 (token, head) rows per kv head.
int mq_tiles(int max_query_len, int group) { return max_query_len * group > 8 ? 2 : 1; }
int row_groups(int max_query_len, int group) {
    const int nc = 8 * mq_tiles(max_query_len, group);
    return (max_query_len * group + nc - 1) / nc;
}
}  // namespace

extern "C" PKV_API size_t pkv_decode_multi_workspace_size(int num_seqs, int total_q, int max_query_len,
                                                          int num_q_heads, int num_kv_heads, int head_dim,
                                                          int max_context) {
    if (num_seqs <= 0 || total_q <= 0 || max_query_len <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || max_context <= 0 || num_q_heads % num_kv_heads != 0)
        return 0;
    const size_t parts = (static_cast<size_t>(max_context) + PKV_DEFAULT_PARTITION - 1) / PKV_DEFAULT_PARTITION;
    if (parts <= 1) return 0;
    const size_t rows = static_cast<size_t>(total_q) * num_q_heads * parts;
    const size_t counters =
        static_cast<size_t>(num_seqs) * num_kv_heads * row_groups(max_query_len, num_q_heads / num_kv_heads);
    return align256(rows * head_dim * sizeof(float)) + 2 * align256(rows * sizeof(float)) +
           align256(counters * sizeof(int));
}

namespace {
// pkv_decode_attention_multi, optionally appending the new tokens first (k_new/v_new non-null:
// pkv_decode_step_multi, with its flags).
int decode_multi_impl(void *out, const void *q, const void *k_new, const void *v_new, const void *k_cache,
                      const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                      const int32_t *query_start, int num_seqs, int total_q, int max_query_len, int max_blocks_per_seq,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale,
                      void *workspace, size_t workspace_bytes, unsigned flags, pkv_stream_t stream) {
    if (flags & ~PKV_STEP_OVERLAP) return PKV_ERR_INVALID_ARG;
    int st = check_common(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks);
    if (st != PKV_OK) return st;
    if (!out || !pkv_internal::aligned(out, 8) || !query_start || !pkv_internal::aligned(query_start, 4))
        return PKV_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID_ARG;
    if (k_new && (!pkv_internal::aligned16(k_new) || !pkv_internal::aligned16(v_new))) return PKV_ERR_INVALID_ARG;
    if (total_q < 0 || max_query_len <= 0) return PKV_ERR_INVALID_ARG;
    if (max_query_len > (k_new ? PKV_MAX_STEP_QUERY_LEN : PKV_MAX_QUERY_LEN)) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || total_q == 0) return PKV_OK;
    const int group = num_q_heads / num_kv_heads;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    const int part = PKV_DEFAULT_PARTITION;
    const int max_parts = static_cast<int>((cap + part - 1) / part);
    DecodeParams p{};
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const unsigned char *>(k_cache);
    p.v_cache = static_cast<const unsigned char *>(v_cache);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<__half *>(out);
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.q_scale = scale * kLog2e;
    p.partition_size = part;
    p.max_partitions = max_parts;
    p.direct_single = 1;
    p.query_start = query_start;
    p.total_q = total_q;
    p.max_query_len = max_query_len;
    p.n_row_groups = row_groups(max_query_len, group);
    p.mq_tiles = mq_tiles(max_query_len, group);
    p.k_new = static_cast<const __half *>(k_new);
    p.v_new = static_cast<const __half *>(v_new);
    p.k_cache_w = static_cast<__half *>(const_cast<void *>(k_cache));
    p.v_cache_w = static_cast<__half *>(const_cast<void *>(v_cache));
    p.overlap = (k_new && (flags & PKV_STEP_OVERLAP)) ? 1 : 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (max_parts > 1) {
        const size_t need = pkv_decode_multi_workspace_size(num_seqs, total_q, max_query_len, num_q_heads,
                                                            num_kv_heads, head_dim, static_cast<int>(cap));
        if (!workspace || workspace_bytes < need || !pkv_internal::aligned(workspace, 256)) return PKV_ERR_WORKSPACE;
        const size_t rows = static_cast<size_t>(total_q) * num_q_heads * max_parts;
        unsigned char *ws = static_cast<unsigned char *>(workspace);
        p.o_part = reinterpret_cast<float *>(ws);
        p.m_part = reinterpret_cast<float *>(ws + align256(rows * kD * sizeof(float)));
        p.l_part = reinterpret_cast<float *>(ws + align256(rows * kD * sizeof(float)) + align256(rows * sizeof(float)));
        p.counters = reinterpret_cast<int *>(ws + counters_offset(rows));
    }
    return dispatch_partition(p, num_seqs, group, s);
}
}  // namespace

extern "C" PKV_API int pkv_decode_attention_multi(void *out, const void *q, const void *k_cache, const void *v_cache,
                                                  const int32_t *block_tables, const int32_t *context_lens,
                                                  const int32_t *query_start, int num_seqs, int total_q,
                                                  int max_query_len, int max_blocks_per_seq, int num_q_heads,
                                                  int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                                  float scale, void *workspace, size_t workspace_bytes,
                                                  pkv_stream_t stream) {
    return decode_multi_impl(out, q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens, query_start,
                             num_seqs, total_q, max_query_len, max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim,
                             block_size, num_blocks, scale, workspace, workspace_bytes, 0, stream);
}

extern "C" PKV_API int pkv_decode_step_multi(void *out, const void *q, const void *k_new, const void *v_new,
                                             void *k_cache, void *v_cache, const int32_t *block_tables,
                                             const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                                             int total_q, int max_query_len, int max_blocks_per_seq, int num_q_heads,
                                             int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                             float scale, void *workspace, size_t workspace_bytes, unsigned flags,
                                             pkv_stream_t stream) {
    if (!k_new || !v_new) return PKV_ERR_INVALID_ARG;
    return decode_multi_impl(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start, num_seqs,
                             total_q, max_query_len, max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim,
                             block_size, num_blocks, scale, workspace, workspace_bytes, flags, stream);
}

// ------------------------------------------------------------------ int8 keys and values

extern "C" PKV_API int pkv_decode_attention_int8kv(void *out, const void *q, const void *k_codes,
                                                   const float *k_scale, const void *v_codes, const float *v_scale,
                                                   const int32_t *block_tables, const int32_t *context_lens,
                                                   int num_seqs, int max_blocks_per_seq, int num_q_heads,
                                                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                                   float scale, void *workspace, size_t workspace_bytes,
                                                   pkv_stream_t stream) {
    if (!k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_codes, v_codes, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, nullptr, nullptr,
                                 workspace, workspace_bytes, stream, k_scale, PKV_DEFAULT_PARTITION, v_scale);
}

extern "C" PKV_API int pkv_decode_step_int8kv(void *out, const void *q, const void *k_new, const void *v_new,
                                              void *k_codes, float *k_scale, void *v_codes, float *v_scale,
                                              const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                                              int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                                              int head_dim, int block_size, int64_t num_blocks, float scale,
                                              void *workspace, size_t workspace_bytes, unsigned flags,
                                              pkv_stream_t stream) {
    if (!k_new || !v_new || !k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_codes, v_codes, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream, k_scale, PKV_DEFAULT_PARTITION, v_scale, flags);
}

// ------------------------------------------------------------------ fp8 (E4M3) keys and values

extern "C" PKV_API int pkv_decode_attention_fp8kv(void *out, const void *q, const void *k_codes,
                                                  const float *k_scale, const void *v_codes, const float *v_scale,
                                                  const int32_t *block_tables, const int32_t *context_lens,
                                                  int num_seqs, int max_blocks_per_seq, int num_q_heads,
                                                  int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                                  float scale, void *workspace, size_t workspace_bytes,
                                                  pkv_stream_t stream) {
    if (!k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_codes, v_codes, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, nullptr, nullptr,
                                 workspace, workspace_bytes, stream, k_scale, PKV_DEFAULT_PARTITION, v_scale, 0u, true);
}

extern "C" PKV_API int pkv_decode_step_fp8kv(void *out, const void *q, const void *k_new, const void *v_new,
                                             void *k_codes, float *k_scale, void *v_codes, float *v_scale,
                                             const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                                             int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                                             int head_dim, int block_size, int64_t num_blocks, float scale,
                                             void *workspace, size_t workspace_bytes, unsigned flags,
                                             pkv_stream_t stream) {
    if (!k_new || !v_new || !k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_codes, v_codes, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream, k_scale, PKV_DEFAULT_PARTITION, v_scale, flags,
                                 true);
}

// ------------------------------------------------------------------ allocation-free variant
//
// For callers that cannot allocate device memory (plugins hosted by a runtime that owns all
// device memory and hands them only input/output pointers; serving loops that forbid allocator
// calls, and the device synchronisation cudaMalloc implies, once they are running): the split
// partials go to this file-scope array instead of a caller workspace.  On the host the symbol
// names a stand-in, not device memory, so it is never passed to a kernel directly; its device
// address is looked up once per device with cudaGetSymbolAddress while that device is current
// and kept for the life of the process (a cudaDeviceReset of that device invalidates it).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_address[kMaxDevices] = {};
}  // namespace

extern "C" PKV_API int pkv_decode_attention_noalloc(void *out, const void *q, const void *k_cache,
                                                    const void *v_cache, const int32_t *block_tables,
                                                    const int32_t *context_lens, int num_seqs,
                                                    int max_blocks_per_seq, int num_q_heads, int num_kv_heads,
                                                    int head_dim, int block_size, int64_t num_blocks, float scale,
                                                    pkv_stream_t stream) {
    // Every argument is checked before any CUDA call, so a refused call enqueues nothing (in
    // particular no clear of the counters at an offset computed from bad sizes).
    int st = check_common(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks);
    if (st != PKV_OK) return st;
    if (!out || !pkv_internal::aligned(out, 8)) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;  // <= 2^31 - 1 (checked)
    const size_t need = pkv_decode_workspace_size(num_seqs, num_q_heads, head_dim, static_cast<int>(cap),
                                                  PKV_DEFAULT_PARTITION);
    if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (!g_noalloc_address[dev]) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) return PKV_ERR_CUDA;
            g_noalloc_address[dev] = addr;
        }
        scratch = g_noalloc_address[dev];
    }
    // The split's completion counters must start at zero; every call leaves them zero, but the
    // array is shared by all calls, so clear them here rather than trust an earlier call.
    const int max_parts = static_cast<int>((cap + PKV_DEFAULT_PARTITION - 1) / PKV_DEFAULT_PARTITION);
    if (max_parts > 1) {  // need (checked above) covers this counter region
        const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_parts;
        if (cudaMemsetAsync(static_cast<unsigned char *>(scratch) + counters_offset(rows), 0,
                            static_cast<size_t>(num_seqs) * num_q_heads * sizeof(int),
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    return pkv_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, scratch,
                                PKV_NOALLOC_SCRATCH_BYTES, stream);
}

namespace pkv_internal {

int encode_fp16_cache_map(void *map, const void *base, int64_t rows) {
    return encode_cache_map(static_cast<CUtensorMap *>(map), base, rows);
}

int encode_q_map(void *map, const void *q, int num_seqs, int num_q_heads, int group) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn || group <= 0 || 128 % group != 0) return PKV_ERR_CUDA;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_q_heads),
                                static_cast<cuuint64_t>(num_seqs)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes),
                                   static_cast<cuuint64_t>(num_q_heads) * kRowBytes};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(128 / group)};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = fn(static_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(q),
                          dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

int check_decode_args(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
                      const int32_t *context_lens, int num_seqs, int max_blocks_per_seq, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks) {
    return check_common(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq, num_q_heads,
                        num_kv_heads, head_dim, block_size, num_blocks);
}

int launch_split_pass(const SplitPass &a, void *stream) {
    DecodeParams p{};
    p.q = static_cast<const __half *>(a.q);
    p.k_cache = static_cast<const unsigned char *>(a.k_cache);
    p.v_cache = static_cast<const unsigned char *>(a.v_cache);
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.out = static_cast<__half *>(a.out);
    p.o_part = a.o_part;
    p.m_part = a.m_part;
    p.l_part = a.l_part;
    p.max_blocks_per_seq = a.max_blocks_per_seq;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.block_size = a.block_size;
    p.num_blocks = a.num_blocks;
    p.q_scale = a.scale * kLog2e;
    p.partition_size = a.partition_size;
    p.max_partitions = a.max_partitions;
    p.direct_single = 0;
    p.counters = a.counters;
    p.token_offset = a.token_offset;
    p.slot_offset = a.slot_offset;
    p.k_new = static_cast<const __half *>(a.k_new);
    p.v_new = static_cast<const __half *>(a.v_new);
    p.k_cache_w = static_cast<__half *>(const_cast<void *>(a.k_cache));
    p.v_cache_w = static_cast<__half *>(const_cast<void *>(a.v_cache));
    p.prefix_ctas = a.prefix_ctas;
    p.prefix_chunks = a.prefix_chunks;
    p.overlap = a.overlap ? 1 : 0;
    if (a.separate_merge && a.prefix_ctas == 0) p.counters = nullptr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int group = a.num_q_heads / a.num_kv_heads;
    const int st = dispatch_partition(p, a.num_seqs, group, s, a.grid_partitions);
    if (st != PKV_OK || (!a.separate_merge && a.prefix_ctas == 0)) return st;
    // the merge as a programmatic dependent of the pass: launched as the pass's CTAs drain
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.num_kv_heads, a.num_seqs);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaErrorInvalidValue;
    switch (group) {
        case 1: e = cudaLaunchKernelEx(&cfg, merge_groups_kernel<1>, p); break;
        case 2: e = cudaLaunchKernelEx(&cfg, merge_groups_kernel<2>, p); break;
        case 4: e = cudaLaunchKernelEx(&cfg, merge_groups_kernel<4>, p); break;
        case 8: e = cudaLaunchKernelEx(&cfg, merge_groups_kernel<8>, p); break;
        default: return PKV_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int decode_take_error(int *code) {
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_decode_error, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    }
    *code = value;
    return PKV_OK;
}

}  // namespace pkv_internal
