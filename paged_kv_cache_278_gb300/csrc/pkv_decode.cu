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
//     ((token, head) rows as the columns, causal masks per column).  A CUDA-core engine (packed
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

constexpr int kD = PKV_HEAD_DIM;        // 128
constexpr int kChunk = 16;              // tokens per shared-memory tile
constexpr int kRowBytes = kD * 2;       // one fp16 K or V row
// Warps per CTA and bulk-copy stages per warp (each stage holds one 16-token chunk of K and V).
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4
#endif
#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 2
#endif
#ifndef PKV_DECODE_MIN_CTAS
#define PKV_DECODE_MIN_CTAS 3
#endif
// Resident CTAs per SM the int8-key kernel is compiled for: its stages are 6 KB, not 8 KB, so four
// CTAs (53 KB of shared memory, 128 registers per thread) fit an SM and keep as many bytes in flight
// as three fp16 CTAs.
#ifndef PKV_DECODE_KQ_MIN_CTAS
#define PKV_DECODE_KQ_MIN_CTAS 4
#endif
// 1: K and V of a stage land on separate mbarriers, so a chunk's q.K starts as soon as its K has
// arrived and the next K copy into the stage is issued before the chunk's P.V runs.  Measured 1-2.5%
// slower on every workload (twice the barrier traffic for no gain in bytes in flight): off.
#ifndef PKV_DECODE_SPLIT_KV
#define PKV_DECODE_SPLIT_KV 0
#endif
// 1: q.K and P.V use packed two-lane FMAs (fma.rn.f32x2), halving FMA issue slots.
#ifndef PKV_DECODE_FFMA2
#define PKV_DECODE_FFMA2 1
#endif
// 1: with at least PKV_DECODE_TC_MIN_GROUP query heads per kv head, q.K and P.V run on the tensor
// cores (mma.m16n8k16); smaller groups use the CUDA-core engine.  Every group size takes the
// tensor cores by default: for MHA (one live column of eight) it measured 0.6% faster than the
// CUDA-core engine, which issues more instructions per chunk.
#ifndef PKV_DECODE_TC
#define PKV_DECODE_TC 1
#endif
#ifndef PKV_DECODE_TC_MIN_GROUP
#define PKV_DECODE_TC_MIN_GROUP 1
#endif
// Independent accumulator chains of a chunk's q.K MMAs on the fp16 tensor-core engines (the
// k-steps are dealt round-robin and the chains added at the end; 1 = one dependent chain of 8
// MMAs).  2 measured 0.2-1 % faster on every fp16 workload (most on the 16-column multi-token
// engine), 4 no better than 2.
#ifndef PKV_QK_CHAINS
#define PKV_QK_CHAINS 2
#endif
constexpr int kWarps = PKV_DECODE_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = PKV_DECODE_STAGES;
constexpr bool kSplitKV = PKV_DECODE_SPLIT_KV != 0;
constexpr int kBarsPerStage = kSplitKV ? 2 : 1;
constexpr float kRescaleThreshold = 8.0f;          // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

struct DecodeParams {
    const __half *q;
    const unsigned char *k_cache;
    const unsigned char *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    __half *out;
    float *o_part;
    float *m_part;
    float *l_part;
    int max_blocks_per_seq;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    int64_t num_blocks;
    float q_scale;            // scale * log2(e)
    int partition_size;
    int max_partitions;
    int direct_single;        // write fp16 out directly for single-partition requests
    int *counters;            // per (request, kv head) completion counters: fused merge when non-null
    int token_offset;         // first logical token covered by partition 0 (shared-prefix length, else 0)
    int slot_offset;          // partial slots [0, slot_offset) already hold the shared prefix's partials
    const __half *k_new;      // non-null: append k_new/v_new [B][Hkv][D] at position ctx_b - 1 first
    const __half *v_new;
    __half *k_cache_w;        // writable views of the caches for that append
    __half *v_cache_w;
    const int32_t *query_start;  // several new tokens per request: request b owns q/out rows
    int total_q;                 //   query_start[b] .. query_start[b+1]-1 (null: one token per request)
    int max_query_len;
    int n_row_groups;            // groups of 8 x mq_tiles (token, head) rows of one kv head
    int mq_tiles;                // 8-column MMA tiles per CTA for several tokens per request (1 or 2)
    const float *k_scale;     // int8 key cache: float32 scale per (block, kv head, slot); null for fp16 keys
    float *k_scale_w;         // writable view of k_scale for the fused append
    const float *v_scale;     // int8 values too: float32 scale per (block, kv head, slot); null for fp16 values
    float *v_scale_w;
    CUtensorMap tmap_k;       // tensor-core engine: the caches as 2-D [NB*Hkv*bs rows][128] fp16,
    CUtensorMap tmap_v;       //   16 x 64 boxes, 128-byte swizzle (int8 keys: 16 x 128-byte boxes)
};

constexpr int kMergeTile = 512;  // partitions whose weights the fused merge stages at a time

// Shared-memory carve-up (bytes), identical on host and device.  TC selects the tensor-core
// engine's fp16 P buffer; its K/V tiles are two 2 KB halves (dims 0-63, 64-127) of 16 rows x
// 128 B in the tensor copies' 128-byte swizzle (16-byte chunk c of row r stored at c ^ (r % 8)).
// KQ (int8 keys): the K tile is one 2 KB box of 16 int8 rows in the same swizzle, and each stage
// also holds the chunk's 16 float32 key scales.
constexpr int kHalfTile = kChunk * 128;
// KQ: 0 fp16 K/V, 1 int8 keys, 2 int8 keys and values.
template <bool TC, int KQ = 0, int NT = 1>
struct SmemLayout {
    static constexpr int row = kRowBytes;
    static constexpr int tile = kChunk * row;
    static constexpr int k_tile = KQ ? kChunk * kD : tile;
    static constexpr int v_tile = KQ == 2 ? kChunk * kD : tile;
    static constexpr int stage = k_tile + v_tile;
    static constexpr int scale_stride = KQ == 2 ? 2 * kChunk * 4 : kChunk * 4;  // K scales (| V scales) per stage
    static constexpr int stages = 0;
    static constexpr int stage_bytes = kWarps * kStages * stage;
    static constexpr int scales = stages + stage_bytes;
    static constexpr int bars = scales + (KQ ? kWarps * kStages * scale_stride : 0);
    static constexpr int probs = bars + kWarps * kStages * kBarsPerStage * 8;
    __host__ __device__ static constexpr int probs_per_warp(int g) { return TC ? NT * 2 * 8 * kChunk * 2 : kChunk * g * 4; }
    __host__ __device__ static constexpr int newrow(int g) { return probs + kWarps * probs_per_warp(g); }
    __host__ __device__ static constexpr int table(int g) { return newrow(g) + 2 * kRowBytes; }
    __host__ __device__ static constexpr int total(int g, int partition_size) {
        return table(g) + (partition_size / kChunk + 1) * 4;
    }
};

// Output rows of a CTA's G packed columns.  One token per request: the G query heads of (request,
// kv head), consecutive rows from row0.
struct HeadRows {
    int64_t row0;
    __device__ __forceinline__ int64_t row(int hh) const { return row0 + hh; }
    __device__ __forceinline__ bool live(int) const { return true; }
};
// Several tokens per request: column hh of row group rg is row r = NC rg + hh of the request's
// n * G rows for kv head kvh, i.e. token r / G, head r % G.  Columns past the last token are
// dead; their reads are redirected to the last token's row so every access stays in bounds.
template <int G, int NC = 8>
struct TokenRows {
    int64_t qs;
    int n, rg, hq, kvh;
    __device__ __forceinline__ int64_t row(int hh) const {
        const int r = rg * NC + hh;
        const int i = r / G < n ? r / G : n - 1;
        return (qs + i) * hq + kvh * G + r % G;
    }
    __device__ __forceinline__ bool live(int hh) const { return (rg * NC + hh) / G < n; }
};

// Log-sum-exp merge of partial slots [0, n_total) of the G packed columns (query heads, or
// (token, head) rows) of one CTA's kv head into fp16 out; called by every thread of one CTA
// (it synchronises the CTA).
// STAGE_BYTES: the caller's shared memory available for the staging (its stage buffers).
template <int G, int STAGE_BYTES, class Rows>
__device__ void merge_group(const DecodeParams &P, const Rows &rows, int n_total, unsigned char *smem) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Slots: (packed head, 4 consecutive dims) -> float4 loads of o; partitions are split over
    // GROUPS thread groups when there are fewer slots than threads, and loads are unrolled so a
    // thread keeps 8 rows in flight.  All weights w = l exp(m - M) of a tile are staged first.
    constexpr int SLOTS = G * (kD / 4);
    constexpr int GROUPS = SLOTS >= kThreads ? 1 : kThreads / SLOTS;
    constexpr int PER_THREAD = SLOTS >= kThreads ? SLOTS / kThreads : 1;
    static_assert(SLOTS % kThreads == 0 || kThreads % SLOTS == 0, "slot split");
    // partitions staged at a time: the largest of 512, 256, 128 whose staging fits
    constexpr int kFixed = G * 4 + 16 + GROUPS * SLOTS * 20;
    constexpr int TILE = 2 * G * kMergeTile * 4 + kFixed <= STAGE_BYTES         ? kMergeTile
                         : 2 * G * (kMergeTile / 2) * 4 + kFixed <= STAGE_BYTES ? kMergeTile / 2
                                                                                 : kMergeTile / 4;
    static_assert(2 * G * TILE * 4 + kFixed <= STAGE_BYTES, "merge staging must fit the stages");
    float *s_wt = reinterpret_cast<float *>(smem);                  // [2][G][TILE]
    float *s_max = s_wt + 2 * G * TILE;                        // [G]
    float4 *s_acc = reinterpret_cast<float4 *>(s_max + G + 4 - (G % 4 == 0 ? 4 : G % 4));  // [GROUPS][SLOTS]
    float *s_sum = reinterpret_cast<float *>(s_acc + GROUPS * SLOTS);                     // [GROUPS][SLOTS]
    const int grp = GROUPS > 1 ? threadIdx.x / SLOTS : 0;
    const int slot0 = GROUPS > 1 ? threadIdx.x % SLOTS : threadIdx.x;
    float4 macc[PER_THREAD];
    float msum[PER_THREAD];
#pragma unroll
    for (int k = 0; k < PER_THREAD; ++k) {
        macc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        msum[k] = 0.f;
    }
    auto o_row = [&](int hh, int d4) {
        return reinterpret_cast<const float4 *>(P.o_part + rows.row(hh) * P.max_partitions * kD) + d4;
    };
    auto accumulate = [&](int k, float w, float4 v) {
        macc[k].x = fmaf(w, v.x, macc[k].x);
        macc[k].y = fmaf(w, v.y, macc[k].y);
        macc[k].z = fmaf(w, v.z, macc[k].z);
        macc[k].w = fmaf(w, v.w, macc[k].w);
        msum[k] += w;
    };
    if (n_total <= TILE) {
        // Fast path, about one L2 round trip: issue this thread's first PRE partial rows, stage
        // every (m, l) of the group in shared memory meanwhile, then weight the rows in registers.
        constexpr int PRE = 8;
        float4 pre[PER_THREAD][PRE];
#pragma unroll
        for (int k = 0; k < PER_THREAD; ++k) {
            const int slot = slot0 + k * kThreads;
            const float4 *o = o_row(slot / (kD / 4), slot % (kD / 4));
#pragma unroll
            for (int jj = 0; jj < PRE; ++jj) {
                const int pp = grp + jj * GROUPS;
                pre[k][jj] = pp < n_total ? __ldcg(o + static_cast<int64_t>(pp) * (kD / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float *s_mm = s_wt;
        float *s_ll = s_wt + G * TILE;
        for (int i = threadIdx.x; i < G * n_total; i += kThreads) {
            const int hh = i / n_total, pp = i - hh * n_total;
            const int64_t prow = rows.row(hh) * P.max_partitions + pp;
            s_mm[hh * TILE + pp] = __ldcg(P.m_part + prow);
            s_ll[hh * TILE + pp] = __ldcg(P.l_part + prow);
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < PER_THREAD; ++k) {
            const int slot = slot0 + k * kThreads;
            const int hh = slot / (kD / 4);
            const float *mm = s_mm + hh * TILE;
            const float *ll = s_ll + hh * TILE;
            float M = -INFINITY;
            for (int pp = 0; pp < n_total; ++pp) M = fmaxf(M, mm[pp]);
#pragma unroll
            for (int jj = 0; jj < PRE; ++jj) {
                const int pp = grp + jj * GROUPS;
                if (pp < n_total) accumulate(k, ll[pp] * expf(mm[pp] - M), pre[k][jj]);
            }
            const float4 *o = o_row(hh, slot % (kD / 4));
            // the remaining rows in batches of 8 independent loads (one L2 round trip per batch: +1.6 %
            // on the 32k-token step with its 64-way merges, +3.4 % with 128-way)
            int pp = grp + PRE * GROUPS;
            for (; pp + 7 * GROUPS < n_total; pp += 8 * GROUPS) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = __ldcg(o + static_cast<int64_t>(pp + u * GROUPS) * (kD / 4));
#pragma unroll
                for (int u = 0; u < 8; ++u) accumulate(k, ll[pp + u * GROUPS] * expf(mm[pp + u * GROUPS] - M), v[u]);
            }
            for (; pp < n_total; pp += GROUPS)
                accumulate(k, ll[pp] * expf(mm[pp] - M), __ldcg(o + static_cast<int64_t>(pp) * (kD / 4)));
        }
    } else {
        // Long contexts: maxima first, then tiles of weights, each tile's rows streamed.
        for (int hh = warp; hh < G; hh += kWarps) {
            const float *m = P.m_part + rows.row(hh) * P.max_partitions;
            float M = -INFINITY;
#pragma unroll 4
            for (int pp = lane; pp < n_total; pp += 32) M = fmaxf(M, __ldcg(m + pp));
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(pkv::kFullMask, M, sh));
            if (lane == 0) s_max[hh] = M;
        }
        for (int p0 = 0; p0 < n_total; p0 += TILE) {
            const int n = min(TILE, n_total - p0);
            __syncthreads();  // s_max ready / previous tile consumed
            for (int i = threadIdx.x; i < G * n; i += kThreads) {
                const int hh = i / n, pp = i - hh * n;
                const int64_t prow = rows.row(hh) * P.max_partitions + p0 + pp;
                s_wt[hh * TILE + pp] = __ldcg(P.l_part + prow) * expf(__ldcg(P.m_part + prow) - s_max[hh]);
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < PER_THREAD; ++k) {
                const int slot = slot0 + k * kThreads;
                const int hh = slot / (kD / 4);
                const float4 *o = o_row(hh, slot % (kD / 4)) + static_cast<int64_t>(p0) * (kD / 4);
                const float *w = s_wt + hh * TILE;
#pragma unroll 8
                for (int pp = grp; pp < n; pp += GROUPS) accumulate(k, w[pp], __ldcg(o + static_cast<int64_t>(pp) * (kD / 4)));
            }
        }
    }
    if (GROUPS > 1) {
        s_acc[grp * SLOTS + slot0] = macc[0];
        s_sum[grp * SLOTS + slot0] = msum[0];
        __syncthreads();
        if (grp != 0) return;
        for (int g2 = 1; g2 < GROUPS; ++g2) {
            const float4 v = s_acc[g2 * SLOTS + slot0];
            macc[0].x += v.x;
            macc[0].y += v.y;
            macc[0].z += v.z;
            macc[0].w += v.w;
            msum[0] += s_sum[g2 * SLOTS + slot0];
        }
    }
#pragma unroll
    for (int k = 0; k < PER_THREAD; ++k) {
        const int slot = slot0 + k * kThreads;
        const int hh = slot / (kD / 4), d4 = slot % (kD / 4);
        if (!rows.live(hh)) continue;
        const float inv = 1.f / msum[k];
        __half2 lo = __floats2half2_rn(macc[k].x * inv, macc[k].y * inv);
        __half2 hi = __floats2half2_rn(macc[k].z * inv, macc[k].w * inv);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t *>(&lo);
        packed.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(P.out + rows.row(hh) * kD + d4 * 4) = packed;
    }
}

// ---------------------------------------------------------------- CUDA-core engine
// LPT lanes share a token row for q . K (each holding 128/LPT dims of q in fp32, pre-scaled by
// scale*log2 e); partial dots are finished with a shuffle reduce-scatter after which each lane
// holds scores of one packed head for a few tokens; P goes through a per-warp shared buffer to
// P . V, where each lane owns 4 output dims of every packed head.  Used for G <= 2, where the
// packed-head tile would leave most of a tensor-core MMA empty.
template <int G, int LPT>
struct FmaEngine {
    static constexpr int TG = 32 / LPT;            // token groups per warp (q.K stage)
    static constexpr int TPL = kChunk / TG;        // tokens per lane per chunk (q.K stage)
    static constexpr int NP = kD / LPT / 8;        // 16-byte pieces of a row per lane
    static constexpr int N = TPL * G;              // partial dot products per lane
    static constexpr int LOG_LPT = ilog2(LPT);
    static constexpr int LOG_N = ilog2(N);
    static constexpr int HALVING = LOG_LPT < LOG_N ? LOG_LPT : LOG_N;
    static constexpr int HELD = N >> HALVING;      // finished scores per lane
    static constexpr int DUP_BITS = LOG_LPT - HALVING;
    static constexpr int kRow = kRowBytes;         // shared-memory row stride
    static_assert((1 << LOG_LPT) == LPT && (1 << LOG_N) == N, "powers of two");
    static_assert(NP >= 1 && NP * 8 * LPT == kD, "lane split of a row");
    // A lane's finished scores are (packed head my_head, chunk token held_tok(k)); HELD divides TPL
    // and base is a multiple of HELD, so all of a lane's scores share one head.
    static_assert(TPL % HELD == 0, "a lane's finished scores must share one head");

    float qf[G][NP * 8];
    float m_head[G], l_lane[G], acc[G][4];  // reference max (warp-uniform), lane share of l, P.V sums
    float m_mine, top_mine;                 // m_head[my_head]; true running max of this lane's scores
    int c, r, base, my_head;
    bool owner;

    __device__ __forceinline__ int held_tok(int k) const { return r + TG * ((base + k) % TPL); }

    __device__ __forceinline__ void init(const DecodeParams &P, int b, int kvh, int lane) {
        c = lane & (LPT - 1);
        r = lane / LPT;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const uint4 *qrow =
                reinterpret_cast<const uint4 *>(P.q + (static_cast<int64_t>(b) * P.num_q_heads + kvh * G + hh) * kD);
#pragma unroll
            for (int np = 0; np < NP; ++np) {
                const uint4 raw = __ldg(qrow + c + LPT * np);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = pkv::half2_bits_to_float2(w[e]);
                    qf[hh][np * 8 + 2 * e] = f.x * P.q_scale;
                    qf[hh][np * 8 + 2 * e + 1] = f.y * P.q_scale;
                }
            }
        }
        base = 0;
#pragma unroll
        for (int s = 0; s < HALVING; ++s)
            if (lane & (LPT >> (s + 1))) base += N >> (s + 1);
        owner = (c & ((1 << DUP_BITS) - 1)) == 0;
        my_head = base / TPL;
        m_mine = -INFINITY;
        top_mine = -INFINITY;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            m_head[hh] = -INFINITY;
            l_lane[hh] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[hh][e] = 0.f;
        }
    }

    // q . K, online softmax and the chunk's probabilities into the warp's scratch (ends synchronised).
    __device__ __forceinline__ void qk(uint32_t k_tile, uint32_t, int valid, int lane, unsigned char *scratch, int) {
        float *s_prob = reinterpret_cast<float *>(scratch);
        // ---- q . K partial sums: v[h * TPL + i] over this lane's dims
        float v[N];
#pragma unroll
        for (int it = 0; it < TPL; ++it) {
            const int t = r + TG * it;
            float kf[NP * 8];
#pragma unroll
            for (int np = 0; np < NP; ++np) {
                const uint4 raw = pkv::lds128(k_tile + t * kRow + (c + LPT * np) * 16);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = pkv::half2_bits_to_float2(w[e]);
                    kf[np * 8 + 2 * e] = f.x;
                    kf[np * 8 + 2 * e + 1] = f.y;
                }
            }
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
#if PKV_DECODE_FFMA2
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int e = 0; e < NP * 8; e += 2) pkv::fma2(s0, s1, qf[hh][e], qf[hh][e + 1], kf[e], kf[e + 1]);
                v[hh * TPL + it] = s0 + s1;
#else
                float sacc = 0.f;
#pragma unroll
                for (int e = 0; e < NP * 8; ++e) sacc = fmaf(qf[hh][e], kf[e], sacc);
                v[hh * TPL + it] = sacc;
#endif
            }
        }
        // ---- reduce-scatter across the LPT lanes of a token group
#pragma unroll
        for (int s = 0; s < HALVING; ++s) {
            const int mask = LPT >> (s + 1);
            const int half = N >> (s + 1);
            const bool upper = (lane & mask) != 0;
#pragma unroll
            for (int k = 0; k < half; ++k) {
                const float send = upper ? v[k] : v[k + half];
                const float keep = upper ? v[k + half] : v[k];
                v[k] = keep + __shfl_xor_sync(pkv::kFullMask, send, mask);
            }
        }
#pragma unroll
        for (int s = HALVING; s < LOG_LPT; ++s) v[0] += __shfl_xor_sync(pkv::kFullMask, v[0], LPT >> (s + 1));

        // ---- online softmax (log2 domain) with lazy rescale
        bool need = false;
#pragma unroll
        for (int k = 0; k < HELD; ++k) {
            if (held_tok(k) >= valid) v[k] = -INFINITY;
            need |= v[k] > m_mine + kRescaleThreshold;
            top_mine = fmaxf(top_mine, v[k]);
        }
        if (__any_sync(pkv::kFullMask, need)) {
            float mx[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) mx[hh] = -INFINITY;
#pragma unroll
            for (int k = 0; k < HELD; ++k)
#pragma unroll
                for (int hh = 0; hh < G; ++hh) mx[hh] = fmaxf(mx[hh], my_head == hh ? v[k] : -INFINITY);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
#pragma unroll
                for (int sh = 0; sh < 5; ++sh) mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(pkv::kFullMask, mx[hh], 16 >> sh));
            }
            m_mine = 0.f;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float mn = fmaxf(m_head[hh], mx[hh]);
                const float alpha = exp2f(m_head[hh] - mn);
                m_head[hh] = mn;
                l_lane[hh] *= alpha;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[hh][e] *= alpha;
                m_mine += (my_head == hh) ? mn : 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < HELD; ++k) {
            const float p = exp2f(v[k] - m_mine);  // 0 for masked tokens
            if (owner) {
#pragma unroll
                for (int hh = 0; hh < G; ++hh) l_lane[hh] += (my_head == hh) ? p : 0.f;
                if (held_tok(k) < valid) s_prob[held_tok(k) * G + my_head] = p;
            }
        }
        __syncwarp();
    }

    // P . V of the chunk whose probabilities qk() left in scratch.
    __device__ __forceinline__ void pv(uint32_t v_tile, int valid, int lane, unsigned char *scratch) {
        const float *s_prob = reinterpret_cast<const float *>(scratch);
        // ---- P . V: this lane owns dims [4*lane, 4*lane+4) of every packed head
#pragma unroll
        for (int t = 0; t < kChunk; ++t) {
            if (t < valid) {
                const uint2 raw = pkv::lds64(v_tile + t * kRow + lane * 8);
                const float2 v01 = pkv::half2_bits_to_float2(raw.x);
                const float2 v23 = pkv::half2_bits_to_float2(raw.y);
                float pr[G];
#pragma unroll
                for (int hh = 0; hh < G; ++hh) pr[hh] = s_prob[t * G + hh];
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
#if PKV_DECODE_FFMA2
                    pkv::fma2(acc[hh][0], acc[hh][1], pr[hh], pr[hh], v01.x, v01.y);
                    pkv::fma2(acc[hh][2], acc[hh][3], pr[hh], pr[hh], v23.x, v23.y);
#else
                    acc[hh][0] = fmaf(pr[hh], v01.x, acc[hh][0]);
                    acc[hh][1] = fmaf(pr[hh], v01.y, acc[hh][1]);
                    acc[hh][2] = fmaf(pr[hh], v23.x, acc[hh][2]);
                    acc[hh][3] = fmaf(pr[hh], v23.y, acc[hh][3]);
#endif
                }
            }
        }
    }

    // Per-warp (m, l, acc) of every packed head, re-referenced to the true max, into shared memory.
    __device__ __forceinline__ void finish(int warp, int lane, float *c_acc, float *c_m, float *c_l) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float l = l_lane[hh];
            float top = my_head == hh ? top_mine : -INFINITY;
#pragma unroll
            for (int sh = 0; sh < 5; ++sh) {
                l += __shfl_xor_sync(pkv::kFullMask, l, 16 >> sh);
                top = fmaxf(top, __shfl_xor_sync(pkv::kFullMask, top, 16 >> sh));
            }
            float m = m_head[hh];
            if (top > -INFINITY) {  // this warp saw tokens: m_head <= top < m_head + 2^8
                const float f = exp2f(m - top);
                l *= f;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[hh][e] *= f;
                m = top;
            }
            *reinterpret_cast<float4 *>(c_acc + (warp * G + hh) * kD + lane * 4) =
                make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
            if (lane == 0) {
                c_m[warp * G + hh] = m;
                c_l[warp * G + hh] = l;
            }
        }
    }
};

// ---------------------------------------------------------------- tensor-core engine
// With G >= 4 query heads per kv head both products are real MMA tiles (N = 8 head columns,
// G of them live): per 16-token chunk
//   S^T[16 tok x 8] = K_tile[16 x 128] . Q^T[128 x 8]        8 x mma.m16n8k16 (K from shared
//                                                           memory by ldmatrix, Q^T as fp16
//                                                           fragments held in registers)
//   O^T[128 x 8]  += V_tile^T[128 x 16] . P^T[16 x 8]        8 m-tiles x 2 (P = hi + lo fp16)
// with fp32 accumulation throughout.  K/V tiles arrive by 2-D tensor copies in the 128-byte
// swizzle, which keeps every ldmatrix bank-conflict free.  Each lane owns heads 2*(lane%4) and +1
// of the fragments; lanes whose heads are >= G carry padding columns.
template <int G>
struct TcEngine {
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "up to 8 heads in the 8 MMA columns");

    // Byte offset of 16-byte chunk `c16` (0..15 across the 128 dims) of row r in a swizzled tile.
    __device__ __forceinline__ static uint32_t swz(int r, int c16) {
        return (c16 >> 3) * kHalfTile + r * 128 + (((c16 & 7) ^ (r & 7)) << 4);
    }

    uint32_t qb[kD / 16][2];  // Q^T B-fragments of the 8 k-steps (fp16x2)
    float o[kD / 16][4];      // O^T accumulators: (dim 16 mt + lane/4 (+8), head h0 (+1))
    float m_ref[2], top[2], l_part[2];
    float q_scale;

    __device__ __forceinline__ void reset(const DecodeParams &P) {
#pragma unroll
        for (int mt = 0; mt < kD / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m_ref[0] = m_ref[1] = top[0] = top[1] = -INFINITY;
        l_part[0] = l_part[1] = 0.f;
        q_scale = P.q_scale;
    }

    __device__ __forceinline__ void init(const DecodeParams &P, int b, int kvh, int lane) {
        const int head = lane >> 2;
        const __half *qrow =
            P.q + (static_cast<int64_t>(b) * P.num_q_heads + kvh * G + (head < G ? head : 0)) * kD;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                qb[ks][j] = head < G ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + (lane & 3) * 2 + j * 8))
                                     : 0u;
        reset(P);
    }

    // Raw q . K of the chunk's 16 tokens (rows g, g + 8) for the lane's columns h0, h0 + 1
    // (PKV_QK_CHAINS independent accumulator chains over the k-steps, added at the end).
    __device__ __forceinline__ void dots(float (&s)[4], uint32_t k_tile, int lane) const {
        float chain[PKV_QK_CHAINS > 1 ? PKV_QK_CHAINS - 1 : 1][4] = {};
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t a[4];
            pkv::ldsm_x4(a, k_tile + swz(lane & 15, ks * 2 + (lane >> 4)));
            float(&acc)[4] = ks % PKV_QK_CHAINS == 0 ? s : chain[ks % PKV_QK_CHAINS - 1];
            pkv::mma16816(acc, a, qb[ks][0], qb[ks][1]);
        }
#pragma unroll
        for (int c = 0; c < PKV_QK_CHAINS - 1; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[e] += chain[c][e];
    }

    __device__ __forceinline__ void qk(uint32_t k_tile, uint32_t, int valid, int lane, unsigned char *scratch, int) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        dots(s, k_tile, lane);
        const int g = lane >> 2;
        s[0] = g < valid ? s[0] * q_scale : -INFINITY;
        s[1] = g < valid ? s[1] * q_scale : -INFINITY;
        s[2] = g + 8 < valid ? s[2] * q_scale : -INFINITY;
        s[3] = g + 8 < valid ? s[3] * q_scale : -INFINITY;
        softmax(s, lane, scratch);
    }

    // Online softmax of the chunk's scaled, masked log2-domain scores s (token g / g + 8, heads
    // h0 / h0 + 1); the weights go to the warp's scratch as fp16 hi / lo parts for pv() (ends
    // synchronised).  kAnyMasked: a column may have no visible token yet (its reference max still
    // -inf), so a masked score's weight is forced to 0 instead of exp2(-inf - -inf).
    // kVScale: the weights stored for P.V are multiplied by the chunk's value row scales (float32 at
    // vs_tile, one per token); l keeps the unscaled weights.  The reference max then follows the
    // running max exactly (no lazy margin), so a weight is at most 1 and weight x scale at most
    // 65504 / 127: it cannot overflow fp16.
    template <bool kAnyMasked = false, bool kVScale = false>
    __device__ __forceinline__ void softmax(float (&s)[4], int lane, unsigned char *scratch, uint32_t vs_tile = 0) {
        const int g = lane >> 2;
        float cm0 = fmaxf(s[0], s[2]), cm1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int sh = 4; sh <= 16; sh <<= 1) {
            cm0 = fmaxf(cm0, __shfl_xor_sync(pkv::kFullMask, cm0, sh));
            cm1 = fmaxf(cm1, __shfl_xor_sync(pkv::kFullMask, cm1, sh));
        }
        top[0] = fmaxf(top[0], cm0);
        top[1] = fmaxf(top[1], cm1);
        constexpr float kMargin = kVScale ? 0.f : kRescaleThreshold;
        if (__any_sync(pkv::kFullMask, cm0 > m_ref[0] + kMargin || cm1 > m_ref[1] + kMargin)) {
            const float n0 = fmaxf(m_ref[0], cm0), n1 = fmaxf(m_ref[1], cm1);
            float a0 = exp2f(m_ref[0] - n0), a1 = exp2f(m_ref[1] - n1);
            if (kAnyMasked) {  // a column still without a visible token: nothing to rescale (-inf - -inf)
                a0 = n0 == -INFINITY ? 1.f : a0;
                a1 = n1 == -INFINITY ? 1.f : a1;
            }
            m_ref[0] = n0;
            m_ref[1] = n1;
            l_part[0] *= a0;
            l_part[1] *= a1;
#pragma unroll
            for (int mt = 0; mt < kD / 16; ++mt) {
                o[mt][0] *= a0;
                o[mt][1] *= a1;
                o[mt][2] *= a0;
                o[mt][3] *= a1;
            }
        }
        float p[4] = {exp2f(s[0] - m_ref[0]), exp2f(s[1] - m_ref[1]), exp2f(s[2] - m_ref[0]),
                      exp2f(s[3] - m_ref[1])};
        if (kAnyMasked) {
#pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = s[e] == -INFINITY ? 0.f : p[e];
        }
        l_part[0] += p[0] + p[2];
        l_part[1] += p[1] + p[3];
        if (kVScale) {
            const float vg = pkv::lds32f(vs_tile + 4 * g), v8 = pkv::lds32f(vs_tile + 4 * (g + 8));
#pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = p[e] == 0.f ? 0.f : p[e] * (e < 2 ? vg : v8);  // masked rows: 0
        }
        // P^T through shared memory as fp16 hi / lo: [2][8 heads][16 tokens]
        __half *ph = reinterpret_cast<__half *>(scratch);
        __half *pl = ph + 8 * kChunk;
        const int h0 = (lane & 3) * 2;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = (h0 + (e & 1)) * kChunk + g + (e >> 1) * 8;
            const __half hi = __float2half_rn(p[e]);
            ph[idx] = hi;
            pl[idx] = __float2half_rn(p[e] - __half2float(hi));
        }
        __syncwarp();
    }

    // O^T += V_tile^T . P^T with the weights softmax() left in scratch.
    __device__ __forceinline__ void pv(uint32_t v_tile, int, int lane, unsigned char *scratch) {
        const __half *ph = reinterpret_cast<const __half *>(scratch);
        const __half *pl = ph + 8 * kChunk;
        const int n = lane >> 2, k0 = (lane & 3) * 2;
        const uint32_t bh0 = *reinterpret_cast<const uint32_t *>(ph + n * kChunk + k0);
        const uint32_t bh1 = *reinterpret_cast<const uint32_t *>(ph + n * kChunk + k0 + 8);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t *>(pl + n * kChunk + k0);
        const uint32_t bl1 = *reinterpret_cast<const uint32_t *>(pl + n * kChunk + k0 + 8);
#pragma unroll
        for (int mt = 0; mt < kD / 16; ++mt) {
            uint32_t a[4];
            pkv::ldsm_x4_trans(a, v_tile + swz((lane >> 4) * 8 + (lane & 7), mt * 2 + ((lane >> 3) & 1)));
            pkv::mma16816(o[mt], a, bh0, bh1);
            pkv::mma16816(o[mt], a, bl0, bl1);
        }
    }

    // Columns go to slots c0 .. c0 + G - 1 of the combine area's nc columns per warp.  kPermDims:
    // the accumulator rows are dims in the int8-value order (row g of m-tile mt = dim 16 g + 2 mt,
    // row g + 8 = dim 16 g + 2 mt + 1).
    template <bool kPermDims = false>
    __device__ __forceinline__ void finish(int warp, int lane, float *c_acc, float *c_m, float *c_l, int nc = G,
                                           int c0 = 0) {
        float l[2] = {l_part[0], l_part[1]};
#pragma unroll
        for (int sh = 4; sh <= 16; sh <<= 1) {
            l[0] += __shfl_xor_sync(pkv::kFullMask, l[0], sh);
            l[1] += __shfl_xor_sync(pkv::kFullMask, l[1], sh);
        }
        float f[2] = {1.f, 1.f}, m[2] = {m_ref[0], m_ref[1]};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (top[j] > -INFINITY) {  // re-reference to the true max: m_ref <= top < m_ref + 2^8
                f[j] = exp2f(m_ref[j] - top[j]);
                l[j] *= f[j];
                m[j] = top[j];
            }
        }
        const int g = lane >> 2, h0 = (lane & 3) * 2;
#pragma unroll
        for (int mt = 0; mt < kD / 16; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = h0 + (e & 1);
                const int dim = kPermDims ? 16 * g + 2 * mt + (e >> 1) : mt * 16 + g + (e >> 1) * 8;
                if (h < G) c_acc[(warp * nc + c0 + h) * kD + dim] = o[mt][e] * f[e & 1];
            }
        if (g == 0) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
                if (h0 + j < G) {
                    c_m[warp * nc + c0 + h0 + j] = m[j];
                    c_l[warp * nc + c0 + h0 + j] = l[j];
                }
        }
    }
};

// ---------------------------------------------------------------- int8-key tensor-core engine
// Same products as TcEngine with K stored as int8 codes (one float32 scale per token row).  The
// dot product is over all 128 dims, so any fixed permutation of the dims applied to both Q and K
// leaves it unchanged: MMA k-slot 2t+e (e = 0, 1) of k-step ks stands for dim 32t + 4ks + e and
// slot 2t+8+e for dim 32t + 4ks + 2 + e (t = lane % 4).  A lane then needs dims [32t, 32t+32) of
// its two token rows g and g+8: four conflict-free 16-byte shared loads per chunk from the
// swizzled int8 tile, converted to exact fp16 integers in registers (byte permute + one fp16x2
// subtract).  The row scale multiplies the finished dot product of each token.
template <int G>
struct TcEngineQ : TcEngine<G> {
    __device__ __forceinline__ static uint32_t swz8(int r, int c16) { return r * 128 + ((c16 ^ (r & 7)) << 4); }

    __device__ __forceinline__ void init(const DecodeParams &P, int b, int kvh, int lane) {
        const int head = lane >> 2;
        const uint4 *qrow = reinterpret_cast<const uint4 *>(
            P.q + (static_cast<int64_t>(b) * P.num_q_heads + kvh * G + (head < G ? head : 0)) * kD + 32 * (lane & 3));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 w = head < G ? __ldg(qrow + i) : make_uint4(0u, 0u, 0u, 0u);
            this->qb[2 * i][0] = w.x;
            this->qb[2 * i][1] = w.y;
            this->qb[2 * i + 1][0] = w.z;
            this->qb[2 * i + 1][1] = w.w;
        }
        this->reset(P);
    }

    __device__ __forceinline__ void qk(uint32_t k_tile, uint32_t s_tile, int valid, int lane, unsigned char *scratch,
                                       int) {
        float s[4];
        int8_scores(s, k_tile, s_tile, valid, lane);
        this->softmax(s, lane, scratch);
    }

    // Scaled, masked log2-domain scores of the chunk from the int8 keys and their row scales.
    __device__ __forceinline__ void int8_scores(float (&s)[4], uint32_t k_tile, uint32_t s_tile, int valid,
                                                int lane) const {
        const int g = lane >> 2, t = lane & 3;
        const uint4 r0 = pkv::lds128(k_tile + swz8(g, 2 * t)), r1 = pkv::lds128(k_tile + swz8(g, 2 * t + 1));
        const uint4 r8 = pkv::lds128(k_tile + swz8(g + 8, 2 * t)), r9 = pkv::lds128(k_tile + swz8(g + 8, 2 * t + 1));
        const uint32_t wg[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const uint32_t w8[8] = {r8.x, r8.y, r8.z, r8.w, r9.x, r9.y, r9.z, r9.w};
        s[0] = s[1] = s[2] = s[3] = 0.f;
        // one accumulator chain: two measured 0.2-0.9 % slower here (the conversions between the
        // MMAs already hide their latency)
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            const uint32_t xg = wg[ks] ^ 0x80808080u, x8 = w8[ks] ^ 0x80808080u;
            const uint32_t a[4] = {pkv::i8x2_to_h2(xg, 0x4140), pkv::i8x2_to_h2(x8, 0x4140),
                                   pkv::i8x2_to_h2(xg, 0x4342), pkv::i8x2_to_h2(x8, 0x4342)};
            pkv::mma16816(s, a, this->qb[ks][0], this->qb[ks][1]);
        }
        const float fg = this->q_scale * pkv::lds32f(s_tile + 4 * g);
        const float f8 = this->q_scale * pkv::lds32f(s_tile + 4 * (g + 8));
        s[0] = g < valid ? s[0] * fg : -INFINITY;
        s[1] = g < valid ? s[1] * fg : -INFINITY;
        s[2] = g + 8 < valid ? s[2] * f8 : -INFINITY;
        s[3] = g + 8 < valid ? s[3] * f8 : -INFINITY;
    }
};

// ---------------------------------------------------------------- int8 keys and values
// TcEngineQ's q.K, with the value rows int8 too.  Each value row's scale multiplies its token's
// weight in P (l keeps the unscaled weights).  For O^T += V^T P^T the MMA's M dimension (dims)
// may be permuted freely as long as the output is written back in order: row g of m-tile mt
// stands for dim 16 g + 2 mt and row g + 8 for dim 16 g + 2 mt + 1, so a lane (g = lane / 4)
// needs dims [16 g, 16 g + 16) of its four token rows (2t, 2t+1, 2t+8, 2t+9): four conflict-free
// 16-byte loads per chunk from the swizzled int8 tile, paired across tokens with a byte
// permute and converted to exact fp16 integers as for the keys.
template <int G>
struct TcEngineQV : TcEngineQ<G> {
    __device__ __forceinline__ void qk(uint32_t k_tile, uint32_t s_tile, int valid, int lane, unsigned char *scratch,
                                       int) {
        float s[4];
        this->int8_scores(s, k_tile, s_tile, valid, lane);
        this->template softmax<false, true>(s, lane, scratch, s_tile + kChunk * 4);
    }

    __device__ __forceinline__ void pv(uint32_t v_tile, int, int lane, unsigned char *scratch) {
        const __half *ph = reinterpret_cast<const __half *>(scratch);
        const __half *pl = ph + 8 * kChunk;
        const int g = lane >> 2, t = lane & 3, k0 = t * 2;
        const uint32_t bh0 = *reinterpret_cast<const uint32_t *>(ph + g * kChunk + k0);
        const uint32_t bh1 = *reinterpret_cast<const uint32_t *>(ph + g * kChunk + k0 + 8);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t *>(pl + g * kChunk + k0);
        const uint32_t bl1 = *reinterpret_cast<const uint32_t *>(pl + g * kChunk + k0 + 8);
        const uint4 r0 = pkv::lds128(v_tile + TcEngineQ<G>::swz8(2 * t, g));
        const uint4 r1 = pkv::lds128(v_tile + TcEngineQ<G>::swz8(2 * t + 1, g));
        const uint4 r8 = pkv::lds128(v_tile + TcEngineQ<G>::swz8(2 * t + 8, g));
        const uint4 r9 = pkv::lds128(v_tile + TcEngineQ<G>::swz8(2 * t + 9, g));
        const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
        const uint32_t w8[4] = {r8.x, r8.y, r8.z, r8.w}, w9[4] = {r9.x, r9.y, r9.z, r9.w};
#pragma unroll
        for (int mt = 0; mt < kD / 16; ++mt) {
            // bytes 2mt, 2mt+1 (dims 16g + 2mt, +1) of the two token rows, interleaved token-wise
            const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
            const uint32_t xa = __byte_perm(w0[mt >> 1], w1[mt >> 1], sel) ^ 0x80808080u;
            const uint32_t xb = __byte_perm(w8[mt >> 1], w9[mt >> 1], sel) ^ 0x80808080u;
            const uint32_t a[4] = {pkv::i8x2_to_h2(xa, 0x4140), pkv::i8x2_to_h2(xa, 0x4342),
                                   pkv::i8x2_to_h2(xb, 0x4140), pkv::i8x2_to_h2(xb, 0x4342)};
            pkv::mma16816(this->o[mt], a, bh0, bh1);
            pkv::mma16816(this->o[mt], a, bl0, bl1);
        }
    }

    __device__ __forceinline__ void finish(int warp, int lane, float *c_acc, float *c_m, float *c_l) {
        TcEngine<G>::template finish<true>(warp, lane, c_acc, c_m, c_l);
    }
};

// ---------------------------------------------------------------- several new tokens per request
// The 8 MMA columns carry (token, head) rows r = 8 rg + c of the request's n * G rows for this kv
// head (token r / G, head r % G), so a verified draft or a prefill chunk is the same tile as a
// packed-GQA decode.  Each column masks the cached positions after its own token's position
// ctx - n + token (causal); dead columns (past the last token) see nothing.
template <int G>
struct TcEngineM : TcEngine<8> {
    int lim[2];  // last visible logical position of the lane's accumulator columns h0, h0 + 1

    __device__ __forceinline__ void init(const DecodeParams &P, int, int, int) { reset(P); }

    // Columns c0 .. c0 + 7 of row group rg, whose groups are nc rows wide.
    __device__ __forceinline__ void bind(const DecodeParams &P, int kvh, int lane, int rg, int64_t qs, int n, int ctx,
                                         int nc = 8, int c0 = 0) {
        const int r = rg * nc + c0 + (lane >> 2);
        const bool live = r / G < n;
        const __half *qrow = P.q + ((qs + (live ? r / G : 0)) * P.num_q_heads + kvh * G + r % G) * kD;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                qb[ks][j] = live ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + (lane & 3) * 2 + j * 8)) : 0u;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int tok = (rg * nc + c0 + (lane & 3) * 2 + j) / G;
            lim[j] = tok < n ? ctx - n + tok : -1;
        }
    }

    __device__ __forceinline__ void qk(uint32_t k_tile, uint32_t, int valid, int lane, unsigned char *scratch,
                                       int tok0) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        dots(s, k_tile, lane);
        const int g = lane >> 2;
        const int p0 = tok0 + g, p8 = tok0 + g + 8;
        s[0] = g < valid && p0 <= lim[0] ? s[0] * q_scale : -INFINITY;
        s[1] = g < valid && p0 <= lim[1] ? s[1] * q_scale : -INFINITY;
        s[2] = g + 8 < valid && p8 <= lim[0] ? s[2] * q_scale : -INFINITY;
        s[3] = g + 8 < valid && p8 <= lim[1] ? s[3] * q_scale : -INFINITY;
        softmax<true>(s, lane, scratch);
    }
};

// Two column tiles (16 (token, head) rows) per CTA: each chunk's K/V tile, staged once, feeds two
// independent 8-column engines, so a request with up to 16 rows per kv head is one stream of the
// cache instead of two.
template <int G>
struct TcEngineM2 {
    TcEngineM<G> e[2];
    static constexpr int kScratch = 2 * 8 * kChunk * 2;  // one engine's P^T buffers

    __device__ __forceinline__ void init(const DecodeParams &P, int b, int kvh, int lane) {
        e[0].init(P, b, kvh, lane);
        e[1].init(P, b, kvh, lane);
    }
    __device__ __forceinline__ void bind(const DecodeParams &P, int kvh, int lane, int rg, int64_t qs, int n, int ctx) {
        e[0].bind(P, kvh, lane, rg, qs, n, ctx, 16, 0);
        e[1].bind(P, kvh, lane, rg, qs, n, ctx, 16, 8);
    }
    __device__ __forceinline__ void qk(uint32_t k_tile, uint32_t s_tile, int valid, int lane, unsigned char *scratch,
                                       int tok0) {
        e[0].qk(k_tile, s_tile, valid, lane, scratch, tok0);
        e[1].qk(k_tile, s_tile, valid, lane, scratch + kScratch, tok0);
    }
    __device__ __forceinline__ void pv(uint32_t v_tile, int valid, int lane, unsigned char *scratch) {
        e[0].pv(v_tile, valid, lane, scratch);
        e[1].pv(v_tile, valid, lane, scratch + kScratch);
    }
    __device__ __forceinline__ void finish(int warp, int lane, float *c_acc, float *c_m, float *c_l) {
        e[0].finish(warp, lane, c_acc, c_m, c_l, 16, 0);
        e[1].finish(warp, lane, c_acc, c_m, c_l, 16, 8);
    }
};

template <int G, int LPT, bool TC, int KQ, int MQ>
using EngineFor = typename std::conditional<
    MQ == 2, TcEngineM2<G>,
    typename std::conditional<MQ == 1, TcEngineM<G>,
    typename std::conditional<
        KQ == 2, TcEngineQV<G>,
        typename std::conditional<
            KQ == 1, TcEngineQ<G>,
            typename std::conditional<TC, TcEngine<(TC ? G : 4)>, FmaEngine<G, LPT>>::type>::type>::type>::type>::type;

// MQ: 0 one token per request; 1 or 2 several tokens per request, with that many 8-column tiles.
template <int G, int LPT, bool TC, int KQ, int MQ>
__global__ void __launch_bounds__(kThreads, (!TC && G >= 8) || MQ == 2
                                                ? 2
                                                : (KQ ? PKV_DECODE_KQ_MIN_CTAS : PKV_DECODE_MIN_CTAS))
    decode_partition_kernel(const __grid_constant__ DecodeParams P) {
    static_assert(!KQ || TC, "int8 keys run on the tensor-core engine");
    static_assert(!MQ || (TC && !KQ), "several tokens per request run on the fp16 tensor-core engine");
    using L = SmemLayout<TC, KQ, MQ == 2 ? 2 : 1>;
    using Engine = EngineFor<G, LPT, TC, KQ, MQ>;
    constexpr int kRow = L::row;
    constexpr int NC = MQ ? 8 * MQ : G;  // packed output columns per CTA

    extern __shared__ __align__(1024) unsigned char smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_rg = MQ ? P.n_row_groups : 1;
    const int part = MQ ? blockIdx.x / n_rg : blockIdx.x;
    const int rg = MQ ? blockIdx.x - part * n_rg : 0;  // row group (fastest: groups share K/V in L2)
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
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
    const int start = P.token_offset + part * P.partition_size;
    int32_t first_ids[kStages];
#pragma unroll
    for (int k = 0; k < kStages; ++k) {
        const int tok = start + (warp + k * kWarps) * kChunk;
        first_ids[k] = (lane == 0 && tok < cap)
                           ? __ldg(P.block_tables + static_cast<int64_t>(b) * P.max_blocks_per_seq + tok / bs)
                           : 0;
    }
    Engine eng;
    eng.init(P, b, kvh, lane);
    int ctx = __ldg(P.context_lens + b);
    if (ctx > cap) {
        if (part == 0 && kvh == 0 && threadIdx.x == 0) pkv::record_error(&g_decode_error, PKV_DEV_BAD_CONTEXT);
        ctx = cap;
    }
    if (ctx < 0) ctx = 0;
    if constexpr (MQ) {
        if (ctx < q_len) {  // the new tokens must already be in the cache
            if (part == 0 && kvh == 0 && rg == 0 && threadIdx.x == 0)
                pkv::record_error(&g_decode_error, PKV_DEV_BAD_CONTEXT);
            return;
        }
        eng.bind(P, kvh, lane, rg, qs_b, q_len, ctx);
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
        if (part == 0 && P.counters != nullptr) {
            pkv::pdl_wait_primary();  // the prefix kernel's partials
            merge_group<G, L::stage_bytes>(P, HeadRows{static_cast<int64_t>(b) * Hq + kvh * G}, P.slot_offset, smem);
        } else if (waits_for_prefix()) {
            pkv::pdl_wait_primary();
        }
        return;
    }
    if (part >= n_parts) return;

    const int n_tok = min(P.partition_size, ctx - start);
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
    // parts: 1 = K (with the int8 keys' scales), 2 = V, 3 = both.  Without split K/V both land on
    // one barrier with one expect_tx for their sum.
    auto issue_from = [=](int i, int64_t phys, int parts) {
        const int cidx = warp + i * kWarps;
        const int tok0 = start + cidx * kChunk;
        const int valid = min(kChunk, n_tok - cidx * kChunk);
        const int lb = tok0 / bs;
        const int off = tok0 - lb * bs;
        const int64_t byte_off = phys * block_stride + kvh * head_stride + static_cast<int64_t>(off) * kRowBytes;
        const uint32_t bytes = static_cast<uint32_t>(valid) * kRowBytes;
        const int st = i % kStages;
        const uint32_t bar_k = bar0 + 8 * st;
        const uint32_t bar_v = bar_v0 + 8 * st;
        const uint32_t dst = stage0 + st * L::stage;
        // TC: whole 16-row boxes (a ragged tail's extra rows stay inside the block and are masked)
        const uint32_t k_bytes = KQ ? L::k_tile + kChunk * 4 : (TC ? 2 * kHalfTile : bytes);
        const uint32_t v_bytes = KQ == 2 ? L::v_tile + kChunk * 4 : (TC ? 2 * kHalfTile : bytes);
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
            if constexpr (KQ == 2) {  // one 16-row box of int8 values and their 16 scales
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
        issue_from(i, s_table[tok0 / bs - lb0], parts);
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

    static_assert(kWarps * NC * (kD + 2) * 4 <= L::stage_bytes, "combine area must fit the stages");

    // ---- fused append: the CTA holding the request's last position writes the new token's K/V
    // row for its kv head into the cache (lanes 0-15: K, 16-31: V of warp own_warp) and patches the
    // row in its shared-memory tile once the chunk has landed, so the attention sees the new token
    // whatever the order of the global write and the bulk copy.
    const int new_pos = ctx - 1;
    const bool appends = P.k_new != nullptr && part == n_parts - 1;
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
            // Lanes 0-15 quantise the K row (8 dims each; scale from a 16-lane max), 16-31 move V.
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
            const float sc = __fdiv_rn(amax, 127.f);
            if (lane < 16) {
                uint32_t c[2] = {0u, 0u};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    c[e >> 2] |= (static_cast<uint32_t>(pkv::quantize_int8(f[e], sc)) & 0xffu) << (8 * (e & 3));
                const uint2 codes = make_uint2(c[0], c[1]);
                *reinterpret_cast<uint2 *>(s_newrow + lane * 8) = codes;
                if (lane == 0) *reinterpret_cast<float *>(s_newrow + kD) = sc;
                if (id_ok) {
                    *reinterpret_cast<uint2 *>(reinterpret_cast<unsigned char *>(P.k_cache_w) + grow * kD + lane * 8) =
                        codes;
                    if (lane == 0) P.k_scale_w[grow] = sc;
                }
            } else if (KQ == 2) {  // lanes 16-31 quantise the V row the same way
                const int l16 = lane & 15;
                uint32_t c[2] = {0u, 0u};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    c[e >> 2] |= (static_cast<uint32_t>(pkv::quantize_int8(f[e], sc)) & 0xffu) << (8 * (e & 3));
                const uint2 codes = make_uint2(c[0], c[1]);
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
        // the appended token's V row and a ragged tail's V rows, once V has landed
        auto fix_v = [&]() {
            bool touched = false;
            // (int8 values need no clearing: codes are finite and the scaled weights of the unused
            // rows are forced to zero)
            if (TC && KQ != 2 && valid < kChunk) {
                for (int x = lane; x < (kChunk - valid) * 16; x += 32)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(v_tile + TcEngine<4>::swz(valid + x / 16, x % 16)),
                                 "r"(0)
                                 : "memory");
                touched = true;
            }
            if (own) {
                if (KQ == 2 && lane >= 16) {  // int8 value row (8 bytes a lane) and its scale
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
                } else if (KQ != 2 && lane >= 16) {
                    const uint4 nr = *reinterpret_cast<const uint4 *>(s_newrow + lane * 16);
                    const uint32_t row = TC ? TcEngine<4>::swz(nr_row, lane & 15) : nr_row * kRow + (lane & 15) * 16;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(v_tile + row), "r"(nr.x), "r"(nr.y),
                                 "r"(nr.z), "r"(nr.w)
                                 : "memory");
                }
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
    float *c_acc = reinterpret_cast<float *>(smem);                  // [kWarps][NC][kD]
    float *c_m = c_acc + kWarps * NC * kD;                           // [kWarps][NC]
    float *c_l = c_m + kWarps * NC;                                  // [kWarps][NC]
    eng.finish(warp, lane, c_acc, c_m, c_l);
    __syncthreads();
    const TokenRows<G, NC> token_rows{qs_b, q_len, rg, Hq, kvh};
#pragma unroll 1
    for (int idx = threadIdx.x; idx < NC * kD; idx += kThreads) {
        const int hh = idx / kD, d = idx % kD;
        if (MQ && !token_rows.live(hh)) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, c_m[w * NC + hh]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float cm = c_m[w * NC + hh];
            // 0 for warps without chunks; with causal masking a column can have seen no token at all
            const float f = (MQ && cm == -INFINITY) ? 0.f : exp2f(cm - M);
            L = fmaf(c_l[w * NC + hh], f, L);
            O = fmaf(c_acc[(w * NC + hh) * kD + d], f, O);
        }
        const int64_t row = MQ ? token_rows.row(hh) : static_cast<int64_t>(b) * Hq + kvh * G + hh;
        const float o = (MQ && L == 0.f) ? 0.f : O / L;
        if (direct) {
            P.out[row * kD + d] = __float2half_rn(o);
        } else {
            const int64_t prow = row * P.max_partitions + P.slot_offset + part;
            P.o_part[prow * kD + d] = o;
            if (d == 0) {
                P.m_part[prow] = M * kLn2;
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
    if (threadIdx.x == 0) s_last = pkv::atomic_add_acq_rel_gpu(counter, 1) == n_parts - 1;
    __syncthreads();
    if (!s_last) return;
    if (P.slot_offset > 0) pkv::pdl_wait_primary();  // shared-prefix pass: the prefix kernel's partials
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
    const int kvh = blockIdx.x, b = blockIdx.y;
    // the suffix pass's partition count for this request (same clamps)
    const int cap = P.max_blocks_per_seq * P.block_size;
    int ctx = __ldg(P.context_lens + b);
    ctx = max(min(ctx, cap), P.token_offset);
    const int n_parts = (ctx - P.token_offset + P.partition_size - 1) / P.partition_size;
    merge_group<G, kMergeStageBytes>(P, HeadRows{static_cast<int64_t>(b) * P.num_q_heads + kvh * G},
                                     P.slot_offset + n_parts, smem);
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

template <int G, int KQ, int MQ>
int launch_partition(const DecodeParams &p_in, int num_seqs, cudaStream_t stream, int grid_parts) {
    constexpr int LPT = lanes_per_token<G>();
    constexpr bool TC = KQ || MQ || (PKV_DECODE_TC && G >= PKV_DECODE_TC_MIN_GROUP);
    auto kernel = decode_partition_kernel<G, LPT, TC, KQ, MQ>;
    DecodeParams p = p_in;
    if (TC) {
        const int64_t rows = p.num_blocks * p.num_kv_heads * p.block_size;
        if (rows >= 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // box row coordinates are signed 32-bit
        int st = KQ ? encode_code_map(&p.tmap_k, p.k_cache, rows) : encode_cache_map(&p.tmap_k, p.k_cache, rows);
        if (st == PKV_OK)
            st = KQ == 2 ? encode_code_map(&p.tmap_v, p.v_cache, rows) : encode_cache_map(&p.tmap_v, p.v_cache, rows);
        if (st != PKV_OK) return st;
    }
    using L = SmemLayout<TC, KQ, MQ == 2 ? 2 : 1>;
    const int smem = L::total(G, p.partition_size);
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
    const dim3 grid(static_cast<unsigned>(gx), p.num_kv_heads, num_seqs);
    if (p.slot_offset == 0) {
        kernel<<<grid, kThreads, smem, stream>>>(p);
        return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
    }
    // Suffix pass after the shared-prefix kernel: launched as a programmatic dependent so it
    // streams the suffixes while the prefix kernel runs; only its merges wait for the prefix.
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
    if (p.query_start)
        return p.mq_tiles == 2 ? launch_partition<G, 0, 2>(p, num_seqs, stream, grid_parts)
                               : launch_partition<G, 0, 1>(p, num_seqs, stream, grid_parts);
    if (p.k_scale && p.v_scale) return launch_partition<G, 2, 0>(p, num_seqs, stream, grid_parts);
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
// k_scale non-null: k_cache holds int8 codes with these float32 row scales.
int decode_attention_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                          int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int64_t num_blocks, float scale, const void *k_new, const void *v_new, void *workspace,
                          size_t workspace_bytes, pkv_stream_t stream, const float *k_scale = nullptr,
                          int partition_size = PKV_DEFAULT_PARTITION, const float *v_scale = nullptr) {
    int st = check_common(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks);
    if (st != PKV_OK) return st;
    if (k_scale && !pkv_internal::aligned16(k_scale)) return PKV_ERR_INVALID_ARG;
    if (v_scale && (!k_scale || !pkv_internal::aligned16(v_scale))) return PKV_ERR_INVALID_ARG;
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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (max_parts <= 1) return dispatch_partition(p, num_seqs, num_q_heads / num_kv_heads, s);

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
                                       size_t workspace_bytes, pkv_stream_t stream) {
    if (!k_new || !v_new) return PKV_ERR_INVALID_ARG;
    if (prefix_len > 0)
        return pkv_internal::shared_prefix_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                                  max_blocks_per_seq, num_q_heads, num_kv_heads, head_dim, block_size,
                                                  num_blocks, scale, prefix_len, k_new, v_new, workspace,
                                                  workspace_bytes, stream);
    if (prefix_len < 0) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream);
}

extern "C" PKV_API int pkv_decode_step_partition(void *out, const void *q, const void *k_new, const void *v_new,
                                                 void *k_cache, void *v_cache, const int32_t *block_tables,
                                                 const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                                 int64_t num_blocks, float scale, int partition_size,
                                                 void *workspace, size_t workspace_bytes, pkv_stream_t stream) {
    if (!k_new || !v_new || partition_size < 0) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream, nullptr,
                                 partition_size > 0 ? partition_size : PKV_DEFAULT_PARTITION);
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
                                             size_t workspace_bytes, pkv_stream_t stream) {
    if (!k_new || !v_new || !k_scale) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_codes, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream, k_scale);
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

extern "C" PKV_API int pkv_decode_attention_multi(void *out, const void *q, const void *k_cache, const void *v_cache,
                                                  const int32_t *block_tables, const int32_t *context_lens,
                                                  const int32_t *query_start, int num_seqs, int total_q,
                                                  int max_query_len, int max_blocks_per_seq, int num_q_heads,
                                                  int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                                  float scale, void *workspace, size_t workspace_bytes,
                                                  pkv_stream_t stream) {
    int st = check_common(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks);
    if (st != PKV_OK) return st;
    if (!out || !pkv_internal::aligned(out, 8) || !query_start || !pkv_internal::aligned(query_start, 4))
        return PKV_ERR_INVALID_ARG;
    if (total_q < 0 || max_query_len <= 0) return PKV_ERR_INVALID_ARG;
    if (max_query_len > PKV_MAX_QUERY_LEN) return PKV_ERR_UNSUPPORTED;
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
                                              void *workspace, size_t workspace_bytes, pkv_stream_t stream) {
    if (!k_new || !v_new || !k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    return decode_attention_impl(out, q, k_codes, v_codes, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_new, v_new,
                                 workspace, workspace_bytes, stream, k_scale, PKV_DEFAULT_PARTITION, v_scale);
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
    if (a.separate_merge) p.counters = nullptr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int group = a.num_q_heads / a.num_kv_heads;
    const int st = dispatch_partition(p, a.num_seqs, group, s, a.grid_partitions);
    if (st != PKV_OK || !a.separate_merge) return st;
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
