// pkv_engine.cuh -- the decode engines shared by the decode kernels' translation units: the
// split-context parameter block, the shared-memory layout of a decode CTA, the log-sum-exp merge
// of partial slots, and the per-warp engines that turn a staged 16-token K/V chunk into online-
// softmax state (CUDA-core FMAs; tensor-core mma.m16n8k16 over fp16, int8-key and int8 K + V
// caches; several tokens per request).  Everything here has internal linkage: each translation
// unit that includes it gets its own copy.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "pkv.h"
#include "pkv_device.cuh"

namespace {

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
// Copy stages per warp of the 16-column multi-token kernel (it runs at 2 CTAs per SM).
#ifndef PKV_DECODE_MQ2_STAGES
#define PKV_DECODE_MQ2_STAGES 2
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
    int kv_fp8;               // with k_scale and v_scale: the codes are E4M3 (fp8), not int8
    int overlap;              // 1: stream the cache history before the preceding kernel completes
    int stagger;              // automatic split: odd partitions start this many tokens early, so the
                              //   partitions alternate partition_size -/+ stagger tokens (0: all equal)
    int prefix_ctas;          // shared-prefix step in one grid: CTAs [0, prefix_ctas) are prefix tiles
    int prefix_chunks;        //   128-token prefix chunks (partial slots [0, prefix_chunks))
    int grid_parts;           //   suffix partitions per (request, kv head) in the grid
    int num_seqs;             //   requests
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
// Row stride (floats) of the warps' partial results in the combine area: 4 floats of padding so
// the fragment-ordered stores of eight rows at once spread over all 32 banks.
constexpr int kAccStride = kD + 4;
// KQ: 0 fp16 K/V, 1 int8 keys, 2 int8 keys and values, 3 fp8 (E4M3) keys and values.  NR: new token rows staged for a fused
// append (one for a single-token step; up to PKV_MAX_STEP_QUERY_LEN for a several-token step).
// The 16-row engine (NT = 2) keeps P in registers and needs no per-warp weight buffer.
template <bool TC, int KQ = 0, int NT = 1, int NS = kStages, int NR = 1>
struct SmemLayout {
    static constexpr int row = kRowBytes;
    static constexpr int tile = kChunk * row;
    static constexpr int k_tile = KQ ? kChunk * kD : tile;
    static constexpr int v_tile = KQ >= 2 ? kChunk * kD : tile;
    static constexpr int stage = k_tile + v_tile;
    static constexpr int scale_stride = KQ >= 2 ? 2 * kChunk * 4 : kChunk * 4;  // K scales (| V scales) per stage
    static constexpr int stages = 0;
    static constexpr int stage_bytes = kWarps * NS * stage;
    static constexpr int scales = stages + stage_bytes;
    static constexpr int bars = scales + (KQ ? kWarps * NS * scale_stride : 0);
    static constexpr int probs = bars + kWarps * NS * kBarsPerStage * 8;
    static_assert(probs % 16 == 0, "the weight rows are read by ldmatrix (16-byte rows)");
    __host__ __device__ static constexpr int probs_per_warp(int g) {
        return TC ? (NT == 2 ? 0 : NT * 2 * 8 * kChunk * 2) : kChunk * g * 4;
    }
    __host__ __device__ static constexpr int newrow(int g) { return probs + kWarps * probs_per_warp(g); }
    __host__ __device__ static constexpr int table(int g) { return newrow(g) + NR * 2 * kRowBytes; }
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
            *reinterpret_cast<float4 *>(c_acc + (warp * G + hh) * kAccStride + lane * 4) =
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
        float p[4] = {pkv::exp2_approx(s[0] - m_ref[0]), pkv::exp2_approx(s[1] - m_ref[1]),
                      pkv::exp2_approx(s[2] - m_ref[0]), pkv::exp2_approx(s[3] - m_ref[1])};
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
        // P^T through shared memory as fp16 hi / lo rows, [2][16 tokens][8 heads] (16 bytes a row):
        // this lane's two columns of tokens g and g + 8, one 32-bit store each
        const uint32_t base = pkv::smem_addr(scratch) + (lane & 3) * 4;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const __half2 hi = __floats2half2_rn(p[2 * r], p[2 * r + 1]);
            const __half2 lo = __floats2half2_rn(p[2 * r] - __low2float(hi), p[2 * r + 1] - __high2float(hi));
            const uint32_t row = base + (g + 8 * r) * 16;
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(row), "r"(*reinterpret_cast<const uint32_t *>(&hi)) : "memory");
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(row + 256), "r"(*reinterpret_cast<const uint32_t *>(&lo))
                         : "memory");
        }
        __syncwarp();
    }

    // The B fragments of P^T (16 tokens x 8 heads; hi then lo) that softmax() left in scratch: one
    // transposing matrix load, lanes 8m .. 8m + 7 addressing the rows of matrix m (hi tokens 0-7,
    // hi 8-15, lo 0-7, lo 8-15), so each lane gets tokens 2t, 2t + 1 (and + 8) of head lane / 4.
    __device__ __forceinline__ static void weights(uint32_t (&b)[4], int lane, const unsigned char *scratch) {
        pkv::ldsm_x4_trans(b, pkv::smem_addr(scratch) + (lane >> 4) * 256 + ((lane >> 3) & 1) * 128 + (lane & 7) * 16);
    }

    // O^T += V_tile^T . P^T with the weights softmax() left in scratch.
    __device__ __forceinline__ void pv(uint32_t v_tile, int, int lane, unsigned char *scratch) {
        uint32_t b[4];
        weights(b, lane, scratch);
        const uint32_t bh0 = b[0], bh1 = b[1], bl0 = b[2], bl1 = b[3];
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
                if (h < G) c_acc[(warp * nc + c0 + h) * kAccStride + dim] = o[mt][e] * f[e & 1];
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
        const int g = lane >> 2, t = lane & 3;
        uint32_t b[4];
        TcEngine<G>::weights(b, lane, scratch);
        const uint32_t bh0 = b[0], bh1 = b[1], bl0 = b[2], bl1 = b[3];
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

// ---------------------------------------------------------------- fp8 (E4M3) keys and values
// TcEngineQV's tiles, dim permutations, scales and weights with E4M3 codes: each code pair
// becomes an fp16x2 MMA operand by one hardware conversion (exact), in place of the int8 codes'
// sign flip, byte permute and fp16 subtract.  The value pairs are still formed across tokens by
// one byte permute per A register pair.  Unused value rows of a ragged tail are cleared before
// P.V (E4M3 has NaN codes, and NaN x 0 is NaN).
template <int G>
struct TcEngineF8 : TcEngineQ<G> {
    __device__ __forceinline__ void qk(uint32_t k_tile, uint32_t s_tile, int valid, int lane, unsigned char *scratch,
                                       int) {
        const int g = lane >> 2, t = lane & 3;
        const uint4 r0 = pkv::lds128(k_tile + TcEngineQ<G>::swz8(g, 2 * t));
        const uint4 r1 = pkv::lds128(k_tile + TcEngineQ<G>::swz8(g, 2 * t + 1));
        const uint4 r8 = pkv::lds128(k_tile + TcEngineQ<G>::swz8(g + 8, 2 * t));
        const uint4 r9 = pkv::lds128(k_tile + TcEngineQ<G>::swz8(g + 8, 2 * t + 1));
        const uint32_t wg[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const uint32_t w8[8] = {r8.x, r8.y, r8.z, r8.w, r9.x, r9.y, r9.z, r9.w};
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t a[4];
            pkv::e4m3x4_to_h2x2(wg[ks], a[0], a[2]);
            pkv::e4m3x4_to_h2x2(w8[ks], a[1], a[3]);
            pkv::mma16816(s, a, this->qb[ks][0], this->qb[ks][1]);
        }
        const float fg = this->q_scale * pkv::lds32f(s_tile + 4 * g);
        const float f8 = this->q_scale * pkv::lds32f(s_tile + 4 * (g + 8));
        s[0] = g < valid ? s[0] * fg : -INFINITY;
        s[1] = g < valid ? s[1] * fg : -INFINITY;
        s[2] = g + 8 < valid ? s[2] * f8 : -INFINITY;
        s[3] = g + 8 < valid ? s[3] * f8 : -INFINITY;
        this->template softmax<false, true>(s, lane, scratch, s_tile + kChunk * 4);
    }

    __device__ __forceinline__ void pv(uint32_t v_tile, int, int lane, unsigned char *scratch) {
        const int g = lane >> 2, t = lane & 3;
        uint32_t b[4];
        TcEngine<G>::weights(b, lane, scratch);
        const uint32_t bh0 = b[0], bh1 = b[1], bl0 = b[2], bl1 = b[3];
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
            const uint32_t xa = __byte_perm(w0[mt >> 1], w1[mt >> 1], sel);
            const uint32_t xb = __byte_perm(w8[mt >> 1], w9[mt >> 1], sel);
            uint32_t a[4];
            pkv::e4m3x4_to_h2x2(xa, a[0], a[1]);
            pkv::e4m3x4_to_h2x2(xb, a[2], a[3]);
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

// Sixteen (token, head) rows of one kv head as the M dimension of the MMAs (several tokens per
// request, more than 8 rows per kv head): per 16-token chunk
//   S[16 rows x 16 tok] = Q[16 x 128] . K^T     2 n-tiles x 8 k-steps of mma.m16n8k16, K by ldmatrix
//   O[16 rows x 128]   += P[16 x 16] . V         16 n-tiles x 2 (P = hi + lo), V by ldmatrix.trans
// with fp32 accumulation.  Q stays in registers as A fragments, and P goes from the S accumulators
// straight into A fragments (no shared-memory round trip), so one engine holds what two 8-column
// engines held and the kernel fits three CTAs per SM.  Lane l owns rows g = l / 4 and g + 8 for the
// online softmax; each row masks the cached positions after its own token's (causal).
template <int G>
struct TcEngineR16 {
    uint32_t qa[kD / 16][4];  // Q A-fragments of the 8 k-steps
    float o[kD / 8][4];       // O: n-tile j = dims 8j .. 8j + 7: (row g, dims 8j + 2t, +1), (row g + 8, same)
    uint32_t ph[4], pl[4];    // the chunk's P as A fragments, fp16 hi and lo parts
    float m_ref[2], top[2], l_part[2];  // rows g, g + 8 (log2 units; l_part this lane's share)
    int lim[2];                         // last visible logical position of rows g, g + 8 (-1: dead row)
    float q_scale;

    __device__ __forceinline__ void init(const DecodeParams &P, int, int, int) {
#pragma unroll
        for (int j = 0; j < kD / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        m_ref[0] = m_ref[1] = top[0] = top[1] = -INFINITY;
        l_part[0] = l_part[1] = 0.f;
        q_scale = P.q_scale;
    }

    // Rows rg * 16 .. rg * 16 + 15 of the request's n * G rows for kv head kvh (row r = token r / G,
    // head r % G); rows past the last token are dead (zero q, nothing visible).
    __device__ __forceinline__ void bind(const DecodeParams &P, int kvh, int lane, int rg, int64_t qs, int n, int ctx) {
        const int g = lane >> 2, t = lane & 3;
        const __half *qrow[2];
        bool live[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = rg * 16 + g + 8 * i;
            live[i] = r / G < n;
            qrow[i] = P.q + ((qs + (live[i] ? r / G : 0)) * P.num_q_heads + kvh * G + r % G) * kD;
            lim[i] = live[i] ? ctx - n + r / G : -1;
        }
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = k & 1, d = ks * 16 + 2 * t + (k >> 1) * 8;
                qa[ks][k] = live[i] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[i] + d)) : 0u;
            }
    }

    __device__ __forceinline__ void qk(uint32_t k_tile, uint32_t, int valid, int lane, unsigned char *, int tok0) {
        const int t = lane & 3;
        float s[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t b[4];
            pkv::ldsm_x4(b, k_tile + TcEngine<8>::swz((lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)));
            pkv::mma16816(s[0], qa[ks], b[0], b[1]);
            pkv::mma16816(s[1], qa[ks], b[2], b[3]);
        }
        // mask (past the chunk's tokens, or after the row's own position) and scale: token
        // 8j + 2t + c of the chunk is visible to row i iff 8j + c <= cut[i]
        float cm[2] = {-INFINITY, -INFINITY};
        const int cut[2] = {min(valid - 1, lim[0] - tok0) - 2 * t, min(valid - 1, lim[1] - tok0) - 2 * t};
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = e >> 1;
                s[j][e] = 8 * j + (e & 1) <= cut[i] ? s[j][e] * q_scale : -INFINITY;
                cm[i] = fmaxf(cm[i], s[j][e]);
            }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            cm[i] = fmaxf(cm[i], __shfl_xor_sync(pkv::kFullMask, cm[i], 1));
            cm[i] = fmaxf(cm[i], __shfl_xor_sync(pkv::kFullMask, cm[i], 2));
            top[i] = fmaxf(top[i], cm[i]);
        }
        // online softmax with the lazy 2^8 margin; a row with nothing visible yet keeps weight 0
        if (__any_sync(pkv::kFullMask, cm[0] > m_ref[0] + kRescaleThreshold || cm[1] > m_ref[1] + kRescaleThreshold)) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float mn = fmaxf(m_ref[i], cm[i]);
                const float a = mn == -INFINITY ? 1.f : exp2f(m_ref[i] - mn);
                m_ref[i] = mn;
                l_part[i] *= a;
#pragma unroll
                for (int j = 0; j < kD / 8; ++j) {
                    o[j][2 * i] *= a;
                    o[j][2 * i + 1] *= a;
                }
            }
        }
        // 2^(-inf) = 0 for masked tokens; a row that has seen nothing yet (reference max still
        // -inf) has only masked tokens, so it subtracts 0 instead
        const float m_use[2] = {m_ref[0] == -INFINITY ? 0.f : m_ref[0], m_ref[1] == -INFINITY ? 0.f : m_ref[1]};
        float p[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = e >> 1;
                p[j][e] = pkv::exp2_approx(s[j][e] - m_use[i]);
                l_part[i] += p[j][e];
            }
        // A fragments of P (rows g / g + 8 x tokens 2t, 2t + 1 / + 8), hi + lo parts
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = k >> 1, e = (k & 1) * 2;  // a0 (j 0, row g), a1 (j 0, row g + 8), a2 (j 1, g), a3 (j 1, g + 8)
            const __half2 hi = __floats2half2_rn(p[j][e], p[j][e + 1]);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(p[j][e] - hf.x, p[j][e + 1] - hf.y);
            ph[k] = *reinterpret_cast<const uint32_t *>(&hi);
            pl[k] = *reinterpret_cast<const uint32_t *>(&lo);
        }
    }

    __device__ __forceinline__ void pv(uint32_t v_tile, int, int lane, unsigned char *) {
#pragma unroll
        for (int j2 = 0; j2 < kD / 16; ++j2) {
            uint32_t b[4];
            pkv::ldsm_x4_trans(b, v_tile + TcEngine<8>::swz((lane & 7) + ((lane >> 3) & 1) * 8, 2 * j2 + (lane >> 4)));
            pkv::mma16816(o[2 * j2], ph, b[0], b[1]);
            pkv::mma16816(o[2 * j2 + 1], ph, b[2], b[3]);
            pkv::mma16816(o[2 * j2], pl, b[0], b[1]);
            pkv::mma16816(o[2 * j2 + 1], pl, b[2], b[3]);
        }
    }

    // Rows g and g + 8 into the combine area's 16 columns per warp, re-referenced to the true max.
    __device__ __forceinline__ void finish(int warp, int lane, float *c_acc, float *c_m, float *c_l) {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float l = l_part[i];
            l += __shfl_xor_sync(pkv::kFullMask, l, 1);
            l += __shfl_xor_sync(pkv::kFullMask, l, 2);
            float m = m_ref[i], f = 1.f;
            if (top[i] > -INFINITY) {  // m_ref <= top < m_ref + 2^8
                f = exp2f(m_ref[i] - top[i]);
                l *= f;
                m = top[i];
            }
            const int row = g + 8 * i;
            float *acc = c_acc + (warp * 16 + row) * kAccStride + 2 * t;
#pragma unroll
            for (int j = 0; j < kD / 8; ++j)
                *reinterpret_cast<float2 *>(acc + 8 * j) = make_float2(o[j][2 * i] * f, o[j][2 * i + 1] * f);
            if (t == 0) {
                c_m[warp * 16 + row] = m;
                c_l[warp * 16 + row] = l;
            }
        }
    }

    // Where each warp owns distinct rows (a shared-prefix tile: row r of the B * G rows of one kv
    // head is request r / G, head r % G, i.e. bound with qs = 0 and n = B), no warp combine: the
    // rows' partial result (max in natural-log units, weight sum, o / l) is stored as `slot` of
    // the split layout.  rg: the warp's 16-row group; rows past n_rows are not stored.
    __device__ __forceinline__ void store_partial(const DecodeParams &P, int lane, int rg, int n_rows, int kvh,
                                                  int slot) {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float l = l_part[i];
            l += __shfl_xor_sync(pkv::kFullMask, l, 1);
            l += __shfl_xor_sync(pkv::kFullMask, l, 2);
            float m = m_ref[i], f = 1.f;
            if (top[i] > -INFINITY) {  // m_ref <= top < m_ref + 2^8
                f = exp2f(m_ref[i] - top[i]);
                l *= f;
                m = top[i];
            }
            const int r = rg * 16 + g + 8 * i;
            if (r >= n_rows) continue;
            const int64_t row = static_cast<int64_t>(r / G) * P.num_q_heads + kvh * G + r % G;
            const int64_t prow = row * P.max_partitions + slot;
            const float s = f / l;
            float *o_out = P.o_part + prow * kD + 2 * t;
#pragma unroll
            for (int j = 0; j < kD / 8; ++j)
                *reinterpret_cast<float2 *>(o_out + 8 * j) = make_float2(o[j][2 * i] * s, o[j][2 * i + 1] * s);
            if (t == 0) {
                P.m_part[prow] = m * kLn2;
                P.l_part[prow] = l;
            }
        }
    }
};

template <int G, int LPT, bool TC, int KQ, int MQ>
using EngineFor = typename std::conditional<
    MQ == 2, TcEngineR16<G>,
    typename std::conditional<MQ == 1, TcEngineM<G>,
    typename std::conditional<
        KQ == 3, TcEngineF8<G>,
    typename std::conditional<
        KQ == 2, TcEngineQV<G>,
        typename std::conditional<
            KQ == 1, TcEngineQ<G>,
            typename std::conditional<TC, TcEngine<(TC ? G : 4)>, FmaEngine<G, LPT>>::type>::type>::type>::type>::type>::type;

}  // namespace
