// pkv_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pkv_internal {

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline bool aligned16(const void *p) { return aligned(p, 16); }

// Each kernel translation unit owns one device error word; these read it for
// the current device and reset it to zero.  Return PKV_OK or PKV_ERR_CUDA.
int append_take_error(int *code);
int decode_take_error(int *code);
int prefix_take_error(int *code);

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A cache tensor [rows][128] fp16 as a tensor map (CUtensorMap, passed as void*) for 2-D tensor
// copies of 16-row x 64-dim boxes in the 128-byte swizzle.  PKV_OK or PKV_ERR_CUDA.
int encode_fp16_cache_map(void *map, const void *base, int64_t rows);
// q [num_seqs][num_q_heads][128] fp16 as a 3-D tensor map read in (64 dims, group heads, 128 / group
// requests) boxes in the 128-byte swizzle: 128 query rows of one kv head.  PKV_OK or PKV_ERR_CUDA.
int encode_q_map(void *map, const void *q, int num_seqs, int num_q_heads, int group);

// Host-side argument checks shared by every decode entry point (PKV_OK or an error status).
int check_decode_args(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
                      const int32_t *context_lens, int num_seqs, int max_blocks_per_seq, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks);

// One split pass of the decode kernel writing partial slots [slot_offset, slot_offset + parts)
// for the tokens from token_offset on, with the log-sum-exp merge of slots
// [0, slot_offset + parts) fused in (counters must be zero; they are left zero), or, with
// separate_merge, done by a merge kernel launched after the pass (counters unused).
struct SplitPass {
    void *out;
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    int num_seqs, max_blocks_per_seq, num_q_heads, num_kv_heads, block_size;
    int64_t num_blocks;
    float scale;
    int partition_size, max_partitions, token_offset, slot_offset, grid_partitions;
    float *o_part, *m_part, *l_part;
    int *counters;
    const void *k_new, *v_new;  // non-null: fused append of the new token (caches are written)
    bool separate_merge;
    int prefix_ctas = 0;    // > 0: the shared-prefix step in one grid, these prefix tiles first
    int prefix_chunks = 0;  //   (128-token prefix chunks; the merge is fused, separate_merge false)
    bool overlap = false;   //   PKV_STEP_OVERLAP
};
int launch_split_pass(const SplitPass &a, void *stream);

// Shared-prefix decode (prefix kernel + suffix pass), optionally appending the new tokens.
int shared_prefix_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                         int max_blocks_per_seq, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, float scale, int prefix_len, const void *k_new, const void *v_new,
                         void *workspace, size_t workspace_bytes, void *stream, bool overlap = false);

}  // namespace pkv_internal
