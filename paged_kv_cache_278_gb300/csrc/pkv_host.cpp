// pkv_host.cpp -- host half of the library: the KV block pool, the host slot
// mapping, status strings and the device error report.
//
// The pool implements paged allocation of the cache in fixed-size blocks,
// allocation on demand, release at the end of a request (all-or-nothing, so a
// failed request leaves nothing behind) and reference counts for blocks shared
// as a common prompt prefix ("推理优化这件事，为什么值得反复复盘", sec. 4.2;
// "为什么“推理优化”不是锦上添花", sec. 3.2, scheme 1: pages indexed through a
// page table).
#include <cuda_runtime.h>

#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"
#include "pkv_internal.h"

struct pkv_pool {
    std::vector<int32_t> free_list;  // stack; back() is handed out next
    std::vector<int32_t> refcount;   // 0 = free
};

namespace {

uint64_t splitmix64(uint64_t &state) {
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Unbiased draw in [0, n) by rejection.
uint64_t draw_below(uint64_t &state, uint64_t n) {
    const uint64_t limit = UINT64_MAX - UINT64_MAX % n;
    uint64_t x;
    do {
        x = splitmix64(state);
    } while (x >= limit);
    return x % n;
}

}  // namespace

extern "C" {

PKV_API const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_OUT_OF_BLOCKS: return "out of KV-cache blocks";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_DEVICE_CHECK: return "device-side index check failed";
        default: return "unknown status";
    }
}

PKV_API int pkv_version(void) { return 10000; }

PKV_API int pkv_pool_create(int64_t num_blocks, uint64_t seed, pkv_pool **out) {
    if (!out || num_blocks <= 0 || num_blocks > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_pool *pool = new (std::nothrow) pkv_pool;
    if (!pool) return PKV_ERR_INVALID_ARG;
    try {
        pool->free_list.resize(static_cast<size_t>(num_blocks));
        pool->refcount.assign(static_cast<size_t>(num_blocks), 0);
    } catch (...) {
        delete pool;
        return PKV_ERR_INVALID_ARG;
    }
    for (int64_t i = 0; i < num_blocks; ++i) pool->free_list[i] = static_cast<int32_t>(i);
    uint64_t state = seed;
    for (int64_t i = num_blocks - 1; i > 0; --i) {  // Fisher-Yates
        const int64_t j = static_cast<int64_t>(draw_below(state, static_cast<uint64_t>(i) + 1));
        const int32_t tmp = pool->free_list[i];
        pool->free_list[i] = pool->free_list[j];
        pool->free_list[j] = tmp;
    }
    *out = pool;
    return PKV_OK;
}

PKV_API void pkv_pool_destroy(pkv_pool *pool) { delete pool; }

PKV_API int pkv_pool_alloc(pkv_pool *pool, int n, int32_t *ids) {
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    if (static_cast<size_t>(n) > pool->free_list.size()) return PKV_ERR_OUT_OF_BLOCKS;
    for (int i = 0; i < n; ++i) {
        const int32_t id = pool->free_list.back();
        pool->free_list.pop_back();
        pool->refcount[id] = 1;
        ids[i] = id;
    }
    return PKV_OK;
}

PKV_API int pkv_pool_share(pkv_pool *pool, int n, const int32_t *ids) {
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    const int64_t nb = static_cast<int64_t>(pool->refcount.size());
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= nb || pool->refcount[ids[i]] <= 0 || pool->refcount[ids[i]] == INT32_MAX)
            return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) ++pool->refcount[ids[i]];
    return PKV_OK;
}

PKV_API int pkv_pool_free(pkv_pool *pool, int n, const int32_t *ids) {
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    const int64_t nb = static_cast<int64_t>(pool->refcount.size());
    std::unordered_map<int32_t, int> drops;  // validate everything before changing anything
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= nb) return PKV_ERR_INVALID_ARG;
        if (++drops[ids[i]] > pool->refcount[ids[i]]) return PKV_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n; ++i) {
        if (--pool->refcount[ids[i]] == 0) pool->free_list.push_back(ids[i]);
    }
    return PKV_OK;
}

PKV_API int64_t pkv_pool_num_free(const pkv_pool *pool) {
    return pool ? static_cast<int64_t>(pool->free_list.size()) : -1;
}

PKV_API int pkv_pool_refcount(const pkv_pool *pool, int32_t id) {
    if (!pool || id < 0 || static_cast<size_t>(id) >= pool->refcount.size()) return -1;
    return pool->refcount[id];
}

PKV_API int pkv_pool_reserve(pkv_pool *pool, int32_t *table_row, int max_blocks, int cur_tokens, int new_tokens,
                             int block_size) {
    if (!pool || !table_row || max_blocks <= 0 || block_size <= 0 || cur_tokens < 0 || new_tokens < cur_tokens)
        return PKV_ERR_INVALID_ARG;
    const int64_t have = (static_cast<int64_t>(cur_tokens) + block_size - 1) / block_size;
    const int64_t want = (static_cast<int64_t>(new_tokens) + block_size - 1) / block_size;
    if (want > max_blocks) return PKV_ERR_INVALID_ARG;
    if (want == have) return PKV_OK;
    return pkv_pool_alloc(pool, static_cast<int>(want - have), table_row + have);
}

PKV_API int pkv_pool_fork(pkv_pool *pool, const int32_t *src_row, int32_t *dst_row, int max_blocks, int num_tokens,
                          int block_size) {
    if (!pool || !src_row || !dst_row || max_blocks <= 0 || block_size <= 0 || num_tokens < 0)
        return PKV_ERR_INVALID_ARG;
    const int64_t n = (static_cast<int64_t>(num_tokens) + block_size - 1) / block_size;
    if (n > max_blocks) return PKV_ERR_INVALID_ARG;
    const int st = pkv_pool_share(pool, static_cast<int>(n), src_row);
    if (st != PKV_OK) return st;
    for (int64_t i = 0; i < n; ++i) dst_row[i] = src_row[i];
    return PKV_OK;
}

PKV_API int pkv_pool_prepare_append(pkv_pool *pool, int32_t *table_row, int max_blocks, int cur_tokens,
                                    int block_size, int32_t *copy_src, int32_t *copy_dst, int *n_copies) {
    if (!pool || !table_row || max_blocks <= 0 || block_size <= 0 || cur_tokens < 0 || !copy_src || !copy_dst ||
        !n_copies)
        return PKV_ERR_INVALID_ARG;
    *n_copies = 0;
    const int64_t blk = cur_tokens / block_size;
    if (blk >= max_blocks) return PKV_ERR_INVALID_ARG;
    if (cur_tokens % block_size == 0) return pkv_pool_alloc(pool, 1, table_row + blk);  // a fresh block
    const int32_t old = table_row[blk];
    const int64_t nb = static_cast<int64_t>(pool->refcount.size());
    if (old < 0 || old >= nb || pool->refcount[old] <= 0) return PKV_ERR_INVALID_ARG;
    if (pool->refcount[old] == 1) return PKV_OK;  // private: append in place
    int32_t fresh = -1;
    const int st = pkv_pool_alloc(pool, 1, &fresh);
    if (st != PKV_OK) return st;
    --pool->refcount[old];  // still >= 1: the other requests keep it
    table_row[blk] = fresh;
    *copy_src = old;
    *copy_dst = fresh;
    *n_copies = 1;
    return PKV_OK;
}

PKV_API int pkv_pool_free_table(pkv_pool *pool, const int32_t *table_row, int num_tokens, int block_size) {
    if (!pool || !table_row || num_tokens < 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
    const int64_t n = (static_cast<int64_t>(num_tokens) + block_size - 1) / block_size;
    if (n > 0x7fffffff) return PKV_ERR_INVALID_ARG;
    return pkv_pool_free(pool, static_cast<int>(n), table_row);
}

PKV_API int pkv_pool_swap(pkv_pool *from, pkv_pool *to, int32_t *table_row, int max_blocks, int num_tokens,
                          int block_size, int32_t *src_ids, int32_t *dst_ids) {
    if (!from || !to || from == to || !table_row || max_blocks <= 0 || num_tokens < 0 || block_size <= 0)
        return PKV_ERR_INVALID_ARG;
    const int64_t n = (static_cast<int64_t>(num_tokens) + block_size - 1) / block_size;
    if (n > max_blocks) return PKV_ERR_INVALID_ARG;
    if (n == 0) return PKV_OK;
    if (!src_ids || !dst_ids) return PKV_ERR_INVALID_ARG;
    const int64_t nb = static_cast<int64_t>(from->refcount.size());
    std::unordered_map<int32_t, int> seen;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t id = table_row[i];
        if (id < 0 || id >= nb || from->refcount[id] != 1 || ++seen[id] > 1) return PKV_ERR_INVALID_ARG;
    }
    const int st = pkv_pool_alloc(to, static_cast<int>(n), dst_ids);
    if (st != PKV_OK) return st;
    for (int64_t i = 0; i < n; ++i) {
        src_ids[i] = table_row[i];
        from->refcount[table_row[i]] = 0;
        from->free_list.push_back(table_row[i]);
        table_row[i] = dst_ids[i];
    }
    return PKV_OK;
}

PKV_API int pkv_slot_mapping(int64_t *slots, const int32_t *block_tables, const int32_t *positions, int num_seqs,
                             int max_blocks_per_seq, int block_size) {
    if (!slots || !block_tables || !positions || num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0)
        return PKV_ERR_INVALID_ARG;
    for (int b = 0; b < num_seqs; ++b) {
        const int pos = positions[b];
        if (pos < 0) continue;
        if (pos / block_size >= max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
        if (block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + pos / block_size] < 0)
            return PKV_ERR_INVALID_ARG;
    }
    for (int b = 0; b < num_seqs; ++b) {
        const int pos = positions[b];
        if (pos < 0) {
            slots[b] = -1;
            continue;
        }
        const int64_t block = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + pos / block_size];
        slots[b] = block * block_size + pos % block_size;
    }
    return PKV_OK;
}

PKV_API int pkv_get_device_error(pkv_stream_t stream, int *code) {
    if (!code) return PKV_ERR_INVALID_ARG;
    *code = PKV_DEV_OK;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
    int a = 0, d = 0, p = 0;
    int st = pkv_internal::append_take_error(&a);
    if (st != PKV_OK) return st;
    st = pkv_internal::decode_take_error(&d);
    if (st != PKV_OK) return st;
    st = pkv_internal::prefix_take_error(&p);
    if (st != PKV_OK) return st;
    *code = a ? a : (d ? d : p);
    return PKV_OK;
}

}  // extern "C"
