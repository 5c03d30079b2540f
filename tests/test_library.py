"""libpkv.so on the CPU: it loads, exports every symbol include/pkv.h declares, rejects bad
arguments before touching the GPU, and its host block pool / slot mapping behave (no kernels run)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
from paged_kv_cache_278_gb300 import _lib
from paged_kv_cache_278_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_symbols():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h), encoding="utf-8").read()
            names += re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES), "the binding's signature table must match the header"


def declared_prototypes():
    """{name: [parameter type text, ...]} of every PKV_API function in include/."""
    protos = {}
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        for m in re.finditer(r"PKV_API\s+([\w\s\*]+?)\b(pkv_\w+)\s*\(([^)]*)\)", text):
            params = [x.strip() for x in m.group(3).split(",")]
            protos[m.group(2)] = [] if params == ["void"] or params == [""] else params
    return protos


def _ctype_for(param: str):
    """The ctypes type a C parameter declaration must be bound with."""
    decl = " ".join(param.replace("*", " * ").split())
    if "*" in decl:
        return "pointer"
    base = decl.rsplit(" ", 1)[0].replace("const ", "")
    return {"int": ctypes.c_int, "int32_t": ctypes.c_int32, "uint32_t": ctypes.c_uint32, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t, "float": ctypes.c_float,
            "uint64_t": ctypes.c_uint64, "unsigned": ctypes.c_uint, "pkv_stream_t": "pointer"}[base]


def test_binding_signatures_match_the_header(lib):
    """Argument count and kind of every ctypes binding against its C prototype, so a slip in the
    table cannot shift arguments into the wrong parameters."""
    protos = declared_prototypes()
    assert set(protos) == set(_lib.SIGNATURES)
    pointer_types = (ctypes.c_void_p, ctypes.c_char_p)
    for name, params in protos.items():
        bound = _lib.SIGNATURES[name][1]
        assert len(bound) == len(params), (name, len(bound), len(params))
        for decl, ct in zip(params, bound):
            want = _ctype_for(decl)
            if want == "pointer":
                assert ct in pointer_types or issubclass(ct, ctypes._Pointer), (name, decl, ct)
            else:
                assert ct is want, (name, decl, ct)


def test_only_api_symbols_are_visible(lib):
    # the C ABI is the only surface: hidden visibility keeps kernels and helpers private
    out = os.popen(f"nm -D --defined-only {_lib.LIB_PATH}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {n for n in exported if n.startswith("pkv_")} == set(declared_symbols())


def test_status_strings(lib):
    for code in range(0, -7, -1):
        assert isinstance(_lib.status_string(code), str)
    assert _lib.status_string(-6) == "device-side index check failed"
    assert _lib.status_string(123) == "unknown status"
    assert lib.pkv_version() >= 10000


def test_invalid_arguments_rejected_without_launch(lib):
    null = None
    p = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    # null pointers
    assert lib.pkv_append(null, p, p, p, p, 1, 1, 128, 16, 4, null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_attention(null, p, p, p, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                    null) == _lib.PKV_ERR_INVALID_ARG
    # head_dim other than 128, block size not a multiple of 16, group size 3
    assert lib.pkv_decode_attention(p, p, p, p, p, p, 1, 1, 1, 1, 64, 16, 4, 1.0, null, 0,
                                    null) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_decode_attention(p, p, p, p, p, p, 1, 1, 1, 1, 128, 8, 4, 1.0, null, 0,
                                    null) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_decode_attention(p, p, p, p, p, p, 1, 1, 3, 1, 128, 16, 4, 1.0, null, 0,
                                    null) == _lib.PKV_ERR_UNSUPPORTED
    # q heads not a multiple of kv heads
    assert lib.pkv_decode_attention(p, p, p, p, p, p, 1, 1, 6, 4, 128, 16, 4, 1.0, null, 0,
                                    null) == _lib.PKV_ERR_INVALID_ARG
    # misaligned cache pointer
    bad = ctypes.c_void_p(24)
    assert lib.pkv_decode_attention(p, p, bad, p, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                    null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_append(bad, p, p, p, p, 1, 1, 128, 16, 4, null) == _lib.PKV_ERR_INVALID_ARG
    # split needed (4096-token tables) but no workspace
    assert lib.pkv_decode_attention(p, p, p, p, p, p, 1, 256, 1, 1, 128, 16, 4096, 1.0, null, 0,
                                    null) == _lib.PKV_ERR_WORKSPACE
    # partition size not a multiple of 16; too few partitions for the table
    assert lib.pkv_decode_partition(p, p, p, p, p, p, p, p, 1, 4, 1, 1, 128, 16, 4, 1.0, 40, 2,
                                    null) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_decode_partition(p, p, p, p, p, p, p, p, 1, 64, 1, 1, 128, 16, 64, 1.0, 64, 2,
                                    null) == _lib.PKV_ERR_INVALID_ARG
    # empty batches are a successful no-op
    assert lib.pkv_append(p, p, p, p, p, 0, 1, 128, 16, 4, null) == _lib.PKV_OK


def test_int8k_multi_copy_invalid_arguments(lib):
    null = None
    p = ctypes.c_void_p(16)
    bad = ctypes.c_void_p(24)
    # int8-key append / decode / step: null scale array, misaligned scales, head_dim 64
    assert lib.pkv_append_int8k(p, null, p, p, p, p, 1, 1, 128, 16, 4, null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_append_int8k(p, p, p, p, p, p, 1, 1, 64, 16, 4, null) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_decode_attention_int8k(p, p, p, null, p, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                          null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_attention_int8k(p, p, p, bad, p, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                          null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_step_int8k(p, p, null, p, p, p, p, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0, 0,
                                     null) == _lib.PKV_ERR_INVALID_ARG
    # int8 keys and values: null value scales, misaligned value scales, null value codes, head_dim 64
    assert lib.pkv_append_int8kv(p, p, p, null, p, p, p, 1, 1, 128, 16, 4, null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_append_int8kv(p, p, p, p, p, p, p, 1, 1, 64, 16, 4, null) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_decode_attention_int8kv(p, p, p, p, p, null, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                           null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_attention_int8kv(p, p, p, p, p, bad, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                           null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_attention_int8kv(p, p, p, p, null, p, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                           null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_step_int8kv(p, p, p, p, p, p, p, null, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0, 0,
                                      null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_append_int8kv(p, p, p, p, null, null, null, 0, 1, 128, 16, 4, null) == _lib.PKV_OK
    # fp8 keys and values: the same argument rules
    assert lib.pkv_append_fp8kv(p, p, p, null, p, p, p, 1, 1, 128, 16, 4, null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_append_fp8kv(p, p, p, p, p, p, p, 1, 1, 64, 16, 4, null) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_decode_attention_fp8kv(p, p, p, p, p, null, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                          null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_attention_fp8kv(p, p, p, p, p, bad, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                          null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_attention_fp8kv(p, p, p, null, p, p, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                          null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_step_fp8kv(p, p, p, p, p, p, p, null, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, null, 0, 0,
                                     null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_step_fp8kv(p, p, p, p, p, p, p, p, p, p, 0, 1, 1, 1, 128, 16, 4, 1.0, null, 0, 8,
                                     null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_append_fp8kv(p, p, p, p, null, null, null, 0, 1, 128, 16, 4, null) == _lib.PKV_OK
    # several tokens per request: null query_start, query length beyond the limit, no workspace
    assert lib.pkv_decode_attention_multi(p, p, p, p, p, p, null, 1, 4, 4, 1, 1, 1, 128, 16, 4, 1.0, null, 0,
                                          null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_attention_multi(p, p, p, p, p, p, p, 1, 4, _lib.PKV_MAX_QUERY_LEN + 1, 1, 1, 1, 128, 16,
                                          4, 1.0, null, 0, null) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_decode_attention_multi(p, p, p, p, p, p, p, 1, 4, 4, 256, 1, 1, 128, 16, 4096, 1.0, null, 0,
                                          null) == _lib.PKV_ERR_WORKSPACE
    # block copy: null id arrays, head_dim not a multiple of 8
    assert lib.pkv_copy_blocks(p, p, null, p, 1, 1, 128, 16, 4, null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(p, p, p, p, 1, 1, 12, 16, 4, null) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_copy_blocks(p, p, null, null, 0, 1, 128, 16, 4, null) == _lib.PKV_OK


def test_noalloc_validates_before_any_cuda_call(lib):
    """The allocation-free entry refuses bad or oversize requests before its first CUDA call (on
    this GPU-less machine any CUDA call would fail with CUDA, so each status below also shows
    that none was made)."""
    null = None
    p = ctypes.c_void_p(16)
    call = lambda maxb, bs, hq=1, hkv=1, b=1, hd=128, out=p: lib.pkv_decode_attention_noalloc(
        out, p, p, p, p, p, b, maxb, hq, hkv, hd, bs, 4, 1.0, null)
    # table capacity max_blocks_per_seq * block_size beyond 2^31 - 1 tokens
    assert call(2 ** 31 // 16, 16) == _lib.PKV_ERR_INVALID_ARG
    assert call(2 ** 30, 256) == _lib.PKV_ERR_INVALID_ARG
    # valid shape whose split needs more than the static scratch: 16 x 32 heads x 64 partitions
    assert lib.pkv_decode_workspace_size(16, 32, 128, 64 * 1024, 1024) > _lib.PKV_NOALLOC_SCRATCH_BYTES
    assert call(64 * 1024 // 16, 16, hq=32, hkv=32, b=16) == _lib.PKV_ERR_WORKSPACE
    # the other argument rules of pkv_decode_attention
    assert call(4, 16, out=null) == _lib.PKV_ERR_INVALID_ARG
    assert call(4, 16, out=ctypes.c_void_p(20)) == _lib.PKV_ERR_INVALID_ARG
    assert call(4, 16, hd=64) == _lib.PKV_ERR_UNSUPPORTED
    assert call(4, 16, hq=6, hkv=4) == _lib.PKV_ERR_INVALID_ARG
    assert call(4, 16, b=0) == _lib.PKV_OK


def test_step_partition_arguments(lib):
    null = None
    p = ctypes.c_void_p(16)
    args = lambda part, flags=0: (p, p, p, p, p, p, p, p, 1, 1, 1, 1, 128, 16, 4, 1.0, part, null, 0, flags, null)
    assert lib.pkv_decode_step_partition(*args(-16)) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_step_partition(*args(24)) == _lib.PKV_ERR_UNSUPPORTED       # not a multiple of 16
    assert lib.pkv_decode_step_partition(*args(_lib.PKV_MAX_PARTITION + 16)) == _lib.PKV_ERR_UNSUPPORTED
    no_new = (p, p, null, p) + args(512)[4:]
    assert lib.pkv_decode_step_partition(*no_new) == _lib.PKV_ERR_INVALID_ARG
    # flags: bits other than PKV_STEP_OVERLAP are refused before any CUDA call
    assert lib.pkv_decode_step_partition(*args(512, 2)) == _lib.PKV_ERR_INVALID_ARG


def test_step_flags(lib):
    null = None
    p = ctypes.c_void_p(16)
    step = lambda flags, prefix=0, b=1: lib.pkv_decode_step(p, p, p, p, p, p, p, p, b, 4, 1, 1, 128, 16, 4, 1.0,
                                                            prefix, null, 0, flags, null)
    assert step(4) == _lib.PKV_ERR_INVALID_ARG
    assert step(0x80000000) == _lib.PKV_ERR_INVALID_ARG
    assert step(4, prefix=16) == _lib.PKV_ERR_INVALID_ARG
    # a valid flag on an empty batch: nothing to launch
    assert step(_lib.PKV_STEP_OVERLAP, b=0) == _lib.PKV_OK
    assert step(0, b=0) == _lib.PKV_OK
    assert lib.pkv_decode_step_int8k(p, p, p, p, p, p, p, p, p, 0, 1, 1, 1, 128, 16, 4, 1.0, null, 0, 8,
                                     null) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_step_int8kv(p, p, p, p, p, p, p, p, p, p, 0, 1, 1, 1, 128, 16, 4, 1.0, null, 0, 8,
                                      null) == _lib.PKV_ERR_INVALID_ARG
    # several-token step: unknown flags, missing new rows, drafts longer than PKV_MAX_STEP_QUERY_LEN
    multi = lambda kn, maxq, flags, b=1: lib.pkv_decode_step_multi(p, p, kn, p, p, p, p, p, p, b, 4, maxq, 4, 1, 1,
                                                                   128, 16, 4, 1.0, null, 0, flags, null)
    assert multi(p, 4, 2) == _lib.PKV_ERR_INVALID_ARG
    assert multi(null, 4, 0) == _lib.PKV_ERR_INVALID_ARG
    assert multi(p, _lib.PKV_MAX_STEP_QUERY_LEN + 1, 0) == _lib.PKV_ERR_UNSUPPORTED
    assert multi(p, _lib.PKV_MAX_STEP_QUERY_LEN, _lib.PKV_STEP_OVERLAP, b=0) == _lib.PKV_OK


def test_multi_workspace_size(lib):
    # one default partition: none needed
    part = _lib.PKV_DEFAULT_PARTITION
    assert lib.pkv_decode_multi_workspace_size(2, 10, 8, 32, 8, 128, part) == 0
    rows = 10 * 32 * (8192 // part)
    up = lambda x: x + (-x) % 256
    groups = -(-8 * 4 // 16)  # more than 8 rows per kv head: 16-row groups
    expect = up(rows * 128 * 4) + 2 * up(rows * 4) + up(2 * 8 * groups * 4)
    assert lib.pkv_decode_multi_workspace_size(2, 10, 8, 32, 8, 128, 8192) == expect


def test_workspace_size(lib):
    assert lib.pkv_decode_workspace_size(4, 32, 128, 512, 512) == 0
    rows = 4 * 32 * 64
    up = lambda x: x + (-x) % 256
    expect = up(rows * 128 * 4) + 2 * up(rows * 4) + up(4 * 32 * 4)
    assert lib.pkv_decode_workspace_size(4, 32, 128, 32768, 512) == expect


# ------------------------------------------------------------------ host block pool

def test_pool_is_seeded_permutation(lib):
    a = pkv.BlockPool(1000, seed=7)
    ids = a.alloc(1000)
    assert sorted(ids) == list(range(1000))
    assert ids != list(range(1000)) and ids != list(range(999, -1, -1))
    b = pkv.BlockPool(1000, seed=7)
    assert b.alloc(1000) == ids
    c = pkv.BlockPool(1000, seed=8)
    assert c.alloc(1000) != ids
    assert a.num_free() == 0


def test_pool_alloc_is_all_or_nothing(lib):
    pool = pkv.BlockPool(10, seed=1)
    got = pool.alloc(7)
    with pytest.raises(pkv.PkvError) as e:
        pool.alloc(4)
    assert e.value.status == _lib.PKV_ERR_OUT_OF_BLOCKS
    assert pool.num_free() == 3
    pool.free(got)
    assert pool.num_free() == 10


def test_pool_refcounts_and_failure_path_release(lib):
    pool = pkv.BlockPool(64, seed=3)
    prefix = pool.alloc(4)
    pool.share(prefix)                       # a second request references the prefix
    assert all(pool.refcount(i) == 2 for i in prefix)
    mine = pool.alloc(2)
    pool.free(prefix + mine)                 # request 1 ends: prefix survives
    assert all(pool.refcount(i) == 1 for i in prefix) and all(pool.refcount(i) == 0 for i in mine)
    assert pool.num_free() == 64 - 4
    # double free is rejected and changes nothing
    with pytest.raises(pkv.PkvError):
        pool.free([prefix[0], prefix[0]])
    assert pool.refcount(prefix[0]) == 1
    with pytest.raises(pkv.PkvError):
        pool.share([mine[0]])                # sharing a free block
    with pytest.raises(pkv.PkvError):
        pool.free([64])
    pool.free(prefix)
    assert pool.num_free() == 64
    assert pool.refcount(-1) == -1


def test_pool_reserve_grows_tables(lib):
    pool = pkv.BlockPool(100, seed=5)
    row = torch.full((8,), -1, dtype=torch.int32)
    pool.reserve(row, 0, 33, 16)             # 3 blocks
    assert (row[:3] >= 0).all() and (row[3:] == -1).all()
    pool.reserve(row, 33, 48, 16)            # still 3 blocks
    assert (row[3:] == -1).all()
    pool.reserve(row, 48, 49, 16)            # crosses into block 4
    assert (row[:4] >= 0).all() and len(set(row[:4].tolist())) == 4
    with pytest.raises(pkv.PkvError):
        pool.reserve(row, 49, 8 * 16 + 1, 16)
    assert pool.num_free() == 96


def test_slot_mapping_matches_oracle(lib):
    rng = np.random.default_rng(0)
    for bs in (16, 32, 64, 128):
        b, maxb = 9, 12
        bt = rng.permutation(b * maxb).reshape(b, maxb).astype(np.int32)
        pos = rng.integers(-1, maxb * bs, size=b).astype(np.int32)
        got = pkv.slot_mapping(torch.from_numpy(bt), torch.from_numpy(pos), bs).numpy()
        ref = oracle.slot_mapping(bt, pos, bs)
        assert np.array_equal(got, ref)
    with pytest.raises(pkv.PkvError):        # position beyond the table
        pkv.slot_mapping(torch.zeros((1, 2), dtype=torch.int32), torch.tensor([32], dtype=torch.int32), 16)


def test_pool_fork_and_copy_on_write(lib):
    pool = pkv.BlockPool(20, seed=9)
    parent = torch.full((6,), -1, dtype=torch.int32)
    pool.reserve(parent, 0, 40, 16)                     # 3 blocks, the last one half full
    child = torch.full((6,), -1, dtype=torch.int32)
    pool.fork(parent, child, 40, 16)
    assert torch.equal(child[:3], parent[:3]) and (child[3:] == -1).all()
    assert all(pool.refcount(int(i)) == 2 for i in parent[:3])
    assert pool.num_free() == 17
    # the child writes position 40, inside the shared third block: copy on write
    shared = int(parent[2])
    pair = pool.prepare_append(child, 40, 16)
    assert pair is not None and pair[0] == shared and pair[1] == int(child[2]) and pair[1] != shared
    assert pool.refcount(shared) == 1 and pool.refcount(pair[1]) == 1
    assert torch.equal(child[:2], parent[:2])
    # the parent now owns its third block alone: it appends in place
    assert pool.prepare_append(parent, 40, 16) is None
    assert int(parent[2]) == shared
    # position 48 starts a fresh block for each
    assert pool.prepare_append(child, 48, 16) is None and int(child[3]) >= 0
    assert pool.num_free() == 15
    pool.free_table(child, 49, 16)                      # child ends: only its private blocks return
    assert pool.num_free() == 17
    assert all(pool.refcount(int(i)) == 1 for i in parent[:3])
    pool.free_table(parent, 41, 16)
    assert pool.num_free() == 20


def test_pool_copy_on_write_failure_changes_nothing(lib):
    pool = pkv.BlockPool(4, seed=2)
    a = torch.full((4,), -1, dtype=torch.int32)
    pool.reserve(a, 0, 64, 16)                          # the whole pool
    b = torch.full((4,), -1, dtype=torch.int32)
    pool.fork(a, b, 64, 16)
    before = b.clone()
    with pytest.raises(pkv.PkvError) as e:
        pool.prepare_append(b, 20, 16)                  # shared block, no free block to copy into
    assert e.value.status == _lib.PKV_ERR_OUT_OF_BLOCKS
    assert torch.equal(b, before) and all(pool.refcount(int(i)) == 2 for i in a)
    with pytest.raises(pkv.PkvError):
        pool.prepare_append(b, 64, 16)                  # beyond the table row
    with pytest.raises(pkv.PkvError):
        pool.fork(a, torch.full((2,), -1, dtype=torch.int32), 64, 16)   # row too short
    stale = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    pool.free_table(a, 64, 16)
    pool.free_table(b, 64, 16)
    with pytest.raises(pkv.PkvError):
        pool.prepare_append(stale, 5, 16)               # block not allocated
    assert pool.num_free() == 4


def test_copy_on_write_flow_against_the_oracle(lib):
    """Host pool + oracle copy and append: a forked request that diverges attends to its own
    tokens, and its parent's output does not move."""
    rng = np.random.default_rng(4)
    hkv, hq, d, bs, ctx = 2, 4, 128, 16, 37
    nb = 12
    kpool = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    vpool = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    pool = pkv.BlockPool(nb, seed=1)
    parent = torch.full((4,), -1, dtype=torch.int32)
    pool.reserve(parent, 0, ctx, bs)
    child = torch.full((4,), -1, dtype=torch.int32)
    pool.fork(parent, child, ctx, bs)
    q = np.repeat(rng.standard_normal((1, hq, d)).astype(np.float16), 2, axis=0)
    bt = torch.stack([parent, child]).numpy()
    before = oracle.decode(q, kpool, vpool, bt, np.array([ctx, ctx], np.int32), 0.1)
    assert np.array_equal(before[0], before[1])
    pair = pool.prepare_append(child, ctx, bs)
    assert pair is not None
    oracle.copy_blocks(kpool, vpool, [pair[0]], [pair[1]])
    k_new = rng.standard_normal((1, hkv, d)).astype(np.float16)
    v_new = rng.standard_normal((1, hkv, d)).astype(np.float16)
    slot = int(child[ctx // bs]) * bs + ctx % bs
    oracle.append(kpool, vpool, np.array([slot], np.int64), k_new, v_new)
    bt = torch.stack([parent, child]).numpy()
    after = oracle.decode(q, kpool, vpool, bt, np.array([ctx, ctx + 1], np.int32), 0.1)
    assert np.array_equal(after[0], before[0])
    assert not np.allclose(after[1], before[1])


def test_pool_swap_out_and_in(lib):
    dev_pool, host_pool = pkv.BlockPool(12, seed=1), pkv.BlockPool(6, seed=2)
    row = torch.full((5,), -1, dtype=torch.int32)
    dev_pool.reserve(row, 0, 50, 16)                        # 4 device blocks
    before = row.clone()
    src, dst = dev_pool.swap_to(host_pool, row, 50, 16)     # swap out
    assert torch.equal(src, before[:4]) and torch.equal(row[:4], dst) and row[4] == -1
    assert dev_pool.num_free() == 12 and host_pool.num_free() == 2
    assert all(host_pool.refcount(int(i)) == 1 for i in dst)
    back_src, back_dst = host_pool.swap_to(dev_pool, row, 50, 16)   # swap in (to fresh device blocks)
    assert torch.equal(back_src, dst) and torch.equal(row[:4], back_dst)
    assert dev_pool.num_free() == 8 and host_pool.num_free() == 6
    # shared blocks cannot leave; too little room changes nothing
    other = torch.full((5,), -1, dtype=torch.int32)
    dev_pool.fork(row, other, 50, 16)
    snap = row.clone()
    with pytest.raises(pkv.PkvError) as e:
        dev_pool.swap_to(host_pool, row, 50, 16)
    assert e.value.status == _lib.PKV_ERR_INVALID_ARG and torch.equal(row, snap)
    dev_pool.free_table(other, 50, 16)
    small = pkv.BlockPool(3, seed=3)
    with pytest.raises(pkv.PkvError) as e:
        dev_pool.swap_to(small, row, 50, 16)
    assert e.value.status == _lib.PKV_ERR_OUT_OF_BLOCKS and torch.equal(row, snap)
    assert small.num_free() == 3 and dev_pool.num_free() == 8
    assert lib.pkv_copy_blocks_between(None, None, 1, None, None, 1, None, None, 1, 1, 128, 16,
                                       None) == _lib.PKV_ERR_INVALID_ARG


def test_swap_round_trip_against_the_oracle(lib):
    """Host pool logic + oracle copies: a request swapped out to a host pool and back into other
    device blocks attends exactly as before."""
    rng = np.random.default_rng(9)
    hkv, hq, d, bs, ctx = 2, 4, 128, 16, 45
    kdev = rng.standard_normal((10, hkv, bs, d)).astype(np.float16)
    vdev = rng.standard_normal((10, hkv, bs, d)).astype(np.float16)
    khost = np.zeros((4, hkv, bs, d), np.float16)
    vhost = np.zeros_like(khost)
    dev_pool, host_pool = pkv.BlockPool(10, seed=4), pkv.BlockPool(4, seed=5)
    row = torch.full((3,), -1, dtype=torch.int32)
    dev_pool.reserve(row, 0, ctx, bs)
    q = rng.standard_normal((1, hq, d)).astype(np.float16)
    ctxs = np.array([ctx], np.int32)
    before = oracle.decode(q, kdev, vdev, row.numpy()[None], ctxs, 0.2)
    src, dst = dev_pool.swap_to(host_pool, row, ctx, bs)
    oracle.copy_blocks_between(khost, vhost, kdev, vdev, src.numpy(), dst.numpy())
    kdev[src.numpy()] = np.nan                                # the freed device blocks get reused
    vdev[src.numpy()] = np.nan
    dev_pool.alloc(dev_pool.num_free())                        # take every free block: swap-in must wait
    with pytest.raises(pkv.PkvError):
        host_pool.swap_to(dev_pool, row, ctx, bs)
    dev_pool.free(list(range(10)))
    src2, dst2 = host_pool.swap_to(dev_pool, row, ctx, bs)
    oracle.copy_blocks_between(kdev, vdev, khost, vhost, src2.numpy(), dst2.numpy())
    after = oracle.decode(q, kdev, vdev, row.numpy()[None], ctxs, 0.2)
    assert np.array_equal(before, after)
