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
