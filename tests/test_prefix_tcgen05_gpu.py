"""The 5th-generation tensor-core form of the shared-prefix tile, against the float64 oracle.

The shared prefix's chunk is the one dense contraction on the path (128 query rows x 128 tokens x
128 dims per CTA).  Its tcgen05 form -- Q through a 3-D tensor map, K and V by 2-D tensor copies,
S = Q K^T and O = P V accumulated in tensor memory with V as an MN-major operand, the rows' softmax
read back with tcgen05.ld -- is built with PKV_PREFIX_TCGEN05=1 (and the merge fused into the
suffix pass) into libpkv_tc5.so beside the product library.  The product default is the mma.sync
tile, measured faster on the shared-prefix step; the variant library keeps the tcgen05 form checked on the
same cases as the default one.
"""
import os

import pytest
import torch

import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error
from paged_kv_cache_278_gb300 import _lib
from paged_kv_cache_278_gb300.build import PKG_DIR, build
from test_shared_prefix_gpu import run, run_no_append, with_prefix

pytestmark = pytest.mark.gpu

TC5_LIB = os.path.join(PKG_DIR, "libpkv_tc5.so")


@pytest.fixture(scope="module", autouse=True)
def tcgen05_library():
    build(extra_flags=["-DPKV_PREFIX_TCGEN05=1", "-DPKV_PREFIX_SEPARATE_MERGE=0"], lib_path=TC5_LIB)
    mp = pytest.MonkeyPatch()
    mp.setattr(pkv, "_L", lambda: _lib.load(TC5_LIB))
    yield
    mp.undo()


def test_full_size_workload_layer_0():
    case = workloads.shared_prefix(0, device="cuda")
    err, *_ = run(case, 1024)
    assert err <= ATTN_TOL, err
    assert_no_device_error()


@pytest.mark.parametrize("group,hkv", [(1, 4), (4, 2), (8, 1)])
@pytest.mark.parametrize("prefix_len,bs", [(16, 16), (80, 16), (1024, 16), (256, 128)])
def test_ragged_prefixes(group, hkv, prefix_len, bs):
    case = with_prefix(300 + prefix_len + group, prefix_len, [1, 17, 511, 513, 1300], group * hkv, hkv, bs=bs)
    err, *_ = run(case, prefix_len)
    assert err <= ATTN_TOL, err
    assert_no_device_error()


def test_rows_span_two_row_tiles_with_prefix_only_requests():
    suffixes = [0 if i % 2 == 0 else 100 + 37 * i % 900 for i in range(160)]
    case = with_prefix(310, 256, suffixes, 4, 4)
    err, outs = run_no_append(case, 256)
    assert err <= ATTN_TOL, err
    assert torch.equal(outs[0], outs[1])
    assert_no_device_error()
