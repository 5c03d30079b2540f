"""The one-grid form of the shared-prefix step (prefix tiles and suffix partitions as CTAs of one
launch, merged where their last piece lands), against the float64 oracle.

Built with PKV_PREFIX_ONE_GRID=1 into libpkv_onegrid.so beside the product library: the prefix
tiles run the 16-row tensor-core engine over eight TMA-staged 16-token tiles each and store their
rows' partials; a pair whose last piece is a prefix tile is merged by the merge launch after the
grid.  The product default is the three-launch cascade, measured faster; the variant library keeps the
one-grid form checked on the same cases.
"""
import os

import pytest
import torch

import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, host_inputs, max_err, oracle_step
from paged_kv_cache_278_gb300 import _lib
from paged_kv_cache_278_gb300.build import PKG_DIR, build
from test_shared_prefix_gpu import run, run_no_append, with_prefix

pytestmark = pytest.mark.gpu

ONE_GRID_LIB = os.path.join(PKG_DIR, "libpkv_onegrid.so")


@pytest.fixture(scope="module", autouse=True)
def one_grid_library():
    build(extra_flags=["-DPKV_PREFIX_ONE_GRID=1"], lib_path=ONE_GRID_LIB)
    mp = pytest.MonkeyPatch()
    mp.setattr(pkv, "_L", lambda: _lib.load(ONE_GRID_LIB))
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


def test_rows_span_row_tiles_with_prefix_only_requests():
    suffixes = [0 if i % 2 == 0 else 100 + 37 * i % 900 for i in range(40)]
    case = with_prefix(310, 256, suffixes, 4, 4)
    err, outs = run_no_append(case, 256)
    assert err <= ATTN_TOL, err
    assert torch.equal(outs[0], outs[1])
    assert_no_device_error()


def test_steps_with_overlap_reuse_the_workspace():
    """Four layers of one-launch steps with PKV_STEP_OVERLAP sharing one workspace (the counters a
    layer leaves complete are folded and cleared by its merge launch)."""
    cases = [with_prefix(320 + l, 256, [1, 40, 700, 129, 1000], 32, 8) for l in range(4)]
    refs = [oracle_step(host_inputs(c), c) for c in cases]
    devs = [c.to("cuda") for c in cases]
    c0 = cases[0]
    ws = pkv.make_step_workspace(c0.num_seqs, c0.num_q_heads, c0.max_blocks_per_seq * c0.block_size, 256, "cuda")
    outs = [torch.empty_like(d.q) for d in devs]
    for rep in range(2):
        for l, d in enumerate(devs):
            pkv.decode_step(outs[l], d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                            d.scale, 256, ws, overlap=True)
        torch.cuda.synchronize()
        for o, ref in zip(outs, refs):
            assert max_err(o, ref) <= ATTN_TOL
    assert_no_device_error()
