"""A bounded device wait that runs out.

Every mbarrier wait in the decode kernel gives up after a time limit, records
PKV_DEV_WAIT_TIMEOUT in the device error word, lets the warp's other copies in flight land
(bounded waits again) and finishes the CTA, so the context stays usable.  To drive that path
without a fault, a separate build of the library (compiled with PKV_WAIT_TEST=1 into
libpkv_waittest.so beside the product library, loaded only here) arms the first copy stage of
warp 0 of the grid's first CTA for its bytes but issues no copy for it, and shortens the limit to
1 ms.  Nothing is in flight for that stage, so the wait can only run out; every copy that is
issued is an ordinary in-bounds one.

Checked: the error word says PKV_DEV_WAIT_TIMEOUT; every output row outside the sabotaged
(request 0, kv head 0) group still matches the float64 oracle; the split's completion counters
are back at zero; and the product library's next call, on a fresh workspace, matches the oracle
with a clean error word.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, host_inputs, max_err
from paged_kv_cache_278_gb300 import _lib
from paged_kv_cache_278_gb300.build import PKG_DIR, build

pytestmark = pytest.mark.gpu

TEST_LIB = os.path.join(PKG_DIR, "libpkv_waittest.so")


@pytest.fixture(scope="module")
def waittest_lib():
    build(extra_flags=["-DPKV_WAIT_TEST=1"], lib_path=TEST_LIB)
    return _lib.load(TEST_LIB)


def _device_error(lib):
    code = ctypes.c_int(-1)
    assert lib.pkv_get_device_error(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                    ctypes.byref(code)) == _lib.PKV_OK
    return code.value


def _decode(lib, out, c, ws):
    return lib.pkv_decode_attention(
        out.data_ptr(), c.q.data_ptr(), c.k_cache.data_ptr(), c.v_cache.data_ptr(), c.block_tables.data_ptr(),
        c.context_lens.data_ptr(), c.num_seqs, c.max_blocks_per_seq, c.num_q_heads, c.num_kv_heads, c.head_dim,
        c.block_size, c.num_blocks, ctypes.c_float(c.scale), ws.data_ptr(), ws.numel(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_wait_runs_out_is_recorded_and_context_stays_usable(waittest_lib):
    # GQA-4, contexts that need the split (so the fused merge and its counters are involved)
    host_case = workloads.random_case(951, [3000, 40, 1500, 2100], 32, 8, block_size=16)
    h = host_inputs(host_case)
    expect = oracle.decode(h["q"], h["k_cache"], h["v_cache"], h["block_tables"], h["context_lens"],
                           host_case.scale)
    c = host_case.to("cuda")
    g = c.num_q_heads // c.num_kv_heads
    pkv.device_error()  # clear the product library's word
    _device_error(waittest_lib)  # and the test build's

    ws = pkv.make_workspace(c.num_seqs, c.num_q_heads, c.max_blocks_per_seq * c.block_size, "cuda")
    out = torch.full_like(c.q, float("nan"))
    assert _decode(waittest_lib, out, c, ws) == _lib.PKV_OK
    torch.cuda.synchronize()
    assert _device_error(waittest_lib) == _lib.PKV_DEV_WAIT_TIMEOUT

    # every row outside (request 0, kv head 0) is untouched by the abort
    got = out.float().cpu().numpy().astype(np.float64)
    mask = np.ones(got.shape[:2], dtype=bool)
    mask[0, :g] = False
    assert np.isfinite(got).all()
    assert float(np.abs(got[mask] - expect[mask]).max()) <= ATTN_TOL

    # the aborted CTA still took part in the completion counters: all back at zero
    rows = c.num_seqs * c.num_q_heads * (-(-c.max_blocks_per_seq * c.block_size // pkv.PKV_DEFAULT_PARTITION))
    up = lambda x: x + (-x) % 256
    off = up(rows * 128 * 4) + 2 * up(rows * 4)
    counters = ws[off:off + c.num_seqs * c.num_q_heads * 4].view(torch.int32)
    assert int(counters.abs().sum().item()) == 0

    # the product library on the same context, fresh workspace: correct and clean
    out2 = torch.empty_like(c.q)
    pkv.decode_attention(out2, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale,
                         workspace=pkv.make_workspace(c.num_seqs, c.num_q_heads,
                                                      c.max_blocks_per_seq * c.block_size, "cuda"))
    torch.cuda.synchronize()
    assert max_err(out2, expect) <= ATTN_TOL
    assert pkv.device_error() == pkv.PKV_DEV_OK
