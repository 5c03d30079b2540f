"""The allocation-free decode entry point, called through the C ABI.

pkv_decode_attention_noalloc serves callers that cannot allocate device memory: plugins whose
host runtime owns all device memory and passes them only input and output pointers, and serving
loops that ban allocator calls (and the device synchronisation cudaMalloc implies) once they are
running.  It keeps the split partials in the library's own static device array instead of a
caller workspace.

Its output must match the float64 oracle and the workspace entry point's (pkv_decode_attention)
within the attention tolerance every other GPU test uses, on two calls in a row with different
inputs and shapes (the array keeps the previous call's contents; the first call's split fills
most of the array), and an oversize request must be refused before launch.  This file is
collected last, so a stop-at-first-failure run has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import host_inputs, max_err
from paged_kv_cache_278_gb300 import _lib

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3


def _noalloc(lib, out, c, max_blocks=None):
    s = torch.cuda.current_stream()
    return lib.pkv_decode_attention_noalloc(
        out.data_ptr(), c.q.data_ptr(), c.k_cache.data_ptr(), c.v_cache.data_ptr(), c.block_tables.data_ptr(),
        c.context_lens.data_ptr(), c.num_seqs, c.max_blocks_per_seq if max_blocks is None else max_blocks,
        c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size, c.num_blocks, ctypes.c_float(c.scale),
        ctypes.c_void_p(s.cuda_stream))


def _with_workspace(c):
    out = torch.empty_like(c.q)
    ws = pkv.make_workspace(c.num_seqs, c.num_q_heads, c.max_blocks_per_seq * c.block_size, c.q.device)
    pkv.decode_attention(out, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, workspace=ws)
    return out


def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls():
    lib = _lib.load()
    cases = [
        # ragged GQA-4 batch whose split needs 8 x 32 x 118 partial rows: 15.7 MB of the 16 MiB array
        workloads.random_case(901, [120000, 1, 0, 700, 2049, 513, 3000, 40], 32, 8, block_size=16),
        # a different shape on the second call: MHA, block 64, long contexts
        workloads.random_case(902, [3000, 6100, 40], 16, 16, block_size=64),
    ]
    need = pkv.decode_workspace_size(8, 32, cases[0].max_blocks_per_seq * 16)
    assert 0.9 * _lib.PKV_NOALLOC_SCRATCH_BYTES < need <= _lib.PKV_NOALLOC_SCRATCH_BYTES
    for host_case in cases:
        h = host_inputs(host_case)
        expect = oracle.decode(h["q"], h["k_cache"], h["v_cache"], h["block_tables"], h["context_lens"],
                               host_case.scale)
        c = host_case.to("cuda")
        ref = _with_workspace(c)
        out = torch.full_like(c.q, float("nan"))
        assert _noalloc(lib, out, c) == _lib.PKV_OK
        torch.cuda.synchronize()
        assert max_err(out, expect) <= ATTN_TOL
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= ATTN_TOL, err
    assert pkv.device_error() == pkv.PKV_DEV_OK


def test_noalloc_refuses_requests_beyond_its_scratch():
    lib = _lib.load()
    # 16 requests x 32 heads x 64 default partitions need more than 16 MiB of partials.
    # Every buffer is allocated at the size the call names (contexts are 0), so nothing could
    # be read out of bounds even if the call were not refused.
    b, hq, hkv = 16, 32, 32
    maxb = 64 * pkv.PKV_DEFAULT_PARTITION // 16
    assert pkv.decode_workspace_size(b, hq, maxb * 16) > _lib.PKV_NOALLOC_SCRATCH_BYTES
    c = workloads.random_case(903, [0] * b, hq, hkv, block_size=16, extra_blocks=4).to("cuda")
    c.block_tables = torch.zeros((b, maxb), dtype=torch.int32, device="cuda")
    out = torch.zeros_like(c.q)
    assert _noalloc(lib, out, c, max_blocks=maxb) == _lib.PKV_ERR_WORKSPACE


def test_noalloc_captured_in_a_graph_and_replayed():
    """The use the entry exists for: after one eager call (the address look-up), the call is
    captured into a CUDA graph in global capture mode and replayed with new queries written into
    the captured input buffer.  Each replay must clear the counters again (the captured memset)
    and equal the workspace entry point's output on the same inputs."""
    lib = _lib.load()
    c = workloads.random_case(904, [5000, 1, 2049, 0, 700, 1025], 32, 8, block_size=16).to("cuda")
    out = torch.zeros_like(c.q)
    assert _noalloc(lib, out, c) == _lib.PKV_OK        # eager: caches the scratch address
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream, capture_error_mode="global"):
            assert _noalloc(lib, out, c) == _lib.PKV_OK
    gen = torch.Generator(device="cuda").manual_seed(905)
    for _ in range(2):
        c.q.copy_(torch.randn(c.q.shape, generator=gen, device="cuda").half())
        out.fill_(float("nan"))
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        ref = _with_workspace(c)
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= ATTN_TOL, err
    assert pkv.device_error() == pkv.PKV_DEV_OK
