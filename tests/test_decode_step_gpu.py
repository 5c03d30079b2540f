"""pkv_decode_step (append fused into the decode kernel) against the oracle's append + decode,
and bit-for-bit against the two-call path (pkv_append + pkv_decode_attention)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, gpu_step, host_inputs, max_err, oracle_step
from test_shared_prefix_gpu import with_prefix

pytestmark = pytest.mark.gpu


def step(case, prefix_len=0):
    ws = pkv.make_step_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * case.block_size,
                                 prefix_len, "cuda")
    out = torch.empty_like(case.q)
    pkv.decode_step(out, case.q, case.k_new, case.v_new, case.k_cache, case.v_cache, case.block_tables,
                    case.context_lens, case.scale, prefix_len, ws)
    return out


def check_pool(dev, h):
    assert np.array_equal(dev.k_cache.cpu().numpy().view(np.uint16), h["k_cache"].view(np.uint16))
    assert np.array_equal(dev.v_cache.cpu().numpy().view(np.uint16), h["v_cache"].view(np.uint16))


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 64])
def test_decode_step_matches_oracle_and_two_call_path(group, bs):
    ctxs = [0, 1, 15, 16, 17, 511, 512, 513, 1537, 2100]
    case = workloads.random_case(300 + group + bs, ctxs, 2 * group, 2, block_size=bs, extra_blocks=4)
    h = host_inputs(case)
    ref = oracle_step(h, case)
    dev = case.to("cuda")
    out = step(dev)
    assert max_err(out, ref) <= ATTN_TOL
    check_pool(dev, h)                       # the append is bit-exact over the whole pool
    two = gpu_step(case.to("cuda"))          # pkv_append + pkv_decode_attention
    assert torch.equal(out, two)
    assert_no_device_error()


def test_decode_step_single_pass_tables():
    case = workloads.random_case(7, [1, 100, 512, 0], 8, 8, block_size=16)
    h = host_inputs(case)
    ref = oracle_step(h, case)
    dev = case.to("cuda")
    out = step(dev)
    assert max_err(out, ref) <= ATTN_TOL
    check_pool(dev, h)
    assert_no_device_error()


@pytest.mark.parametrize("prefix_len", [64, 1024])
def test_decode_step_with_shared_prefix(prefix_len):
    case = with_prefix(400 + prefix_len, prefix_len, [1, 40, 700, 129], 32, 8)
    h = host_inputs(case)
    ref = oracle_step(h, case)
    dev = case.to("cuda")
    out = step(dev, prefix_len)
    assert max_err(out, ref) <= ATTN_TOL
    check_pool(dev, h)
    assert_no_device_error()


def test_decode_step_full_size_mha7b():
    case = workloads.mha7b(5, device="cuda")
    h = host_inputs(case)
    ref = oracle_step(h, case)
    out = step(case)
    assert max_err(out, ref) <= ATTN_TOL
    assert_no_device_error()
