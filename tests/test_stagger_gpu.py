"""The automatic split with partitions of alternating length.

When every request can span at least 8 partitions and the grid fills at least three waves of
resident CTAs, odd partitions start a quarter partition early (lengths P - P/4 and P + P/4 alternate
and the last one ends at the context), so the CTAs of one wave do not all end together.  Results
must still equal the oracle: the ragged batch below puts contexts on both sides of every such
boundary (on GB300's 152 SMs its 2,048 CTAs are 4.5 waves), and the long-context workload runs in
the benchmark's launch configuration (512-token partitions, fused append)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, host_inputs, max_err, oracle_step

pytestmark = pytest.mark.gpu

P = pkv.PKV_DEFAULT_PARTITION
EDGES = [0, 1, 16, 17, 767, 768, 769, 1023, 1024, 1025, 1791, 1792, 1793, 2047, 2048, 2049, 2815, 2816, 2817,
         3071, 3072, 3073, 3839, 3840, 3841, 4095, 4096, 4097, 5000, 6143, 6144, 6145, 7167, 7168, 7169, 8191, 8192]


def ragged_contexts(seed):
    rng = np.random.default_rng(seed)
    ctxs = EDGES + rng.integers(1, 8 * P + 1, 64 - len(EDGES)).tolist()
    return [int(c) for c in rng.permutation(ctxs)]


def test_staggered_ragged_decode():
    ctxs = ragged_contexts(5)
    case = workloads.random_case(1300, ctxs, 16, 4, block_size=16, extra_blocks=5)
    assert case.max_blocks_per_seq * 16 == 8 * P                      # 8 partitions per request
    h = host_inputs(case)
    ref = oracle.decode(h["q"], h["k_cache"], h["v_cache"], h["block_tables"], h["context_lens"], case.scale)
    dev = case.to("cuda")
    out = torch.full_like(dev.q, float("nan"))
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * 16, "cuda")
    pkv.decode_attention(out, dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens, case.scale,
                         workspace=ws)
    assert max_err(out, ref) <= ATTN_TOL
    # the explicit uniform partitions and their merge give the same attention
    parts = torch.empty((case.num_seqs, case.num_q_heads, 8, 128), dtype=torch.float32, device="cuda")
    m = torch.empty((case.num_seqs, case.num_q_heads, 8), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    pkv.decode_partition(parts, m, l, dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                         case.scale, P)
    uni = torch.empty_like(out)
    pkv.merge(uni, parts, m, l, dev.context_lens, P)
    assert (out.float() - uni.float()).abs().max().item() <= 2 * ATTN_TOL
    assert_no_device_error()


def test_staggered_ragged_step():
    ctxs = [max(c, 1) for c in ragged_contexts(6)]
    case = workloads.random_case(1310, ctxs, 16, 4, block_size=16, extra_blocks=5)
    h = host_inputs(case)
    ref = oracle_step(h, case)
    dev = case.to("cuda")
    out = torch.empty_like(dev.q)
    ws = pkv.make_step_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * 16, 0, "cuda")
    pkv.decode_step(out, dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                    case.scale, 0, ws, overlap=True)
    assert max_err(out, ref) <= ATTN_TOL
    assert np.array_equal(dev.k_cache.cpu().numpy().view(np.uint16), h["k_cache"].view(np.uint16))
    assert np.array_equal(dev.v_cache.cpu().numpy().view(np.uint16), h["v_cache"].view(np.uint16))
    assert_no_device_error()


@pytest.mark.parametrize("bs", [16, 128])
def test_long_context_step_in_the_bench_configuration(bs):
    """32k-token contexts, 512-token partitions, the new token appended by the decode kernel:
    every request and head against the oracle, the appended rows bit-exact."""
    case = workloads.long_context(0, bs, device="cuda")
    h = host_inputs(case)
    ref = oracle_step(h, case)
    out = torch.empty_like(case.q)
    ws = pkv.make_step_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * bs, 0, "cuda",
                                 partition_size=512)
    pkv.decode_step(out, case.q, case.k_new, case.v_new, case.k_cache, case.v_cache, case.block_tables,
                    case.context_lens, case.scale, 0, ws, partition_size=512, overlap=True)
    assert max_err(out, ref) <= ATTN_TOL
    slots = oracle.slot_mapping(h["block_tables"], h["positions"], bs)
    blk, off = slots // bs, slots % bs
    got = case.k_cache[torch.from_numpy(blk).cuda(), :, torch.from_numpy(off).cuda()].cpu().numpy()
    assert np.array_equal(got.view(np.uint16), h["k_cache"][blk, :, off].view(np.uint16))
    assert_no_device_error()
    del case
    torch.cuda.empty_cache()
