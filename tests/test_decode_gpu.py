"""Decode attention on the GPU against the float64 oracle, element by element, at sizes that
span several 16-token tiles, several split partitions and ragged tails."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, gpu_step, host_inputs, max_err, oracle_step

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 15, 16, 17, 100, 511, 512, 513, 1000, 1537, 2100]


def run_parity(case):
    h = host_inputs(case)
    ref = oracle_step(h, case)
    out = gpu_step(case.to("cuda"))
    err = max_err(out, ref)
    assert_no_device_error()
    return err, out, ref


def test_tiny_workload():
    case = workloads.tiny()
    err, _, _ = run_parity(case)
    assert err <= ATTN_TOL, err


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
def test_ragged_batch(group, bs):
    case = workloads.random_case(10 * group + bs, RAGGED, 2 * group, 2, block_size=bs, extra_blocks=4)
    err, _, _ = run_parity(case)
    assert err <= ATTN_TOL, (group, bs, err)


@pytest.mark.parametrize("group", [1, 4])
def test_single_pass_only(group):
    # every table fits one partition: no workspace, one kernel
    case = workloads.random_case(77 + group, [1, 7, 16, 33, 255, 256, 500], 4 * group, 4, block_size=16)
    assert case.max_blocks_per_seq * 16 <= pkv.PKV_DEFAULT_PARTITION
    h = host_inputs(case)
    ref = oracle_step(h, case)
    out = gpu_step(case.to("cuda"), workspace=None)
    assert max_err(out, ref) <= ATTN_TOL
    assert_no_device_error()


def test_one_key_output_is_v_exactly():
    case = workloads.random_case(5, [1, 1, 1], 8, 2, block_size=16)
    dev = case.to("cuda")
    out = gpu_step(dev)
    # after the append the only cached token is the new one
    v = case.v_new.float()
    for b in range(3):
        for h in range(8):
            assert torch.equal(out[b, h].cpu().float(), v[b, h // 4])


def test_uniform_scores_give_mean_of_v():
    case = workloads.random_case(6, [300, 1200], 4, 4, block_size=32)
    case.q.zero_()
    h = host_inputs(case)
    oracle_step(h, case, decode=False)
    out = gpu_step(case.to("cuda"))
    for b, c in enumerate([300, 1200]):
        # mean over the context of V, gathered by the oracle's own decode with q = 0
        ref = oracle.decode(h["q"][b:b + 1], h["k_cache"], h["v_cache"], h["block_tables"][b:b + 1],
                            h["context_lens"][b:b + 1], case.scale)[0]
        assert max_err(out[b], ref) <= ATTN_TOL


def test_block_relabel_gives_bit_identical_output():
    case = workloads.random_case(7, [700, 33, 1500], 16, 4, block_size=16, extra_blocks=10)
    out1 = gpu_step(case.to("cuda"))
    g = torch.Generator().manual_seed(1)
    relabel = torch.randperm(case.num_blocks, generator=g)
    case2 = case.to("cpu")
    case2.k_cache = torch.empty_like(case.k_cache)
    case2.v_cache = torch.empty_like(case.v_cache)
    case2.k_cache[relabel] = case.k_cache
    case2.v_cache[relabel] = case.v_cache
    bt = case.block_tables.long()
    case2.block_tables = torch.where(bt >= 0, relabel[bt.clamp(min=0)], -1).to(torch.int32)
    out2 = gpu_step(case2.to("cuda"))
    assert torch.equal(out1, out2)


def test_peaky_softmax_long_context():
    # 1% of keys scaled by 8 (the long-context recipe), 3 requests of 8k tokens, block 64
    case = workloads.random_case(8, [8192, 8000, 4097], 32, 8, block_size=64, peaky_fraction=0.01,
                                 peaky_factor=8.0)
    err, _, _ = run_parity(case)
    assert err <= ATTN_TOL, err


def test_large_values_stay_within_tolerance():
    # |out| up to ~4: fp16 rounding alone is up to ~1e-3 there
    case = workloads.random_case(9, [64, 3000], 8, 8, block_size=16)
    case.v_cache.mul_(4.0)
    case.v_new.mul_(4.0)
    err, _, _ = run_parity(case)
    assert err <= ATTN_TOL, err


def test_side_stream_and_graph_capture():
    case = workloads.random_case(10, [900, 45, 2049], 32, 8, block_size=16)
    h = host_inputs(case)
    ref = oracle_step(h, case)
    dev = case.to("cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = gpu_step(dev)
    torch.cuda.current_stream().wait_stream(s)
    assert max_err(out, ref) <= ATTN_TOL
    # capture append + decode into a CUDA graph and replay it (the append rewrites the same slot)
    dev2 = case.to("cuda")
    slots = pkv.slot_mapping(case.block_tables, case.positions, 16).cuda()
    out_g = torch.empty_like(dev2.q)
    ws = pkv.make_workspace(dev2.num_seqs, dev2.num_q_heads, dev2.max_blocks_per_seq * 16, "cuda")
    g = torch.cuda.CUDAGraph()
    s2 = torch.cuda.Stream()
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s2):
        pkv.append(dev2.k_cache, dev2.v_cache, slots, dev2.k_new, dev2.v_new)   # warm up outside capture
        pkv.decode_attention(out_g, dev2.q, dev2.k_cache, dev2.v_cache, dev2.block_tables, dev2.context_lens,
                             dev2.scale, workspace=ws)
    torch.cuda.current_stream().wait_stream(s2)
    with torch.cuda.graph(g):
        pkv.append(dev2.k_cache, dev2.v_cache, slots, dev2.k_new, dev2.v_new)
        pkv.decode_attention(out_g, dev2.q, dev2.k_cache, dev2.v_cache, dev2.block_tables, dev2.context_lens,
                             dev2.scale, workspace=ws)
    out_g.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out)
    assert_no_device_error()


def test_workspace_reuse_leaves_counters_zero():
    # one workspace across calls with different contexts: the fused merge's completion counters
    # must come back to zero after every call, or later calls would merge too early or never
    first = workloads.random_case(21, [4000, 513, 1025, 77], 16, 4, block_size=16, extra_blocks=8)
    ws = pkv.make_workspace(first.num_seqs, first.num_q_heads, first.max_blocks_per_seq * 16, "cuda")
    for seed, ctxs in [(21, [4000, 513, 1025, 77]), (22, [600, 3999, 0, 2048]), (23, [1, 2, 3, 4000])]:
        case = workloads.random_case(seed, ctxs, 16, 4, block_size=16, extra_blocks=8)
        case.block_tables = torch.nn.functional.pad(case.block_tables,
                                                    (0, first.max_blocks_per_seq - case.max_blocks_per_seq),
                                                    value=-1)
        h = host_inputs(case)
        ref = oracle_step(h, case)
        out = gpu_step(case.to("cuda"), workspace=ws)
        assert max_err(out, ref) <= ATTN_TOL
        torch.cuda.synchronize()
        rows = 4 * 16 * -(-first.max_blocks_per_seq * 16 // pkv.PKV_DEFAULT_PARTITION)
        up = lambda x: x + (-x) % 256
        counters = ws[up(rows * 128 * 4) + 2 * up(rows * 4):].view(torch.int32)
        assert int(counters.abs().sum()) == 0
    assert_no_device_error()


def test_context_beyond_one_merge_tile():
    # 270,000 tokens = 528 partitions of 512: the fused merge takes its tiled branch
    case = workloads.random_case(31, [270000, 700], 2, 1, block_size=128)
    h = host_inputs(case)
    ref = oracle_step(h, case)
    dev = case.to("cuda")
    out = torch.empty_like(dev.q)
    ws = pkv.make_step_workspace(2, 2, case.max_blocks_per_seq * 128, device="cuda", partition_size=512)
    pkv.decode_step(out, dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                    case.scale, workspace=ws, partition_size=512)
    assert max_err(out, ref) <= ATTN_TOL
    assert_no_device_error()


@pytest.mark.parametrize("part", [16, 256, 512, 1536, 4096])
def test_step_with_explicit_partition(part):
    # the fused step at other partition sizes, down to one 16-token chunk per CTA
    case = workloads.random_case(32 + part, [5000, 1, 2049, 333, 4097], 16, 4, block_size=16, extra_blocks=5)
    h = host_inputs(case)
    ref = oracle_step(h, case)
    dev = case.to("cuda")
    out = torch.empty_like(dev.q)
    ws = pkv.make_step_workspace(5, 16, case.max_blocks_per_seq * 16, device="cuda", partition_size=part)
    pkv.decode_step(out, dev.q, dev.k_new, dev.v_new, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                    case.scale, workspace=ws, partition_size=part)
    assert max_err(out, ref) <= ATTN_TOL
    assert_no_device_error()
