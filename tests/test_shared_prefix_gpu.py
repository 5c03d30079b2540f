"""Shared-prefix decode (prefix chunks on the tensor cores + suffix split decode + fused merge)
against the float64 oracle on the full, un-shared definition."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, host_inputs, max_err, oracle_step

pytestmark = pytest.mark.gpu


def with_prefix(seed, prefix_len, suffixes, hq, hkv, bs=16, extra_blocks=3):
    """Requests that share the first prefix_len tokens' blocks, then private suffixes."""
    g = torch.Generator().manual_seed(seed)
    n_pre = prefix_len // bs
    need = [-(-s // bs) for s in suffixes]
    nb = n_pre + sum(need) + extra_blocks
    perm = torch.randperm(nb, generator=g)
    bt = torch.full((len(suffixes), n_pre + max(need + [1])), -1, dtype=torch.int32)
    pos = n_pre
    for i, n in enumerate(need):
        bt[i, :n_pre] = perm[:n_pre].to(torch.int32)
        bt[i, n_pre:n_pre + n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    ctx = [prefix_len + s for s in suffixes]
    return workloads._finish("prefix", hq, hkv, 128, bs, nb, bt, ctx, workloads._gen(seed + 1, "cpu"), "cpu")


def run(case, prefix_len):
    h = host_inputs(case)
    ref = oracle_step(h, case)
    dev = case.to("cuda")
    slots = pkv.slot_mapping(case.block_tables, case.positions, case.block_size).cuda()
    pkv.append(dev.k_cache, dev.v_cache, slots, dev.k_new, dev.v_new)
    ws = pkv.make_shared_prefix_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * case.block_size,
                                          prefix_len, "cuda")
    out = torch.empty_like(dev.q)
    pkv.decode_attention_shared_prefix(out, dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                                       case.scale, prefix_len, ws)
    return max_err(out, ref), out, dev, ws


@pytest.mark.parametrize("layer", [0, 31])
def test_shared_prefix_workload_full_size(layer):
    case = workloads.shared_prefix(layer, device="cuda")
    err, out, dev, _ = run(case, 1024)
    assert err <= ATTN_TOL, err
    # same answer as the plain decode over the same (already appended) cache
    ref2 = torch.empty_like(out)
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * 16, "cuda")
    pkv.decode_attention(ref2, dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens, case.scale,
                         workspace=ws)
    assert (out.float() - ref2.float()).abs().max().item() <= ATTN_TOL
    assert_no_device_error()


@pytest.mark.parametrize("group,hkv", [(1, 4), (4, 2), (8, 1)])
@pytest.mark.parametrize("prefix_len,bs", [(16, 16), (80, 16), (1024, 16), (192, 64), (256, 128)])
def test_ragged_prefixes(group, hkv, prefix_len, bs):
    # a suffix of 1 token (only the appended one), ragged suffixes, a long one
    case = with_prefix(100 + prefix_len + group, prefix_len, [1, 17, 511, 513, 1300], group * hkv, hkv, bs=bs)
    err, *_ = run(case, prefix_len)
    assert err <= ATTN_TOL, err
    assert_no_device_error()


def test_many_rows_span_two_row_tiles():
    # 40 requests x 4 q heads = 160 query rows per kv head: two 128-row tiles in the prefix kernel
    case = with_prefix(7, 128, list(range(1, 41)), 8, 2)
    err, *_ = run(case, 128)
    assert err <= ATTN_TOL, err
    assert_no_device_error()


def test_workspace_reuse_and_counters():
    case = with_prefix(8, 256, [300, 40, 1], 16, 4)
    err1, out1, dev, ws = run(case, 256)
    assert err1 <= ATTN_TOL
    out2 = torch.empty_like(out1)
    pkv.decode_attention_shared_prefix(out2, dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                                       case.scale, 256, ws)
    assert torch.equal(out1, out2)
    assert_no_device_error()


def test_prefix_mismatch_is_recorded():
    case = with_prefix(9, 64, [30, 30], 4, 1).to("cuda")
    case.block_tables[1, 2] = case.block_tables[1, 5]   # request 1 no longer shares block 2 of the prefix
    ws = pkv.make_shared_prefix_workspace(2, 4, case.max_blocks_per_seq * 16, 64, "cuda")
    out = torch.empty_like(case.q)
    pkv.decode_attention_shared_prefix(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                                       case.context_lens, case.scale, 64, ws)
    assert pkv.device_error() == pkv.PKV_DEV_PREFIX_MISMATCH
    with pytest.raises(pkv.PkvError):   # prefix length not a multiple of the block size
        pkv.decode_attention_shared_prefix(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                                           case.context_lens, case.scale, 40, ws)


def run_no_append(case, prefix_len):
    """decode_attention_shared_prefix over the cache as generated (no new token), twice."""
    h = host_inputs(case)
    ref = oracle.decode(h["q"], h["k_cache"], h["v_cache"], h["block_tables"], h["context_lens"], case.scale)
    dev = case.to("cuda")
    ws = pkv.make_shared_prefix_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * case.block_size,
                                          prefix_len, "cuda")
    outs = []
    for _ in range(2):
        out = torch.empty_like(dev.q)
        pkv.decode_attention_shared_prefix(out, dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                                           case.scale, prefix_len, ws)
        outs.append(out)
    return max_err(outs[0], ref), outs


@pytest.mark.parametrize("group,hkv", [(1, 4), (4, 2), (8, 1)])
def test_prefix_only_requests_merged_by_the_prefix_kernel(group, hkv):
    # every context is exactly the prefix: no suffix partition exists, so the prefix kernel's
    # last chunk CTA completes every request's count and merges it
    case = with_prefix(200 + group, 512, [0] * 6, group * hkv, hkv)
    err, outs = run_no_append(case, 512)
    assert err <= ATTN_TOL, err
    assert torch.equal(outs[0], outs[1])
    assert_no_device_error()


def test_mixed_prefix_only_and_long_suffixes_two_row_tiles():
    # 160 requests x 1 q head per kv head (two 128-row tiles); every other request has no suffix,
    # the others up to 1000 tokens: merges fall to both kernels, results repeat bit for bit
    suffixes = [0 if i % 2 == 0 else 100 + 37 * i % 900 for i in range(160)]
    case = with_prefix(210, 256, suffixes, 4, 4)
    err, outs = run_no_append(case, 256)
    assert err <= ATTN_TOL, err
    assert torch.equal(outs[0], outs[1])
    assert_no_device_error()
