"""Several new tokens per request (a verified draft, a prefill chunk) on the GPU against the
float64 oracle: causal attention of each new token over its request's paged cache."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, max_err

pytestmark = pytest.mark.gpu


def run_multi(case, ns, seed, workspace="auto"):
    rng = np.random.default_rng(seed)
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    t = int(qs[-1])
    q = rng.standard_normal((t, case.num_q_heads, case.head_dim)).astype(np.float16)
    h = case.to("cpu")
    ref = oracle.decode_multi(q, h.k_cache.numpy(), h.v_cache.numpy(), h.block_tables.numpy(), h.context_lens.numpy(),
                              qs, case.scale)
    dev = case.to("cuda")
    qd = torch.from_numpy(q).cuda()
    out = torch.full_like(qd, float("nan"))
    maxq = max(1, max(ns))
    if workspace == "auto":
        workspace = pkv.make_multi_workspace(case.num_seqs, t, maxq, case.num_q_heads, case.num_kv_heads,
                                             case.max_blocks_per_seq * case.block_size, "cuda")
    pkv.decode_attention_multi(out, qd, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                               torch.from_numpy(qs).cuda(), maxq, case.scale, workspace=workspace)
    return out, ref, workspace


CTXS = [1, 5, 16, 17, 100, 513, 1000, 2100, 3, 40]
NS = [1, 3, 4, 8, 2, 16, 5, 7, 3, 0]


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 64])
def test_multi_ragged(group, bs):
    case = workloads.random_case(600 + 10 * group + bs, CTXS, 2 * group, 2, block_size=bs, extra_blocks=3)
    out, ref, _ = run_multi(case, NS, group + bs)
    assert max_err(out, ref) <= ATTN_TOL, (group, bs)
    assert_no_device_error()


def test_multi_one_token_each_is_decode():
    ctxs = [700, 1, 2049, 33]
    case = workloads.random_case(620, ctxs, 32, 8, block_size=16)
    out, ref, _ = run_multi(case, [1, 1, 1, 1], 3)
    assert max_err(out, ref) <= ATTN_TOL
    # with one new token per request the result is the ordinary decode's
    dev = case.to("cuda")
    qd = out.clone()
    qd.copy_(torch.from_numpy(np.random.default_rng(3).standard_normal(qd.shape).astype(np.float16)))
    single = torch.empty_like(qd)
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * 16, "cuda")
    pkv.decode_attention(single, qd, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens, case.scale,
                         workspace=ws)
    assert max_err(single, ref) <= ATTN_TOL
    assert_no_device_error()


@pytest.mark.parametrize("group,n,ctx", [(4, 256, 1000), (1, 1024, 3000), (8, 40, 5000)])
def test_multi_long_chunk(group, n, ctx):
    case = workloads.random_case(630 + group, [ctx, 77], 2 * group, 2, block_size=32)
    out, ref, _ = run_multi(case, [n, 5], 5)
    assert max_err(out, ref) <= ATTN_TOL
    assert_no_device_error()


def test_multi_workspace_reuse_and_bad_rows():
    case = workloads.random_case(640, [3000, 600, 1200], 16, 4, block_size=16, extra_blocks=2)
    ws = pkv.make_multi_workspace(3, 64, 32, 16, 4, case.max_blocks_per_seq * 16, "cuda")
    for seed, ns in [(1, [4, 9, 2]), (2, [32, 1, 31])]:
        out, ref, _ = run_multi(case, ns, seed, workspace=ws)
        assert max_err(out, ref) <= ATTN_TOL
        torch.cuda.synchronize()
    assert_no_device_error()
    # a request claiming more new tokens than its context is skipped and recorded; the others
    # are still computed
    bad = workloads.random_case(641, [3, 900], 8, 4, block_size=16)
    dev = bad.to("cuda")
    qs = torch.tensor([0, 5, 7], dtype=torch.int32, device="cuda")
    q = torch.randn((7, 8, 128), generator=torch.Generator().manual_seed(1)).half().cuda()
    out = torch.zeros_like(q)
    wsb = pkv.make_multi_workspace(2, 7, 5, 8, 4, bad.max_blocks_per_seq * 16, "cuda")
    pkv.decode_attention_multi(out, q, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens, qs, 5,
                               bad.scale, workspace=wsb)
    assert pkv.device_error() == pkv.PKV_DEV_BAD_CONTEXT
    h = bad.to("cpu")
    ref = oracle.decode_multi(q[5:].cpu().numpy(), h.k_cache.numpy(), h.v_cache.numpy(), h.block_tables.numpy()[1:],
                              h.context_lens.numpy()[1:], np.array([0, 2], np.int32), bad.scale)
    assert max_err(out[5:], ref) <= ATTN_TOL
    assert not out[:5].any()


@pytest.mark.parametrize("nq", [4, 8])
def test_multi_full_size_gqa8b_sampled(nq):
    """The 8B-shaped GQA workload (batch 64, 2049-token contexts, block 16) with nq new tokens per
    request, as the benchmark runs it; requests 0, 31 and 63 compared with the oracle."""
    case = workloads.gqa8b(0, 1, 16, device="cuda")
    b = case.num_seqs
    g = torch.Generator(device="cuda")
    g.manual_seed(7000 + nq)
    q = torch.randn((b * nq, case.num_q_heads, 128), generator=g, device="cuda").half()
    qs = torch.arange(0, (b + 1) * nq, nq, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, float("nan"))
    ws = pkv.make_multi_workspace(b, b * nq, nq, case.num_q_heads, case.num_kv_heads,
                                  case.max_blocks_per_seq * 16, "cuda")
    pkv.decode_attention_multi(out, q, case.k_cache, case.v_cache, case.block_tables, case.context_lens, qs, nq,
                               case.scale, workspace=ws)
    kc, vc = case.k_cache.cpu().numpy(), case.v_cache.cpu().numpy()
    bt, cl = case.block_tables.cpu().numpy(), case.context_lens.cpu().numpy()
    for r in (0, 31, 63):
        ref = oracle.decode_multi(q[r * nq:(r + 1) * nq].cpu().numpy(), kc, vc, bt[r:r + 1], cl[r:r + 1],
                                  np.array([0, nq], np.int32), case.scale)
        assert max_err(out[r * nq:(r + 1) * nq], ref) <= ATTN_TOL, r
    assert torch.isfinite(out.float()).all()
    assert_no_device_error()
