"""pkv_decode_step_multi (several new tokens per request appended inside the attention launch)
against the float64 oracle's append + causal multi-token attention, and bit for bit against the
two-call path (pkv_append + pkv_decode_attention_multi): the cache after the step, and the
attention output."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, max_err

pytestmark = pytest.mark.gpu


def new_rows(case, ns, seed):
    """q, k_new, v_new for ns[b] new tokens of request b at positions ctx_b - n_b .. ctx_b - 1."""
    rng = np.random.default_rng(seed)
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    t = int(qs[-1])
    q = rng.standard_normal((t, case.num_q_heads, case.head_dim)).astype(np.float16)
    kn = rng.standard_normal((t, case.num_kv_heads, case.head_dim)).astype(np.float16)
    vn = rng.standard_normal((t, case.num_kv_heads, case.head_dim)).astype(np.float16)
    ctx = case.context_lens.cpu().numpy()
    pos = np.concatenate([np.arange(c - n, c) for c, n in zip(ctx, ns)]).astype(np.int32)
    return qs, q, kn, vn, pos


def oracle_step_multi(case, qs, q, kn, vn, pos):
    h = case.to("cpu")
    k, v, bt = h.k_cache.numpy().copy(), h.v_cache.numpy().copy(), h.block_tables.numpy()
    rows = np.repeat(np.arange(len(qs) - 1), np.diff(qs))
    slots = oracle.slot_mapping(bt[rows], pos, case.block_size)
    oracle.append(k, v, slots, kn, vn)
    return oracle.decode_multi(q, k, v, bt, h.context_lens.numpy(), qs, case.scale), k, v


def gpu_step_multi(case, qs, q, kn, vn, maxq, fused=True, overlap=False, workspace=None):
    dev = case.to("cuda")
    qd, knd, vnd = (torch.from_numpy(a).cuda() for a in (q, kn, vn))
    qsd = torch.from_numpy(qs).cuda()
    out = torch.full_like(qd, float("nan"))
    t = qd.shape[0]
    if workspace is None:
        workspace = pkv.make_multi_workspace(case.num_seqs, t, maxq, case.num_q_heads, case.num_kv_heads,
                                             case.max_blocks_per_seq * case.block_size, "cuda")
    if fused:
        pkv.decode_step_multi(out, qd, knd, vnd, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens, qsd,
                              maxq, case.scale, workspace=workspace, overlap=overlap)
    else:
        rows = np.repeat(np.arange(len(qs) - 1), np.diff(qs))
        pos = np.concatenate([np.arange(c - n, c) for c, n in zip(case.context_lens.cpu().numpy(), np.diff(qs))])
        slots = torch.from_numpy(oracle.slot_mapping(case.block_tables.cpu().numpy()[rows], pos.astype(np.int32),
                                                     case.block_size)).cuda()
        pkv.append(dev.k_cache, dev.v_cache, slots, knd, vnd)
        pkv.decode_attention_multi(out, qd, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens, qsd, maxq,
                                   case.scale, workspace=workspace)
    return out, dev


def check_pool(dev, k, v):
    assert np.array_equal(dev.k_cache.cpu().numpy().view(np.uint16), k.view(np.uint16))
    assert np.array_equal(dev.v_cache.cpu().numpy().view(np.uint16), v.view(np.uint16))


CTXS = [1, 5, 16, 17, 100, 513, 1000, 2100, 3, 40, 1026, 1030]
NS = [1, 3, 4, 8, 2, 16, 5, 7, 3, 0, 4, 16]   # the last two cross the 1024-token partition boundary


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 64])
def test_step_multi_matches_oracle_and_two_call_path(group, bs):
    case = workloads.random_case(1100 + 10 * group + bs, CTXS, 2 * group, 2, block_size=bs, extra_blocks=3)
    qs, q, kn, vn, pos = new_rows(case, NS, group + bs)
    ref, k, v = oracle_step_multi(case, qs, q, kn, vn, pos)
    out, dev = gpu_step_multi(case, qs, q, kn, vn, max(NS))
    assert max_err(out, ref) <= ATTN_TOL, (group, bs)
    check_pool(dev, k, v)                                  # the fused append is bit-exact over the pool
    two, dev2 = gpu_step_multi(case, qs, q, kn, vn, max(NS), fused=False)
    assert torch.equal(out, two)
    check_pool(dev2, k, v)
    assert_no_device_error()


@pytest.mark.parametrize("group,n", [(4, 4), (8, 2), (1, 16), (2, 9)])
def test_step_multi_uniform_lengths(group, n):
    ctxs = [2049 + 7 * i for i in range(12)]
    case = workloads.random_case(1150 + group + n, ctxs, 4 * group, 4, block_size=16, extra_blocks=3)
    ns = [n] * len(ctxs)
    qs, q, kn, vn, pos = new_rows(case, ns, n)
    ref, k, v = oracle_step_multi(case, qs, q, kn, vn, pos)
    out, dev = gpu_step_multi(case, qs, q, kn, vn, n)
    assert max_err(out, ref) <= ATTN_TOL
    check_pool(dev, k, v)
    assert_no_device_error()


def test_step_multi_whole_context_is_new():
    """Every cached position is a new token (a first prefill chunk of up to 16 tokens)."""
    ns = [16, 1, 7, 16]
    case = workloads.random_case(1170, ns, 16, 4, block_size=16, extra_blocks=2)
    qs, q, kn, vn, pos = new_rows(case, ns, 3)
    ref, k, v = oracle_step_multi(case, qs, q, kn, vn, pos)
    out, dev = gpu_step_multi(case, qs, q, kn, vn, 16)
    assert max_err(out, ref) <= ATTN_TOL
    check_pool(dev, k, v)
    assert_no_device_error()


def test_step_multi_layers_with_overlap():
    """Four layers (own caches, one shared workspace) with PKV_STEP_OVERLAP, eager and as a replayed
    graph: each layer equals the oracle and, bit for bit, the calls without the flag."""
    cases = [workloads.random_case(1180 + l, CTXS, 16, 4, block_size=16, extra_blocks=3) for l in range(4)]
    rows = [new_rows(c, NS, 40 + l) for l, c in enumerate(cases)]
    refs = [oracle_step_multi(c, *r)[0] for c, r in zip(cases, rows)]
    devs = [c.to("cuda") for c in cases]
    ins = [tuple(torch.from_numpy(a).cuda() for a in (r[1], r[2], r[3])) + (torch.from_numpy(r[0]).cuda(),)
           for r in rows]
    c0 = cases[0]
    ws = pkv.make_multi_workspace(c0.num_seqs, int(rows[0][0][-1]), 16, 16, 4, c0.max_blocks_per_seq * 16, "cuda")
    outs = [torch.empty_like(i[0]) for i in ins]

    def run(overlap):
        for l, (d, (qd, knd, vnd, qsd)) in enumerate(zip(devs, ins)):
            pkv.decode_step_multi(outs[l], qd, knd, vnd, d.k_cache, d.v_cache, d.block_tables, d.context_lens, qsd,
                                  16, d.scale, workspace=ws, overlap=overlap)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        run(True)
    torch.cuda.synchronize()
    for o, ref in zip(outs, refs):
        assert max_err(o, ref) <= ATTN_TOL
    first = [o.clone() for o in outs]
    with torch.cuda.stream(stream):
        run(False)
    torch.cuda.synchronize()
    assert all(torch.equal(o, f) for o, f in zip(outs, first))
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run(True)
        for _ in range(4):
            g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(o, f) for o, f in zip(outs, first))
    assert_no_device_error()


def test_step_multi_refuses_long_drafts():
    case = workloads.random_case(1190, [100, 200], 8, 2, block_size=16)
    qs, q, kn, vn, pos = new_rows(case, [17, 3], 1)
    with pytest.raises(pkv.PkvError):
        gpu_step_multi(case, qs, q, kn, vn, 17)


def test_step_multi_bad_block_id_skips_the_write_and_is_recorded():
    """A new token whose block id is outside the pool: its cache write is skipped (every access
    stays in bounds), the error is recorded, the other requests' rows and results are exact, and
    the context stays usable."""
    pkv.device_error()  # clear
    ctxs, ns = [300, 700, 40], [4, 3, 2]
    case = workloads.random_case(1195, ctxs, 8, 2, block_size=16, extra_blocks=3)
    qs, q, kn, vn, pos = new_rows(case, ns, 5)
    ref, k, v = oracle_step_multi(case, qs, q, kn, vn, pos)
    bad = case.to("cpu")
    bad.block_tables = case.block_tables.clone()  # (to("cpu") of a CPU case shares its tensors)
    bad.block_tables[1, (ctxs[1] - 1) // 16] = case.num_blocks + 9   # the block of request 1's last new token
    out, dev = gpu_step_multi(bad, qs, q, kn, vn, max(ns))
    assert pkv.device_error() == pkv.PKV_DEV_BAD_BLOCK_ID
    rows = np.repeat(np.arange(3), ns)
    keep = rows != 1
    assert max_err(out[torch.from_numpy(keep).cuda()], ref[keep]) <= ATTN_TOL
    # the same step with the valid table, on a fresh copy of the pool, is exact
    out2, dev2 = gpu_step_multi(case, qs, q, kn, vn, max(ns))
    assert max_err(out2, ref) <= ATTN_TOL
    check_pool(dev2, k, v)
    assert_no_device_error()


def test_step_multi_binding_checks_shapes():
    case = workloads.random_case(1197, [100, 200], 8, 2, block_size=16)
    qs, q, kn, vn, pos = new_rows(case, [3, 2], 1)
    dev = case.to("cuda")
    qd, knd, vnd = (torch.from_numpy(a).cuda() for a in (q, kn, vn))
    qsd = torch.from_numpy(qs).cuda()
    out = torch.empty_like(qd)
    with pytest.raises(ValueError):   # k_new must have one row per new token
        pkv.decode_step_multi(out, qd, knd[:-1], vnd, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                              qsd, 3, case.scale)
    with pytest.raises(ValueError):   # query_start must have num_seqs + 1 entries
        pkv.decode_step_multi(out, qd, knd, vnd, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                              qsd[:-1], 3, case.scale)
    with pytest.raises(pkv.PkvError):  # the one-launch step takes up to PKV_MAX_STEP_QUERY_LEN new tokens
        pkv.decode_step_multi(out, qd, knd, vnd, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                              qsd, pkv.PKV_MAX_STEP_QUERY_LEN + 1, case.scale)
    assert_no_device_error()
