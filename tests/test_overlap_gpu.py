"""Step calls with PKV_STEP_OVERLAP, as a model runs its layers: each layer's step on its own
caches, back to back on one stream, sharing one split workspace (eagerly, and as a replayed CUDA
graph).  Each layer's kernels stream their cache history while the previous layer's kernel drains
and touch q, the new rows, the workspace and out only after it completes.  Every layer must equal
the float64 oracle (append bit-exact, attention within tolerance) and, bit for bit, the same steps
called without the flag."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, host_inputs, max_err, oracle_step
from test_shared_prefix_gpu import with_prefix
import test_int8k_gpu as i8k
import test_int8kv_gpu as i8kv
import test_fp8kv_gpu as f8kv

pytestmark = pytest.mark.gpu

LAYERS = 4
LENS = [0, 1, 17, 1024, 1025, 2100, 4000, 300]


def run_layers(fn, outs, stream, overlap):
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for l in range(len(outs)):
            fn(l, outs[l], overlap)
    torch.cuda.synchronize()


def replay_graph(fn, outs, stream, times):
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(len(outs)):
                fn(l, outs[l], True)
        for _ in range(times):
            g.replay()
    torch.cuda.synchronize()


def check_overlap(fn, outs, refs):
    """fn(l, out, overlap) runs layer l's step.  The appends rewrite the same rows with the same
    values, so every run sees the same caches."""
    stream = torch.cuda.Stream()
    run_layers(fn, outs, stream, True)
    for l, ref in enumerate(refs):
        assert max_err(outs[l], ref) <= ATTN_TOL, l
    first = [o.clone() for o in outs]
    for o in outs:
        o.fill_(7.0)
    run_layers(fn, outs, stream, False)
    for l in range(len(outs)):
        assert torch.equal(outs[l], first[l]), l
    for o in outs:
        o.fill_(7.0)
    replay_graph(fn, outs, stream, 5)
    for l in range(len(outs)):
        assert torch.equal(outs[l], first[l]), l
    assert_no_device_error()


@pytest.mark.parametrize("group,bs", [(1, 16), (4, 16), (8, 64)])
def test_fp16_steps(group, bs):
    cases = [workloads.random_case(700 + 10 * l + group, LENS, 4 * group, 4, block_size=bs, extra_blocks=3)
             for l in range(LAYERS)]
    hosts = [host_inputs(c) for c in cases]
    refs = [oracle_step(h, c) for h, c in zip(hosts, cases)]
    devs = [c.to("cuda") for c in cases]
    c0 = cases[0]
    ws = pkv.make_step_workspace(c0.num_seqs, c0.num_q_heads, c0.max_blocks_per_seq * bs, 0, "cuda")
    outs = [torch.empty_like(d.q) for d in devs]

    def fn(l, out, overlap):
        d = devs[l]
        pkv.decode_step(out, d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.scale,
                        0, ws, overlap=overlap)

    check_overlap(fn, outs, refs)
    for d, h in zip(devs, hosts):
        assert np.array_equal(d.k_cache.cpu().numpy().view(np.uint16), h["k_cache"].view(np.uint16))
        assert np.array_equal(d.v_cache.cpu().numpy().view(np.uint16), h["v_cache"].view(np.uint16))


def test_fp16_steps_explicit_partition():
    cases = [workloads.random_case(760 + l, LENS, 32, 8, block_size=16, extra_blocks=3) for l in range(LAYERS)]
    refs = [oracle_step(host_inputs(c), c) for c in cases]
    devs = [c.to("cuda") for c in cases]
    c0 = cases[0]
    ws = pkv.make_step_workspace(c0.num_seqs, c0.num_q_heads, c0.max_blocks_per_seq * 16, 0, "cuda",
                                 partition_size=512)
    outs = [torch.empty_like(d.q) for d in devs]

    def fn(l, out, overlap):
        d = devs[l]
        pkv.decode_step(out, d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.scale,
                        0, ws, partition_size=512, overlap=overlap)

    check_overlap(fn, outs, refs)


def test_shared_prefix_steps():
    cases = [with_prefix(780 + l, 256, [1, 40, 700, 129, 1000], 32, 8) for l in range(LAYERS)]
    refs = [oracle_step(host_inputs(c), c) for c in cases]
    devs = [c.to("cuda") for c in cases]
    c0 = cases[0]
    ws = pkv.make_step_workspace(c0.num_seqs, c0.num_q_heads, c0.max_blocks_per_seq * c0.block_size, 256, "cuda")
    outs = [torch.empty_like(d.q) for d in devs]

    def fn(l, out, overlap):
        d = devs[l]
        pkv.decode_step(out, d.q, d.k_new, d.v_new, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.scale,
                        256, ws, overlap=overlap)

    check_overlap(fn, outs, refs)


@pytest.mark.parametrize("group", [1, 4])
def test_int8k_steps(group):
    cases = [workloads.random_case(800 + 10 * l + group, LENS, 4 * group, 4, block_size=16, extra_blocks=3)
             for l in range(LAYERS)]
    refs, pools = [], []
    for c in cases:
        codes, scales, v = i8k.quantised_pool(c)
        h = c.to("cpu")
        bt = h.block_tables.numpy()
        co, so, vo = codes.copy(), scales.copy(), v.copy()
        oracle.append_quant_k(co, so, vo, oracle.slot_mapping(bt, h.positions.numpy(), c.block_size),
                              h.k_new.numpy(), h.v_new.numpy())
        refs.append(oracle.decode_quant_k(h.q.numpy(), co, so, vo, bt, h.context_lens.numpy(), c.scale))
        pools.append(i8k.to_dev(codes, scales, v))
    devs = [c.to("cuda") for c in cases]
    c0 = cases[0]
    ws = pkv.make_workspace(c0.num_seqs, c0.num_q_heads, c0.max_blocks_per_seq * 16, "cuda")
    outs = [torch.empty_like(d.q) for d in devs]

    def fn(l, out, overlap):
        d, (kc, ks, vc) = devs[l], pools[l]
        pkv.decode_step_int8k(out, d.q, d.k_new, d.v_new, kc, ks, vc, d.block_tables, d.context_lens, d.scale,
                              workspace=ws, overlap=overlap)

    check_overlap(fn, outs, refs)


def test_int8kv_steps():
    cases = [workloads.random_case(850 + l, LENS, 32, 8, block_size=16, extra_blocks=3) for l in range(LAYERS)]
    refs, pools = [], []
    for c in cases:
        pool = i8kv.quantised_pool(c)
        h = c.to("cpu")
        bt = h.block_tables.numpy()
        host = tuple(a.copy() for a in pool)
        oracle.append_quant_kv(*host, oracle.slot_mapping(bt, h.positions.numpy(), c.block_size),
                               h.k_new.numpy(), h.v_new.numpy())
        refs.append(oracle.decode_quant_kv(h.q.numpy(), *host, bt, h.context_lens.numpy(), c.scale))
        pools.append(i8kv.to_dev(*pool))
    devs = [c.to("cuda") for c in cases]
    c0 = cases[0]
    ws = pkv.make_workspace(c0.num_seqs, c0.num_q_heads, c0.max_blocks_per_seq * 16, "cuda")
    outs = [torch.empty_like(d.q) for d in devs]

    def fn(l, out, overlap):
        d, (kc, ks, vc, vs) = devs[l], pools[l]
        pkv.decode_step_int8kv(out, d.q, d.k_new, d.v_new, kc, ks, vc, vs, d.block_tables, d.context_lens, d.scale,
                               workspace=ws, overlap=overlap)

    check_overlap(fn, outs, refs)


def test_fp8kv_steps():
    cases = [workloads.random_case(870 + l, LENS, 32, 8, block_size=16, extra_blocks=3) for l in range(LAYERS)]
    refs, pools = [], []
    for c in cases:
        pool = f8kv.quantised_pool(c)
        h = c.to("cpu")
        bt = h.block_tables.numpy()
        host = tuple(a.copy() for a in pool)
        oracle.append_fp8_kv(*host, oracle.slot_mapping(bt, h.positions.numpy(), c.block_size),
                             h.k_new.numpy(), h.v_new.numpy())
        refs.append(oracle.decode_fp8_kv(h.q.numpy(), *host, bt, h.context_lens.numpy(), c.scale))
        pools.append(f8kv.to_dev(*pool))
    devs = [c.to("cuda") for c in cases]
    c0 = cases[0]
    ws = pkv.make_workspace(c0.num_seqs, c0.num_q_heads, c0.max_blocks_per_seq * 16, "cuda")
    outs = [torch.empty_like(d.q) for d in devs]

    def fn(l, out, overlap):
        d, (kc, ks, vc, vs) = devs[l], pools[l]
        pkv.decode_step_fp8kv(out, d.q, d.k_new, d.v_new, kc, ks, vc, vs, d.block_tables, d.context_lens, d.scale,
                              workspace=ws, overlap=overlap)

    check_overlap(fn, outs, refs)


def test_full_size_gqa8b_layers_sampled():
    """Four layers of the 8B-shaped GQA step (64 requests, 2,049-token contexts) with the flag, in a
    replayed graph: layer 0 against the oracle on sampled requests, every layer bit-identical to
    the calls without the flag."""
    cases = [workloads.gqa8b(l, device="cuda") for l in range(LAYERS)]
    c0 = cases[0]
    ws = pkv.make_step_workspace(c0.num_seqs, c0.num_q_heads, c0.max_blocks_per_seq * c0.block_size, 0, "cuda")
    outs = [torch.empty_like(c.q) for c in cases]
    sample = [0, 17, 63]
    h = host_inputs(c0)

    def fn(l, out, overlap):
        c = cases[l]
        pkv.decode_step(out, c.q, c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale,
                        0, ws, overlap=overlap)

    stream = torch.cuda.Stream()
    replay_graph(fn, outs, stream, 3)
    first = [o.clone() for o in outs]
    run_layers(fn, outs, stream, False)
    for l in range(LAYERS):
        assert torch.equal(outs[l], first[l]), l
    slots = oracle.slot_mapping(h["block_tables"], h["positions"], c0.block_size)
    oracle.append(h["k_cache"], h["v_cache"], slots, h["k_new"], h["v_new"])
    ref = oracle.decode(h["q"][sample], h["k_cache"], h["v_cache"], h["block_tables"][sample],
                        h["context_lens"][sample], c0.scale)
    assert max_err(first[0][sample], ref) <= ATTN_TOL
    assert_no_device_error()
