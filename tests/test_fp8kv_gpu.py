"""The optional fp8 (E4M3) K + V cache on the GPU against the float64 oracle.

Append must match the oracle's key and value codes and scales bit for bit (the hardware
conversion's round-to-nearest-even against the oracle's brute-force nearest code); decode over
the fp8 cache must match the oracle's decode over the dequantised keys and values within the
attention tolerance, for every group size, several block sizes, ragged batches, split contexts,
peaky scores, NaN codes past the context, and the fused append of the decode step."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, max_err

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 15, 16, 17, 100, 511, 512, 513, 1000, 1537, 2100]


def quantised_pool(case):
    """Host (k_codes, k_scale, v_codes, v_scale): every row of the case's fp16 pool quantised by
    the oracle."""
    k = case.k_cache.cpu().numpy()
    v = case.v_cache.cpu().numpy()
    nb, hkv, bs, d = k.shape
    kc, vc = np.zeros((nb, hkv, bs, d), np.uint8), np.zeros((nb, hkv, bs, d), np.uint8)
    ks, vs = np.zeros((nb, hkv, bs), np.float32), np.zeros((nb, hkv, bs), np.float32)
    rows_k = np.ascontiguousarray(k.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    rows_v = np.ascontiguousarray(v.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    oracle.append_fp8_kv(kc, ks, vc, vs, np.arange(nb * bs, dtype=np.int64), rows_k, rows_v)
    return kc, ks, vc, vs


def to_dev(*arrays):
    return tuple(torch.from_numpy(a).cuda() for a in arrays)


def assert_pool_equal(dev, host):
    for d, h in zip(dev, host):
        got = d.cpu().numpy()
        assert got.dtype == h.dtype
        if h.dtype == np.float32:
            assert np.array_equal(got.view(np.uint32), h.view(np.uint32))
        else:
            assert np.array_equal(got, h)


def run_decode(case, pool):
    dev = case.to("cuda")
    kc, ks, vc, vs = to_dev(*pool)
    out = torch.empty_like(dev.q)
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * case.block_size, "cuda")
    pkv.decode_attention_fp8kv(out, dev.q, kc, ks, vc, vs, dev.block_tables, dev.context_lens, case.scale,
                               workspace=ws)
    return out


def oracle_decode(case, pool):
    h = case.to("cpu")
    return oracle.decode_fp8_kv(h.q.numpy(), *pool, h.block_tables.numpy(), h.context_lens.numpy(), case.scale)


def test_append_fp8kv_bit_exact():
    rng = np.random.default_rng(23)
    nb, hkv, bs, d, t = 40, 8, 16, 128, 300
    kn = rng.standard_normal((t, hkv, d)).astype(np.float16)
    vn = rng.standard_normal((t, hkv, d)).astype(np.float16)
    for x in (kn, vn):
        x[0, 0] = 0                                                    # zero row: scale 0
        x[1, 1] = np.tile(np.array([28, -28, 1.0, 0.5, 0.03125, 1.0625, 1.1875, -0.75], np.float16), 16)  # ties
        x[2, 2] = np.clip(rng.standard_normal(d) * 3e4, -65504, 65504).astype(np.float16)  # large
        x[3, 3] = (rng.standard_normal(d) * 1e-6).astype(np.float16)   # fp16 subnormals
        x[6, 4] = np.tile(np.array([28, 6.1035e-05, 1.831e-04, -6.1035e-05], np.float16), 32)  # E4M3 subnormals, -0
        x[4, :] = (rng.standard_normal((hkv, d)) * 10.0 ** rng.uniform(-4, 4, (hkv, 1))).astype(np.float16)
    vn[7, 5] = 0                                                       # zero value row, nonzero key row
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[5::37] = -1
    pool = (rng.integers(0, 256, (nb, hkv, bs, d)).astype(np.uint8),
            rng.standard_normal((nb, hkv, bs)).astype(np.float32),
            rng.integers(0, 256, (nb, hkv, bs, d)).astype(np.uint8),
            rng.standard_normal((nb, hkv, bs)).astype(np.float32))
    dev = to_dev(*pool)
    pkv.append_fp8kv(*dev, torch.from_numpy(slots).cuda(), torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda())
    oracle.append_fp8_kv(*pool, slots, kn, vn)
    assert_pool_equal(dev, pool)
    blk, off = divmod(int(slots[6]), bs)
    assert slots[6] >= 0 and pool[0][blk, 4, off, :4].tolist() == [0x7e, 0x00, 0x02, 0x80]  # 448, 0, 2^-8, -0
    assert_no_device_error()


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 64, 256])
def test_decode_fp8kv_ragged(group, bs):
    case = workloads.random_case(620 + 10 * group + bs, RAGGED, 2 * group, 2, block_size=bs, extra_blocks=4)
    pool = quantised_pool(case)
    assert max_err(run_decode(case, pool), oracle_decode(case, pool)) <= ATTN_TOL, (group, bs)
    assert_no_device_error()


@pytest.mark.parametrize("group", [1, 4])
def test_decode_fp8kv_nan_codes_past_the_context(group):
    """Every code at a position at or past a request's context length is a NaN code and every
    scale there NaN: the ragged tails' unused rows must not reach the result."""
    ctxs = [1, 15, 17, 100, 513, 1030]
    case = workloads.random_case(640 + group, ctxs, 4 * group, 4, block_size=16, extra_blocks=4)
    pool = tuple(a.copy() for a in quantised_pool(case))
    bt = case.block_tables.cpu().numpy()
    live = np.zeros((case.num_blocks, 16), bool)
    for b, c in enumerate(ctxs):
        for p in range(c):
            live[bt[b, p // 16], p % 16] = True
    dead = ~live
    for codes in (pool[0], pool[2]):
        codes.transpose(0, 2, 1, 3)[dead] = 0x7f
    for sc in (pool[1], pool[3]):
        sc.transpose(0, 2, 1)[dead] = np.nan
    out = run_decode(case, pool)
    assert torch.isfinite(out.float()).all()
    assert max_err(out, oracle_decode(case, pool)) <= ATTN_TOL
    assert_no_device_error()


@pytest.mark.parametrize("group,bs", [(1, 16), (2, 32), (4, 128), (8, 16)])
def test_decode_step_fp8kv_fused_append(group, bs):
    ctxs = [1, 16, 17, 513, 2049, 300, 0, 1024]
    case = workloads.random_case(720 + group + bs, ctxs, 4 * group, 4, block_size=bs, extra_blocks=3)
    pool = quantised_pool(case)
    h = case.to("cpu")
    bt, ctx = h.block_tables.numpy(), h.context_lens.numpy()
    # oracle: quantise-append the new token at ctx - 1, then decode
    want = tuple(a.copy() for a in pool)
    slots = oracle.slot_mapping(bt, h.positions.numpy(), bs)
    oracle.append_fp8_kv(*want, slots, h.k_new.numpy(), h.v_new.numpy())
    ref = oracle.decode_fp8_kv(h.q.numpy(), *want, bt, ctx, case.scale)
    dev = case.to("cuda")
    got = to_dev(*pool)
    out = torch.empty_like(dev.q)
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * bs, "cuda")
    pkv.decode_step_fp8kv(out, dev.q, dev.k_new, dev.v_new, *got, dev.block_tables, dev.context_lens, case.scale,
                          workspace=ws)
    assert max_err(out, ref) <= ATTN_TOL
    assert_pool_equal(got, want)
    assert_no_device_error()


def test_decode_fp8kv_peaky_long_context():
    case = workloads.random_case(82, [8192, 8000, 4097], 32, 8, block_size=64, peaky_fraction=0.01,
                                 peaky_factor=8.0)
    pool = quantised_pool(case)
    assert max_err(run_decode(case, pool), oracle_decode(case, pool)) <= ATTN_TOL
    assert_no_device_error()


def test_decode_fp8kv_block_relabel_bit_identical():
    case = workloads.random_case(83, [700, 33, 1500], 16, 4, block_size=16, extra_blocks=10)
    pool = quantised_pool(case)
    out1 = run_decode(case, pool)
    relabel = torch.randperm(case.num_blocks, generator=torch.Generator().manual_seed(4)).numpy()
    pool2 = tuple(np.empty_like(a) for a in pool)
    for a2, a in zip(pool2, pool):
        a2[relabel] = a
    case2 = case.to("cpu")
    bt = case.block_tables.cpu().long().numpy()
    case2.block_tables = torch.from_numpy(np.where(bt >= 0, relabel[np.clip(bt, 0, None)], -1).astype(np.int32))
    out2 = run_decode(case2, pool2)
    assert torch.equal(out1, out2)


def test_fp8kv_full_size_gqa8b_sampled():
    """The 8B-shaped GQA workload with fp8 keys and values: every pool row quantised by the
    library's append kernel (bit-exact against the oracle's quantiser), then one fused decode
    step; requests 0, 31 and 63 compared with the oracle."""
    case = workloads.gqa8b(0, device="cuda")
    nb, hkv, bs, d = case.k_cache.shape
    dev = pkv.empty_fp8kv_cache(nb, hkv, bs, "cuda")
    rows_k = case.k_cache.permute(0, 2, 1, 3).reshape(nb * bs, hkv, d).contiguous()
    rows_v = case.v_cache.permute(0, 2, 1, 3).reshape(nb * bs, hkv, d).contiguous()
    pkv.append_fp8kv(*dev, torch.arange(nb * bs, device="cuda"), rows_k, rows_v)
    pool = quantised_pool(case)
    assert_pool_equal(dev, pool)
    h = case.to("cpu")
    bt, ctx = h.block_tables.numpy(), h.context_lens.numpy()
    slots = oracle.slot_mapping(bt, h.positions.numpy(), bs)
    oracle.append_fp8_kv(*pool, slots, h.k_new.numpy(), h.v_new.numpy())
    out = torch.empty_like(case.q)
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * bs, "cuda")
    pkv.decode_step_fp8kv(out, case.q, case.k_new, case.v_new, *dev, case.block_tables, case.context_lens,
                          case.scale, workspace=ws)
    for r in (0, 31, 63):
        ref = oracle.decode_fp8_kv(h.q.numpy()[r:r + 1], *pool, bt[r:r + 1], ctx[r:r + 1], case.scale)
        assert max_err(out[r:r + 1], ref) <= ATTN_TOL, r
    assert_no_device_error()


def test_decode_fp8kv_values_near_fp16_max():
    """Value rows up to the fp16 maximum (row scales near 65504 / 448): the weights folded with the
    value scales stay finite.  Compared relative to the output's magnitude (fp16 output rounding)."""
    case = workloads.random_case(84, [3000, 17, 1025], 16, 4, block_size=16, peaky_fraction=0.02, peaky_factor=6.0)
    g = torch.Generator().manual_seed(6)
    big = torch.randn(case.v_cache.shape, generator=g) * 2e4
    case.v_cache = big.clamp(-65504, 65504).half().to(case.v_cache.device)
    pool = quantised_pool(case)
    assert pool[3].max() > 65504 / 448 * 0.95
    ref = oracle_decode(case, pool)
    out = run_decode(case, pool)
    assert max_err(out, ref) <= ATTN_TOL * np.abs(ref).max()
    assert_no_device_error()


def test_fp8kv_binding_checks_dtypes():
    case = workloads.random_case(85, [40, 3], 8, 2, block_size=16).to("cuda")
    nb, hkv, bs, d = case.k_cache.shape
    kc, ks, vc, vs = pkv.empty_fp8kv_cache(nb, hkv, bs, "cuda")
    out = torch.empty_like(case.q)
    with pytest.raises(ValueError):   # int8 codes are not fp8 codes
        pkv.decode_attention_fp8kv(out, case.q, kc.view(torch.int8), ks, vc, vs, case.block_tables,
                                   case.context_lens, case.scale)
    with pytest.raises(ValueError):   # scales per (block, kv head, slot)
        pkv.decode_attention_fp8kv(out, case.q, kc, ks[:, :, :1].contiguous(), vc, vs, case.block_tables,
                                   case.context_lens, case.scale)
    assert_no_device_error()
