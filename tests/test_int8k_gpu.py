"""The int8-key cache on the GPU against the float64 oracle.

The quantiser (append) must match the oracle's codes and scales bit for bit; decode over the
int8 keys must match the oracle's decode over the dequantised keys (code * scale) within the
attention tolerance, for every group size, several block sizes, ragged batches, split contexts,
peaky scores and the fused append of the decode step."""
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
    """Host (codes, scales, v) for the case's fp16 pool: every pool row quantised by the oracle."""
    k = case.k_cache.cpu().numpy()
    v = case.v_cache.cpu().numpy()
    nb, hkv, bs, d = k.shape
    codes = np.zeros((nb, hkv, bs, d), np.int8)
    scales = np.zeros((nb, hkv, bs), np.float32)
    v_out = np.zeros_like(v)
    rows_k = np.ascontiguousarray(k.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    rows_v = np.ascontiguousarray(v.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    oracle.append_quant_k(codes, scales, v_out, np.arange(nb * bs, dtype=np.int64), rows_k, rows_v)
    assert np.array_equal(v_out.view(np.uint16), v.view(np.uint16))
    return codes, scales, v


def to_dev(codes, scales, v):
    return (torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), torch.from_numpy(v).cuda())


def run_decode(case, codes, scales, v):
    dev = case.to("cuda")
    kc, ks, vc = to_dev(codes, scales, v)
    out = torch.empty_like(dev.q)
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * case.block_size, "cuda")
    pkv.decode_attention_int8k(out, dev.q, kc, ks, vc, dev.block_tables, dev.context_lens, case.scale, workspace=ws)
    return out


def test_append_int8k_bit_exact():
    rng = np.random.default_rng(12)
    nb, hkv, bs, d, t = 40, 8, 16, 128, 300
    kn = rng.standard_normal((t, hkv, d)).astype(np.float16)
    kn[0, 0] = 0                                                       # zero row: scale 0
    kn[1, 1] = np.tile(np.array([63.5, -63.5, 0.25, 0.75, -1.25, 10, 0.5, 1.5], np.float16), 16)  # ties
    kn[2, 2] = np.clip(rng.standard_normal(d) * 3e4, -65504, 65504).astype(np.float16)  # large
    kn[3, 3] = (rng.standard_normal(d) * 1e-6).astype(np.float16)      # fp16 subnormals
    kn[4, :] = (rng.standard_normal((hkv, d)) * 10.0 ** rng.uniform(-4, 4, (hkv, 1))).astype(np.float16)
    vn = rng.standard_normal((t, hkv, d)).astype(np.float16)
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[5::37] = -1
    codes = rng.integers(-128, 128, (nb, hkv, bs, d)).astype(np.int8)
    scales = rng.standard_normal((nb, hkv, bs)).astype(np.float32)
    v = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    kc, ks, vc = to_dev(codes, scales, v)
    pkv.append_int8k(kc, ks, vc, torch.from_numpy(slots).cuda(), torch.from_numpy(kn).cuda(),
                     torch.from_numpy(vn).cuda())
    oracle.append_quant_k(codes, scales, v, slots, kn, vn)
    assert np.array_equal(kc.cpu().numpy(), codes)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    assert np.array_equal(vc.cpu().numpy().view(np.uint16), v.view(np.uint16))
    assert_no_device_error()


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 64, 256])
def test_decode_int8k_ragged(group, bs):
    case = workloads.random_case(400 + 10 * group + bs, RAGGED, 2 * group, 2, block_size=bs, extra_blocks=4)
    codes, scales, v = quantised_pool(case)
    h = case.to("cpu")
    ref = oracle.decode_quant_k(h.q.numpy(), codes, scales, v, h.block_tables.numpy(), h.context_lens.numpy(),
                                case.scale)
    out = run_decode(case, codes, scales, v)
    assert max_err(out, ref) <= ATTN_TOL, (group, bs)
    assert_no_device_error()


@pytest.mark.parametrize("group,bs", [(1, 16), (2, 32), (4, 128), (8, 16)])
def test_decode_step_int8k_fused_append(group, bs):
    ctxs = [1, 16, 17, 513, 2049, 300, 0, 1024]
    case = workloads.random_case(500 + group + bs, ctxs, 4 * group, 4, block_size=bs, extra_blocks=3)
    codes, scales, v = quantised_pool(case)
    h = case.to("cpu")
    bt, ctx = h.block_tables.numpy(), h.context_lens.numpy()
    # oracle: quantise-append the new token at ctx - 1, then decode
    co, so, vo = codes.copy(), scales.copy(), v.copy()
    slots = oracle.slot_mapping(bt, h.positions.numpy(), bs)
    oracle.append_quant_k(co, so, vo, slots, h.k_new.numpy(), h.v_new.numpy())
    ref = oracle.decode_quant_k(h.q.numpy(), co, so, vo, bt, ctx, case.scale)
    dev = case.to("cuda")
    kc, ks, vc = to_dev(codes, scales, v)
    out = torch.empty_like(dev.q)
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * bs, "cuda")
    pkv.decode_step_int8k(out, dev.q, dev.k_new, dev.v_new, kc, ks, vc, dev.block_tables, dev.context_lens,
                          case.scale, workspace=ws)
    assert max_err(out, ref) <= ATTN_TOL
    assert np.array_equal(kc.cpu().numpy(), co)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert np.array_equal(vc.cpu().numpy().view(np.uint16), vo.view(np.uint16))
    assert_no_device_error()


def test_decode_int8k_peaky_long_context():
    case = workloads.random_case(77, [8192, 8000, 4097], 32, 8, block_size=64, peaky_fraction=0.01,
                                 peaky_factor=8.0)
    codes, scales, v = quantised_pool(case)
    h = case.to("cpu")
    ref = oracle.decode_quant_k(h.q.numpy(), codes, scales, v, h.block_tables.numpy(), h.context_lens.numpy(),
                                case.scale)
    out = run_decode(case, codes, scales, v)
    assert max_err(out, ref) <= ATTN_TOL
    assert_no_device_error()


def test_decode_int8k_block_relabel_bit_identical():
    case = workloads.random_case(78, [700, 33, 1500], 16, 4, block_size=16, extra_blocks=10)
    codes, scales, v = quantised_pool(case)
    out1 = run_decode(case, codes, scales, v)
    relabel = torch.randperm(case.num_blocks, generator=torch.Generator().manual_seed(2)).numpy()
    c2, s2, v2 = np.empty_like(codes), np.empty_like(scales), np.empty_like(v)
    c2[relabel], s2[relabel], v2[relabel] = codes, scales, v
    case2 = case.to("cpu")
    bt = case.block_tables.cpu().long().numpy()
    case2.block_tables = torch.from_numpy(np.where(bt >= 0, relabel[np.clip(bt, 0, None)], -1).astype(np.int32))
    out2 = run_decode(case2, c2, s2, v2)
    assert torch.equal(out1, out2)


def test_int8k_full_size_mha7b_sampled():
    """The 7B-shaped workload as the benchmark runs it with int8 keys: every pool row quantised by
    the library's append kernel (codes and scales bit-exact against the oracle's quantiser), then
    one fused decode step; requests 0, 7 and 15 compared with the oracle."""
    case = workloads.mha7b(0, device="cuda")
    nb, hkv, bs, d = case.k_cache.shape
    kc, ks, vc = pkv.empty_int8k_cache(nb, hkv, bs, "cuda")
    vc.copy_(case.v_cache)
    rows_k = case.k_cache.permute(0, 2, 1, 3).reshape(nb * bs, hkv, d).contiguous()
    rows_v = case.v_cache.permute(0, 2, 1, 3).reshape(nb * bs, hkv, d).contiguous()
    pkv.append_int8k(kc, ks, vc, torch.arange(nb * bs, device="cuda"), rows_k, rows_v)
    codes, scales, v = quantised_pool(case)
    assert np.array_equal(kc.cpu().numpy(), codes)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    h = case.to("cpu")
    bt, ctx = h.block_tables.numpy(), h.context_lens.numpy()
    co, so, vo = codes.copy(), scales.copy(), v.copy()
    slots = oracle.slot_mapping(bt, h.positions.numpy(), bs)
    oracle.append_quant_k(co, so, vo, slots, h.k_new.numpy(), h.v_new.numpy())
    out = torch.empty_like(case.q)
    ws = pkv.make_workspace(case.num_seqs, case.num_q_heads, case.max_blocks_per_seq * bs, "cuda")
    pkv.decode_step_int8k(out, case.q, case.k_new, case.v_new, kc, ks, vc, case.block_tables, case.context_lens,
                          case.scale, workspace=ws)
    for r in (0, 7, 15):
        ref = oracle.decode_quant_k(h.q.numpy()[r:r + 1], co, so, vo, bt[r:r + 1], ctx[r:r + 1], case.scale)
        assert max_err(out[r:r + 1], ref) <= ATTN_TOL, r
    assert_no_device_error()
