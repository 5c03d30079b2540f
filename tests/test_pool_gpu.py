"""Copy-on-write of shared blocks on the GPU: the block-copy kernel against the oracle's copy
(bit for bit), its handling of bad ids, and a fork-then-diverge decode step driven by the host
block pool, compared with the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
from gpu_util import ATTN_TOL, assert_no_device_error, max_err

pytestmark = pytest.mark.gpu


def _pairs(rng, nb, n):
    ids = rng.permutation(nb)[:2 * n]
    return ids[:n].astype(np.int32), ids[n:].astype(np.int32)


@pytest.mark.parametrize("hkv,bs", [(8, 16), (32, 128), (2, 48)])
def test_copy_blocks_bit_exact(hkv, bs):
    rng = np.random.default_rng(hkv * 1000 + bs)
    nb, d, n = 700, 128, 211
    kc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    vc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    src, dst = _pairs(rng, nb, n)
    kd, vd = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    pkv.copy_blocks(kd, vd, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    oracle.copy_blocks(kc, vc, src, dst)
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), kc.view(np.uint16))
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), vc.view(np.uint16))
    assert_no_device_error()


def test_copy_blocks_empty_and_bad_ids():
    rng = np.random.default_rng(3)
    kc = torch.from_numpy(rng.standard_normal((10, 2, 16, 128)).astype(np.float16)).cuda()
    vc = torch.from_numpy(rng.standard_normal((10, 2, 16, 128)).astype(np.float16)).cuda()
    k0, v0 = kc.clone(), vc.clone()
    empty = torch.empty(0, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(kc, vc, empty, empty)
    # out-of-range ids skip their pair and raise the device error word; the valid pair is copied
    pkv.copy_blocks(kc, vc, torch.tensor([10, 1, 2], dtype=torch.int32, device="cuda"),
                    torch.tensor([3, -1, 4], dtype=torch.int32, device="cuda"))
    assert pkv.device_error() == pkv.PKV_DEV_BAD_BLOCK_ID
    k0[4], v0[4] = k0[2], v0[2]
    assert torch.equal(kc, k0) and torch.equal(vc, v0)
    assert_no_device_error()


@pytest.mark.parametrize("bs", [16, 64])
def test_fork_then_diverge_decode_step(bs):
    """One parent of 1000 tokens forks into three children (beam-style); all four then append a
    different token at position 1000, inside the shared last block.  Each child copies that block
    on write; the fused append + decode must match the oracle's copy, append and decode."""
    rng = np.random.default_rng(bs)
    hq, hkv, d, ctx, kids = 32, 8, 128, 1000, 3
    nb = 4 * (-(-(ctx + 1) // bs)) + 8
    kc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    vc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    pool = pkv.BlockPool(nb, seed=bs)
    maxb = -(-(ctx + 1) // bs)
    rows = [torch.full((maxb,), -1, dtype=torch.int32) for _ in range(kids + 1)]
    pool.reserve(rows[0], 0, ctx, bs)
    for r in rows[1:]:
        pool.fork(rows[0], r, ctx, bs)
    # the children diverge first (each copies the shared block); the parent, left as the block's
    # only holder, then appends in place
    pairs = [pool.prepare_append(r, ctx, bs) for r in rows[1:]] + [pool.prepare_append(rows[0], ctx, bs)]
    if ctx % bs:
        assert all(p is not None for p in pairs[:-1]) and pairs[-1] is None
    else:
        assert all(p is None for p in pairs)
    src = np.array([p[0] for p in pairs if p], np.int32)
    dst = np.array([p[1] for p in pairs if p], np.int32)
    bt = torch.stack(rows)
    b = kids + 1
    q = rng.standard_normal((b, hq, d)).astype(np.float16)
    k_new = rng.standard_normal((b, hkv, d)).astype(np.float16)
    v_new = rng.standard_normal((b, hkv, d)).astype(np.float16)
    lens = np.full(b, ctx + 1, np.int32)
    scale = d ** -0.5
    # oracle: copy, append, decode
    ko, vo = kc.copy(), vc.copy()
    oracle.copy_blocks(ko, vo, src, dst)
    slots = oracle.slot_mapping(bt.numpy(), np.full(b, ctx, np.int32), bs)
    oracle.append(ko, vo, slots, k_new, v_new)
    ref = oracle.decode(q, ko, vo, bt.numpy(), lens, scale)
    # GPU: copy_blocks, then the fused step
    kd, vd = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    if len(src):
        pkv.copy_blocks(kd, vd, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    out = torch.empty((b, hq, d), dtype=torch.float16, device="cuda")
    ws = pkv.make_step_workspace(b, hq, maxb * bs, device="cuda")
    pkv.decode_step(out, torch.from_numpy(q).cuda(), torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(),
                    kd, vd, bt.cuda(), torch.from_numpy(lens).cuda(), scale, workspace=ws)
    assert max_err(out, ref) <= ATTN_TOL
    # the caches match the oracle's bit for bit after copy + append
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), ko.view(np.uint16))
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), vo.view(np.uint16))
    assert_no_device_error()
    for r in rows:
        pool.free_table(r, ctx + 1, bs)
    assert pool.num_free() == nb


def test_swap_out_to_pinned_host_and_back():
    """A request's blocks go to a page-locked host pool (the copy kernel writes host memory
    directly) and come back into other device blocks; the host pool matches the oracle's copy bit
    for bit and the decode output over the new table is bit-identical to the one before."""
    rng = np.random.default_rng(77)
    hq, hkv, d, bs, nb, nh = 16, 4, 128, 16, 64, 24
    ctxs = [300, 170]
    kc = torch.from_numpy(rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)).cuda()
    vc = torch.from_numpy(rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)).cuda()
    kh = torch.zeros((nh, hkv, bs, d), dtype=torch.float16).pin_memory()
    vh = torch.zeros((nh, hkv, bs, d), dtype=torch.float16).pin_memory()
    dev_pool, host_pool = pkv.BlockPool(nb, seed=11), pkv.BlockPool(nh, seed=12)
    maxb = -(-max(ctxs) // bs)
    rows = [torch.full((maxb,), -1, dtype=torch.int32) for _ in ctxs]
    for r, c in zip(rows, ctxs):
        dev_pool.reserve(r, 0, c, bs)
    q = torch.from_numpy(rng.standard_normal((2, hq, d)).astype(np.float16)).cuda()
    lens = torch.tensor(ctxs, dtype=torch.int32, device="cuda")
    scale = d ** -0.5

    def decode():
        out = torch.empty_like(q)
        pkv.decode_attention(out, q, kc, vc, torch.stack(rows).cuda(), lens, scale)
        return out

    before = decode()
    host_before = (kc.cpu().numpy(), vc.cpu().numpy())
    # swap request 0 out: ids passed in pinned host memory
    src, dst = dev_pool.swap_to(host_pool, rows[0], ctxs[0], bs)
    pkv.copy_blocks_between(kh, vh, kc, vc, src.pin_memory(), dst.pin_memory(), device="cuda")
    torch.cuda.synchronize()
    ko, vo = np.zeros(kh.shape, np.float16), np.zeros(vh.shape, np.float16)
    oracle.copy_blocks_between(ko, vo, host_before[0], host_before[1], src.numpy(), dst.numpy())
    assert np.array_equal(kh.numpy().view(np.uint16), ko.view(np.uint16))
    assert np.array_equal(vh.numpy().view(np.uint16), vo.view(np.uint16))
    # the freed device blocks are reused by someone else
    kc[src.long().cuda()] = float("nan")
    vc[src.long().cuda()] = float("nan")
    # swap back in (ids on the device this time) to whatever blocks the pool hands out
    src2, dst2 = host_pool.swap_to(dev_pool, rows[0], ctxs[0], bs)
    pkv.copy_blocks_between(kc, vc, kh, vh, src2.cuda(), dst2.cuda())
    after = decode()
    assert torch.equal(before, after)
    assert_no_device_error()
