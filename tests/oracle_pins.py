"""Pins of the float64 CPU oracle against things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with

* the pages' own worked example (the KV-size formula),
* hand-worked fixtures under tests/golden/,
* a textbook contiguous attention (scipy's softmax and numpy matmuls over
  un-paged K/V, scattered into the paged pool block by block here),
* closed forms (one key -> v; equal keys or q = 0 -> mean of V; a dominant
  key -> its v; an empty context -> 0; merge of one partition -> identity),
* a pure-Python brute force with math.exp and math.fsum,
* invariances the definition implies (relabelling physical block ids, GQA
  equal to MHA with K/V repeated per group, split size).

``tests/test_oracle.py`` runs them on the oracle; ``tests/test_oracle_mutants.py``
runs them on deliberately broken copies of the oracle to show that a
plausible slip (a dropped term, a wrong sign or index, a swapped operand) is
caught by at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import softmax

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


# ------------------------------------------------------------------ test-side constructions

def random_contiguous(rng, ctxs, hkv, d, value_scale=1.0):
    """Per-request contiguous K, V: list of fp16 arrays [Hkv, ctx_b, D]."""
    ks = [(rng.standard_normal((hkv, c, d)) * value_scale).astype(np.float16) for c in ctxs]
    vs = [rng.standard_normal((hkv, c, d)).astype(np.float16) for c in ctxs]
    return ks, vs


def scatter_to_pool(ks, vs, bs, rng, extra_blocks=2):
    """Store contiguous per-request K/V in a paged pool [NB, Hkv, bs, D] whose physical
    block ids are a random permutation; block i of request b holds its tokens
    [i*bs, (i+1)*bs).  Unused pool memory is filled with NaN so that any read outside the
    context shows up."""
    hkv, d = ks[0].shape[0], ks[0].shape[2]
    need = [-(-k.shape[1] // bs) for k in ks]
    nb = sum(need) + extra_blocks
    perm = rng.permutation(nb)
    kpool = np.full((nb, hkv, bs, d), np.nan, np.float16)
    vpool = np.full((nb, hkv, bs, d), np.nan, np.float16)
    bt = np.full((len(ks), max(1, max(need))), -1, np.int32)
    nxt = 0
    for b, (k, v) in enumerate(zip(ks, vs)):
        for i in range(need[b]):
            phys = perm[nxt]
            nxt += 1
            bt[b, i] = phys
            lo, hi = i * bs, min((i + 1) * bs, k.shape[1])
            kpool[phys, :, :hi - lo, :] = k[:, lo:hi, :]
            vpool[phys, :, :hi - lo, :] = v[:, lo:hi, :]
    ctx = np.array([k.shape[1] for k in ks], np.int32)
    return kpool, vpool, bt, ctx


def textbook_attention(q, ks, vs, scale):
    """softmax(scale q K^T) V per request and q head on contiguous float64 K/V."""
    b, hq, d = q.shape
    hkv = ks[0].shape[0]
    g = hq // hkv
    out = np.zeros((b, hq, d))
    for i in range(b):
        if ks[i].shape[1] == 0:
            continue
        for h in range(hq):
            kk = ks[i][h // g].astype(np.float64)
            vv = vs[i][h // g].astype(np.float64)
            w = softmax(scale * (kk @ q[i, h].astype(np.float64)))
            out[i, h] = w @ vv
    return out


# ------------------------------------------------------------------ pins

def pin_half_decoding(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_kv_bytes_worked_example(orc):
    g = golden("kv_cache_bytes.json")
    got = orc.kv_cache_bytes(g["batch"], g["layers"], g["heads"], g["head_dim"], g["tokens"],
                             g["elem_bytes"])
    assert got == g["expected_bytes"]
    assert round(got / 1e9, 1) == g["printed_gb"]
    # the batch factor multiplies; a pool of S tokens per layer and kv head is NB*bs*D*2 per tensor
    assert orc.kv_cache_bytes(8, 32, 8, 128, 2048, 2) == 8 * orc.kv_cache_bytes(1, 32, 8, 128,
                                                                                  2048, 2)
    nb, hkv, bs, d = 128, 8, 16, 128
    assert orc.kv_cache_bytes(1, 1, hkv, d, nb * bs, 2) == 2 * nb * hkv * bs * d * 2


def pin_append_golden(orc):
    g = golden("append_tiny.json")
    kc = np.array(g["k_cache_before"], np.float16)
    vc = np.array(g["v_cache_before"], np.float16)
    orc.append(kc, vc, np.array(g["slot_mapping"], np.int64),
               np.array(g["k_new"], np.float16), np.array(g["v_new"], np.float16))
    assert np.array_equal(kc, np.array(g["k_cache_after"], np.float16))
    assert np.array_equal(vc, np.array(g["v_cache_after"], np.float16))


def pin_copy_blocks_golden(orc):
    g = golden("copy_blocks_tiny.json")
    kc = np.array(g["k_cache_before"], np.float16)
    vc = np.array(g["v_cache_before"], np.float16)
    orc.copy_blocks(kc, vc, g["src"], g["dst"])
    assert np.array_equal(kc, np.array(g["k_cache_after"], np.float16))
    assert np.array_equal(vc, np.array(g["v_cache_after"], np.float16))


def pin_copy_blocks_between_golden(orc):
    """The same hand-worked pool copied into a second, 2-block pool (swap out): the destination
    receives source blocks 3 and 0 as its blocks 0 and 1; the source is left as it was."""
    g = golden("copy_blocks_tiny.json")
    sk = np.array(g["k_cache_before"], np.float16)
    sv = np.array(g["v_cache_before"], np.float16)
    dk = np.zeros((2,) + sk.shape[1:], np.float16)
    dv = np.zeros_like(dk)
    orc.copy_blocks_between(dk, dv, sk, sv, [3, 0], [0, 1])
    assert np.array_equal(dk, np.array([g["k_cache_before"][3], g["k_cache_before"][0]], np.float16))
    assert np.array_equal(dv, np.array([g["v_cache_before"][3], g["v_cache_before"][0]], np.float16))
    assert np.array_equal(sk, np.array(g["k_cache_before"], np.float16))


def pin_copy_on_write_keeps_attention(orc):
    """A request whose table points at a copied block must attend exactly as before the copy,
    and appending into the copy must leave the original block's readers unchanged."""
    rng = np.random.default_rng(11)
    hkv, d, bs, ctx = 2, 16, 4, 10
    ks, vs = random_contiguous(rng, [ctx, ctx], hkv, d)
    ks[1], vs[1] = ks[0].copy(), vs[0].copy()
    kpool, vpool, bt, _ = scatter_to_pool(ks, vs, bs, rng, extra_blocks=3)
    bt[1] = bt[0]                                     # request 1 forks request 0
    q = rng.standard_normal((2, 2 * hkv, d)).astype(np.float16)
    ctxs = np.array([ctx, ctx], np.int32)
    before = orc.decode(q, kpool, vpool, bt, ctxs, 0.25)
    free = [i for i in range(kpool.shape[0]) if i not in set(bt[0].tolist())]
    last = ctx // bs                                  # block holding position ctx (partially full)
    orc.copy_blocks(kpool, vpool, [int(bt[1, last])], [free[0]])
    bt[1, last] = free[0]
    after = orc.decode(q, kpool, vpool, bt, ctxs, 0.25)
    assert np.array_equal(before, after)
    # request 1 appends its own token into the copy; request 0 is unaffected
    k_new = rng.standard_normal((1, hkv, d)).astype(np.float16)
    v_new = rng.standard_normal((1, hkv, d)).astype(np.float16)
    orc.append(kpool, vpool, np.array([free[0] * bs + ctx % bs], np.int64), k_new, v_new)
    ctxs2 = np.array([ctx, ctx + 1], np.int32)
    out = orc.decode(q, kpool, vpool, bt, ctxs2, 0.25)
    assert np.array_equal(out[0], before[0])
    ref = textbook_attention(q[1:], [np.concatenate([ks[1], k_new.transpose(1, 0, 2)], axis=1)],
                             [np.concatenate([vs[1], v_new.transpose(1, 0, 2)], axis=1)], 0.25)
    assert np.abs(out[1] - ref[0]).max() < 1e-12


def pin_quantize_golden(orc):
    g = golden("quantize_k_rows.json")
    for row in g["rows"]:
        codes, sc = orc.quantize_k_row(np.array(row["k"], np.float16))
        assert sc == np.float32(row["scale"]), (row["note"], sc)
        assert codes.tolist() == row["codes"], (row["note"], codes)


def pin_quantize_properties(orc):
    """On random rows: every code in [-127, 127], the largest |k| maps to +-127, the rounding
    error is at most half a step (plus the float32 quotient's rounding), and doubling the row
    doubles the scale and keeps the codes."""
    rng = np.random.default_rng(5)
    for i in range(50):
        k = (rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 2)).astype(np.float16)
        codes, sc = orc.quantize_k_row(k)
        kd = k.astype(np.float64)
        assert np.abs(codes.astype(np.int32)).max() == 127
        assert codes[np.argmax(np.abs(kd))] == (127 if kd[np.argmax(np.abs(kd))] > 0 else -127)
        assert np.all(np.abs(kd - codes * np.float64(sc)) <= np.float64(sc) * (0.5 + 1e-5))
        codes2, sc2 = orc.quantize_k_row((k.astype(np.float32) * 2).astype(np.float16))
        assert sc2 == 2 * sc and np.array_equal(codes2, codes)


def pin_append_quant_k(orc):
    """The int8 append stores, per (token, kv head), the quantiser's codes and scale, and V bit
    for bit as the fp16 append does; negative slots write nothing."""
    rng = np.random.default_rng(6)
    nb, hkv, bs, d, t = 5, 3, 4, 16, 6
    codes = np.zeros((nb, hkv, bs, d), np.int8)
    scales = np.full((nb, hkv, bs), -1.0, np.float32)
    vq = np.zeros((nb, hkv, bs, d), np.float16)
    vref = vq.copy()
    kref = vq.copy()
    slots = np.array([7, -1, 0, 19, 12, -5], np.int64)
    kn = rng.standard_normal((t, hkv, d)).astype(np.float16)
    vn = rng.standard_normal((t, hkv, d)).astype(np.float16)
    orc.append_quant_k(codes, scales, vq, slots, kn, vn)
    orc.append(kref, vref, slots, kn, vn)
    assert np.array_equal(vq.view(np.uint16), vref.view(np.uint16))
    for ti, sl in enumerate(slots):
        if sl < 0:
            continue
        for j in range(hkv):
            c, sc = orc.quantize_k_row(kn[ti, j])
            assert np.array_equal(codes[sl // bs, j, sl % bs], c) and scales[sl // bs, j, sl % bs] == sc
    written = np.zeros((nb, bs), bool)
    for sl in slots[slots >= 0]:
        written[sl // bs, sl % bs] = True
    assert np.all(scales.transpose(0, 2, 1)[~written] == -1.0)
    assert not codes.transpose(0, 2, 1, 3)[~written].any()


def pin_decode_quant_k(orc):
    """With scales that are powers of two the dequantised keys are exact fp16 values: decode over
    the int8 cache must equal decode over that fp16 cache; with arbitrary scales it must equal a
    textbook contiguous attention over the dequantised keys."""
    rng = np.random.default_rng(8)
    hq, hkv, d, bs = 4, 2, 32, 4
    ctxs = [9, 1, 0, 16]
    nb = 20
    codes = rng.integers(-127, 128, size=(nb, hkv, bs, d)).astype(np.int8)
    scales = (2.0 ** rng.integers(-9, -4, size=(nb, hkv, bs))).astype(np.float32)
    v = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    bt = rng.permutation(nb)[:16].reshape(4, 4).astype(np.int32)
    q = rng.standard_normal((4, hq, d)).astype(np.float16)
    ctx = np.array(ctxs, np.int32)
    kf16 = (codes.astype(np.float64) * scales[..., None]).astype(np.float16)
    assert np.array_equal(kf16.astype(np.float64), codes.astype(np.float64) * scales[..., None])
    got = orc.decode_quant_k(q, codes, scales, v, bt, ctx, 0.3)
    ref = orc.decode(q, kf16, v, bt, ctx, 0.3)
    assert np.abs(got - ref).max() <= 1e-15
    scales = rng.uniform(1e-3, 5e-2, size=(nb, hkv, bs)).astype(np.float32)
    got = orc.decode_quant_k(q, codes, scales, v, bt, ctx, 0.3)
    kdq = codes.astype(np.float64) * scales[..., None].astype(np.float64)
    ks, vs = [], []
    for b, c in enumerate(ctxs):
        rows_k = [kdq[bt[b, p // bs], :, p % bs] for p in range(c)]
        rows_v = [v[bt[b, p // bs], :, p % bs] for p in range(c)]
        ks.append(np.stack(rows_k, 1) if c else np.zeros((hkv, 0, d)))
        vs.append(np.stack(rows_v, 1) if c else np.zeros((hkv, 0, d), np.float16))
    ref = textbook_attention(q, ks, vs, 0.3)
    assert np.abs(got - ref).max() <= 1e-12


def pin_quant_kv(orc):
    """int8 K + V: the append stores the quantiser's codes and scales for both rows; with scales
    that are powers of two the decode equals the fp16 decode of the exact dequantised cache, and
    with the values' codes and scales it equals the int8-key decode over those dequantised values."""
    rng = np.random.default_rng(31)
    nb, hkv, bs, d = 6, 2, 4, 16
    kc = np.zeros((nb, hkv, bs, d), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nb, hkv, bs), np.float32)
    vs = np.zeros_like(ks)
    slots = np.array([3, 22, -1, 9], np.int64)
    kn = rng.standard_normal((4, hkv, d)).astype(np.float16)
    vn = rng.standard_normal((4, hkv, d)).astype(np.float16)
    orc.append_quant_kv(kc, ks, vc, vs, slots, kn, vn)
    for ti, sl in enumerate(slots):
        if sl < 0:
            continue
        for j in range(hkv):
            c, sc = orc.quantize_k_row(vn[ti, j])
            assert np.array_equal(vc[sl // bs, j, sl % bs], c) and vs[sl // bs, j, sl % bs] == sc
            c, sc = orc.quantize_k_row(kn[ti, j])
            assert np.array_equal(kc[sl // bs, j, sl % bs], c) and ks[sl // bs, j, sl % bs] == sc
    hq, ctxs = 4, [7, 0, 16, 1]
    nb = 20
    kc = rng.integers(-127, 128, size=(nb, hkv, bs, d)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(nb, hkv, bs, d)).astype(np.int8)
    ks = (2.0 ** rng.integers(-9, -4, size=(nb, hkv, bs))).astype(np.float32)
    vs = (2.0 ** rng.integers(-9, -4, size=(nb, hkv, bs))).astype(np.float32)
    bt = rng.permutation(nb)[:16].reshape(4, 4).astype(np.int32)
    q = rng.standard_normal((4, hq, d)).astype(np.float16)
    ctx = np.array(ctxs, np.int32)
    k16 = (kc.astype(np.float64) * ks[..., None]).astype(np.float16)
    v16 = (vc.astype(np.float64) * vs[..., None]).astype(np.float16)
    got = orc.decode_quant_kv(q, kc, ks, vc, vs, bt, ctx, 0.3)
    assert np.abs(got - orc.decode(q, k16, v16, bt, ctx, 0.3)).max() <= 1e-15
    vs = rng.uniform(1e-3, 5e-2, size=(nb, hkv, bs)).astype(np.float32)
    vdq = vc.astype(np.float64) * vs[..., None].astype(np.float64)
    got = orc.decode_quant_kv(q, kc, ks, vc, vs, bt, ctx, 0.3)
    ks_rows = [[kc[bt[b, p // bs], :, p % bs].astype(np.float64) * ks[bt[b, p // bs], :, p % bs][:, None]
                for p in range(c)] for b, c in enumerate(ctxs)]
    kk = [np.stack(r, 1) if r else np.zeros((hkv, 0, d)) for r in ks_rows]
    vv = [np.stack([vdq[bt[b, p // bs], :, p % bs] for p in range(c)], 1) if c else np.zeros((hkv, 0, d))
          for b, c in enumerate(ctxs)]
    ref = textbook_attention(q, kk, vv, 0.3)
    assert np.abs(got - ref).max() <= 1e-12


def _torch_e4m3_values():
    """float64 values of the 256 E4M3 codes by torch's own float8_e4m3fn type (a library
    decoder, not the oracle's); None where torch lacks the type."""
    import torch
    if not hasattr(torch, "float8_e4m3fn"):
        return None
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def pin_e4m3_decoding(orc):
    """All 256 codes against torch's float8_e4m3fn, and the format's landmarks by hand: 0, the
    smallest subnormal 2^-9, the smallest normal 2^-6, 1.0, the largest finite 448, -0, NaN."""
    got = orc.e4m3_to_double(np.arange(256, dtype=np.uint8))
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3c: 1.5,
            0x77: 240.0, 0x7e: 448.0, 0xb8: -1.0, 0xfe: -448.0}
    for c, v in hand.items():
        assert got[c] == v, (hex(c), got[c])
    assert got[0x80] == 0.0 and np.signbit(got[0x80])
    assert np.isnan(got[0x7f]) and np.isnan(got[0xff]) and np.isfinite(np.delete(got, [0x7f, 0xff])).all()
    ref = _torch_e4m3_values()
    if ref is not None:
        both_nan = np.isnan(ref) & np.isnan(got)
        assert np.array_equal(got[~both_nan], ref[~both_nan]) and both_nan.sum() == 2


def pin_e4m3_encoding(orc):
    """Every finite code's value encodes back to that code; a point halfway between neighbours
    goes to the even code and a hair off it to the nearer one; magnitudes past 448 clamp to 448;
    random float32 values within +-448 agree with torch's round-to-nearest-even conversion."""
    vals = orc.e4m3_to_double(np.arange(0x7f, dtype=np.uint8))
    assert np.array_equal(orc.e4m3_from_float(vals.astype(np.float32)), np.arange(0x7f, dtype=np.uint8))
    assert np.array_equal(orc.e4m3_from_float(-vals[1:].astype(np.float32)), np.arange(1, 0x7f, dtype=np.uint8) | 0x80)
    mid = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    lower = np.arange(0x7e, dtype=np.uint8)
    even = np.where(lower % 2 == 0, lower, lower + 1).astype(np.uint8)
    assert np.array_equal(orc.e4m3_from_float(mid), even)
    assert np.array_equal(orc.e4m3_from_float(np.nextafter(mid, np.float32(0))), lower)
    assert np.array_equal(orc.e4m3_from_float(np.nextafter(mid, np.float32(1e9))), lower + 1)
    assert orc.e4m3_from_float(np.float32(1e6)) == 0x7e and orc.e4m3_from_float(np.float32(-470.0)) == 0xfe
    import torch
    if hasattr(torch, "float8_e4m3fn"):
        rng = np.random.default_rng(17)
        y = (rng.standard_normal(4000) * 10.0 ** rng.uniform(-4, 2.6, 4000)).astype(np.float32)
        y = np.clip(y, -448, 448)
        ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(orc.e4m3_from_float(y), ref)


def pin_quantize_fp8_golden(orc):
    g = golden("quantize_fp8_rows.json")
    for row in g["rows"]:
        codes, sc = orc.quantize_fp8_row(np.array(row["x"], np.float16))
        assert sc == np.float32(row["scale"]), (row["note"], sc)
        assert codes.tolist() == row["codes"], (row["note"], codes)


def pin_quantize_fp8_properties(orc):
    """On random rows: the largest |x| maps to +-448, every code's value is within half a code
    spacing of x / s, the codes equal torch's conversion of the float32 quotients, and doubling
    the row doubles the scale and keeps the codes."""
    import torch
    rng = np.random.default_rng(19)
    for i in range(40):
        x = (rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 2)).astype(np.float16)
        codes, sc = orc.quantize_fp8_row(x)
        xd = x.astype(np.float64)
        i_max = np.argmax(np.abs(xd))
        assert codes[i_max] == (0x7e if xd[i_max] > 0 else 0xfe)
        y = (x.astype(np.float32) / sc).astype(np.float64)
        v = orc.e4m3_to_double(codes)
        spacing = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6))) - 3)
        assert np.all(np.abs(y - v) <= spacing / 2)
        if hasattr(torch, "float8_e4m3fn"):
            q = torch.from_numpy(x.astype(np.float32) / np.float32(sc)).to(torch.float8_e4m3fn)
            assert np.array_equal(q.view(torch.uint8).numpy(), codes)
        codes2, sc2 = orc.quantize_fp8_row((x.astype(np.float32) * 2).astype(np.float16))
        assert sc2 == 2 * sc and np.array_equal(codes2, codes)


def pin_fp8_kv(orc):
    """fp8 K + V: the append stores the quantiser's codes and scales for both rows and nothing
    else; with power-of-two scales the dequantised cache is exactly fp16 and the decode equals the
    fp16 decode of it; with arbitrary scales it equals a textbook attention over the cache
    dequantised through torch's float8 decoder."""
    import torch
    rng = np.random.default_rng(37)
    nb, hkv, bs, d = 6, 2, 4, 16
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.full((nb, hkv, bs), -1.0, np.float32)
    vs = ks.copy()
    slots = np.array([3, 22, -1, 9], np.int64)
    kn = rng.standard_normal((4, hkv, d)).astype(np.float16)
    vn = rng.standard_normal((4, hkv, d)).astype(np.float16)
    orc.append_fp8_kv(kc, ks, vc, vs, slots, kn, vn)
    written = np.zeros((nb, bs), bool)
    for ti, sl in enumerate(slots):
        if sl < 0:
            continue
        written[sl // bs, sl % bs] = True
        for j in range(hkv):
            c, sc = orc.quantize_fp8_row(vn[ti, j])
            assert np.array_equal(vc[sl // bs, j, sl % bs], c) and vs[sl // bs, j, sl % bs] == sc
            c, sc = orc.quantize_fp8_row(kn[ti, j])
            assert np.array_equal(kc[sl // bs, j, sl % bs], c) and ks[sl // bs, j, sl % bs] == sc
    assert np.all(ks.transpose(0, 2, 1)[~written] == -1.0) and not vc.transpose(0, 2, 1, 3)[~written].any()
    hq, ctxs = 4, [7, 0, 16, 1]
    nb = 20
    finite = np.delete(np.arange(256), [0x7f, 0xff])
    kc = rng.choice(finite, size=(nb, hkv, bs, d)).astype(np.uint8)
    vc = rng.choice(finite, size=(nb, hkv, bs, d)).astype(np.uint8)
    ks = (2.0 ** rng.integers(-9, -4, size=(nb, hkv, bs))).astype(np.float32)
    vs = (2.0 ** rng.integers(-9, -4, size=(nb, hkv, bs))).astype(np.float32)
    bt = rng.permutation(nb)[:16].reshape(4, 4).astype(np.int32)
    q = rng.standard_normal((4, hq, d)).astype(np.float16)
    ctx = np.array(ctxs, np.int32)
    table = _torch_e4m3_values()
    if table is None:
        table = orc.e4m3_to_double(np.arange(256, dtype=np.uint8))
    k64 = table[kc] * ks[..., None]
    v64 = table[vc] * vs[..., None]
    k16, v16 = k64.astype(np.float16), v64.astype(np.float16)
    assert np.array_equal(k16.astype(np.float64), k64) and np.array_equal(v16.astype(np.float64), v64)
    got = orc.decode_fp8_kv(q, kc, ks, vc, vs, bt, ctx, 0.3)
    assert np.abs(got - orc.decode(q, k16, v16, bt, ctx, 0.3)).max() <= 1e-15
    ks = rng.uniform(1e-3, 5e-2, size=(nb, hkv, bs)).astype(np.float32)
    vs = rng.uniform(1e-3, 5e-2, size=(nb, hkv, bs)).astype(np.float32)
    k64 = table[kc] * ks[..., None].astype(np.float64)
    v64 = table[vc] * vs[..., None].astype(np.float64)
    got = orc.decode_fp8_kv(q, kc, ks, vc, vs, bt, ctx, 0.3)
    kk = [np.stack([k64[bt[b, p // bs], :, p % bs] for p in range(c)], 1) if c else np.zeros((hkv, 0, d))
          for b, c in enumerate(ctxs)]
    vv = [np.stack([v64[bt[b, p // bs], :, p % bs] for p in range(c)], 1) if c else np.zeros((hkv, 0, d))
          for b, c in enumerate(ctxs)]
    ref = textbook_attention(q, kk, vv, 0.3)
    assert np.abs(got - ref).max() <= 1e-12


def pin_decode_multi_causal(orc):
    """Several new tokens per request: a textbook causal attention (scipy softmax over the
    scores with every later position masked) on contiguous K/V, and row by row the single-token
    decode with the context cut at that row's position."""
    rng = np.random.default_rng(21)
    hq, hkv, d, bs = 4, 2, 16, 4
    ctxs, ns = [9, 5, 12, 3], [3, 1, 4, 3]
    ks, vs = random_contiguous(rng, ctxs, hkv, d)
    kpool, vpool, bt, ctx = scatter_to_pool(ks, vs, bs, rng)
    qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    q = rng.standard_normal((qs[-1], hq, d)).astype(np.float16)
    got = orc.decode_multi(q, kpool, vpool, bt, ctx, qs, 0.3)
    g = hq // hkv
    for b, (c, n) in enumerate(zip(ctxs, ns)):
        for i in range(n):
            t = qs[b] + i
            pos = c - n + i
            for h in range(hq):
                kk = ks[b][h // g].astype(np.float64)
                vv = vs[b][h // g].astype(np.float64)
                sc = 0.3 * (kk @ q[t, h].astype(np.float64))
                sc[pos + 1:] = -np.inf
                assert np.abs(got[t, h] - softmax(sc) @ vv).max() <= 1e-12
            cut = ctx.copy()
            cut[b] = pos + 1
            one = orc.decode(q[t:t + 1], kpool, vpool, bt[b:b + 1], cut[b:b + 1], 0.3)
            assert np.abs(got[t] - one[0]).max() <= 1e-15


def pin_slot_mapping_by_enumeration(orc):
    """Walk every block table in order, naming each pool slot by the (request, position)
    stored there; the slot mapping must be the inverse of that enumeration."""
    rng = np.random.default_rng(11)
    for bs in (1, 2, 16, 64):
        ctxs = [0, 1, bs, 3 * bs + 1, 5 * bs - 1]
        need = [-(-c // bs) for c in ctxs]
        nb = sum(need) + 3
        perm = rng.permutation(nb)
        bt = np.full((len(ctxs), max(need)), -1, np.int32)
        owner = {}
        nxt = 0
        for b, n in enumerate(need):
            for i in range(n):
                bt[b, i] = perm[nxt]
                for o in range(bs):
                    owner[(b, i * bs + o)] = int(perm[nxt]) * bs + o
                nxt += 1
        for b, c in enumerate(ctxs):
            pos = np.full(len(ctxs), -1, np.int32)
            for p in range(c):
                pos[b] = p
                got = orc.slot_mapping(bt, pos, bs)
                assert got[b] == owner[(b, p)]
                assert all(got[i] == -1 for i in range(len(ctxs)) if i != b)


def pin_two_keys_golden(orc):
    g = golden("attention_two_keys.json")
    out = orc.decode(np.array(g["q"], np.float16), np.array(g["k_cache"], np.float16),
                     np.array(g["v_cache"], np.float16), np.array(g["block_tables"], np.int32),
                     np.array(g["context_lens"], np.int32), g["scale"])
    assert np.allclose(out, np.array(g["expected_out"]), rtol=0, atol=g["tolerance"])


def pin_textbook_contiguous(orc):
    rng = np.random.default_rng(3)
    for bs, hq, hkv, d, ctxs in [(16, 4, 2, 128, [1, 15, 16, 17, 100]),
                                 (2, 3, 3, 8, [5, 2, 9]),
                                 (64, 8, 1, 64, [200, 64, 1])]:
        ks, vs = random_contiguous(rng, ctxs, hkv, d)
        q = rng.standard_normal((len(ctxs), hq, d)).astype(np.float16)
        kp, vp, bt, ctx = scatter_to_pool(ks, vs, bs, rng)
        scale = 1.0 / math.sqrt(d)
        got = orc.decode(q, kp, vp, bt, ctx, scale)
        ref = textbook_attention(q, ks, vs, scale)
        assert np.abs(got - ref).max() < 1e-12


def pin_one_key_is_v(orc):
    rng = np.random.default_rng(4)
    ks, vs = random_contiguous(rng, [1, 1], 2, 16, value_scale=5.0)
    q = rng.standard_normal((2, 4, 16)).astype(np.float16)
    kp, vp, bt, ctx = scatter_to_pool(ks, vs, 4, rng)
    got = orc.decode(q, kp, vp, bt, ctx, 0.25)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(got[b, h], vs[b][h // 2, 0].astype(np.float64))


def pin_uniform_scores_mean_v(orc):
    rng = np.random.default_rng(5)
    ctxs = [37, 5]
    # (a) every key identical -> all scores equal -> out = mean of V
    k_row = rng.standard_normal(32).astype(np.float16)
    ks = [np.broadcast_to(k_row, (1, c, 32)).copy() for c in ctxs]
    vs = [rng.standard_normal((1, c, 32)).astype(np.float16) for c in ctxs]
    q = rng.standard_normal((2, 1, 32)).astype(np.float16)
    kp, vp, bt, ctx = scatter_to_pool(ks, vs, 8, rng)
    got = orc.decode(q, kp, vp, bt, ctx, 0.3)
    for b in range(2):
        assert np.abs(got[b, 0] - vs[b][0].astype(np.float64).mean(axis=0)).max() < 1e-14
    # (b) q = 0 -> all scores zero -> out = mean of V, whatever K is
    ks2, vs2 = random_contiguous(rng, ctxs, 1, 32, value_scale=3.0)
    kp, vp, bt, ctx = scatter_to_pool(ks2, vs2, 8, rng)
    got = orc.decode(np.zeros((2, 1, 32), np.float16), kp, vp, bt, ctx, 0.3)
    for b in range(2):
        assert np.abs(got[b, 0] - vs2[b][0].astype(np.float64).mean(axis=0)).max() < 1e-14


def pin_dominant_key(orc):
    rng = np.random.default_rng(6)
    d, c = 8, 20
    k = (rng.standard_normal((1, c, d)) * 0.1).astype(np.float16)
    k[0, 13] = 0
    k[0, 13, 2] = 8.0
    v = rng.standard_normal((1, c, d)).astype(np.float16)
    q = np.zeros((1, 1, d), np.float16)
    q[0, 0, 2] = 8.0
    kp, vp, bt, ctx = scatter_to_pool([k], [v], 4, rng)
    got = orc.decode(q, kp, vp, bt, ctx, 1.0)          # score 64 vs |others| < ~3
    assert np.abs(got[0, 0] - v[0, 13].astype(np.float64)).max() < 1e-20


def pin_block_relabel_invariance(orc):
    rng = np.random.default_rng(7)
    ks, vs = random_contiguous(rng, [33, 7, 64], 2, 32)
    q = rng.standard_normal((3, 4, 32)).astype(np.float16)
    kp, vp, bt, ctx = scatter_to_pool(ks, vs, 16, rng)
    base = orc.decode(q, kp, vp, bt, ctx, 0.2)
    relabel = rng.permutation(kp.shape[0])          # new id of old block i is relabel[i]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[relabel] = kp
    vp2[relabel] = vp
    bt2 = np.where(bt >= 0, relabel[np.maximum(bt, 0)], -1).astype(np.int32)
    again = orc.decode(q, kp2, vp2, bt2, ctx, 0.2)
    assert np.array_equal(base, again)


def pin_gqa_is_repeated_mha(orc):
    rng = np.random.default_rng(8)
    g = 4
    ks, vs = random_contiguous(rng, [21, 50], 2, 16)
    q = rng.standard_normal((2, 2 * g, 16)).astype(np.float16)
    kp, vp, bt, ctx = scatter_to_pool(ks, vs, 8, rng)
    gqa = orc.decode(q, kp, vp, bt, ctx, 0.25)
    ks_r = [np.repeat(k, g, axis=0) for k in ks]
    vs_r = [np.repeat(v, g, axis=0) for v in vs]
    kp_r, vp_r, bt_r, ctx_r = scatter_to_pool(ks_r, vs_r, 8, rng)
    mha = orc.decode(q, kp_r, vp_r, bt_r, ctx_r, 0.25)
    assert np.abs(gqa - mha).max() < 1e-15


def pin_brute_force_python(orc):
    rng = np.random.default_rng(9)
    for trial in range(20):
        ctxs = [int(x) for x in rng.integers(1, 6, size=2)]
        ks, vs = random_contiguous(rng, ctxs, 1, 4)
        q = rng.standard_normal((2, 2, 4)).astype(np.float16)
        kp, vp, bt, ctx = scatter_to_pool(ks, vs, 2, rng)
        scale = 0.7
        got = orc.decode(q, kp, vp, bt, ctx, scale)
        for b in range(2):
            for h in range(2):
                qq = [float(x) for x in q[b, h]]
                sc = [scale * math.fsum(qq[d] * float(ks[b][0, p, d]) for d in range(4))
                      for p in range(ctxs[b])]
                mx = max(sc)
                w = [math.exp(s - mx) for s in sc]
                tot = math.fsum(w)
                for d in range(4):
                    ref = math.fsum(w[p] * float(vs[b][0, p, d]) for p in range(ctxs[b])) / tot
                    assert abs(got[b, h, d] - ref) <= 1e-14 * max(1.0, abs(ref))


def pin_empty_context(orc):
    rng = np.random.default_rng(10)
    ks, vs = random_contiguous(rng, [0, 3], 1, 8)
    q = rng.standard_normal((2, 1, 8)).astype(np.float16)
    kp, vp, bt, ctx = scatter_to_pool(ks, vs, 2, rng)
    got = orc.decode(q, kp, vp, bt, ctx, 1.0)
    assert np.array_equal(got[0], np.zeros((1, 8)))
    o, m, l = orc.decode_partition(q, kp, vp, bt, ctx, 1.0, 2, 2)
    assert np.array_equal(orc.merge(o, m, l, ctx, 2)[0], np.zeros((1, 8)))


def pin_partition_merge_is_decode(orc):
    rng = np.random.default_rng(12)
    ctxs = [1, 16, 17, 100, 511, 512, 513, 1300]
    ks, vs = random_contiguous(rng, ctxs, 2, 32, value_scale=2.0)
    q = rng.standard_normal((len(ctxs), 8, 32)).astype(np.float16)
    kp, vp, bt, ctx = scatter_to_pool(ks, vs, 16, rng)
    ref = textbook_attention(q, ks, vs, 0.3)
    for part in (16, 48, 512, 2048):
        maxp = -(-max(ctxs) // part)
        o, m, l = orc.decode_partition(q, kp, vp, bt, ctx, 0.3, part, maxp)
        got = orc.merge(o, m, l, ctx, part)
        assert np.abs(got - ref).max() < 1e-12, part
        # unused partitions are marked empty
        for b, c in enumerate(ctxs):
            np_b = -(-c // part)
            assert np.all(l[b, :, np_b:] == 0) and np.all(np.isneginf(m[b, :, np_b:]))


def pin_partition_statistics(orc):
    """One partition covering the whole context: m is the max score, l = sum exp(s - m),
    o the normalised output -- checked against scores computed here with numpy."""
    rng = np.random.default_rng(13)
    ctxs = [9, 40]
    ks, vs = random_contiguous(rng, ctxs, 1, 16, value_scale=3.0)
    q = rng.standard_normal((2, 2, 16)).astype(np.float16)
    kp, vp, bt, ctx = scatter_to_pool(ks, vs, 4, rng)
    o, m, l = orc.decode_partition(q, kp, vp, bt, ctx, 0.5, 64, 1)
    ref = textbook_attention(q, ks, vs, 0.5)
    for b in range(2):
        for h in range(2):
            s = 0.5 * (ks[b][0].astype(np.float64) @ q[b, h].astype(np.float64))
            assert abs(m[b, h, 0] - s.max()) < 1e-13
            assert abs(l[b, h, 0] - np.exp(s - s.max()).sum()) < 1e-12
            assert np.abs(o[b, h, 0] - ref[b, h]).max() < 1e-12
    # merging a single partition returns it unchanged
    merged = orc.merge(o, m, l, ctx, 64)
    assert np.array_equal(merged, o[:, :, 0, :])


ALL_PINS = [
    pin_half_decoding,
    pin_kv_bytes_worked_example,
    pin_append_golden,
    pin_copy_blocks_golden,
    pin_copy_blocks_between_golden,
    pin_copy_on_write_keeps_attention,
    pin_quantize_golden,
    pin_quantize_properties,
    pin_append_quant_k,
    pin_decode_quant_k,
    pin_decode_multi_causal,
    pin_quant_kv,
    pin_e4m3_decoding,
    pin_e4m3_encoding,
    pin_quantize_fp8_golden,
    pin_quantize_fp8_properties,
    pin_fp8_kv,
    pin_slot_mapping_by_enumeration,
    pin_two_keys_golden,
    pin_textbook_contiguous,
    pin_one_key_is_v,
    pin_uniform_scores_mean_v,
    pin_dominant_key,
    pin_block_relabel_invariance,
    pin_gqa_is_repeated_mha,
    pin_brute_force_python,
    pin_empty_context,
    pin_partition_merge_is_decode,
    pin_partition_statistics,
]
