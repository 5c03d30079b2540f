"""float64 CPU oracle for paged-KV-cache decode attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product library
never imports, links or loads anything here, and this package imports nothing
from the product package.

The arithmetic lives in ``pkv_oracle.c`` (plain C loops in double precision,
compiled with ``-ffp-contract=off`` so that x86 and Arm give the same bits).
This module only builds that file with gcc, loads it with ctypes and moves
numpy arrays in and out.  Every function cites, in ``pkv_oracle.c``, the
passage of the pages it follows:

* ``kv_cache_bytes``  -- "推理优化这件事，为什么值得反复复盘", sec. 4.1
  (2 x L x H x D x S x bytes) and the batch factor of
  "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.1;
* ``slot_mapping``, ``append`` -- in-place append into a paged cache
  ("为什么“推理优化”不是锦上添花", sec. 3.1 and 3.2;
  "LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.3);
* ``decode`` -- read every cached K/V, score, softmax, weighted sum
  ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.2);
* ``decode_partition``, ``merge`` -- the same over consecutive token ranges,
  recombined by the log-sum-exp identity (not on the pages; see the C file);
* ``quantize_k_row``, ``append_quant_k(v)``, ``decode_quant_k(v)`` -- the int8
  cache ("推理优化这件事，为什么值得反复复盘", sec. 4.4);
* ``e4m3_to_double``, ``e4m3_from_float``, ``quantize_fp8_row``,
  ``append_fp8_kv``, ``decode_fp8_kv`` -- the 8-bit floating-point (E4M3) cache
  ("LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 2 and 4.2).

Every function is pinned by ``tests/test_oracle.py`` against something other
than itself (numpy's binary16 decoder, torch's float8_e4m3fn conversions, a
contiguous textbook softmax, closed forms, a pure-Python brute force, the
pages' worked size example, hand-worked goldens).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()

_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i8p = ctypes.POINTER(ctypes.c_int8)
_f32p = ctypes.POINTER(ctypes.c_float)
_u8p = ctypes.POINTER(ctypes.c_uint8)

GCC_FLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c99", "-shared", "-fPIC"]


def compile_source(src: str, out: str) -> str:
    """gcc a C source into a shared object (no FP contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into liboracle.so next to it when missing or stale."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
            compile_source(SOURCE, _LIB)
    return _LIB


def _p(a: np.ndarray, ptr_t):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ptr_t)


def _bits(a: np.ndarray) -> np.ndarray:
    """fp16 (or raw uint16) array -> contiguous uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


class Oracle:
    """numpy front end over one compiled copy of pkv_oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_halves_to_doubles.restype = None
        lib.oracle_halves_to_doubles.argtypes = [_f64p, _u16p, ctypes.c_int64]
        lib.oracle_kv_cache_bytes.restype = ctypes.c_int64
        lib.oracle_kv_cache_bytes.argtypes = [ctypes.c_int64] * 6
        lib.oracle_slot_mapping.restype = None
        lib.oracle_slot_mapping.argtypes = [_i64p, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int]
        lib.oracle_append.restype = None
        lib.oracle_append.argtypes = [_u16p, _u16p, _i64p, _u16p, _u16p] + [ctypes.c_int] * 4
        lib.oracle_decode.restype = None
        lib.oracle_decode.argtypes = ([_f64p, _u16p, _u16p, _u16p, _i32p, _i32p]
                                      + [ctypes.c_int] * 6 + [ctypes.c_double])
        lib.oracle_decode_partition.restype = None
        lib.oracle_decode_partition.argtypes = ([_f64p, _f64p, _f64p, _u16p, _u16p, _u16p,
                                                 _i32p, _i32p] + [ctypes.c_int] * 6
                                                + [ctypes.c_double, ctypes.c_int, ctypes.c_int])
        lib.oracle_copy_blocks.restype = None
        lib.oracle_copy_blocks.argtypes = [_u16p, _u16p, _i32p, _i32p] + [ctypes.c_int] * 4
        lib.oracle_quantize_k_row.restype = None
        lib.oracle_quantize_k_row.argtypes = [_i8p, ctypes.POINTER(ctypes.c_float), _u16p, ctypes.c_int]
        lib.oracle_append_quant_k.restype = None
        lib.oracle_append_quant_k.argtypes = [_i8p, _f32p, _u16p, _i64p, _u16p, _u16p] + [ctypes.c_int] * 4
        lib.oracle_decode_quant_k.restype = None
        lib.oracle_decode_quant_k.argtypes = [_f64p, _u16p, _i8p, _f32p, _u16p, _i32p, _i32p] + \
            [ctypes.c_int] * 6 + [ctypes.c_double]
        lib.oracle_decode_multi.restype = None
        lib.oracle_decode_multi.argtypes = [_f64p, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p] + \
            [ctypes.c_int] * 6 + [ctypes.c_double]
        lib.oracle_copy_blocks_between.restype = None
        lib.oracle_copy_blocks_between.argtypes = [_u16p, _u16p, _u16p, _u16p, _i32p, _i32p] + [ctypes.c_int] * 4
        lib.oracle_append_quant_kv.restype = None
        lib.oracle_append_quant_kv.argtypes = [_i8p, _f32p, _i8p, _f32p, _i64p, _u16p, _u16p] + [ctypes.c_int] * 4
        lib.oracle_decode_quant_kv.restype = None
        lib.oracle_decode_quant_kv.argtypes = [_f64p, _u16p, _i8p, _f32p, _i8p, _f32p, _i32p, _i32p] + \
            [ctypes.c_int] * 6 + [ctypes.c_double]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_quantize_fp8_row.restype = None
        lib.oracle_quantize_fp8_row.argtypes = [_u8p, ctypes.POINTER(ctypes.c_float), _u16p, ctypes.c_int]
        lib.oracle_append_fp8_kv.restype = None
        lib.oracle_append_fp8_kv.argtypes = [_u8p, _f32p, _u8p, _f32p, _i64p, _u16p, _u16p] + [ctypes.c_int] * 4
        lib.oracle_decode_fp8_kv.restype = None
        lib.oracle_decode_fp8_kv.argtypes = [_f64p, _u16p, _u8p, _f32p, _u8p, _f32p, _i32p, _i32p] + \
            [ctypes.c_int] * 6 + [ctypes.c_double]
        lib.oracle_merge.restype = None
        lib.oracle_merge.argtypes = [_f64p, _f64p, _f64p, _f64p, _i32p] + [ctypes.c_int] * 5
        self.lib = lib
        self.path = lib_path

    def half_to_double(self, a: np.ndarray) -> np.ndarray:
        """Decode binary16 values (fp16 or uint16 bit patterns) to float64."""
        bits = _bits(a)
        out = np.empty(bits.shape, np.float64)
        self.lib.oracle_halves_to_doubles(_p(out, _f64p), _p(bits, _u16p), bits.size)
        return out

    def kv_cache_bytes(self, batch: int, layers: int, heads: int, head_dim: int, tokens: int,
                       elem_bytes: int) -> int:
        return int(self.lib.oracle_kv_cache_bytes(batch, layers, heads, head_dim, tokens,
                                                  elem_bytes))

    def slot_mapping(self, block_tables, positions, block_size: int) -> np.ndarray:
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        out = np.empty(pos.shape[0], np.int64)
        self.lib.oracle_slot_mapping(_p(out, _i64p), _p(bt, _i32p), _p(pos, _i32p), pos.shape[0],
                                     bt.shape[1], block_size)
        return out

    def append(self, k_cache: np.ndarray, v_cache: np.ndarray, slots, k_new, v_new) -> None:
        """In place on k_cache / v_cache ([NB, Hkv, bs, D] fp16 or uint16 arrays)."""
        nb, hkv, bs, d = k_cache.shape
        kc, vc = _bits(k_cache), _bits(v_cache)
        assert np.shares_memory(kc, k_cache) and np.shares_memory(vc, v_cache)
        kn, vn = _bits(k_new), _bits(v_new)
        sl = np.ascontiguousarray(slots, dtype=np.int64)
        assert kn.shape == (sl.shape[0], hkv, d) and vn.shape == kn.shape
        self.lib.oracle_append(_p(kc, _u16p), _p(vc, _u16p), _p(sl, _i64p), _p(kn, _u16p),
                               _p(vn, _u16p), sl.shape[0], hkv, d, bs)

    def copy_blocks(self, k_cache: np.ndarray, v_cache: np.ndarray, src, dst) -> None:
        """In place: whole blocks dst[i] <- src[i] of both caches."""
        nb, hkv, bs, d = k_cache.shape
        kc, vc = _bits(k_cache), _bits(v_cache)
        assert np.shares_memory(kc, k_cache) and np.shares_memory(vc, v_cache)
        sr = np.ascontiguousarray(src, dtype=np.int32)
        ds = np.ascontiguousarray(dst, dtype=np.int32)
        self.lib.oracle_copy_blocks(_p(kc, _u16p), _p(vc, _u16p), _p(sr, _i32p), _p(ds, _i32p), sr.shape[0], hkv,
                                    d, bs)

    def copy_blocks_between(self, dst_k: np.ndarray, dst_v: np.ndarray, src_k: np.ndarray, src_v: np.ndarray, src,
                            dst) -> None:
        """In place on dst_k / dst_v: whole blocks dst[i] <- src[i] of the source pools."""
        nb, hkv, bs, d = src_k.shape
        assert dst_k.shape[1:] == src_k.shape[1:] and dst_v.shape == dst_k.shape and src_v.shape == src_k.shape
        dk, dv = _bits(dst_k), _bits(dst_v)
        assert np.shares_memory(dk, dst_k) and np.shares_memory(dv, dst_v)
        sk, sv = _bits(src_k), _bits(src_v)
        sr = np.ascontiguousarray(src, dtype=np.int32)
        ds = np.ascontiguousarray(dst, dtype=np.int32)
        self.lib.oracle_copy_blocks_between(_p(dk, _u16p), _p(dv, _u16p), _p(sk, _u16p), _p(sv, _u16p), _p(sr, _i32p),
                                            _p(ds, _i32p), sr.shape[0], hkv, d, bs)

    def quantize_k_row(self, k_row) -> tuple[np.ndarray, float]:
        """(int8 codes [D], float32 scale) of one fp16 K row."""
        kb = _bits(np.ascontiguousarray(k_row))
        codes = np.empty(kb.shape[0], np.int8)
        sc = ctypes.c_float(0.0)
        self.lib.oracle_quantize_k_row(_p(codes, _i8p), ctypes.byref(sc), _p(kb, _u16p), kb.shape[0])
        return codes, np.float32(sc.value)

    def append_quant_k(self, k_codes: np.ndarray, k_scale: np.ndarray, v_cache: np.ndarray, slots, k_new,
                       v_new) -> None:
        """In place on k_codes (int8 [NB,Hkv,bs,D]), k_scale (float32 [NB,Hkv,bs]) and v_cache (fp16)."""
        nb, hkv, bs, d = k_codes.shape
        assert k_codes.dtype == np.int8 and k_codes.flags.c_contiguous
        assert k_scale.dtype == np.float32 and k_scale.shape == (nb, hkv, bs) and k_scale.flags.c_contiguous
        vc = _bits(v_cache)
        assert np.shares_memory(vc, v_cache)
        kn, vn = _bits(k_new), _bits(v_new)
        sl = np.ascontiguousarray(slots, dtype=np.int64)
        assert kn.shape == (sl.shape[0], hkv, d) and vn.shape == kn.shape
        self.lib.oracle_append_quant_k(_p(k_codes, _i8p), _p(k_scale, _f32p), _p(vc, _u16p), _p(sl, _i64p),
                                       _p(kn, _u16p), _p(vn, _u16p), sl.shape[0], hkv, d, bs)

    def decode_quant_k(self, q, k_codes, k_scale, v_cache, block_tables, context_lens, scale: float) -> np.ndarray:
        """float64 [B, Hq, D] decode over the int8-K / fp16-V cache (keys dequantised exactly)."""
        qb, vc = _bits(q), _bits(v_cache)
        kc = np.ascontiguousarray(k_codes, dtype=np.int8)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        b, hq, d = qb.shape
        nb, hkv, bs, d2 = kc.shape
        assert d2 == d and hq % hkv == 0 and ks.shape == (nb, hkv, bs)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.empty((b, hq, d), np.float64)
        self.lib.oracle_decode_quant_k(_p(out, _f64p), _p(qb, _u16p), _p(kc, _i8p), _p(ks, _f32p), _p(vc, _u16p),
                                       _p(bt, _i32p), _p(cl, _i32p), b, bt.shape[1], hq, hkv, d, bs, float(scale))
        return out

    def append_quant_kv(self, k_codes, k_scale, v_codes, v_scale, slots, k_new, v_new) -> None:
        """In place on the int8 K + V cache: codes int8 [NB,Hkv,bs,D], scales float32 [NB,Hkv,bs]."""
        nb, hkv, bs, d = k_codes.shape
        for a, dt in ((k_codes, np.int8), (v_codes, np.int8), (k_scale, np.float32), (v_scale, np.float32)):
            assert a.dtype == dt and a.flags.c_contiguous
        assert v_codes.shape == k_codes.shape and k_scale.shape == (nb, hkv, bs) and v_scale.shape == k_scale.shape
        kn, vn = _bits(k_new), _bits(v_new)
        sl = np.ascontiguousarray(slots, dtype=np.int64)
        assert kn.shape == (sl.shape[0], hkv, d) and vn.shape == kn.shape
        self.lib.oracle_append_quant_kv(_p(k_codes, _i8p), _p(k_scale, _f32p), _p(v_codes, _i8p), _p(v_scale, _f32p),
                                        _p(sl, _i64p), _p(kn, _u16p), _p(vn, _u16p), sl.shape[0], hkv, d, bs)

    def decode_quant_kv(self, q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens,
                        scale: float) -> np.ndarray:
        """float64 [B, Hq, D] decode over the int8 K + V cache (both dequantised exactly)."""
        qb = _bits(q)
        kc = np.ascontiguousarray(k_codes, dtype=np.int8)
        vc = np.ascontiguousarray(v_codes, dtype=np.int8)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        b, hq, d = qb.shape
        nb, hkv, bs, d2 = kc.shape
        assert d2 == d and hq % hkv == 0 and vc.shape == kc.shape and ks.shape == vs.shape == (nb, hkv, bs)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.empty((b, hq, d), np.float64)
        self.lib.oracle_decode_quant_kv(_p(out, _f64p), _p(qb, _u16p), _p(kc, _i8p), _p(ks, _f32p), _p(vc, _i8p),
                                        _p(vs, _f32p), _p(bt, _i32p), _p(cl, _i32p), b, bt.shape[1], hq, hkv, d, bs,
                                        float(scale))
        return out

    def e4m3_to_double(self, codes) -> np.ndarray:
        """float64 values of E4M3 codes (uint8), elementwise."""
        c = np.asarray(codes, dtype=np.uint8)
        return np.array([self.lib.oracle_e4m3_to_double(int(x)) for x in c.ravel()], np.float64).reshape(c.shape)

    def e4m3_from_float(self, y) -> np.ndarray:
        """E4M3 codes (uint8) nearest to float32 values y (ties to even, clamped to +-448)."""
        a = np.asarray(y, dtype=np.float32)
        return np.array([self.lib.oracle_e4m3_from_float(float(x)) for x in a.ravel()], np.uint8).reshape(a.shape)

    def quantize_fp8_row(self, row) -> tuple[np.ndarray, float]:
        """(E4M3 codes uint8 [D], float32 scale) of one fp16 row."""
        rb = _bits(np.ascontiguousarray(row))
        codes = np.empty(rb.shape[0], np.uint8)
        sc = ctypes.c_float(0.0)
        self.lib.oracle_quantize_fp8_row(_p(codes, _u8p), ctypes.byref(sc), _p(rb, _u16p), rb.shape[0])
        return codes, np.float32(sc.value)

    def append_fp8_kv(self, k_codes, k_scale, v_codes, v_scale, slots, k_new, v_new) -> None:
        """In place on the fp8 K + V cache: codes uint8 [NB,Hkv,bs,D], scales float32 [NB,Hkv,bs]."""
        nb, hkv, bs, d = k_codes.shape
        for a, dt in ((k_codes, np.uint8), (v_codes, np.uint8), (k_scale, np.float32), (v_scale, np.float32)):
            assert a.dtype == dt and a.flags.c_contiguous
        assert v_codes.shape == k_codes.shape and k_scale.shape == (nb, hkv, bs) and v_scale.shape == k_scale.shape
        kn, vn = _bits(k_new), _bits(v_new)
        sl = np.ascontiguousarray(slots, dtype=np.int64)
        assert kn.shape == (sl.shape[0], hkv, d) and vn.shape == kn.shape
        self.lib.oracle_append_fp8_kv(_p(k_codes, _u8p), _p(k_scale, _f32p), _p(v_codes, _u8p), _p(v_scale, _f32p),
                                      _p(sl, _i64p), _p(kn, _u16p), _p(vn, _u16p), sl.shape[0], hkv, d, bs)

    def decode_fp8_kv(self, q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens,
                      scale: float) -> np.ndarray:
        """float64 [B, Hq, D] decode over the fp8 K + V cache (both dequantised exactly)."""
        qb = _bits(q)
        kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
        vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        b, hq, d = qb.shape
        nb, hkv, bs, d2 = kc.shape
        assert d2 == d and hq % hkv == 0 and vc.shape == kc.shape and ks.shape == vs.shape == (nb, hkv, bs)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.empty((b, hq, d), np.float64)
        self.lib.oracle_decode_fp8_kv(_p(out, _f64p), _p(qb, _u16p), _p(kc, _u8p), _p(ks, _f32p), _p(vc, _u8p),
                                      _p(vs, _f32p), _p(bt, _i32p), _p(cl, _i32p), b, bt.shape[1], hq, hkv, d, bs,
                                      float(scale))
        return out

    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale: float) -> np.ndarray:
        """float64 [B, Hq, D] attention output of one decode step."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        b, hq, d = qb.shape
        nb, hkv, bs, d2 = kc.shape
        assert d2 == d and hq % hkv == 0
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.empty((b, hq, d), np.float64)
        self.lib.oracle_decode(_p(out, _f64p), _p(qb, _u16p), _p(kc, _u16p), _p(vc, _u16p),
                               _p(bt, _i32p), _p(cl, _i32p), b, bt.shape[1], hq, hkv, d, bs,
                               float(scale))
        return out

    def decode_multi(self, q, k_cache, v_cache, block_tables, context_lens, query_start,
                     scale: float) -> np.ndarray:
        """float64 [total_q, Hq, D]: causal attention of each request's new tokens (rows
        query_start[b]..query_start[b+1]-1 of q) over its cache."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        t, hq, d = qb.shape
        nb, hkv, bs, d2 = kc.shape
        assert d2 == d and hq % hkv == 0
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        qs = np.ascontiguousarray(query_start, dtype=np.int32)
        assert qs.shape == (bt.shape[0] + 1,) and qs[-1] == t
        out = np.empty((t, hq, d), np.float64)
        self.lib.oracle_decode_multi(_p(out, _f64p), _p(qb, _u16p), _p(kc, _u16p), _p(vc, _u16p), _p(bt, _i32p),
                                     _p(cl, _i32p), _p(qs, _i32p), bt.shape[0], bt.shape[1], hq, hkv, d, bs,
                                     float(scale))
        return out

    def decode_partition(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                         partition_size: int, max_partitions: int):
        """(o [B,Hq,P,D], m [B,Hq,P], l [B,Hq,P]) float64 split-context partials."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        b, hq, d = qb.shape
        nb, hkv, bs, _ = kc.shape
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        o = np.empty((b, hq, max_partitions, d), np.float64)
        m = np.empty((b, hq, max_partitions), np.float64)
        l = np.empty((b, hq, max_partitions), np.float64)
        self.lib.oracle_decode_partition(_p(o, _f64p), _p(m, _f64p), _p(l, _f64p), _p(qb, _u16p),
                                         _p(kc, _u16p), _p(vc, _u16p), _p(bt, _i32p),
                                         _p(cl, _i32p), b, bt.shape[1], hq, hkv, d, bs,
                                         float(scale), partition_size, max_partitions)
        return o, m, l

    def merge(self, o_part, m_part, l_part, context_lens, partition_size: int) -> np.ndarray:
        """float64 [B, Hq, D] log-sum-exp merge of split-context partials."""
        o = np.ascontiguousarray(o_part, dtype=np.float64)
        m = np.ascontiguousarray(m_part, dtype=np.float64)
        l = np.ascontiguousarray(l_part, dtype=np.float64)
        b, hq, p, d = o.shape
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.empty((b, hq, d), np.float64)
        self.lib.oracle_merge(_p(out, _f64p), _p(o, _f64p), _p(m, _f64p), _p(l, _f64p),
                              _p(cl, _i32p), b, hq, d, partition_size, p)
        return out


_default = None


def default() -> Oracle:
    """The oracle built from pkv_oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        path = build()
        with _lock:
            if _default is None:
                _default = Oracle(path)
    return _default


def half_to_double(a):
    return default().half_to_double(a)


def kv_cache_bytes(*args):
    return default().kv_cache_bytes(*args)


def slot_mapping(block_tables, positions, block_size):
    return default().slot_mapping(block_tables, positions, block_size)


def append(k_cache, v_cache, slots, k_new, v_new):
    return default().append(k_cache, v_cache, slots, k_new, v_new)


def decode(q, k_cache, v_cache, block_tables, context_lens, scale):
    return default().decode(q, k_cache, v_cache, block_tables, context_lens, scale)


def decode_partition(q, k_cache, v_cache, block_tables, context_lens, scale, partition_size,
                     max_partitions):
    return default().decode_partition(q, k_cache, v_cache, block_tables, context_lens, scale,
                                      partition_size, max_partitions)


def merge(o_part, m_part, l_part, context_lens, partition_size):
    return default().merge(o_part, m_part, l_part, context_lens, partition_size)


def copy_blocks(k_cache, v_cache, src, dst):
    return default().copy_blocks(k_cache, v_cache, src, dst)


def quantize_k_row(k_row):
    return default().quantize_k_row(k_row)


def copy_blocks_between(dst_k, dst_v, src_k, src_v, src, dst):
    return default().copy_blocks_between(dst_k, dst_v, src_k, src_v, src, dst)


def append_quant_kv(k_codes, k_scale, v_codes, v_scale, slots, k_new, v_new):
    return default().append_quant_kv(k_codes, k_scale, v_codes, v_scale, slots, k_new, v_new)


def decode_quant_kv(q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens, scale):
    return default().decode_quant_kv(q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens, scale)


def decode_multi(q, k_cache, v_cache, block_tables, context_lens, query_start, scale):
    return default().decode_multi(q, k_cache, v_cache, block_tables, context_lens, query_start, scale)


def append_quant_k(k_codes, k_scale, v_cache, slots, k_new, v_new):
    return default().append_quant_k(k_codes, k_scale, v_cache, slots, k_new, v_new)


def decode_quant_k(q, k_codes, k_scale, v_cache, block_tables, context_lens, scale):
    return default().decode_quant_k(q, k_codes, k_scale, v_cache, block_tables, context_lens, scale)


def e4m3_to_double(codes):
    return default().e4m3_to_double(codes)


def e4m3_from_float(y):
    return default().e4m3_from_float(y)


def quantize_fp8_row(row):
    return default().quantize_fp8_row(row)


def append_fp8_kv(k_codes, k_scale, v_codes, v_scale, slots, k_new, v_new):
    return default().append_fp8_kv(k_codes, k_scale, v_codes, v_scale, slots, k_new, v_new)


def decode_fp8_kv(q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens, scale):
    return default().decode_fp8_kv(q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens, scale)
