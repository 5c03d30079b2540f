"""paged_kv_cache_278_gb300 -- decode attention over a paged KV cache on GB300.

A thin Python binding over libpkv.so (C ABI in include/pkv.h).  Every step of
the hot path runs in the library's CUDA kernels; this module only checks
tensor shapes/dtypes, passes raw device pointers and the current CUDA stream,
and turns status codes into exceptions.  PyTorch is used for device memory
and streams only.

    import paged_kv_cache_278_gb300 as pkv
    pkv.append(k_cache, v_cache, slot_mapping, k_new, v_new)          # in-place append
    pkv.decode_attention(out, q, k_cache, v_cache, block_tables,        # softmax(q K^T) V
                         context_lens, scale, workspace=ws)
    o, m, l = ...; pkv.decode_partition(o, m, l, q, ...); pkv.merge(out, o, m, l, context_lens, 512)

Cache tensors are fp16 [num_blocks, num_kv_heads, block_size, head_dim].
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (PKV_MAX_QUERY_LEN, PKV_DEFAULT_PARTITION, PKV_DEV_BAD_BLOCK_ID, PKV_DEV_BAD_CONTEXT, PKV_DEV_BAD_SLOT,
                   PKV_DEV_OK, PKV_DEV_PREFIX_MISMATCH, PKV_DEV_SMEM_MISALIGNED, PKV_DEV_WAIT_TIMEOUT, PKV_HEAD_DIM, PKV_MAX_PARTITION,
                   PKV_STEP_OVERLAP, PKV_MAX_STEP_QUERY_LEN, PkvError)

__all__ = [
    "append", "decode_attention", "decode_partition", "merge", "decode_workspace_size", "make_workspace",
    "decode_attention_shared_prefix", "make_shared_prefix_workspace", "PKV_DEV_PREFIX_MISMATCH",
    "decode_step", "make_step_workspace", "copy_blocks", "append_int8k", "decode_attention_int8k",
    "decode_step_int8k", "empty_int8k_cache", "decode_attention_multi", "decode_step_multi", "make_multi_workspace",
    "copy_blocks_between", "empty_int8kv_cache", "append_int8kv", "decode_attention_int8kv", "decode_step_int8kv",
    "empty_fp8kv_cache", "append_fp8kv", "decode_attention_fp8kv", "decode_step_fp8kv",
    "device_error", "slot_mapping", "BlockPool", "PkvError", "library_path",
    "PKV_DEFAULT_PARTITION", "PKV_MAX_PARTITION", "PKV_HEAD_DIM",
    "PKV_DEV_OK", "PKV_DEV_BAD_BLOCK_ID", "PKV_DEV_BAD_CONTEXT", "PKV_DEV_BAD_SLOT", "PKV_DEV_WAIT_TIMEOUT",
    "PKV_DEV_SMEM_MISALIGNED", "PKV_STEP_OVERLAP", "PKV_MAX_STEP_QUERY_LEN",
]


def library_path() -> str:
    return _lib.LIB_PATH


def _L():
    return _lib.load()


def _stream(device: torch.device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _flags(overlap: bool) -> int:
    return _lib.PKV_STEP_OVERLAP if overlap else 0


def _need(t: torch.Tensor, name: str, dtype, ndim: int, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _cache_shape(k_cache, v_cache):
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4, k_cache.device)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    return tuple(k_cache.shape)


def append(k_cache: torch.Tensor, v_cache: torch.Tensor, slot_mapping: torch.Tensor, k_new: torch.Tensor,
           v_new: torch.Tensor, stream=None) -> None:
    """Write k_new/v_new [T, Hkv, D] into the cache slots slot_mapping [T] (int64; -1 = skip)."""
    nb, hkv, bs, d = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    t = slot_mapping.shape[0]
    if k_new.shape != (t, hkv, d) or v_new.shape != (t, hkv, d):
        raise ValueError(f"k_new/v_new must be [{t}, {hkv}, {d}]")
    st = _L().pkv_append(k_cache.data_ptr(), v_cache.data_ptr(), slot_mapping.data_ptr(), k_new.data_ptr(),
                         v_new.data_ptr(), t, hkv, d, bs, nb, _stream(dev, stream))
    _lib.check(st, "pkv_append")


def decode_workspace_size(num_seqs: int, num_q_heads: int, max_context: int,
                          partition_size: int = PKV_DEFAULT_PARTITION, head_dim: int = PKV_HEAD_DIM) -> int:
    return int(_L().pkv_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context, partition_size))


def make_workspace(num_seqs: int, num_q_heads: int, max_context: int, device) -> torch.Tensor | None:
    """Allocate (with torch) the zero-filled workspace decode_attention needs; None when it needs
    none.  Its completion counters start at zero and every call leaves them zero."""
    n = decode_workspace_size(num_seqs, num_q_heads, max_context)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _decode_inputs(q, k_cache, v_cache, block_tables, context_lens):
    nb, hkv, bs, d = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", torch.float16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    b, hq, dq = q.shape
    if dq != d:
        raise ValueError("q head_dim differs from the cache's")
    if block_tables.shape[0] != b or context_lens.shape[0] != b:
        raise ValueError("block_tables / context_lens batch differs from q")
    return nb, hkv, bs, d, b, hq, dev


def decode_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out [B, Hq, D] fp16 = softmax(scale q K^T) V over each request's paged context."""
    nb, hkv, bs, d, b, hq, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    _need(out, "out", torch.float16, 3, dev)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    st = _L().pkv_decode_attention(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   block_tables.data_ptr(), context_lens.data_ptr(), b, block_tables.shape[1],
                                   hq, hkv, d, bs, nb, float(scale), ws_ptr, ws_bytes, _stream(dev, stream))
    _lib.check(st, "pkv_decode_attention")
    return out


def make_shared_prefix_workspace(num_seqs: int, num_q_heads: int, max_context: int, prefix_len: int,
                                 device) -> torch.Tensor:
    """Allocate (with torch) the zero-filled workspace decode_attention_shared_prefix needs."""
    n = int(_L().pkv_shared_prefix_workspace_size(num_seqs, num_q_heads, PKV_HEAD_DIM, max_context, prefix_len))
    if n == 0:
        raise ValueError("invalid shared-prefix workspace request")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode_attention_shared_prefix(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                   scale: float, prefix_len: int, workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """Same result as decode_attention for tables that all start with the same prefix_len tokens'
    blocks; the prefix's K/V is read once per kv head for the whole batch."""
    nb, hkv, bs, d, b, hq, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    _need(out, "out", torch.float16, 3, dev)
    _need(workspace, "workspace", torch.uint8, 1, dev)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    st = _L().pkv_decode_attention_shared_prefix(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), b, block_tables.shape[1], hq, hkv, d, bs, nb, float(scale), int(prefix_len),
        workspace.data_ptr(), workspace.numel(), _stream(dev, stream))
    _lib.check(st, "pkv_decode_attention_shared_prefix")
    return out


def make_step_workspace(num_seqs: int, num_q_heads: int, max_context: int, prefix_len: int = 0,
                        device=None, partition_size: int = 0) -> torch.Tensor | None:
    """Zero-filled workspace for decode_step (None when it needs none); partition_size as decode_step's."""
    if partition_size and not prefix_len:
        n = decode_workspace_size(num_seqs, num_q_heads, max_context, partition_size)
    else:
        n = int(_L().pkv_decode_step_workspace_size(num_seqs, num_q_heads, PKV_HEAD_DIM, max_context, prefix_len))
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode_step(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                context_lens: torch.Tensor, scale: float, prefix_len: int = 0,
                workspace: torch.Tensor | None = None, stream=None, partition_size: int = 0,
                overlap: bool = False) -> torch.Tensor:
    """One decode step: write each request's new token [B, Hkv, D] at position context_lens - 1,
    then out = softmax(scale q K^T) V over the whole context (append fused into the decode kernel).
    partition_size > 0 (prefix_len 0 only) overrides the split-context partition.  overlap=True
    passes PKV_STEP_OVERLAP: the step's kernels start streaming the cache history while the
    previous kernel on the stream drains, which that kernel must not write (another layer's step
    is fine; the previous step on the same cache is not)."""
    nb, hkv, bs, d, b, hq, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    _need(out, "out", torch.float16, 3, dev)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if k_new.shape != (b, hkv, d) or v_new.shape != (b, hkv, d):
        raise ValueError(f"k_new/v_new must be [{b}, {hkv}, {d}]")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    if partition_size:
        if prefix_len:
            raise ValueError("partition_size applies to steps without a shared prefix")
        st = _L().pkv_decode_step_partition(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                            k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
                                            context_lens.data_ptr(), b, block_tables.shape[1], hq, hkv, d, bs, nb,
                                            float(scale), int(partition_size), ws_ptr, ws_bytes, _flags(overlap),
                                            _stream(dev, stream))
        _lib.check(st, "pkv_decode_step_partition")
        return out
    st = _L().pkv_decode_step(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                              v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(), b,
                              block_tables.shape[1], hq, hkv, d, bs, nb, float(scale), int(prefix_len), ws_ptr,
                              ws_bytes, _flags(overlap), _stream(dev, stream))
    _lib.check(st, "pkv_decode_step")
    return out


def decode_partition(o_part: torch.Tensor, m_part: torch.Tensor, l_part: torch.Tensor, q: torch.Tensor,
                     k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                     context_lens: torch.Tensor, scale: float, partition_size: int = PKV_DEFAULT_PARTITION,
                     stream=None) -> None:
    """Split-context partials: o_part [B,Hq,P,D], m_part/l_part [B,Hq,P] (fp32)."""
    nb, hkv, bs, d, b, hq, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    _need(o_part, "o_part", torch.float32, 4, dev)
    _need(m_part, "m_part", torch.float32, 3, dev)
    _need(l_part, "l_part", torch.float32, 3, dev)
    p = o_part.shape[2]
    if o_part.shape != (b, hq, p, d) or m_part.shape != (b, hq, p) or l_part.shape != (b, hq, p):
        raise ValueError("partial buffers must be [B, Hq, P, D] and [B, Hq, P]")
    st = _L().pkv_decode_partition(o_part.data_ptr(), m_part.data_ptr(), l_part.data_ptr(), q.data_ptr(),
                                   k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
                                   context_lens.data_ptr(), b, block_tables.shape[1], hq, hkv, d, bs, nb,
                                   float(scale), partition_size, p, _stream(dev, stream))
    _lib.check(st, "pkv_decode_partition")


def merge(out: torch.Tensor, o_part: torch.Tensor, m_part: torch.Tensor, l_part: torch.Tensor,
          context_lens: torch.Tensor, partition_size: int = PKV_DEFAULT_PARTITION, stream=None) -> torch.Tensor:
    """Log-sum-exp merge of decode_partition's partials into out [B, Hq, D] fp16."""
    _need(o_part, "o_part", torch.float32, 4)
    dev = o_part.device
    _need(m_part, "m_part", torch.float32, 3, dev)
    _need(l_part, "l_part", torch.float32, 3, dev)
    _need(out, "out", torch.float16, 3, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    b, hq, p, d = o_part.shape
    if out.shape != (b, hq, d) or m_part.shape != (b, hq, p) or l_part.shape != (b, hq, p):
        raise ValueError("shape mismatch between out and the partial buffers")
    st = _L().pkv_merge(out.data_ptr(), o_part.data_ptr(), m_part.data_ptr(), l_part.data_ptr(),
                        context_lens.data_ptr(), b, hq, d, partition_size, p, _stream(dev, stream))
    _lib.check(st, "pkv_merge")
    return out


def device_error(device=None, stream=None) -> int:
    """Synchronise and return (then clear) the device error word: PKV_DEV_OK if no kernel
    recorded an out-of-range index."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    code = ctypes.c_int(0)
    with torch.cuda.device(dev):
        st = _L().pkv_get_device_error(_stream(dev, stream), ctypes.byref(code))
    _lib.check(st, "pkv_get_device_error")
    return code.value


# ---------------------------------------------------------------- several new tokens per request

def make_multi_workspace(num_seqs: int, total_q: int, max_query_len: int, num_q_heads: int, num_kv_heads: int,
                         max_context: int, device) -> torch.Tensor | None:
    """Zero-filled workspace for decode_attention_multi (None when it needs none)."""
    n = int(_L().pkv_decode_multi_workspace_size(num_seqs, total_q, max_query_len, num_q_heads, num_kv_heads,
                                                 PKV_HEAD_DIM, max_context))
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode_attention_multi(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, query_start: torch.Tensor,
                           max_query_len: int, scale: float, workspace: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """Causal attention of each request's new tokens (q rows query_start[b]..query_start[b+1]-1,
    already appended, so context_lens counts them) over its paged cache; out like q."""
    nb, hkv, bs, d = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", torch.float16, 3, dev)
    _need(out, "out", torch.float16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(query_start, "query_start", torch.int32, 1, dev)
    t, hq, dq = q.shape
    b = context_lens.shape[0]
    if dq != d or out.shape != q.shape:
        raise ValueError("q / out shapes disagree with the cache")
    if block_tables.shape[0] != b or query_start.shape[0] != b + 1:
        raise ValueError("block_tables [B, ...], context_lens [B] and query_start [B + 1] disagree")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    st = _L().pkv_decode_attention_multi(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                         block_tables.data_ptr(), context_lens.data_ptr(), query_start.data_ptr(), b,
                                         t, int(max_query_len), block_tables.shape[1], hq, hkv, d, bs, nb,
                                         float(scale), ws_ptr, ws_bytes, _stream(dev, stream))
    _lib.check(st, "pkv_decode_attention_multi")
    return out


def decode_step_multi(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, query_start: torch.Tensor, max_query_len: int, scale: float,
                      workspace: torch.Tensor | None = None, stream=None, overlap: bool = False) -> torch.Tensor:
    """One several-token step: write request b's new tokens (k_new/v_new rows query_start[b]..,
    [total_q, Hkv, D]) at positions context_lens[b] - n_b .., then the causal attention of
    decode_attention_multi, in one launch; max_query_len <= PKV_MAX_STEP_QUERY_LEN.  overlap as
    decode_step's."""
    nb, hkv, bs, d = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", torch.float16, 3, dev)
    _need(out, "out", torch.float16, 3, dev)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(query_start, "query_start", torch.int32, 1, dev)
    t, hq, dq = q.shape
    b = context_lens.shape[0]
    if dq != d or out.shape != q.shape:
        raise ValueError("q / out shapes disagree with the cache")
    if k_new.shape != (t, hkv, d) or v_new.shape != (t, hkv, d):
        raise ValueError(f"k_new/v_new must be [{t}, {hkv}, {d}]")
    if block_tables.shape[0] != b or query_start.shape[0] != b + 1:
        raise ValueError("block_tables [B, ...], context_lens [B] and query_start [B + 1] disagree")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    st = _L().pkv_decode_step_multi(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                    k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
                                    context_lens.data_ptr(), query_start.data_ptr(), b, t, int(max_query_len),
                                    block_tables.shape[1], hq, hkv, d, bs, nb, float(scale), ws_ptr, ws_bytes,
                                    _flags(overlap), _stream(dev, stream))
    _lib.check(st, "pkv_decode_step_multi")
    return out


# ---------------------------------------------------------------- int8 key cache

def _int8k_shape(k_codes, k_scale, v_cache):
    _need(k_codes, "k_codes", torch.int8, 4)
    dev = k_codes.device
    _need(k_scale, "k_scale", torch.float32, 3, dev)
    _need(v_cache, "v_cache", torch.float16, 4, dev)
    if k_codes.shape != v_cache.shape or k_scale.shape != k_codes.shape[:3]:
        raise ValueError("k_codes [NB,Hkv,bs,D], k_scale [NB,Hkv,bs] and v_cache [NB,Hkv,bs,D] disagree")
    return tuple(k_codes.shape)


def empty_int8k_cache(num_blocks: int, num_kv_heads: int, block_size: int, device,
                      head_dim: int = PKV_HEAD_DIM):
    """Zero-filled (k_codes int8, k_scale float32, v_cache fp16) for the int8-key cache."""
    return (torch.zeros((num_blocks, num_kv_heads, block_size, head_dim), dtype=torch.int8, device=device),
            torch.zeros((num_blocks, num_kv_heads, block_size), dtype=torch.float32, device=device),
            torch.zeros((num_blocks, num_kv_heads, block_size, head_dim), dtype=torch.float16, device=device))


def append_int8k(k_codes: torch.Tensor, k_scale: torch.Tensor, v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                 k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Quantise k_new [T, Hkv, D] into k_codes/k_scale and copy v_new into v_cache at slot_mapping [T]."""
    nb, hkv, bs, d = _int8k_shape(k_codes, k_scale, v_cache)
    dev = k_codes.device
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    t = slot_mapping.shape[0]
    if k_new.shape != (t, hkv, d) or v_new.shape != (t, hkv, d):
        raise ValueError(f"k_new/v_new must be [{t}, {hkv}, {d}]")
    st = _L().pkv_append_int8k(k_codes.data_ptr(), k_scale.data_ptr(), v_cache.data_ptr(), slot_mapping.data_ptr(),
                               k_new.data_ptr(), v_new.data_ptr(), t, hkv, d, bs, nb, _stream(dev, stream))
    _lib.check(st, "pkv_append_int8k")


def _int8k_decode_inputs(q, k_codes, k_scale, v_cache, block_tables, context_lens, out, workspace):
    nb, hkv, bs, d = _int8k_shape(k_codes, k_scale, v_cache)
    dev = k_codes.device
    _need(q, "q", torch.float16, 3, dev)
    _need(out, "out", torch.float16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    b, hq, dq = q.shape
    if dq != d or out.shape != q.shape:
        raise ValueError("q / out shapes disagree with the cache")
    if block_tables.shape[0] != b or context_lens.shape[0] != b:
        raise ValueError("block_tables / context_lens batch differs from q")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    return nb, hkv, bs, d, b, hq, dev, ws_ptr, ws_bytes


def decode_attention_int8k(out: torch.Tensor, q: torch.Tensor, k_codes: torch.Tensor, k_scale: torch.Tensor,
                           v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """decode_attention over the int8-key cache (keys dequantised as code * row scale)."""
    nb, hkv, bs, d, b, hq, dev, ws_ptr, ws_bytes = _int8k_decode_inputs(q, k_codes, k_scale, v_cache, block_tables,
                                                                        context_lens, out, workspace)
    st = _L().pkv_decode_attention_int8k(out.data_ptr(), q.data_ptr(), k_codes.data_ptr(), k_scale.data_ptr(),
                                         v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(), b,
                                         block_tables.shape[1], hq, hkv, d, bs, nb, float(scale), ws_ptr, ws_bytes,
                                         _stream(dev, stream))
    _lib.check(st, "pkv_decode_attention_int8k")
    return out


def decode_step_int8k(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      k_codes: torch.Tensor, k_scale: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, workspace: torch.Tensor | None = None,
                      stream=None, overlap: bool = False) -> torch.Tensor:
    """decode_step over the int8-key cache: quantise + write the new token at ctx - 1, then attend.
    overlap as decode_step's."""
    nb, hkv, bs, d, b, hq, dev, ws_ptr, ws_bytes = _int8k_decode_inputs(q, k_codes, k_scale, v_cache, block_tables,
                                                                        context_lens, out, workspace)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    if k_new.shape != (b, hkv, d) or v_new.shape != (b, hkv, d):
        raise ValueError(f"k_new/v_new must be [{b}, {hkv}, {d}]")
    st = _L().pkv_decode_step_int8k(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                    k_codes.data_ptr(), k_scale.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
                                    context_lens.data_ptr(), b, block_tables.shape[1], hq, hkv, d, bs, nb, float(scale),
                                    ws_ptr, ws_bytes, _flags(overlap), _stream(dev, stream))
    _lib.check(st, "pkv_decode_step_int8k")
    return out


# ---------------------------------------------------------------- int8 keys and values

def _int8kv_shape(k_codes, k_scale, v_codes, v_scale, codes=torch.int8):
    _need(k_codes, "k_codes", codes, 4)
    dev = k_codes.device
    _need(v_codes, "v_codes", codes, 4, dev)
    _need(k_scale, "k_scale", torch.float32, 3, dev)
    _need(v_scale, "v_scale", torch.float32, 3, dev)
    if v_codes.shape != k_codes.shape or k_scale.shape != k_codes.shape[:3] or v_scale.shape != k_scale.shape:
        raise ValueError("codes [NB,Hkv,bs,D] and scales [NB,Hkv,bs] disagree")
    return tuple(k_codes.shape)


def empty_int8kv_cache(num_blocks: int, num_kv_heads: int, block_size: int, device, head_dim: int = PKV_HEAD_DIM):
    """Zero-filled (k_codes, k_scale, v_codes, v_scale) for the int8 K + V cache."""
    codes = lambda: torch.zeros((num_blocks, num_kv_heads, block_size, head_dim), dtype=torch.int8, device=device)
    scales = lambda: torch.zeros((num_blocks, num_kv_heads, block_size), dtype=torch.float32, device=device)
    return codes(), scales(), codes(), scales()


def append_int8kv(k_codes, k_scale, v_codes, v_scale, slot_mapping, k_new, v_new, stream=None) -> None:
    """Quantise k_new and v_new [T, Hkv, D] into the int8 K + V cache at slot_mapping [T]."""
    nb, hkv, bs, d = _int8kv_shape(k_codes, k_scale, v_codes, v_scale)
    dev = k_codes.device
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    t = slot_mapping.shape[0]
    if k_new.shape != (t, hkv, d) or v_new.shape != (t, hkv, d):
        raise ValueError(f"k_new/v_new must be [{t}, {hkv}, {d}]")
    st = _L().pkv_append_int8kv(k_codes.data_ptr(), k_scale.data_ptr(), v_codes.data_ptr(), v_scale.data_ptr(),
                                slot_mapping.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), t, hkv, d, bs, nb,
                                _stream(dev, stream))
    _lib.check(st, "pkv_append_int8kv")


def _int8kv_inputs(q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens, out, workspace,
                   codes=torch.int8):
    nb, hkv, bs, d = _int8kv_shape(k_codes, k_scale, v_codes, v_scale, codes)
    dev = k_codes.device
    _need(q, "q", torch.float16, 3, dev)
    _need(out, "out", torch.float16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    b, hq, dq = q.shape
    if dq != d or out.shape != q.shape:
        raise ValueError("q / out shapes disagree with the cache")
    if block_tables.shape[0] != b or context_lens.shape[0] != b:
        raise ValueError("block_tables / context_lens batch differs from q")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    return nb, hkv, bs, d, b, hq, dev, ws_ptr, ws_bytes


def decode_attention_int8kv(out, q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens, scale: float,
                            workspace=None, stream=None) -> torch.Tensor:
    """decode_attention over the int8 K + V cache."""
    nb, hkv, bs, d, b, hq, dev, ws_ptr, ws_bytes = _int8kv_inputs(q, k_codes, k_scale, v_codes, v_scale, block_tables,
                                                                  context_lens, out, workspace)
    st = _L().pkv_decode_attention_int8kv(out.data_ptr(), q.data_ptr(), k_codes.data_ptr(), k_scale.data_ptr(),
                                          v_codes.data_ptr(), v_scale.data_ptr(), block_tables.data_ptr(),
                                          context_lens.data_ptr(), b, block_tables.shape[1], hq, hkv, d, bs, nb,
                                          float(scale), ws_ptr, ws_bytes, _stream(dev, stream))
    _lib.check(st, "pkv_decode_attention_int8kv")
    return out


def decode_step_int8kv(out, q, k_new, v_new, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens,
                       scale: float, workspace=None, stream=None, overlap: bool = False) -> torch.Tensor:
    """decode_step over the int8 K + V cache; overlap as decode_step's."""
    nb, hkv, bs, d, b, hq, dev, ws_ptr, ws_bytes = _int8kv_inputs(q, k_codes, k_scale, v_codes, v_scale, block_tables,
                                                                  context_lens, out, workspace)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    if k_new.shape != (b, hkv, d) or v_new.shape != (b, hkv, d):
        raise ValueError(f"k_new/v_new must be [{b}, {hkv}, {d}]")
    st = _L().pkv_decode_step_int8kv(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                     k_codes.data_ptr(), k_scale.data_ptr(), v_codes.data_ptr(), v_scale.data_ptr(),
                                     block_tables.data_ptr(), context_lens.data_ptr(), b, block_tables.shape[1], hq, hkv,
                                     d, bs, nb, float(scale), ws_ptr, ws_bytes, _flags(overlap), _stream(dev, stream))
    _lib.check(st, "pkv_decode_step_int8kv")
    return out


# ---------------------------------------------------------------- fp8 (E4M3) keys and values
# Codes are uint8 tensors holding E4M3 bit patterns (view them as torch.float8_e4m3fn to read
# their values); scales float32 per (block, kv head, slot), as for the int8 K + V cache.

def empty_fp8kv_cache(num_blocks: int, num_kv_heads: int, block_size: int, device, head_dim: int = PKV_HEAD_DIM):
    """Zero-filled (k_codes, k_scale, v_codes, v_scale) for the fp8 K + V cache (codes uint8)."""
    codes = lambda: torch.zeros((num_blocks, num_kv_heads, block_size, head_dim), dtype=torch.uint8, device=device)
    scales = lambda: torch.zeros((num_blocks, num_kv_heads, block_size), dtype=torch.float32, device=device)
    return codes(), scales(), codes(), scales()


def append_fp8kv(k_codes, k_scale, v_codes, v_scale, slot_mapping, k_new, v_new, stream=None) -> None:
    """Quantise k_new and v_new [T, Hkv, D] into the fp8 K + V cache at slot_mapping [T]."""
    nb, hkv, bs, d = _int8kv_shape(k_codes, k_scale, v_codes, v_scale, torch.uint8)
    dev = k_codes.device
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    t = slot_mapping.shape[0]
    if k_new.shape != (t, hkv, d) or v_new.shape != (t, hkv, d):
        raise ValueError(f"k_new/v_new must be [{t}, {hkv}, {d}]")
    st = _L().pkv_append_fp8kv(k_codes.data_ptr(), k_scale.data_ptr(), v_codes.data_ptr(), v_scale.data_ptr(),
                               slot_mapping.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), t, hkv, d, bs, nb,
                               _stream(dev, stream))
    _lib.check(st, "pkv_append_fp8kv")


def decode_attention_fp8kv(out, q, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens, scale: float,
                           workspace=None, stream=None) -> torch.Tensor:
    """decode_attention over the fp8 K + V cache."""
    nb, hkv, bs, d, b, hq, dev, ws_ptr, ws_bytes = _int8kv_inputs(q, k_codes, k_scale, v_codes, v_scale, block_tables,
                                                                  context_lens, out, workspace, torch.uint8)
    st = _L().pkv_decode_attention_fp8kv(out.data_ptr(), q.data_ptr(), k_codes.data_ptr(), k_scale.data_ptr(),
                                         v_codes.data_ptr(), v_scale.data_ptr(), block_tables.data_ptr(),
                                         context_lens.data_ptr(), b, block_tables.shape[1], hq, hkv, d, bs, nb,
                                         float(scale), ws_ptr, ws_bytes, _stream(dev, stream))
    _lib.check(st, "pkv_decode_attention_fp8kv")
    return out


def decode_step_fp8kv(out, q, k_new, v_new, k_codes, k_scale, v_codes, v_scale, block_tables, context_lens,
                      scale: float, workspace=None, stream=None, overlap: bool = False) -> torch.Tensor:
    """decode_step over the fp8 K + V cache; overlap as decode_step's."""
    nb, hkv, bs, d, b, hq, dev, ws_ptr, ws_bytes = _int8kv_inputs(q, k_codes, k_scale, v_codes, v_scale, block_tables,
                                                                  context_lens, out, workspace, torch.uint8)
    _need(k_new, "k_new", torch.float16, 3, dev)
    _need(v_new, "v_new", torch.float16, 3, dev)
    if k_new.shape != (b, hkv, d) or v_new.shape != (b, hkv, d):
        raise ValueError(f"k_new/v_new must be [{b}, {hkv}, {d}]")
    st = _L().pkv_decode_step_fp8kv(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                    k_codes.data_ptr(), k_scale.data_ptr(), v_codes.data_ptr(), v_scale.data_ptr(),
                                    block_tables.data_ptr(), context_lens.data_ptr(), b, block_tables.shape[1], hq, hkv,
                                    d, bs, nb, float(scale), ws_ptr, ws_bytes, _flags(overlap), _stream(dev, stream))
    _lib.check(st, "pkv_decode_step_fp8kv")
    return out


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src: torch.Tensor, dst: torch.Tensor,
                stream=None) -> None:
    """k_cache[dst[i]] <- k_cache[src[i]] (and V), whole blocks, bit for bit (copy-on-write)."""
    nb, hkv, bs, d = _cache_shape(k_cache, v_cache)
    dev = k_cache.device
    _need(src, "src", torch.int32, 1, dev)
    _need(dst, "dst", torch.int32, 1, dev)
    if src.shape != dst.shape:
        raise ValueError("src and dst differ in length")
    st = _L().pkv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), src.data_ptr(), dst.data_ptr(), src.numel(),
                              hkv, d, bs, nb, _stream(dev, stream))
    _lib.check(st, "pkv_copy_blocks")


def _gpu_addressable(t: torch.Tensor, name: str, device):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.is_cuda:
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device}")
    elif not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or page-locked host memory")


def copy_blocks_between(dst_k: torch.Tensor, dst_v: torch.Tensor, src_k: torch.Tensor, src_v: torch.Tensor,
                        src_ids: torch.Tensor, dst_ids: torch.Tensor, device=None, stream=None) -> None:
    """dst_k[dst_ids[i]] <- src_k[src_ids[i]] (and V), whole blocks, bit for bit.  Pools and id arrays may
    be CUDA tensors or pinned host tensors (the copy kernel addresses host memory directly)."""
    dev = torch.device(device) if device is not None else next(
        (t.device for t in (dst_k, src_k, src_ids) if t.is_cuda), torch.device("cuda"))
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    for t, name in ((dst_k, "dst_k"), (dst_v, "dst_v"), (src_k, "src_k"), (src_v, "src_v")):
        if t.dtype != torch.float16 or t.dim() != 4:
            raise ValueError(f"{name} must be fp16 [blocks, Hkv, bs, D]")
        _gpu_addressable(t, name, dev)
    for t, name in ((src_ids, "src_ids"), (dst_ids, "dst_ids")):
        if t.dtype != torch.int32 or t.dim() != 1:
            raise ValueError(f"{name} must be int32 [n]")
        _gpu_addressable(t, name, dev)
    if dst_k.shape != dst_v.shape or src_k.shape != src_v.shape or dst_k.shape[1:] != src_k.shape[1:]:
        raise ValueError("pools differ in geometry")
    if src_ids.shape != dst_ids.shape:
        raise ValueError("src_ids and dst_ids differ in length")
    _, hkv, bs, d = src_k.shape
    st = _L().pkv_copy_blocks_between(dst_k.data_ptr(), dst_v.data_ptr(), dst_k.shape[0], src_k.data_ptr(),
                                      src_v.data_ptr(), src_k.shape[0], src_ids.data_ptr(), dst_ids.data_ptr(),
                                      src_ids.numel(), hkv, d, bs, _stream(dev, stream))
    _lib.check(st, "pkv_copy_blocks_between")


def slot_mapping(block_tables: torch.Tensor, positions: torch.Tensor, block_size: int) -> torch.Tensor:
    """Host slot of each request's new token: int64 [B] (CPU tensors in, CPU tensor out)."""
    bt = block_tables.to(torch.int32).contiguous().cpu()
    pos = positions.to(torch.int32).contiguous().cpu()
    out = torch.empty(pos.shape[0], dtype=torch.int64)
    st = _L().pkv_slot_mapping(ctypes.cast(out.data_ptr(), _lib.c_i64p), ctypes.cast(bt.data_ptr(), _lib.c_i32p),
                               ctypes.cast(pos.data_ptr(), _lib.c_i32p), pos.shape[0], bt.shape[1], block_size)
    _lib.check(st, "pkv_slot_mapping")
    return out


class BlockPool:
    """Host pool of KV-cache block ids (free list + reference counts), backed by pkv_pool_*."""

    def __init__(self, num_blocks: int, seed: int = 0):
        h = ctypes.c_void_p()
        _lib.check(_L().pkv_pool_create(num_blocks, seed, ctypes.byref(h)), "pkv_pool_create")
        self._h = h
        self.num_blocks = num_blocks

    def close(self):
        if self._h is not None and self._h.value:
            _L().pkv_pool_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _ids(ids):
        arr = (ctypes.c_int32 * len(ids))(*[int(i) for i in ids])
        return arr

    def alloc(self, n: int) -> list[int]:
        arr = (ctypes.c_int32 * max(n, 1))()
        _lib.check(_L().pkv_pool_alloc(self._h, n, arr), "pkv_pool_alloc")
        return list(arr[:n])

    def share(self, ids) -> None:
        _lib.check(_L().pkv_pool_share(self._h, len(ids), self._ids(ids)), "pkv_pool_share")

    def free(self, ids) -> None:
        _lib.check(_L().pkv_pool_free(self._h, len(ids), self._ids(ids)), "pkv_pool_free")

    def num_free(self) -> int:
        return int(_L().pkv_pool_num_free(self._h))

    def refcount(self, block_id: int) -> int:
        return int(_L().pkv_pool_refcount(self._h, block_id))

    @staticmethod
    def _row(table_row: torch.Tensor) -> "ctypes._Pointer":
        if table_row.dtype != torch.int32 or table_row.device.type != "cpu" or not table_row.is_contiguous():
            raise ValueError("table rows must be contiguous CPU int32 tensors")
        return ctypes.cast(table_row.data_ptr(), _lib.c_i32p)

    def fork(self, src_row: torch.Tensor, dst_row: torch.Tensor, num_tokens: int, block_size: int) -> None:
        """dst_row shares the blocks holding src_row's first num_tokens tokens."""
        st = _L().pkv_pool_fork(self._h, self._row(src_row), self._row(dst_row), dst_row.numel(), num_tokens,
                                block_size)
        _lib.check(st, "pkv_pool_fork")

    def prepare_append(self, table_row: torch.Tensor, cur_tokens: int, block_size: int):
        """Make position cur_tokens writable; returns (src, dst) block ids to copy first, or None."""
        src, dst, n = ctypes.c_int32(-1), ctypes.c_int32(-1), ctypes.c_int(0)
        st = _L().pkv_pool_prepare_append(self._h, self._row(table_row), table_row.numel(), cur_tokens, block_size,
                                          ctypes.byref(src), ctypes.byref(dst), ctypes.byref(n))
        _lib.check(st, "pkv_pool_prepare_append")
        return (src.value, dst.value) if n.value else None

    def swap_to(self, other: "BlockPool", table_row: torch.Tensor, num_tokens: int, block_size: int):
        """Move the request's blocks into `other` (swap out / in); returns (src_ids, dst_ids) int32 CPU
        tensors of the block pairs to copy with copy_blocks_between.  table_row is rewritten."""
        n = -(-num_tokens // block_size)
        src = torch.empty(max(n, 1), dtype=torch.int32)
        dst = torch.empty(max(n, 1), dtype=torch.int32)
        st = _L().pkv_pool_swap(self._h, other._h, self._row(table_row), table_row.numel(), num_tokens, block_size,
                                self._row(src), self._row(dst))
        _lib.check(st, "pkv_pool_swap")
        return src[:n], dst[:n]

    def free_table(self, table_row: torch.Tensor, num_tokens: int, block_size: int) -> None:
        _lib.check(_L().pkv_pool_free_table(self._h, self._row(table_row), num_tokens, block_size),
                   "pkv_pool_free_table")

    def reserve(self, table_row: torch.Tensor, cur_tokens: int, new_tokens: int, block_size: int) -> None:
        """Grow a CPU int32 block-table row in place to cover new_tokens tokens."""
        if table_row.dtype != torch.int32 or table_row.device.type != "cpu" or not table_row.is_contiguous():
            raise ValueError("table_row must be a contiguous CPU int32 tensor")
        st = _L().pkv_pool_reserve(self._h, ctypes.cast(table_row.data_ptr(), _lib.c_i32p), table_row.numel(),
                                   cur_tokens, new_tokens, block_size)
        _lib.check(st, "pkv_pool_reserve")
