"""Helpers for the GPU parity tests: run one decode step through the C ABI and the same step
through the float64 oracle, on the same seeded inputs.  The oracle's inputs are host copies of
the generator's tensors taken before any library kernel touches them."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv

ATTN_TOL = 2e-3      # max |fp16 GPU output - float64 oracle|, fp32 accumulation


def host_inputs(case):
    """numpy copies of a Case (fp16 stays fp16)."""
    return {
        "q": case.q.cpu().numpy(),
        "k_cache": case.k_cache.cpu().numpy(),
        "v_cache": case.v_cache.cpu().numpy(),
        "k_new": case.k_new.cpu().numpy(),
        "v_new": case.v_new.cpu().numpy(),
        "block_tables": case.block_tables.cpu().numpy(),
        "context_lens": case.context_lens.cpu().numpy(),
        "positions": case.positions.cpu().numpy(),
    }


def oracle_step(h, case, decode=True):
    """Oracle append (in place on h's caches) then decode; returns float64 [B, Hq, D] or None."""
    slots = oracle.slot_mapping(h["block_tables"], h["positions"], case.block_size)
    oracle.append(h["k_cache"], h["v_cache"], slots, h["k_new"], h["v_new"])
    if not decode:
        return None
    return oracle.decode(h["q"], h["k_cache"], h["v_cache"], h["block_tables"], h["context_lens"], case.scale)


def gpu_step(case, workspace="auto", stream=None):
    """Library append + decode on the case's device tensors (caches modified in place)."""
    dev = case.q.device
    slots = pkv.slot_mapping(case.block_tables.cpu(), case.positions.cpu(), case.block_size).to(dev)
    pkv.append(case.k_cache, case.v_cache, slots, case.k_new, case.v_new, stream=stream)
    out = torch.empty_like(case.q)
    if workspace == "auto":
        workspace = pkv.make_workspace(case.num_seqs, case.num_q_heads,
                                       case.max_blocks_per_seq * case.block_size, dev)
    pkv.decode_attention(out, case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                         case.scale, workspace=workspace, stream=stream)
    return out


def max_err(gpu_out: torch.Tensor, ref: np.ndarray) -> float:
    got = gpu_out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.abs(got - ref).max()) if got.size else 0.0


def assert_no_device_error():
    code = pkv.device_error()
    assert code == pkv.PKV_DEV_OK, f"device error word = {code}"
