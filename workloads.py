"""Seeded synthetic inputs for one decode step over a paged KV cache.

This module is shared by the tests, the benchmark and the CPU oracle's
callers.  It only draws numbers and builds the input structures (pools, block
tables, context lengths, new-token positions); it holds none of the method's
arithmetic -- no slot computation, no gather, no scores, no softmax -- so the
CUDA library and the oracle each do that work on their own.

Shapes follow the Llama-class models the pages measure (32 layers, 32 heads
of dimension 128, fp16 K/V: "推理优化这件事，为什么值得反复复盘", sec. 4.1;
"LLM推理优化：从硬件瓶颈到KV Cache的工程实践", sec. 4.1), with the 8-kv-head
GQA variant of the 8B model.  Values are N(0, 1) drawn in fp32 and rounded to
fp16; physical block ids are a seeded random permutation of the pool, so a
request's blocks are scattered the way an allocator that recycles blocks
leaves them.

Conventions (the same readings the oracle documents):
  * cache tensors are fp16 [num_blocks, num_kv_heads, block_size, head_dim];
  * ``context_lens[b]`` counts the cached tokens including the one appended by
    this step; the appended token's logical position is ``positions[b]``
    (= context_lens[b] - 1);
  * ``block_tables`` is int32 [B, max_blocks]; entries a request does not own
    are -1 and are never read;
  * ``k_cache``/``v_cache`` hold the pool *before* this step's append; the
    slot that receives the new token holds an earlier random value.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

LAYERS = 32
HEAD_DIM = 128


@dataclass
class Case:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    block_tables: torch.Tensor   # int32 [B, max_blocks], -1 where unused
    context_lens: torch.Tensor   # int32 [B]
    positions: torch.Tensor      # int32 [B], logical position of the appended token
    q: torch.Tensor              # fp16 [B, Hq, D]
    k_new: torch.Tensor          # fp16 [B, Hkv, D]
    v_new: torch.Tensor          # fp16 [B, Hkv, D]
    k_cache: torch.Tensor        # fp16 [NB, Hkv, bs, D]
    v_cache: torch.Tensor        # fp16 [NB, Hkv, bs, D]
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def to(self, device) -> "Case":
        kw = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
              for k, v in self.__dict__.items()}
        return Case(**kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_fp16(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.float16)


def _blocks_needed(n_tokens: int, bs: int) -> int:
    return -(-n_tokens // bs)


def _tables_from_permutation(perm: torch.Tensor, blocks_per_seq, max_blocks: int,
                             shared_prefix=None) -> torch.Tensor:
    """Hand out consecutive runs of a permutation of the pool as block tables."""
    b = len(blocks_per_seq)
    bt = torch.full((b, max_blocks), -1, dtype=torch.int32)
    pos = 0
    if shared_prefix is not None:
        pos = len(shared_prefix)
    for i, n in enumerate(blocks_per_seq):
        row = []
        if shared_prefix is not None:
            row.extend(shared_prefix)
        row.extend(perm[pos:pos + n].tolist())
        pos += n
        bt[i, :len(row)] = torch.tensor(row, dtype=torch.int32)
    return bt


def _finish(name, hq, hkv, d, bs, nb, bt, ctx, g_vals, device, meta=None,
            peaky_fraction=0.0, peaky_factor=1.0) -> Case:
    b = bt.shape[0]
    ctx_t = torch.tensor(ctx, dtype=torch.int32)
    k_cache = torch.randn((nb, hkv, bs, d), generator=g_vals, device=device, dtype=torch.float32)
    v_cache = _normal_fp16((nb, hkv, bs, d), g_vals, device)
    q = _normal_fp16((b, hq, d), g_vals, device)
    k_new = torch.randn((b, hkv, d), generator=g_vals, device=device, dtype=torch.float32)
    v_new = _normal_fp16((b, hkv, d), g_vals, device)
    if peaky_fraction > 0.0:
        # a fraction of (token, all kv heads) K rows scaled before fp16 rounding
        row_pick = torch.rand((nb, 1, bs, 1), generator=g_vals, device=device) < peaky_fraction
        k_cache = torch.where(row_pick, k_cache * peaky_factor, k_cache)
        new_pick = torch.rand((b, 1, 1), generator=g_vals, device=device) < peaky_fraction
        k_new = torch.where(new_pick, k_new * peaky_factor, k_new)
    return Case(name=name, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                num_blocks=nb, block_tables=bt.to(device), context_lens=ctx_t.to(device),
                positions=(ctx_t - 1).to(device), q=q, k_new=k_new.to(torch.float16),
                v_new=v_new, k_cache=k_cache.to(torch.float16), v_cache=v_cache,
                scale=1.0 / math.sqrt(d), meta=dict(meta or {}))


def random_case(seed: int, context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int = 128,
                block_size: int = 16, extra_blocks: int = 3, device="cpu", name="random",
                peaky_fraction=0.0, peaky_factor=1.0) -> Case:
    """Ragged batch: request b holds context_lens[b] tokens (0 allowed), blocks scattered
    over a pool with `extra_blocks` blocks nobody owns."""
    ctx = [int(c) for c in context_lens]
    need = [_blocks_needed(c, block_size) for c in ctx]
    nb = sum(need) + extra_blocks
    g_struct = _gen(seed, "cpu")
    perm = torch.randperm(nb, generator=g_struct)
    bt = _tables_from_permutation(perm, need, max(1, max(need)))
    return _finish(name, num_q_heads, num_kv_heads, head_dim, block_size, nb, bt, ctx,
                   _gen(seed + 1, device), device, peaky_fraction=peaky_fraction,
                   peaky_factor=peaky_factor)


# --------------------------------------------------------------------------------------
# The five workload shapes.  Structure (context lengths, tables) depends on the
# workload seed only, so every layer of a request shares one block table;
# values depend on (seed, layer, step).
# --------------------------------------------------------------------------------------

def tiny(device="cpu", seed=1000) -> Case:
    """batch 1, 32 q = 32 kv heads, head_dim 128, context 512, block_size 16: 32 blocks
    drawn from a seeded permutation of a 64-block pool."""
    g = _gen(seed, "cpu")
    perm = torch.randperm(64, generator=g)
    bt = perm[:32].to(torch.int32).view(1, 32)
    return _finish("tiny", 32, 32, HEAD_DIM, 16, 64, bt, [512], _gen(seed + 1, device), device)


def mha7b_structure(seed=2000):
    g = _gen(seed, "cpu")
    ctx = torch.randint(200, 4001, (16,), generator=g).tolist()
    need = [_blocks_needed(c, 16) for c in ctx]
    nb = sum(need)
    perm = torch.randperm(nb, generator=g)
    bt = _tables_from_permutation(perm, need, max(need))
    return ctx, nb, bt


def mha7b(layer: int = 0, device="cpu", seed=2000) -> Case:
    """7B-shaped MHA decode: batch 16, 32 heads, head_dim 128, block_size 16, context
    lengths uniform in [200, 4000] per request; the pool holds exactly the requests' blocks."""
    ctx, nb, bt = mha7b_structure(seed)
    return _finish("mha7b", 32, 32, HEAD_DIM, 16, nb, bt, ctx,
                   _gen(seed + 1 + layer, device), device, meta={"layer": layer})


GQA_PREFILL = 2048
GQA_STEPS = 128


def gqa8b_structure(block_size=16, seed=3000):
    need = _blocks_needed(GQA_PREFILL + GQA_STEPS, block_size)
    nb = 64 * need
    g = _gen(seed + block_size, "cpu")
    perm = torch.randperm(nb, generator=g)
    bt = _tables_from_permutation(perm, [need] * 64, need)
    return nb, bt


def gqa8b(layer: int = 0, step: int = 1, block_size: int = 16, device="cpu", seed=3000) -> Case:
    """8B-shaped GQA decode: batch 64, 32 q / 8 kv heads, head_dim 128, 2048 prefilled
    tokens; decode step t (1..128) appends logical position 2047 + t, so ctx = 2048 + t.
    The pool is sized for 2176 tokens per request."""
    assert 1 <= step <= GQA_STEPS
    nb, bt = gqa8b_structure(block_size, seed)
    ctx = [GQA_PREFILL + step] * 64
    return _finish("gqa8b", 32, 8, HEAD_DIM, block_size, nb, bt, ctx,
                   _gen(seed + 10000 * block_size + 1000 * step + layer, device), device,
                   meta={"layer": layer, "step": step})


def shared_prefix_structure(seed=4000):
    g = _gen(seed, "cpu")
    suffix = torch.randint(128, 1025, (32,), generator=g).tolist()
    need = [_blocks_needed(s, 16) for s in suffix]
    nb = 64 + sum(need)
    perm = torch.randperm(nb, generator=g)
    prefix_ids = perm[:64].tolist()
    bt = _tables_from_permutation(perm, need, 64 + max(need), shared_prefix=prefix_ids)
    ctx = [1024 + s for s in suffix]
    return ctx, nb, bt, prefix_ids


def shared_prefix(layer: int = 0, device="cpu", seed=4000) -> Case:
    """batch 32, 32 q / 8 kv heads, block_size 16: every block table starts with the same
    64 blocks (a 1024-token common prefix) followed by a private suffix of 128..1024 tokens
    (the last of which is appended by this step)."""
    ctx, nb, bt, prefix_ids = shared_prefix_structure(seed)
    return _finish("shared_prefix", 32, 8, HEAD_DIM, 16, nb, bt, ctx,
                   _gen(seed + 1 + layer, device), device,
                   meta={"layer": layer, "prefix_blocks": prefix_ids})


LONG_CONTEXT = 32768


def long_context_structure(block_size=16, seed=5000):
    need = LONG_CONTEXT // block_size
    nb = 4 * need
    g = _gen(seed + block_size, "cpu")
    perm = torch.randperm(nb, generator=g)
    bt = _tables_from_permutation(perm, [need] * 4, need)
    return nb, bt


def long_context(layer: int = 0, block_size: int = 16, device="cpu", seed=5000) -> Case:
    """batch 4, 32 q / 8 kv heads, context 32768, block_size in {16, 32, 64, 128}; 1% of
    the token rows of K (all kv heads of that token) scaled by 8 before fp16 rounding,
    which makes the softmax peaky."""
    nb, bt = long_context_structure(block_size, seed)
    return _finish("long_context", 32, 8, HEAD_DIM, block_size, nb, bt, [LONG_CONTEXT] * 4,
                   _gen(seed + 10000 * block_size + 1 + layer, device), device,
                   meta={"layer": layer}, peaky_fraction=0.01, peaky_factor=8.0)


WORKLOADS = {
    "tiny": tiny,
    "mha7b": mha7b,
    "gqa8b": gqa8b,
    "shared_prefix": shared_prefix,
    "long_context": long_context,
}
