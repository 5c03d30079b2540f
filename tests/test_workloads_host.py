"""The seeded workload generators (CPU only): each workload has the structure its definition
states — batch, heads, context lengths, pool size, block tables that cover every context with
distinct blocks (a shared prefix only where the workload has one) — and the same seed gives the
same bytes."""
import torch

import workloads


def owned_blocks(bt, ctx, bs):
    """The physical ids each request's context covers, per request."""
    return [bt[b, : -(-c // bs)].tolist() for b, c in enumerate(ctx)]


def assert_valid_tables(bt, ctx, nb, bs, shared=()):
    assert bt.dtype == torch.int32
    rows = owned_blocks(bt, ctx, bs)
    for b, row in enumerate(rows):
        assert all(0 <= i < nb for i in row), b
        assert (bt[b, len(row):] == -1).all() or len(row) == bt.shape[1]
    private = [i for row in rows for i in row[len(shared):]]
    assert len(private) == len(set(private)), "a private block is used twice"
    assert not set(private) & set(shared)
    for row in rows:
        assert row[: len(shared)] == list(shared)


def test_tiny():
    c = workloads.tiny()
    assert (c.num_seqs, c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size, c.num_blocks) == (1, 32, 32, 128,
                                                                                                  16, 64)
    assert c.context_lens.tolist() == [512] and c.positions.tolist() == [511]
    assert_valid_tables(c.block_tables, [512], 64, 16)
    assert c.k_cache.dtype == torch.float16 and tuple(c.k_cache.shape) == (64, 32, 16, 128)


def test_mha7b_structure():
    ctx, nb, bt = workloads.mha7b_structure()
    assert len(ctx) == 16 and all(200 <= c <= 4000 for c in ctx)
    assert nb == sum(-(-c // 16) for c in ctx)  # the pool holds exactly the requests' blocks
    assert_valid_tables(bt, ctx, nb, 16)
    assert sorted(i for row in owned_blocks(bt, ctx, 16) for i in row) == list(range(nb))
    ctx2, nb2, bt2 = workloads.mha7b_structure()
    assert ctx2 == ctx and nb2 == nb and torch.equal(bt2, bt)


def test_gqa8b_structure():
    for bs in (16, 64):
        nb, bt = workloads.gqa8b_structure(bs)
        need = -(-(workloads.GQA_PREFILL + workloads.GQA_STEPS) // bs)
        assert nb == 64 * need and tuple(bt.shape) == (64, need)
        assert_valid_tables(bt, [workloads.GQA_PREFILL + workloads.GQA_STEPS] * 64, nb, bs)


def test_shared_prefix_structure():
    ctx, nb, bt, prefix = workloads.shared_prefix_structure()
    assert len(ctx) == 32 and all(1024 + 128 <= c <= 1024 + 1024 for c in ctx)
    assert len(prefix) == 64
    assert nb == 64 + sum(-(-(c - 1024) // 16) for c in ctx)
    assert_valid_tables(bt, ctx, nb, 16, shared=prefix)


def test_long_context_structure():
    for bs in (16, 32, 64, 128):
        nb, bt = workloads.long_context_structure(bs)
        assert nb == 4 * 32768 // bs
        assert_valid_tables(bt, [32768] * 4, nb, bs)


def test_random_case_is_seeded_and_shaped():
    a = workloads.random_case(5, [0, 1, 17, 300], 8, 2, block_size=32, extra_blocks=3)
    b = workloads.random_case(5, [0, 1, 17, 300], 8, 2, block_size=32, extra_blocks=3)
    for name in ("block_tables", "context_lens", "positions", "q", "k_new", "v_new", "k_cache", "v_cache"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.float16 else x,
                           y.view(torch.int16) if y.dtype == torch.float16 else y), name
    assert a.context_lens.tolist() == [0, 1, 17, 300]
    assert a.positions.tolist()[1:] == [0, 16, 299]
    assert_valid_tables(a.block_tables, [0, 1, 17, 300], a.num_blocks, 32)
    assert tuple(a.q.shape) == (4, 8, 128) and tuple(a.k_new.shape) == (4, 2, 128)
    c = workloads.random_case(6, [0, 1, 17, 300], 8, 2, block_size=32, extra_blocks=3)
    assert not torch.equal(c.q.view(torch.int16), a.q.view(torch.int16))
