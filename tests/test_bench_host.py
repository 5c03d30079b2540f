"""Host logic of bench.py without a GPU: the whole-job reduction over ranks (gloo, world size 2),
the bytes model, and the reference arm's argument handling."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, units = bench.reduce_over_ranks(1.0 + rank, 100.0 * (rank + 1), world)
    q.put((rank, ms, units))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, units in got:
        assert ms == 2.0          # slowest rank
        assert units == 300.0     # units of all ranks


def test_reduce_single_rank_is_identity():
    assert bench.reduce_over_ranks(3.5, 7.0, 1) == (3.5, 7.0)


def test_decode_bytes_model():
    # K+V of every token, q and out per head, table entries, context lengths
    b = bench.decode_bytes([16, 17], num_kv_heads=2, num_q_heads=8, head_dim=128, bs=16)
    assert b == 2 * 33 * 2 * 128 * 2 + 2 * 2 * 8 * 128 * 2 + (1 + 2) * 4 + 4 * 2
    # a shared prefix counts once
    shared = bench.decode_bytes([1100, 1200], 8, 32, 128, 16, unique_prefix_tokens=1024)
    assert shared == bench.decode_bytes([1100, 1200], 8, 32, 128, 16) - 1024 * 8 * 128 * 2 * 2


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_kernel_hash_ignores_comments_not_code():
    src = """// header\n__global__ void k(int *p) { /* note */ p[0] = 1; }  // trailing\n"""
    same = """// another header\n__global__ void k(int *p) {\n    p[0] = 1;\n}\n"""
    changed = """__global__ void k(int *p) { p[0] = 2; }\n"""
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(changed)

