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



def test_decode_bytes_model_by_hand():
    # two requests (ctx 20 and 33), Hkv 2, Hq 4, D 128, bs 16
    ctx, hkv, hq, d, bs = [20, 33], 2, 4, 128, 16
    kv_row = d * 2                                   # one fp16 K or V row
    tables = (2 + 3) * 4 + 4 * 2                     # ceil(20/16) + ceil(33/16) ids, context lengths
    qo = 2 * 2 * hq * d * 2                          # q in, out back
    fp16 = 53 * hkv * 2 * kv_row + qo + tables
    assert bench.decode_bytes(ctx, hkv, hq, d, bs) == fp16
    # int8 keys: a key row is 128 codes + a float32 scale; values stay fp16
    assert bench.decode_bytes(ctx, hkv, hq, d, bs, kv="int8k") == 53 * hkv * ((d + 4) + kv_row) + qo + tables
    # int8 keys and values; fp8 keys and values (the same bytes)
    assert bench.decode_bytes(ctx, hkv, hq, d, bs, kv="int8kv") == 53 * hkv * 2 * (d + 4) + qo + tables
    assert bench.decode_bytes(ctx, hkv, hq, d, bs, kv="fp8kv") == 53 * hkv * 2 * (d + 4) + qo + tables
    # several new tokens per request: q and out counted per token
    assert bench.decode_bytes(ctx, hkv, hq, d, bs, q_len=3) == fp16 + 2 * qo
    # a shared 16-token prefix counted once: unique tokens = 20 + 33 - 16
    assert bench.decode_bytes(ctx, hkv, hq, d, bs, unique_prefix_tokens=16) == fp16 - 16 * hkv * 2 * kv_row


def test_decode_bytes_of_the_mha7b_workload():
    # the 7B-shaped workload's algorithmic bytes per layer, as the results quote them (480.89 MB)
    import workloads
    ctx, nb, bt = workloads.mha7b_structure()
    assert abs(bench.decode_bytes(ctx, 32, 32, 128, 16) / 1e6 - 480.89) < 0.01


@pytest.mark.parametrize("argv", [
    ["--warmup", "2"],                                                   # fewer than 3 warm-up steps
    ["--workload", "shared_prefix", "--kv", "int8k"],                    # the cascade reads fp16 K/V
    ["--workload", "shared_prefix", "--kv", "int8kv"],
    ["--workload", "shared_prefix", "--kv", "fp8kv"],
    ["--query-len", "4", "--kv", "fp8kv"],
    ["--query-len", "4", "--kv", "int8k"],                               # several tokens: fp16 path only
    ["--query-len", "4", "--workload", "shared_prefix"],
    ["--query-len", "2", "--impl", "reference"],                         # the reference arm times single tokens
    ["--kv", "fp8"],                                                     # not a cache format
])
def test_bench_refuses_unsupported_combinations(argv):
    with pytest.raises(SystemExit) as e:
        bench.main(argv)
    assert e.value.code == 2
