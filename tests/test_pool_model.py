"""Host block pool against a plain Python model (CPU only): random sequences of request
creation and growth, single-token appends with copy-on-write, forks, swaps between a device
pool and a host pool, and releases.  After every call the library's free counts and reference
counts must equal the model's, every live table entry must be a held block, and every failing
call (too few blocks, a shared block that may not leave) must change nothing."""
import random

import pytest
import torch

import paged_kv_cache_278_gb300 as pkv
from paged_kv_cache_278_gb300 import _lib

BS = 16
MAX_BLOCKS = 24
NB = (96, 48)  # device pool, host swap pool


class Model:
    def __init__(self):
        self.count = [dict(), dict()]  # per pool: block id -> references

    def free_blocks(self, p):
        return NB[p] - sum(1 for c in self.count[p].values() if c > 0)

    def take(self, p, i):
        assert self.count[p].get(i, 0) == 0, f"pool {p} handed out held block {i}"
        self.count[p][i] = 1

    def ref(self, p, i, d):
        self.count[p][i] = self.count[p].get(i, 0) + d
        assert self.count[p][i] >= 0


def nblk(tokens):
    return -(-tokens // BS)


def check(pools, model, reqs):
    for p in (0, 1):
        assert pools[p].num_free() == model.free_blocks(p)
        for i in range(NB[p]):
            assert pools[p].refcount(i) == model.count[p].get(i, 0), (p, i)
    for r in reqs:
        for k in range(nblk(r["tokens"])):
            i = int(r["row"][k])
            assert 0 <= i < NB[r["pool"]] and model.count[r["pool"]].get(i, 0) >= 1


def expect_error(fn, status):
    with pytest.raises(pkv.PkvError) as e:
        fn()
    assert e.value.status == status


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_pool_matches_model(seed):
    rng = random.Random(seed)
    pools = (pkv.BlockPool(NB[0], seed=seed), pkv.BlockPool(NB[1], seed=seed + 100))
    model = Model()
    reqs = []
    for _ in range(400):
        op = rng.choice(["new", "new", "append", "append", "append", "fork", "free", "swap"])
        if op == "new" or not reqs:
            tokens = rng.randint(1, 160)
            row = torch.full((MAX_BLOCKS,), -1, dtype=torch.int32)
            if nblk(tokens) > model.free_blocks(0):
                expect_error(lambda: pools[0].reserve(row, 0, tokens, BS), _lib.PKV_ERR_OUT_OF_BLOCKS)
                assert (row == -1).all()
            else:
                pools[0].reserve(row, 0, tokens, BS)
                for k in range(nblk(tokens)):
                    model.take(0, int(row[k]))
                reqs.append({"pool": 0, "row": row, "tokens": tokens})
        elif op == "append":
            r = rng.choice(reqs)
            p, row, t = r["pool"], r["row"], r["tokens"]
            if t >= MAX_BLOCKS * BS:
                continue
            before = row.clone()
            shared = t % BS != 0 and model.count[p][int(row[t // BS])] > 1
            needs_block = t % BS == 0 or shared
            if needs_block and model.free_blocks(p) == 0:
                expect_error(lambda: pools[p].prepare_append(row, t, BS), _lib.PKV_ERR_OUT_OF_BLOCKS)
                assert torch.equal(row, before)
            else:
                pair = pools[p].prepare_append(row, t, BS)
                if t % BS == 0:
                    assert pair is None
                    model.take(p, int(row[t // BS]))
                elif shared:
                    old, new = pair
                    assert old == int(before[t // BS]) and new == int(row[t // BS]) and new != old
                    model.ref(p, old, -1)
                    model.take(p, new)
                else:
                    assert pair is None and torch.equal(row, before)
                r["tokens"] = t + 1
        elif op == "fork":
            src = rng.choice(reqs)
            n = rng.randint(1, src["tokens"])
            row = torch.full((MAX_BLOCKS,), -1, dtype=torch.int32)
            pools[src["pool"]].fork(src["row"], row, n, BS)
            for k in range(nblk(n)):
                assert int(row[k]) == int(src["row"][k])
                model.ref(src["pool"], int(row[k]), +1)
            reqs.append({"pool": src["pool"], "row": row, "tokens": n})
        elif op == "free":
            r = reqs.pop(rng.randrange(len(reqs)))
            pools[r["pool"]].free_table(r["row"], r["tokens"], BS)
            for k in range(nblk(r["tokens"])):
                model.ref(r["pool"], int(r["row"][k]), -1)
        else:  # swap to the other pool
            r = rng.choice(reqs)
            p, q, n = r["pool"], 1 - r["pool"], nblk(r["tokens"])
            before = r["row"].clone()
            if any(model.count[p][int(r["row"][k])] > 1 for k in range(n)):
                expect_error(lambda: pools[p].swap_to(pools[q], r["row"], r["tokens"], BS), _lib.PKV_ERR_INVALID_ARG)
                assert torch.equal(r["row"], before)
            elif n > model.free_blocks(q):
                expect_error(lambda: pools[p].swap_to(pools[q], r["row"], r["tokens"], BS),
                             _lib.PKV_ERR_OUT_OF_BLOCKS)
                assert torch.equal(r["row"], before)
            else:
                src, dst = pools[p].swap_to(pools[q], r["row"], r["tokens"], BS)
                assert src.tolist() == before[:n].tolist() and dst.tolist() == r["row"][:n].tolist()
                for k in range(n):
                    model.ref(p, int(src[k]), -1)
                    model.take(q, int(dst[k]))
                r["pool"] = q
        check(pools, model, reqs)
    for r in reqs:
        pools[r["pool"]].free_table(r["row"], r["tokens"], BS)
    assert pools[0].num_free() == NB[0] and pools[1].num_free() == NB[1]
    pools[0].close()
    pools[1].close()
