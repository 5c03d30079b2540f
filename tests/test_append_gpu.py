"""pkv_append on the GPU: bit-exact against the oracle's append over the WHOLE pool (every
untouched byte included), padding slots skipped."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import assert_no_device_error, host_inputs, oracle_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("hkv", [1, 8, 32])
def test_append_bit_exact_whole_pool(bs, hkv):
    case = workloads.random_case(100 + bs + hkv, [0, 1, bs - 1, bs, bs + 1, 3 * bs + 7, 700], 2 * hkv, hkv,
                                 block_size=bs, extra_blocks=5, device="cpu")
    h = host_inputs(case)
    oracle_step(h, case, decode=False)
    dev = case.to("cuda")
    slots = pkv.slot_mapping(case.block_tables, case.positions, bs).cuda()
    pkv.append(dev.k_cache, dev.v_cache, slots, dev.k_new, dev.v_new)
    assert np.array_equal(dev.k_cache.cpu().numpy().view(np.uint16), h["k_cache"].view(np.uint16))
    assert np.array_equal(dev.v_cache.cpu().numpy().view(np.uint16), h["v_cache"].view(np.uint16))
    assert_no_device_error()


def test_append_skips_negative_slots_and_copies_bits():
    # NaN/Inf/subnormal/-0 payloads must land bit for bit; slot -1 must not write anything
    nb, hkv, bs, d = 4, 2, 16, 128
    k_cache = torch.zeros((nb, hkv, bs, d), dtype=torch.float16, device="cuda")
    v_cache = torch.zeros_like(k_cache)
    special = np.array([0x7e00, 0x7c00, 0xfc00, 0x0001, 0x8000, 0x3c00, 0x7bff, 0x8400], np.uint16)
    k_new = torch.from_numpy(np.tile(special, 3 * hkv * d // 8).view(np.float16).reshape(3, hkv, d)).cuda()
    v_new = torch.from_numpy(np.tile(special[::-1].copy(), 3 * hkv * d // 8).view(np.float16)
                             .reshape(3, hkv, d)).cuda()
    slots = torch.tensor([5, -1, 63], dtype=torch.int64, device="cuda")
    pkv.append(k_cache, v_cache, slots, k_new, v_new)
    kc = k_cache.cpu().numpy().view(np.uint16).copy()
    ref = np.zeros_like(kc)
    kn = k_new.cpu().numpy().view(np.uint16)
    ref[0, :, 5, :] = kn[0]
    ref[3, :, 15, :] = kn[2]
    assert np.array_equal(kc, ref)
    vc = v_cache.cpu().numpy().view(np.uint16).copy()
    vref = np.zeros_like(vc)
    vn = v_new.cpu().numpy().view(np.uint16)
    vref[0, :, 5, :] = vn[0]
    vref[3, :, 15, :] = vn[2]
    assert np.array_equal(vc, vref)
    assert_no_device_error()


def test_append_many_tokens_matches_oracle():
    # T = 4096 tokens (a chunk of prefill) scattered over a shuffled pool
    rng = np.random.default_rng(5)
    nb, hkv, bs, d, t = 512, 8, 16, 128, 4096
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[::97] = -1
    k_cache = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    v_cache = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    k_new = rng.standard_normal((t, hkv, d)).astype(np.float16)
    v_new = rng.standard_normal((t, hkv, d)).astype(np.float16)
    kd, vd = torch.from_numpy(k_cache).cuda(), torch.from_numpy(v_cache).cuda()
    pkv.append(kd, vd, torch.from_numpy(slots).cuda(), torch.from_numpy(k_new).cuda(),
               torch.from_numpy(v_new).cuda())
    oracle.append(k_cache, v_cache, slots, k_new, v_new)
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), k_cache.view(np.uint16))
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), v_cache.view(np.uint16))
    assert_no_device_error()
