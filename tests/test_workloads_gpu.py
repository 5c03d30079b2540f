"""The five workload shapes at full size, in the launch configuration the benchmark times
(pkv.append + pkv.decode_attention with the default split), against the oracle on
every request and head of the sampled layers / steps."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, assert_no_device_error, gpu_step, host_inputs, max_err, oracle_step

pytestmark = pytest.mark.gpu


def check(case):
    h = host_inputs(case)                 # host copies before any library kernel runs
    ref = oracle_step(h, case)
    out = gpu_step(case)
    err = max_err(out, ref)
    # the append is bit-exact: compare the slots this step wrote
    slots = oracle.slot_mapping(h["block_tables"], h["positions"], case.block_size)
    blk, off = slots // case.block_size, slots % case.block_size
    got_k = case.k_cache[torch.from_numpy(blk).cuda(), :, torch.from_numpy(off).cuda()].cpu().numpy()
    assert np.array_equal(got_k.view(np.uint16), h["k_cache"][blk, :, off].view(np.uint16))
    assert_no_device_error()
    del case
    torch.cuda.empty_cache()
    return err


@pytest.mark.parametrize("layer", [0, 31])
def test_mha7b(layer):
    err = check(workloads.mha7b(layer, device="cuda"))
    assert err <= ATTN_TOL, err


@pytest.mark.parametrize("bs", [16, 64])
@pytest.mark.parametrize("layer,step", [(0, 1), (31, 64), (0, 128)])
def test_gqa8b(bs, layer, step):
    err = check(workloads.gqa8b(layer, step, bs, device="cuda"))
    assert err <= ATTN_TOL, err


@pytest.mark.parametrize("layer", [0, 31])
def test_shared_prefix(layer):
    case = workloads.shared_prefix(layer, device="cuda")
    h = host_inputs(case)
    # reference on an un-shared pool: every request gets private copies of the 64 prefix blocks
    prefix = case.meta["prefix_blocks"]
    b = case.num_seqs
    bt = h["block_tables"].copy()
    kc, vc = h["k_cache"], h["v_cache"]
    extra_k = np.concatenate([kc[prefix]] * b)
    extra_v = np.concatenate([vc[prefix]] * b)
    for i in range(b):
        bt[i, :64] = case.num_blocks + i * 64 + np.arange(64)
    h2 = dict(h, k_cache=np.concatenate([kc, extra_k]), v_cache=np.concatenate([vc, extra_v]), block_tables=bt)
    ref = oracle_step(h2, case)
    out = gpu_step(case)
    assert max_err(out, ref) <= ATTN_TOL
    assert_no_device_error()


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_long_context(bs):
    err = check(workloads.long_context(0, bs, device="cuda"))
    assert err <= ATTN_TOL, err
