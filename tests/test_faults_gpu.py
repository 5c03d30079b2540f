"""Bad indices coming from device memory are caught by the kernels' own bounds checks: they are
clamped or skipped (every access stays inside the buffers), recorded in the device error word,
and the context stays usable.  Argument errors are refused on the host before any launch."""
import numpy as np
import pytest
import torch

import paged_kv_cache_278_gb300 as pkv
import workloads
from gpu_util import ATTN_TOL, gpu_step, host_inputs, max_err, oracle_step

pytestmark = pytest.mark.gpu


def fresh(seed=1):
    pkv.device_error()  # clear
    return workloads.random_case(seed, [100, 700, 40], 8, 2, block_size=16, extra_blocks=3).to("cuda")


def test_block_id_out_of_range_is_recorded():
    case = fresh()
    case.block_tables[1, 2] = case.num_blocks + 5          # inside the context of request 1
    out = torch.empty_like(case.q)
    ws = pkv.make_workspace(3, 8, case.max_blocks_per_seq * 16, "cuda")
    pkv.decode_attention(out, case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                         case.scale, workspace=ws)
    assert pkv.device_error() == pkv.PKV_DEV_BAD_BLOCK_ID
    assert pkv.device_error() == pkv.PKV_DEV_OK            # cleared by the read
    case.block_tables[1, 2] = -7
    pkv.decode_attention(out, case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                         case.scale, workspace=ws)
    assert pkv.device_error() == pkv.PKV_DEV_BAD_BLOCK_ID


def test_context_longer_than_table_is_recorded():
    case = fresh(2)
    case.context_lens[0] = case.max_blocks_per_seq * 16 + 1
    out = torch.empty_like(case.q)
    ws = pkv.make_workspace(3, 8, case.max_blocks_per_seq * 16, "cuda")
    pkv.decode_attention(out, case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                         case.scale, workspace=ws)
    assert pkv.device_error() == pkv.PKV_DEV_BAD_CONTEXT


def test_slot_out_of_range_is_skipped_and_recorded():
    case = fresh(3)
    before_k = case.k_cache.clone()
    slots = torch.tensor([case.num_blocks * 16, -1, case.num_blocks * 16 + 99], dtype=torch.int64,
                         device="cuda")
    pkv.append(case.k_cache, case.v_cache, slots, case.k_new, case.v_new)
    assert pkv.device_error() == pkv.PKV_DEV_BAD_SLOT
    assert torch.equal(case.k_cache, before_k)


def test_context_is_usable_after_recorded_errors():
    case = workloads.random_case(4, [300, 1200], 8, 2, block_size=16)
    h = host_inputs(case)
    ref = oracle_step(h, case)
    out = gpu_step(case.to("cuda"))
    assert max_err(out, ref) <= ATTN_TOL
    assert pkv.device_error() == pkv.PKV_DEV_OK


def test_host_side_argument_errors():
    case = fresh(5)
    out = torch.empty_like(case.q)
    with pytest.raises(pkv.PkvError) as e:   # split needed (tables of two default partitions), no workspace
        nblk = 2 * pkv.PKV_DEFAULT_PARTITION // 16
        big = torch.zeros((3, nblk), dtype=torch.int32, device="cuda")
        pkv.decode_attention(out, case.q, case.k_cache, case.v_cache, big, case.context_lens, case.scale)
    assert e.value.status == -5
    with pytest.raises(pkv.PkvError):        # workspace one byte short
        need = pkv.decode_workspace_size(3, 8, nblk * 16)
        ws = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
        pkv.decode_attention(out, case.q, case.k_cache, case.v_cache, big, case.context_lens, case.scale,
                             workspace=ws)
    with pytest.raises(ValueError):          # wrong dtype caught by the binding
        pkv.decode_attention(out.float(), case.q, case.k_cache, case.v_cache, case.block_tables,
                             case.context_lens, case.scale)
    with pytest.raises(pkv.PkvError) as e:   # head_dim 64 is not supported by the decode kernels
        kc = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device="cuda")
        q = torch.zeros((3, 8, 64), dtype=torch.float16, device="cuda")
        pkv.decode_attention(torch.empty_like(q), q, kc, kc, case.block_tables, case.context_lens, 0.1)
    assert e.value.status == -2
    assert pkv.device_error() == pkv.PKV_DEV_OK
