"""GPU checkpoint flush and load (kda_ckpt_flush / kda_ckpt_load) against the
oracle's element copies: whole states through the address function, bit for
bit (ROCm/ATOM pull request 2945, Changes: under ReplaySSM the checkpoint load
and the flush go through state_at)."""
import numpy as np
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import workloads

import oracle
from _harness import lib_for, pool_np

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_flush_then_load_round_trip(state_dtype):
    lib = lib_for(state_dtype)
    g = torch.Generator().manual_seed(70)
    pool = workloads.make_pool(g, 256, 12, 128, 128, state_dtype)
    plane = workloads.make_pool(g, 96, 12, 128, 128, state_dtype)
    slots = torch.randperm(256, generator=g)[:64].to(torch.int32)
    entries = torch.randperm(96, generator=g)[:64].to(torch.int32)
    slots[5], entries[9] = -1, -1  # skipped pairs
    ref_pool, ref_plane = pool_np(pool), pool_np(plane)
    oracle.ckpt_transfer(ref_pool, ref_plane, slots.numpy(), entries.numpy(), load=False)
    dp, dl = pool.cuda(), plane.cuda()
    ds, de = slots.cuda(), entries.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_ckpt_flush(dp, dl, ds, de, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(pool_np(dl.cpu()), ref_plane) and np.array_equal(pool_np(dp.cpu()), ref_pool)
    # load the entries back into a scrambled pool: the flushed slots come back bit for bit
    dp2 = workloads.make_pool(g, 256, 12, 128, 128, state_dtype).cuda()
    ref2 = pool_np(dp2.cpu())
    oracle.ckpt_transfer(ref2, ref_plane, slots.numpy(), entries.numpy(), load=True)
    lib.kda_ckpt_load(dp2, dl, ds, de, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = pool_np(dp2.cpu())
    assert np.array_equal(got, ref2)
    keep = ((slots >= 0) & (entries >= 0)).numpy()
    assert np.array_equal(got[slots.numpy()[keep]], pool_np(pool)[slots.numpy()[keep]])


def test_out_of_range_pair_sets_status_and_is_skipped():
    lib = lib_for(torch.float32)
    pool = torch.randn(8, 2, 16, 16, device="cuda")
    plane = torch.zeros(4, 2, 16, 16, device="cuda")
    slots = torch.tensor([1, 8, 2], dtype=torch.int32, device="cuda")
    entries = torch.tensor([0, 1, 3], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_ckpt_flush(pool, plane, slots, entries, status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_ERR_SLOT_RANGE
    assert torch.equal(plane[0], pool[1]) and torch.equal(plane[3], pool[2]) and not plane[1].any()


def test_image_of_the_other_dtype_is_refused():
    lib16 = lib_for(torch.float16)
    lib32 = lib_for(torch.float32)
    pool = torch.zeros(4, 2, 16, 16, dtype=torch.float16, device="cuda")
    plane = torch.zeros(2, 2, 16, 16, dtype=torch.float16, device="cuda")
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp32_id = lib32.kda_layout_id(kda.PoolDesc(pool.data_ptr(), kda.KDA_F32, 2, 16, 16, 4, 2 * 16 * 16))
    with pytest.raises(kda.KdaError) as e:
        lib16.kda_ckpt_load(pool, plane, ids, ids, status, layout_id=fp32_id)
    assert e.value.code == kda.KDA_ERR_LAYOUT
