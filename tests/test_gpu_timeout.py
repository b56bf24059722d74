"""The bounded pipeline waits, exercised without a fault.

With the test hook KDA_LAUNCH_TEST_WITHHOLD_STATE (include/kda.h) every tile
arms its state tile's barrier but the copy is never issued, so each wait on it
runs out at its 1 s bound.  The call must then report KDA_ERR_TIMEOUT through
the status word, write neither states nor outputs of those tiles, and leave the
context usable: the next plain call on the same stream matches the oracle.
Nothing here faults, traps or spins without a bound.
"""
import time

import numpy as np
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import workloads

from _harness import (assert_out_match, assert_pool_match, gpu_decode, gpu_verify, lib_for, oracle_decode,
                      oracle_verify, pool_np)

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]

SD = [torch.float32, torch.float16]


@pytest.mark.parametrize("state_dtype", SD)
def test_withheld_state_copy_times_out_and_writes_nothing(state_dtype):
    lib = lib_for(state_dtype)
    inp = workloads.make_decode(n=4, hv=2, k=64, v=64, num_slots=8, state_dtype=state_dtype, seed=81)
    d = inp.to("cuda")
    before = pool_np(d.pool.cpu())
    o = torch.full((4, 2, 64), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    lib.kda_decode_step(d.pool, d.init_slot, d.q, d.k, d.v, d.a, d.b, o, status,
                        flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(status.item()) == kda.KDA_ERR_TIMEOUT
    assert 0.9 <= elapsed < 30.0, f"the bounded waits took {elapsed:.2f} s"
    assert pool_np(d.pool.cpu()).tobytes() == before.tobytes()
    assert torch.isnan(o).all()
    # the context still works: a plain call on the same inputs matches the oracle
    gpool, o2, st = gpu_decode(inp)
    assert st == 0
    ref, o_ref = oracle_decode(inp)
    assert_out_match(o2, o_ref, state_dtype, "o after the timeout")
    assert_pool_match(gpool, ref, inp.init_slot.numpy(), "pool after the timeout")


def test_withheld_state_copy_times_out_two_tiles_a_cta():
    """An fp16-pool launch past one wave (N=64 x HV=12 x 2 column tiles) runs
    two tiles a CTA: with both state copies withheld, each CTA's first wait
    runs out, it waits (bounded) on both tiles' barriers, and the call reports
    the timeout with nothing written; the context stays usable."""
    lib = lib_for(torch.float16)
    inp = workloads.make_decode(n=64, hv=12, k=64, v=128, num_slots=72, state_dtype=torch.float16, seed=84)
    d = inp.to("cuda")
    before = pool_np(d.pool.cpu())
    o = torch.full((64, 12, 128), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    lib.kda_decode_step(d.pool, d.init_slot, d.q, d.k, d.v, d.a, d.b, o, status,
                        flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(status.item()) == kda.KDA_ERR_TIMEOUT
    assert 0.9 <= elapsed < 30.0, f"the bounded waits took {elapsed:.2f} s"
    assert pool_np(d.pool.cpu()).tobytes() == before.tobytes()
    assert torch.isnan(o).all()
    gpool, o2, st = gpu_decode(inp)
    assert st == 0
    ref, o_ref = oracle_decode(inp)
    assert_out_match(o2, o_ref, torch.float16, "o after the timeout")
    assert_pool_match(gpool, ref, inp.init_slot.numpy(), "pool after the timeout")


@pytest.mark.parametrize("state_dtype", SD)
def test_withheld_state_copy_times_out_in_verify(state_dtype):
    lib = lib_for(state_dtype)
    inp = workloads.make_verify(n=2, t=3, hv=2, k=64, v=64, num_slots=12, state_dtype=state_dtype, seed=82)
    d = inp.to("cuda")
    before = pool_np(d.pool.cpu())
    o = torch.full((2, 3, 2, 64), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_spec_verify(d.pool, d.init_slot, d.snap_slot, d.q, d.k, d.v, d.a, d.b, o, status,
                        flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_ERR_TIMEOUT
    assert pool_np(d.pool.cpu()).tobytes() == before.tobytes()  # no snapshot stored
    assert torch.isnan(o).all()
    gpool, o2, st = gpu_verify(inp)
    assert st == 0
    ref, o_ref = oracle_verify(inp)
    assert_out_match(o2, o_ref, state_dtype, "o after the timeout")
    assert_pool_match(gpool, ref, inp.snap_slot.numpy(), "snapshots after the timeout")


def test_reset_requests_need_no_state_and_do_not_wait():
    """A request that resets reads no state, so the hook leaves it alone: with
    every request reset the call completes normally and matches the oracle."""
    inp = workloads.make_decode(n=4, hv=2, k=64, v=64, num_slots=8, state_dtype=torch.float32, seed=83)
    inp.reset = torch.ones(4, dtype=torch.uint8)
    d = inp.to("cuda")
    o = torch.empty(4, 2, 64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib_for(torch.float32).kda_decode_step(d.pool, d.init_slot, d.q, d.k, d.v, d.a, d.b, o, status, reset=d.reset,
                                           flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, o_ref = oracle_decode(inp)
    assert_out_match(o.cpu(), o_ref, torch.float32, "o")
    assert np.isfinite(o.cpu().numpy()).all()
