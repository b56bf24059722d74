"""Pins of the oracle's prefill (no GPU): prefill over a prompt is the
recurrence run token by token, so it must equal T chained decode steps, equal
the last snapshot of a speculative verify over the same tokens, and be
invariant to where the prompt is split into two calls."""
import numpy as np
import pytest
import torch

import oracle
from kda_linear_attention_gated_gb300 import workloads

pytestmark = pytest.mark.usefixtures("oracle_mod")


def pnp(pool):
    return pool.numpy().copy() if pool.dtype == torch.float32 else pool.view(torch.int16).numpy().view(np.uint16).copy()


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_prefill_equals_chained_decode(state_dtype):
    inp = workloads.make_prefill(lens=(9,), hv=2, k=16, v=32, num_slots=4, state_dtype=state_dtype,
                                 qkv_dtype=torch.float32, seed=1, reset_p=0.0, same_slot_p=1.0)
    pool = pnp(inp.pool)
    o = oracle.prefill(pool, inp.init_slot, inp.final_slot, inp.q, inp.k, inp.v, inp.a, inp.b,
                       cu_seqlens=inp.cu_seqlens)
    ref = pnp(inp.pool)
    if state_dtype == torch.float16:
        # the decode chain rounds to fp16 after every token, prefill only at the end: compare
        # against the fp32 pool twin instead, then round once
        twin = inp.pool.float().numpy().copy()
        outs = [oracle.decode_step(twin, inp.init_slot, inp.q[t:t + 1], inp.k[t:t + 1], inp.v[t:t + 1],
                                   inp.a[t:t + 1], inp.b[t:t + 1]) for t in range(9)]
        np.testing.assert_allclose(o, np.concatenate(outs), rtol=0, atol=1e-6)
        return
    outs = [oracle.decode_step(ref, inp.init_slot, inp.q[t:t + 1], inp.k[t:t + 1], inp.v[t:t + 1],
                               inp.a[t:t + 1], inp.b[t:t + 1]) for t in range(9)]
    np.testing.assert_allclose(o, np.concatenate(outs), rtol=0, atol=1e-6)  # the chain rounds to fp32 per token
    np.testing.assert_allclose(pool, ref, rtol=0, atol=1e-6)


def test_prefill_equals_last_verify_snapshot():
    inp = workloads.make_prefill(lens=(6, 6), hv=3, k=16, v=16, num_slots=20, state_dtype=torch.float16,
                                 qkv_dtype=torch.float32, seed=2, reset_p=0.5, same_slot_p=0.0)
    pool = pnp(inp.pool)
    o = oracle.prefill(pool, inp.init_slot, inp.final_slot, inp.q, inp.k, inp.v, inp.a, inp.b,
                       cu_seqlens=inp.cu_seqlens, reset=inp.reset)
    ref = pnp(inp.pool)
    snaps = np.full((2, 6), -1, np.int32)
    snaps[:, 5] = inp.final_slot.numpy()
    free = np.setdiff1d(np.arange(20), np.concatenate([inp.init_slot.numpy(), inp.final_slot.numpy()]))
    snaps[:, :5] = free[:10].reshape(2, 5)
    ov = oracle.spec_verify(ref, inp.init_slot, snaps, inp.q.reshape(2, 6, 3, 16), inp.k.reshape(2, 6, 3, 16),
                            inp.v.reshape(2, 6, 3, 16), inp.a.reshape(2, 6, 3, 16), inp.b.reshape(2, 6, 3),
                            reset=inp.reset)
    assert np.array_equal(o.reshape(2, 6, 3, 16), ov)
    fs = inp.final_slot.numpy()
    assert np.array_equal(pool[fs], ref[fs])


def test_split_prompt_equals_whole_prompt():
    inp = workloads.make_prefill(lens=(23,), hv=2, k=32, v=16, num_slots=6, state_dtype=torch.float32,
                                 qkv_dtype=torch.float32, seed=3, reset_p=1.0, same_slot_p=1.0, gate_scale=True)
    whole = pnp(inp.pool)
    ow = oracle.prefill(whole, inp.init_slot, inp.final_slot, inp.q, inp.k, inp.v, inp.a, inp.b,
                        cu_seqlens=inp.cu_seqlens, reset=inp.reset, a_log=inp.a_log, dt_bias=inp.dt_bias)
    # fp64 carry across the split: the first call's state goes to an fp32 slot, so allow its rounding
    part = pnp(inp.pool)
    o1 = oracle.prefill(part, inp.init_slot, inp.final_slot, inp.q[:10], inp.k[:10], inp.v[:10], inp.a[:10],
                        inp.b[:10], reset=inp.reset, a_log=inp.a_log, dt_bias=inp.dt_bias)
    o2 = oracle.prefill(part, inp.final_slot, inp.final_slot, inp.q[10:], inp.k[10:], inp.v[10:], inp.a[10:],
                        inp.b[10:], a_log=inp.a_log, dt_bias=inp.dt_bias)
    assert np.array_equal(o1, ow[:10])
    np.testing.assert_allclose(o2, ow[10:], rtol=0, atol=1e-6)
    np.testing.assert_allclose(part, whole, rtol=0, atol=1e-6)


def test_padding_and_unstored_final():
    inp = workloads.make_prefill(lens=(4, 5, 3), hv=2, k=16, v=16, num_slots=8, state_dtype=torch.float32,
                                 qkv_dtype=torch.float32, seed=4, reset_p=0.0, same_slot_p=0.0)
    init = inp.init_slot.clone()
    final = inp.final_slot.clone()
    init[0] = -1       # padding request
    final[1] = -1      # state not kept
    before = pnp(inp.pool)
    pool = pnp(inp.pool)
    o = oracle.prefill(pool, init, final, inp.q, inp.k, inp.v, inp.a, inp.b, cu_seqlens=inp.cu_seqlens)
    assert (o[:4] == 0).all() and (o[4:] != 0).any()
    changed = np.nonzero([not np.array_equal(pool[s], before[s]) for s in range(8)])[0].tolist()
    assert changed == [int(final[2])]


@pytest.mark.parametrize("reset", [0, 1])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_empty_first_part_split_equals_whole_prompt(state_dtype, reset):
    """A prompt split as 0 | T, init and final slots distinct: the empty call
    must leave the final slot holding the request's initial state (zero on a
    reset), so that the second call, from the final slot, reproduces the whole
    prompt bit for bit.  A rule that left an empty request alone would make
    the second call start from whatever the final slot held before."""
    T = 11
    inp = workloads.make_prefill(lens=(T,), hv=2, k=16, v=32, num_slots=6, state_dtype=state_dtype,
                                 qkv_dtype=torch.float32, seed=5, reset_p=float(reset), same_slot_p=0.0)
    assert int(inp.init_slot[0]) != int(inp.final_slot[0])
    rs = np.array([reset], np.uint8)
    whole = pnp(inp.pool)
    ow = oracle.prefill(whole, inp.init_slot, inp.final_slot, inp.q, inp.k, inp.v, inp.a, inp.b,
                        cu_seqlens=inp.cu_seqlens, reset=rs)
    part = pnp(inp.pool)
    empty = lambda x: x[:0]  # noqa: E731
    o1 = oracle.prefill(part, inp.init_slot, inp.final_slot, *(empty(x) for x in (inp.q, inp.k, inp.v, inp.a, inp.b)),
                        cu_seqlens=np.array([0, 0], np.int32), reset=rs)
    assert o1.shape == (0, 2, 32)
    f, i = int(inp.final_slot[0]), int(inp.init_slot[0])
    before = pnp(inp.pool)
    if reset:
        assert not part[f].any()
    else:
        assert part[f].tobytes() == before[i].tobytes()
    others = [s for s in range(6) if s != f]
    assert part[others].tobytes() == before[others].tobytes()
    o2 = oracle.prefill(part, inp.final_slot, inp.final_slot, inp.q, inp.k, inp.v, inp.a, inp.b,
                        cu_seqlens=inp.cu_seqlens)
    assert np.array_equal(o2, ow)
    assert part.tobytes() == whole.tobytes()


def test_empty_middle_part_changes_nothing():
    """T1 | 0 | T2 on one slot equals T1 | T2: an empty call from a slot to the
    same slot rewrites its state with itself."""
    inp = workloads.make_prefill(lens=(14,), hv=2, k=16, v=16, num_slots=4, state_dtype=torch.float16,
                                 qkv_dtype=torch.float32, seed=6, reset_p=0.0, same_slot_p=1.0)
    s = inp.init_slot
    a = pnp(inp.pool)
    oracle.prefill(a, s, s, inp.q[:5], inp.k[:5], inp.v[:5], inp.a[:5], inp.b[:5])
    b = a.copy()
    oracle.prefill(b, s, s, inp.q[:0], inp.k[:0], inp.v[:0], inp.a[:0], inp.b[:0],
                   cu_seqlens=np.array([0, 0], np.int32))
    assert a.tobytes() == b.tobytes()
    oracle.prefill(a, s, s, inp.q[5:], inp.k[5:], inp.v[5:], inp.a[5:], inp.b[5:])
    oracle.prefill(b, s, s, inp.q[5:], inp.k[5:], inp.v[5:], inp.a[5:], inp.b[5:])
    assert a.tobytes() == b.tobytes()
