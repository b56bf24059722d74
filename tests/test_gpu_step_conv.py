"""GPU parity of the speculative step with the short convolution fused in front
(kda_step_conv).

Bit for bit against the two-kernel path on the same inputs: kda_conv_step over
the same requests (cu_seqlens, accepted, reset; a padding request's window slot
-1), then kda_step with q, k and v taken from the conv's y.  Pool, window, y
and o must be identical and the read counters back at zero.  Then against the
fp64 oracle: the conv's y and window against the oracle's conv_step, and the
recurrence against the oracle's step fed the kernel's own q/k/v values.
"""
import numpy as np
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import workloads

import oracle
from _harness import assert_out_match, assert_pool_match, lib_for, pool_np
from test_gpu_conv import assert_y16_match, storage
from test_gpu_conv_decode import bits

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]

PDL, EARLY = kda.KDA_LAUNCH_PDL, kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE


def split_y(y, inp):
    total, hv, K, V = y.shape[0], inp.pool.shape[1], inp.pool.shape[2], inp.pool.shape[3]
    h = inp.h_qk
    return (y[:, : h * K].reshape(total, h, K).contiguous(), y[:, h * K: 2 * h * K].reshape(total, h, K).contiguous(),
            y[:, 2 * h * K:].reshape(total, hv, V).contiguous())


def two_kernels(d, inp, pool, W, flags=0):
    lib = lib_for(inp.pool.dtype)
    total, hv, V = inp.x.shape[0], inp.pool.shape[1], inp.pool.shape[3]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full_like(d.x, float("nan"))
    lib.kda_conv_step(W, d.conv_slot, d.x, d.weight, y, st, bias=d.bias, cu_seqlens=d.cu_seqlens, max_t=inp.max_t,
                      accepted=d.accepted, reset=d.reset, flags=flags)
    q, k, v = split_y(y, inp)
    o = torch.full((total, hv, V), float("nan"), device="cuda")
    lib.kda_step(pool, d.slot_table, q, k, v, d.a, d.b, o, st, cu_seqlens=d.cu_seqlens, max_t=inp.max_t,
                 accepted=d.accepted, reset=d.reset, a_log=d.a_log, dt_bias=d.dt_bias, flags=flags)
    return o, y, st


def fused(d, inp, pool, W, counters, flags=0, with_y=True):
    lib = lib_for(inp.pool.dtype)
    total, hv, V = inp.x.shape[0], inp.pool.shape[1], inp.pool.shape[3]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full_like(d.x, float("nan")) if with_y else None
    o = torch.full((total, hv, V), float("nan"), device="cuda")
    lib.kda_step_conv(pool, W, d.slot_table, d.conv_slot, d.x, d.weight, d.a, d.b, o, st, counters,
                      cu_seqlens=d.cu_seqlens, max_t=inp.max_t, accepted=d.accepted, reset=d.reset, a_log=d.a_log,
                      dt_bias=d.dt_bias, bias=d.bias, y=y, h_qk=inp.h_qk, flags=flags)
    return o, y, st


def assert_fused_equals_two_kernels(inp, flags=0):
    d = inp.to("cuda")
    pool_a, W_a = d.pool.clone(), d.window.clone()
    pool_b, W_b = d.pool.clone(), d.window.clone()
    counters = torch.zeros(inp.slot_table.shape[0], inp.h_qk, dtype=torch.int32, device="cuda")
    o_a, y_a, st_a = two_kernels(d, inp, pool_a, W_a, flags)
    o_b, y_b, st_b = fused(d, inp, pool_b, W_b, counters, flags)
    torch.cuda.synchronize()
    assert int(st_a.item()) == 0 and int(st_b.item()) == 0, (int(st_a.item()), int(st_b.item()))
    assert torch.equal(bits(y_a), bits(y_b)), "y differs"
    assert torch.equal(bits(W_a), bits(W_b)), "window differs"
    assert torch.equal(bits(o_a), bits(o_b)), "o differs"
    assert torch.equal(bits(pool_a), bits(pool_b)), "pool differs"
    assert int(counters.abs().sum().item()) == 0, "read counters not back at zero"


# ---------------------------------------------------------------------------
# bit for bit against the two-kernel path
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wdt", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("state_dtype", [torch.float16, torch.float32])
def test_step_conv_verify_shape(state_dtype, wdt):
    """8 requests x 8 tokens (1 accepted + 7 drafts), HV = 12, K = V = 128, a
    kernel-4 window of 10 entries: the one-wave verify shape."""
    inp = workloads.make_step_conv(n=8, num_spec=7, state_dtype=state_dtype, dtype=wdt, seed=61, reset_p=0.25)
    assert_fused_equals_two_kernels(inp)


@pytest.mark.parametrize("state_dtype", [torch.float16, torch.float32])
def test_step_conv_serving_scale(state_dtype):
    """32 requests x 8 tokens: past one wave (the wide shape on an fp16 pool)."""
    inp = workloads.make_step_conv(n=32, num_spec=7, state_dtype=state_dtype, seed=62)
    assert_fused_equals_two_kernels(inp, flags=PDL)


@pytest.mark.parametrize("h_qk", [12, 4, 1])
@pytest.mark.parametrize("state_dtype", [torch.float16, torch.float32])
def test_step_conv_varlen_padding_grouped_gate_scale(state_dtype, h_qk):
    """Requests of 5, 1, 3, 0, 5, 8, 2 and 7 tokens (num_spec 7), padding
    requests, resets, grouped q/k heads and the learned gate scale."""
    inp = workloads.make_step_conv(n=8, num_spec=7, t_lens=[5, 1, 3, 0, 5, 8, 2, 7], h_qk=h_qk,
                                   state_dtype=state_dtype, seed=63 + h_qk, reset_p=0.3, pad_p=0.25, gate_scale=True)
    assert_fused_equals_two_kernels(inp)


@pytest.mark.parametrize("kw,num_spec", [(1, 4), (2, 4), (3, 2), (4, 1), (4, 4)])
@pytest.mark.parametrize("state_dtype", [torch.float16, torch.float32])
def test_step_conv_kernel_widths(state_dtype, kw, num_spec):
    inp = workloads.make_step_conv(n=8, num_spec=num_spec, kw=kw, state_dtype=state_dtype, seed=70 + 8 * kw + num_spec,
                                   reset_p=0.25, bias=kw % 2 == 0)
    assert_fused_equals_two_kernels(inp)


@pytest.mark.parametrize("state_dtype", [torch.float16, torch.float32])
def test_step_conv_bad_window_slot(state_dtype):
    """A window slot outside the pool: KDA_ERR_SLOT_RANGE, that request's state
    slots and every window untouched, the counters zero."""
    inp = workloads.make_step_conv(n=6, num_spec=3, h_qk=4, state_dtype=state_dtype, seed=75, num_wslots=16)
    inp.conv_slot[2] = 16
    d = inp.to("cuda")
    pool, W = d.pool.clone(), d.window.clone()
    c = torch.zeros(6, 4, dtype=torch.int32, device="cuda")
    o, y, st = fused(d, inp, pool, W, c)
    torch.cuda.synchronize()
    assert int(st.item()) == kda.KDA_ERR_SLOT_RANGE
    assert int(c.abs().sum().item()) == 0
    for s in inp.slot_table[2].tolist():
        assert torch.equal(bits(pool[s]), bits(d.pool[s]))
    bad_win = [int(inp.conv_slot[r]) for r in range(6) if r != 2]
    untouched = [s for s in range(16) if s not in bad_win]
    assert torch.equal(bits(W[untouched]), bits(d.window[untouched]))


# ---------------------------------------------------------------------------
# against the fp64 oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wdt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("state_dtype", [torch.float16, torch.float32])
def test_step_conv_against_oracle(state_dtype, wdt):
    """n = 5 requests of 4, 1, 3, 0 and 4 tokens, HV = 4 on 2 q/k heads,
    K = V = 32, kernel 4, num_spec 3, resets, padding and the gate scale: the
    oracle's conv_step gives the window (exact) and y (the conv bar); its step,
    fed the kernel's own q/k/v, gives the pool and o (the decode bars)."""
    inp = workloads.make_step_conv(n=5, num_spec=3, t_lens=[4, 1, 3, 0, 4], h_qk=2, hv=4, k=32, v=32, num_slots=40,
                                   num_wslots=9, state_dtype=state_dtype, dtype=wdt, seed=80, reset_p=0.4,
                                   pad_p=0.2, gate_scale=True)
    d = inp.to("cuda")
    pool, W = d.pool.clone(), d.window.clone()
    c = torch.zeros(5, 2, dtype=torch.int32, device="cuda")
    o, y, st = fused(d, inp, pool, W, c)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Wref, name = storage(inp.window)
    xs, _ = storage(inp.x)
    yref = oracle.conv_step(Wref, name, inp.conv_slot.numpy(), xs, inp.weight, inp.bias,
                            cu_seqlens=inp.cu_seqlens.numpy(), accepted=inp.accepted.numpy(),
                            reset=None if inp.reset is None else inp.reset.numpy(), silu=True)
    gW, _ = storage(W.cpu())
    assert np.array_equal(gW, Wref), "window differs from the oracle's"
    gy, _ = storage(y.cpu())
    if wdt == torch.float32:
        assert np.abs(gy.astype(np.float64) - yref.astype(np.float64)).max() <= 1e-5
    else:
        assert_y16_match(gy, yref, wdt)
    q, k, v = split_y(y.cpu(), inp)
    ref = pool_np(inp.pool)
    o_ref = oracle.step(ref, inp.slot_table.numpy(), q.double().numpy(), k.double().numpy(), v.double().numpy(),
                        inp.a.numpy(), inp.b.numpy(), cu_seqlens=inp.cu_seqlens.numpy(),
                        accepted=inp.accepted.numpy(), reset=None if inp.reset is None else inp.reset.numpy(),
                        a_log=inp.a_log.numpy(), dt_bias=inp.dt_bias.numpy())
    touched = [s for s in inp.slot_table.numpy().ravel() if s >= 0]
    assert_pool_match(pool.cpu(), ref, touched, "pool")
    assert_out_match(o.cpu(), o_ref, state_dtype, "o")
