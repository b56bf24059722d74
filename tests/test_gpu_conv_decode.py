"""GPU parity of the decode step with the short convolution fused in front
(kda_decode_conv_step).

Bit for bit against the two-kernel path on the same inputs: kda_conv_step with
one token a request, then kda_decode_step (kda_step in place for grouped q/k
heads) with q, k and v taken from the conv's y.  Pool, window, y and o must be
identical, and the read counters must be back at zero after every call.  Then
against the fp64 oracle: the conv's y and window against the oracle's
conv_step (the conv bar: one 16-bit step, windows exact), and the recurrence
against the oracle's step fed the same q/k/v values (the decode bars).
"""
import numpy as np
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import workloads

import oracle
from _harness import assert_out_match, assert_pool_match, lib_for, pool_np
from test_gpu_conv import assert_y16_match, storage

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]

PDL, EARLY = kda.KDA_LAUNCH_PDL, kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE


def split_y(y, inp):
    """q [n, h_qk, K], k [n, h_qk, K], v [n, HV, V] from the conv's outputs (q | k | v channels)."""
    n, hv, K, V = inp.x.shape[0], inp.pool.shape[1], inp.pool.shape[2], inp.pool.shape[3]
    h = inp.h_qk
    q = y[:, : h * K].reshape(n, h, K).contiguous()
    k = y[:, h * K: 2 * h * K].reshape(n, h, K).contiguous()
    v = y[:, 2 * h * K:].reshape(n, hv, V).contiguous()
    return q, k, v


def two_kernels(d, inp, pool, W, silu=True, flags=0):
    """kda_conv_step then the decode on device copies pool and W; returns o, y, status."""
    lib = lib_for(inp.pool.dtype)
    n, hv, V = inp.x.shape[0], inp.pool.shape[1], inp.pool.shape[3]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full_like(d.x, float("nan"))
    lib.kda_conv_step(W, d.conv_slot, d.x, d.weight, y, st, bias=d.bias, max_t=1, reset=d.reset, silu=silu,
                      flags=flags)
    q, k, v = split_y(y, inp)
    o = torch.full((n, hv, V), float("nan"), device="cuda")
    if inp.h_qk == hv and d.a_log is None:
        lib.kda_decode_step(pool, d.slot_ids, q, k, v, d.a, d.b, o, st, reset=d.reset, flags=flags)
    else:
        lib.kda_step(pool, d.slot_ids.view(n, 1).contiguous(), q, k, v, d.a, d.b, o, st, reset=d.reset,
                     a_log=d.a_log, dt_bias=d.dt_bias, in_place=True, flags=flags)
    return o, y, st


def fused(d, inp, pool, W, counters, silu=True, flags=0, with_y=True):
    lib = lib_for(inp.pool.dtype)
    n, hv, V = inp.x.shape[0], inp.pool.shape[1], inp.pool.shape[3]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full_like(d.x, float("nan")) if with_y else None
    o = torch.full((n, hv, V), float("nan"), device="cuda")
    lib.kda_decode_conv_step(pool, W, d.slot_ids, d.conv_slot, d.x, d.weight, d.a, d.b, o, st, counters,
                             bias=d.bias, y=y, reset=d.reset, h_qk=inp.h_qk, silu=silu, a_log=d.a_log,
                             dt_bias=d.dt_bias, flags=flags)
    return o, y, st


def bits(t):
    t = t.cpu()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def assert_fused_equals_two_kernels(inp, silu=True, flags=0, steps=1):
    """steps > 1: a rolling chain on the same pool and window (new inputs each step)."""
    d = inp.to("cuda")
    pool_a, W_a = d.pool.clone(), d.window.clone()
    pool_b, W_b = d.pool.clone(), d.window.clone()
    counters = torch.zeros(inp.x.shape[0], inp.h_qk, dtype=torch.int32, device="cuda")
    g = torch.Generator().manual_seed(123)
    for s in range(steps):
        if s > 0:  # the next token's inputs
            d.x = torch.randn(inp.x.shape, generator=g).to(inp.x.dtype).cuda()
            d.a = torch.randn(inp.a.shape, generator=g).cuda()
            d.b = torch.randn(inp.b.shape, generator=g).cuda()
            d.reset = None
        o_a, y_a, st_a = two_kernels(d, inp, pool_a, W_a, silu, flags)
        o_b, y_b, st_b = fused(d, inp, pool_b, W_b, counters, silu, flags)
        torch.cuda.synchronize()
        assert int(st_a.item()) == 0 and int(st_b.item()) == 0, (int(st_a.item()), int(st_b.item()))
        assert torch.equal(bits(y_a), bits(y_b)), f"step {s}: y differs"
        assert torch.equal(bits(W_a), bits(W_b)), f"step {s}: window differs"
        assert torch.equal(bits(o_a), bits(o_b)), f"step {s}: o differs"
        assert torch.equal(bits(pool_a), bits(pool_b)), f"step {s}: pool differs"
        assert int(counters.abs().sum().item()) == 0, "read counters not back at zero"


# ---------------------------------------------------------------------------
# bit for bit against the two-kernel path
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wdt", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_layer_shape_equals_conv_then_decode(state_dtype, wdt):
    """N = 64, HV = 12, K = V = 128, kernel 4, a 3-entry window, resets: the
    fp16 launch has one CTA per head (no shared q/k window), the fp32 one two
    (two 32-column tiles each; the read counters decide the writer)."""
    inp = workloads.make_decode_conv(n=64, state_dtype=state_dtype, dtype=wdt, seed=11, reset_p=0.1)
    assert_fused_equals_two_kernels(inp)


@pytest.mark.parametrize("n,h_qk", [(64, 4), (64, 1), (5, 12), (5, 3)])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_grouped_heads_and_small_launches(state_dtype, n, h_qk):
    """Grouped q/k heads (up to 12 value heads x 2 CTAs, or x 4 and x 8 one-tile
    CTAs within one wave, reading one q/k window) and launches within one wave."""
    inp = workloads.make_decode_conv(n=n, h_qk=h_qk, state_dtype=state_dtype, seed=12 + h_qk, reset_p=0.2)
    assert_fused_equals_two_kernels(inp)


@pytest.mark.parametrize("kw,L", [(1, 1), (2, 1), (2, 2), (3, 2), (3, 3), (4, 4)])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_kernel_widths_and_window_lengths(state_dtype, kw, L):
    """Every width 1 .. 4 with both window lengths a one-token step allows
    (kernel - 1: each entry moves down one; kernel: entries stay), with and
    without SiLU and bias."""
    inp = workloads.make_decode_conv(n=16, kw=kw, L=L, state_dtype=state_dtype, seed=20 + 4 * kw + L,
                                     reset_p=0.25, bias=kw % 2 == 0)
    assert_fused_equals_two_kernels(inp, silu=kw != 3)


@pytest.mark.parametrize("K,V", [(64, 80), (128, 48), (32, 128)])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_ragged_key_and_value_sizes(state_dtype, K, V):
    """K below 128 (the per-row bound checks) and V not a multiple of the
    tile (a partial second fp16 tile at V = 80, none at V = 48)."""
    inp = workloads.make_decode_conv(n=64, hv=6, h_qk=3, k=K, v=V, state_dtype=state_dtype, seed=30 + K + V)
    assert_fused_equals_two_kernels(inp)


@pytest.mark.parametrize("h_qk", [12, 4])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_learned_gate_scale(state_dtype, h_qk):
    """The layer's learned gate scale and bias (a_log, dt_bias): against the
    conv step then the in-place kda_step with the same gate arguments, over
    a 2-step chain."""
    inp = workloads.make_decode_conv(n=64, h_qk=h_qk, state_dtype=state_dtype, seed=45 + h_qk, reset_p=0.1,
                                     gate_scale=True)
    assert_fused_equals_two_kernels(inp, steps=2)


@pytest.mark.parametrize("flags", [0, PDL])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_rolling_chain(state_dtype, flags):
    """Three steps in a row on the same pool and window: each step's window
    is the next one's history, and the counters start each call at zero."""
    inp = workloads.make_decode_conv(n=24, h_qk=4, state_dtype=state_dtype, seed=40)
    assert_fused_equals_two_kernels(inp, flags=flags, steps=3)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_early_state_reads_after_another_layer(state_dtype):
    """KDA_LAUNCH_PDL_EARLY_STATE behind a step on another layer's pool and
    window (so nothing it reads early is written by the kernel before it)."""
    l0 = workloads.make_decode_conv(n=32, state_dtype=state_dtype, seed=41)
    l1 = workloads.make_decode_conv(n=32, state_dtype=state_dtype, seed=42)
    d0, d1 = l0.to("cuda"), l1.to("cuda")
    c = torch.zeros(32, 12, dtype=torch.int32, device="cuda")
    ref0, ref1 = (d0.pool.clone(), d0.window.clone()), (d1.pool.clone(), d1.window.clone())
    o0r, _, s0 = two_kernels(d0, l0, *ref0)
    o1r, _, s1 = two_kernels(d1, l1, *ref1)
    got0, got1 = (d0.pool.clone(), d0.window.clone()), (d1.pool.clone(), d1.window.clone())
    o0, _, t0 = fused(d0, l0, *got0, c, flags=PDL)
    o1, _, t1 = fused(d1, l1, *got1, c, flags=EARLY)
    torch.cuda.synchronize()
    assert [int(s.item()) for s in (s0, s1, t0, t1)] == [0, 0, 0, 0]
    for a, b in ((o0r, o0), (o1r, o1), (ref0[0], got0[0]), (ref0[1], got0[1]), (ref1[0], got1[0]),
                 (ref1[1], got1[1])):
        assert torch.equal(bits(a), bits(b))
    assert int(c.abs().sum().item()) == 0


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_without_y_output(state_dtype):
    inp = workloads.make_decode_conv(n=8, h_qk=4, state_dtype=state_dtype, seed=43)
    d = inp.to("cuda")
    pa, Wa, pb, Wb = d.pool.clone(), d.window.clone(), d.pool.clone(), d.window.clone()
    c = torch.zeros(8, 4, dtype=torch.int32, device="cuda")
    oa, _, sa = fused(d, inp, pa, Wa, c)
    ob, _, sb = fused(d, inp, pb, Wb, c, with_y=False)
    torch.cuda.synchronize()
    assert int(sa.item()) == 0 and int(sb.item()) == 0
    assert torch.equal(bits(oa), bits(ob)) and torch.equal(bits(pa), bits(pb)) and torch.equal(bits(Wa), bits(Wb))


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_bad_window_slot_skips_the_request(state_dtype):
    """A window slot outside the pool: KDA_ERR_SLOT_RANGE, that request's state
    and every window left alone, its counters untouched (zero); the other
    requests as on the two-kernel path."""
    inp = workloads.make_decode_conv(n=6, h_qk=3, state_dtype=state_dtype, seed=44, num_wslots=16)
    bad = 2
    inp.conv_slot[bad] = 16
    d = inp.to("cuda")
    pool, W = d.pool.clone(), d.window.clone()
    c = torch.zeros(6, 3, dtype=torch.int32, device="cuda")
    o, y, st = fused(d, inp, pool, W, c)
    torch.cuda.synchronize()
    assert int(st.item()) == kda.KDA_ERR_SLOT_RANGE
    assert int(c.abs().sum().item()) == 0
    s = int(inp.slot_ids[bad])
    assert torch.equal(bits(pool[s]), bits(d.pool[s]))
    good = [r for r in range(6) if r != bad]
    sub = workloads.DecodeConvInputs(inp.pool, inp.slot_ids[good], inp.window, inp.conv_slot[good], inp.x[good],
                                     inp.weight, inp.bias, inp.a[good], inp.b[good], None, inp.h_qk)
    ds = sub.to("cuda")
    pr, Wr = d.pool.clone(), d.window.clone()
    o_r, _, st_r = two_kernels(ds, sub, pr, Wr)
    torch.cuda.synchronize()
    assert int(st_r.item()) == 0
    assert torch.equal(bits(pool), bits(pr)) and torch.equal(bits(W), bits(Wr))
    assert torch.equal(bits(o[good]), bits(o_r))


# ---------------------------------------------------------------------------
# against the fp64 oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wdt,gate_scale", [(torch.bfloat16, False), (torch.float32, False), (torch.bfloat16, True)])
@pytest.mark.parametrize("kw,L", [(4, 3), (4, 4)])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_fused_against_oracle(state_dtype, kw, L, wdt, gate_scale):
    """n = 5, HV = 4 value heads on 2 q/k heads, K = V = 32, resets.  The
    oracle's convolution gives the window (exact) and y (the conv bar); its
    recurrence, fed the kernel's own q/k/v values, gives the pool and o
    (the decode bars), so a 16-bit y one step from the oracle's cannot
    masquerade as a recurrence error."""
    inp = workloads.make_decode_conv(n=5, hv=4, h_qk=2, k=32, v=32, kw=kw, L=L, num_slots=12, num_wslots=9,
                                     state_dtype=state_dtype, dtype=wdt, seed=50 + L, reset_p=0.4,
                                     gate_scale=gate_scale)
    d = inp.to("cuda")
    pool, W = d.pool.clone(), d.window.clone()
    c = torch.zeros(5, 2, dtype=torch.int32, device="cuda")
    o, y, st = fused(d, inp, pool, W, c)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the convolution
    Wref, name = storage(inp.window)
    xs, _ = storage(inp.x)
    yref = oracle.conv_step(Wref, name, inp.conv_slot.numpy(), xs, inp.weight, inp.bias,
                            reset=None if inp.reset is None else inp.reset.numpy(), silu=True)
    gW, _ = storage(W.cpu())
    assert np.array_equal(gW, Wref), "window differs from the oracle's"
    gy, _ = storage(y.cpu())
    if wdt == torch.float32:
        assert np.abs(gy.astype(np.float64) - yref.astype(np.float64)).max() <= 1e-5
    else:
        assert_y16_match(gy, yref, wdt)
    # the recurrence on the kernel's q/k/v
    q, k, v = split_y(y.cpu(), inp)
    ref = pool_np(inp.pool)
    o_ref = oracle.step(ref, inp.slot_ids.numpy().reshape(5, 1), q.double().numpy(), k.double().numpy(),
                        v.double().numpy(), inp.a.numpy(), inp.b.numpy(),
                        reset=None if inp.reset is None else inp.reset.numpy(),
                        a_log=None if inp.a_log is None else inp.a_log.numpy(),
                        dt_bias=None if inp.dt_bias is None else inp.dt_bias.numpy(), in_place=True)
    assert_pool_match(pool.cpu(), ref, inp.slot_ids.numpy(), "pool")
    assert_out_match(o.cpu(), o_ref, state_dtype, "o")
