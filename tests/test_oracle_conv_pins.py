"""Pins of the oracle's short convolution and bfloat16 rounding (no GPU).

The convolution in front of the recurrence keeps a paged window of the last
kernel - 1 + num_spec inputs per request; a step reads its kernel - 1 history
entries at the accepted index and writes back the kept old entries followed by
its inputs (ROCm/ATOM pull request 2894, review thread on the conv window).
The pins: bfloat16 rounding against torch's fp32 -> bf16 conversion (a direct
RNE from fp32); the convolution against torch.nn.functional.conv1d (a library
routine) with a zero history; and the window rule by chaining steps, which
must equal one longer step, and by rejecting drafts, which must equal never
having taken them.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from kda_linear_attention_gated_gb300 import workloads

pytestmark = pytest.mark.usefixtures("oracle_mod")


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def storage(t):
    """float32 array, or uint16 bits for fp16 / bf16, plus the dtype name."""
    name = str(t.dtype).split(".")[1]
    return (t.numpy().copy() if t.dtype == torch.float32 else bits(t)), name


def as_tensor(a, name):
    if name == "float32":
        return torch.from_numpy(np.asarray(a, np.float32))
    return torch.from_numpy(np.asarray(a, np.uint16).view(np.int16)).view(getattr(torch, name))


def test_bf16_rounding_matches_torch_from_fp32():
    rng = np.random.default_rng(0)
    raw = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = raw.view(np.float32)
    f = f[np.isfinite(f)]
    # exact midpoints between neighbouring bf16 values and their fp32 neighbours
    hi = (rng.integers(0, 2**16, size=20000, dtype=np.uint64).astype(np.uint32) << 16)
    mids = (hi | 0x8000).view(np.float32)
    mids = mids[np.isfinite(mids)]
    cand = np.concatenate([f, mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf)),
                           np.array([0.0, -0.0, 1e-40, -1e-40, 3.3895314e38, 3.39e38], np.float32)])
    got = oracle.f64_to_bf16_rne(cand.astype(np.float64))
    ref = bits(torch.from_numpy(cand).to(torch.bfloat16))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("kw", [1, 2, 4])
def test_conv_matches_conv1d_from_zero_history(kw):
    """Reset requests start from a zero history: y = silu(conv1d(left-padded x) + b)."""
    inp = workloads.make_conv(n=3, t=5, channels=40, kw=kw, num_spec=4, num_slots=5, dtype=torch.float32,
                              seed=kw, reset_p=1.0)
    W, name = storage(inp.window)
    y = oracle.conv_step(W, name, inp.conv_slot, inp.x.numpy(), inp.weight, inp.bias, accepted=inp.accepted,
                         reset=inp.reset)
    x = inp.x.double().reshape(3, 5, 40).permute(0, 2, 1)             # [N, C, T]
    ref = F.conv1d(F.pad(x, (kw - 1, 0)), inp.weight.double()[:, None, :], inp.bias.double(), groups=40)
    ref = F.silu(ref).permute(0, 2, 1).reshape(15, 40).float().numpy()
    np.testing.assert_array_max_ulp(y, ref, maxulp=1)


def run(inp, window, **kw):
    W, name = storage(window)
    x, _ = storage(inp.x) if "x" not in kw else kw.pop("x")
    y = oracle.conv_step(W, name, inp.conv_slot, x, inp.weight, inp.bias, **kw)
    return W, y, name


def test_chained_steps_equal_one_long_step():
    """Two steps, every draft of the first accepted, equal one step over both token runs."""
    kw, spec = 4, 4
    L = kw - 1 + spec
    inp = workloads.make_conv(n=2, t=10, channels=24, kw=kw, num_spec=spec, num_slots=4, dtype=torch.float32,
                              seed=7, accepted=False)
    x = inp.x.reshape(2, 10, 24)
    acc0 = torch.tensor([3, 5], dtype=torch.int32)  # the previous step's accepted counts
    # one step of 10 tokens needs a window of at least 10 + kw - 2 entries: use the long form
    W0, name = storage(inp.window)
    # split: 5 + 5 tokens
    first = workloads.ConvInputs(inp.window, inp.conv_slot, x[:, :5].reshape(10, 24), inp.weight, inp.bias)
    Wa, y1, _ = run(first, inp.window, accepted=acc0)
    second = workloads.ConvInputs(as_tensor(Wa, name), inp.conv_slot, x[:, 5:].reshape(10, 24), inp.weight,
                                  inp.bias)
    Wb, y2, _ = run(second, as_tensor(Wa, name), accepted=torch.full((2,), 5, dtype=torch.int32))
    # reference: a window of L' = 10 + kw - 2 holding the same history at the same accepted index
    Lp = 10 + kw - 2
    big = np.zeros((4, Lp, 24), np.float32)
    big[:, :L] = W0
    longer = workloads.ConvInputs(torch.from_numpy(big), inp.conv_slot, x.reshape(20, 24), inp.weight, inp.bias)
    Wl, yl, _ = run(longer, torch.from_numpy(big), accepted=acc0)
    yl = yl.reshape(2, 10, 24)
    assert np.array_equal(np.concatenate([y1.reshape(2, 5, 24), y2.reshape(2, 5, 24)], 1), yl)
    # both windows end with the same last L inputs
    for s in inp.conv_slot.tolist():
        assert np.array_equal(Wb[s], Wl[s][Lp - L:])


def test_rejected_drafts_are_as_if_never_taken():
    """A step of qlen tokens of which a are accepted, then a step from accepted
    index a - 1, gives what taking only the a tokens gives (history = the last
    kw - 1 entries of the window)."""
    kw, spec = 4, 4
    L = kw - 1 + spec
    qlen = spec + 1
    inp = workloads.make_conv(n=3, t=qlen, channels=16, kw=kw, num_spec=spec, num_slots=6, dtype=torch.float32,
                              seed=8, accepted=True)
    inp.accepted[:] = qlen  # the whole window is valid history at the first step
    g = torch.Generator().manual_seed(80)
    x2 = torch.randn((3 * qlen, 16), generator=g)
    a = torch.tensor([1, 3, 5], dtype=torch.int32)
    # path A: all qlen tokens, then continue from accepted index a - 1
    Wa, _, name = run(inp, inp.window, accepted=inp.accepted)
    nxt = workloads.ConvInputs(as_tensor(Wa, name), inp.conv_slot, x2, inp.weight, inp.bias)
    _, ya, _ = run(nxt, as_tensor(Wa, name), accepted=a)
    # path B: per request, only its a accepted tokens, then continue from the window's end
    x1 = inp.x.reshape(3, qlen, 16)
    Wb, name = storage(inp.window)
    yb = []
    for r in range(3):
        one = workloads.ConvInputs(as_tensor(Wb, name), inp.conv_slot[r:r + 1], x1[r, :int(a[r])].contiguous(),
                                   inp.weight, inp.bias)
        Wb, _, _ = run(one, as_tensor(Wb, name), accepted=inp.accepted[r:r + 1])
        nxt_r = workloads.ConvInputs(as_tensor(Wb, name), inp.conv_slot[r:r + 1],
                                     x2.reshape(3, qlen, 16)[r].contiguous(), inp.weight, inp.bias)
        Wc = Wb.copy()
        _, y_r, _ = run(nxt_r, as_tensor(Wc, name), accepted=torch.tensor([L - kw + 2], dtype=torch.int32))
        yb.append(y_r)
    np.testing.assert_array_equal(ya.reshape(3, qlen, 16), np.stack(yb))


def test_pointwise_kernel_closed_form():
    inp = workloads.make_conv(n=2, t=3, channels=8, kw=1, num_spec=2, num_slots=3, dtype=torch.float32, seed=9)
    _, y, _ = run(inp, inp.window, accepted=inp.accepted)
    s = inp.x.double() * inp.weight.double()[:, 0] + inp.bias.double()
    np.testing.assert_array_max_ulp(y, (s / (1 + torch.exp(-s))).float().numpy(), maxulp=1)


def test_padding_and_reset():
    inp = workloads.make_conv(n=4, t=5, channels=8, kw=4, num_spec=4, num_slots=6, dtype=torch.bfloat16,
                              seed=14, pad_p=0.5, reset_p=0.5)
    pad = inp.conv_slot < 0
    assert pad.any() and not pad.all()
    W0, name = storage(inp.window)
    W, y, _ = run(inp, inp.window, accepted=inp.accepted, reset=inp.reset)
    y = y.reshape(4, 5, 8)
    assert (y[pad.numpy()] == 0).all()
    used = inp.conv_slot[~pad].long().numpy()
    unused = np.setdiff1d(np.arange(6), used)
    assert np.array_equal(W[unused], W0[unused])
    # a reset request's first output only sees its first input
    for r in np.nonzero((~pad & (inp.reset > 0)).numpy())[0]:
        s = inp.x[r * 5].double() * inp.weight.double()[:, 3] + inp.bias.double()
        ref = bits((s / (1 + torch.exp(-s))).to(torch.float32).to(torch.bfloat16))
        got = y[r, 0]
        # one rounding (oracle, from fp64) against fp64 -> fp32 -> bf16: at most one bf16 step apart
        assert np.abs(got.astype(np.int32) - ref.astype(np.int32)).max() <= 1


def test_window_layout_errors():
    inp = workloads.make_conv(n=1, t=5, channels=4, kw=4, num_spec=4, num_slots=2, dtype=torch.float32, seed=11)
    W, name = storage(inp.window)
    with pytest.raises(ValueError):   # history past the window: accepted index 5 of a 7-entry window
        oracle.conv_step(W, name, inp.conv_slot, inp.x.numpy(), inp.weight, inp.bias,
                         accepted=np.array([6], np.int32))


@pytest.mark.parametrize("seed,lens,kw,spec", [(90, [5, 1, 3, 0, 5, 8, 2, 7], 4, 7), (91, [1, 1, 4], 3, 3),
                                               (92, None, 2, 4), (93, [2, 0, 5], 4, 4)])
def test_fused_step_inputs_obey_the_window_rule(seed, lens, kw, spec):
    """The speculative fused-step inputs (make_step_conv) draw each request's
    accepted index among the values its length admits: the kept old entries,
    max(0, L - T_r), lie below acc + kw - 1.  The oracle's conv_step checks
    that rule (it raises on a violation) and leaves padding requests' windows
    alone, so it runs cleanly over the generated step and moves only the
    windows of requests with tokens."""
    inp = workloads.make_step_conv(n=len(lens) if lens else 6, num_spec=spec, t_lens=lens, kw=kw, h_qk=2, hv=4,
                                   k=16, v=16, num_slots=80, num_wslots=12, seed=seed, pad_p=0.3)
    L = kw - 1 + spec
    t = [inp.max_t] * inp.slot_table.shape[0] if lens is None else lens
    for r, tr in enumerate(t):
        acc = int(inp.accepted[r]) - 1
        assert 0 <= acc <= spec and max(0, L - tr) <= acc + kw - 1
        pad = bool((inp.slot_table[r] < 0).all())
        assert pad == (int(inp.conv_slot[r]) < 0)
    W, name = storage(inp.window)
    before = W.copy()
    xs, _ = storage(inp.x)
    oracle.conv_step(W, name, inp.conv_slot.numpy(), xs, inp.weight, inp.bias,
                     cu_seqlens=None if inp.cu_seqlens is None else inp.cu_seqlens.numpy(),
                     accepted=inp.accepted.numpy(), silu=True)
    moved = {int(inp.conv_slot[r]) for r, tr in enumerate(t) if tr > 0 and int(inp.conv_slot[r]) >= 0}
    for s in range(W.shape[0]):
        if s not in moved:
            assert np.array_equal(W[s], before[s]), f"window {s} changed"
