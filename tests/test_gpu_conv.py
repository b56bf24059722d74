"""GPU parity of the short convolution with its paged window (kda_conv_step)
against the fp64 oracle.

y: fp32 within max-abs 1e-5; fp16 / bf16 within one step of the oracle's
value rounded once from fp64 (the GPU rounds from its fp32 sum).  The window
holds copies of inputs and old entries, so it must match bit for bit, and
windows of slots no request uses must not change.
"""
import numpy as np
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import workloads

import oracle
from _harness import CONV_Y_ABS, lib_for

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]

DT = [torch.float32, torch.float16, torch.bfloat16]


def storage(t):
    name = str(t.dtype).split(".")[1]
    if t.dtype == torch.float32:
        return t.numpy().copy(), name
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy(), name


def offset_copy(t):
    """The same values in a buffer whose base is one element past a 4-element boundary."""
    buf = torch.empty(t.numel() + 4, dtype=t.dtype, device=t.device)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def gpu_conv(inp, silu=True, flags=0, offset=False, offset_wb=False):
    d = inp.to("cuda")
    y = torch.full_like(d.x, float("nan"))
    if offset:  # rules out 4-channel accesses
        d.window, d.x, y = offset_copy(d.window), offset_copy(d.x), offset_copy(y)
    if offset_wb:  # rules out 16-byte weight rows and bias vectors
        d.weight, d.bias = offset_copy(d.weight), offset_copy(d.bias)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib_for(torch.float32).kda_conv_step(d.window, d.conv_slot, d.x, d.weight, y, status, bias=d.bias,
                                         cu_seqlens=d.cu_seqlens, max_t=inp.max_t, accepted=d.accepted,
                                         reset=d.reset, silu=silu, flags=flags)
    torch.cuda.synchronize()
    return d.window.cpu(), y.cpu(), int(status.item())


def oracle_conv(inp, silu=True):
    W, name = storage(inp.window)
    x, _ = storage(inp.x)
    y = oracle.conv_step(W, name, inp.conv_slot.numpy(), x, inp.weight, inp.bias,
                         cu_seqlens=None if inp.cu_seqlens is None else inp.cu_seqlens.numpy(),
                         accepted=None if inp.accepted is None else inp.accepted.numpy(),
                         reset=None if inp.reset is None else inp.reset.numpy(), silu=silu)
    return W, y


def compare(inp, silu=True, flags=0, offset=False, offset_wb=False, scale=1.0):
    """scale: the inputs' magnitude against the generator's unit scale; the
    fp32 sum's error grows with it, so both absolute bars are multiplied by it."""
    gw, gy, st = gpu_conv(inp, silu, flags, offset, offset_wb)
    rw, ry = oracle_conv(inp, silu)
    assert st == 0, lib_for(torch.float32).kda_strerror(st)
    gws, _ = storage(gw)
    assert np.array_equal(gws, rw), "window differs"
    gys, _ = storage(gy)
    if inp.x.dtype == torch.float32:
        assert np.isfinite(gys).all()
        assert np.abs(gys.astype(np.float64) - ry.astype(np.float64)).max() <= 1e-5 * scale
    else:
        assert_y16_match(gys, ry, inp.x.dtype, CONV_Y_ABS * scale)


def y16_values(bits, dtype):
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(dtype).double().numpy()


def assert_y16_match(gys, ry, dtype, abs_floor=CONV_Y_ABS):
    """fp16 / bf16 y: within one step of the oracle's value, or within
    CONV_Y_ABS of it (the fp32 sum's error, which is many steps near zero)."""
    steps = np.abs(gys.astype(np.int32) - ry.astype(np.int32))
    diff = np.abs(y16_values(gys, dtype) - y16_values(ry, dtype))
    bad = (steps > 1) & (diff > abs_floor)
    assert not bad.any(), f"y off by {steps[bad].max()} steps, {diff[bad].max():.3e} absolute"


EARLY = kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE


@pytest.mark.parametrize("flags", [0, EARLY])
@pytest.mark.parametrize("dtype", DT)
def test_conv_layer_shape(dtype, flags):
    """8 requests x 5 tokens (4 drafts), 4608 channels (q, k and v of one layer),
    kernel 4, window 7, accepted index per request, resets and padding."""
    compare(workloads.make_conv(n=8, t=5, dtype=dtype, seed=60, reset_p=0.25, pad_p=0.2), flags=flags)


@pytest.mark.parametrize("flags", [0, EARLY])
@pytest.mark.parametrize("dtype", DT)
def test_conv_variable_lengths(dtype, flags):
    inp = workloads.make_conv(n=5, t_lens=[5, 0, 3, 5, 1], channels=300, dtype=dtype, seed=61)
    inp.accepted[:] = 5  # the whole window is history: every token count is valid
    compare(inp, flags=flags)


def test_conv_early_reads_back_to_back():
    """Six launches in a row on one stream, each on its own window pool, with
    programmatic dependent launch and early reads (each reads its window
    while the previous one still runs): every one matches the oracle."""
    sets = [workloads.make_conv(n=16, t=5, dtype=torch.bfloat16, seed=80 + i, reset_p=0.25, pad_p=0.1)
            for i in range(6)]
    devs = [s.to("cuda") for s in sets]
    ys = [torch.full_like(d.x, float("nan")) for d in devs]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = lib_for(torch.float32)
    for d, y, s in zip(devs, ys, sets):
        lib.kda_conv_step(d.window, d.conv_slot, d.x, d.weight, y, status, bias=d.bias, cu_seqlens=d.cu_seqlens,
                          max_t=s.max_t, accepted=d.accepted, reset=d.reset, flags=EARLY)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for d, y, s in zip(devs, ys, sets):
        rw, ry = oracle_conv(s)
        assert np.array_equal(storage(d.window.cpu())[0], rw)
        assert_y16_match(storage(y.cpu())[0], ry, torch.bfloat16)


@pytest.mark.parametrize("dtype", DT)
def test_conv_one_channel_per_thread_path(dtype):
    """Shapes and addresses that rule out 4-channel accesses -- 301 channels,
    and a window, input and output one element past a 4-element boundary --
    take the one-channel path, with the same results."""
    compare(workloads.make_conv(n=5, t=5, channels=301, dtype=dtype, seed=65, reset_p=0.2))
    compare(workloads.make_conv(n=4, t=5, channels=256, dtype=dtype, seed=66, reset_p=0.2), offset=True)


@pytest.mark.parametrize("channels", [4608, 301])
@pytest.mark.parametrize("flags", [0, EARLY])
@pytest.mark.parametrize("dtype", DT)
def test_conv_long_requests_and_window(dtype, flags, channels):
    """Requests of 13, 20, 9 and 1 tokens on a 22-entry window (19 drafts):
    the inputs and the kept old entries run past one batch of 8 registers, so
    the history carries from batch to batch, the kept entries (9 to 21 of
    them) move in the loop, and the last inputs are read again for the window;
    4-channel and 1-channel paths."""
    inp = workloads.make_conv(n=4, t_lens=[13, 20, 9, 1], channels=channels, num_spec=19, dtype=dtype,
                              seed=69, reset_p=0.25)
    inp.accepted[:] = 20  # the whole window is history: every token count is valid
    compare(inp, flags=flags)


@pytest.mark.parametrize("flags", [0, EARLY])
@pytest.mark.parametrize("dtype", DT)
def test_conv_unaligned_weights_and_bias(dtype, flags):
    """Weights and bias one element past a 16-byte boundary, everything else
    aligned: the 4-channel, kernel-width-4 path reads them element by element,
    with the same results."""
    compare(workloads.make_conv(n=6, t=5, dtype=dtype, seed=67, reset_p=0.2), flags=flags, offset_wb=True)


@pytest.mark.parametrize("dtype", DT)
def test_conv_silu_saturates(dtype):
    """Inputs and window scaled by 64 (exact in every dtype here) put the
    pre-activations at hundreds in both directions: SiLU's limits, y = s for
    large s and y = -0 or a vanishing negative for very negative s.  Every
    term of the fp32 sum is 64 times larger, so its error is, and the
    absolute bars are scaled to match (one fp32 ulp at 256 is already 3e-5)."""
    inp = workloads.make_conv(n=6, t=5, dtype=dtype, seed=68, reset_p=0.2)
    inp.x = inp.x * 64
    inp.window = inp.window * 64
    compare(inp, scale=64.0)


@pytest.mark.parametrize("kw", [1, 2, 3, 4, 8])
def test_conv_kernel_widths_and_no_activation(kw):
    inp = workloads.make_conv(n=4, t=3, channels=200, kw=kw, num_spec=2, dtype=torch.float32, seed=62 + kw)
    compare(inp, silu=(kw % 2 == 0))


def test_conv_decode_rolling_window_chain():
    """Plain decode (qlen 1, window kernel - 1) over 6 calls equals conv1d over
    the 6 tokens from a zero start."""
    n, C, kw = 3, 64, 4
    g = torch.Generator().manual_seed(63)
    W = torch.zeros(4, kw - 1, C, device="cuda")
    w = torch.randn(C, kw, generator=g)
    xs = torch.randn(6, n, C, generator=g)
    slots = torch.tensor([2, 0, 3], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = lib_for(torch.float32)
    ys = []
    for t in range(6):
        y = torch.empty(n, C, device="cuda")
        lib.kda_conv_step(W, slots, xs[t].cuda(), w.cuda(), y, status, silu=False)
        ys.append(y.cpu())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = torch.nn.functional.conv1d(torch.nn.functional.pad(xs.permute(1, 2, 0).double(), (kw - 1, 0)),
                                     w.double()[:, None, :], groups=C).permute(2, 0, 1)
    assert (torch.stack(ys).double() - ref).abs().max() <= 1e-5


def test_conv_bad_accepted_index_sets_status():
    inp = workloads.make_conv(n=3, t=5, channels=64, dtype=torch.float32, seed=64)
    inp.accepted[1] = 6  # history would run past the 7-entry window
    gw, gy, st = gpu_conv(inp)
    assert st == kda.KDA_ERR_ARG
    s = int(inp.conv_slot[1])
    assert torch.equal(gw[s], inp.window[s])  # that request was skipped
