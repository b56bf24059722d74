"""Test harness: run one call through the C ABI on the GPU and the same call
through the CPU oracle, on identical seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300.workloads import StepInputs

FP32_ATOL = 1e-5          # max-abs bound for an fp32 pool (states and outputs)
F16_STATE_ULPS = 1        # stored fp16 states: within 1 ulp of the oracle's RNE value ...
# ... except in the bottom binades, |S| < 2^-13, where one fp16 step is 2^-24
# (6.0e-8): that is below the rounding error of any fp32 carry through terms of
# magnitude up to about 1 (an fp32 ulp there is 2^-23 .. 2^-24), so a second
# step (1.2e-7 in all) is allowed there and nowhere else
F16_LOW_BINADE = 2.0 ** -13
F16_LOW_ULPS = 2
F16_OFF_FRACTION = 1e-3   # and at most this share of the stored elements off by any ulp
F16_OUT_RTOL = 2e-3       # outputs with an fp16 pool: relative
F16_OUT_ATOL = 1e-6       # ... with an absolute floor for outputs near zero
# Short-convolution outputs stored as fp16 / bf16: within one step of the
# oracle's once-rounded value, or within CONV_Y_ABS of it.  The kernel sums the
# KW + 1 terms (bias and KW products) in fp32, an error of up to about
# (KW + 1) 2^-24 sum |terms| (7.7e-7 at most on the layer-shape workloads,
# tests/test_tolerances.py); where the output is near zero (|y| ~ 1e-6, a bf16
# step of 1.5e-8) that is several steps, so a step count alone cannot bound it.
CONV_Y_ABS = 2.0 ** -19

_LIBS: dict = {}


def lib_for(state_dtype) -> kda.KdaLibrary:
    if state_dtype not in _LIBS:
        _LIBS[state_dtype] = kda.KdaLibrary(state_dtype)
    return _LIBS[state_dtype]


def pool_np(pool: torch.Tensor) -> np.ndarray:
    """CPU NumPy view of a pool: float32, or fp16 bit patterns as uint16."""
    p = pool.detach().cpu().contiguous()
    if p.dtype == torch.float16:
        return p.view(torch.int16).numpy().view(np.uint16).copy()
    return p.numpy().copy()


def f16_ulp_distance(x_bits: np.ndarray, y_bits: np.ndarray) -> np.ndarray:
    """Distance in representable steps between fp16 bit patterns (sign-magnitude -> ordered)."""
    def ordered(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(ordered(x_bits) - ordered(y_bits))


def gpu_decode(inp: StepInputs, state_dtype=None, stream=None):
    """Returns (pool after, o, status) as CPU tensors / int."""
    d = inp.to("cuda")
    lib = lib_for(state_dtype or inp.pool.dtype)
    n, hv, v = d.v.shape
    o = torch.full((n, hv, v), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_decode_step(d.pool, d.init_slot, d.q, d.k, d.v, d.a, d.b, o, status,
                        reset=d.reset, stream=stream)
    torch.cuda.synchronize()
    return d.pool.cpu(), o.cpu(), int(status.item())


def gpu_verify(inp: StepInputs, state_dtype=None):
    d = inp.to("cuda")
    lib = lib_for(state_dtype or inp.pool.dtype)
    n, t, hv, v = d.v.shape
    o = torch.full((n, t, hv, v), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_spec_verify(d.pool, d.init_slot, d.snap_slot, d.q, d.k, d.v, d.a, d.b, o, status,
                        reset=d.reset)
    torch.cuda.synchronize()
    return d.pool.cpu(), o.cpu(), int(status.item())


def oracle_decode(inp: StepInputs, nthreads=8):
    P = pool_np(inp.pool)
    o = oracle.decode_step(P, inp.init_slot.numpy(), inp.q, inp.k, inp.v, inp.a, inp.b,
                           reset=None if inp.reset is None else inp.reset.numpy(),
                           slot_stride=None, nthreads=nthreads)
    return P, o


def oracle_verify(inp: StepInputs, nthreads=8):
    P = pool_np(inp.pool)
    o = oracle.spec_verify(P, inp.init_slot.numpy(), inp.snap_slot.numpy(), inp.q, inp.k, inp.v,
                           inp.a, inp.b, reset=None if inp.reset is None else inp.reset.numpy(),
                           nthreads=nthreads)
    return P, o


def assert_pool_match(gpu_pool: torch.Tensor, ref: np.ndarray, touched_slots, what=""):
    """Slots not in touched_slots must be bit-identical to ref (which the oracle
    left untouched too); touched slots within the pool dtype's tolerance."""
    g = pool_np(gpu_pool)
    touched = np.zeros(g.shape[0], bool)
    touched[np.asarray(touched_slots, np.int64).ravel()] = True
    assert g[~touched].tobytes() == ref[~touched].tobytes(), f"{what}: untouched slots changed"
    if g.dtype == np.uint16:
        dist = f16_ulp_distance(g[touched], ref[touched])
        low = np.abs(ref[touched].view(np.float16).astype(np.float64)) < F16_LOW_BINADE
        bound = np.where(low, F16_LOW_ULPS, F16_STATE_ULPS)
        worst = int(np.argmax(dist - bound))
        assert (dist <= bound).all(), (
            f"{what}: fp16 state off by {dist.ravel()[worst]} ulp at reference value "
            f"{ref[touched].view(np.float16).ravel()[worst]}")
        off = float((dist > 0).mean())
        assert off <= F16_OFF_FRACTION, f"{what}: {off:.2e} of the fp16 states are off by an ulp"
        return dist
    diff = np.abs(g[touched].astype(np.float64) - ref[touched].astype(np.float64))
    assert np.isfinite(g[touched]).all()
    assert diff.max() <= FP32_ATOL, f"{what}: fp32 state max abs diff {diff.max():.3e}"
    return diff


def assert_out_match(o_gpu: torch.Tensor, o_ref: np.ndarray, state_dtype, what=""):
    og = o_gpu.numpy().astype(np.float64)
    assert np.isfinite(og).all(), f"{what}: non-finite output"
    d = np.abs(og - o_ref)
    if state_dtype == torch.float16:
        lim = F16_OUT_RTOL * np.abs(o_ref) + F16_OUT_ATOL
        assert (d <= lim).all(), f"{what}: output rel diff {(d / (np.abs(o_ref) + 1e-30)).max():.3e}"
    else:
        assert d.max() <= FP32_ATOL, f"{what}: output max abs diff {d.max():.3e}"
    return d
