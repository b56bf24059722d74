"""fp64 CPU oracle for the KDA decode / speculative-verify state update.

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library and its
Python binding never import this package, and this package imports nothing
from them.

The arithmetic lives in ``kda_oracle.c`` (plain fp64 loops).  This module
compiles it with the host C compiler on first use, loads it with ctypes and
marshals NumPy arrays in and out.  Inputs of any float type are widened to
fp64 exactly before the call (bf16, fp16 and fp32 all embed in fp64).

What it computes, per request n, value head h and token t (KDA gated delta
rule; ROCm/ATOM pull requests 2945 "Summary"/"Changes" and 2130 "What"):

    khat = k / sqrt(sum k^2 + 1e-6);  qhat = q / sqrt(sum q^2 + 1e-6)
    beta = sigmoid(b);                alpha_i = exp(-softplus(a_i))
    S <- diag(alpha) S;  u = S^T khat;  S <- S + beta khat (v - u)^T
    o = S^T qhat / sqrt(K)

with S read from the pool slot (widened) or zero on reset, carried in fp64
between tokens, and rounded to the pool's element type (fp32, or fp16 to
nearest even) only where it is stored.

Parity pins (tests/test_oracle_pins.py): dense-matrix brute force in NumPy and
50-digit mpmath, closed forms (identity step, full forget, delta-rule recall,
basis key), the per-token norm bound, and an exhaustive check of the fp16
rounding against NumPy's float64 -> float16 conversion.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_kda.so")
_lock = threading.Lock()
_lib = None

F32 = 0
F16 = 1


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into liboracle_kda.so (gcc, -O2, OpenMP)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = ctypes.POINTER(ctypes.c_int32)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_f64_to_f16_rne.restype = ctypes.c_uint16
            lib.oracle_f64_to_f16_rne.argtypes = [ctypes.c_double]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f64_to_f16_rne_array.argtypes = [dp, ctypes.POINTER(ctypes.c_uint16), ctypes.c_int64]
            lib.oracle_f16_to_f64_array.argtypes = [ctypes.POINTER(ctypes.c_uint16), dp, ctypes.c_int64]
            common = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int]
            lib.oracle_decode_step.restype = ctypes.c_int
            lib.oracle_decode_step.argtypes = common + [i32p, u8p, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            lib.oracle_spec_verify.restype = ctypes.c_int
            lib.oracle_spec_verify.argtypes = common + [ctypes.c_int, i32p, i32p, u8p,
                                                        dp, dp, dp, dp, dp, dp, ctypes.c_int]
            lib.oracle_step.restype = ctypes.c_int
            lib.oracle_step.argtypes = common + [ctypes.c_int, i32p, ctypes.c_int, i32p, ctypes.c_int, i32p,
                                                 ctypes.c_int, u8p, dp, dp, dp, dp, dp, dp, dp, dp,
                                                 ctypes.c_int]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
            lib.oracle_f64_to_bf16_rne_array.argtypes = [dp, ctypes.POINTER(ctypes.c_uint16), ctypes.c_int64]
            lib.oracle_conv_step.restype = ctypes.c_int
            lib.oracle_conv_step.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int64, ctypes.c_int, i32p, ctypes.c_int,
                                             i32p, i32p, u8p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                             dp, dp, ctypes.c_void_p]
            lib.oracle_ckpt_transfer.restype = ctypes.c_int
            lib.oracle_ckpt_transfer.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                                 ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                                 ctypes.c_int, i32p, i32p, ctypes.c_int]
            lib.oracle_prefill.restype = ctypes.c_int
            lib.oracle_prefill.argtypes = common + [ctypes.c_int, i32p, ctypes.c_int, i32p, i32p, u8p,
                                                    dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact widening to a contiguous fp64 array (accepts NumPy or torch CPU tensors)."""
    if hasattr(x, "detach"):  # torch tensor: widen in torch (bf16 has no NumPy type)
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def f64_to_f16_rne(x) -> np.ndarray:
    """Round fp64 values to IEEE binary16 (nearest, ties to even); returns uint16 bits."""
    x = _f64(x)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f64_to_f16_rne_array(_ptr(x.reshape(-1), ctypes.c_double),
                                        _ptr(out.reshape(-1), ctypes.c_uint16), x.size)
    return out


def f16_to_f64(bits) -> np.ndarray:
    """Widen IEEE binary16 bit patterns (uint16) to fp64 exactly."""
    bits = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_f16_to_f64_array(_ptr(bits.reshape(-1), ctypes.c_uint16),
                                    _ptr(out.reshape(-1), ctypes.c_double), bits.size)
    return out


def _pool_args(pool: np.ndarray, slot_stride):
    """pool: NumPy float32 [num_slots, HV, K, V] or uint16 (fp16 bits) of that shape."""
    if not pool.flags.c_contiguous:
        raise ValueError("oracle pool must be C-contiguous")
    if pool.dtype == np.float32:
        dtype = F32
    elif pool.dtype in (np.uint16, np.float16):
        dtype = F16
    else:
        raise ValueError(f"oracle pool dtype {pool.dtype} is neither fp32 nor fp16")
    num_slots, hv, k, v = pool.shape
    if slot_stride is None:
        slot_stride = hv * k * v
    return [pool.ctypes.data, dtype, num_slots, hv, k, v, slot_stride]


def decode_step(pool: np.ndarray, slot_ids, q, k, v, a, b, reset=None,
                slot_stride=None, nthreads: int = 1) -> np.ndarray:
    """One decode token per request; updates ``pool`` in place; returns o fp64 [N, HV, V].

    q, k, a: [N, HV, K]; v: [N, HV, V]; b: [N, HV] (any float type, widened exactly).
    """
    slot_ids = np.ascontiguousarray(np.asarray(slot_ids, dtype=np.int32))
    n = slot_ids.shape[0]
    args = _pool_args(pool, slot_stride)
    hv, vdim = args[3], args[5]
    q64, k64, v64, a64, b64 = (_f64(x) for x in (q, k, v, a, b))
    o = np.zeros((n, hv, vdim), dtype=np.float64)
    rs = None if reset is None else np.ascontiguousarray(np.asarray(reset, dtype=np.uint8))
    rc = _load().oracle_decode_step(
        *args, n, _ptr(slot_ids, ctypes.c_int32),
        None if rs is None else _ptr(rs, ctypes.c_uint8),
        _ptr(q64, ctypes.c_double), _ptr(k64, ctypes.c_double), _ptr(v64, ctypes.c_double),
        _ptr(a64, ctypes.c_double), _ptr(b64, ctypes.c_double), _ptr(o, ctypes.c_double),
        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_decode_step failed ({rc}): slot id out of range")
    return o


def spec_verify(pool: np.ndarray, init_slot, snap_slot, q, k, v, a, b, reset=None,
                slot_stride=None, nthreads: int = 1) -> np.ndarray:
    """T tokens per request; writes the state after token t to snap_slot[n, t].

    q, k, a: [N, T, HV, K]; v: [N, T, HV, V]; b: [N, T, HV].  Returns o fp64 [N, T, HV, V].
    """
    init_slot = np.ascontiguousarray(np.asarray(init_slot, dtype=np.int32))
    snap_slot = np.ascontiguousarray(np.asarray(snap_slot, dtype=np.int32))
    n, t = snap_slot.shape
    args = _pool_args(pool, slot_stride)
    hv, vdim = args[3], args[5]
    q64, k64, v64, a64, b64 = (_f64(x) for x in (q, k, v, a, b))
    o = np.zeros((n, t, hv, vdim), dtype=np.float64)
    rs = None if reset is None else np.ascontiguousarray(np.asarray(reset, dtype=np.uint8))
    rc = _load().oracle_spec_verify(
        *args, n, t, _ptr(init_slot, ctypes.c_int32), _ptr(snap_slot, ctypes.c_int32),
        None if rs is None else _ptr(rs, ctypes.c_uint8),
        _ptr(q64, ctypes.c_double), _ptr(k64, ctypes.c_double), _ptr(v64, ctypes.c_double),
        _ptr(a64, ctypes.c_double), _ptr(b64, ctypes.c_double), _ptr(o, ctypes.c_double),
        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_spec_verify failed ({rc}): slot id out of range")
    return o


def step(pool: np.ndarray, slot_table, q, k, v, a, b, cu_seqlens=None, accepted=None, reset=None,
         a_log=None, dt_bias=None, in_place=False, slot_stride=None, nthreads: int = 1) -> np.ndarray:
    """The general step: packed variable-length requests, a [N, C] slot table
    (initial state at column accepted[r] - 1, token j's state to column j),
    padding requests (negative initial slot), grouped q/k heads and the learned
    gate scale.  Returns o fp64 [total, HV, V].

    q, k: [total, H, K]; v: [total, HV, V]; a: [total, HV, K]; b: [total, HV];
    without cu_seqlens every request has total / N tokens.
    """
    slot_table = np.ascontiguousarray(np.asarray(slot_table, dtype=np.int32))
    n, ncols = slot_table.shape
    args = _pool_args(pool, slot_stride)
    hv, vdim = args[3], args[5]
    q64, k64, v64, a64, b64 = (_f64(x) for x in (q, k, v, a, b))
    total, h_qk = q64.shape[0], q64.shape[1]
    cu = None if cu_seqlens is None else np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    t_uniform = 0 if cu is not None else (total // n if n else 0)
    acc = None if accepted is None else np.ascontiguousarray(np.asarray(accepted, dtype=np.int32))
    rs = None if reset is None else np.ascontiguousarray(np.asarray(reset, dtype=np.uint8))
    al = None if a_log is None else _f64(a_log)
    db = None if dt_bias is None else _f64(dt_bias)
    o = np.zeros((total, hv, vdim), dtype=np.float64)
    opt = lambda x, t: None if x is None else _ptr(x, t)
    rc = _load().oracle_step(
        *args, n, h_qk, opt(cu, ctypes.c_int32), t_uniform, _ptr(slot_table, ctypes.c_int32), ncols,
        opt(acc, ctypes.c_int32), int(bool(in_place)), opt(rs, ctypes.c_uint8),
        _ptr(q64, ctypes.c_double), _ptr(k64, ctypes.c_double), _ptr(v64, ctypes.c_double),
        _ptr(a64, ctypes.c_double), _ptr(b64, ctypes.c_double), opt(al, ctypes.c_double),
        opt(db, ctypes.c_double), _ptr(o, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_step failed ({rc}): " + ("slot id out of range" if rc == -1 else "layout"))
    return o


def f64_to_bf16_rne(x) -> np.ndarray:
    """Round fp64 values to bfloat16 (nearest, ties to even, one rounding); returns uint16 bits."""
    x = _f64(x)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f64_to_bf16_rne_array(_ptr(x.reshape(-1), ctypes.c_double),
                                         _ptr(out.reshape(-1), ctypes.c_uint16), x.size)
    return out


CONV_DTYPES = {"float32": 0, "float16": 1, "bfloat16": 2}


def conv_step(window: np.ndarray, dtype: str, conv_slot, x: np.ndarray, weight, bias=None, cu_seqlens=None,
              accepted=None, reset=None, silu=True) -> np.ndarray:
    """The causal short convolution with its paged window (see oracle_conv_step).

    window: [num_slots, L, C] as float32, or uint16 bit patterns for fp16/bf16
    (``dtype`` names which); x: [total, C] of the same storage; weight fp64
    [C, KW]; bias [C] or None.  Updates ``window`` in place and returns y with
    x's storage type, [total, C]."""
    code = CONV_DTYPES[dtype]
    window = window if window.flags.c_contiguous else None
    if window is None:
        raise ValueError("window must be C-contiguous")
    num_slots, L, C = window.shape
    x = np.ascontiguousarray(x)
    total = x.shape[0]
    conv_slot = np.ascontiguousarray(np.asarray(conv_slot, dtype=np.int32))
    n = conv_slot.shape[0]
    w = _f64(weight)
    kw = w.shape[1]
    b = None if bias is None else _f64(bias)
    cu = None if cu_seqlens is None else np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    acc = None if accepted is None else np.ascontiguousarray(np.asarray(accepted, dtype=np.int32))
    rs = None if reset is None else np.ascontiguousarray(np.asarray(reset, dtype=np.uint8))
    y = np.zeros_like(x)
    opt = lambda a, t: None if a is None else _ptr(a, t)  # noqa: E731
    rc = _load().oracle_conv_step(window.ctypes.data, code, num_slots, C, L, L * C, n,
                                  opt(cu, ctypes.c_int32), 0 if cu is not None else (total // n if n else 0),
                                  _ptr(conv_slot, ctypes.c_int32), opt(acc, ctypes.c_int32),
                                  opt(rs, ctypes.c_uint8), kw, int(bool(silu)), x.ctypes.data,
                                  _ptr(w, ctypes.c_double), opt(b, ctypes.c_double), y.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_conv_step failed ({rc})")
    return y


def ckpt_transfer(pool: np.ndarray, plane: np.ndarray, slots, entries, load: bool) -> None:
    """Checkpoint flush (load=False: plane[entries] <- pool[slots]) or load
    (pool[slots] <- plane[entries]) of whole slot states; negative indices
    skip.  pool [num_slots, HV, K, V] and plane [num_entries, HV, K, V] share
    an element type (float32, or uint16 fp16 bits)."""
    if pool.dtype != plane.dtype or pool.shape[1:] != plane.shape[1:]:
        raise ValueError("pool and plane differ in element type or state shape")
    if not (pool.flags.c_contiguous and plane.flags.c_contiguous):
        raise ValueError("pool and plane must be C-contiguous")
    slots = np.ascontiguousarray(np.asarray(slots, dtype=np.int32))
    entries = np.ascontiguousarray(np.asarray(entries, dtype=np.int32))
    state = int(np.prod(pool.shape[1:]))
    rc = _load().oracle_ckpt_transfer(pool.ctypes.data, pool.shape[0], state, plane.ctypes.data, plane.shape[0],
                                      state, state, pool.itemsize, slots.shape[0], _ptr(slots, ctypes.c_int32),
                                      _ptr(entries, ctypes.c_int32), int(bool(load)))
    if rc != 0:
        raise ValueError("oracle_ckpt_transfer: index out of range")


def prefill(pool: np.ndarray, init_slot, final_slot, q, k, v, a, b, cu_seqlens=None, reset=None,
            a_log=None, dt_bias=None, slot_stride=None, nthreads: int = 1) -> np.ndarray:
    """Prefill over packed prompts: the state from init_slot[r] (zero on reset;
    negative: padding), the state after the last token to final_slot[r]
    (negative: not stored).  q, k: [total, H, K]; v: [total, HV, V];
    a: [total, HV, K]; b: [total, HV].  Returns o fp64 [total, HV, V]."""
    init_slot = np.ascontiguousarray(np.asarray(init_slot, dtype=np.int32))
    final_slot = np.ascontiguousarray(np.asarray(final_slot, dtype=np.int32))
    n = init_slot.shape[0]
    args = _pool_args(pool, slot_stride)
    hv, vdim = args[3], args[5]
    q64, k64, v64, a64, b64 = (_f64(x) for x in (q, k, v, a, b))
    total, h_qk = q64.shape[0], q64.shape[1]
    cu = None if cu_seqlens is None else np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    t_uniform = 0 if cu is not None else (total // n if n else 0)
    rs = None if reset is None else np.ascontiguousarray(np.asarray(reset, dtype=np.uint8))
    al = None if a_log is None else _f64(a_log)
    db = None if dt_bias is None else _f64(dt_bias)
    o = np.zeros((total, hv, vdim), dtype=np.float64)
    opt = lambda x, t: None if x is None else _ptr(x, t)  # noqa: E731
    rc = _load().oracle_prefill(
        *args, n, h_qk, opt(cu, ctypes.c_int32), t_uniform, _ptr(init_slot, ctypes.c_int32),
        _ptr(final_slot, ctypes.c_int32), opt(rs, ctypes.c_uint8), _ptr(q64, ctypes.c_double),
        _ptr(k64, ctypes.c_double), _ptr(v64, ctypes.c_double), _ptr(a64, ctypes.c_double),
        _ptr(b64, ctypes.c_double), opt(al, ctypes.c_double), opt(db, ctypes.c_double),
        _ptr(o, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_prefill failed ({rc})")
    return o
