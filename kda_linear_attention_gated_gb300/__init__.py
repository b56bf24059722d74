"""Python binding of the GB300 KDA recurrent-state library (include/kda.h).

Argument marshalling only: every step of the state update runs in the CUDA
kernels of ``libkda_h0.so`` (fp32 pool) / ``libkda_h1.so`` (fp16 pool).  There
is no CPU fallback: if the library is missing, ``KdaLibrary`` raises.

    import torch, kda_linear_attention_gated_gb300 as kda
    lib = kda.KdaLibrary(torch.float16)          # loads libkda_h1.so
    pool = torch.zeros(256, 12, 128, 128, dtype=torch.float16, device="cuda")
    lib.kda_decode_step(pool, slot_ids, q, k, v, a, b, o, status)

Tensors are PyTorch CUDA tensors (PyTorch supplies device memory and the
stream); the calls are asynchronous on ``stream`` (default: the current
PyTorch stream).  Names follow the C ABI one to one.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_DIR, SOURCES, build, lib_path  # noqa: F401  (re-exported)

__all__ = ["KdaError", "KdaLibrary", "PoolDesc", "build", "lib_path",
           "KDA_F32", "KDA_F16", "KDA_BF16", "KDA_OK", "KDA_ERR_NULL",
           "KDA_ERR_DTYPE_MISMATCH", "KDA_ERR_DTYPE_UNSUPPORTED", "KDA_ERR_LAYERS_DISAGREE",
           "KDA_ERR_SHAPE", "KDA_ERR_ALIGN", "KDA_ERR_LAUNCH", "KDA_ERR_SLOT_RANGE",
           "KDA_ERR_ARG", "KDA_ERR_TIMEOUT", "KDA_ERR_LAYOUT", "KDA_LAUNCH_PDL", "KDA_LAUNCH_PDL_EARLY_STATE",
           "KDA_LAUNCH_TEST_WITHHOLD_STATE", "EXPORTED_SYMBOLS"]

KDA_F32, KDA_F16, KDA_BF16 = 0, 1, 2
KDA_LAUNCH_PDL, KDA_LAUNCH_PDL_EARLY_STATE = 1, 2
KDA_LAUNCH_TEST_WITHHOLD_STATE = 1 << 30  # test hook of the timeout path (include/kda.h)
(KDA_OK, KDA_ERR_NULL, KDA_ERR_DTYPE_MISMATCH, KDA_ERR_DTYPE_UNSUPPORTED,
 KDA_ERR_LAYERS_DISAGREE, KDA_ERR_SHAPE, KDA_ERR_ALIGN, KDA_ERR_LAUNCH,
 KDA_ERR_SLOT_RANGE, KDA_ERR_ARG, KDA_ERR_TIMEOUT, KDA_ERR_LAYOUT) = range(12)

EXPORTED_SYMBOLS = ("kda_build_state_dtype", "kda_pool_check", "kda_state_bytes",
                    "kda_decode_step", "kda_spec_verify", "kda_step", "kda_prefill", "kda_prefill_workspace_bytes",
                    "kda_prefill_chunked", "kda_prefill_chunked_noalloc", "kda_conv_step", "kda_decode_conv_step",
                    "kda_step_conv",
                    "kda_layout_id", "kda_ckpt_flush", "kda_ckpt_load", "kda_stage_host", "kda_strerror")


class KdaError(RuntimeError):
    def __init__(self, code: int, what: str, msg: str):
        super().__init__(f"{what}: {msg} (status {code})")
        self.code = code


class PoolDesc(ctypes.Structure):
    """Mirror of ``struct kda_pool`` (include/kda.h)."""
    _fields_ = [("base", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("hv", ctypes.c_int32),
                ("k", ctypes.c_int32), ("v", ctypes.c_int32), ("num_slots", ctypes.c_int64),
                ("slot_stride", ctypes.c_int64)]


class StepArgs(ctypes.Structure):
    """Mirror of ``struct kda_step_args`` (include/kda.h)."""
    _fields_ = [("n", ctypes.c_int32), ("total", ctypes.c_int32), ("max_t", ctypes.c_int32),
                ("h_qk", ctypes.c_int32), ("num_cols", ctypes.c_int32), ("in_place", ctypes.c_int32),
                ("qkv_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("slot_table", ctypes.c_void_p),
                ("accepted", ctypes.c_void_p), ("reset", ctypes.c_void_p), ("q", ctypes.c_void_p),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("a", ctypes.c_void_p),
                ("b", ctypes.c_void_p), ("a_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("o", ctypes.c_void_p)]


class PrefillArgs(ctypes.Structure):
    """Mirror of ``struct kda_prefill_args`` (include/kda.h)."""
    _fields_ = [("n", ctypes.c_int32), ("total", ctypes.c_int32), ("max_t", ctypes.c_int32),
                ("h_qk", ctypes.c_int32), ("qkv_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("init_slot", ctypes.c_void_p), ("final_slot", ctypes.c_void_p),
                ("reset", ctypes.c_void_p), ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("a_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("o", ctypes.c_void_p)]


class ConvWindowDesc(ctypes.Structure):
    """Mirror of ``struct kda_conv_window`` (include/kda.h)."""
    _fields_ = [("base", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("channels", ctypes.c_int32),
                ("state_len", ctypes.c_int32), ("reserved", ctypes.c_int32), ("num_slots", ctypes.c_int64),
                ("slot_stride", ctypes.c_int64)]


class ConvArgs(ctypes.Structure):
    """Mirror of ``struct kda_conv_args`` (include/kda.h)."""
    _fields_ = [("n", ctypes.c_int32), ("total", ctypes.c_int32), ("max_t", ctypes.c_int32),
                ("kernel_width", ctypes.c_int32), ("activation", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("conv_slot", ctypes.c_void_p), ("accepted", ctypes.c_void_p),
                ("reset", ctypes.c_void_p), ("x", ctypes.c_void_p), ("weight", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class DecodeConvArgs(ctypes.Structure):
    """Mirror of ``struct kda_decode_conv_args`` (include/kda.h)."""
    _fields_ = [("n", ctypes.c_int32), ("h_qk", ctypes.c_int32), ("kernel_width", ctypes.c_int32),
                ("activation", ctypes.c_int32), ("slot_ids", ctypes.c_void_p), ("conv_slot", ctypes.c_void_p),
                ("reset", ctypes.c_void_p), ("x", ctypes.c_void_p), ("weight", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("o", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("counters", ctypes.c_void_p), ("a_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p)]


class StepConvArgs(ctypes.Structure):
    """Mirror of ``struct kda_step_conv_args`` (include/kda.h)."""
    _fields_ = [("kernel_width", ctypes.c_int32), ("activation", ctypes.c_int32), ("conv_slot", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("counters", ctypes.c_void_p)]


class HostCopy(ctypes.Structure):
    """Mirror of ``struct kda_host_copy`` (include/kda.h)."""
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_int64)]


class CkptPlaneDesc(ctypes.Structure):
    """Mirror of ``struct kda_ckpt_plane`` (include/kda.h)."""
    _fields_ = [("base", ctypes.c_void_p), ("layout_id", ctypes.c_uint32), ("reserved", ctypes.c_int32),
                ("num_entries", ctypes.c_int64), ("entry_stride", ctypes.c_int64)]


def _dtype_code(dt) -> int:
    import torch
    table = {torch.float32: KDA_F32, torch.float16: KDA_F16, torch.bfloat16: KDA_BF16}
    if dt not in table:
        raise ValueError(f"dtype {dt} has no kda_dtype code")
    return table[dt]


def pool_desc(pool) -> PoolDesc:
    """Descriptor of a [num_slots, hv, k, v] tensor whose inner three dims are dense."""
    if pool.dim() != 4:
        raise ValueError("a state pool is a [num_slots, hv, k, v] tensor")
    ns, hv, k, v = pool.shape
    if pool.stride(3) != 1 or pool.stride(2) != v or pool.stride(1) != k * v:
        raise ValueError("the [hv, k, v] part of a state pool must be dense (v innermost)")
    return PoolDesc(pool.data_ptr(), _dtype_code(pool.dtype), hv, k, v, ns, pool.stride(0))


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _expect(name, t, shape, dtypes) -> None:
    """Shape/dtype/contiguity/device check, so that no kernel indexes past a buffer."""
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


_libs: dict[bool, ctypes.CDLL] = {}
_lock = threading.Lock()


def _load(state16: bool) -> ctypes.CDLL:
    with _lock:
        if state16 in _libs:
            return _libs[state16]
        path = lib_path(state16)
        if not os.path.exists(path):
            raise RuntimeError(
                f"KDA CUDA library {path} is missing; build it with "
                "kda_linear_attention_gated_gb300.build() (there is no CPU fallback)")
        import torch  # noqa: F401  -- loads the CUDA runtime the library shares
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(PoolDesc)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        lib.kda_build_state_dtype.restype = ctypes.c_int
        lib.kda_build_state_dtype.argtypes = []
        lib.kda_pool_check.restype = ctypes.c_int
        lib.kda_pool_check.argtypes = [P, i32]
        lib.kda_state_bytes.restype = ctypes.c_int
        lib.kda_state_bytes.argtypes = [P, ctypes.POINTER(ctypes.c_int64)]
        lib.kda_decode_step.restype = ctypes.c_int
        u32 = ctypes.c_uint32
        lib.kda_decode_step.argtypes = [P, vp, vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, u32, vp]
        lib.kda_spec_verify.restype = ctypes.c_int
        lib.kda_spec_verify.argtypes = [P, vp, vp, vp, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, u32, vp]
        lib.kda_step.restype = ctypes.c_int
        lib.kda_step.argtypes = [P, ctypes.POINTER(StepArgs), vp, u32, vp]
        lib.kda_prefill.restype = ctypes.c_int
        lib.kda_prefill.argtypes = [P, ctypes.POINTER(PrefillArgs), vp, u32, vp]
        lib.kda_prefill_workspace_bytes.restype = ctypes.c_int
        lib.kda_prefill_workspace_bytes.argtypes = [P, i32, i32, ctypes.POINTER(ctypes.c_int64)]
        lib.kda_prefill_chunked.restype = ctypes.c_int
        lib.kda_prefill_chunked.argtypes = [P, ctypes.POINTER(PrefillArgs), vp, ctypes.c_int64, vp, u32, vp]
        lib.kda_prefill_chunked_noalloc.restype = ctypes.c_int
        lib.kda_prefill_chunked_noalloc.argtypes = [P, ctypes.POINTER(PrefillArgs), vp, u32, vp]
        lib.kda_conv_step.restype = ctypes.c_int
        lib.kda_conv_step.argtypes = [ctypes.POINTER(ConvWindowDesc), ctypes.POINTER(ConvArgs), vp, u32, vp]
        lib.kda_step_conv.restype = ctypes.c_int
        lib.kda_step_conv.argtypes = [P, ctypes.POINTER(StepArgs), ctypes.POINTER(ConvWindowDesc),
                                      ctypes.POINTER(StepConvArgs), vp, u32, vp]
        lib.kda_decode_conv_step.restype = ctypes.c_int
        lib.kda_decode_conv_step.argtypes = [P, ctypes.POINTER(ConvWindowDesc), ctypes.POINTER(DecodeConvArgs),
                                             vp, u32, vp]
        lib.kda_layout_id.restype = ctypes.c_uint32
        lib.kda_layout_id.argtypes = [P]
        for fn in (lib.kda_ckpt_flush, lib.kda_ckpt_load):
            fn.restype = ctypes.c_int
            fn.argtypes = [P, ctypes.POINTER(CkptPlaneDesc), vp, vp, i32, vp, u32, vp]
        lib.kda_stage_host.restype = ctypes.c_int
        lib.kda_stage_host.argtypes = [ctypes.POINTER(HostCopy), i32, u32, vp]
        lib.kda_strerror.restype = ctypes.c_char_p
        lib.kda_strerror.argtypes = [i32]
        _libs[state16] = lib
        return lib


class KdaLibrary:
    """One build of the library: ``state_dtype`` torch.float32 -> libkda_h0, float16 -> libkda_h1."""

    def __init__(self, state_dtype):
        import torch
        if state_dtype not in (torch.float32, torch.float16):
            raise ValueError("the state pool dtype of a build is fp32 or fp16")
        self.state_dtype = state_dtype
        self.lib = _load(state_dtype == torch.float16)
        self.path = lib_path(state_dtype == torch.float16)

    # -- helpers ------------------------------------------------------------
    def _check(self, rc: int, what: str) -> None:
        if rc != KDA_OK:
            raise KdaError(rc, what, self.kda_strerror(rc))

    @staticmethod
    def _stream(stream) -> int | None:
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)

    # -- the C ABI, one to one ---------------------------------------------
    def kda_build_state_dtype(self) -> int:
        return self.lib.kda_build_state_dtype()

    def kda_strerror(self, code: int) -> str:
        return self.lib.kda_strerror(int(code)).decode()

    def kda_pool_check_raw(self, descs) -> int:
        arr = (PoolDesc * len(descs))(*descs)
        return self.lib.kda_pool_check(arr, len(descs))

    def kda_pool_check(self, pools) -> None:
        """Raise KdaError unless every layer's pool is valid for this build."""
        self._check(self.kda_pool_check_raw([pool_desc(p) for p in pools]), "kda_pool_check")

    def kda_state_bytes(self, pool) -> int:
        desc = pool if isinstance(pool, PoolDesc) else pool_desc(pool)
        out = ctypes.c_int64(0)
        self._check(self.lib.kda_state_bytes(ctypes.byref(desc), ctypes.byref(out)), "kda_state_bytes")
        return out.value

    def kda_decode_step_raw(self, desc: PoolDesc, slot_ids, reset, n, q, k, v, qkv_dtype,
                            a, b, o, status, stream, flags=0) -> int:
        return self.lib.kda_decode_step(ctypes.byref(desc), slot_ids, reset, n, q, k, v,
                                        qkv_dtype, a, b, o, status, flags, stream)

    def kda_decode_step(self, pool, slot_ids, q, k, v, a, b, o, status, reset=None,
                        stream=None, flags=0) -> None:
        """One decode token per request; ``pool`` is updated in place (see include/kda.h)."""
        import torch
        desc = pool_desc(pool)
        n, hv, kd, vd = int(slot_ids.shape[0]), desc.hv, desc.k, desc.v
        qkv_types = (torch.float32, torch.float16, torch.bfloat16)
        _expect("slot_ids", slot_ids, (n,), (torch.int32,))
        for name, t in (("q", q), ("k", k)):
            _expect(name, t, (n, hv, kd), (q.dtype,) if name == "k" else qkv_types)
        _expect("v", v, (n, hv, vd), (q.dtype,))
        _expect("a", a, (n, hv, kd), (torch.float32,))
        _expect("b", b, (n, hv), (torch.float32,))
        _expect("o", o, (n, hv, vd), (torch.float32,))
        _expect("status", status, (1,), (torch.int32,))
        if reset is not None:
            _expect("reset", reset, (n,), (torch.uint8,))
        rc = self.kda_decode_step_raw(
            desc, _ptr(slot_ids), _ptr(reset), int(slot_ids.shape[0]), _ptr(q), _ptr(k),
            _ptr(v), _dtype_code(q.dtype), _ptr(a), _ptr(b), _ptr(o), _ptr(status),
            self._stream(stream), flags)
        self._check(rc, "kda_decode_step")

    def kda_spec_verify(self, pool, init_slot, snap_slot, q, k, v, a, b, o, status,
                        reset=None, stream=None, flags=0) -> None:
        """T tokens per request; the state after token t goes to snap_slot[n, t]."""
        import torch
        desc = pool_desc(pool)
        n, t = int(snap_slot.shape[0]), int(snap_slot.shape[1])
        hv, kd, vd = desc.hv, desc.k, desc.v
        qkv_types = (torch.float32, torch.float16, torch.bfloat16)
        _expect("init_slot", init_slot, (n,), (torch.int32,))
        _expect("snap_slot", snap_slot, (n, t), (torch.int32,))
        _expect("q", q, (n, t, hv, kd), qkv_types)
        _expect("k", k, (n, t, hv, kd), (q.dtype,))
        _expect("v", v, (n, t, hv, vd), (q.dtype,))
        _expect("a", a, (n, t, hv, kd), (torch.float32,))
        _expect("b", b, (n, t, hv), (torch.float32,))
        _expect("o", o, (n, t, hv, vd), (torch.float32,))
        _expect("status", status, (1,), (torch.int32,))
        if reset is not None:
            _expect("reset", reset, (n,), (torch.uint8,))
        rc = self.lib.kda_spec_verify(
            ctypes.byref(desc), _ptr(init_slot), _ptr(snap_slot), _ptr(reset), n, t,
            _ptr(q), _ptr(k), _ptr(v), _dtype_code(q.dtype), _ptr(a), _ptr(b), _ptr(o),
            _ptr(status), flags, self._stream(stream))
        self._check(rc, "kda_spec_verify")

    def kda_step_raw(self, desc: PoolDesc, args: StepArgs, status, stream, flags=0) -> int:
        return self.lib.kda_step(ctypes.byref(desc), ctypes.byref(args), status, flags, stream)

    def kda_step(self, pool, slot_table, q, k, v, a, b, o, status, cu_seqlens=None, max_t=None,
                 accepted=None, reset=None, a_log=None, dt_bias=None, in_place=False, stream=None,
                 flags=0) -> None:
        """The general step (see kda_step_args in include/kda.h): packed tokens
        q, k [total, H, K], v [total, HV, V], a [total, HV, K], b [total, HV],
        o [total, HV, V]; slot_table [N, C]; cu_seqlens [N + 1] (then max_t is
        required) or None (every request has total / N tokens)."""
        import torch
        desc = pool_desc(pool)
        hv, kd, vd = desc.hv, desc.k, desc.v
        n, ncols = int(slot_table.shape[0]), int(slot_table.shape[1])
        total, h_qk = int(q.shape[0]), int(q.shape[1])
        qkv_types = (torch.float32, torch.float16, torch.bfloat16)
        _expect("slot_table", slot_table, (n, ncols), (torch.int32,))
        _expect("q", q, (total, h_qk, kd), qkv_types)
        _expect("k", k, (total, h_qk, kd), (q.dtype,))
        _expect("v", v, (total, hv, vd), (q.dtype,))
        _expect("a", a, (total, hv, kd), (torch.float32,))
        _expect("b", b, (total, hv), (torch.float32,))
        _expect("o", o, (total, hv, vd), (torch.float32,))
        _expect("status", status, (1,), (torch.int32,))
        if cu_seqlens is not None:
            _expect("cu_seqlens", cu_seqlens, (n + 1,), (torch.int32,))
            if max_t is None:
                raise ValueError("max_t is required with cu_seqlens")
        elif max_t is None:
            max_t = total // n if n else 0
        if accepted is not None:
            _expect("accepted", accepted, (n,), (torch.int32,))
        if reset is not None:
            _expect("reset", reset, (n,), (torch.uint8,))
        if a_log is not None:
            _expect("a_log", a_log, (hv,), (torch.float32,))
        if dt_bias is not None:
            _expect("dt_bias", dt_bias, (hv, kd), (torch.float32,))
        args = StepArgs(n, total, int(max_t), h_qk, ncols, int(bool(in_place)), _dtype_code(q.dtype), 0,
                        _ptr(cu_seqlens), _ptr(slot_table), _ptr(accepted), _ptr(reset), _ptr(q), _ptr(k),
                        _ptr(v), _ptr(a), _ptr(b), _ptr(a_log), _ptr(dt_bias), _ptr(o))
        self._check(self.kda_step_raw(desc, args, _ptr(status), self._stream(stream), flags), "kda_step")

    def kda_conv_step_raw(self, win: ConvWindowDesc, args: ConvArgs, status, stream, flags=0) -> int:
        return self.lib.kda_conv_step(ctypes.byref(win), ctypes.byref(args), status, flags, stream)

    def kda_conv_step(self, window, conv_slot, x, weight, y, status, bias=None, cu_seqlens=None, max_t=None,
                      accepted=None, reset=None, silu=True, stream=None, flags=0) -> None:
        """The short convolution with its paged window (see kda_conv_args in
        include/kda.h): window [num_slots, L, C] (C innermost), x and y
        [total, C] of the window's dtype, weight fp32 [C, KW], bias [C]."""
        import torch
        if window.dim() != 3 or window.stride(2) != 1 or window.stride(1) != window.shape[2]:
            raise ValueError("a conv window pool is a [num_slots, L, C] tensor, dense in [L, C]")
        ns, L, C = window.shape
        n, total, kw = int(conv_slot.shape[0]), int(x.shape[0]), int(weight.shape[1])
        _expect("conv_slot", conv_slot, (n,), (torch.int32,))
        _expect("x", x, (total, C), (window.dtype,))
        _expect("y", y, (total, C), (window.dtype,))
        _expect("weight", weight, (C, kw), (torch.float32,))
        _expect("status", status, (1,), (torch.int32,))
        if bias is not None:
            _expect("bias", bias, (C,), (torch.float32,))
        if cu_seqlens is not None:
            _expect("cu_seqlens", cu_seqlens, (n + 1,), (torch.int32,))
            if max_t is None:
                raise ValueError("max_t is required with cu_seqlens")
        elif max_t is None:
            max_t = total // n if n else 0
        if accepted is not None:
            _expect("accepted", accepted, (n,), (torch.int32,))
        if reset is not None:
            _expect("reset", reset, (n,), (torch.uint8,))
        win = ConvWindowDesc(window.data_ptr(), _dtype_code(window.dtype), C, L, 0, ns, window.stride(0))
        args = ConvArgs(n, total, int(max_t), kw, int(bool(silu)), 0, _ptr(cu_seqlens), _ptr(conv_slot),
                        _ptr(accepted), _ptr(reset), _ptr(x), _ptr(weight), _ptr(bias), _ptr(y))
        self._check(self.kda_conv_step_raw(win, args, _ptr(status), self._stream(stream), flags), "kda_conv_step")

    def kda_decode_conv_step_raw(self, desc: PoolDesc, win: ConvWindowDesc, args: DecodeConvArgs, status, stream,
                                 flags=0) -> int:
        return self.lib.kda_decode_conv_step(ctypes.byref(desc), ctypes.byref(win), ctypes.byref(args), status,
                                             flags, stream)

    def kda_decode_conv_step(self, pool, window, slot_ids, conv_slot, x, weight, a, b, o, status, counters,
                             bias=None, y=None, reset=None, h_qk=None, silu=True, a_log=None, dt_bias=None,
                             stream=None, flags=0) -> None:
        """One decode token per request with the short convolution fused in
        front of the recurrence (see kda_decode_conv_args in include/kda.h):
        x [n, C] of the window's dtype with C = 2 h_qk K + HV V (q | k | v
        channels), window [num_slots, L, C], weight fp32 [C, KW], counters
        int32 [n, h_qk] (zero; left zero)."""
        import torch
        desc = pool_desc(pool)
        if window.dim() != 3 or window.stride(2) != 1 or window.stride(1) != window.shape[2]:
            raise ValueError("a conv window pool is a [num_slots, L, C] tensor, dense in [L, C]")
        ns, L, C = window.shape
        n, kw = int(slot_ids.shape[0]), int(weight.shape[1])
        hv, kd, vd = desc.hv, desc.k, desc.v
        h_qk = hv if h_qk is None else int(h_qk)
        _expect("slot_ids", slot_ids, (n,), (torch.int32,))
        _expect("conv_slot", conv_slot, (n,), (torch.int32,))
        _expect("x", x, (n, C), (window.dtype,))
        _expect("weight", weight, (C, kw), (torch.float32,))
        _expect("a", a, (n, hv, kd), (torch.float32,))
        _expect("b", b, (n, hv), (torch.float32,))
        _expect("o", o, (n, hv, vd), (torch.float32,))
        _expect("counters", counters, (n, h_qk), (torch.int32,))
        _expect("status", status, (1,), (torch.int32,))
        if bias is not None:
            _expect("bias", bias, (C,), (torch.float32,))
        if y is not None:
            _expect("y", y, (n, C), (window.dtype,))
        if reset is not None:
            _expect("reset", reset, (n,), (torch.uint8,))
        if a_log is not None:
            _expect("a_log", a_log, (hv,), (torch.float32,))
        if dt_bias is not None:
            _expect("dt_bias", dt_bias, (hv, kd), (torch.float32,))
        win = ConvWindowDesc(window.data_ptr(), _dtype_code(window.dtype), C, L, 0, ns, window.stride(0))
        args = DecodeConvArgs(n, h_qk, kw, int(bool(silu)), _ptr(slot_ids), _ptr(conv_slot), _ptr(reset), _ptr(x),
                              _ptr(weight), _ptr(bias), _ptr(a), _ptr(b), _ptr(o), _ptr(y), _ptr(counters),
                              _ptr(a_log), _ptr(dt_bias))
        self._check(self.kda_decode_conv_step_raw(desc, win, args, _ptr(status), self._stream(stream), flags),
                    "kda_decode_conv_step")

    def kda_step_conv_raw(self, desc: PoolDesc, args: StepArgs, win: ConvWindowDesc, cargs: StepConvArgs, status,
                          stream, flags=0) -> int:
        return self.lib.kda_step_conv(ctypes.byref(desc), ctypes.byref(args), ctypes.byref(win), ctypes.byref(cargs),
                                      status, flags, stream)

    def kda_step_conv(self, pool, window, slot_table, conv_slot, x, weight, a, b, o, status, counters,
                      cu_seqlens=None, max_t=None, accepted=None, reset=None, a_log=None, dt_bias=None, bias=None,
                      y=None, h_qk=None, silu=True, stream=None, flags=0) -> None:
        """The general speculative step with the short convolution fused in
        front (see kda_step_conv_args in include/kda.h): packed tokens x
        [total, C] of the window's dtype (q | k | v channels, C = 2 h_qk K +
        HV V), a [total, HV, K], b [total, HV], o [total, HV, V]; slot_table
        [N, num_cols]; window [num_slots, L, C]; counters int32 [N, h_qk]."""
        import torch
        desc = pool_desc(pool)
        hv, kd, vd = desc.hv, desc.k, desc.v
        if window.dim() != 3 or window.stride(2) != 1 or window.stride(1) != window.shape[2]:
            raise ValueError("a conv window pool is a [num_slots, L, C] tensor, dense in [L, C]")
        ns, L, C = window.shape
        n, ncols = int(slot_table.shape[0]), int(slot_table.shape[1])
        total, kw = int(x.shape[0]), int(weight.shape[1])
        h_qk = hv if h_qk is None else int(h_qk)
        _expect("slot_table", slot_table, (n, ncols), (torch.int32,))
        _expect("conv_slot", conv_slot, (n,), (torch.int32,))
        _expect("x", x, (total, C), (window.dtype,))
        _expect("weight", weight, (C, kw), (torch.float32,))
        _expect("a", a, (total, hv, kd), (torch.float32,))
        _expect("b", b, (total, hv), (torch.float32,))
        _expect("o", o, (total, hv, vd), (torch.float32,))
        _expect("counters", counters, (n, h_qk), (torch.int32,))
        _expect("status", status, (1,), (torch.int32,))
        for name, t, shape in (("bias", bias, (C,)), ("a_log", a_log, (hv,)), ("dt_bias", dt_bias, (hv, kd))):
            if t is not None:
                _expect(name, t, shape, (torch.float32,))
        if y is not None:
            _expect("y", y, (total, C), (window.dtype,))
        if cu_seqlens is not None:
            _expect("cu_seqlens", cu_seqlens, (n + 1,), (torch.int32,))
            if max_t is None:
                raise ValueError("max_t is required with cu_seqlens")
        elif max_t is None:
            max_t = total // n if n else 0
        if accepted is not None:
            _expect("accepted", accepted, (n,), (torch.int32,))
        if reset is not None:
            _expect("reset", reset, (n,), (torch.uint8,))
        wd = _dtype_code(window.dtype)
        args = StepArgs(n, total, int(max_t), h_qk, ncols, 0, wd, 0, _ptr(cu_seqlens), _ptr(slot_table),
                        _ptr(accepted), _ptr(reset), None, None, None, _ptr(a), _ptr(b), _ptr(a_log), _ptr(dt_bias),
                        _ptr(o))
        win = ConvWindowDesc(window.data_ptr(), wd, C, L, 0, ns, window.stride(0))
        cargs = StepConvArgs(kw, int(bool(silu)), _ptr(conv_slot), _ptr(x), _ptr(weight), _ptr(bias), _ptr(y),
                             _ptr(counters))
        self._check(self.kda_step_conv_raw(desc, args, win, cargs, _ptr(status), self._stream(stream), flags),
                    "kda_step_conv")

    def kda_stage_host_raw(self, copies, stream, flags=0) -> int:
        """copies: a list of (dst device address, src pinned host address, bytes)."""
        arr = (HostCopy * max(1, len(copies)))(*[HostCopy(d, s_, b) for d, s_, b in copies])
        return self.lib.kda_stage_host(arr, len(copies), flags, stream)

    def kda_stage_host(self, pairs, stream=None, flags=0) -> None:
        """Copy each (dst, src) pair -- dst a contiguous CUDA tensor, src a
        contiguous pinned CPU tensor of the same byte size -- with one kernel
        launch (see kda_stage_host in include/kda.h)."""
        copies = []
        for dst, src in pairs:
            if not dst.is_cuda or src.is_cuda or not dst.is_contiguous() or not src.is_contiguous():
                raise ValueError("kda_stage_host copies a contiguous pinned CPU tensor into a contiguous CUDA tensor")
            nb = dst.numel() * dst.element_size()
            if src.numel() * src.element_size() != nb:
                raise ValueError("source and destination differ in size")
            copies.append((dst.data_ptr(), src.data_ptr(), nb))
        self._check(self.kda_stage_host_raw(copies, self._stream(stream), flags), "kda_stage_host")

    def kda_layout_id(self, pool) -> int:
        desc = pool if isinstance(pool, PoolDesc) else pool_desc(pool)
        return int(self.lib.kda_layout_id(ctypes.byref(desc)))

    def plane_desc(self, plane, pool, layout_id=None) -> CkptPlaneDesc:
        """Descriptor of a [num_entries, hv, k, v] checkpoint plane serving ``pool``."""
        if plane.dim() != 4 or tuple(plane.shape[1:]) != tuple(pool.shape[1:]) or plane.dtype != pool.dtype:
            raise ValueError("a checkpoint plane is [num_entries, hv, k, v] of the pool's dtype")
        if not plane[0].is_contiguous():
            raise ValueError("each plane entry must be dense")
        lid = self.kda_layout_id(pool) if layout_id is None else layout_id
        return CkptPlaneDesc(plane.data_ptr(), lid, 0, plane.shape[0], plane.stride(0))

    def _ckpt(self, fn, name, pool, plane, slots, entries, status, layout_id, stream, flags):
        import torch
        n = int(slots.shape[0])
        _expect("slots", slots, (n,), (torch.int32,))
        _expect("entries", entries, (n,), (torch.int32,))
        _expect("status", status, (1,), (torch.int32,))
        desc, pdesc = pool_desc(pool), self.plane_desc(plane, pool, layout_id)
        self._check(fn(ctypes.byref(desc), ctypes.byref(pdesc), _ptr(slots), _ptr(entries), n, _ptr(status),
                       flags, self._stream(stream)), name)

    def kda_ckpt_flush(self, pool, plane, slots, entries, status, layout_id=None, stream=None, flags=0) -> None:
        """plane[entries[i]] <- pool[slots[i]] (whole states, bit for bit)."""
        self._ckpt(self.lib.kda_ckpt_flush, "kda_ckpt_flush", pool, plane, slots, entries, status, layout_id,
                   stream, flags)

    def kda_ckpt_load(self, pool, plane, slots, entries, status, layout_id=None, stream=None, flags=0) -> None:
        """pool[slots[i]] <- plane[entries[i]] (whole states, bit for bit)."""
        self._ckpt(self.lib.kda_ckpt_load, "kda_ckpt_load", pool, plane, slots, entries, status, layout_id,
                   stream, flags)

    def kda_prefill_raw(self, desc: PoolDesc, args: PrefillArgs, status, stream, flags=0) -> int:
        return self.lib.kda_prefill(ctypes.byref(desc), ctypes.byref(args), status, flags, stream)

    def kda_prefill_workspace_bytes(self, pool, n: int, total: int) -> int:
        out = ctypes.c_int64(0)
        desc = pool if isinstance(pool, PoolDesc) else pool_desc(pool)
        self._check(self.lib.kda_prefill_workspace_bytes(ctypes.byref(desc), n, total, ctypes.byref(out)),
                    "kda_prefill_workspace_bytes")
        return out.value

    def kda_prefill_chunked(self, pool, init_slot, final_slot, q, k, v, a, b, o, status, workspace=None,
                            **kw) -> None:
        """kda_prefill in two passes (see include/kda.h); ``workspace`` is a CUDA
        tensor of at least kda_prefill_workspace_bytes bytes, made here when None."""
        import torch
        need = self.kda_prefill_workspace_bytes(pool, int(init_slot.shape[0]), int(q.shape[0]))
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        self.kda_prefill(pool, init_slot, final_slot, q, k, v, a, b, o, status,
                         _workspace=(workspace.data_ptr(), workspace.numel() * workspace.element_size()), **kw)

    def kda_prefill_chunked_noalloc(self, pool, init_slot, final_slot, q, k, v, a, b, o, status, **kw) -> None:
        """kda_prefill in two passes on the library's own scratch buffer: nothing is allocated."""
        self.kda_prefill(pool, init_slot, final_slot, q, k, v, a, b, o, status, _noalloc=True, **kw)

    def kda_prefill(self, pool, init_slot, final_slot, q, k, v, a, b, o, status, cu_seqlens=None, max_t=None,
                    reset=None, a_log=None, dt_bias=None, stream=None, flags=0, _workspace=None,
                    _noalloc=False) -> None:
        """Prefill over packed prompts (see kda_prefill_args in include/kda.h)."""
        import torch
        desc = pool_desc(pool)
        hv, kd, vd = desc.hv, desc.k, desc.v
        n = int(init_slot.shape[0])
        total, h_qk = int(q.shape[0]), int(q.shape[1])
        qkv_types = (torch.float32, torch.float16, torch.bfloat16)
        _expect("init_slot", init_slot, (n,), (torch.int32,))
        _expect("final_slot", final_slot, (n,), (torch.int32,))
        _expect("q", q, (total, h_qk, kd), qkv_types)
        _expect("k", k, (total, h_qk, kd), (q.dtype,))
        _expect("v", v, (total, hv, vd), (q.dtype,))
        _expect("a", a, (total, hv, kd), (torch.float32,))
        _expect("b", b, (total, hv), (torch.float32,))
        _expect("o", o, (total, hv, vd), (torch.float32,))
        _expect("status", status, (1,), (torch.int32,))
        if cu_seqlens is not None:
            _expect("cu_seqlens", cu_seqlens, (n + 1,), (torch.int32,))
            if max_t is None:
                raise ValueError("max_t is required with cu_seqlens")
        elif max_t is None:
            max_t = total // n if n else 0
        if reset is not None:
            _expect("reset", reset, (n,), (torch.uint8,))
        if a_log is not None:
            _expect("a_log", a_log, (hv,), (torch.float32,))
        if dt_bias is not None:
            _expect("dt_bias", dt_bias, (hv, kd), (torch.float32,))
        args = PrefillArgs(n, total, int(max_t), h_qk, _dtype_code(q.dtype), 0, _ptr(cu_seqlens), _ptr(init_slot),
                           _ptr(final_slot), _ptr(reset), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(a_log),
                           _ptr(dt_bias), _ptr(o))
        if _noalloc:
            self._check(self.lib.kda_prefill_chunked_noalloc(ctypes.byref(desc), ctypes.byref(args), _ptr(status),
                                                             flags, self._stream(stream)),
                        "kda_prefill_chunked_noalloc")
        elif _workspace is None:
            self._check(self.kda_prefill_raw(desc, args, _ptr(status), self._stream(stream), flags), "kda_prefill")
        else:
            self._check(self.lib.kda_prefill_chunked(ctypes.byref(desc), ctypes.byref(args), _workspace[0],
                                                     _workspace[1], _ptr(status), flags, self._stream(stream)),
                        "kda_prefill_chunked")

