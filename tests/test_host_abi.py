"""Host-side tests of the C ABI (no GPU): the libraries build, load, export
every symbol include/kda.h declares, and refuse bad pools on the host.

kda_pool_check and kda_state_bytes touch no device memory, so they run here
on fake (never dereferenced) base addresses.  The refusal rules are those of
ROCm/ATOM pull request 2945 (Changes, Testing): layers must agree on the
dtype, a pool of the other dtype is refused, and only fp32/fp16 are accepted.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import PoolDesc

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kda.h")
FAKE_BASE = 0x7F0000000000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def libs(built_libs):
    return {torch.float32: kda.KdaLibrary(torch.float32), torch.float16: kda.KdaLibrary(torch.float16)}


def desc(dtype=kda.KDA_F32, hv=12, k=128, v=128, num_slots=256, slot_stride=None, base=FAKE_BASE):
    return PoolDesc(base, dtype, hv, k, v, num_slots, hv * k * v if slot_stride is None else slot_stride)


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|uint32_t|const char\*)\s+(kda_\w+)\s*\(", text, re.M)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(kda.EXPORTED_SYMBOLS)


@pytest.mark.parametrize("state16", [False, True])
def test_library_exports_every_declared_symbol(built_libs, state16):
    path = kda.lib_path(state16)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, re.M))
    for sym in declared_functions():
        assert sym in exported, f"{sym} missing from {os.path.basename(path)}"
    lib = ctypes.CDLL(path)
    for sym in declared_functions():
        assert getattr(lib, sym) is not None


def test_build_dtype(libs):
    assert libs[torch.float32].kda_build_state_dtype() == kda.KDA_F32
    assert libs[torch.float16].kda_build_state_dtype() == kda.KDA_F16


@pytest.mark.parametrize("sd", [torch.float32, torch.float16])
def test_pool_check_accepts_agreeing_layers(libs, sd):
    code = kda.KDA_F32 if sd == torch.float32 else kda.KDA_F16
    pools = [desc(code, base=FAKE_BASE + i * (1 << 32)) for i in range(69)]
    assert libs[sd].kda_pool_check_raw(pools) == kda.KDA_OK


def test_pool_check_refusals(libs):
    L32, L16 = libs[torch.float32], libs[torch.float16]
    # a pool of the other dtype
    assert L32.kda_pool_check_raw([desc(kda.KDA_F16)]) == kda.KDA_ERR_DTYPE_MISMATCH
    assert L16.kda_pool_check_raw([desc(kda.KDA_F32)]) == kda.KDA_ERR_DTYPE_MISMATCH
    # bf16 refused by both builds
    for L in (L32, L16):
        assert L.kda_pool_check_raw([desc(kda.KDA_BF16)]) == kda.KDA_ERR_DTYPE_UNSUPPORTED
        assert L.kda_pool_check_raw([desc(7)]) == kda.KDA_ERR_DTYPE_UNSUPPORTED
    # layers that disagree on dtype or shape
    assert L32.kda_pool_check_raw([desc(), desc(kda.KDA_F16)]) == kda.KDA_ERR_LAYERS_DISAGREE
    assert L16.kda_pool_check_raw([desc(kda.KDA_F16), desc(kda.KDA_F32)]) == kda.KDA_ERR_LAYERS_DISAGREE
    assert L32.kda_pool_check_raw([desc(), desc(hv=8)]) == kda.KDA_ERR_LAYERS_DISAGREE
    assert L32.kda_pool_check_raw([desc(), desc(k=64)]) == kda.KDA_ERR_LAYERS_DISAGREE
    # shapes
    for bad in (dict(k=8), dict(k=136), dict(v=24), dict(v=0), dict(hv=0), dict(num_slots=0),
                dict(slot_stride=12 * 128 * 128 - 4)):
        assert L32.kda_pool_check_raw([desc(**bad)]) == kda.KDA_ERR_SHAPE, bad
    # alignment
    assert L32.kda_pool_check_raw([desc(base=FAKE_BASE + 4)]) == kda.KDA_ERR_ALIGN
    assert L16.kda_pool_check_raw([desc(kda.KDA_F16, slot_stride=12 * 128 * 128 + 2)]) == kda.KDA_ERR_ALIGN
    assert L16.kda_pool_check_raw([desc(kda.KDA_F16, slot_stride=12 * 128 * 128 + 8)]) == kda.KDA_OK
    # nulls and counts
    assert L32.kda_pool_check_raw([desc(base=0)]) == kda.KDA_ERR_NULL
    assert L32.lib.kda_pool_check(None, 1) == kda.KDA_ERR_NULL
    arr = (PoolDesc * 1)(desc())
    assert L32.lib.kda_pool_check(arr, 0) == kda.KDA_ERR_ARG


def test_state_bytes(libs):
    L = libs[torch.float32]
    assert L.kda_state_bytes(desc()) == 12 * 128 * 128 * 4
    assert L.kda_state_bytes(desc(kda.KDA_F16)) == 12 * 128 * 128 * 2
    with pytest.raises(kda.KdaError) as e:
        L.kda_state_bytes(desc(kda.KDA_BF16))
    assert e.value.code == kda.KDA_ERR_DTYPE_UNSUPPORTED


def test_step_refusals_before_any_launch(libs):
    """Argument errors come back synchronously from the host checks; the
    pointers below are never dereferenced because every call is refused."""
    L32 = libs[torch.float32]
    P = 0x7F0000100000
    args = lambda d, **kw: dict(dict(desc=d, slot_ids=P, reset=None, n=4, q=P, k=P, v=P,  # noqa: E731
                                     qkv_dtype=kda.KDA_BF16, a=P, b=P, o=P, status=P, stream=None), **kw)
    call = lambda **kw: L32.kda_decode_step_raw(**kw)  # noqa: E731
    assert call(**args(desc(kda.KDA_F16))) == kda.KDA_ERR_DTYPE_MISMATCH
    assert call(**args(desc(kda.KDA_BF16))) == kda.KDA_ERR_DTYPE_UNSUPPORTED
    assert call(**args(desc(), qkv_dtype=9)) == kda.KDA_ERR_DTYPE_UNSUPPORTED
    assert call(**args(desc(), n=-1)) == kda.KDA_ERR_ARG
    assert call(**args(desc(), q=None)) == kda.KDA_ERR_NULL
    assert call(**args(desc(), status=None)) == kda.KDA_ERR_NULL
    assert call(**args(desc(), a=P + 2)) == kda.KDA_ERR_ALIGN
    assert call(**args(desc(), a=P + 4)) == kda.KDA_ERR_ALIGN
    assert call(**args(desc(), v=P + 8)) == kda.KDA_ERR_ALIGN
    assert call(**args(desc(), b=P + 2)) == kda.KDA_ERR_ALIGN
    assert call(**args(desc(), q=P + 1)) == kda.KDA_ERR_ALIGN
    assert call(**args(desc(k=100))) == kda.KDA_ERR_SHAPE
    # n == 0 is a no-op that succeeds without touching the GPU
    assert call(**args(desc(), n=0)) == kda.KDA_OK
    # verify: snapshot ids are required
    rc = L32.lib.kda_spec_verify(ctypes.byref(desc()), P, None, None, 4, 8, P, P, P,
                                 kda.KDA_F32, P, P, P, P, 0, None)
    assert rc == kda.KDA_ERR_NULL
    rc = L32.lib.kda_spec_verify(ctypes.byref(desc()), P, P, None, 4, 0, P, P, P,
                                 kda.KDA_F32, P, P, P, P, 0, None)
    assert rc == kda.KDA_OK
    # unknown launch flags
    assert call(**args(desc(), flags=4)) == kda.KDA_ERR_ARG
    assert call(**args(desc(), n=0, flags=kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE)) == kda.KDA_OK
    assert call(**args(desc(), n=0, flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE)) == kda.KDA_OK  # the test hook


def test_general_step_refusals_before_any_launch(libs):
    """kda_step's host checks (include/kda.h, kda_step_args): every call below
    is refused before a launch, so the fake pointers are never dereferenced."""
    L32 = libs[torch.float32]
    P = 0x7F0000100000

    def args(**kw):
        f = dict(n=4, total=32, max_t=8, h_qk=12, num_cols=8, in_place=0, qkv_dtype=kda.KDA_F32,
                 reserved=0, cu_seqlens=None, slot_table=P, accepted=None, reset=None, q=P, k=P, v=P,
                 a=P, b=P, a_log=None, dt_bias=None, o=P)
        f.update(kw)
        return kda.StepArgs(**f)

    call = lambda a, d=None, status=P, flags=0: L32.kda_step_raw(d or desc(), a, status, None, flags)  # noqa
    assert L32.lib.kda_step(ctypes.byref(desc()), None, P, 0, None) == kda.KDA_ERR_NULL
    assert call(args(), d=desc(kda.KDA_F16)) == kda.KDA_ERR_DTYPE_MISMATCH
    assert call(args(qkv_dtype=7)) == kda.KDA_ERR_DTYPE_UNSUPPORTED
    assert call(args(h_qk=5)) == kda.KDA_ERR_SHAPE          # 12 % 5 != 0
    assert call(args(h_qk=0)) == kda.KDA_ERR_SHAPE
    assert call(args(num_cols=0)) == kda.KDA_ERR_SHAPE
    assert call(args(max_t=9, total=36)) == kda.KDA_ERR_SHAPE  # more tokens than columns
    assert call(args(total=31)) == kda.KDA_ERR_SHAPE         # not n * max_t without offsets
    assert call(args(in_place=1, total=4, max_t=1, cu_seqlens=P)) == kda.KDA_ERR_SHAPE
    assert call(args(in_place=1, total=5, max_t=1)) == kda.KDA_ERR_SHAPE
    assert call(args(reserved=1)) == kda.KDA_ERR_ARG
    assert call(args(n=-1)) == kda.KDA_ERR_ARG
    assert call(args(), flags=8) == kda.KDA_ERR_ARG
    assert call(args(slot_table=None)) == kda.KDA_ERR_NULL
    assert call(args(), status=None) == kda.KDA_ERR_NULL
    assert call(args(a=P + 4)) == kda.KDA_ERR_ALIGN
    assert call(args(cu_seqlens=P + 2, total=20)) == kda.KDA_ERR_ALIGN
    assert call(args(dt_bias=P + 1)) == kda.KDA_ERR_ALIGN
    # nothing to do: succeeds without touching the GPU
    assert call(args(n=0, total=0)) == kda.KDA_OK
    assert call(args(n=0, total=0), flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE) == kda.KDA_OK  # the test hook
    assert call(args(total=0, cu_seqlens=P)) == kda.KDA_OK


def test_conv_step_refusals_before_any_launch(libs):
    """kda_conv_step's host checks (include/kda.h, kda_conv_args)."""
    L = libs[torch.float16]  # the conv window's dtype is independent of the pool build
    P = 0x7F0000100000

    def win(**kw):
        f = dict(base=P, dtype=kda.KDA_BF16, channels=4608, state_len=7, reserved=0, num_slots=64,
                 slot_stride=7 * 4608)
        f.update(kw)
        return kda.ConvWindowDesc(**f)

    def args(**kw):
        f = dict(n=8, total=40, max_t=5, kernel_width=4, activation=1, reserved=0, cu_seqlens=None,
                 conv_slot=P, accepted=None, reset=None, x=P, weight=P, bias=None, y=P)
        f.update(kw)
        return kda.ConvArgs(**f)

    call = lambda w, a, status=P, flags=0: L.kda_conv_step_raw(w, a, status, None, flags)  # noqa: E731
    assert L.lib.kda_conv_step(None, ctypes.byref(args()), P, 0, None) == kda.KDA_ERR_NULL
    assert call(win(dtype=7), args()) == kda.KDA_ERR_DTYPE_UNSUPPORTED
    assert call(win(channels=0), args()) == kda.KDA_ERR_SHAPE
    assert call(win(), args(kernel_width=9)) == kda.KDA_ERR_SHAPE
    assert call(win(state_len=2), args()) == kda.KDA_ERR_SHAPE      # fewer than kernel - 1 entries
    assert call(win(state_len=33, slot_stride=33 * 4608), args()) == kda.KDA_ERR_SHAPE
    assert call(win(slot_stride=7 * 4608 - 1), args()) == kda.KDA_ERR_SHAPE
    assert call(win(), args(total=39)) == kda.KDA_ERR_SHAPE
    assert call(win(), args(activation=2)) == kda.KDA_ERR_ARG
    assert call(win(reserved=1), args()) == kda.KDA_ERR_ARG
    assert call(win(), args(), flags=16) == kda.KDA_ERR_ARG
    assert call(win(), args(), flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE) == kda.KDA_ERR_ARG  # not a conv option
    assert call(win(), args(conv_slot=None)) == kda.KDA_ERR_NULL
    assert call(win(), args(x=P + 1)) == kda.KDA_ERR_ALIGN
    assert call(win(), args(weight=P + 2)) == kda.KDA_ERR_ALIGN
    assert call(win(), args(n=0, total=0)) == kda.KDA_OK


def test_decode_conv_step_refusals_before_any_launch(libs):
    """kda_decode_conv_step's host checks (include/kda.h, kda_decode_conv_args):
    the pool's, the window's, and the channel count tying the two together."""
    L = libs[torch.float32]
    P = 0x7F0000100000
    C = 2 * 12 * 128 + 12 * 128  # q | k | v channels of hv = h_qk = 12, K = V = 128

    def win(**kw):
        f = dict(base=P, dtype=kda.KDA_BF16, channels=C, state_len=3, reserved=0, num_slots=64, slot_stride=3 * C)
        f.update(kw)
        return kda.ConvWindowDesc(**f)

    def args(**kw):
        f = dict(n=8, h_qk=12, kernel_width=4, activation=1, slot_ids=P, conv_slot=P, reset=None, x=P, weight=P,
                 bias=None, a=P, b=P, o=P, y=None, counters=P)
        f.update(kw)
        return kda.DecodeConvArgs(**f)

    call = lambda w, a, d=None, status=P, flags=0: L.kda_decode_conv_step_raw(  # noqa: E731
        d or desc(), w, a, status, None, flags)
    assert L.lib.kda_decode_conv_step(ctypes.byref(desc()), None, ctypes.byref(args()), P, 0, None) == kda.KDA_ERR_NULL
    assert call(win(), args(), d=desc(kda.KDA_F16)) == kda.KDA_ERR_DTYPE_MISMATCH  # the fp32 build
    assert call(win(dtype=7), args()) == kda.KDA_ERR_DTYPE_UNSUPPORTED
    assert call(win(channels=C - 1), args()) == kda.KDA_ERR_SHAPE                   # not q | k | v
    assert call(win(channels=2 * 4 * 128 + 12 * 128), args()) == kda.KDA_ERR_SHAPE  # h_qk = 4 laid out, 12 given
    assert call(win(channels=2 * 4 * 128 + 12 * 128), args(h_qk=4, n=0)) == kda.KDA_OK  # grouped: accepted
    assert call(win(), args(h_qk=5)) == kda.KDA_ERR_SHAPE                          # does not divide hv
    assert call(win(), args(kernel_width=5)) == kda.KDA_ERR_SHAPE                  # widths 1 .. 4
    assert call(win(state_len=2), args()) == kda.KDA_ERR_SHAPE                      # fewer than kernel - 1
    assert call(win(state_len=5, slot_stride=5 * C), args()) == kda.KDA_ERR_SHAPE   # more than one step keeps
    assert call(win(slot_stride=3 * C - 1), args()) == kda.KDA_ERR_SHAPE
    assert call(win(), args(activation=2)) == kda.KDA_ERR_ARG
    assert call(win(reserved=1), args()) == kda.KDA_ERR_ARG
    assert call(win(), args(n=-1)) == kda.KDA_ERR_ARG
    assert call(win(), args(), flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE) == kda.KDA_ERR_ARG
    for name in ("slot_ids", "conv_slot", "x", "weight", "a", "b", "o", "counters"):
        assert call(win(), args(**{name: None})) == kda.KDA_ERR_NULL, name
    assert call(win(), args(a=P + 4)) == kda.KDA_ERR_ALIGN    # a moves by 16-byte bulk copy
    assert call(win(), args(x=P + 1)) == kda.KDA_ERR_ALIGN
    assert call(win(), args(y=P + 1)) == kda.KDA_ERR_ALIGN
    assert call(win(), args(counters=P + 2)) == kda.KDA_ERR_ALIGN
    assert call(win(), args(a_log=P + 2)) == kda.KDA_ERR_ALIGN
    assert call(win(), args(dt_bias=P + 1)) == kda.KDA_ERR_ALIGN
    assert call(win(), args(n=0)) == kda.KDA_OK               # nothing to do: no launch


def test_step_conv_refusals_before_any_launch(libs):
    """kda_step_conv's host checks (include/kda.h, kda_step_conv_args): those of
    kda_step, the window's, and the fused form's own (speculative, at most 8
    tokens a request, q/k/v left to the convolution)."""
    L = libs[torch.float16]
    P = 0x7F0000100000
    C = 2 * 12 * 128 + 12 * 128

    def win(**kw):
        f = dict(base=P, dtype=kda.KDA_BF16, channels=C, state_len=7, reserved=0, num_slots=64, slot_stride=7 * C)
        f.update(kw)
        return kda.ConvWindowDesc(**f)

    def step(**kw):
        f = dict(n=8, total=64, max_t=8, h_qk=12, num_cols=8, in_place=0, qkv_dtype=kda.KDA_BF16, reserved=0,
                 cu_seqlens=None, slot_table=P, accepted=None, reset=None, q=None, k=None, v=None, a=P, b=P,
                 a_log=None, dt_bias=None, o=P)
        f.update(kw)
        return kda.StepArgs(**f)

    def conv(**kw):
        f = dict(kernel_width=4, activation=1, conv_slot=P, x=P, weight=P, bias=None, y=None, counters=P)
        f.update(kw)
        return kda.StepConvArgs(**f)

    def call(st=None, w=None, cv=None, d=None, flags=0):
        return L.kda_step_conv_raw(d or desc(kda.KDA_F16), st or step(), w or win(), cv or conv(), P, None, flags)

    assert L.lib.kda_step_conv(ctypes.byref(desc(kda.KDA_F16)), None, ctypes.byref(win()), ctypes.byref(conv()),
                               P, 0, None) == kda.KDA_ERR_NULL
    assert call(d=desc(kda.KDA_F32)) == kda.KDA_ERR_DTYPE_MISMATCH
    assert call(w=win(dtype=7)) == kda.KDA_ERR_DTYPE_UNSUPPORTED
    assert call(st=step(in_place=1)) == kda.KDA_ERR_ARG                      # the decode form is elsewhere
    assert call(st=step(q=P)) == kda.KDA_ERR_ARG                             # the convolution makes q/k/v
    assert call(st=step(qkv_dtype=kda.KDA_F16)) == kda.KDA_ERR_ARG           # not the window's dtype
    assert call(cv=conv(activation=2)) == kda.KDA_ERR_ARG
    assert call(flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE) == kda.KDA_ERR_ARG
    assert call(st=step(max_t=9, num_cols=9, total=72)) == kda.KDA_ERR_SHAPE  # one chunk of 8 at most
    assert call(w=win(channels=C - 1)) == kda.KDA_ERR_SHAPE
    assert call(st=step(h_qk=5)) == kda.KDA_ERR_SHAPE
    assert call(st=step(total=63)) == kda.KDA_ERR_SHAPE
    assert call(cv=conv(kernel_width=5)) == kda.KDA_ERR_SHAPE
    assert call(w=win(state_len=2)) == kda.KDA_ERR_SHAPE
    assert call(w=win(state_len=33, slot_stride=33 * C)) == kda.KDA_ERR_SHAPE
    assert call(w=win(slot_stride=7 * C - 1)) == kda.KDA_ERR_SHAPE
    for name in ("conv_slot", "x", "weight", "counters"):
        assert call(cv=conv(**{name: None})) == kda.KDA_ERR_NULL, name
    assert call(st=step(slot_table=None)) == kda.KDA_ERR_NULL
    assert call(cv=conv(x=P + 1)) == kda.KDA_ERR_ALIGN
    assert call(cv=conv(counters=P + 2)) == kda.KDA_ERR_ALIGN
    assert call(st=step(a=P + 2)) == kda.KDA_ERR_ALIGN
    assert call(st=step(n=0, total=0)) == kda.KDA_OK  # nothing to do: no launch


def test_layout_id_names_dtype_and_shape(libs):
    """Pull request 2130, What: the checkpoint layout id names the dtype, so an
    fp16 build cannot read an fp32 build's checkpoint images."""
    L = libs[torch.float32]
    base = L.kda_layout_id(desc())
    assert base != 0 and L.kda_layout_id(desc()) == base
    others = {L.kda_layout_id(desc(kda.KDA_F16)), L.kda_layout_id(desc(hv=8)), L.kda_layout_id(desc(k=64)),
              L.kda_layout_id(desc(v=64))}
    assert base not in others and len(others) == 4
    assert L.kda_layout_id(desc(num_slots=9, slot_stride=12 * 128 * 128 + 64)) == base  # slots do not matter
    assert L.lib.kda_layout_id(None) == 0


def test_ckpt_refusals_before_any_launch(libs):
    L32, L16 = libs[torch.float32], libs[torch.float16]
    P = 0x7F0000100000
    d32, d16 = desc(), desc(kda.KDA_F16)
    plane = lambda lid, **kw: kda.CkptPlaneDesc(**{**dict(base=P, layout_id=lid, reserved=0, num_entries=8,  # noqa
                                                         entry_stride=12 * 128 * 128), **kw})
    lid32, lid16 = L32.kda_layout_id(d32), L16.kda_layout_id(d16)
    call = lambda L, d, pl, n=4, slots=P, status=P: L.lib.kda_ckpt_flush(  # noqa: E731
        ctypes.byref(d), ctypes.byref(pl), slots, P, n, status, 0, None)
    assert call(L32, d32, plane(lid16)) == kda.KDA_ERR_LAYOUT     # an fp16 image in the fp32 build
    assert call(L16, d16, plane(lid32)) == kda.KDA_ERR_LAYOUT
    assert call(L16, d32, plane(lid32)) == kda.KDA_ERR_DTYPE_MISMATCH
    assert call(L32, d32, plane(lid32, entry_stride=100)) == kda.KDA_ERR_SHAPE
    assert call(L32, d32, plane(lid32, reserved=1)) == kda.KDA_ERR_ARG
    assert call(L32, d32, plane(lid32), n=-1) == kda.KDA_ERR_ARG
    assert call(L32, d32, plane(lid32), slots=None) == kda.KDA_ERR_NULL
    assert call(L32, d32, plane(lid32, base=P + 8)) == kda.KDA_ERR_ALIGN
    assert call(L32, d32, plane(lid32), n=0) == kda.KDA_OK
    assert L32.lib.kda_ckpt_load(ctypes.byref(d32), None, P, P, 1, P, 0, None) == kda.KDA_ERR_NULL


def test_prefill_refusals_before_any_launch(libs):
    L32 = libs[torch.float32]
    P = 0x7F0000100000

    def args(**kw):
        f = dict(n=2, total=64, max_t=32, h_qk=12, qkv_dtype=kda.KDA_BF16, reserved=0, cu_seqlens=None,
                 init_slot=P, final_slot=P, reset=None, q=P, k=P, v=P, a=P, b=P, a_log=None, dt_bias=None, o=P)
        f.update(kw)
        return kda.PrefillArgs(**f)

    call = lambda a, d=None, flags=0: L32.kda_prefill_raw(d or desc(), a, P, None, flags)  # noqa: E731
    assert L32.lib.kda_prefill(ctypes.byref(desc()), None, P, 0, None) == kda.KDA_ERR_NULL
    assert call(args(), d=desc(kda.KDA_F16)) == kda.KDA_ERR_DTYPE_MISMATCH
    assert call(args(h_qk=7)) == kda.KDA_ERR_SHAPE
    assert call(args(total=63)) == kda.KDA_ERR_SHAPE
    assert call(args(reserved=2)) == kda.KDA_ERR_ARG
    assert call(args(final_slot=None)) == kda.KDA_ERR_NULL
    assert call(args(k=P + 8)) == kda.KDA_ERR_ALIGN
    assert call(args(n=0, total=0)) == kda.KDA_OK
    assert call(args(), flags=kda.KDA_LAUNCH_TEST_WITHHOLD_STATE) == kda.KDA_ERR_ARG  # not a prefill option


def test_strerror_covers_every_code(libs):
    L = libs[torch.float32]
    msgs = {c: L.kda_strerror(c) for c in range(12)}
    assert msgs[0] == "ok"
    assert len(set(msgs.values())) == 12
    assert L.kda_strerror(99) == "unknown kda status code"


def test_binding_rejects_cpu_and_misshapen_tensors(libs):
    L = libs[torch.float32]
    pool = torch.zeros(4, 2, 16, 16)
    z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt)  # noqa: E731
    with pytest.raises(ValueError):  # CPU tensors never reach the library
        L.kda_decode_step(pool, z(2, dt=torch.int32), z(2, 2, 16), z(2, 2, 16), z(2, 2, 16),
                          z(2, 2, 16), z(2, 2), z(2, 2, 16), z(1, dt=torch.int32))
    with pytest.raises(ValueError):  # wrong shape
        L.kda_decode_step(pool, z(2, dt=torch.int32), z(2, 2, 8), z(2, 2, 16), z(2, 2, 16),
                          z(2, 2, 16), z(2, 2), z(2, 2, 16), z(1, dt=torch.int32))
    with pytest.raises(ValueError):  # pool whose head part is not dense
        kda.pool_desc(torch.zeros(4, 2, 16, 32)[..., :16])


def test_library_missing_fails_loudly(monkeypatch, tmp_path):
    import kda_linear_attention_gated_gb300 as pkg
    monkeypatch.setattr(pkg, "lib_path", lambda s: str(tmp_path / "nope.so"))
    monkeypatch.setattr(pkg, "_libs", {})
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        pkg.KdaLibrary(torch.float32)


def test_source_hash_ignores_comments_and_layout_but_not_code(tmp_path):
    """The profile summaries' staleness check (bench.py): comments and
    whitespace do not change the hash, string literals and preprocessor line
    breaks are kept, and any code change does."""
    import bench
    src = 'int a = 1; // note\n/* two\n lines */ const char* s = "x // y";\n#define X 1 /* t */\n'
    assert bench.code_text(src) == 'int a = 1;\nconst char* s = "x // y";\n#define X 1'
    f = tmp_path / "k.cu"
    f.write_text(src)
    h0 = bench.source_hash([str(f)])
    f.write_text("  // a new comment\n\n" + src.replace("// note", "// edited   note").replace("int a", "int   a"))
    assert bench.source_hash([str(f)]) == h0  # comments, blank lines and runs of spaces
    f.write_text(src.replace("int a = 1;", "int a = 2;"))
    assert bench.source_hash([str(f)]) != h0  # code
