"""GPU parity of the general step (kda_step) against the fp64 oracle.

The general step reads a request's initial state from the accepted column of
its slot table and stores each token's state to that token's column
(state_at(c, slot) of ROCm/ATOM pull request 2945, Changes), over packed
variable-length requests, with padding requests, dropped snapshots, grouped
q/k heads and the learned gate scale.  Tolerances are those of the plain
steps (tests/_harness.py); slot placement is bit-exact.
"""
import numpy as np
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import workloads

import oracle
from _harness import assert_out_match, assert_pool_match, lib_for, pool_np

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]

SD = [torch.float32, torch.float16]


def gpu_general(inp, flags=0):
    d = inp.to("cuda")
    lib = lib_for(inp.pool.dtype)
    total, hv, v = d.v.shape
    o = torch.full((total, hv, v), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_step(d.pool, d.slot_table, d.q, d.k, d.v, d.a, d.b, o, status, cu_seqlens=d.cu_seqlens,
                 max_t=inp.max_t, accepted=d.accepted, reset=d.reset, a_log=d.a_log, dt_bias=d.dt_bias,
                 in_place=inp.in_place, flags=flags)
    torch.cuda.synchronize()
    return d.pool.cpu(), o.cpu(), int(status.item())


def oracle_general(inp):
    P = pool_np(inp.pool)
    o = oracle.step(P, inp.slot_table.numpy(), inp.q, inp.k, inp.v, inp.a, inp.b,
                    cu_seqlens=None if inp.cu_seqlens is None else inp.cu_seqlens.numpy(),
                    accepted=None if inp.accepted is None else inp.accepted.numpy(),
                    reset=None if inp.reset is None else inp.reset.numpy(),
                    a_log=inp.a_log, dt_bias=inp.dt_bias, in_place=inp.in_place, nthreads=8)
    return P, o


def written_slots(inp):
    """The slots a step stores to: token j's column for j < T_r (when kept), or
    the initial slot in place; none for a padding request."""
    table = inp.slot_table.numpy()
    n = table.shape[0]
    c0 = np.zeros(n, np.int64) if inp.accepted is None else inp.accepted.numpy().astype(np.int64) - 1
    lens = inp.meta["lens"]
    out = []
    for r in range(n):
        if table[r, c0[r]] < 0:
            continue
        if inp.in_place:
            out.append(table[r, c0[r]])
        else:
            out.extend(s for s in table[r, :lens[r]] if s >= 0)
    return np.array(out, np.int64)


def check(inp, flags=0):
    gp, o, st = gpu_general(inp, flags)
    ref, o_ref = oracle_general(inp)
    assert st == 0, kda.KdaLibrary(inp.pool.dtype).kda_strerror(st)
    assert_out_match(o, o_ref, inp.pool.dtype, "o")
    assert_pool_match(gp, ref, written_slots(inp), "pool")


@pytest.mark.parametrize("state_dtype", SD)
def test_spec_step_from_accepted_columns(state_dtype):
    """N=8 requests x 8 tokens at the layer shape, initial state at a random accepted column."""
    check(workloads.make_general(n=8, t=8, num_cols=8, state_dtype=state_dtype, seed=40, reset_p=0.2))


@pytest.mark.parametrize("state_dtype", SD)
def test_spec_step_variable_lengths(state_dtype):
    """Packed requests of 5, 0, 13, 1, 8 and 9 tokens (two token chunks past 8), ragged K and V."""
    check(workloads.make_general(n=6, t_lens=[5, 0, 13, 1, 8, 9], num_cols=13, hv=4, k=64, v=48,
                                 num_slots=6 * 13 + 3, state_dtype=state_dtype, seed=41, reset_p=0.3))


@pytest.mark.parametrize("state_dtype", SD)
def test_padding_requests_and_dropped_snapshots(state_dtype):
    inp = workloads.make_general(n=12, t=6, num_cols=7, hv=6, k=128, v=64, num_slots=90,
                                 state_dtype=state_dtype, seed=42, pad_p=0.3, drop_p=0.3)
    assert (inp.slot_table < 0).all(dim=1).any()
    check(inp)


@pytest.mark.parametrize("state_dtype", SD)
@pytest.mark.parametrize("h_qk", [1, 3, 12])
def test_grouped_heads_and_gate_scale(state_dtype, h_qk):
    check(workloads.make_general(n=4, t=5, num_cols=5, hv=12, h_qk=h_qk, num_slots=24,
                                 state_dtype=state_dtype, seed=43 + h_qk, gate_scale=True))


@pytest.mark.parametrize("state_dtype", SD)
@pytest.mark.parametrize("flags", [0, kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE])
def test_in_place_decode_general(state_dtype, flags):
    """Decode at N=64, HV=12, K=V=128 from accepted columns of a 4-column table,
    bf16 q/k/v on 4 q/k heads, learned gate scale, padding and resets."""
    check(workloads.make_general(n=64, num_cols=4, hv=12, h_qk=4, num_slots=256, state_dtype=state_dtype,
                                 qkv_dtype=torch.bfloat16, seed=48, in_place=True, pad_p=0.1, reset_p=0.1,
                                 gate_scale=True), flags)


@pytest.mark.parametrize("state_dtype", SD)
def test_general_step_matches_plain_verify_bits(state_dtype):
    """With one q/k head per value head, no gate scale and column 0 as the
    initial slot, kda_step is kda_spec_verify from that slot: the same bits."""
    n, t = 4, 6
    inp = workloads.make_verify(n=n, t=t, hv=12, k=128, v=128, num_slots=64, state_dtype=state_dtype,
                                seed=49, reset_p=0.25)
    flat = lambda x: x.reshape(n * t, *x.shape[2:])  # noqa: E731
    gen = workloads.GeneralInputs(inp.pool, inp.snap_slot.clone(), flat(inp.q), flat(inp.k), flat(inp.v),
                                  flat(inp.a), flat(inp.b), None, None, inp.reset, None, None, False, t,
                                  dict(lens=[t] * n))
    gp, o, st = gpu_general(gen)
    d = inp.to("cuda")
    init = inp.snap_slot[:, 0].contiguous().to("cuda")
    o2 = torch.empty(n, t, 12, 128, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib_for(state_dtype).kda_spec_verify(d.pool, init, d.snap_slot, d.q, d.k, d.v, d.a, d.b, o2, st2,
                                         reset=d.reset)
    torch.cuda.synchronize()
    assert st == 0 and int(st2.item()) == 0
    assert torch.equal(gp, d.pool.cpu()) and torch.equal(o.reshape(n, t, 12, 128), o2.cpu())


@pytest.mark.parametrize("state_dtype", SD)
def test_bad_accepted_column_and_offsets_set_status(state_dtype):
    """An accepted column outside 1..C, or token offsets past max_t, is
    KDA_ERR_ARG on the device; that request's tiles are skipped, the others run."""
    inp = workloads.make_general(n=4, t_lens=[2, 3, 1, 2], num_cols=3, hv=2, k=32, v=32, num_slots=20,
                                 state_dtype=state_dtype, seed=50)
    inp.accepted[1] = 4  # column 3 of 3
    gp, o, st = gpu_general(inp)
    assert st == kda.KDA_ERR_ARG
    ok = [0, 2, 3]
    ref, o_ref = oracle_general(_without(inp, 1))
    cu = inp.cu_seqlens.long()
    for r in ok:
        sl = slice(int(cu[r]), int(cu[r + 1]))
        assert_out_match(o[sl], o_ref[sl], state_dtype, f"request {r}")
    bad_slots = set(inp.slot_table[1].tolist())
    assert_pool_match(gp, ref, written_slots(_without(inp, 1)), "pool")
    for s in bad_slots:
        assert torch.equal(gp[s], inp.pool[s])
    # offsets: request 2 claims 4 tokens with max_t = 3
    inp2 = workloads.make_general(n=3, t_lens=[1, 2, 3], num_cols=3, hv=2, k=32, v=32, num_slots=12,
                                  state_dtype=state_dtype, seed=51)
    inp2.cu_seqlens = torch.tensor([0, 1, 2, 6], dtype=torch.int32)  # T_2 = 4 > max_t
    inp2.q = torch.cat([inp2.q, inp2.q[:1]]); inp2.k = torch.cat([inp2.k, inp2.k[:1]])
    inp2.v = torch.cat([inp2.v, inp2.v[:1]]); inp2.a = torch.cat([inp2.a, inp2.a[:1]])
    inp2.b = torch.cat([inp2.b, inp2.b[:1]])
    _, _, st2 = gpu_general(inp2)
    assert st2 == kda.KDA_ERR_ARG


def _without(inp, r):
    """The same inputs with request r turned into padding (its row all -1)."""
    table = inp.slot_table.clone()
    table[r] = -1
    acc = inp.accepted.clone()
    acc[r] = 1
    return workloads.GeneralInputs(inp.pool, table, inp.q, inp.k, inp.v, inp.a, inp.b, inp.cu_seqlens, acc,
                                   inp.reset, inp.a_log, inp.dt_bias, inp.in_place, inp.max_t, dict(inp.meta))


# Launches of more than one wave of the default verify shape (3 CTAs per SM;
# 456 CTAs on 152 SMs) run the wide shape on an fp16 pool with 16-bit inputs:
# 4 CTAs per SM, two staging buffers.  N=32 requests x 12 heads x 4 column
# tiles is 1536 CTAs.

@pytest.mark.parametrize("qkv_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("flags", [0, kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE])
def test_serving_scale_step_wide_launch(qkv_dtype, flags):
    """The general step at serving scale, N=32 x 8 tokens on an fp16 pool:
    accepted columns, learned gate scale, resets and padding."""
    check(workloads.make_general(n=32, t=8, num_cols=8, hv=12, num_slots=256, state_dtype=torch.float16,
                                 qkv_dtype=qkv_dtype, seed=52, reset_p=0.1, pad_p=0.05, gate_scale=True),
          flags)


def test_wide_launch_variable_lengths_past_one_chunk():
    """A wide launch (40 requests: 1920 CTAs) of packed requests of 13, 1, 8,
    16, 0 and 9 tokens: two chunks of 8 for some, the two staging buffers
    reused across the chunk boundary, empty requests beside them."""
    lens = [13, 1, 8, 16, 0, 9] * 6 + [13, 16, 9, 5]
    check(workloads.make_general(n=40, t_lens=lens, num_cols=16, hv=12, num_slots=40 * 16 + 8,
                                 state_dtype=torch.float16, qkv_dtype=torch.bfloat16, seed=54, reset_p=0.1,
                                 gate_scale=True))


@pytest.mark.parametrize("qkv_dtype", [torch.bfloat16, torch.float16])
def test_wide_launch_equals_one_wave_launches_bits(qkv_dtype):
    """Requests are independent, so one launch of 32 requests (the wide shape)
    must give the same bits as four launches of 8 (the default shape)."""
    n, t, part = 32, 8, 8
    inp = workloads.make_verify(n=n, t=t, hv=12, k=128, v=128, num_slots=n * (t + 1), state_dtype=torch.float16,
                                qkv_dtype=qkv_dtype, seed=53, reset_p=0.2)
    lib = lib_for(torch.float16)
    d = inp.to("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool_wide = d.pool.clone()
    o_wide = torch.empty(n, t, 12, 128, device="cuda")
    lib.kda_spec_verify(pool_wide, d.init_slot, d.snap_slot, d.q, d.k, d.v, d.a, d.b, o_wide, st, reset=d.reset)
    pool_parts = d.pool.clone()
    o_parts = torch.empty(n, t, 12, 128, device="cuda")
    for r0 in range(0, n, part):
        sl = slice(r0, r0 + part)
        o_sl = torch.empty(part, t, 12, 128, device="cuda")
        lib.kda_spec_verify(pool_parts, d.init_slot[sl].contiguous(), d.snap_slot[sl].contiguous(),
                            d.q[sl].contiguous(), d.k[sl].contiguous(), d.v[sl].contiguous(),
                            d.a[sl].contiguous(), d.b[sl].contiguous(), o_sl, st, reset=d.reset[sl].contiguous())
        o_parts[sl] = o_sl
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(pool_wide, pool_parts)
    assert torch.equal(o_wide, o_parts)
