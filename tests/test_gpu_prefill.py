"""GPU prefill (kda_prefill) against the fp64 oracle: outputs of every token,
the final state stored once (fp32 pool max-abs 1e-5, fp16 within one ulp of
the oracle's single rounding), nothing else written."""
import numpy as np
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import workloads

import oracle
from _harness import assert_out_match, assert_pool_match, lib_for, pool_np

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]
SD = [torch.float32, torch.float16]


def run(inp, flags=0, chunked=False):
    d = inp.to("cuda")
    total, hv, v = d.v.shape
    o = torch.full((total, hv, v), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = lib_for(inp.pool.dtype)
    call = lib.kda_prefill_chunked if chunked else lib.kda_prefill
    call(d.pool, d.init_slot, d.final_slot, d.q, d.k, d.v, d.a, d.b, o, status, cu_seqlens=d.cu_seqlens,
         max_t=inp.max_t, reset=d.reset, a_log=d.a_log, dt_bias=d.dt_bias, flags=flags)
    torch.cuda.synchronize()
    P = pool_np(inp.pool)
    o_ref = oracle.prefill(P, inp.init_slot.numpy(), inp.final_slot.numpy(), inp.q, inp.k, inp.v, inp.a, inp.b,
                           cu_seqlens=inp.cu_seqlens.numpy(), reset=inp.reset.numpy(), a_log=inp.a_log,
                           dt_bias=inp.dt_bias, nthreads=8)
    return d.pool.cpu(), o.cpu(), int(status.item()), P, o_ref


def written(inp):
    """Final slots a call writes: every non-padding request with a final slot,
    an empty one included (it stores its initial state there)."""
    return [int(f) for f, i in zip(inp.final_slot, inp.init_slot) if f >= 0 and i >= 0]


CHUNKED = [False, True]


@pytest.mark.parametrize("chunked", CHUNKED)
@pytest.mark.parametrize("state_dtype", SD)
def test_prefill_layer_shape(state_dtype, chunked):
    """Prompts of 200 and 37 tokens (many chunks, ragged last chunk), HV=12, K=V=128, bf16 q/k/v."""
    inp = workloads.make_prefill(lens=(200, 37), state_dtype=state_dtype, seed=90)
    gp, o, st, P, o_ref = run(inp, chunked=chunked)
    assert st == 0
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gp, P, written(inp), "pool")


@pytest.mark.parametrize("chunked", CHUNKED)
@pytest.mark.parametrize("state_dtype", SD)
def test_prefill_varlen_grouped_heads_gate_scale_padding(state_dtype, chunked):
    inp = workloads.make_prefill(lens=(13, 0, 64, 1, 9), h_qk=4, state_dtype=state_dtype, num_slots=16,
                                 qkv_dtype=torch.float32, seed=91, gate_scale=True, pad_p=0.3)
    gp, o, st, P, o_ref = run(inp, flags=kda.KDA_LAUNCH_PDL, chunked=chunked)
    assert st == 0
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gp, P, written(inp), "pool")


@pytest.mark.parametrize("chunked", CHUNKED)
def test_prefill_long_prompt_sampled(chunked):
    """One 2048-token prompt on an fp16 pool: final state and a sample of outputs."""
    inp = workloads.make_prefill(lens=(2048,), state_dtype=torch.float16, num_slots=4, seed=92, reset_p=1.0)
    gp, o, st, P, o_ref = run(inp, chunked=chunked)
    assert st == 0
    idx = np.r_[0:16, 1000:1016, 2032:2048]
    assert_out_match(o[idx], o_ref[idx], torch.float16, "o")
    assert_pool_match(gp, P, written(inp), "pool")


@pytest.mark.parametrize("state_dtype", SD)
def test_chunked_prefill_ragged_shapes(state_dtype):
    """K = 48, V = 80 (a partial 32-column tile), prompts shorter and longer than a chunk."""
    inp = workloads.make_prefill(lens=(5, 16, 17, 40), hv=3, k=48, v=80, num_slots=12, state_dtype=state_dtype,
                                 qkv_dtype=torch.float32, seed=93)
    gp, o, st, P, o_ref = run(inp, chunked=True)
    assert st == 0
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gp, P, written(inp), "pool")


def test_chunked_prefill_workspace_too_small_is_refused():
    inp = workloads.make_prefill(lens=(20,), hv=2, k=16, v=16, num_slots=4, state_dtype=torch.float32,
                                 qkv_dtype=torch.float32, seed=94)
    d = inp.to("cuda")
    lib = lib_for(torch.float32)
    o = torch.empty(20, 2, 16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    need = lib.kda_prefill_workspace_bytes(d.pool, 1, 20)
    # one 56,576-byte block per (16-token chunk slot, head): W', Q' and Ke as three
    # bf16 parts of [16][136], c [128] fp32, U and O_intra [16][132] fp32
    assert need == (20 // 16 + 1) * 2 * 56576
    with pytest.raises(kda.KdaError) as e:
        lib.kda_prefill_chunked(d.pool, d.init_slot, d.final_slot, d.q, d.k, d.v, d.a, d.b, o, status,
                                workspace=torch.empty(need - 256, dtype=torch.uint8, device="cuda"),
                                cu_seqlens=d.cu_seqlens, max_t=20, reset=d.reset)
    assert e.value.code == kda.KDA_ERR_ARG


@pytest.mark.parametrize("chunked", CHUNKED)
@pytest.mark.parametrize("state_dtype", SD)
def test_prefill_empty_prompts_store_their_initial_state(state_dtype, chunked):
    """Requests with no tokens beside ones with tokens, init and final slots
    distinct, with and without reset: an empty request's final slot gets its
    initial state bit for bit (zeros on a reset), as the oracle says."""
    inp = workloads.make_prefill(lens=(0, 7, 0, 0, 20), hv=12, k=128, v=128, num_slots=12, state_dtype=state_dtype,
                                 qkv_dtype=torch.bfloat16, seed=95, reset_p=0.0, same_slot_p=0.0)
    inp.reset[:] = torch.tensor([0, 0, 1, 0, 1], dtype=torch.uint8)
    gp, o, st, P, o_ref = run(inp, chunked=chunked)
    assert st == 0
    before = pool_np(inp.pool)
    for r, lr in enumerate(inp.meta["lens"]):
        if lr == 0:
            f, i = int(inp.final_slot[r]), int(inp.init_slot[r])
            expect = np.zeros_like(before[i]) if int(inp.reset[r]) else before[i]
            assert pool_np(gp)[f].tobytes() == expect.tobytes()
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gp, P, written(inp), "pool")


@pytest.mark.parametrize("chunked", CHUNKED)
@pytest.mark.parametrize("state_dtype", SD)
def test_prefill_call_without_tokens(state_dtype, chunked):
    """total == 0 (every prompt empty, max_t 0, NULL token buffers): the call
    still moves each request's initial state to its final slot."""
    inp = workloads.make_prefill(lens=(0, 0, 0), hv=3, k=48, v=80, num_slots=8, state_dtype=state_dtype,
                                 qkv_dtype=torch.float32, seed=96, reset_p=0.5, same_slot_p=0.0, pad_p=0.3)
    gp, o, st, P, o_ref = run(inp, chunked=chunked)
    assert st == 0 and o.shape[0] == 0
    assert_pool_match(gp, P, written(inp), "pool")


@pytest.mark.parametrize("n_prompts", [8, 16])
def test_chunked_prefill_wide_scan_tilings(n_prompts):
    """8 prompts (96 heads: four 16-column blocks per scan CTA) and 16 prompts
    (192 heads: eight blocks per CTA), ragged lengths, fp16 pool: the scan
    shapes a batch takes, against the oracle."""
    lens = tuple(17 + 9 * i for i in range(n_prompts))
    inp = workloads.make_prefill(lens=lens, state_dtype=torch.float16, num_slots=2 * n_prompts + 2, seed=97)
    gp, o, st, P, o_ref = run(inp, chunked=True)
    assert st == 0
    assert_out_match(o, o_ref, torch.float16, "o")
    assert_pool_match(gp, P, written(inp), "pool")
