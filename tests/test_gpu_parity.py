"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle on
the same seeded inputs.

Tolerances (the method's statement of the target): fp32 pool -- states and
outputs within max-abs 1e-5; fp16 pool -- stored states within 1 fp16 ulp of
the oracle's round-to-nearest-even value (the GPU rounds from fp32, the oracle
from fp64, so a value near a rounding midpoint may land one step apart; in the
bottom binades, |S| < 2^-13, where an fp16 step of 2^-24 is below the fp32
carry's own rounding error, two steps) and outputs within 2e-3 relative.  Slot placement is checked bit-exact: every slot
the call must not write is compared byte for byte.
"""
import numpy as np
import pytest
import torch

from kda_linear_attention_gated_gb300 import workloads
import kda_linear_attention_gated_gb300 as kda

from _harness import (assert_out_match, assert_pool_match, f16_ulp_distance, gpu_decode,
                      gpu_verify, lib_for, oracle_decode, oracle_verify, pool_np)

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]


# ---------------------------------------------------------------------------
# the configured workloads
# ---------------------------------------------------------------------------
def test_tiny_chain_of_eight_decode_calls():
    """1 request, HV=2, K=V=16, 8 sequential decode calls on a 1-slot fp32 pool."""
    tiny = workloads.make_tiny(seed=0)
    gpool = tiny["pool"].clone()
    ref = pool_np(tiny["pool"])
    import oracle
    for t in range(8):
        inp = workloads.StepInputs(gpool, tiny["slot"], tiny["q"][t], tiny["k"][t], tiny["v"][t],
                                   tiny["a"][t], tiny["b"][t])
        gpool, o, st = gpu_decode(inp)
        assert st == 0
        o_ref = oracle.decode_step(ref, tiny["slot"].numpy(), tiny["q"][t], tiny["k"][t],
                                   tiny["v"][t], tiny["a"][t], tiny["b"][t])
        assert_out_match(o, o_ref, torch.float32, f"token {t}")
        assert_pool_match(gpool, ref, [0], f"token {t}")
        # carry each side's own state forward (both are fp32 pools)


@pytest.mark.parametrize("state_dtype,seed", [(torch.float32, 0), (torch.float16, 1)])
def test_decode_n64_hv12_k128_v128(state_dtype, seed):
    """N=64 requests x HV=12, K=V=128, bf16 q/k/v, 256-slot pool; the whole pool compared."""
    inp = workloads.make_decode(state_dtype=state_dtype, seed=seed)
    gpool, o, st = gpu_decode(inp)
    ref, o_ref = oracle_decode(inp)
    assert st == 0
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gpool, ref, inp.init_slot.numpy(), "pool")


@pytest.mark.parametrize("state_dtype", [torch.float16, torch.float32])
def test_spec_verify_n8_t8(state_dtype):
    """8 requests x 8 tokens; the state after each token lands in its own snapshot slot."""
    inp = workloads.make_verify(state_dtype=state_dtype, seed=2)
    gpool, o, st = gpu_verify(inp)
    ref, o_ref = oracle_verify(inp)
    assert st == 0
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gpool, ref, inp.snap_slot.numpy(), "pool")
    # init slots were only read
    g = pool_np(gpool)
    assert g[inp.init_slot.long().numpy()].tobytes() == pool_np(inp.pool)[inp.init_slot.long().numpy()].tobytes()


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("qkv_dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("K,V", [(16, 16), (48, 80), (128, 16), (32, 128), (112, 48)])
def test_decode_ragged_shapes_and_input_types(state_dtype, qkv_dtype, K, V):
    """K, V multiples of 16 that leave a partial column tile; resets mixed in."""
    inp = workloads.make_decode(n=5, hv=3, k=K, v=V, num_slots=9, state_dtype=state_dtype,
                                qkv_dtype=qkv_dtype, seed=K * 1000 + V, reset_p=0.4)
    gpool, o, st = gpu_decode(inp)
    ref, o_ref = oracle_decode(inp)
    assert st == 0
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gpool, ref, inp.init_slot.numpy(), "pool")


# An fp16-pool decode whose one-tile grid exceeds one wave (8 CTAs per SM: 1216
# on 152 SMs) runs two 64-column tiles per CTA.  V = 80 gives each head a full
# and a 16-column tile; V = 48 gives one tile, the CTA's second slot empty.
@pytest.mark.parametrize("n,hv,K,V", [(64, 12, 128, 80), (128, 12, 64, 48)])
def test_fp16_decode_two_tiles_a_cta_ragged(n, hv, K, V):
    inp = workloads.make_decode(n=n, hv=hv, k=K, v=V, num_slots=n + 7, state_dtype=torch.float16,
                                qkv_dtype=torch.bfloat16, seed=K * 1000 + V + 7, reset_p=0.2)
    gpool, o, st = gpu_decode(inp)
    ref, o_ref = oracle_decode(inp)
    assert st == 0
    assert_out_match(o, o_ref, torch.float16, "o")
    assert_pool_match(gpool, ref, inp.init_slot.numpy(), "pool")


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("T", [1, 3, 8, 13])
def test_verify_token_counts_and_resets(state_dtype, T):
    inp = workloads.make_verify(n=3, t=T, hv=2, k=64, v=48, num_slots=3 * (T + 1) + 2,
                                state_dtype=state_dtype, seed=T, reset_p=0.5)
    gpool, o, st = gpu_verify(inp)
    ref, o_ref = oracle_verify(inp)
    assert st == 0
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gpool, ref, inp.snap_slot.numpy(), "pool")


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_verify_init_slot_equal_to_a_snapshot_slot(state_dtype):
    """A request may write its first snapshot over the slot it was read from."""
    inp = workloads.make_verify(n=2, t=4, hv=2, k=32, v=32, num_slots=12, state_dtype=state_dtype,
                                seed=21)
    inp.snap_slot[:, 0] = inp.init_slot
    gpool, o, st = gpu_verify(inp)
    ref, o_ref = oracle_verify(inp)
    assert st == 0
    assert_out_match(o, o_ref, state_dtype, "o")
    assert_pool_match(gpool, ref, inp.snap_slot.numpy(), "pool")


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_padded_slot_stride(state_dtype):
    """A pool whose slots are padded (slot_stride > HV*K*V) is addressed through state_at."""
    hv, K, V, ns, pad = 2, 32, 48, 6, 64
    inp = workloads.make_decode(n=4, hv=hv, k=K, v=V, num_slots=ns, state_dtype=state_dtype,
                                qkv_dtype=torch.float32, seed=31)
    stride = hv * K * V + pad
    flat = torch.full((ns * stride,), 7.0, dtype=state_dtype)
    view = flat.as_strided((ns, hv, K, V), (stride, K * V, V, 1))
    view.copy_(inp.pool)
    gflat = flat.cuda()
    gview = gflat.as_strided((ns, hv, K, V), (stride, K * V, V, 1))
    d = inp.to("cuda")
    o = torch.empty(4, hv, V, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib_for(state_dtype).kda_decode_step(gview, d.init_slot, d.q, d.k, d.v, d.a, d.b, o, status)
    torch.cuda.synchronize()
    import oracle
    ref_flat = pool_np(flat)
    o_ref = oracle.decode_step(ref_flat.reshape(ns, stride)[:, : hv * K * V].reshape(ns, hv, K, V).copy(),
                               inp.init_slot.numpy(), inp.q, inp.k, inp.v, inp.a, inp.b)
    assert int(status.item()) == 0
    assert_out_match(o.cpu(), o_ref, state_dtype, "o")
    g = pool_np(gflat).reshape(ns, stride)
    r = ref_flat.reshape(ns, stride)
    assert g[:, hv * K * V:].tobytes() == r[:, hv * K * V:].tobytes()  # the padding is never written


def test_empty_calls_are_noops():
    for sd in (torch.float32, torch.float16):
        inp = workloads.make_decode(n=0, hv=2, k=16, v=16, num_slots=4, state_dtype=sd, seed=0)
        gpool, o, st = gpu_decode(inp)
        assert st == 0 and gpool.equal(inp.pool) and o.numel() == 0
        inp = workloads.make_verify(n=2, t=0, hv=2, k=16, v=16, num_slots=4, state_dtype=sd, seed=0)
        gpool, o, st = gpu_verify(inp)
        assert st == 0 and gpool.equal(inp.pool)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_out_of_range_slot_sets_status_and_skips(state_dtype):
    inp = workloads.make_decode(n=6, hv=2, k=32, v=32, num_slots=8, state_dtype=state_dtype, seed=41)
    inp.init_slot[2] = 8       # one past the end
    inp.init_slot[4] = -3
    gpool, o, st = gpu_decode(inp)
    assert st == kda.KDA_ERR_SLOT_RANGE
    good = [0, 1, 3, 5]
    sub = workloads.StepInputs(inp.pool, inp.init_slot[good], inp.q[good], inp.k[good],
                               inp.v[good], inp.a[good], inp.b[good])
    ref, o_ref = oracle_decode(sub)
    assert_out_match(o[good], o_ref, state_dtype, "o")
    assert_pool_match(gpool, ref, inp.init_slot[good].numpy(), "pool")
    # verify: a bad snapshot id skips that request only
    v = workloads.make_verify(n=3, t=2, hv=2, k=32, v=32, num_slots=12, state_dtype=state_dtype, seed=42)
    v.snap_slot[1, 1] = 12
    gpool, o, st = gpu_verify(v)
    assert st == kda.KDA_ERR_SLOT_RANGE
    assert pool_np(gpool)[v.snap_slot[1, 0].item()].tobytes() == pool_np(v.pool)[v.snap_slot[1, 0].item()].tobytes()


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_identity_step_is_bit_exact(state_dtype):
    """alpha = 1, beta = 0: widen then store must give back the pool's own bits."""
    inp = workloads.make_decode(n=16, hv=12, k=128, v=128, num_slots=32, state_dtype=state_dtype,
                                seed=51)
    inp.a[:] = -float("inf")
    inp.b[:] = -float("inf")
    gpool, o, st = gpu_decode(inp)
    assert st == 0
    assert pool_np(gpool).tobytes() == pool_np(inp.pool).tobytes()
    ref, o_ref = oracle_decode(inp)
    assert_out_match(o, o_ref, state_dtype, "o")


def _saturate_gates(inp):
    """Rows of a at +inf, -inf, +100 and -100 (alpha = 0, 1, ~4e-44, ~1),
    b per head at +inf, -inf, +100, -100, 0 in turn (beta = 1, 0, ~1, ~4e-44, 1/2)."""
    k = inp.a.shape[-1]
    for i, val in enumerate((float("inf"), -float("inf"), 100.0, -100.0)):
        inp.a[..., i * k // 4:(i + 1) * k // 4] = val
    vals = (float("inf"), -float("inf"), 100.0, -100.0, 0.0)
    for h in range(inp.b.shape[-1]):
        inp.b[..., h] = vals[h % len(vals)]
    return inp


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_saturated_gates_match_oracle(state_dtype):
    """The decay and the update gate at their limits: alpha exactly 0 and 1,
    beta exactly 1 and 0, and values past the point where e^a overflows."""
    dec = _saturate_gates(workloads.make_decode(n=8, hv=10, k=128, v=128, num_slots=16,
                                                state_dtype=state_dtype, seed=57))
    gpool, o, st = gpu_decode(dec)
    assert st == 0
    ref, o_ref = oracle_decode(dec)
    assert np.isfinite(o.numpy()).all()
    assert_out_match(o, o_ref, state_dtype, "decode o")
    assert_pool_match(gpool, ref, dec.init_slot.numpy(), "decode pool")
    ver = _saturate_gates(workloads.make_verify(n=4, t=5, hv=10, k=128, v=128, num_slots=32,
                                                state_dtype=state_dtype, seed=58))
    gpool, o, st = gpu_verify(ver)
    assert st == 0
    ref, o_ref = oracle_verify(ver)
    assert np.isfinite(o.numpy()).all()
    assert_out_match(o, o_ref, state_dtype, "verify o")
    assert_pool_match(gpool, ref, ver.snap_slot.numpy(), "verify snapshots")


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_zero_k_and_q_rows_match_oracle(state_dtype):
    """All-zero k or q rows (the norm's epsilon keeps khat = 0 and qhat = 0, no
    NaN): the update is the decay alone and the output is zero where q is."""
    dec = workloads.make_decode(n=8, hv=4, k=128, v=128, num_slots=16, state_dtype=state_dtype, seed=59)
    dec.k[::2, 1] = 0.0
    dec.q[1::3, 2] = 0.0
    gpool, o, st = gpu_decode(dec)
    assert st == 0
    ref, o_ref = oracle_decode(dec)
    assert np.isfinite(o.numpy()).all()
    assert_out_match(o, o_ref, state_dtype, "decode o")
    assert_pool_match(gpool, ref, dec.init_slot.numpy(), "decode pool")
    ver = workloads.make_verify(n=4, t=5, hv=4, k=128, v=128, num_slots=32, state_dtype=state_dtype, seed=60)
    ver.k[:, 1::2, 1] = 0.0   # tokens 1 and 3 of head 1
    ver.q[2, :, 3] = 0.0      # every token of request 2, head 3
    gpool, o, st = gpu_verify(ver)
    assert st == 0
    ref, o_ref = oracle_verify(ver)
    assert np.isfinite(o.numpy()).all()
    assert_out_match(o, o_ref, state_dtype, "verify o")
    assert_pool_match(gpool, ref, ver.snap_slot.numpy(), "verify snapshots")


def test_verify_equals_chained_decode_on_fp32_pool():
    """An fp32 pool stores the fp32 carry exactly, so T decode calls and one
    T-token verify agree up to the order of the fp32 sums over K (the two
    kernels split that reduction differently): within a few fp32 ulps."""
    inp = workloads.make_verify(n=4, t=6, hv=12, k=128, v=128, num_slots=64,
                                state_dtype=torch.float32, seed=61)
    gpool_v, o_v, st = gpu_verify(inp)
    assert st == 0
    pool = inp.pool.clone()
    for t in range(6):
        step = workloads.StepInputs(pool, inp.init_slot, inp.q[:, t], inp.k[:, t], inp.v[:, t],
                                    inp.a[:, t], inp.b[:, t])
        pool, o_d, st = gpu_decode(step)
        assert st == 0
        np.testing.assert_allclose(o_d.numpy(), o_v[:, t].numpy(), rtol=0, atol=2e-6)
        for r in range(4):
            np.testing.assert_allclose(pool[inp.init_slot[r]].numpy(),
                                       gpool_v[inp.snap_slot[r, t]].numpy(), rtol=0, atol=2e-6)


def test_fp16_build_against_fp32_twin():
    """The fp32-twin check of ROCm/ATOM pull request 2945 (Testing): the fp16
    build's stored states equal RNE(fp32 build's states) on the exactly widened
    pool, within one fp16 step (the builds tile V differently, so their fp32
    sums may differ in the last bit), and the outputs agree."""
    inp16 = workloads.make_verify(n=8, t=8, hv=12, k=128, v=128, state_dtype=torch.float16, seed=2)
    inp32 = workloads.StepInputs(inp16.pool.float(), inp16.init_slot, inp16.q, inp16.k, inp16.v,
                                 inp16.a, inp16.b, inp16.snap_slot)
    p16, o16, s16 = gpu_verify(inp16)
    p32, o32, s32 = gpu_verify(inp32)
    assert s16 == 0 and s32 == 0
    snaps = inp16.snap_slot.long().flatten()
    twin = pool_np(p32[snaps].half())
    dist = f16_ulp_distance(pool_np(p16[snaps]), twin)
    assert dist.max() <= 1
    assert (dist == 0).mean() > 0.99
    np.testing.assert_allclose(o16.numpy(), o32.numpy(), rtol=1e-5, atol=1e-6)


def test_results_do_not_depend_on_the_stream():
    inp = workloads.make_decode(n=8, hv=4, k=64, v=64, num_slots=16, seed=71)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        p1, o1, st1 = gpu_decode(inp, stream=s)
    p2, o2, st2 = gpu_decode(inp)
    assert st1 == st2 == 0 and torch.equal(p1, p2) and torch.equal(o1, o2)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_launch_flags_do_not_change_results(state_dtype):
    """Programmatic dependent launch (with and without early state loads) gives
    the same bits as a plain launch, also when captured in a CUDA graph of
    back-to-back steps on different pools."""
    inp = workloads.make_decode(n=24, hv=12, k=128, v=128, num_slots=64, state_dtype=state_dtype,
                                seed=81, reset_p=0.2)
    lib = lib_for(state_dtype)
    d = inp.to("cuda")
    pools = [d.pool.clone() for _ in range(3)]
    outs = [torch.empty(24, 12, 128, device="cuda") for _ in range(3)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = [0, kda.KDA_LAUNCH_PDL, kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(3):
                lib.kda_decode_step(pools[i], d.init_slot, d.q, d.k, d.v, d.a, d.b, outs[i], status,
                                    reset=d.reset, flags=flags[i])
        g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in (1, 2):
        assert torch.equal(pools[i], pools[0]) and torch.equal(outs[i], outs[0])
    ref, o_ref = oracle_decode(inp)
    assert_out_match(outs[2].cpu(), o_ref, state_dtype, "o")
    assert_pool_match(pools[2].cpu(), ref, inp.init_slot.numpy(), "pool")


def test_pdl_chain_on_one_pool_without_early_state():
    """Back-to-back steps on the same pool with KDA_LAUNCH_PDL alone (the state
    is read only after the previous step completed) equal the plain chain."""
    inp = workloads.make_verify(n=4, t=5, hv=12, k=128, v=128, num_slots=64,
                                state_dtype=torch.float32, seed=82)
    lib = lib_for(torch.float32)
    d = inp.to("cuda")
    results = []
    for flags in (0, kda.KDA_LAUNCH_PDL):
        pool = d.pool.clone()
        o = torch.empty(5, 4, 12, 128, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        for t in range(5):
            lib.kda_decode_step(pool, d.init_slot, d.q[:, t].contiguous(), d.k[:, t].contiguous(),
                                d.v[:, t].contiguous(), d.a[:, t].contiguous(), d.b[:, t].contiguous(),
                                o[t], status, flags=flags)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        results.append((pool.cpu(), o.cpu()))
    assert torch.equal(results[0][0], results[1][0]) and torch.equal(results[0][1], results[1][1])
