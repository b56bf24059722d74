"""Full-size parity: the 69-layer decode sweep.

69 KDA layers (ROCm/ATOM pull request 2130, What: 69 layers each stream a
[12, 128, 128] state per token), each with its own 256-slot pool, N requests
per layer, HV=12, K=V=128, fp32 inputs, resets ~ Bernoulli(0.05), slot ids the
first N of a seeded permutation.  All 69 steps run as one CUDA graph with the
launch flags the benchmark uses (programmatic dependent launch with early state
loads: every layer has its own pool, so no launch reads what the previous one
writes).  Slots no request touches hold a sentinel and must come back bit for
bit; sampled layers are compared with the fp64 oracle in full.
"""
import numpy as np
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import workloads

from _harness import assert_out_match, assert_pool_match, lib_for, oracle_decode, oracle_verify

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs", "oracle_mod")]

LAYERS = 69
SENTINEL = -7.25  # no state a step writes here; untouched slots must keep it


def _warm(lib, d, n):
    """One launch outside the capture (on a copy of the pool), so the library's
    one-time setup (function attributes, tensor-map entry point) is done."""
    o = torch.empty(n, 12, 128, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_decode_step(d.pool.clone(), d.init_slot, d.q, d.k, d.v, d.a, d.b, o, status, reset=d.reset)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("n", [1, 16, 64, 128])
def test_69_layer_sweep(state_dtype, n):
    lib = lib_for(state_dtype)
    host = [workloads.make_sweep_layer(layer, n, state_dtype, sentinel=SENTINEL)
            for layer in range(LAYERS)]
    dev = [h.to("cuda") for h in host]
    outs = [torch.full((n, 12, 128), float("nan"), device="cuda") for _ in range(LAYERS)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE
    _warm(lib, dev[0], n)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for layer in range(LAYERS):
                d = dev[layer]
                lib.kda_decode_step(d.pool, d.init_slot, d.q, d.k, d.v, d.a, d.b, outs[layer],
                                    status, reset=d.reset, flags=flags)
        graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    sentinel_bits = torch.tensor([SENTINEL], dtype=state_dtype).view(
        torch.int32 if state_dtype == torch.float32 else torch.int16).item()
    ibits = torch.int32 if state_dtype == torch.float32 else torch.int16
    for layer in range(LAYERS):
        untouched = torch.ones(256, dtype=torch.bool, device="cuda")
        untouched[dev[layer].init_slot.long()] = False
        assert bool((dev[layer].pool[untouched].view(ibits) == sentinel_bits).all()), \
            f"layer {layer}: a slot no request uses was written"
        assert bool(torch.isfinite(outs[layer]).all()), f"layer {layer}: output not written"

    rng = np.random.default_rng(1000 + n)
    sampled = sorted({0, LAYERS - 1, *rng.choice(LAYERS, size=3, replace=False).tolist()})
    for layer in sampled:
        ref, o_ref = oracle_decode(host[layer])
        assert_out_match(outs[layer].cpu(), o_ref, state_dtype, f"layer {layer} o")
        assert_pool_match(dev[layer].pool.cpu(), ref, host[layer].init_slot.numpy(), f"layer {layer} pool")
    del dev, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_decode_bench_launch_configuration_sampled(state_dtype):
    """The benchmark's own launch pattern -- a CUDA graph of steps over rotating
    copies of the N=64, HV=12, K=V=128 pool with PDL flags -- checked on the
    outputs of every step against the oracle run on the same sequence (each
    copy is updated once, so each step sees the initial pool)."""
    lib = lib_for(state_dtype)
    inp = workloads.make_decode(n=64, hv=12, k=128, v=128, num_slots=256, state_dtype=state_dtype,
                                qkv_dtype=torch.bfloat16, seed=0 if state_dtype == torch.float32 else 1)
    R = 6
    d = inp.to("cuda")
    pools = [d.pool.clone() for _ in range(R)]
    outs = [torch.empty(64, 12, 128, device="cuda") for _ in range(R)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = kda.KDA_LAUNCH_PDL | kda.KDA_LAUNCH_PDL_EARLY_STATE
    _warm(lib, d, 64)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(R):
                lib.kda_decode_step(pools[i], d.init_slot, d.q, d.k, d.v, d.a, d.b, outs[i], status,
                                    flags=flags)
        graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, o_ref = oracle_decode(inp)
    for i in range(R):
        assert_out_match(outs[i].cpu(), o_ref, state_dtype, f"step {i} o")
        assert_pool_match(pools[i].cpu(), ref, inp.init_slot.numpy(), f"step {i} pool")


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_pool_past_2_31_elements(state_dtype):
    """A pool of 11,000 (fp32) or 16,400 (fp16) slots at the layer shape holds
    more than 2^31 elements (over 4 GB): decode, verify and the checkpoint flush
    on the highest slots must equal the oracle on a small pool holding the same
    states, and the neighbouring slots must not change."""
    lib = lib_for(state_dtype)
    num_slots = 11000 if state_dtype == torch.float32 else 16400
    assert num_slots * 12 * 128 * 128 > 2 ** 31
    g = torch.Generator().manual_seed(97)
    small = workloads.make_decode(n=16, hv=12, k=128, v=128, num_slots=16, state_dtype=state_dtype, seed=97)
    high = torch.arange(num_slots - 16, num_slots, dtype=torch.int32)[torch.randperm(16, generator=g)]
    big = torch.empty(num_slots, 12, 128, 128, dtype=state_dtype, device="cuda")
    big[num_slots - 20:num_slots - 16] = SENTINEL
    big[high.long().cuda()] = small.pool.cuda()[small.init_slot.long().cuda()]
    d = small.to("cuda")
    o = torch.empty(16, 12, 128, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_decode_step(big, high.cuda(), d.q, d.k, d.v, d.a, d.b, o, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, o_ref = oracle_decode(small)
    got_small = small.pool.clone()
    got_small[small.init_slot.long()] = big[high.long().cuda()].cpu()
    assert_out_match(o.cpu(), o_ref, state_dtype, "decode o")
    assert_pool_match(got_small, ref, small.init_slot.numpy(), "decode pool")
    assert bool((big[num_slots - 20:num_slots - 16] == SENTINEL).all())
    # verify: initial states from the top 4 slots, snapshots into the 8 below them
    ver = workloads.make_verify(n=2, t=4, hv=12, k=128, v=128, num_slots=12, state_dtype=state_dtype,
                                qkv_dtype=torch.float32, seed=98)
    init_big = torch.tensor([num_slots - 1, num_slots - 2], dtype=torch.int32)
    snap_big = torch.arange(num_slots - 10, num_slots - 2, dtype=torch.int32).reshape(2, 4)
    big[init_big.long().cuda()] = ver.pool.cuda()[ver.init_slot.long().cuda()]
    dv = ver.to("cuda")
    ov = torch.empty(2, 4, 12, 128, device="cuda")
    lib.kda_spec_verify(big, init_big.cuda(), snap_big.cuda(), dv.q, dv.k, dv.v, dv.a, dv.b, ov, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    vref, vo_ref = oracle_verify(ver)
    assert_out_match(ov.cpu(), vo_ref, state_dtype, "verify o")
    got = ver.pool.clone()
    got[ver.snap_slot.long().reshape(-1)] = big[snap_big.long().reshape(-1).cuda()].cpu()
    assert_pool_match(got, vref, ver.snap_slot.numpy(), "verify snapshots")
    # checkpoint flush of the top slots into a small plane, bit for bit
    plane = torch.empty(4, 12, 128, 128, dtype=state_dtype, device="cuda")
    ids = torch.tensor([num_slots - 1, num_slots - 3, num_slots - 5, num_slots - 7], dtype=torch.int32,
                       device="cuda")
    ent = torch.arange(4, dtype=torch.int32, device="cuda")
    lib.kda_ckpt_flush(big, plane, ids, ent, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(plane, big[ids.long()])
    del big
    torch.cuda.empty_cache()
