"""kda_stage_host: device-mapped pinned host memory copied into device
buffers by one kernel launch, bit for bit; pageable sources and host
destinations are refused before any launch."""
import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from _harness import lib_for

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("built_libs")]


@pytest.mark.parametrize("flags", [0, kda.KDA_LAUNCH_PDL])
def test_stage_copies_every_region_bit_for_bit(flags):
    g = torch.Generator().manual_seed(11)
    sizes = [16, 4096, 986368 - 4096 - 16, 48, 393216]
    srcs = [torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory() for n in sizes]
    dsts = [torch.zeros(n, dtype=torch.uint8, device="cuda") for n in sizes]
    lib = lib_for(torch.float32)
    torch.cuda.synchronize()
    lib.kda_stage_host(list(zip(dsts, srcs)), flags=flags)
    torch.cuda.synchronize()
    for d, s in zip(dsts, srcs):
        assert torch.equal(d.cpu(), s)


def test_stage_refuses_pageable_and_misplaced_buffers():
    lib = lib_for(torch.float32)
    pageable = torch.zeros(64, dtype=torch.uint8)
    pinned = torch.zeros(64, dtype=torch.uint8).pin_memory()
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.kda_stage_host_raw([(dev.data_ptr(), pageable.data_ptr(), 64)], s) == kda.KDA_ERR_ARG
    assert lib.kda_stage_host_raw([(pinned.data_ptr(), pinned.data_ptr(), 64)], s) == kda.KDA_ERR_ARG
    assert lib.kda_stage_host_raw([(dev.data_ptr(), pinned.data_ptr(), 40)], s) == kda.KDA_ERR_ARG
    assert lib.kda_stage_host_raw([(dev.data_ptr() + 8, pinned.data_ptr(), 32)], s) == kda.KDA_ERR_ALIGN
    assert lib.kda_stage_host_raw([(dev.data_ptr(), pinned.data_ptr(), 64)] * 9, s) == kda.KDA_ERR_ARG
    assert lib.kda_stage_host_raw([], s) == kda.KDA_OK
    torch.cuda.synchronize()


def test_decode_writes_its_output_into_host_mapped_memory():
    """The end-to-end path: inputs staged from pinned host memory by
    kda_stage_host, and a decode whose o is pinned host memory (the device
    writes it over the host link), against the same decode into device memory."""
    from kda_linear_attention_gated_gb300 import workloads
    inp = workloads.make_decode(n=16, hv=12, k=128, v=128, num_slots=32, state_dtype=torch.float32,
                                qkv_dtype=torch.bfloat16, seed=12)
    lib = lib_for(torch.float32)
    ref = inp.to("cuda")
    o_ref = torch.empty(16, 12, 128, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kda_decode_step(ref.pool, ref.init_slot, ref.q, ref.k, ref.v, ref.a, ref.b, o_ref, status)
    d = inp.to("cuda")
    names = ("init_slot", "q", "k", "v", "a", "b")
    host = {n_: getattr(inp, n_).contiguous().pin_memory() for n_ in names}
    dev = {n_: torch.empty_like(getattr(d, n_)) for n_ in names}
    o_host = torch.full((16, 12, 128), float("nan")).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    lib.kda_stage_host([(dev[n_], host[n_]) for n_ in names], flags=kda.KDA_LAUNCH_PDL)
    rc = lib.kda_decode_step_raw(kda.pool_desc(d.pool), dev["init_slot"].data_ptr(), None, 16, dev["q"].data_ptr(),
                                 dev["k"].data_ptr(), dev["v"].data_ptr(), kda.KDA_BF16, dev["a"].data_ptr(),
                                 dev["b"].data_ptr(), o_host.data_ptr(), status.data_ptr(), s, kda.KDA_LAUNCH_PDL)
    assert rc == kda.KDA_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(o_host, o_ref.cpu())
    assert torch.equal(d.pool.cpu(), ref.pool.cpu())
