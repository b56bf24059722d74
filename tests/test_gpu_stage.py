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
