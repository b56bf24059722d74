"""kda_prefill_chunked_noalloc: the two-pass prefill on the library's own
file-scope scratch buffer.  It must give the oracle's results, allocate no
device memory per call, and refuse work larger than its buffer before any
launch."""
import ctypes

import pytest
import torch

import kda_linear_attention_gated_gb300 as kda
from kda_linear_attention_gated_gb300 import PoolDesc, PrefillArgs, workloads

import oracle
from _harness import assert_out_match, assert_pool_match, lib_for, pool_np

SCRATCH = 128 << 20


def test_too_large_for_the_scratch_is_refused_before_any_launch(built_libs):
    lib = kda.KdaLibrary(torch.float32)
    P = 0x7F0000100000
    desc = PoolDesc(P, kda.KDA_F32, 12, 128, 128, 16, 12 * 128 * 128)
    need = lib.kda_prefill_workspace_bytes(desc, 1, 65536)
    assert need > SCRATCH
    args = PrefillArgs(1, 65536, 65536, 12, kda.KDA_BF16, 0, None, P, P, None, P, P, P, P, P, None, None, P)
    rc = lib.lib.kda_prefill_chunked_noalloc(ctypes.byref(desc), ctypes.byref(args), P, 0, None)
    assert rc == kda.KDA_ERR_SHAPE
    # 4 prompts x 512 tokens at the layer shape fit; 8 x 1024 do not
    assert lib.kda_prefill_workspace_bytes(desc, 4, 2048) <= SCRATCH
    assert lib.kda_prefill_workspace_bytes(desc, 8, 8192) > SCRATCH


@pytest.mark.gpu
@pytest.mark.usefixtures("built_libs", "oracle_mod")
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16])
def test_noalloc_prefill_matches_workspace_entry_and_allocates_nothing(state_dtype):
    """Two no-alloc calls in a row, each on a fresh copy of the pool, against
    kda_prefill_chunked with a caller workspace (and against the oracle): the
    same outputs and final states within the parity tolerances, and no device
    memory allocated by the second call."""
    inp = workloads.make_prefill(lens=(200, 0, 37), state_dtype=state_dtype, seed=95, same_slot_p=0.3)
    d = inp.to("cuda")
    total, hv, v = d.v.shape
    lib = lib_for(state_dtype)
    kw = dict(cu_seqlens=d.cu_seqlens, max_t=inp.max_t, reset=d.reset)
    args = (d.init_slot, d.final_slot, d.q, d.k, d.v, d.a, d.b)

    def buffers():
        return (d.pool.clone(), torch.full((total, hv, v), float("nan"), device="cuda"),
                torch.zeros(1, dtype=torch.int32, device="cuda"))

    pool_w, o_w, st_w = buffers()
    ws = torch.empty(lib.kda_prefill_workspace_bytes(d.pool, len(inp.meta["lens"]), total), dtype=torch.uint8,
                     device="cuda")
    lib.kda_prefill_chunked(pool_w, *args, o_w, st_w, workspace=ws, **kw)
    # first call: may load the module and look up the scratch address
    pool_1, o_1, st_1 = buffers()
    lib.kda_prefill_chunked_noalloc(pool_1, *args, o_1, st_1, **kw)
    pool_2, o_2, st_2 = buffers()
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    lib.kda_prefill_chunked_noalloc(pool_2, *args, o_2, st_2, **kw)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0 and torch.cuda.memory_allocated() == alloc0
    assert int(st_w.item()) == 0 and int(st_1.item()) == 0 and int(st_2.item()) == 0
    written = [int(f) for f, i in zip(inp.final_slot, inp.init_slot) if f >= 0 and i >= 0]
    ref_pool, ref_o = pool_np(pool_w), o_w.cpu().numpy().astype("float64")
    for pool_x, o_x in ((pool_1, o_1), (pool_2, o_2)):
        assert_out_match(o_x.cpu(), ref_o, state_dtype, "o vs workspace entry")
        assert_pool_match(pool_x.cpu(), ref_pool, written, "pool vs workspace entry")
    P = pool_np(inp.pool)
    o_ref = oracle.prefill(P, inp.init_slot.numpy(), inp.final_slot.numpy(), inp.q, inp.k, inp.v, inp.a, inp.b,
                           cu_seqlens=inp.cu_seqlens.numpy(), reset=inp.reset.numpy(), nthreads=8)
    assert_out_match(o_2.cpu(), o_ref, state_dtype, "o vs oracle")
    assert_pool_match(pool_2.cpu(), P, written, "pool vs oracle")
