// Checkpoint flush and load of whole slot states through the address
// function (ROCm/ATOM pull request 2945, Changes: under ReplaySSM the
// checkpoint load and the flush go through state_at).  A pure copy: each CTA
// moves one 16 KB piece of one state with coalesced 16-byte streaming loads
// and stores (the bytes are touched once, so they bypass L1 and are marked
// evict-first in L2).
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int CKPT_THREADS = 256;
constexpr int CKPT_VEC_PER_THREAD = 4;                                  // 4 x 16 B
constexpr int CKPT_PIECE = CKPT_THREADS * CKPT_VEC_PER_THREAD * 16;     // bytes per CTA

struct CkptParams {
    char* pool;
    int64_t num_slots;
    int64_t slot_bytes;      // bytes between slots
    char* plane;
    int64_t num_entries;
    int64_t entry_bytes;     // bytes between entries
    int64_t state_bytes;     // bytes of one state, a multiple of 16
    int n;
    const int32_t* slots;
    const int32_t* entries;
    int load;                // 1: plane -> pool, 0: pool -> plane
    int32_t* status;
};

__global__ void __launch_bounds__(CKPT_THREADS) kda_ckpt_kernel(const CkptParams p) {
    const int64_t pieces = (p.state_bytes + CKPT_PIECE - 1) / CKPT_PIECE;
    const int64_t i = (int64_t)blockIdx.x / pieces;
    const int64_t piece = (int64_t)blockIdx.x - i * pieces;
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize();
    const int32_t s = p.slots[i], e = p.entries[i];
    if (s >= p.num_slots || e >= p.num_entries) {
        if (threadIdx.x == 0 && piece == 0) atomicCAS(p.status, 0, STATUS_SLOT_RANGE);
        return;
    }
    if (s < 0 || e < 0) return;
    const char* src = p.load ? p.plane + (int64_t)e * p.entry_bytes : p.pool + (int64_t)s * p.slot_bytes;
    char* dst = p.load ? p.pool + (int64_t)s * p.slot_bytes : p.plane + (int64_t)e * p.entry_bytes;
    const int64_t base = piece * CKPT_PIECE;
    uint4 v[CKPT_VEC_PER_THREAD];
#pragma unroll
    for (int j = 0; j < CKPT_VEC_PER_THREAD; ++j) {
        const int64_t off = base + ((int64_t)j * CKPT_THREADS + threadIdx.x) * 16;
        if (off < p.state_bytes) v[j] = __ldcs(reinterpret_cast<const uint4*>(src + off));
    }
#pragma unroll
    for (int j = 0; j < CKPT_VEC_PER_THREAD; ++j) {
        const int64_t off = base + ((int64_t)j * CKPT_THREADS + threadIdx.x) * 16;
        if (off < p.state_bytes) __stcs(reinterpret_cast<uint4*>(dst + off), v[j]);
    }
}

}  // namespace kda
