// Staging of host inputs by a kernel: up to STAGE_MAX_COPIES regions of
// pinned host memory that is mapped into the device's address space are
// copied into device buffers with plain 16-byte loads over the host link, one
// thread per 16 bytes.  The copy runs on the SMs beside other kernels, so a
// step's small inputs avoid the copy engine's fixed cost per transfer.
//
// With KDA_LAUNCH_PDL the loads go out before the wait for the previous
// kernel on the stream (the host wrote the sources before the launch) and the
// stores to the device buffers come after it, so a previous kernel that still
// reads a buffer is never overtaken.
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int STAGE_MAX_COPIES = 8;
constexpr int STAGE_THREADS = 256;

struct StageParams {
    uint4* dst[STAGE_MAX_COPIES];
    const uint4* src[STAGE_MAX_COPIES];
    int64_t end[STAGE_MAX_COPIES];  // exclusive prefix sums of the copies' 16-byte counts
    int n;
    uint32_t flags;
};

__global__ void __launch_bounds__(STAGE_THREADS) kda_stage_kernel(const StageParams p) {
    cudaTriggerProgrammaticLaunchCompletion();
    const int64_t e = (int64_t)blockIdx.x * STAGE_THREADS + threadIdx.x;
    const bool in = p.n > 0 && e < p.end[p.n - 1];
    int c = 0;
#pragma unroll
    for (int i = 0; i < STAGE_MAX_COPIES - 1; ++i) c += (i < p.n - 1 && e >= p.end[i]) ? 1 : 0;
    const int64_t off = e - (c > 0 ? p.end[c - 1] : 0);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (in) v = p.src[c][off];
    if (p.flags & LAUNCH_PDL) cudaGridDependencySynchronize();
    if (in) p.dst[c][off] = v;
}

}  // namespace kda
