// The causal short convolution in front of the KDA recurrence, with its paged
// window, fused into one pass: convolution, SiLU and the window update.
//
// The conv pool keeps, per request slot, the last L = kernel - 1 + num_spec
// inputs of each channel (ROCm/ATOM pull request 2894, review thread on the
// conv window: the window is sized kernel - 1 + num_spec; a step reads its
// kernel - 1 history entries starting at the accepted index and writes back
// the kept old entries followed by the step's inputs).  Layout here:
// [slot][L][C], oldest entry first and the channel innermost, so that a warp's
// 32 consecutive channels of one entry are one coalesced access.
//
// One thread per (request, channel).  With acc = accepted[r] - 1 (0 without),
// m = acc + KW - 1 valid entries and kept = max(0, L - T) old ones:
//   history h_i = W[acc + i] (i < KW - 1; zero on reset), z = h ++ x,
//   y_t = act(bias + sum_i w_i z_{t+i})      (w_{KW-1} weighs the newest input)
//   new window = W[m - kept .. m - 1] (zero on reset) ++ the last min(T, L) inputs.
// Every read of the window happens before any write to it.  The arithmetic is
// fp32; y is rounded to the window's dtype to nearest even.
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int CONV_KW_MAX = 8;   // kernel widths 1 .. 8
constexpr int CONV_L_MAX = 32;   // window entries up to 32
constexpr int CONV_THREADS = 256;

struct ConvParams {
    void* window;
    int64_t num_slots;
    int64_t slot_stride;          // elements
    int C, L, KW;
    int n, t;                     // requests; tokens per request without cu (bound with cu)
    int total;                    // rows of x and y: every request's tokens lie below it
    const int32_t* cu;            // [n + 1] or nullptr
    const int32_t* conv_slot;     // [n]
    const int32_t* accepted;      // [n] or nullptr
    const uint8_t* reset;         // [n] or nullptr
    const void* x;                // [total][C]
    const float* w;               // [C][KW]
    const float* bias;            // [C] or nullptr
    void* y;                      // [total][C]
    int silu;
    int32_t* status;
};

__device__ __forceinline__ float conv_ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float conv_ld(const __half* p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ float conv_ld(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void conv_st(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void conv_st(__half* p, int64_t i, float v) { p[i] = __float2half_rn(v); }
__device__ __forceinline__ void conv_st(__nv_bfloat16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }

template <typename ET>
__global__ void __launch_bounds__(CONV_THREADS) kda_conv_kernel(const ConvParams p) {
    const int cblocks = (p.C + CONV_THREADS - 1) / CONV_THREADS;
    const int r = (int)blockIdx.x / cblocks;
    const int c = ((int)blockIdx.x - r * cblocks) * CONV_THREADS + (int)threadIdx.x;
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize();  // nothing here is read before the previous kernel is done

    int tb = r * p.t, T = p.t;
    if (p.cu != nullptr) {
        tb = p.cu[r];
        T = p.cu[r + 1] - tb;
    }
    const int32_t slot = p.conv_slot[r];
    const int acc = p.accepted != nullptr ? p.accepted[r] - 1 : 0;
    const int m = acc + p.KW - 1;
    const int kept = max(0, p.L - T);
    // uniform over the CTA: one request
    if (slot >= p.num_slots) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, STATUS_SLOT_RANGE);
        return;
    }
    if (tb < 0 || T < 0 || T > p.t || tb + T > p.total || (slot >= 0 && T > 0 && (acc < 0 || m > p.L || m < kept))) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, STATUS_ARG);
        return;
    }
    if (c >= p.C) return;
    ET* y = static_cast<ET*>(p.y);
    if (slot < 0) {  // padding: zero outputs, window untouched
        for (int t = 0; t < T; ++t) conv_st(y, (int64_t)(tb + t) * p.C + c, 0.f);
        return;
    }
    if (T == 0) return;

    const ET* x = static_cast<const ET*>(p.x);
    ET* W = static_cast<ET*>(p.window) + (int64_t)slot * p.slot_stride + c;
    const bool rst = p.reset != nullptr && p.reset[r] != 0;
    // w[i] weighs history entry i (i < KW - 1); wlast weighs the current input
    float w[CONV_KW_MAX], z[CONV_KW_MAX], old[CONV_L_MAX];
#pragma unroll
    for (int i = 0; i < CONV_KW_MAX; ++i) {
        w[i] = i < p.KW - 1 ? __ldg(p.w + (int64_t)c * p.KW + i) : 0.f;
        z[i] = (i < p.KW - 1 && !rst) ? conv_ld(W, (int64_t)(acc + i) * p.C) : 0.f;
    }
    const float wlast = __ldg(p.w + (int64_t)c * p.KW + p.KW - 1);
#pragma unroll
    for (int e = 0; e < CONV_L_MAX; ++e)
        old[e] = (e < kept && !rst) ? conv_ld(W, (int64_t)(m - kept + e) * p.C) : 0.f;
    const float bias = p.bias != nullptr ? __ldg(p.bias + c) : 0.f;

    for (int t = 0; t < T; ++t) {
        const float xv = conv_ld(x, (int64_t)(tb + t) * p.C + c);
        float s = bias;
#pragma unroll
        for (int i = 0; i < CONV_KW_MAX; ++i) s = fmaf(w[i], z[i], s);  // w is 0 past KW - 2
        s = fmaf(wlast, xv, s);
        const float out = p.silu ? s / (1.0f + expf(-s)) : s;
        conv_st(y, (int64_t)(tb + t) * p.C + c, out);
        // slide the history by one: z_i <- z_(i+1), the last history entry <- x_t
#pragma unroll
        for (int i = 0; i < CONV_KW_MAX; ++i) {
            if (i < p.KW - 2) z[i] = z[i + 1 < CONV_KW_MAX ? i + 1 : i];
            else if (i == p.KW - 2) z[i] = xv;
        }
    }
    // the new window: kept old entries, then the last min(T, L) inputs (a copy)
#pragma unroll
    for (int e = 0; e < CONV_L_MAX; ++e)
        if (e < kept) conv_st(W, (int64_t)e * p.C, old[e]);
    const int nin = min(T, p.L);
    const ET* xs = x + (int64_t)(tb + T - nin) * p.C + c;
    for (int e = 0; e < nin; ++e) W[(int64_t)(kept + e) * p.C] = xs[(int64_t)e * p.C];
}

}  // namespace kda
