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
// One thread per (request, 1 or 4 channels).  With acc = accepted[r] - 1 (0 without),
// m = acc + KW - 1 valid entries and kept = max(0, L - T) old ones:
//   history h_i = W[acc + i] (i < KW - 1; zero on reset), z = h ++ x,
//   y_t = act(bias + sum_i w_i z_{t+i})      (w_{KW-1} weighs the newest input)
//   new window = W[m - kept .. m - 1] (zero on reset) ++ the last min(T, L) inputs.
// Every read of the window happens before any write to it.  The arithmetic is
// fp32, SiLU as s sigmoid(s); y is rounded to the window's dtype to nearest even.
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int CONV_KW_MAX = 8;   // kernel widths 1 .. 8
// Kernel widths of the convolution fused into the recurrence kernels: 1 .. 4
// (a history of up to three entries, held in registers).
constexpr int DCONV_KW_MAX = 4;
constexpr int DCONV_H = DCONV_KW_MAX - 1;
constexpr int CONV_L_MAX = 32;   // window entries up to 32
constexpr int CONV_THREADS = 256;      // threads per CTA, one channel each
constexpr int CONV_VEC_THREADS = 128;  // threads per CTA, four channels each ...
constexpr int CONV_VEC_KW_MAX = 4;     // ... for kernel widths up to 4

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
    uint32_t flags;               // KDA_LAUNCH_* bits
    int32_t* status;
};

__device__ __forceinline__ float conv_f32(float v) { return v; }
__device__ __forceinline__ float conv_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float conv_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void conv_round(float v, float& e) { e = v; }
__device__ __forceinline__ void conv_round(float v, __half& e) { e = __float2half_rn(v); }
__device__ __forceinline__ void conv_round(float v, __nv_bfloat16& e) { e = __float2bfloat16_rn(v); }

// SiLU, s sigmoid(s) = s / (1 + e^-s), with the fast exponential and division
// intrinsics: a few instructions in place of the full-precision forms, which
// made the token loop instruction-bound.  The error is relative to y, about
// 1e-6 at the layer's pre-activation range (the exponential's documented bound
// is 2 + floor(1.173 |x|) ulp, the division's 2 ulp), far below a 16-bit
// output's step and below the fp32 sum's own error near y = 0.  For s below
// about -87 the divisor passes 2^126 and the quotient is -0, the limit of y.
__device__ __forceinline__ float silu_fast(float s) { return __fdividef(s, 1.0f + __expf(-s)); }

// VC consecutive channels of one window entry or token row as one access.
template <int BYTES> struct ConvRaw;
template <> struct ConvRaw<2> { using T = unsigned short; };
template <> struct ConvRaw<4> { using T = unsigned int; };
template <> struct ConvRaw<8> { using T = uint2; };
template <> struct ConvRaw<16> { using T = uint4; };

template <typename ET, int VC>
struct ConvIO {
    using R = typename ConvRaw<VC * (int)sizeof(ET)>::T;
    static __device__ __forceinline__ R ld(const ET* p) { return *reinterpret_cast<const R*>(p); }
    static __device__ __forceinline__ void st(ET* p, R v) { *reinterpret_cast<R*>(p) = v; }
    static __device__ __forceinline__ void widen(R r, float (&f)[VC]) {
        ET e[VC];
        memcpy(e, &r, sizeof(R));
#pragma unroll
        for (int v = 0; v < VC; ++v) f[v] = conv_f32(e[v]);
    }
    static __device__ __forceinline__ R narrow(const float (&f)[VC]) {  // to nearest even
        ET e[VC];
#pragma unroll
        for (int v = 0; v < VC; ++v) conv_round(f[v], e[v]);
        R r;
        memcpy(&r, e, sizeof(R));
        return r;
    }
};

// VC channels per thread (1, or 4 when C and every address allow 4-channel
// accesses), CT threads per CTA, kernel widths up to KWM; grid = requests x
// ceil(C / (VC CT)).
//
// With KDA_LAUNCH_PDL_EARLY_STATE the reads that do not depend on the previous
// kernel on the stream -- token offsets, slot id, accepted index, reset flag,
// weights, bias and the window entries -- go out before the wait for it, so
// they overlap its tail; the inputs x are read, and everything is written,
// after the wait.
// KWF: the kernel width fixed at compile time (0: read from the parameters).
template <typename ET, int VC, int CT, int KWM, int KWF>
__global__ void __launch_bounds__(CT) kda_conv_kernel(const ConvParams p) {
    static_assert(KWF <= KWM, "fixed kernel width");
#define KWR (KWF > 0 ? KWF : p.KW)
    using IO = ConvIO<ET, VC>;
    using R = typename IO::R;
    const int cblocks = (p.C / VC + CT - 1) / CT;
    const int r = (int)blockIdx.x / cblocks;
    const int c = (((int)blockIdx.x - r * cblocks) * CT + (int)threadIdx.x) * VC;  // first channel
    cudaTriggerProgrammaticLaunchCompletion();
    const bool early = (p.flags & LAUNCH_PDL_EARLY_STATE) != 0;
    if (!early) cudaGridDependencySynchronize();  // nothing here is read before the previous kernel is done

    int tb = r * p.t, T = p.t;
    if (p.cu != nullptr) {
        tb = p.cu[r];
        T = p.cu[r + 1] - tb;
    }
    const int32_t slot = p.conv_slot[r];
    const int acc = p.accepted != nullptr ? p.accepted[r] - 1 : 0;
    const bool rst = p.reset != nullptr && p.reset[r] != 0;
    const int m = acc + KWR - 1;
    const int kept = max(0, p.L - T);
    constexpr int CB = 8;  // window entries or tokens per batch of loads
    // kept old entries per batch: a full-length step (T = L - KW + 2) keeps
    // KW - 2 of them, so one batch of KWM - 2 covers it; more go through the loop
    constexpr int CBK = KWM > 2 ? KWM - 2 : 1;
    const bool range_ok = tb >= 0 && T > 0 && T <= p.t && tb + T <= p.total;
    const ET* x = static_cast<const ET*>(p.x) + (int64_t)tb * p.C + min(c, p.C - VC);  // token t at x[t C]
    // The first CB inputs of this request go out before anything that waits
    // for the slot id or the accepted index (rows clamped into the request,
    // the channels into range; only read once the token range is checked).
    R x0[CB];
    auto load_x0 = [&]() {
        if (range_ok)
#pragma unroll
            for (int u = 0; u < CB; ++u) x0[u] = IO::ld(x + (int64_t)min(u, T - 1) * p.C);
    };
    if (!early) load_x0();
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
    ET* y = static_cast<ET*>(p.y) + (int64_t)tb * p.C + c;  // token t at y[t C]
    const R zero = R{};    // +0 in every channel, for all three element types
    if (slot < 0) {  // padding: zero outputs, window untouched
        if (early) cudaGridDependencySynchronize();
        for (int t = 0; t < T; ++t) IO::st(y + (int64_t)t * p.C, zero);
        return;
    }
    if (T == 0) return;

    // Each thread owns its VC channels of the slot's window, so its own
    // program order is the only order its reads and writes need.  Loads go
    // out in batches of CB, unconditionally, from indices clamped into the
    // window or the request's tokens, so that a batch is in flight at once;
    // the values out of range are dropped where they are used.
    ET* W = static_cast<ET*>(p.window) + (int64_t)slot * p.slot_stride + c;
    const int nh = KWR - 1;  // history entries
    // the history entries and the first batch of kept old entries, read
    // together (the kept entries W[m - kept + e] move to W[e])
    R hr[KWM], kv[CBK];
#pragma unroll
    for (int i = 0; i < KWM; ++i) hr[i] = IO::ld(W + (int64_t)min(acc + i, p.L - 1) * p.C);
#pragma unroll
    for (int u = 0; u < CBK; ++u) kv[u] = IO::ld(W + (int64_t)min(m - kept + u, p.L - 1) * p.C);
    // w[i] weighs history entry i (i < KW - 1); wlast weighs the current input.
    // A channel's KW = 4 weights are one 16-byte row, and four channels' biases
    // one 16-byte vector, read as such where the arrays are 16-byte aligned.
    float w[KWM][VC], z[KWM][VC], wlast[VC], bias[VC];
    bool w_rows = false, b_vec = false;
    if constexpr (VC == 4 && KWF == 4) w_rows = (reinterpret_cast<uintptr_t>(p.w) & 15u) == 0;
    if constexpr (VC == 4) b_vec = p.bias != nullptr && (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0;
    if constexpr (VC == 4 && KWF == 4) {
        if (w_rows) {
#pragma unroll
            for (int v = 0; v < VC; ++v) {
                const float4 wr = __ldg(reinterpret_cast<const float4*>(p.w + (int64_t)(c + v) * 4));
                w[0][v] = wr.x;
                w[1][v] = wr.y;
                w[2][v] = wr.z;
                wlast[v] = wr.w;
#pragma unroll
                for (int i = 3; i < KWM; ++i) w[i][v] = 0.f;
            }
        }
    }
    if (!w_rows) {
#pragma unroll
        for (int i = 0; i < KWM; ++i)
#pragma unroll
            for (int v = 0; v < VC; ++v) w[i][v] = i < nh ? __ldg(p.w + (int64_t)(c + v) * KWR + i) : 0.f;
#pragma unroll
        for (int v = 0; v < VC; ++v) wlast[v] = __ldg(p.w + (int64_t)(c + v) * KWR + KWR - 1);
    }
    if constexpr (VC == 4) {
        if (b_vec) {
            const float4 bv = __ldg(reinterpret_cast<const float4*>(p.bias + c));
            bias[0] = bv.x;
            bias[1] = bv.y;
            bias[2] = bv.z;
            bias[3] = bv.w;
        }
    }
    if (!b_vec)
#pragma unroll
        for (int v = 0; v < VC; ++v) bias[v] = p.bias != nullptr ? __ldg(p.bias + c + v) : 0.f;
    if (early) {
        cudaGridDependencySynchronize();
        load_x0();
    }
#pragma unroll
    for (int i = 0; i < KWM; ++i) {
        float hv[VC];
        IO::widen(hr[i], hv);
#pragma unroll
        for (int v = 0; v < VC; ++v) z[i][v] = i < nh && !rst ? hv[v] : 0.f;
    }

    // the kept old entries W[m - kept + e] -> W[e] (zero on reset), ascending:
    // a source never lies below its destination (m >= kept), so no batch reads
    // what an earlier one wrote
#pragma unroll
    for (int u = 0; u < CBK; ++u)
        if (u < kept) IO::st(W + (int64_t)u * p.C, rst ? zero : kv[u]);
    for (int e0 = CBK; e0 < kept; e0 += CB) {
        R v[CB];
#pragma unroll
        for (int u = 0; u < CB; ++u) v[u] = IO::ld(W + (int64_t)min(m - kept + e0 + u, p.L - 1) * p.C);
#pragma unroll
        for (int u = 0; u < CB; ++u)
            if (e0 + u < kept) IO::st(W + (int64_t)(e0 + u) * p.C, rst ? zero : v[u]);
    }
    for (int t0 = 0; t0 < T; t0 += CB) {
        R xr[CB];
        if (t0 == 0) {
#pragma unroll
            for (int u = 0; u < CB; ++u) xr[u] = x0[u];
        } else {
#pragma unroll
            for (int u = 0; u < CB; ++u) xr[u] = IO::ld(x + (int64_t)min(t0 + u, T - 1) * p.C);
        }
#pragma unroll
        for (int u = 0; u < CB; ++u) {
            // past the last token, leave: the history slide below then runs
            // unconditionally and compiles to register renaming, where a
            // guard around it would keep every history register live through
            // selects
            if (t0 + u >= T) break;
            {
                float xv[VC], out[VC];
                IO::widen(xr[u], xv);
#pragma unroll
                for (int v = 0; v < VC; ++v) {
                    float s = bias[v];
#pragma unroll
                    // w is 0 past KW - 2; with the width fixed at compile time those
                    // terms (0 times a zero history slot) are left out
                    for (int i = 0; i < KWM; ++i)
                        if (KWF == 0 || i < KWF - 1) s = fmaf(w[i][v], z[i][v], s);
                    s = fmaf(wlast[v], xv[v], s);
                    out[v] = p.silu ? silu_fast(s) : s;
                    // slide the history by one: z_i <- z_(i+1), the last history entry <- x_t
#pragma unroll
                    for (int i = 0; i < KWM; ++i)
                        z[i][v] = i < nh - 1 ? z[i + 1 < KWM ? i + 1 : i][v] : (i == nh - 1 ? xv[v] : z[i][v]);
                }
                IO::st(y + (int64_t)(t0 + u) * p.C, IO::narrow(out));
            }
        }
    }

    // then the last min(T, L) inputs, copied exactly: from the first batch's
    // registers when they are all of them, else read again
    const int nin = min(T, p.L);
    if (T <= CB && T <= p.L) {
#pragma unroll
        for (int u = 0; u < CB; ++u)
            if (u < T) IO::st(W + (int64_t)(kept + u) * p.C, x0[u]);
        return;
    }
    const ET* xs = x + (int64_t)(T - nin) * p.C;
    for (int e0 = 0; e0 < nin; e0 += CB) {
        R v[CB];
#pragma unroll
        for (int u = 0; u < CB; ++u) v[u] = IO::ld(xs + (int64_t)min(e0 + u, nin - 1) * p.C);
#pragma unroll
        for (int u = 0; u < CB; ++u)
            if (e0 + u < nin) IO::st(W + (int64_t)(kept + e0 + u) * p.C, v[u]);
    }
}
#undef KWR

}  // namespace kda
