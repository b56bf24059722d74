// KDA gated delta-rule state update: device code for sm_103a.
//
// One CTA owns one (request, value head, column tile of BV state columns).
// The state of a head is [K][V] with V innermost, so a column tile is K rows
// of BV contiguous elements; columns are independent in this recurrence (the
// reductions u = S^T k and S^T q run over K, down a column), so a CTA needs
// nothing from its neighbours.  Each thread owns VEC = 16 / sizeof(state)
// adjacent columns of ROWS rows and moves them as one 16-byte vector per row,
// so a warp's row segment is a run of full 32-byte sectors.
//
// Per token (KDA decode step; ROCm/ATOM pull requests 2130 "What" and 2945
// "Summary"):
//   khat, qhat  L2-normalised k, q (block reduction over K)
//   alpha_i = exp(-softplus(a_i)) = 1 / (1 + e^{a_i});  beta = 1 / (1 + e^{-b})
//   x = alpha_i S_ij                                  (decay, in registers)
//   u_j = sum_i x_ij khat_i,  p_j = sum_i x_ij qhat_i (in-thread, then shuffles
//                                                      over the warp's row groups,
//                                                      then shared memory)
//   S'_ij = x_ij + beta khat_i (v_j - u_j)
//   o_j = (p_j + beta (qhat . khat)(v_j - u_j)) / sqrt(K)
// The last line equals sum_i S'_ij qhat_i / sqrt(K) exactly in real arithmetic
// (expand S'), so one reduction pass serves both u and o and the state is read
// once and written once per launch.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kda {

constexpr int KMAX = 128;        // largest K (and V) a launch accepts
constexpr float L2_EPS = 1e-6f;  // L2-norm epsilon: x / sqrt(sum x^2 + eps)
constexpr int32_t STATUS_SLOT_RANGE = 8;  // KDA_ERR_SLOT_RANGE in kda.h

struct StepParams {
    void* pool;               // state pool base (fp32 or fp16 by build)
    int64_t num_slots;
    int64_t slot_stride;      // elements
    int hv, k, v;
    int n, t;                 // requests, tokens per request (1 for decode)
    const int32_t* init_slot; // [n]
    const int32_t* snap_slot; // [n][t], or nullptr: write back in place
    const uint8_t* reset;     // [n] or nullptr
    const void* q;            // [n][t][hv][k]
    const void* kk;           // [n][t][hv][k]
    const void* vv;           // [n][t][hv][v]
    const float* a;           // [n][t][hv][k]
    const float* b;           // [n][t][hv]
    float* o;                 // [n][t][hv][v]
    int32_t* status;
    float inv_sqrt_k;
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// A 16-byte vector of state elements <-> fp32 registers.
template <typename ST> struct StateVec;

template <> struct StateVec<float> {
    static constexpr int VEC = 4;
    static __device__ __forceinline__ void widen(const uint4& r, float (&x)[VEC]) {
        x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z); x[3] = __uint_as_float(r.w);
    }
    static __device__ __forceinline__ uint4 narrow(const float (&x)[VEC]) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                          __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
};

template <> struct StateVec<__half> {
    static constexpr int VEC = 8;
    static __device__ __forceinline__ float2 w2(uint32_t u) {
        __half2 h = *reinterpret_cast<const __half2*>(&u);
        return __half22float2(h);  // exact: every fp16 value is an fp32 value
    }
    static __device__ __forceinline__ uint32_t n2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    static __device__ __forceinline__ void widen(const uint4& r, float (&x)[VEC]) {
        float2 f;
        f = w2(r.x); x[0] = f.x; x[1] = f.y;
        f = w2(r.y); x[2] = f.x; x[3] = f.y;
        f = w2(r.z); x[4] = f.x; x[5] = f.y;
        f = w2(r.w); x[6] = f.x; x[7] = f.y;
    }
    static __device__ __forceinline__ uint4 narrow(const float (&x)[VEC]) {
        return make_uint4(n2(x[0], x[1]), n2(x[2], x[3]), n2(x[4], x[5]), n2(x[6], x[7]));
    }
};

// state_at(slot, h): the one address function for every state access
// (ROCm/ATOM pull request 2945, Changes), in elements from the pool base.
__device__ __forceinline__ int64_t state_at(const StepParams& p, int64_t slot, int h) {
    return slot * p.slot_stride + (int64_t)h * p.k * p.v;
}

template <typename ST, typename QT, int BV, int NT, bool VERIFY>
__global__ void __launch_bounds__(NT) kda_step_kernel(const StepParams p) {
    using SV = StateVec<ST>;
    constexpr int VEC = SV::VEC;
    constexpr int CL = BV / VEC;          // threads across the tile's columns
    constexpr int RG = NT / CL;           // row groups
    constexpr int ROWS = (KMAX + RG - 1) / RG;
    constexpr int NWARP = NT / 32;
    static_assert(BV % VEC == 0 && CL >= 1 && CL <= 32 && (32 % CL) == 0, "bad BV");
    static_assert(NT % 32 == 0 && NT >= KMAX, "one thread per key channel");

    __shared__ float s_kh[KMAX], s_qh[KMAX], s_al[KMAX];
    __shared__ float s_red[3][NWARP];
    __shared__ float s_up[NWARP][CL][2 * VEC];

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int cl = tid % CL, rg = tid / CL;
    const int vt = (p.v + BV - 1) / BV;
    int64_t bid = blockIdx.x;
    const int tile = (int)(bid % vt);
    bid /= vt;
    const int h = (int)(bid % p.hv);
    const int n = (int)(bid / p.hv);
    const int j0 = tile * BV + cl * VEC;
    const bool col_ok = j0 < p.v;   // V % 16 == 0 and VEC | 16: a vector is all in or all out

    // Slot ids: out of range -> record, skip this tile (uniform over the CTA).
    const int T = VERIFY ? p.t : 1;
    const int32_t slot = p.init_slot[n];
    bool bad = slot < 0 || slot >= p.num_slots;
    if (VERIFY) {
        for (int t = 0; t < T; ++t) {
            const int32_t s = p.snap_slot[(int64_t)n * p.t + t];
            bad |= (s < 0 || s >= p.num_slots);
        }
    }
    if (bad) {
        if (tid == 0) atomicCAS(p.status, 0, STATUS_SLOT_RANGE);
        return;
    }
    const bool rst = p.reset != nullptr && p.reset[n] != 0;
    const int64_t col_off = (int64_t)h * p.k * p.v + j0;

    const QT* q = static_cast<const QT*>(p.q);
    const QT* kv = static_cast<const QT*>(p.kk);
    const QT* vv = static_cast<const QT*>(p.vv);

    // Token 0's small inputs first, so their latency overlaps the state stream.
    int64_t row_nt = ((int64_t)n * T) * p.hv + h;  // index into [n][t][hv]
    float ki = 0.f, qi = 0.f, ai = 0.f, bt = 0.f;
    float vj[VEC];
    auto load_small = [&](int64_t r) {
        if (tid < p.k) {
            ki = to_f32(kv[r * p.k + tid]);
            qi = to_f32(q[r * p.k + tid]);
            ai = __ldg(p.a + r * p.k + tid);
        }
        bt = __ldg(p.b + r);
#pragma unroll
        for (int c = 0; c < VEC; ++c) vj[c] = col_ok ? to_f32(vv[r * p.v + j0 + c]) : 0.f;
    };
    load_small(row_nt);

    // The state tile: one 16-byte streaming load per owned row, all in flight.
    float x[ROWS][VEC];
    {
        const ST* src = static_cast<const ST*>(p.pool) + state_at(p, slot, 0) + col_off;
        uint4 raw[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int row = rg + r * RG;
            if (!rst && col_ok && row < p.k)
                raw[r] = __ldcs(reinterpret_cast<const uint4*>(src + (int64_t)row * p.v));
            else
                raw[r] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) SV::widen(raw[r], x[r]);
    }

    for (int t = 0; t < T; ++t) {
        // L2 norms of k and q, and k.q, over the K channels.
        float kk2 = ki * ki, qq2 = qi * qi, kq = ki * qi;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            kk2 += __shfl_xor_sync(0xffffffffu, kk2, off);
            qq2 += __shfl_xor_sync(0xffffffffu, qq2, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }
        if (lane == 0) { s_red[0][warp] = kk2; s_red[1][warp] = qq2; s_red[2][warp] = kq; }
        __syncthreads();
        kk2 = 0.f; qq2 = 0.f; kq = 0.f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) { kk2 += s_red[0][w]; qq2 += s_red[1][w]; kq += s_red[2][w]; }
        const float rk = 1.0f / sqrtf(kk2 + L2_EPS);
        const float rq = 1.0f / sqrtf(qq2 + L2_EPS);
        const float qk = kq * rk * rq;                 // qhat . khat
        const float beta = 1.0f / (1.0f + expf(-bt));  // sigmoid(b)
        if (tid < p.k) {
            s_kh[tid] = ki * rk;
            s_qh[tid] = qi * rq;
            s_al[tid] = 1.0f / (1.0f + expf(ai));      // exp(-softplus(a))
        }
        float vt_[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) vt_[c] = vj[c];
        __syncthreads();

        // Next token's small inputs, in flight during this token's math.
        if (VERIFY && t + 1 < T) load_small(row_nt + p.hv);

        // Decay and the two partial reductions over this thread's rows.
        float u[VEC], pp[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) { u[c] = 0.f; pp[c] = 0.f; }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int row = rg + r * RG;
            if (row < p.k) {
                const float al = s_al[row], kh = s_kh[row], qh = s_qh[row];
#pragma unroll
                for (int c = 0; c < VEC; ++c) {
                    x[r][c] *= al;
                    u[c] = fmaf(x[r][c], kh, u[c]);
                    pp[c] = fmaf(x[r][c], qh, pp[c]);
                }
            }
        }
        // Sum over the row groups of the warp (lanes that share cl) ...
#pragma unroll
        for (int off = CL; off < 32; off <<= 1) {
#pragma unroll
            for (int c = 0; c < VEC; ++c) {
                u[c] += __shfl_xor_sync(0xffffffffu, u[c], off);
                pp[c] += __shfl_xor_sync(0xffffffffu, pp[c], off);
            }
        }
        // ... then over the warps.
        if (lane < CL) {
#pragma unroll
            for (int c = 0; c < VEC; ++c) { s_up[warp][cl][c] = u[c]; s_up[warp][cl][VEC + c] = pp[c]; }
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            float su = 0.f, sp = 0.f;
#pragma unroll
            for (int w = 0; w < NWARP; ++w) { su += s_up[w][cl][c]; sp += s_up[w][cl][VEC + c]; }
            u[c] = vt_[c] - su;  // d_j = v_j - u_j
            pp[c] = sp;
        }

        if (rg == 0 && col_ok) {
            float* o = p.o + row_nt * p.v + j0;
#pragma unroll
            for (int c = 0; c < VEC; ++c) o[c] = fmaf(beta * qk, u[c], pp[c]) * p.inv_sqrt_k;
        }

        // Delta update and the store (snapshot slot per token, or in place).
        const bool store = VERIFY || (t == T - 1);
        ST* dst = nullptr;
        if (store) {
            const int64_t s = VERIFY ? p.snap_slot[(int64_t)n * T + t] : slot;
            dst = static_cast<ST*>(p.pool) + state_at(p, s, 0) + col_off;
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int row = rg + r * RG;
            if (row < p.k) {
                const float bk = beta * s_kh[row];
#pragma unroll
                for (int c = 0; c < VEC; ++c) x[r][c] = fmaf(bk, u[c], x[r][c]);
                if (store && col_ok)
                    __stcs(reinterpret_cast<uint4*>(dst + (int64_t)row * p.v), SV::narrow(x[r]));
            }
        }
        row_nt += p.hv;
        if (VERIFY && t + 1 < T) __syncthreads();  // s_kh/s_qh/s_al/s_red are rewritten next token
    }
}

}  // namespace kda
