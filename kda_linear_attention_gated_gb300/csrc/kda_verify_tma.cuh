// KDA speculative verify, TMA-staged (sm_103a).
//
// One CTA per tile (request n, value head h, block of BV state columns); one
// warp per 16-byte column chunk, lane l owning rows l, l+32, l+64, l+96, so the
// reductions over K are warp shuffles.  The tile's state is TMA-loaded once
// from init_slot[n] (skipped on reset), carried in fp32 registers across the T
// tokens without rounding, and after each token written, rounded to the pool's
// dtype, into one of three shared-memory snapshot buffers that thread 0
// TMA-stores to snap_slot[n][t] (ROCm/ATOM pull request 2945, Changes: the
// state after each token goes to that token's snapshot slot through state_at).
// Three buffers and one CTA barrier per token: when token t+1 overwrites the
// buffer of token t-2, thread 0 has already seen that store finish reading it
// (bulk wait_group.read before the barrier of token t).
#pragma once

#include "kda_common.cuh"

namespace kda {

template <typename ST, int BV>
struct VerifyTmaShape {
    static constexpr int VEC = StateVec<ST>::VEC;
    static constexpr int ROWBYTES = BV * (int)sizeof(ST);
    static constexpr int NW = ROWBYTES / 16;
    static constexpr int THREADS = 32 * NW;
    static constexpr int ROWS = KMAX / 32;
    static constexpr uint32_t BUF_BYTES = (KMAX * ROWBYTES + 1023u) & ~1023u;
    static constexpr int NBUF = 4;  // 3 snapshot buffers + the load buffer
};

template <typename ST, int BV>
constexpr size_t verify_tma_smem_bytes() {
    using SH = VerifyTmaShape<ST, BV>;
    return 1024 + (size_t)SH::NBUF * SH::BUF_BYTES + 16;
}

template <typename ST, typename QT, int BV>
__global__ void __launch_bounds__(VerifyTmaShape<ST, BV>::THREADS)
kda_verify_tma_kernel(const __grid_constant__ CUtensorMap tmap, const StepParams p) {
    using SH = VerifyTmaShape<ST, BV>;
    using SV = StateVec<ST>;
    constexpr int VEC = SH::VEC;
    constexpr int ROWS = SH::ROWS;
    constexpr uint32_t BUF_BYTES = SH::BUF_BYTES;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SH::NBUF * BUF_BYTES);
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t load_buf = smem_base + 3 * BUF_BYTES;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk = warp;
    const int vt = (p.v + BV - 1) / BV;
    const int tile = blockIdx.x;
    const int cb = tile % vt;
    const int h = (tile / vt) % p.hv;
    const int n = tile / vt / p.hv;
    const int T = p.t;
    const int col0 = cb * BV + chunk * VEC;

    // The next kernel on the stream may be scheduled now; this grid reads
    // nothing the previous kernel may write before that kernel has completed,
    // except slot ids and the state tile when the caller vouches for them
    // (KDA_LAUNCH_PDL_EARLY_STATE).
    cudaTriggerProgrammaticLaunchCompletion();
    const bool early = (p.flags & LAUNCH_PDL_EARLY_STATE) != 0;
    if (!early) cudaGridDependencySynchronize();

    // Slot ids (uniform over the CTA): any out of range -> record and skip.
    const int32_t slot = p.init_slot[n];
    bool bad = slot < 0 || slot >= p.num_slots;
    for (int t = 0; t < T; ++t) {
        const int32_t s = p.snap_slot[(int64_t)n * T + t];
        bad |= (s < 0 || s >= p.num_slots);
    }
    const bool rst = !bad && p.reset != nullptr && p.reset[n] != 0;
    if (bad) {
        if (early) cudaGridDependencySynchronize();
        if (threadIdx.x == 0) atomicCAS(p.status, 0, STATUS_SLOT_RANGE);
        return;
    }

    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        fence_mbar_init();
        if (!rst) {
            prefetch_tmap(&tmap);
            mbar_arrive_expect_tx(full, (uint32_t)p.k * SH::ROWBYTES);
            tma_load_3d(smem + 3 * BUF_BYTES, &tmap, full, cb * BV, h * p.k, slot);
        }
    }
    if (early) cudaGridDependencySynchronize();

    const QT* qp = static_cast<const QT*>(p.q);
    const QT* kp = static_cast<const QT*>(p.kk);
    const QT* vp = static_cast<const QT*>(p.vv);
    struct Small {
        float k[ROWS], q[ROWS], a[ROWS], v[VEC], b;
    };
    auto load_small = [&](int t, Small& sm) {
        const int64_t r = ((int64_t)n * T + t) * p.hv + h;
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            const int row = lane + 32 * rr;
            const bool ok = row < p.k;
            sm.k[rr] = ok ? to_f32(kp[r * p.k + row]) : 0.f;
            sm.q[rr] = ok ? to_f32(qp[r * p.k + row]) : 0.f;
            sm.a[rr] = ok ? __ldg(p.a + r * p.k + row) : 0.f;
        }
#pragma unroll
        for (int c = 0; c < VEC; ++c) sm.v[c] = col0 < p.v ? to_f32(vp[r * p.v + col0 + c]) : 0.f;
        sm.b = __ldg(p.b + r);
    };
    Small cur, nxt;
    load_small(0, cur);
    __syncthreads();  // barrier initialised before anyone waits on it

    float x[ROWS][VEC];
    if (!rst) {
        if (!mbar_wait(full, 0)) {
            if (lane == 0) atomicExch(p.status, STATUS_TIMEOUT);
            // every thread waits once more (bounded) so no copy is left in flight
            mbar_wait(full, 0);
            return;
        }
    }
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
        const int row = lane + 32 * rr;
        if (row < p.k && !rst) {
            SV::widen(lds128(load_buf + swz<SH::ROWBYTES>(row, chunk)), x[rr]);
        } else {
#pragma unroll
            for (int c = 0; c < VEC; ++c) x[rr][c] = 0.f;
        }
    }

    for (int t = 0; t < T; ++t) {
        if (t + 1 < T) load_small(t + 1, nxt);
        const int64_t r = ((int64_t)n * T + t) * p.hv + h;
        float kk2 = 0.f, qq2 = 0.f, kq = 0.f;
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            kk2 = fmaf(cur.k[rr], cur.k[rr], kk2);
            qq2 = fmaf(cur.q[rr], cur.q[rr], qq2);
            kq = fmaf(cur.k[rr], cur.q[rr], kq);
        }
        kk2 = warp_sum(kk2);
        qq2 = warp_sum(qq2);
        kq = warp_sum(kq);
        const float rk = 1.0f / sqrtf(kk2 + L2_EPS);
        const float rq = 1.0f / sqrtf(qq2 + L2_EPS);
        const float beta = 1.0f / (1.0f + expf(-cur.b));
        const float bqk = beta * (kq * rk * rq);
        float kh[ROWS], qh[ROWS];
        float u[VEC], pp[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) { u[c] = 0.f; pp[c] = 0.f; }
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            kh[rr] = cur.k[rr] * rk;
            qh[rr] = cur.q[rr] * rq;
            const float al = 1.0f / (1.0f + expf(cur.a[rr]));  // exp(-softplus(a))
#pragma unroll
            for (int c = 0; c < VEC; ++c) {
                x[rr][c] *= al;
                u[c] = fmaf(x[rr][c], kh[rr], u[c]);
                pp[c] = fmaf(x[rr][c], qh[rr], pp[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            u[c] = cur.v[c] - warp_sum(u[c]);  // d_j = v_j - u_j
            pp[c] = warp_sum(pp[c]);
        }
        if (lane == 0 && col0 < p.v) {
            float* o = p.o + r * p.v + col0;
#pragma unroll
            for (int c = 0; c < VEC; ++c) o[c] = fmaf(bqk, u[c], pp[c]) * p.inv_sqrt_k;
        }
        const uint32_t buf = smem_base + (t % 3) * BUF_BYTES;
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            const int row = lane + 32 * rr;
            const float bk = beta * kh[rr];
#pragma unroll
            for (int c = 0; c < VEC; ++c) x[rr][c] = fmaf(bk, u[c], x[rr][c]);
            if (row < p.k) sts128(buf + swz<SH::ROWBYTES>(row, chunk), SV::narrow(x[rr]));
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            const int32_t snap = p.snap_slot[(int64_t)n * T + t];
            tma_store_3d(&tmap, smem + (t % 3) * BUF_BYTES, cb * BV, h * p.k, snap);
            bulk_commit();
            bulk_wait_read<1>();  // the store of token t-1 has read its buffer
        }
        cur = nxt;
    }
    if (threadIdx.x == 0) bulk_wait<0>();
}

}  // namespace kda
