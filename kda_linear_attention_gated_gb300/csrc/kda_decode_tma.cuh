// KDA decode step, one CTA per tile, the tile staged by TMA (sm_103a).
//
// Work unit ("tile"): one (request n, value head h, block of BV state columns)
// with all K rows.  Columns are independent in this recurrence, so a tile needs
// nothing from other tiles.  BV * sizeof(state) is 128, 64 or 32 bytes: one
// TMA box row, one swizzle span.
//
// A CTA owns one tile.  Thread 0 starts one 3-D tensor-map load of the state
// tile and 1-D bulk copies of the q, k and a rows and the tile's slice of v
// into shared memory, all completing on one barrier.  Because the bytes land in
// shared memory rather than registers, a CTA is small in registers and many
// CTAs stay resident per SM, so the SM keeps a deep queue of state bytes in
// flight while the hardware scheduler overlaps loading CTAs with computing
// ones.  Then all threads work the tile:
//   (1) gates: thread i < K turns row i's inputs into khat_i, qhat_i, alpha_i
//       (the norms of k and q are a block reduction);
//   (2) thread (row group rg, 16-byte column chunk cl) reads rows rg, rg + RG,
//       ... of its chunk from shared memory, decays them and accumulates
//       u = S^T khat and p = S^T qhat; warp shuffles and one shared-memory pass
//       finish the sums over K;
//   (3) it reads its rows again, applies the delta update and writes them back
//       to the slot with coalesced 16-byte stores.
// The stage barrier wait is bounded (1 s); a wait that runs out makes the whole
// CTA record KDA_ERR_TIMEOUT, wait once more (bounded) for its copies, and exit.
//
// Math per tile (ROCm/ATOM pull requests 2130 "What", 2945 "Summary"):
//   khat = k / sqrt(|k|^2 + eps), qhat likewise; beta = 1 / (1 + e^-b)
//   alpha_i = exp(-softplus(a_i)) = 1 / (1 + e^{a_i})
//   x_ij = alpha_i S_ij;  u_j = sum_i x_ij khat_i;  p_j = sum_i x_ij qhat_i
//   S'_ij = x_ij + beta khat_i (v_j - u_j)
//   o_j = (p_j + beta (qhat . khat)(v_j - u_j)) / sqrt(K)   (= sum_i S'_ij qhat_i / sqrt(K))
#pragma once

#include "kda_common.cuh"

namespace kda {

template <typename ST, int BV, int NT>
struct DecodeShape {
    static constexpr int VEC = StateVec<ST>::VEC;
    static constexpr int ROWBYTES = BV * (int)sizeof(ST);
    static constexpr int CL = ROWBYTES / 16;     // 16-byte column chunks per row
    static constexpr int RG = NT / CL;           // row groups
    static constexpr int ROWS = KMAX / RG;       // rows per thread
    static constexpr int NWARP = NT / 32;
    static constexpr uint32_t TILE_BYTES = (KMAX * ROWBYTES + 1023u) & ~1023u;
    // input area: q row, k row (any q/k/v type, <= 4 bytes), a row (fp32), v slice
    static constexpr uint32_t IN_Q = 0, IN_K = KMAX * 4, IN_A = 2 * KMAX * 4, IN_V = 3 * KMAX * 4;
    static constexpr uint32_t IN_BYTES = (IN_V + BV * 4 + 127u) & ~127u;
    // gates: float4 {khat, qhat, alpha, 0} per row, then v (fp32)
    static constexpr uint32_t GATE_BYTES = KMAX * 16 + BV * 4;
    static constexpr uint32_t RED_BYTES = NWARP * 4 * 4 + NWARP * CL * 2 * VEC * 4;
    static_assert(ROWBYTES == 128 || ROWBYTES == 64 || ROWBYTES == 32, "tile row bytes");
    static_assert(NT % 32 == 0 && NT >= KMAX && RG * CL == NT && KMAX % RG == 0, "thread shape");
    static_assert(32 % CL == 0, "a warp holds whole rows");
    static_assert(IN_BYTES % 128 == 0 && GATE_BYTES % 16 == 0 && RED_BYTES % 16 == 0, "layout");
};

template <typename ST, int BV, int NT>
constexpr size_t decode_smem_bytes() {
    using SH = DecodeShape<ST, BV, NT>;
    // alignment slack, the tile, inputs, gates, reductions, one barrier
    return 1024 + SH::TILE_BYTES + SH::IN_BYTES + SH::GATE_BYTES + SH::RED_BYTES + 16;
}

template <typename ST, typename QT, int BV, int NT, int MINB>
__global__ void __launch_bounds__(NT, MINB)
kda_decode_kernel(const __grid_constant__ CUtensorMap tmap, const StepParams p) {
    using SH = DecodeShape<ST, BV, NT>;
    using SV = StateVec<ST>;
    constexpr int VEC = SH::VEC, CL = SH::CL, RG = SH::RG, ROWS = SH::ROWS, NWARP = SH::NWARP;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);  // swizzle period
    uint8_t* in = smem + SH::TILE_BYTES;
    float4* gates = reinterpret_cast<float4*>(in + SH::IN_BYTES);
    float* gv = reinterpret_cast<float*>(gates + KMAX);
    float* red = gv + BV;          // [NWARP][4]
    float* red2 = red + NWARP * 4;  // [NWARP][CL][2 VEC]
    uint64_t* full = reinterpret_cast<uint64_t*>(red2 + NWARP * CL * 2 * VEC);
    const uint32_t tile_base = smem_u32(smem);
    const uint32_t gate_base = smem_u32(gates);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cl = tid % CL, rg = tid / CL;
    const int vt = (p.v + BV - 1) / BV;
    const int cb = blockIdx.x % vt;
    const int64_t r = blockIdx.x / vt;  // n * hv + h
    const int h = (int)(r % p.hv);
    const int n = (int)(r / p.hv);
    const int col0 = cb * BV + cl * VEC;
    const int qes = (int)sizeof(QT);

    // The next kernel on the stream may be scheduled now.  Nothing the previous
    // kernel may write is read before it completes, except -- when the caller
    // vouches for it (KDA_LAUNCH_PDL_EARLY_STATE) -- the slot id and the state
    // tile, which then stream while that kernel drains.
    cudaTriggerProgrammaticLaunchCompletion();
    const bool early = (p.flags & LAUNCH_PDL_EARLY_STATE) != 0;
    if (!early) cudaGridDependencySynchronize();

    const int32_t slot = p.init_slot[n];
    const bool valid = slot >= 0 && slot < p.num_slots;
    const bool rst = valid && p.reset != nullptr && p.reset[n] != 0;
    if (tid == 0) {
        mbar_init(full, 1);
        fence_mbar_init();
        if (valid && !rst) {
            prefetch_tmap(&tmap);
            mbar_expect_tx(full, (uint32_t)p.k * SH::ROWBYTES);
            tma_load_3d(smem, &tmap, full, cb * BV, h * p.k, slot);
        }
    }
    if (early) cudaGridDependencySynchronize();
    if (!valid) {
        if (tid == 0) atomicCAS(p.status, 0, STATUS_SLOT_RANGE);
        return;  // uniform over the CTA; nothing was issued
    }
    if (tid == 0) {
        const uint32_t qk_bytes = (uint32_t)p.k * qes;
        const uint32_t v_bytes = (uint32_t)min(BV, p.v - cb * BV) * qes;
        mbar_arrive_expect_tx(full, 2 * qk_bytes + (uint32_t)p.k * 4 + v_bytes);
        bulk_load(in + SH::IN_Q, static_cast<const char*>(p.q) + r * qk_bytes, qk_bytes, full);
        bulk_load(in + SH::IN_K, static_cast<const char*>(p.kk) + r * qk_bytes, qk_bytes, full);
        bulk_load(in + SH::IN_A, p.a + r * p.k, (uint32_t)p.k * 4, full);
        bulk_load(in + SH::IN_V, static_cast<const char*>(p.vv) + (r * p.v + (int64_t)cb * BV) * qes,
                  v_bytes, full);
    }
    const float b = __ldg(p.b + r);
    __syncthreads();  // the barrier is initialised before anyone waits on it
    const bool ok = mbar_wait(full, 0);

    // (1) gates: thread tid < K owns row tid.
    float kt = 0.f, qt = 0.f, alpha = 0.f;
    if (ok && tid < p.k) {
        kt = to_f32(reinterpret_cast<const QT*>(in + SH::IN_K)[tid]);
        qt = to_f32(reinterpret_cast<const QT*>(in + SH::IN_Q)[tid]);
        alpha = 1.0f / (1.0f + expf(reinterpret_cast<const float*>(in + SH::IN_A)[tid]));  // exp(-softplus(a))
    }
    float kk2 = warp_sum(kt * kt), qq2 = warp_sum(qt * qt), kq = warp_sum(kt * qt);
    if (lane == 0) {
        red[warp * 4 + 0] = kk2;
        red[warp * 4 + 1] = qq2;
        red[warp * 4 + 2] = kq;
    }
    if (__syncthreads_or(ok ? 0 : 1)) {  // the copies did not land in time: give up
        if (tid == 0) {
            atomicExch(p.status, STATUS_TIMEOUT);
            mbar_wait(full, 0);  // bounded: no copy may still target this CTA's memory
        }
        return;
    }
    kk2 = 0.f;
    qq2 = 0.f;
    kq = 0.f;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
        kk2 += red[w * 4 + 0];
        qq2 += red[w * 4 + 1];
        kq += red[w * 4 + 2];
    }
    const float rk = 1.0f / sqrtf(kk2 + L2_EPS);
    const float rq = 1.0f / sqrtf(qq2 + L2_EPS);
    const float beta = 1.0f / (1.0f + expf(-b));  // sigmoid(b)
    const float bqk = beta * (kq * rk * rq);       // beta (qhat . khat)
    if (tid < p.k) gates[tid] = make_float4(kt * rk, qt * rq, alpha, 0.f);
    if (tid < BV) {
        const int vcols = min(BV, p.v - cb * BV);
        gv[tid] = tid < vcols ? to_f32(reinterpret_cast<const QT*>(in + SH::IN_V)[tid]) : 0.f;
    }
    __syncthreads();

    // (2) decay and the partial sums over this thread's rows.
    float u[VEC], pp[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) { u[c] = 0.f; pp[c] = 0.f; }
    if (!rst) {
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            const int row = rg + RG * rr;
            if (row < p.k) {
                float x[VEC];
                SV::widen(lds128(tile_base + swz<SH::ROWBYTES>(row, cl)), x);
                const uint4 g = lds128(gate_base + row * 16);
                const float kh = __uint_as_float(g.x), qh = __uint_as_float(g.y), al = __uint_as_float(g.z);
#pragma unroll
                for (int c = 0; c < VEC; ++c) {
                    x[c] *= al;
                    u[c] = fmaf(x[c], kh, u[c]);
                    pp[c] = fmaf(x[c], qh, pp[c]);
                }
            }
        }
    }
    // sum over the row groups of this warp (lanes that share cl) ...
#pragma unroll
    for (int off = CL; off < 32; off <<= 1) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            u[c] += __shfl_xor_sync(0xffffffffu, u[c], off);
            pp[c] += __shfl_xor_sync(0xffffffffu, pp[c], off);
        }
    }
    if (lane < CL) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            red2[(warp * CL + cl) * 2 * VEC + c] = u[c];
            red2[(warp * CL + cl) * 2 * VEC + VEC + c] = pp[c];
        }
    }
    __syncthreads();
    // ... then over the warps.
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
        float su = 0.f, sp = 0.f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) {
            su += red2[(w * CL + cl) * 2 * VEC + c];
            sp += red2[(w * CL + cl) * 2 * VEC + VEC + c];
        }
        u[c] = gv[cl * VEC + c] - su;  // d_j = v_j - u_j
        pp[c] = sp;
    }
    if (col0 >= p.v) return;
    if (rg == 0) {
        float* o = p.o + r * p.v + col0;
#pragma unroll
        for (int c = 0; c < VEC; ++c) o[c] = fmaf(bqk, u[c], pp[c]) * p.inv_sqrt_k;
    }

    // (3) the delta update, stored in place with coalesced 16-byte stores.
    ST* dst = static_cast<ST*>(p.pool) + state_at(p, slot, h) + col0;
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) {
        const int row = rg + RG * rr;
        if (row < p.k) {
            float x[VEC];
            if (!rst) {
                SV::widen(lds128(tile_base + swz<SH::ROWBYTES>(row, cl)), x);
            } else {
#pragma unroll
                for (int c = 0; c < VEC; ++c) x[c] = 0.f;
            }
            const uint4 g = lds128(gate_base + row * 16);
            const float bk = beta * __uint_as_float(g.x), al = __uint_as_float(g.z);
#pragma unroll
            for (int c = 0; c < VEC; ++c) x[c] = fmaf(bk, u[c], x[c] * al);
            __stcs(reinterpret_cast<uint4*>(dst + (int64_t)row * p.v), SV::narrow(x));
        }
    }
}

}  // namespace kda
