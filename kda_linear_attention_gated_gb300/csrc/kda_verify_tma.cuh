// KDA speculative verify, one CTA per tile, the tile staged by TMA (sm_103a).
//
// Tile: one (request n, value head h, block of BV state columns) with all K
// rows; BV * sizeof(state) is 64 or 128 bytes, one warp per 16-byte column
// chunk.  The state tile is TMA-loaded once from init_slot[n] (or taken as
// zero on reset); lane l of warp w then carries rows l, l+32, l+64, l+96 of
// chunk w in fp32 registers through the T tokens without rounding.  After each
// token the state, rounded to the pool's dtype, is written to a shared-memory
// staging buffer (three in turn) and TMA-stored, as one coalesced box, to that
// token's snapshot slot snap_slot[n][t] (ROCm/ATOM pull request 2945, Changes:
// the state after each token goes to the token's snapshot slot through
// state_at).
//
// The gates do not depend on the state, so they are worked out for a chunk of
// up to TC tokens at once, from inputs bulk-copied into shared memory together
// (q, k, a rows and the tile's v slice of every token): the per-token norms
// and beta by one warp (a lane per token), then per row
//   w_i = alpha_i khat_i,  z_i = alpha_i qhat_i,  alpha_i,  beta khat_i.
// Each token then costs each warp one pass over its registers:
// u_j = sum_i S_ij w_i and p_j = sum_i S_ij z_i reduce over the lanes by
// shuffles; d_j = v_j - u_j; o_j = (p_j + beta (qhat . khat) d_j) / sqrt(K);
// S_ij <- alpha_i S_ij + (beta khat_i) d_j; and one CTA barrier before thread 0
// issues the snapshot's TMA store.
// Barrier waits are bounded (1 s); one that runs out makes the CTA record
// KDA_ERR_TIMEOUT, wait once more (bounded) for its copies, and exit.
#pragma once

#include "kda_common.cuh"

namespace kda {

template <typename ST, int BV, int QES>
struct VerifyShape {
    static constexpr int VEC = StateVec<ST>::VEC;
    static constexpr int ROWBYTES = BV * (int)sizeof(ST);
    static constexpr int NW = ROWBYTES / 16;  // warps, one per 16-byte column chunk
    static constexpr int NT = 32 * NW;
    static constexpr int ROWS = KMAX / 32;    // rows per lane
    static constexpr int TC = 8;              // tokens per chunk of inputs and gates
    static constexpr uint32_t TILE_BYTES = (KMAX * ROWBYTES + 1023u) & ~1023u;
    // per token inputs: q row, k row (QES-byte elements), a row (fp32), v slice
    static constexpr uint32_t IN_Q = 0, IN_K = KMAX * QES, IN_A = 2 * KMAX * QES;
    static constexpr uint32_t IN_V = IN_A + KMAX * 4, IN_TOK = (IN_V + BV * QES + 15u) & ~15u;
    // per token gates: float4 per row, then v (fp32)
    static constexpr uint32_t G_V = KMAX * 16, G_TOK = G_V + BV * 4;
    static constexpr uint32_t IN_BYTES = TC * IN_TOK, GATE_BYTES = TC * G_TOK;
    // the gates overlay the inputs, which are all read into registers first
    static constexpr uint32_t WORK_BYTES = IN_BYTES > GATE_BYTES ? IN_BYTES : GATE_BYTES;
    // staging buffers for the snapshot stores (the state tile's area is the first)
    static constexpr int NSTAGE = 3;
    // norms [TC][NW][4], per-token scalars [TC] float4, snapshot ids [TC]
    static constexpr uint32_t RED_BYTES = TC * NW * 16 + TC * 16 + TC * 4;
    static_assert(ROWBYTES == 128 || ROWBYTES == 64, "tile row bytes");
    static_assert(NT >= KMAX, "one thread per key row in the gate phase");
    static_assert(IN_K % 16 == 0 && IN_A % 16 == 0 && IN_V % 16 == 0 && G_TOK % 16 == 0 &&
                  WORK_BYTES % 16 == 0 && RED_BYTES % 16 == 0, "layout");
};

template <typename ST, int BV, int QES>
constexpr size_t verify_smem_bytes() {
    using SH = VerifyShape<ST, BV, QES>;
    return SH::NSTAGE * SH::TILE_BYTES + SH::WORK_BYTES + SH::RED_BYTES + 16;
}

template <typename ST, typename QT, int BV>
__global__ void __launch_bounds__(VerifyShape<ST, BV, (int)sizeof(QT)>::NT)
kda_verify_kernel(const __grid_constant__ CUtensorMap tmap, const StepParams p) {
    using SH = VerifyShape<ST, BV, (int)sizeof(QT)>;
    using SV = StateVec<ST>;
    constexpr int VEC = SH::VEC, NW = SH::NW, ROWS = SH::ROWS, TC = SH::TC;

    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* ins = smem + SH::NSTAGE * SH::TILE_BYTES;
    uint8_t* gts = ins;  // overlays the inputs once they are in registers
    float* red = reinterpret_cast<float*>(ins + SH::WORK_BYTES);  // [TC][NW][4]
    float4* scal = reinterpret_cast<float4*>(red + TC * NW * 4);  // [TC] {beta, bqk, rk, rq}
    int32_t* snaps = reinterpret_cast<int32_t*>(scal + TC);       // [TC]
    uint64_t* bar_st = reinterpret_cast<uint64_t*>(snaps + TC);
    uint64_t* bar_in = bar_st + 1;
    const uint32_t tile_base = smem_u32(smem);
    const uint32_t gate_base = smem_u32(gts);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = warp;
    const int vt = (p.v + BV - 1) / BV;
    const int tile = (int)blockIdx.x;
    const int r = tile / vt;  // n * hv + h
    const int cb = tile - r * vt;
    const int n = r / p.hv;
    const int h = r - n * p.hv;
    const int col0 = cb * BV + chunk * VEC;
    const int T = p.t;
    const int qes = (int)sizeof(QT);
    const int vcols = min(BV, p.v - cb * BV);
    if ((tile_base & 1023u) != 0) {  // the swizzled tile needs a 1024-byte aligned base
        if (tid == 0) atomicCAS(p.status, 0, STATUS_SMEM_ALIGN);
        return;
    }

    // Programmatic dependent launch: as in the decode kernel, only the slot ids
    // and the state may be read before the previous kernel completes, and only
    // when the caller vouches for it (KDA_LAUNCH_PDL_EARLY_STATE).
    cudaTriggerProgrammaticLaunchCompletion();
    const bool early = (p.flags & LAUNCH_PDL_EARLY_STATE) != 0;
    if (!early) cudaGridDependencySynchronize();

    const int32_t slot = p.init_slot[n];
    bool bad = slot < 0 || slot >= p.num_slots;
    for (int t = lane; t < T; t += 32) {
        const int32_t s = p.snap_slot[(int64_t)n * T + t];
        bad |= (s < 0 || s >= p.num_slots);
    }
    bad = __any_sync(0xffffffffu, bad);  // the same answer in every warp
    const bool rst = !bad && p.reset != nullptr && p.reset[n] != 0;
    if (tid == 0) {
        mbar_init(bar_st, 1);
        mbar_init(bar_in, 1);
        fence_mbar_init();
        if (!bad && !rst) {
            prefetch_tmap(&tmap);
            mbar_arrive_expect_tx(bar_st, (uint32_t)p.k * SH::ROWBYTES);
            tma_load_3d(smem, &tmap, bar_st, cb * BV, h * p.k, slot);
        }
    }
    if (early) cudaGridDependencySynchronize();
    if (bad) {
        if (tid == 0) atomicCAS(p.status, 0, STATUS_SLOT_RANGE);
        return;  // uniform; nothing was issued
    }
    __syncthreads();  // barriers initialised

    const uint32_t qk_bytes = (uint32_t)p.k * qes;
    const uint32_t v_bytes = (uint32_t)vcols * qes;
    float x[ROWS][VEC];
    bool state_in = false;
    bool alive = true;
    int in_phase = 0;
    for (int t0 = 0; t0 < T; t0 += TC) {
        const int tc = min(TC, T - t0);
        // inputs of tokens t0 .. t0 + tc - 1: lane 0 of warp 0 arms the barrier
        // with the whole byte count, then warp 0 issues the 4 tc copies
        if (warp == 0) {
            if (lane == 0)
                mbar_arrive_expect_tx(bar_in, (uint32_t)tc * (2 * qk_bytes + (uint32_t)p.k * 4 + v_bytes));
            __syncwarp();
            for (int c = lane; c < 4 * tc; c += 32) {
                const int j = c >> 2, kind = c & 3;
                const int64_t rt = ((int64_t)n * T + t0 + j) * p.hv + h;
                uint8_t* in = ins + j * SH::IN_TOK;
                if (kind == 0)
                    bulk_load(in + SH::IN_Q, static_cast<const char*>(p.q) + rt * qk_bytes, qk_bytes, bar_in);
                else if (kind == 1)
                    bulk_load(in + SH::IN_K, static_cast<const char*>(p.kk) + rt * qk_bytes, qk_bytes, bar_in);
                else if (kind == 2)
                    bulk_load(in + SH::IN_A, p.a + rt * p.k, (uint32_t)p.k * 4, bar_in);
                else
                    bulk_load(in + SH::IN_V,
                              static_cast<const char*>(p.vv) + (rt * p.v + (int64_t)cb * BV) * qes, v_bytes,
                              bar_in);
            }
        }
        float bt = 0.f;
        if (tid < tc) {
            bt = __ldg(p.b + ((int64_t)n * T + t0 + tid) * p.hv + h);
            snaps[tid] = p.snap_slot[(int64_t)n * T + t0 + tid];
        }
        const bool ok_in = mbar_wait(bar_in, in_phase);
        in_phase ^= 1;

        // (1) row tid of every token: k, q, alpha; partial norms per warp
        float kt[TC], qt[TC], at[TC], vv[TC];
#pragma unroll
        for (int j = 0; j < TC; ++j) {
            kt[j] = 0.f; qt[j] = 0.f; at[j] = 0.f; vv[j] = 0.f;
            if (ok_in && j < tc) {
                const uint8_t* in = ins + j * SH::IN_TOK;
                if (tid < p.k) {
                    kt[j] = to_f32(reinterpret_cast<const QT*>(in + SH::IN_K)[tid]);
                    qt[j] = to_f32(reinterpret_cast<const QT*>(in + SH::IN_Q)[tid]);
                    at[j] = __frcp_rn(1.0f + expf(reinterpret_cast<const float*>(in + SH::IN_A)[tid]));
                }
                if (tid < vcols) vv[j] = to_f32(reinterpret_cast<const QT*>(in + SH::IN_V)[tid]);
            }
        }
#pragma unroll
        for (int j = 0; j < TC; ++j) {
            const float s1 = warp_sum(kt[j] * kt[j]), s2 = warp_sum(qt[j] * qt[j]), s3 = warp_sum(kt[j] * qt[j]);
            if (lane == 0) {
                float* rj = red + (j * NW + warp) * 4;
                rj[0] = s1;
                rj[1] = s2;
                rj[2] = s3;
            }
        }
        if (tid < TC) red[(tid * NW) * 4 + 3] = bt;
        if (__syncthreads_or(ok_in ? 0 : 1)) {
            alive = false;
            break;
        }
        // (2) per-token scalars, a lane per token
        if (warp == 0 && lane < tc) {
            float kk2 = 0.f, qq2 = 0.f, kq = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                kk2 += red[(lane * NW + w) * 4 + 0];
                qq2 += red[(lane * NW + w) * 4 + 1];
                kq += red[(lane * NW + w) * 4 + 2];
            }
            const float rk = __frsqrt_rn(kk2 + L2_EPS), rq = __frsqrt_rn(qq2 + L2_EPS);
            const float beta = __frcp_rn(1.0f + expf(-red[(lane * NW) * 4 + 3]));  // sigmoid(b)
            scal[lane] = make_float4(beta, beta * (kq * rk * rq), rk, rq);
        }
        __syncthreads();
        // (3) gates of row tid for every token (the inputs are dead now)
#pragma unroll
        for (int j = 0; j < TC; ++j) {
            if (j < tc) {
                const float4 sc = scal[j];
                uint8_t* g = gts + j * SH::G_TOK;
                if (tid < p.k) {
                    const float kh = kt[j] * sc.z, qh = qt[j] * sc.w;
                    reinterpret_cast<float4*>(g)[tid] = make_float4(at[j] * kh, at[j] * qh, at[j], sc.x * kh);
                }
                if (tid < BV) reinterpret_cast<float*>(g + SH::G_V)[tid] = vv[j];
            }
        }
        if (!state_in) {  // the initial state, once, while the gates are written
            const bool ok_st = rst || mbar_wait(bar_st, 0);
            if (__syncthreads_or(ok_st ? 0 : 1)) {
                alive = false;
                break;
            }
#pragma unroll
            for (int rr = 0; rr < ROWS; ++rr) {
                const int row = lane + 32 * rr;
                if (!rst && row < p.k) SV::widen(lds128(tile_base + swz<SH::ROWBYTES>(row, chunk)), x[rr]);
                else
#pragma unroll
                    for (int c = 0; c < VEC; ++c) x[rr][c] = 0.f;
            }
            state_in = true;
        } else {
            __syncthreads();
        }

        // (4) the tokens, each warp on its own: no CTA barrier in this loop
        for (int j = 0; j < tc; ++j) {
            const int t = t0 + j;
            const uint32_t gb = gate_base + j * SH::G_TOK;
            const uint8_t* g = gts + j * SH::G_TOK;
            float u[VEC], pp[VEC];
#pragma unroll
            for (int c = 0; c < VEC; ++c) { u[c] = 0.f; pp[c] = 0.f; }
            float al[ROWS], bk[ROWS];
#pragma unroll
            for (int rr = 0; rr < ROWS; ++rr) {
                const int row = lane + 32 * rr;
                al[rr] = 0.f;
                bk[rr] = 0.f;
                if (row < p.k) {
                    const uint4 gq = lds128(gb + row * 16);
                    const float w = __uint_as_float(gq.x), z = __uint_as_float(gq.y);
                    al[rr] = __uint_as_float(gq.z);
                    bk[rr] = __uint_as_float(gq.w);
#pragma unroll
                    for (int c = 0; c < VEC; ++c) {
                        u[c] = fmaf(x[rr][c], w, u[c]);
                        pp[c] = fmaf(x[rr][c], z, pp[c]);
                    }
                }
            }
            // u and p over the 32 lanes: reduce-scatter, then broadcast d
            constexpr int NV = 2 * VEC, SHIFT = (NV == 16) ? 1 : 2;  // lanes per value: 1 << SHIFT
            float rv[NV];
#pragma unroll
            for (int c = 0; c < VEC; ++c) { rv[c] = u[c]; rv[VEC + c] = pp[c]; }
            const float sum = warp_reduce_scatter<NV>(rv, lane);
            const int idx = lane >> SHIFT;  // value this lane holds: u_idx, or p_(idx - VEC)
            const float* gv = reinterpret_cast<const float*>(g + SH::G_V) + chunk * VEC;
            const float dmine = idx < VEC ? gv[idx] - sum : 0.f;  // d_j = v_j - u_j
            float d[VEC];
#pragma unroll
            for (int c = 0; c < VEC; ++c) d[c] = __shfl_sync(0xffffffffu, dmine, c << SHIFT);
            const bool col_ok = col0 < p.v;
            if (idx >= VEC && (lane & ((1 << SHIFT) - 1)) == 0 && col_ok) {
                const int c = idx - VEC;
                float dc = d[0];
#pragma unroll
                for (int e = 1; e < VEC; ++e) dc = (c == e) ? d[e] : dc;
                p.o[(((int64_t)n * T + t) * p.hv + h) * p.v + col0 + c] = fmaf(scal[j].y, dc, sum) * p.inv_sqrt_k;
            }
            // snapshot: stage the rounded rows, then one TMA store of the box
            const int b = t % SH::NSTAGE;
            const uint32_t stage = tile_base + b * SH::TILE_BYTES;
#pragma unroll
            for (int rr = 0; rr < ROWS; ++rr) {
                const int row = lane + 32 * rr;
                if (row < p.k) {
#pragma unroll
                    for (int c = 0; c < VEC; ++c) x[rr][c] = fmaf(al[rr], x[rr][c], bk[rr] * d[c]);
                    sts128(stage + swz<SH::ROWBYTES>(row, chunk), SV::narrow(x[rr]));
                }
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tma_store_3d(&tmap, smem + b * SH::TILE_BYTES, cb * BV, h * p.k, snaps[j]);
                bulk_commit();
                // the store of token t - 1 has read its buffer, which token t + 2 rewrites
                bulk_wait_read<1>();
            }
        }
        // The next chunk's bulk copies (async proxy) overwrite this chunk's
        // gates (generic proxy): fence, then the barrier before they are issued.
        fence_proxy_async_smem();
        __syncthreads();
    }
    if (tid == 0) bulk_wait<0>();
    if (!alive) {
        if (tid == 0) {
            atomicExch(p.status, STATUS_TIMEOUT);
            mbar_wait(bar_in, in_phase ^ 1);  // bounded: no copy may still target this CTA's memory
            if (!rst) mbar_wait(bar_st, 0);
        }
    }
}

}  // namespace kda
