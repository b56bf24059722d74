// KDA decode step, one CTA per one or two tiles, staged by TMA (sm_103a).
//
// Work unit ("tile"): one (request n, value head h, block of BV state columns)
// with all K rows.  Columns are independent in this recurrence, so a tile needs
// nothing from other tiles.  BV * sizeof(state) is 128, 64 or 32 bytes: one
// TMA box row, one swizzle span.
//
// A CTA owns TPC adjacent tiles of one (request, head): one for an fp32 pool,
// two for an fp16 pool (and for the fused-convolution build on either pool),
// so that an fp16 launch at N = 64 is 768 CTAs, all resident at once (6 per SM
// by shared memory), where one tile per CTA made 1.26 waves of 1536.  Thread 0 starts one 3-D tensor-map load per state tile,
// each on its own barrier, and 1-D bulk copies of the q, k and a rows and the
// tiles' slices of v into shared memory, completing on one more barrier.
// Because the bytes land in shared memory rather than registers, a CTA is
// small in registers and many CTAs stay resident per SM, so the SM keeps a
// deep queue of state bytes in flight while the hardware scheduler overlaps
// loading CTAs with computing ones.  The gates are worked out once for the
// CTA's tiles; then all threads work each tile in turn:
//   (1) gates: thread i < K turns row i's inputs into khat_i, qhat_i, alpha_i
//       (the norms of k and q are a block reduction);
//   (2) thread (row group rg, 16-byte column chunk cl) reads rows rg, rg + RG,
//       ... of its chunk from shared memory and accumulates u = S^T (alpha khat)
//       and p = S^T (alpha qhat) (the decay folded into the gates); warp
//       shuffles and one shared-memory pass finish the sums over K;
//   (3) it reads its rows from shared memory again (one tile a CTA) or takes
//       their raw 16-byte words, kept in registers since (2) (two tiles a CTA,
//       where shared memory caps residency at 6 CTAs per SM and so leaves room
//       for them), applies the delta update and writes the rows back to the
//       slot with coalesced 16-byte stores.
// The CONV build puts the layer's short convolution in front: q, k and v are
// not copied in but formed from the conv window and the pre-activations x
// (thread i < K: the q and k channels of key row i; thread e < TPC BV: value
// column e), and the window is rewritten; see the conv helpers below and
// step (4) in the kernel.
// The inputs and the state tile complete on separate barriers, so the gates
// are computed while the state is still in flight.  Each barrier wait is
// bounded (1 s); a wait that runs out makes the whole CTA record
// KDA_ERR_TIMEOUT, wait once more (bounded) for its copies, and exit.
//
// The request's slot is column accepted[n] - 1 (or 0) of its row of the slot
// table (init_slot, init_stride); q and k may be shared by groups of value
// heads (hqk heads); with MODE_PADDING a negative slot is a padding request
// whose outputs are zeroed and whose state is left alone.
//
// Math per tile (ROCm/ATOM pull requests 2130 "What", 2945 "Summary"):
//   khat = k / sqrt(|k|^2 + eps), qhat likewise; beta = 1 / (1 + e^-b)
//   alpha_i = exp(-softplus(a_i)) = 1 / (1 + e^{a_i}), or with the layer's
//             learned scale exp(-exp(A_log_h) softplus(a_i + dt_bias_h,i))
//   u_j = sum_i S_ij (alpha_i khat_i);  p_j = sum_i S_ij (alpha_i qhat_i)
//   S'_ij = alpha_i S_ij + (beta khat_i) (v_j - u_j)
//   o_j = (p_j + beta (qhat . khat)(v_j - u_j)) / sqrt(K)   (= sum_i S'_ij qhat_i / sqrt(K))
#pragma once

#include "kda_common.cuh"
#include "kda_conv.cuh"

namespace kda {

// The fused short convolution of a decode step (CONV), one channel, in
// stages.  conv_load: the history entries h_0 .. h_(KW-2) of the window at
// W[i C] (zero on reset), the weights and the bias, into registers.
// conv_apply: bias + sum_i w_i h_i + w_(KW-1) x, SiLU when silu, rounded to
// QT: the same fmaf chain in the same order as the conv kernel, so y is
// bit-identical to kda_conv_step's.  The loads can go out before the input
// exists and the input's load before any of them returns.
template <typename QT>
__device__ __forceinline__ void conv_load(QT (&h)[DCONV_H], float (&w)[DCONV_H], float& wl, float& b, const QT* W,
                                          int C, int KW, bool rst, const float* wp, bool w4, const float* bias) {
    QT zero;
    conv_round(0.f, zero);
#pragma unroll
    for (int i = 0; i < DCONV_H; ++i) h[i] = !rst && i < KW - 1 ? W[(int64_t)i * C] : zero;
    if (w4) {  // KW = 4: the channel's weights are one 16-byte row
        const float4 v = __ldg(reinterpret_cast<const float4*>(wp));
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        wl = v.w;
    } else {
#pragma unroll
        for (int i = 0; i < DCONV_H; ++i) w[i] = i < KW - 1 ? __ldg(wp + i) : 0.f;
        wl = __ldg(wp + KW - 1);  // the input's weight
    }
    b = bias != nullptr ? __ldg(bias) : 0.f;
}

template <typename QT>
__device__ __forceinline__ QT conv_apply(const QT (&h)[DCONV_H], const float (&w)[DCONV_H], float wl, float b,
                                         int KW, QT xr, int silu) {
    float s = b;
#pragma unroll
    for (int i = 0; i < DCONV_H; ++i)
        if (i < KW - 1) s = fmaf(w[i], to_f32(h[i]), s);
    s = fmaf(wl, to_f32(xr), s);
    QT out;
    conv_round(silu ? silu_fast(s) : s, out);
    return out;
}

// The window of one channel after a one-token step: its last L - 1 history
// entries (h_(KW-L+e) -> entry e; L is KW - 1 or KW; zero on reset) followed
// by the input.  All kept entries are read before any is written; only the
// channel's one writer runs this, after every reader of the old entries has
// read them.
template <typename QT>
__device__ __forceinline__ void conv_window_store_kept(QT* W, int C, int L, int KW, const QT (&hraw)[DCONV_H], QT xr) {
    const bool shift = KW - L == 1;  // else L == KW: entry e keeps h_e (hraw is zero on reset)
#pragma unroll
    for (int e = 0; e < DCONV_H; ++e)
        if (e < L - 1) W[(int64_t)e * C] = shift ? hraw[e + 1 < DCONV_H ? e + 1 : e] : hraw[e];
    if (L >= 1) W[(int64_t)(L - 1) * C] = xr;
}

template <typename QT>
__device__ __forceinline__ void conv_window_store(QT* W, int C, int L, int KW, bool rst, QT xr) {
    const int shift = KW - L;  // 1, or 0 when L == KW (entry e keeps h_e)
    QT zero;
    conv_round(0.f, zero);
    QT keep[DCONV_H];
#pragma unroll
    for (int e = 0; e < DCONV_H; ++e) keep[e] = !rst && e < L - 1 ? W[(int64_t)(e + shift) * C] : zero;
#pragma unroll
    for (int e = 0; e < DCONV_H; ++e)
        if (e < L - 1) W[(int64_t)e * C] = keep[e];
    if (L >= 1) W[(int64_t)(L - 1) * C] = xr;
}

// TPC: tiles per CTA, adjacent column blocks of one (request, value head).
// They share the inputs and the gates, and their state boxes are all in flight
// from the start.
template <typename ST, int BV, int NT, int QES, int TPC = 1>
struct DecodeShape {
    static constexpr int VEC = StateVec<ST>::VEC;
    static constexpr int ROWBYTES = BV * (int)sizeof(ST);
    static constexpr int CL = ROWBYTES / 16;     // 16-byte column chunks per row
    static constexpr int RG = NT / CL;           // row groups
    static constexpr int ROWS = KMAX / RG;       // rows per thread
    static constexpr int NWARP = NT / 32;
    static constexpr uint32_t TILE_BYTES = (KMAX * ROWBYTES + 1023u) & ~1023u;
    // input area: q row, k row (QES-byte elements), a row (fp32), v slice
    static constexpr uint32_t IN_Q = 0, IN_K = KMAX * QES, IN_A = 2 * KMAX * QES;
    static constexpr uint32_t IN_V = IN_A + KMAX * 4, IN_END = IN_V + TPC * BV * QES;
    // gates: float4 {alpha khat, alpha qhat, alpha, beta khat} per row, then v
    // (fp32); they overlay the input area, which is read into registers first
    static constexpr uint32_t GATE_BYTES = KMAX * 16 + TPC * BV * 4;
    static constexpr uint32_t WORK_BYTES = ((IN_END > GATE_BYTES ? IN_END : GATE_BYTES) + 15u) & ~15u;
    // lanes of a warp that share a column chunk, and the values each keeps
    // after the in-warp reduce-scatter of its 2 VEC partial sums
    static constexpr int NL = 32 / CL, KEEPV = 2 * VEC / NL;
    // norms [NWARP][4], partial sums [NWARP][CL][2 VEC], d [BV]
    static constexpr uint32_t RED_BYTES = NWARP * 4 * 4 + NWARP * CL * 2 * VEC * 4 + BV * 4;
    static_assert(ROWBYTES == 128 || ROWBYTES == 64 || ROWBYTES == 32, "tile row bytes");
    static_assert(NT % 32 == 0 && NT >= KMAX && RG * CL == NT && KMAX % RG == 0, "thread shape");
    static_assert(32 % CL == 0, "a warp holds whole rows");
    static_assert(KEEPV >= 1 && (KEEPV == 1 || KEEPV == 2 || KEEPV == 4), "reduce-scatter split");
    static_assert(BV <= NT, "one thread per column in the finishing step");
    static_assert(IN_K % 16 == 0 && IN_A % 16 == 0 && IN_V % 16 == 0 && RED_BYTES % 16 == 0, "layout");
    // rows rg + RG * i share the swizzle XOR term of row rg (patterns repeat every 8 rows of 128 B,
    // 8 rows of 64 B read as pairs, 8 rows of 32 B read as quads: 1024 B in each case)
    static_assert((RG * ROWBYTES) % 1024 == 0, "row stride must span whole swizzle periods");
};

template <typename ST, int BV, int NT, int QES, int TPC = 1>
constexpr size_t decode_smem_bytes() {
    using SH = DecodeShape<ST, BV, NT, QES, TPC>;
    // the tile, inputs/gates, reductions, two barriers (no alignment slack: the
    // dynamic shared memory base is 1024-byte aligned, which the kernel checks)
    return TPC * SH::TILE_BYTES + SH::WORK_BYTES + SH::RED_BYTES + 8 * (TPC + 1);
}

template <typename ST, typename QT, int BV, int NT, int MINB, bool KEEP, bool FULLK, int TPC = 1, bool CONV = false>
__global__ void __launch_bounds__(NT, MINB)
kda_decode_kernel(const __grid_constant__ CUtensorMap tmap, const StepParams p) {
    using SH = DecodeShape<ST, BV, NT, (int)sizeof(QT), TPC>;
    using SV = StateVec<ST>;
    constexpr int VEC = SH::VEC, CL = SH::CL, RG = SH::RG, ROWS = SH::ROWS, NWARP = SH::NWARP;
    constexpr int KEEPV = SH::KEEPV;

    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* in = smem + TPC * SH::TILE_BYTES;
    float4* gates = reinterpret_cast<float4*>(in);  // overlays the inputs once they are read
    float* gv = reinterpret_cast<float*>(gates + KMAX);
    float* red = reinterpret_cast<float*>(in + SH::WORK_BYTES);  // [NWARP][4]
    float* red2 = red + NWARP * 4;                               // [NWARP][CL][2 VEC]
    float* dsm = red2 + NWARP * CL * 2 * VEC;                    // [BV]: d = v - u
    uint64_t* bar_st = reinterpret_cast<uint64_t*>(dsm + BV);    // state tile landed
    uint64_t* bar_in = bar_st + TPC;                                           // inputs landed
    const uint32_t tile_base0 = smem_u32(smem);
    const uint32_t gate_base = smem_u32(gates);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cl = tid % CL, rg = tid / CL;
    // 32-bit index arithmetic: the host guarantees n * hv * ceil(v / BV) < 2^31
    const int vt = (p.v + BV - 1) / BV;
    const int ct = (vt + TPC - 1) / TPC;  // CTAs per (request, head)
    const int tile = (int)blockIdx.x;
    const int r = tile / ct;  // n * hv + h
    const int cb0 = (tile - r * ct) * TPC;  // first column block of this CTA
    const int n = r / p.hv;
    const int h = r - n * p.hv;
    // the fused convolution's q/k head and the CTAs that read its window
    // (value heads sharing it times CTAs per head); formed once
    const int cgrp = CONV ? p.hv / p.hqk : 1;
    const int chq = CONV ? h / cgrp : 0;
    const int qes = (int)sizeof(QT);
    // The swizzled tile needs a 1024-byte aligned base; report, never guess.
    if ((tile_base0 & 1023u) != 0) {
        if (tid == 0) atomicCAS(p.status, 0, STATUS_SMEM_ALIGN);
        return;
    }

    // The next kernel on the stream may be scheduled now.  Nothing the previous
    // kernel may write is read before it completes, except -- when the caller
    // vouches for it (KDA_LAUNCH_PDL_EARLY_STATE) -- the slot id and the state
    // tile, which then stream while that kernel drains.
    cudaTriggerProgrammaticLaunchCompletion();
    const bool early = (p.flags & LAUNCH_PDL_EARLY_STATE) != 0;
    if (!early) cudaGridDependencySynchronize();

    // The request's slot: column accepted[n] - 1 (or 0) of its row of the
    // slot table; a negative slot is padding when the caller says so.
    int col = 0;
    if (p.accepted != nullptr) col = p.accepted[n] - 1;
    const bool col_ok = col >= 0 && col < p.num_cols;
    const int32_t slot = col_ok ? p.init_slot[(int64_t)n * p.init_stride + col] : -1;
    const bool pad = col_ok && slot < 0 && (p.mode & MODE_PADDING) != 0;
    int32_t cslot = 0;  // the fused convolution's window slot
    if constexpr (CONV) cslot = p.conv.slot[n];
    const bool valid = col_ok && slot >= 0 && slot < p.num_slots && (!CONV || (cslot >= 0 && cslot < p.conv.num_slots));
    const bool rst = valid && p.reset != nullptr && p.reset[n] != 0;
    if (tid == 0) {
        for (int j = 0; j <= TPC; ++j) mbar_init(bar_st + j, 1);
        fence_mbar_init();
        if (valid && !rst) {
            prefetch_tmap(&tmap);
            for (int j = 0; j < TPC && (TPC == 1 || cb0 + j < vt); ++j) {
                mbar_arrive_expect_tx(bar_st + j, (uint32_t)p.k * SH::ROWBYTES);
                if (!(p.flags & LAUNCH_TEST_WITHHOLD_STATE))  // the test hook: the wait runs out
                    tma_load_3d(smem + j * SH::TILE_BYTES, &tmap, bar_st + j, (cb0 + j) * BV, h * p.k, slot);
            }
        }
    }
    // (0) the fused convolution (CONV): thread i < K takes the q and k
    // channels of key row i, thread e < TPC BV value column e of the CTA's
    // tiles.  The history entries, weights and bias are nothing the previous
    // kernel writes, so with early reads they are loaded while it drains; the
    // sums are formed once the inputs' loads are out, after the wait.
    constexpr int NVE = (TPC * BV + NT - 1) / NT;  // value columns per thread
    // a value column's history also rewrites its window (this CTA's alone)
    QT hq_[DCONV_H], hk_[DCONV_H], hv_[NVE][DCONV_H];
    float wq_[DCONV_H], wk_[DCONV_H], wv_[NVE][DCONV_H], lq_ = 0.f, lk_ = 0.f, lv_[NVE], bq_ = 0.f, bk_ = 0.f, bv_[NVE];
    if constexpr (CONV) {
        if (valid) {
            const auto& cp = p.conv;
            const QT* W = static_cast<const QT*>(cp.window) + (int64_t)cslot * cp.slot_stride;
            const bool w4 = cp.KW == 4 && (reinterpret_cast<uintptr_t>(cp.w) & 15u) == 0;
            if (tid < p.k) {
                const int qc = chq * p.k + tid, kc = (p.hqk + chq) * p.k + tid;
                conv_load(hq_, wq_, lq_, bq_, W + qc, cp.C, cp.KW, rst, cp.w + (int64_t)qc * cp.KW, w4,
                          cp.bias != nullptr ? cp.bias + qc : nullptr);
                conv_load(hk_, wk_, lk_, bk_, W + kc, cp.C, cp.KW, rst, cp.w + (int64_t)kc * cp.KW, w4,
                          cp.bias != nullptr ? cp.bias + kc : nullptr);
            }
#pragma unroll
            for (int e = 0; e < NVE; ++e) {
                const int c = tid + e * NT, col = cb0 * BV + c;
                if (c < TPC * BV && col < p.v) {
                    const int vc = 2 * p.hqk * p.k + h * p.v + col;
                    conv_load(hv_[e], wv_[e], lv_[e], bv_[e], W + vc, cp.C, cp.KW, rst, cp.w + (int64_t)vc * cp.KW, w4,
                              cp.bias != nullptr ? cp.bias + vc : nullptr);
                }
            }
        }
    }
    if (early) cudaGridDependencySynchronize();
    if (!valid) {
        if (pad) {  // padding: this CTA's outputs are zero
            for (int e = tid; e < min(TPC * BV, p.v - cb0 * BV); e += NT) p.o[(int64_t)r * p.v + cb0 * BV + e] = 0.f;
        } else if (tid == 0) {
            atomicCAS(p.status, 0, col_ok ? STATUS_SLOT_RANGE : STATUS_ARG);
        }
        return;  // uniform over the CTA; nothing was issued
    }
    if (tid == 0) {
        const uint32_t qk_bytes = (uint32_t)p.k * qes;
        const uint32_t v_bytes = (uint32_t)min(TPC * BV, p.v - cb0 * BV) * qes;
        const int64_t r64 = r;
        if constexpr (CONV) {  // q, k and v come from the convolution below
            mbar_arrive_expect_tx(bar_in, (uint32_t)p.k * 4);
        } else {
            mbar_arrive_expect_tx(bar_in, 2 * qk_bytes + (uint32_t)p.k * 4 + v_bytes);
            const int64_t rqk = (int64_t)n * p.hqk + h / (p.hv / p.hqk);  // grouped q/k heads
            bulk_load(in + SH::IN_Q, static_cast<const char*>(p.q) + rqk * qk_bytes, qk_bytes, bar_in);
            bulk_load(in + SH::IN_K, static_cast<const char*>(p.kk) + rqk * qk_bytes, qk_bytes, bar_in);
            bulk_load(in + SH::IN_V, static_cast<const char*>(p.vv) + (r64 * p.v + (int64_t)cb0 * BV) * qes,
                      v_bytes, bar_in);
        }
        bulk_load(in + SH::IN_A, p.a + r64 * p.k, (uint32_t)p.k * 4, bar_in);
    }
    const float b = __ldg(p.b + r);

    // The input terms, once the previous kernel is done: y, and q, k and v
    // for the decode.
    float cq = 0.f, ck = 0.f, cvv[NVE];
#pragma unroll
    for (int e = 0; e < NVE; ++e) cvv[e] = 0.f;
    if constexpr (CONV) {
        const auto& cp = p.conv;
        const QT* X = static_cast<const QT*>(cp.x) + (int64_t)n * cp.C;
        QT* Y = cp.y != nullptr ? static_cast<QT*>(cp.y) + (int64_t)n * cp.C : nullptr;
        const int qc = chq * p.k + tid, kc = (p.hqk + chq) * p.k + tid;  // this row's q and k channels
        QT xq, xk, xv[NVE];
        if (tid < p.k) {
            xq = X[qc];
            xk = X[kc];
        }
#pragma unroll
        for (int e = 0; e < NVE; ++e) {
            const int c = tid + e * NT, col = cb0 * BV + c;
            if (c < TPC * BV && col < p.v) xv[e] = X[2 * p.hqk * p.k + h * p.v + col];
        }
        if (tid < p.k) {
            const QT yq = conv_apply(hq_, wq_, lq_, bq_, cp.KW, xq, cp.silu);
            const QT yk = conv_apply(hk_, wk_, lk_, bk_, cp.KW, xk, cp.silu);
            cq = to_f32(yq);
            ck = to_f32(yk);
            if (Y != nullptr && h % cgrp == 0 && cb0 == 0) {  // one writer of y per q/k channel
                Y[qc] = yq;
                Y[kc] = yk;
            }
            // the only reader of its q/k windows (one CTA a head, one value
            // head a q/k head): rewrite them now, from the registers, as the
            // value columns' are below; no count, no re-read at the end (two
            // tiles a CTA only: the one-tile kernels have no registers to
            // spare and do it at the end)
            if (TPC > 1 && cgrp * ct == 1) {
                QT* W = static_cast<QT*>(cp.window) + (int64_t)cslot * cp.slot_stride;
                conv_window_store_kept(W + qc, cp.C, cp.L, cp.KW, hq_, xq);
                conv_window_store_kept(W + kc, cp.C, cp.L, cp.KW, hk_, xk);
            }
        }
#pragma unroll
        for (int e = 0; e < NVE; ++e) {
            const int c = tid + e * NT, col = cb0 * BV + c;
            if (c < TPC * BV && col < p.v) {
                const int chv = 2 * p.hqk * p.k + h * p.v + col;
                const QT yv = conv_apply(hv_[e], wv_[e], lv_[e], bv_[e], cp.KW, xv[e], cp.silu);
                cvv[e] = to_f32(yv);
                if (Y != nullptr) Y[chv] = yv;
                conv_window_store_kept(static_cast<QT*>(cp.window) + (int64_t)cslot * cp.slot_stride + chv, cp.C,
                                       cp.L, cp.KW, hv_[e], xv[e]);
            }
        }
    }
    // (4) the fused convolution's q/k window update, the last thing the CTA
    // does (all threads together).  A q/k channel's window is read by every
    // CTA of the request's value heads that share the q/k head: each counts
    // its read once its threads have used the values (they fed the gates,
    // before a barrier; thread 0 counts right after it and keeps the old
    // count, prev, for here), and the one that makes the count complete
    // writes the new entries and puts the count back to zero.  No CTA waits
    // for another.  prev < 0: not counted yet (a timeout before the gates).
    auto conv_window_update = [&](int prev) {
        if constexpr (CONV) {
            const auto& cp = p.conv;
            // the request and q/k head and the reader count, kept by thread 0
            // in spare words of the norm area (no register holds them through
            // the tile loop)
            const int* meta = reinterpret_cast<const int*>(red);
            const int n = meta[7], hq = meta[11], readers = meta[15];
            if (TPC > 1 && readers == 1) return;  // rewritten with the value columns'
            bool last = true;
            if (readers > 1) {
                int* flag = reinterpret_cast<int*>(red) + 3;  // unused word of the norm area
                if (tid == 0) {
                    int* cnt = cp.counters + (int64_t)n * p.hqk + hq;
                    const bool done = (prev >= 0 ? prev : atomicAdd(cnt, 1)) == readers - 1;
                    if (done) atomicExch(cnt, 0);
                    *flag = done ? 1 : 0;
                }
                __syncthreads();
                last = *flag != 0;
            }
            if (last && tid < p.k) {
                const bool rst = p.reset != nullptr && p.reset[n] != 0;
                QT* W = static_cast<QT*>(cp.window) + (int64_t)cp.slot[n] * cp.slot_stride;
                const QT* X = static_cast<const QT*>(cp.x) + (int64_t)n * cp.C;
                const int chq = hq * p.k + tid, chk = (p.hqk + hq) * p.k + tid;
                conv_window_store(W + chq, cp.C, cp.L, cp.KW, rst, X[chq]);
                conv_window_store(W + chk, cp.C, cp.L, cp.KW, rst, X[chk]);
            }
        }
    };
    if constexpr (CONV) {  // for the window update at the end (spare words of the norm area)
        static_assert(NWARP >= 4, "the norm area's spare words 3, 7, 11, 15");
        if (tid == 0) {
            int* meta = reinterpret_cast<int*>(red);
            meta[7] = n;
            meta[11] = chq;
            meta[15] = cgrp * ct;
        }
    }
    __syncthreads();  // the barriers are initialised before anyone waits on them
    // The gates need only the small inputs, so they are worked out while the
    // state tile is still in flight.
    const bool ok = mbar_wait(bar_in, 0);

    // (1) gates: thread tid < K owns row tid.
    float kt = 0.f, qt = 0.f, alpha = 0.f;
    float vts[(TPC * BV + NT - 1) / NT];
#pragma unroll
    for (int e = 0; e < (TPC * BV + NT - 1) / NT; ++e) {
        const int c = tid + e * NT;
        vts[e] = ok && c < TPC * BV && c < p.v - cb0 * BV
                     ? (CONV ? cvv[e] : to_f32(reinterpret_cast<const QT*>(in + SH::IN_V)[c])) : 0.f;
    }
    if (ok && tid < p.k) {
        kt = CONV ? ck : to_f32(reinterpret_cast<const QT*>(in + SH::IN_K)[tid]);
        qt = CONV ? cq : to_f32(reinterpret_cast<const QT*>(in + SH::IN_Q)[tid]);
        const bool scaled = p.a_log != nullptr;
        alpha = gate_alpha(reinterpret_cast<const float*>(in + SH::IN_A)[tid], scaled,
                           scaled ? expf(__ldg(p.a_log + h)) : 1.f,
                           p.dt_bias != nullptr ? __ldg(p.dt_bias + (int64_t)h * p.k + tid) : 0.f);
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
            mbar_wait(bar_in, 0);  // bounded: no copy may still target this CTA's memory
            if (!rst)
                for (int j = 0; j < TPC && (TPC == 1 || cb0 + j < vt); ++j) mbar_wait(bar_st + j, 0);
        }
        conv_window_update(-1);
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
    const float rk = __frsqrt_rn(kk2 + L2_EPS);
    const float rq = __frsqrt_rn(qq2 + L2_EPS);
    const float beta = sigmoid_neg(-b);  // sigmoid(b)
    const float bqk = beta * (kq * rk * rq);         // beta (qhat . khat)
    // Per row: w = alpha khat and z = alpha qhat fold the decay into the two
    // reductions (u = sum_i S_ij w_i, p = sum_i S_ij z_i); alpha and beta khat
    // serve the update S' = alpha S + (beta khat) d.
    if (tid < p.k) {
        const float kh = kt * rk, qh = qt * rq;
        gates[tid] = make_float4(alpha * kh, alpha * qh, alpha, beta * kh);
    }
#pragma unroll
    for (int e = 0; e < (TPC * BV + NT - 1) / NT; ++e)
        if (tid + e * NT < TPC * BV) gv[tid + e * NT] = vts[e];
    __syncthreads();
    // the fused convolution: every thread of this CTA has used the window
    // values it read (they fed the gates above), so thread 0 counts the
    // CTA's read now; the result is needed only at the end
    int conv_prev = 0;
    if constexpr (CONV) {
        const int* meta = reinterpret_cast<const int*>(red);  // request, q/k head, readers
        if (tid == 0 && meta[15] > 1) conv_prev = atomicAdd(p.conv.counters + (int64_t)meta[7] * p.hqk + meta[11], 1);
    }

    for (int jt = 0; jt < TPC; ++jt) {
        // tile jt of this CTA: column block cb (past the last block when V
        // is not a multiple of TPC BV: then only the barriers are kept)
        const int cb = cb0 + jt;
        const bool tile_in = TPC == 1 || cb < vt;  // one tile a CTA: the grid covers exactly vt
        const int col0 = cb * BV + cl * VEC;
        const uint32_t tile_base = tile_base0 + jt * SH::TILE_BYTES;
        // This thread's rows are rg + RG * rr.  RG rows span whole swizzle periods,
        // so the XOR term of every row equals that of row rg: one base address,
        // then a constant stride.
        const int nrows = FULLK ? ROWS : min(ROWS, (p.k - rg + RG - 1) / RG);
        const uint32_t srow0 = tile_base + swz<SH::ROWBYTES>(rg, cl);
        const uint32_t grow0 = gate_base + rg * 16;
        constexpr uint32_t SSTRIDE = RG * SH::ROWBYTES, GSTRIDE = RG * 16;

        // (2) the two partial sums over this thread's rows, once the tile is in.
        // Adjacent columns travel as float pairs through the packed FMA (two
        // fmaf per instruction, each rounded as fmaf rounds).
        constexpr int VP = VEC / 2;
        const bool ok_st = rst || !tile_in || mbar_wait(bar_st + jt, 0);
        float2 u[VP], pp[VP];
        uint4 xs[KEEP ? ROWS : 1];  // KEEP: the rows' raw 16-byte words, for pass (3)
#pragma unroll
        for (int c = 0; c < VP; ++c) { u[c] = make_float2(0.f, 0.f); pp[c] = make_float2(0.f, 0.f); }
        if (!rst && ok_st && tile_in) {
#pragma unroll
            for (int rr = 0; rr < ROWS; ++rr) {
                if (FULLK || rr < nrows) {
                    float2 x[VP];
                    const uint4 raw = lds128(srow0 + rr * SSTRIDE);
                    if (KEEP) xs[KEEP ? rr : 0] = raw;
                    SV::widen2(raw, x);
                    const uint4 g = lds128(grow0 + rr * GSTRIDE);
                    const float w = __uint_as_float(g.x), z = __uint_as_float(g.y);
                    const float2 w2 = make_float2(w, w), z2 = make_float2(z, z);
#pragma unroll
                    for (int c = 0; c < VP; ++c) {
                        u[c] = __ffma2_rn(x[c], w2, u[c]);
                        pp[c] = __ffma2_rn(x[c], z2, pp[c]);
                    }
                }
            }
        }
        // Sum over the row groups of this warp (the lanes that share cl) as a
        // reduce-scatter: each step hands the partner lane the half of the values
        // this lane will not keep, so the lane ends with KEEPV finished sums of
        // the 2 VEC values {u[0..VEC), p[0..VEC)} of chunk cl, at index kbase.
        float vals[2 * VEC];
#pragma unroll
        for (int c = 0; c < VP; ++c) {
            vals[2 * c] = u[c].x; vals[2 * c + 1] = u[c].y;
            vals[VEC + 2 * c] = pp[c].x; vals[VEC + 2 * c + 1] = pp[c].y;
        }
        int kbase = 0;
#pragma unroll
        for (int m = 16, cnt = 2 * VEC; m >= CL; m >>= 1, cnt >>= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int j = 0; j < cnt / 2; ++j) {
                const float send = upper ? vals[j] : vals[j + cnt / 2];
                const float keep = upper ? vals[j + cnt / 2] : vals[j];
                vals[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
            kbase += upper ? cnt / 2 : 0;
        }
        {
            float* dst = red2 + (warp * CL + cl) * 2 * VEC + kbase;
            if (KEEPV == 4) *reinterpret_cast<float4*>(dst) = make_float4(vals[0], vals[1], vals[2], vals[3]);
            else if (KEEPV == 2) *reinterpret_cast<float2*>(dst) = make_float2(vals[0], vals[1]);
            else dst[0] = vals[0];
        }
        if (__syncthreads_or(ok_st ? 0 : 1)) {  // the state tile did not land in time
            if (tid == 0) {
                atomicExch(p.status, STATUS_TIMEOUT);
                for (int j = jt; j < TPC && (TPC == 1 || cb0 + j < vt); ++j) mbar_wait(bar_st + j, 0);  // bounded, as above
            }
            conv_window_update(conv_prev);
            return;
        }
        // ... then over the warps: thread j < BV finishes column j, writes its
        // output and leaves d_j = v_j - u_j for the update.
        const int ncols = min(BV, p.v - cb * BV);  // <= 0 past the last column block
        if (tid < ncols) {
            const int jc = tid / VEC, jv = tid - jc * VEC;
            float su = 0.f, sp = 0.f;
#pragma unroll
            for (int w = 0; w < NWARP; ++w) {
                su += red2[(w * CL + jc) * 2 * VEC + jv];
                sp += red2[(w * CL + jc) * 2 * VEC + VEC + jv];
            }
            const float dj = gv[jt * BV + tid] - su;
            dsm[tid] = dj;
            p.o[(int64_t)r * p.v + cb * BV + tid] = fmaf(bqk, dj, sp) * p.inv_sqrt_k;
        }
        __syncthreads();
        if constexpr (TPC == 1 && !CONV) {
            if (col0 >= p.v) return;  // one tile a CTA: nothing follows
        }
        if ((TPC == 1 && !CONV) || col0 < p.v) {  // the tile holds columns: the update and the stores
            float2 d[VP];
#pragma unroll
            for (int c = 0; c < VP; c += 2) {
                const float4 d4 = *reinterpret_cast<const float4*>(dsm + cl * VEC + 2 * c);
                d[c] = make_float2(d4.x, d4.y); d[c + 1] = make_float2(d4.z, d4.w);
            }

            // (3) the delta update S' = alpha S + (beta khat) d (per element
            // fmaf(alpha, S, (beta khat) d), in pairs), stored in place with coalesced
            // 16-byte stores.
            ST* dst = static_cast<ST*>(p.pool) + state_at(p, slot, h) + (int64_t)rg * p.v + col0;
            const int64_t gstride = (int64_t)RG * p.v;
#pragma unroll
            for (int rr = 0; rr < ROWS; ++rr) {
                if (FULLK || rr < nrows) {
                    float2 x[VP];
                    if (rst) {
#pragma unroll
                        for (int c = 0; c < VP; ++c) x[c] = make_float2(0.f, 0.f);
                    } else if (KEEP) {
                        SV::widen2(xs[KEEP ? rr : 0], x);
                    } else {
                        SV::widen2(lds128(srow0 + rr * SSTRIDE), x);
                    }
                    const uint4 g = lds128(grow0 + rr * GSTRIDE);
                    const float al = __uint_as_float(g.z), bk = __uint_as_float(g.w);
                    const float2 al2 = make_float2(al, al), bk2 = make_float2(bk, bk);
#pragma unroll
                    for (int c = 0; c < VP; ++c) x[c] = __ffma2_rn(al2, x[c], __fmul2_rn(bk2, d[c]));
                    __stcs(reinterpret_cast<uint4*>(dst + rr * gstride), SV::narrow2(x));
                }
            }
        }
    }
    conv_window_update(conv_prev);
}

}  // namespace kda
