// Prefill in two passes over chunks of CH = 16 tokens (the chunk form of the
// delta rule, restated from the recurrence; see the verify kernel's header
// for the derivation).  For a chunk with initial state S_0, tokens t < CH,
// c_t = alpha_0 ... alpha_t (elementwise), P_ts = alpha_(s+1) ... alpha_t:
//   W_t = c_t khat_t,  Z_t = c_t qhat_t,
//   A_ts = beta_s sum_i khat_s,i P_ts,i khat_t,i   (s < t),
//   B_ts = beta_s sum_i khat_s,i P_ts,i qhat_t,i   (s <= t),
//   (I + A) [W' | U] = [W | V]          (T = (I + A)^-1: W' = T W, U = T V)
//   D = U - W' S_0                      (the chunk's d_t, one row per token)
//   O = (Z - B W') S_0 + B U            (times 1/sqrt(K): Q' S_0 + O_intra)
//   S_end = diag(c_(CH-1)) S_0 + Ke^T D,  Ke_s = beta_s khat_s P_(CH-1)s.
// Everything but S_0 depends on the chunk's inputs only, so
//   pass 1 (prepare): one CTA per (chunk, head), all chunks at once, writes
//     W'^T, Q'^T, Ke^T ([K][CH] each), c_(CH-1) [K], U and O_intra ([V/32][CH][32])
//     to a workspace;
//   pass 2 (scan): one CTA per (request, head, 32 value columns) walks the
//     request's chunks in order: D = U - W' S, O = Q' S + O_intra,
//     S <- c S + Ke^T D, with each chunk's operands bulk-copied into shared
//     memory one chunk ahead; the final state is stored once.
// The products P are formed by multiplication (no division), so alpha = 0 is
// exact.  Tokens past a request's end are padded as alpha = 1, beta = 0, k = 0.
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int PCH = 16;                                   // tokens per chunk
constexpr int PCH_FLOATS = 3 * KMAX * PCH + KMAX + 2 * KMAX * PCH;  // workspace floats per (chunk, head)
constexpr int PVT = 32;                                   // value columns per scan CTA
#ifndef KDA_PREP_MINB
#define KDA_PREP_MINB 3   // resident prepare CTAs per SM the register budget must allow (168 registers, no spill)
#endif
#ifndef KDA_PSCAN_WARPS
#define KDA_PSCAN_WARPS 8
#endif
constexpr int PSCAN_WARPS = KDA_PSCAN_WARPS;              // scan: warp w owns rows KMAX / PSCAN_WARPS * w ..
constexpr int PSCAN_ROWS = KMAX / PSCAN_WARPS;

// workspace offsets (floats) inside one (chunk, head) block
constexpr int PW_WT = 0;                        // W'^T [KMAX][PCH]
constexpr int PW_QT = PW_WT + KMAX * PCH;       // Q'^T [KMAX][PCH] (already / sqrt(K))
constexpr int PW_KT = PW_QT + KMAX * PCH;       // Ke^T [KMAX][PCH]
constexpr int PW_C = PW_KT + KMAX * PCH;        // c_(CH-1) [KMAX]
constexpr int PW_U = PW_C + KMAX;               // U [KMAX / PVT][PCH][PVT]
constexpr int PW_OI = PW_U + KMAX * PCH;        // O_intra [KMAX / PVT][PCH][PVT] (already / sqrt(K))
static_assert(PW_OI + KMAX * PCH == PCH_FLOATS, "workspace layout");
static_assert((2 * PCH) % PSCAN_WARPS == 0 && KMAX % PSCAN_WARPS == 0, "scan warps split the rows and vectors");

// Chunk j of request r lives at slot floor(tb / PCH) + r + j, tb = the request's
// first token: distinct for every (r, j) and below total / PCH + n.
__device__ __forceinline__ int64_t prefill_chunk_slot(int tb, int r, int j) {
    return (int64_t)(tb / PCH) + r + j;
}

// This row's terms of the 256 row sums of a 16-token chunk (A: 120, B: 136,
// stored in that order: A_ts at t (t - 1) / 2 + s, B_ts at 120 + t (t + 1) / 2 + s),
// those from LO to LO + 31.  Compile-time indices throughout.
__host__ __device__ constexpr int pidx_a(int t, int s) { return t * (t - 1) / 2 + s; }
__host__ __device__ constexpr int pidx_b(int t, int s) { return 120 + t * (t + 1) / 2 + s; }

template <int LO>
__device__ __forceinline__ void pab_terms(float (&out)[32], const float (&bk)[PCH], const float (&kh)[PCH],
                                          const float (&qh)[PCH], const float (&al)[PCH]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) out[i] = 0.f;
#pragma unroll
    for (int s = 0; s < PCH; ++s) {
        float e = bk[s];
        if (pidx_b(s, s) >= LO && pidx_b(s, s) < LO + 32) out[pidx_b(s, s) - LO] = e * qh[s];
#pragma unroll
        for (int t = s + 1; t < PCH; ++t) {
            e *= al[t];
            if (pidx_a(t, s) >= LO && pidx_a(t, s) < LO + 32) out[pidx_a(t, s) - LO] = e * kh[t];
            if (pidx_b(t, s) >= LO && pidx_b(t, s) < LO + 32) out[pidx_b(t, s) - LO] = e * qh[t];
        }
    }
}

// Pass 1.  grid = (n * max_chunks, hv), 128 threads: thread i owns key
// channel i (and value column i for the V-side solve).
template <typename QT>
__global__ void __launch_bounds__(KMAX, KDA_PREP_MINB) kda_prefill_prep_kernel(const StepParams p, float* __restrict__ ws,
                                                                int max_chunks) {
    __shared__ float vs[PCH][KMAX];        // v of the chunk's tokens
    __shared__ float wsm[PCH][KMAX];       // W, then W'
    __shared__ float zsm[PCH][KMAX];       // Z = c qhat
    __shared__ float abw[KMAX / 32][256];  // per warp row sums
    __shared__ float ab[256];              // A then B
    __shared__ float nrm[KMAX / 32][32];
    __shared__ float sc[PCH][4];           // beta, rk, rq

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = (int)blockIdx.x / max_chunks, j = (int)blockIdx.x - r * max_chunks;
    const int h = (int)blockIdx.y;
    cudaGridDependencySynchronize();
    int tb = r * p.t, Tn = p.t;
    if (p.cu != nullptr) {
        tb = p.cu[r];
        Tn = p.cu[r + 1] - tb;
    }
    // bad offsets are reported by the scan pass; here they only stop the work
    if (tb < 0 || Tn < 0 || Tn > p.t || (int64_t)tb + Tn > p.total || j * PCH >= Tn) return;
    if (p.init_slot[r] < 0) return;  // padding request
    const int cl = min(PCH, Tn - j * PCH);
    const int t0 = tb + j * PCH;
    const int hq = h / (p.hv / p.hqk);
    float* w = ws + (prefill_chunk_slot(tb, r, j) * p.hv + h) * PCH_FLOATS;

    // (1) inputs: row tid of k, q, a for every token; value column tid of v.
    // Half a chunk at a time, every load unconditional from an address
    // clamped into the chunk's last token, row 0 or column 0, so that all of
    // a half's loads are in flight at once; values out of range are zeroed.
    float kt[PCH], qt[PCH], al[PCH];
    const bool scaled = p.a_log != nullptr;
    const float gscale = scaled ? expf(__ldg(p.a_log + h)) : 1.f;
    const float gbias = p.dt_bias != nullptr && tid < p.k ? __ldg(p.dt_bias + (int64_t)h * p.k + tid) : 0.f;
    {
        const int row = tid < p.k ? tid : 0, col = tid < p.v ? tid : 0;
        const QT* qp = static_cast<const QT*>(p.q);
        const QT* kp = static_cast<const QT*>(p.kk);
        const QT* vp = static_cast<const QT*>(p.vv);
        constexpr int HALF = PCH / 2;
#pragma unroll
        for (int t1 = 0; t1 < PCH; t1 += HALF) {
            QT kr[HALF], qr[HALF], vr[HALF];
            float ar[HALF];
#pragma unroll
            for (int u = 0; u < HALF; ++u) {
                const int64_t tok = (int64_t)t0 + min(t1 + u, cl - 1);
                const int64_t rq = (tok * p.hqk + hq) * p.k + row, rt = tok * p.hv + h;
                kr[u] = kp[rq];
                qr[u] = qp[rq];
                ar[u] = __ldg(p.a + rt * p.k + row);
                vr[u] = vp[rt * p.v + col];
            }
#pragma unroll
            for (int u = 0; u < HALF; ++u) {
                const int t = t1 + u;
                const bool in_row = t < cl && tid < p.k;
                kt[t] = in_row ? to_f32(kr[u]) : 0.f;
                qt[t] = in_row ? to_f32(qr[u]) : 0.f;
                al[t] = in_row ? gate_alpha(ar[u], scaled, gscale, gbias) : 1.f;
                vs[t][tid] = t < cl && tid < p.v ? to_f32(vr[u]) : 0.f;
            }
        }
    }
    {
        float sq[2 * PCH];
#pragma unroll
        for (int t = 0; t < PCH; ++t) { sq[2 * t] = kt[t] * kt[t]; sq[2 * t + 1] = qt[t] * qt[t]; }
        nrm[warp][lane] = warp_reduce_scatter<2 * PCH>(sq, lane);  // lane L: value L
    }
    __syncthreads();
    if (tid < PCH) {
        float kk2 = 0.f, qq2 = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < KMAX / 32; ++w2) {
            kk2 += nrm[w2][2 * tid];
            qq2 += nrm[w2][2 * tid + 1];
        }
        const float beta = tid < cl ? sigmoid_neg(-__ldg(p.b + (int64_t)(t0 + tid) * p.hv + h)) : 0.f;
        sc[tid][0] = beta;
        sc[tid][1] = __frsqrt_rn(kk2 + L2_EPS);
        sc[tid][2] = __frsqrt_rn(qq2 + L2_EPS);
    }
    __syncthreads();

    // (2) row tid: khat, qhat, W = c khat, Z = c qhat, Ke, c_(CH-1), and its
    // terms of the 256 row sums of A and B
    float kh[PCH], qh[PCH], bk[PCH];
    float c = 1.f;
#pragma unroll
    for (int t = 0; t < PCH; ++t) {
        kh[t] = kt[t] * sc[t][1];
        qh[t] = qt[t] * sc[t][2];
        bk[t] = sc[t][0] * kh[t];
        c *= al[t];
        wsm[t][tid] = c * kh[t];
        zsm[t][tid] = c * qh[t];
    }
    // The workspace rows of W'^T, Q'^T and Ke^T are 64 bytes, one per thread:
    // each is stored as four 16-byte vectors.
    if (tid < p.k) {
        w[PW_C + tid] = c;
        float e = 1.f;  // alpha_(s+1) ... alpha_(CH-1)
        float4* kt4 = reinterpret_cast<float4*>(w + PW_KT + tid * PCH);
        float kv[4];
#pragma unroll
        for (int s = PCH - 1; s >= 0; --s) {
            kv[s & 3] = bk[s] * e;
            e *= al[s];
            if ((s & 3) == 0) kt4[s >> 2] = make_float4(kv[0], kv[1], kv[2], kv[3]);
        }
    }
    {
        float part[32];
#define KDA_PAB(LO)                                                        \
        pab_terms<LO>(part, bk, kh, qh, al);                               \
        abw[warp][LO + lane] = warp_reduce_scatter<32>(part, lane);
        KDA_PAB(0) KDA_PAB(32) KDA_PAB(64) KDA_PAB(96) KDA_PAB(128) KDA_PAB(160) KDA_PAB(192) KDA_PAB(224)
#undef KDA_PAB
    }
    __syncthreads();
    for (int e = tid; e < 256; e += KMAX) {
        float s = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < KMAX / 32; ++w2) s += abw[w2][e];
        ab[e] = s;
    }
    __syncthreads();

    // (3) column tid: forward substitution for W' and U, then Q' and O_intra
    float wp[PCH], u[PCH];
#pragma unroll
    for (int t = 0; t < PCH; ++t) {
        float xw = wsm[t][tid], xu = vs[t][tid];
#pragma unroll
        for (int s = 0; s < t; ++s) {
            const float a = ab[pidx_a(t, s)];
            xw = fmaf(-a, wp[s], xw);
            xu = fmaf(-a, u[s], xu);
        }
        wp[t] = xw;
        u[t] = xu;
    }
    const int vt = tid / PVT, vc = tid - vt * PVT;
    float4* wt4 = reinterpret_cast<float4*>(w + PW_WT + tid * PCH);
    float4* qt4 = reinterpret_cast<float4*>(w + PW_QT + tid * PCH);
    float qv[4];
#pragma unroll
    for (int t = 0; t < PCH; ++t) {
        float qp = zsm[t][tid], oi = 0.f;
#pragma unroll
        for (int s = 0; s <= t; ++s) {
            const float bts = ab[pidx_b(t, s)];
            qp = fmaf(-bts, wp[s], qp);
            oi = fmaf(bts, u[s], oi);
        }
        qv[t & 3] = qp * p.inv_sqrt_k;
        if ((t & 3) == 3 && tid < p.k) {
            wt4[t >> 2] = make_float4(wp[t - 3], wp[t - 2], wp[t - 1], wp[t]);
            qt4[t >> 2] = make_float4(qv[0], qv[1], qv[2], qv[3]);
        }
        if (tid < p.v) {
            w[PW_U + (vt * PCH + t) * PVT + vc] = u[t];
            w[PW_OI + (vt * PCH + t) * PVT + vc] = oi * p.inv_sqrt_k;
        }
    }
}

// Pass 2.  grid = n * hv * ceil(v / NC) CTAs of PSCAN_WARPS warps, NC = 32, 16
// or 8 value columns per CTA (narrower tiles when few requests leave SMs idle).
// Warp w owns rows 16 w .. 16 w + 15 of the state tile; lane l = rq NC + cc
// takes column cc and rows 16 w + rq RPT + i (i < RPT = 16 NC / 32).
template <int NC>
struct PrefillScanSmem {
    static constexpr uint32_t OPS = (3 * KMAX * PCH + KMAX + 2 * PCH * PVT) * 4;  // one chunk's operands
    static constexpr uint32_t BUF = (OPS + 127u) & ~127u;
    static constexpr uint32_t RED = PSCAN_WARPS * 2 * PCH * NC * 4;               // partial sums
    static constexpr uint32_t BYTES = 2 * BUF + RED + 2 * PCH * NC * 4 + 16;
};

template <typename ST, int NC>
__global__ void __launch_bounds__(PSCAN_WARPS * 32, 2) kda_prefill_scan_kernel(const StepParams p,
                                                                           const float* __restrict__ ws) {
    static_assert(NC == 32 || NC == 16 || NC == 8, "columns per scan CTA");
    constexpr int NRQ = 32 / NC;                 // lanes sharing a column
    constexpr int RPT = PSCAN_ROWS / NRQ;        // rows per thread
    constexpr int KEEP = 2 * PCH / NRQ;          // partial sums a lane keeps after the reduce-scatter
    static_assert(PSCAN_ROWS % NRQ == 0, "row split");
    using SM = PrefillScanSmem<NC>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* red = reinterpret_cast<float*>(smem + 2 * SM::BUF);  // [warp][32 vectors][NC]
    float* fin = red + PSCAN_WARPS * 2 * PCH * NC;               // [32 vectors][NC]
    uint64_t* bars = reinterpret_cast<uint64_t*>(fin + 2 * PCH * NC);  // two chunk-operand barriers

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rq = lane / NC, cc = lane - rq * NC;
    const int vtiles = (p.v + NC - 1) / NC;
    const int tile = (int)blockIdx.x;
    const int r = tile / (p.hv * vtiles);
    const int rem = tile - r * p.hv * vtiles;
    const int h = rem / vtiles, cb = rem - h * vtiles;
    const int col = cb * NC + cc;
    const int c32 = (cb * NC) / PVT;             // the 32-column workspace tile holding this CTA's columns
    const int cw = col - c32 * PVT;              // column inside it
    const bool col_ok = col < p.v;
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize();

    int tb = r * p.t, Tn = p.t;
    if (p.cu != nullptr) {
        tb = p.cu[r];
        Tn = p.cu[r + 1] - tb;
    }
    const bool range_ok = tb >= 0 && Tn >= 0 && Tn <= p.t && (int64_t)tb + Tn <= p.total;
    const int32_t slot = p.init_slot[r], fin_slot = p.final_slot[r];
    const bool bad = !range_ok || slot >= p.num_slots || fin_slot >= p.num_slots;
    if (bad) {
        if (tid == 0) atomicCAS(p.status, 0, range_ok ? STATUS_SLOT_RANGE : STATUS_ARG);
        return;
    }
    if (slot < 0) {  // padding: outputs zero, nothing read or stored
        for (int e = tid; e < Tn * NC; e += PSCAN_WARPS * 32) {
            const int c2 = cb * NC + (e % NC);
            if (c2 < p.v) p.o[((int64_t)(tb + e / NC) * p.hv + h) * p.v + c2] = 0.f;
        }
        return;
    }
    // a request with no tokens stores its initial state (zero on a reset) to
    // its final slot: the state after its last token
    if (Tn == 0 && fin_slot < 0) return;
    const int nch = (Tn + PCH - 1) / PCH;
    const int row0 = warp * PSCAN_ROWS + rq * RPT;  // this thread's rows: row0 .. row0 + RPT - 1

    // the state tile, fp32 in registers
    float S[RPT];
    const bool rst = p.reset != nullptr && p.reset[r] != 0;
    const ST* src = static_cast<const ST*>(p.pool) + state_at(p, slot, h);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = row0 + i;
        S[i] = (!rst && col_ok && row < p.k) ? to_f32(src[(int64_t)row * p.v + col]) : 0.f;
    }

    // chunk operands of chunk j -> buffer j % 2, one barrier per buffer
    auto issue = [&](int j) {
        const float* w = ws + (prefill_chunk_slot(tb, r, j) * p.hv + h) * PCH_FLOATS;
        uint8_t* buf = smem + (j & 1) * SM::BUF;
        uint64_t* bar = bars + (j & 1);
        const uint32_t kb = (uint32_t)p.k * PCH * 4, tb2 = PCH * PVT * 4;
        mbar_arrive_expect_tx(bar, 3 * kb + (uint32_t)p.k * 4 + 2 * tb2);
        bulk_load(buf, w + PW_WT, kb, bar);
        bulk_load(buf + KMAX * PCH * 4, w + PW_QT, kb, bar);
        bulk_load(buf + 2 * KMAX * PCH * 4, w + PW_KT, kb, bar);
        bulk_load(buf + 3 * KMAX * PCH * 4, w + PW_C, (uint32_t)p.k * 4, bar);
        bulk_load(buf + (3 * KMAX * PCH + KMAX) * 4, w + PW_U + c32 * PCH * PVT, tb2, bar);
        bulk_load(buf + (3 * KMAX * PCH + KMAX + PCH * PVT) * 4, w + PW_OI + c32 * PCH * PVT, tb2, bar);
    };
    if (tid == 0) {
        mbar_init(bars, 1);
        mbar_init(bars + 1, 1);
        fence_mbar_init();
        if (nch > 0) issue(0);
    }
    __syncthreads();

    // chunk j is buffer j % 2's (j / 2)-th use: barrier parity (j / 2) % 2
    int jfail = -1, issued = nch > 0 ? 1 : 0;
    for (int j = 0; j < nch; ++j) {
        if (j + 1 < nch) {  // its buffer's last reader was chunk j - 1
            if (tid == 0) issue(j + 1);
            ++issued;
        }
        const bool ok = mbar_wait(bars + (j & 1), (j >> 1) & 1);
        if (__syncthreads_or(ok ? 0 : 1)) {
            jfail = j;
            break;
        }
        const float* buf = reinterpret_cast<const float*>(smem + (j & 1) * SM::BUF);
        const float* WT = buf;
        const float* QT_ = buf + KMAX * PCH;
        const float* KT = buf + 2 * KMAX * PCH;
        const float* CC = buf + 3 * KMAX * PCH;
        const float* U = CC + KMAX;
        const float* OI = U + PCH * PVT;

        // partial sums over this thread's rows: v_t = sum_i W'_ti S_i (t < 16),
        // v_(16+t) = sum_i Q'_ti S_i
        float vals[2 * PCH];
#pragma unroll
        for (int t = 0; t < 2 * PCH; ++t) vals[t] = 0.f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int row = row0 + i;
            if (row < p.k) {
                const float4* w4 = reinterpret_cast<const float4*>(WT + row * PCH);
                const float4* q4 = reinterpret_cast<const float4*>(QT_ + row * PCH);
#pragma unroll
                for (int g = 0; g < PCH / 4; ++g) {
                    const float4 a = w4[g], b = q4[g];
                    vals[4 * g] = fmaf(a.x, S[i], vals[4 * g]);
                    vals[4 * g + 1] = fmaf(a.y, S[i], vals[4 * g + 1]);
                    vals[4 * g + 2] = fmaf(a.z, S[i], vals[4 * g + 2]);
                    vals[4 * g + 3] = fmaf(a.w, S[i], vals[4 * g + 3]);
                    vals[PCH + 4 * g] = fmaf(b.x, S[i], vals[PCH + 4 * g]);
                    vals[PCH + 4 * g + 1] = fmaf(b.y, S[i], vals[PCH + 4 * g + 1]);
                    vals[PCH + 4 * g + 2] = fmaf(b.z, S[i], vals[PCH + 4 * g + 2]);
                    vals[PCH + 4 * g + 3] = fmaf(b.w, S[i], vals[PCH + 4 * g + 3]);
                }
            }
        }
        // over the NRQ lanes sharing column cc: a reduce-scatter, each keeps KEEP sums
        int kbase = 0;
#pragma unroll
        for (int m = 16, cnt = 2 * PCH; m >= NC; m >>= 1, cnt >>= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int e = 0; e < cnt / 2; ++e) {
                const float send = upper ? vals[e] : vals[e + cnt / 2];
                const float keep = upper ? vals[e + cnt / 2] : vals[e];
                vals[e] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
            kbase += upper ? cnt / 2 : 0;
        }
#pragma unroll
        for (int e = 0; e < KEEP; ++e) red[(warp * 2 * PCH + kbase + e) * NC + cc] = vals[e];
        __syncthreads();
        // the sums over the warps: 32 vectors x NC columns
        for (int e = tid; e < 2 * PCH * NC; e += PSCAN_WARPS * 32) {
            float sum = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < PSCAN_WARPS; ++w2) sum += red[w2 * 2 * PCH * NC + e];
            fin[e] = sum;
        }
        __syncthreads();
        // d_t = U_t - (W' S)_t for this column; outputs O_t = (Q' S)_t + O_intra_t
        float d[PCH];
#pragma unroll
        for (int t = 0; t < PCH; ++t) d[t] = U[t * PVT + cw] - fin[t * NC + cc];
        const int cl = min(PCH, Tn - j * PCH);
        for (int e = tid; e < cl * NC; e += PSCAN_WARPS * 32) {
            const int t = e / NC, c2 = e - t * NC, gcol = cb * NC + c2;
            if (gcol < p.v)
                p.o[((int64_t)(tb + j * PCH + t) * p.hv + h) * p.v + gcol] =
                    fin[(PCH + t) * NC + c2] + OI[t * PVT + gcol - c32 * PVT];
        }
        // S <- c S + Ke^T D
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int row = row0 + i;
            if (row < p.k) {
                const float4* k4 = reinterpret_cast<const float4*>(KT + row * PCH);
                float x = CC[row] * S[i];
#pragma unroll
                for (int g = 0; g < PCH / 4; ++g) {
                    const float4 kk = k4[g];
                    x = fmaf(kk.x, d[4 * g], x);
                    x = fmaf(kk.y, d[4 * g + 1], x);
                    x = fmaf(kk.z, d[4 * g + 2], x);
                    x = fmaf(kk.w, d[4 * g + 3], x);
                }
                S[i] = x;
            }
        }
        // every thread is done with this buffer and with red/fin before the
        // next issue (generic reads, then async writes: fence first)
        fence_proxy_async_smem();
        __syncthreads();
    }
    if (jfail >= 0) {
        if (tid == 0) {
            atomicExch(p.status, STATUS_TIMEOUT);
            // bounded: no copy may still target this CTA's memory when it exits
            for (int jj = jfail; jj < issued; ++jj) mbar_wait(bars + (jj & 1), (jj >> 1) & 1);
        }
        return;
    }
    if (fin_slot >= 0 && col_ok) {
        ST* dst = static_cast<ST*>(p.pool) + state_at(p, fin_slot, h);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int row = row0 + i;
            if (row < p.k) {
                if constexpr (sizeof(ST) == 4) dst[(int64_t)row * p.v + col] = S[i];
                else dst[(int64_t)row * p.v + col] = __float2half_rn(S[i]);
            }
        }
    }
}

}  // namespace kda
