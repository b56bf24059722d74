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
//     W', Q' and Ke ([CH][K] each, as three bf16 parts), c_(CH-1) [K], U and
//     O_intra ([CH][V], fp32) to a workspace;
//   pass 2 (scan): per (request, head), warps of 16 value columns walk the
//     request's chunks in order on the tensor cores: D = U - W' S,
//     O = Q' S + O_intra, S <- c S + Ke^T D, with each chunk's operands
//     bulk-copied into shared memory one chunk ahead; the final state is
//     stored once.
// The products P are formed by multiplication (no division), so alpha = 0 is
// exact.  Tokens past a request's end are padded as alpha = 1, beta = 0, k = 0.
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int PCH = 16;                                   // tokens per chunk
#ifndef KDA_PREP_MINB
#define KDA_PREP_MINB 3   // resident prepare CTAs per SM the register budget must allow (168 registers, no spill)
#endif

// Workspace block of one (chunk, head), in bytes.  W', Q' (already / sqrt(K))
// and Ke are [PCH tokens][KMAX rows] matrices, each as three bf16 part
// matrices (x = x0 + x1 + x2), rows padded to PT_ROW elements (272 bytes: the
// 8 rows an ldmatrix reads fall in distinct banks); U and O_intra (already
// / sqrt(K)) are [PCH tokens][KMAX columns] fp32, rows padded to PU_ROW.
constexpr int PT_ROW = KMAX + 8;
constexpr int PU_ROW = KMAX + 4;
constexpr uint32_t PART_BYTES = PCH * PT_ROW * 2;
constexpr uint32_t PB_W = 0, PB_Q = 3 * PART_BYTES, PB_K = 6 * PART_BYTES;
constexpr uint32_t PB_C = 9 * PART_BYTES;                  // c_(CH-1) [KMAX] fp32
constexpr uint32_t PB_U = PB_C + KMAX * 4;
constexpr uint32_t PB_OI = PB_U + PCH * PU_ROW * 4;
constexpr uint32_t PCH_BYTES = PB_OI + PCH * PU_ROW * 4;
static_assert(PART_BYTES % 16 == 0 && PB_C % 16 == 0 && PB_U % 16 == 0 && PCH_BYTES % 256 == 0, "workspace layout");

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
// x in three bf16 parts, element [t][i] of part matrices base, base + 1, base + 2
__device__ __forceinline__ void put_parts(__nv_bfloat16* base, int t, int i, float x) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(x);
    const float r = x - __bfloat162float(h0);
    const __nv_bfloat16 h1 = __float2bfloat16_rn(r);
    const __nv_bfloat16 h2 = __float2bfloat16_rn(r - __bfloat162float(h1));
    __nv_bfloat16* e = base + t * PT_ROW + i;
    e[0] = h0;
    e[PCH * PT_ROW] = h1;
    e[2 * PCH * PT_ROW] = h2;
}

template <typename QT>
__global__ void __launch_bounds__(KMAX, KDA_PREP_MINB) kda_prefill_prep_kernel(const StepParams p, uint8_t* __restrict__ ws,
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
    uint8_t* w = ws + (prefill_chunk_slot(tb, r, j) * p.hv + h) * (int64_t)PCH_BYTES;
    __nv_bfloat16* wpart = reinterpret_cast<__nv_bfloat16*>(w + PB_W);
    __nv_bfloat16* qpart = reinterpret_cast<__nv_bfloat16*>(w + PB_Q);
    __nv_bfloat16* kpart = reinterpret_cast<__nv_bfloat16*>(w + PB_K);
    float* wu = reinterpret_cast<float*>(w + PB_U);
    float* woi = reinterpret_cast<float*>(w + PB_OI);

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
    // Column tid of Ke and c_(CH-1); rows past K hold zeros (k = 0 there).
    {
        reinterpret_cast<float*>(w + PB_C)[tid] = c;
        float e = 1.f;  // alpha_(s+1) ... alpha_(CH-1)
#pragma unroll
        for (int s = PCH - 1; s >= 0; --s) {
            put_parts(kpart, s, tid, bk[s] * e);
            e *= al[s];
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
    // row tid of W' and Q', column tid of U and O_intra (zeros past K and V)
#pragma unroll
    for (int t = 0; t < PCH; ++t) {
        float qp = zsm[t][tid], oi = 0.f;
#pragma unroll
        for (int s = 0; s <= t; ++s) {
            const float bts = ab[pidx_b(t, s)];
            qp = fmaf(-bts, wp[s], qp);
            oi = fmaf(bts, u[s], oi);
        }
        put_parts(wpart, t, tid, wp[t]);
        put_parts(qpart, t, tid, qp * p.inv_sqrt_k);
        wu[t * PU_ROW + tid] = u[t];
        woi[t * PU_ROW + tid] = oi * p.inv_sqrt_k;
    }
}

// Pass 2 on the tensor cores.  A CTA holds WPC column blocks of 16 value
// columns, each worked by KS warps that split its K rows (the warps of block
// cbk = w / KS own rows 128 / KS * (w % KS) ..); grid = n * hv * ceil(v / (16
// WPC)).  A warp holds its part of the block's state transposed, S^T (16
// columns x its rows), in m16n8 accumulator fragments: tile nt covers rows
// 8 nt .. 8 nt + 7 and lane (g, qd) = (lane / 4, lane % 4) holds
//   {S[8nt+2qd][c0+g], S[8nt+2qd+1][c0+g], S[8nt+2qd][c0+g+8], S[8nt+2qd+1][c0+g+8]}.
// Two adjacent tiles are exactly the A fragment of a 16 x 16 block of S^T, so
// every product takes the state straight from its accumulators:
//   [X^T | Y^T] = S^T [W'^T | Q'^T]    (16 x K by K x 32: X = W' S, Y = Q' S)
//   D^T = U^T - X^T,  O^T = Y^T + O_intra^T
//   S^T <- S^T diag(c) + D^T Ke        (16 x 16 by 16 x K onto the scaled accumulators)
// With KS > 1 each warp forms X^T and Y^T over its rows only; the KS partial
// sums meet in shared memory and every warp of the block adds them in the same
// order, so all of them hold the same D.  No other sum crosses a warp.
// mma.sync takes bf16 operands and accumulates in fp32; fp32 accuracy comes
// from splitting each factor in three bf16 parts (x = x0 + x1 + x2 exactly)
// and summing the six products x_i y_j with i + j <= 2: the three left out
// are below 2^-23 |x y| together.
template <int WPC, int KS>
struct PrefillScanSmem {
    static constexpr uint32_t XCH = KS > 1 ? WPC * KS * 32 * 16 * 4 : 0;  // partial sums [block][ks][lane][16]
    static constexpr uint32_t BYTES = 2 * PCH_BYTES + XCH + 16;          // two chunk buffers, two barriers
};

template <typename ST, int WPC, int KS, bool FULLK>
__global__ void __launch_bounds__(WPC * KS * 32, 1) kda_prefill_scan_kernel(const StepParams p,
                                                                           const uint8_t* __restrict__ ws) {
    static_assert(WPC == 1 || WPC == 2 || WPC == 4 || WPC == 8, "column blocks per scan CTA");
    static_assert(KS == 1 || KS == 2 || KS == 4, "warps per column block");
    constexpr int NT = WPC * KS * 32, NTILE = KMAX / 8, MT = NTILE / KS;  // MT: row tiles per warp
    using SM = PrefillScanSmem<WPC, KS>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* xch = reinterpret_cast<float*>(smem + 2 * PCH_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * PCH_BYTES + SM::XCH);  // two chunk-operand barriers

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cbk = warp / KS, ks = warp - cbk * KS;
    const int g = lane >> 2, qd = lane & 3;
    const int ctiles = (p.v + 16 * WPC - 1) / (16 * WPC);
    const int tile = (int)blockIdx.x;
    const int r = tile / (p.hv * ctiles);
    const int rem = tile - r * p.hv * ctiles;
    const int h = rem / ctiles, cb = rem - h * ctiles;
    const int c0 = (cb * WPC + cbk) * 16;
    const bool wact = c0 < p.v;  // V is a multiple of 16: a block's columns are all in or all out
    const int t0 = ks * MT;      // this warp's first row tile
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
        for (int e = tid; e < Tn * 16 * WPC; e += NT) {
            const int c2 = cb * 16 * WPC + (e % (16 * WPC));
            if (c2 < p.v) p.o[((int64_t)(tb + e / (16 * WPC)) * p.hv + h) * p.v + c2] = 0.f;
        }
        return;
    }
    // a request with no tokens stores its initial state (zero on a reset) to
    // its final slot: the state after its last token
    if (Tn == 0 && fin_slot < 0) return;
    const int nch = (Tn + PCH - 1) / PCH;
    const int nkt = FULLK ? NTILE : p.k / 8;  // row tiles in use (K is a multiple of 16)

    // this warp's rows of the state, transposed, in accumulator fragments
    float acc[MT][4];
    const bool rst = p.reset != nullptr && p.reset[r] != 0;
    const ST* src = static_cast<const ST*>(p.pool) + state_at(p, slot, h);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int row = 8 * (t0 + mt) + 2 * qd + (e & 1), col = c0 + g + 8 * (e >> 1);
            acc[mt][e] = (!rst && wact && t0 + mt < nkt) ? to_f32(src[(int64_t)row * p.v + col]) : 0.f;
        }

    // chunk j's operand block -> buffer j % 2, one barrier per buffer
    auto issue = [&](int j) {
        const uint8_t* blk = ws + (prefill_chunk_slot(tb, r, j) * p.hv + h) * (int64_t)PCH_BYTES;
        uint64_t* bar = bars + (j & 1);
        mbar_arrive_expect_tx(bar, PCH_BYTES);
        bulk_load(smem + (j & 1) * PCH_BYTES, blk, PCH_BYTES, bar);
    };
    if (tid == 0) {
        mbar_init(bars, 1);
        mbar_init(bars + 1, 1);
        fence_mbar_init();
        if (nch > 0) issue(0);
    }
    __syncthreads();

    // ldmatrix lane addresses (bytes inside a part matrix): lane l reads row
    // (l & 7) of 8 x 8 block l / 8.  W', Q' as B[k = row of S][n = token]:
    // blocks (tokens 0-7 | 8-15) x (k 0-7 | 8-15); Ke as B[k = token][n = row
    // of S], transposed: blocks (tokens 0-7 | 8-15) x (two row tiles)
    const uint32_t lwq = ((lane & 7) + 8 * (lane >> 4)) * (PT_ROW * 2) + 16 * ((lane >> 3) & 1);
    const uint32_t lke = ((lane & 7) + 8 * ((lane >> 3) & 1)) * (PT_ROW * 2) + 16 * (lane >> 4);

    // chunk j is buffer j % 2's (j / 2)-th use: barrier parity (j / 2) % 2
    int jfail = -1, issued = nch > 0 ? 1 : 0;
    for (int j = 0; j < nch; ++j) {
        if (j + 1 < nch) {  // its buffer's last readers were done with chunk j - 1
            if (tid == 0) issue(j + 1);
            ++issued;
        }
        const bool ok = mbar_wait(bars + (j & 1), (j >> 1) & 1);
        if (__syncthreads_or(ok ? 0 : 1)) {
            jfail = j;
            break;
        }
        const uint8_t* buf = smem + (j & 1) * PCH_BYTES;
        const uint32_t bw = smem_u32(buf + PB_W), bq = smem_u32(buf + PB_Q), bke = smem_u32(buf + PB_K);
        const float* cc = reinterpret_cast<const float*>(buf + PB_C);
        const float* U = reinterpret_cast<const float*>(buf + PB_U);
        const float* OI = reinterpret_cast<const float*>(buf + PB_OI);
        // X^T (tiles 0, 1: tokens 0-7, 8-15) and Y^T (tiles 2, 3) over this
        // warp's rows: the leading product and the five small ones in
        // separate sums, each of those per k-step parity (shorter chains)
        float xs[4][4];
        {
            float xh[4][4], xl[2][4][4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) { xh[t][e] = 0.f; xl[0][t][e] = 0.f; xl[1][t][e] = 0.f; }
#pragma unroll
            for (int kk = 0; kk < MT / 2; ++kk) {
                if (!wact || t0 + 2 * kk >= nkt) break;  // (unrolled: the state's tiles keep register indices)
                uint32_t a[3][4];
                split3_bf16x2(acc[2 * kk][0], acc[2 * kk][1], a[0][0], a[1][0], a[2][0]);
                split3_bf16x2(acc[2 * kk][2], acc[2 * kk][3], a[0][1], a[1][1], a[2][1]);
                split3_bf16x2(acc[2 * kk + 1][0], acc[2 * kk + 1][1], a[0][2], a[1][2], a[2][2]);
                split3_bf16x2(acc[2 * kk + 1][2], acc[2 * kk + 1][3], a[0][3], a[1][3], a[2][3]);
                const uint32_t kofs = (t0 / 2 + kk) * 32;
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    uint32_t b[3][4];
#pragma unroll
                    for (int part = 0; part < 3; ++part)
                        ldsm_x4((m ? bq : bw) + part * PART_BYTES + lwq + kofs, b[part][0], b[part][1], b[part][2],
                                b[part][3]);
#pragma unroll
                    for (int nh = 0; nh < 2; ++nh) {
                        float(&dh)[4] = xh[2 * m + nh];
                        float(&dl)[4] = xl[kk & 1][2 * m + nh];
                        const int i0 = 2 * nh, i1 = 2 * nh + 1;
                        mma_16816_bf16(dh, a[0][0], a[0][1], a[0][2], a[0][3], b[0][i0], b[0][i1]);
                        mma_16816_bf16(dl, a[0][0], a[0][1], a[0][2], a[0][3], b[1][i0], b[1][i1]);
                        mma_16816_bf16(dl, a[1][0], a[1][1], a[1][2], a[1][3], b[0][i0], b[0][i1]);
                        mma_16816_bf16(dl, a[0][0], a[0][1], a[0][2], a[0][3], b[2][i0], b[2][i1]);
                        mma_16816_bf16(dl, a[1][0], a[1][1], a[1][2], a[1][3], b[1][i0], b[1][i1]);
                        mma_16816_bf16(dl, a[2][0], a[2][1], a[2][2], a[2][3], b[0][i0], b[0][i1]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) xs[t][e] = xh[t][e] + (xl[0][t][e] + xl[1][t][e]);
        }
        if constexpr (KS > 1) {
            // the block's KS partial sums, added in the same order by every
            // warp of the block
            float4* mine = reinterpret_cast<float4*>(xch + ((cbk * KS + ks) * 32 + lane) * 16);
#pragma unroll
            for (int t = 0; t < 4; ++t) mine[t] = make_float4(xs[t][0], xs[t][1], xs[t][2], xs[t][3]);
            __syncthreads();
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                float4 sum = reinterpret_cast<const float4*>(xch + ((cbk * KS) * 32 + lane) * 16)[t];
#pragma unroll
                for (int k2 = 1; k2 < KS; ++k2) {
                    const float4 o4 = reinterpret_cast<const float4*>(xch + ((cbk * KS + k2) * 32 + lane) * 16)[t];
                    sum.x += o4.x; sum.y += o4.y; sum.z += o4.z; sum.w += o4.w;
                }
                xs[t][0] = sum.x; xs[t][1] = sum.y; xs[t][2] = sum.z; xs[t][3] = sum.w;
            }
        }
        if (wact) {
            // D^T = U^T - X^T; O^T = Y^T + O_intra^T for the chunk's tokens
            const int cl = min(PCH, Tn - j * PCH);
            float dd[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = 8 * nt + 2 * qd + (e & 1), col = c0 + g + 8 * (e >> 1);
                    dd[nt][e] = U[tok * PU_ROW + col] - xs[nt][e];
                    if (ks == 0 && tok < cl)
                        p.o[((int64_t)(tb + j * PCH + tok) * p.hv + h) * p.v + col] = xs[2 + nt][e] + OI[tok * PU_ROW + col];
                }
            // S^T <- S^T diag(c) + D^T Ke on this warp's rows
            uint32_t a[3][4];
            split3_bf16x2(dd[0][0], dd[0][1], a[0][0], a[1][0], a[2][0]);
            split3_bf16x2(dd[0][2], dd[0][3], a[0][1], a[1][1], a[2][1]);
            split3_bf16x2(dd[1][0], dd[1][1], a[0][2], a[1][2], a[2][2]);
            split3_bf16x2(dd[1][2], dd[1][3], a[0][3], a[1][3], a[2][3]);
#pragma unroll
            for (int np = 0; np < MT / 2; ++np) {
                if (t0 + 2 * np < nkt) {
                    uint32_t b[3][4];
#pragma unroll
                    for (int part = 0; part < 3; ++part)
                        ldsm_x4_trans(bke + part * PART_BYTES + lke + (t0 / 2 + np) * 32, b[part][0], b[part][1],
                                      b[part][2], b[part][3]);
#pragma unroll
                    for (int nh = 0; nh < 2; ++nh) {
                        float(&s4)[4] = acc[2 * np + nh];
                        const int row = 8 * (t0 + 2 * np + nh) + 2 * qd;
                        const float c_lo = cc[row], c_hi = cc[row + 1];
                        s4[0] *= c_lo; s4[1] *= c_hi; s4[2] *= c_lo; s4[3] *= c_hi;
                        const int i0 = 2 * nh, i1 = 2 * nh + 1;
                        mma_16816_bf16(s4, a[2][0], a[2][1], a[2][2], a[2][3], b[0][i0], b[0][i1]);
                        mma_16816_bf16(s4, a[1][0], a[1][1], a[1][2], a[1][3], b[1][i0], b[1][i1]);
                        mma_16816_bf16(s4, a[0][0], a[0][1], a[0][2], a[0][3], b[2][i0], b[2][i1]);
                        mma_16816_bf16(s4, a[1][0], a[1][1], a[1][2], a[1][3], b[0][i0], b[0][i1]);
                        mma_16816_bf16(s4, a[0][0], a[0][1], a[0][2], a[0][3], b[1][i0], b[1][i1]);
                        mma_16816_bf16(s4, a[0][0], a[0][1], a[0][2], a[0][3], b[0][i0], b[0][i1]);
                    }
                }
            }
        }
        // every thread is done with this buffer and the partial sums before
        // the next issue (generic reads, then async writes: fence first)
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
    if (fin_slot >= 0 && wact) {
        ST* dst = static_cast<ST*>(p.pool) + state_at(p, fin_slot, h);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = 8 * (t0 + mt) + 2 * qd + (e & 1), col = c0 + g + 8 * (e >> 1);
                if (t0 + mt < nkt) {
                    if constexpr (sizeof(ST) == 4) dst[(int64_t)row * p.v + col] = acc[mt][e];
                    else dst[(int64_t)row * p.v + col] = __float2half_rn(acc[mt][e]);
                }
            }
    }
}

}  // namespace kda
