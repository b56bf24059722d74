// KDA speculative verify, one CTA per tile, the tile staged by TMA (sm_103a).
//
// Tile: one (request n, value head h, block of BV state columns) with all K
// rows; BV * sizeof(state) is 64 or 128 bytes, one warp per 16-byte column
// chunk.  The state tile is TMA-loaded once from init_slot[n] (or taken as
// zero on reset); the per-token inputs are plain coalesced loads, thread r
// taking row r of q, k and a and column r of the v slice.  Lane l of warp w
// then carries rows l, l+32, l+64, l+96 of chunk w in fp32 registers through
// the T tokens without rounding.  After each
// token the state, rounded to the pool's dtype, is written to a swizzled
// shared-memory staging tile and from there to that token's snapshot slot
// snap_slot[n][t] (ROCm/ATOM pull request 2945, Changes: the state after each
// token goes to the token's snapshot slot through state_at) as one TMA box
// store, three staging buffers in turn (two in the wide shape).
//
// The general step: request n owns tokens cu[n] .. cu[n+1] - 1 of packed
// inputs (or n T .. n T + T - 1), reads its initial state from column
// accepted[n] - 1 (or 0) of its row of the slot table and stores token j's
// state to column j; value head h reads q/k head h / (hv / hqk); with
// MODE_PADDING a negative initial slot is a padding request (outputs zero,
// no state read or stored) and a negative snapshot slot is not kept.
//
// Tokens are taken in chunks of up to TC.  Within a chunk the recurrence
//   S_t = D_t S_{t-1} + beta_t khat_t d_t^T,   D_t = diag(alpha_t),
//   d_t = v_t - (D_t S_{t-1})^T khat_t,        o_t = S_t^T qhat_t / sqrt(K)
// unrolls from the chunk's initial state S_0.  With P_ts = D_{s+1} ... D_t
// (P_tt = I) and c_t = alpha_1 ... alpha_t (elementwise):
//   (D_t S_{t-1})^T khat_t = S_0^T (c_t khat_t) + sum_{s<t}  A_ts d_s,
//   S_t^T qhat_t           = S_0^T (c_t qhat_t) + sum_{s<=t} B_ts d_s,
//   A_ts = beta_s sum_i khat_s,i P_ts,ii khat_t,i,
//   B_ts = beta_s sum_i khat_s,i P_ts,ii qhat_t,i.
// So one pass over S_0 gives the 2 TC column sums of every token at once (no
// reduction waits on the previous token), each column solves its T x T
// lower-triangular system for d by forward substitution, and the snapshots
// then need only S_t = alpha_t S_{t-1} + (beta_t khat_t) d_t^T per element.
// Every sum is taken over the raw k and q: khat = k / |k| and the norms, like
// beta, are per-token scalars, so they multiply the 64 sums A and B, the
// column sums and d after the reductions.  The gates, the terms of A and B
// and the squared norms then come from one pass over the rows.
// It is the token-by-token recurrence with its sums taken in another order;
// the products P are formed by multiplication, never division, so alpha = 0
// stays exact.
// Barrier waits are bounded (1 s); one that runs out makes the CTA record
// KDA_ERR_TIMEOUT, wait once more (bounded) for its copies, and exit.
#pragma once

#include <type_traits>

#include "kda_common.cuh"
#include "kda_conv.cuh"

#ifndef KDA_VER_MINB
#define KDA_VER_MINB 3
#endif

namespace kda {

// WIDE: the shape for launches of more than one wave at 3 CTAs per SM (an
// fp16 pool with 16-bit inputs): 4 resident CTAs per SM, from a 128-register
// cap and two staging buffers instead of three.  A one-wave launch runs the
// default shape, whose extra registers and buffer shorten each CTA.
template <typename ST, int BV, int QES, bool WIDE = false>
struct VerifyShape {
    static constexpr int VEC = StateVec<ST>::VEC;
    static constexpr int ROWBYTES = BV * (int)sizeof(ST);
    static constexpr int NW = ROWBYTES / 16;  // warps, one per 16-byte column chunk
    static constexpr int NT = 32 * NW;
    // resident CTAs per SM the register budget must allow: at the configured
    // shapes a launch is about 2.5 CTAs per SM, so 3 keep it in one wave
    static constexpr int MINB = WIDE ? 4 : KDA_VER_MINB;
    static constexpr int ROWS = KMAX / 32;    // rows per lane
    // the row pass: thread r < KMAX takes key row r; with 2 KMAX threads (an
    // fp32 pool's 128-byte rows) thread KMAX + r takes row r as well and the
    // two split its terms of the sums A and B.  RW warps cover the rows once.
    static constexpr bool SPLIT = NT >= 2 * KMAX;
    static constexpr int RW = KMAX / 32;
    static constexpr int TC = 8;              // tokens per chunk
    static constexpr int NA = TC * (TC - 1) / 2, NB = TC * (TC + 1) / 2;  // 28 + 36 = 64 sums
    static constexpr int G = 16 / VEC;        // tokens per group of column sums (2 G VEC = 32 values)
    static constexpr uint32_t TILE_BYTES = (KMAX * ROWBYTES + 1023u) & ~1023u;
    // per token gates: float4 {c k, c q, alpha, k} per row (raw k and q), then v (fp32)
    static constexpr uint32_t G_V = KMAX * 16, G_TOK = G_V + BV * 4;
    static constexpr uint32_t GATE_BYTES = TC * G_TOK;
    static constexpr uint32_t WORK_BYTES = GATE_BYTES;
    // staging buffers for the snapshot stores (the state tile's area is the first)
    static constexpr int NSTAGE = WIDE ? 2 : 3;
    // norms [TC][NW][2] and b [TC], scalars [TC] float4, A and B per warp
    // [NW][64] then summed [64], column sums [TC][2][BV], d [TC][BV], snapshot ids [TC]
    static constexpr uint32_t RED_NORM = 0, RED_B = RED_NORM + TC * NW * 8;
    static constexpr uint32_t RED_SCAL = (RED_B + TC * 4 + 15u) & ~15u, RED_ABW = RED_SCAL + TC * 16;
    static constexpr uint32_t RED_AB = RED_ABW + NW * 64 * 4, RED_RES = RED_AB + 64 * 4;
    static constexpr uint32_t RED_D = RED_RES + TC * 2 * BV * 4, RED_SNAP = RED_D + TC * BV * 4;
    static constexpr uint32_t RED_BYTES = (RED_SNAP + TC * 4 + 15u) & ~15u;
    // tensor-core column sums (fp16 pool, first chunk, K = KMAX): the gates of
    // the 2 TC token-kind rows in three fp16 parts, stored key-major,
    // [3][KMAX][G16_STRIDE] halves: key row i holds its 2 TC values as two
    // 16-byte halves (gate rows 0-7 and 8-15; one thread's two stores per
    // part), the halves swapped in rows with bit 2 set (g16_half), so that
    // the 8 rows a transposing ldmatrix reads, and 8 threads' stores, fall in
    // distinct banks
    static constexpr bool MMA_CS = sizeof(ST) == 2 && 2 * TC == 16 && VEC == 8;
    static constexpr int G16_STRIDE = 2 * TC;
    static constexpr uint32_t G16_ARRAY = KMAX * G16_STRIDE * 2;
    static constexpr uint32_t G16_BYTES = MMA_CS ? 3 * G16_ARRAY : 0;
    static_assert(G16_STRIDE * 2 == 32, "g16_half: 32-byte key rows");
    static_assert(ROWBYTES == 128 || ROWBYTES == 64, "tile row bytes");
    static_assert(NT >= KMAX, "one thread per key row in the gate phase");
    static_assert(NA + NB == 64 && 2 * G * VEC == 32 && TC % G == 0 && TC == 8, "chunk shape");
    static_assert(BV == 32 && TC % NW == 0, "the solve: a lane per column, whole token shares per warp");
    // the gate matrix of the tensor-core column sums has one column per key
    // row, written by thread tid for row tid: exactly KMAX threads
    static_assert(!MMA_CS || NT == KMAX, "tensor-core column sums need one thread per key row");
    static_assert(NSTAGE >= 2, "staging buffers");
    static_assert(!WIDE || (sizeof(ST) == 2 && QES == 2), "the wide shape: fp16 pool, 16-bit inputs");
    static_assert(G_TOK % 16 == 0 &&
                  WORK_BYTES % 16 == 0 && RED_RES % 16 == 0 && RED_D % 16 == 0, "layout");
};

template <typename ST, int BV, int QES, bool WIDE = false>
constexpr size_t verify_smem_bytes() {
    using SH = VerifyShape<ST, BV, QES, WIDE>;
    return SH::NSTAGE * SH::TILE_BYTES + SH::WORK_BYTES + SH::RED_BYTES + SH::G16_BYTES + 16;
}

// Byte offset of 16-byte half h (gate rows 8 h .. 8 h + 7) of key row k in one
// part of the gate matrix.
__device__ __forceinline__ uint32_t g16_half(int k, int h) {
    return (uint32_t)(k * 32 + ((h ^ ((k >> 2) & 1)) << 4));
}

// Position of A_ts (s < t) and of B_ts (s <= t) among a chunk's 64 row sums.
__host__ __device__ constexpr int idx_a(int t, int s) { return t * (t - 1) / 2 + s; }
__host__ __device__ constexpr int idx_b(int t, int s) { return 28 + t * (t + 1) / 2 + s; }

// This row's terms of the row sums LO .. LO + 31 (A and B above): e runs
// through beta_s khat_s,i P_ts,ii for t = s, s + 1, ...  Every index is a
// compile-time constant, so only the 32 requested terms are formed.
template <int LO, int TC>
__device__ __forceinline__ void ab_terms(float (&out)[32], const float (&bk)[TC], const float (&kh)[TC],
                                         const float (&qh)[TC], const float (&al)[TC]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) out[i] = 0.f;
#pragma unroll
    for (int s = 0; s < TC; ++s) {
        float e = bk[s];
        if (idx_b(s, s) >= LO && idx_b(s, s) < LO + 32) out[idx_b(s, s) - LO] = e * qh[s];
#pragma unroll
        for (int t = s + 1; t < TC; ++t) {
            e *= al[t];
            if (idx_a(t, s) >= LO && idx_a(t, s) < LO + 32) out[idx_a(t, s) - LO] = e * kh[t];
            if (idx_b(t, s) >= LO && idx_b(t, s) < LO + 32) out[idx_b(t, s) - LO] = e * qh[t];
        }
    }
}

// The convolution fused in front of a speculative step (CONV), one channel:
// its history right-aligned in DCONV_H slots and its weights left-padded to
// match (slot i holds history entry i - (DCONV_H - (KW - 1)) and the weight
// that multiplies it; the slots before are zero and skipped), so that token
// j's taps are slots j .. j + DCONV_H - 1 of (history ++ the chunk's inputs)
// and then the input itself.  The fmaf chain runs the real taps in ascending
// order and the input last, as the conv kernel does, so y is bit-identical to
// kda_conv_step's.
template <typename QT>
__device__ __forceinline__ void sconv_load(QT (&z)[DCONV_H], float (&w)[DCONV_H], float& wl, float& b, const QT* W,
                                           int C, int KW, int acc, bool rst, const float* wp, const float* bias) {
    QT zero;
    conv_round(0.f, zero);
    const int pad = DCONV_H - (KW - 1);
#pragma unroll
    for (int i = 0; i < DCONV_H; ++i) {
        z[i] = !rst && i >= pad ? W[(int64_t)(acc + i - pad) * C] : zero;
        w[i] = i >= pad ? __ldg(wp + i - pad) : 0.f;
    }
    wl = __ldg(wp + KW - 1);
    b = bias != nullptr ? __ldg(bias) : 0.f;
}

template <typename QT, int TC>
__device__ __forceinline__ QT sconv_token(const QT (&z)[DCONV_H], const float (&w)[DCONV_H], float wl, float b,
                                          const QT (&xs)[TC], int KW, int silu, int j) {
    float s = b;
#pragma unroll
    for (int i = 0; i < DCONV_H; ++i)
        if (i >= DCONV_H - (KW - 1)) s = fmaf(w[i], to_f32(j + i < DCONV_H ? z[(j + i) % DCONV_H] : xs[(j + i + TC - DCONV_H) % TC]), s);
    s = fmaf(wl, to_f32(xs[j]), s);
    QT out;
    conv_round(silu ? silu_fast(s) : s, out);
    return out;
}

// The window of a channel after a step of Tn tokens is the last L entries of
// S = (old entries W[0 .. m-1]) ++ (the inputs x_0 .. x_(Tn-1)), m = acc +
// KW - 1 (old entries zero on reset).  From registers: z holds S[m - DCONV_H
// + i] in its real slots (the history) and xs[j] = S[m + j]; each register's
// destination is computed, no register index is.  Older kept entries (below
// the history) are read again first, in batches read whole before they are
// written: their sources lie at or above their destinations and may be
// register destinations too, so they move before those are written.
template <typename QT, int TC>
__device__ __forceinline__ void sconv_window_store_regs(QT* W, int C, int L, int KW, int m, int Tn, bool rst,
                                                        const QT (&z)[DCONV_H], const QT (&xs)[TC]) {
    QT zero;
    conv_round(0.f, zero);
    const int first = m + Tn - L;     // S index of new entry 0 (>= 0: kept <= m)
    const int lo = m - (KW - 1);      // the lowest S index the registers hold
    for (int e0 = 0; first + e0 < lo && e0 < L; e0 += 8) {
        QT v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u;
            v[u] = first + e < lo && e < L && !rst ? W[(int64_t)(first + e) * C] : zero;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (first + e0 + u < lo && e0 + u < L) W[(int64_t)(e0 + u) * C] = v[u];
    }
#pragma unroll
    for (int i = 0; i < DCONV_H; ++i) {
        const int e = m - DCONV_H + i - first;
        if (i >= DCONV_H - (KW - 1) && e >= 0 && e < L) W[(int64_t)e * C] = z[i];
    }
#pragma unroll
    for (int j = 0; j < TC; ++j) {
        const int e = m + j - first;
        if (j < Tn && e >= 0 && e < L) W[(int64_t)e * C] = xs[j];
    }
}

// The same window update for two channels c0, c1 from memory (the q/k
// windows, written by their last reader at the end): all of a batch of 16
// entries of both channels are read before any is written, so a window of up
// to 16 entries costs one round trip.
template <typename QT>
__device__ __forceinline__ void sconv_window_store2(QT* W, const QT* X, int c0, int c1, int C, int L, int m, int Tn,
                                                    bool rst) {
    QT zero;
    conv_round(0.f, zero);
    const int kept = max(0, L - Tn), nin = min(Tn, L);
    for (int e0 = 0; e0 < L; e0 += 16) {
        QT v0[16], v1[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int e = e0 + u;
            const bool old = e < kept;
            const int64_t src = old ? (int64_t)(m - kept + e) * C : (int64_t)(Tn - nin + e - kept) * C;
            v0[u] = e >= L || (old && rst) ? zero : (old ? W[src + c0] : X[src + c0]);
            v1[u] = e >= L || (old && rst) ? zero : (old ? W[src + c1] : X[src + c1]);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (e0 + u < L) {
                W[(int64_t)(e0 + u) * C + c0] = v0[u];
                W[(int64_t)(e0 + u) * C + c1] = v1[u];
            }
    }
}

// FULLK: K = KMAX, known at compile time (the row guards and loops fold away).
// CONV on an fp32 pool: 2 CTAs per SM (128 registers), the 256-thread tile
// having no room for the convolution's inputs under the 3-CTA cap of 80.
template <typename ST, typename QT, int BV, bool FULLK, bool WIDE = false, bool CONV = false>
__global__ void __launch_bounds__(VerifyShape<ST, BV, (int)sizeof(QT), WIDE>::NT,
                                  CONV && sizeof(ST) == 4 ? 2 : VerifyShape<ST, BV, (int)sizeof(QT), WIDE>::MINB)
kda_verify_kernel(const __grid_constant__ CUtensorMap tmap, const StepParams p) {
// key rows: KMAX in the K = KMAX build, else read from the parameters where used
#define KK (FULLK ? KMAX : p.k)
    using SH = VerifyShape<ST, BV, (int)sizeof(QT), WIDE>;
    using SV = StateVec<ST>;
    constexpr int VEC = SH::VEC, NW = SH::NW, ROWS = SH::ROWS, TC = SH::TC, G = SH::G;

    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* gts = smem + SH::NSTAGE * SH::TILE_BYTES;
    uint8_t* redb = gts + SH::WORK_BYTES;
    float* nrm = reinterpret_cast<float*>(redb + SH::RED_NORM);    // [TC][NW][2]
    float* bsm = reinterpret_cast<float*>(redb + SH::RED_B);       // [TC]
    float4* scal = reinterpret_cast<float4*>(redb + SH::RED_SCAL); // [TC] {beta, 1/|k|, 1/|q|, -}
    float* abw = reinterpret_cast<float*>(redb + SH::RED_ABW);     // [NW][64]
    float* ab = reinterpret_cast<float*>(redb + SH::RED_AB);       // [64]
    float* res = reinterpret_cast<float*>(redb + SH::RED_RES);     // [TC][2][BV]
    float* dsm = reinterpret_cast<float*>(redb + SH::RED_D);       // [TC][BV]
    int32_t* snaps = reinterpret_cast<int32_t*>(redb + SH::RED_SNAP);  // [TC]
    __half* g16 = reinterpret_cast<__half*>(redb + SH::RED_BYTES);  // [3][KMAX][G16_STRIDE] (fp16 pool)
    uint64_t* bar_st = reinterpret_cast<uint64_t*>(redb + SH::RED_BYTES + SH::G16_BYTES);
    const uint32_t tile_base = smem_u32(smem);
    const uint32_t gate_base = smem_u32(gts);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = warp;
    const int rowt = SH::SPLIT ? (tid & (KMAX - 1)) : tid;  // this thread's key row in the row pass
    const int half = SH::SPLIT ? tid / KMAX : 0;             // which half of the terms (uniform per warp)
    const int vt = (p.v + BV - 1) / BV;
    const int tile = (int)blockIdx.x;
    const int r = tile / vt;  // n * hv + h
    const int cb = tile - r * vt;
    const int n = r / p.hv;
    const int h = r - n * p.hv;
    const int T = p.t;  // most tokens a request may have
    const int hq = h / (p.hv / p.hqk);  // q/k head of value head h
    const int vcols = min(BV, p.v - cb * BV);
    if ((tile_base & 1023u) != 0) {  // the swizzled tile needs a 1024-byte aligned base
        if (tid == 0) atomicCAS(p.status, 0, STATUS_SMEM_ALIGN);
        return;
    }

    int tb = n * T, Tn = T;  // request n's packed tokens tb .. tb + Tn - 1 (set below)
    // Row tid of k, q and a, and column tid of this tile's v slice, of tokens
    // t0 .. t0 + tc - 1 (tc >= 1), straight into registers: coalesced loads,
    // none of which depends on a slot id.  Every load is unconditional, from
    // an address clamped into the request's last token, row 0 or column 0,
    // so that all of them are in flight at once; the values past tc or the
    // row or column count are zeroed where they are used.
    // fp16 inputs of a 256-thread (fp32 pool) tile are held as fp32: as 16-bit
    // values they need more registers than its 85-register budget allows
    using RT = typename std::conditional<sizeof(ST) == 4 && std::is_same<QT, __half>::value, float, QT>::type;
    RT kraw[TC], qraw[TC], vraw[TC];
    float araw[TC];
    // CONV: the fused convolution makes q, k and v: thread r the q and k
    // channels of key row r, thread j < vcols the tile's value column j.  The
    // window slot, accepted index and checks are set in the prologue, which
    // also loads each channel's history (at the accepted index), weights and
    // bias (early with KDA_LAUNCH_PDL_EARLY_STATE); load_inputs then issues
    // every input of the chunk before the first sum.  One chunk: the host
    // refuses longer requests.  The value column's inputs stay for its window.
    int32_t cslot = 0;
    int cacc = 0;
    bool conv_ok = false;
    QT zq[DCONV_H], zk[DCONV_H], zv[DCONV_H], xv[TC];
    float wq[DCONV_H], wk[DCONV_H], wv[DCONV_H], lq = 0.f, lk = 0.f, lv = 0.f, bq = 0.f, bk = 0.f, bv = 0.f;
    auto load_inputs = [&](int t0, int tc) {
        const int row = rowt < KK ? rowt : 0, col = tid < vcols ? tid : 0;
        if constexpr (CONV) {
            const auto& cp = p.conv;
            const QT* X = static_cast<const QT*>(cp.x);
            const int qc = hq * KK + row, kc = (p.hqk + hq) * KK + row, vc = 2 * p.hqk * KK + h * p.v + cb * BV + col;
            QT xq[TC], xk[TC];
#pragma unroll
            for (int j = 0; j < TC; ++j) {
                const int64_t tok = (int64_t)tb + t0 + min(j, tc - 1);
                xq[j] = X[tok * cp.C + qc];
                xk[j] = X[tok * cp.C + kc];
                xv[j] = X[tok * cp.C + vc];
                araw[j] = __ldg(p.a + (tok * p.hv + h) * KK + row);
            }
            // y only for a request whose window is valid (a padding request's
            // rows are zeroed where it leaves; a bad one is left alone)
            QT* Y = static_cast<QT*>(cp.y);
            const bool yqk = Y != nullptr && conv_ok && h % (p.hv / p.hqk) == 0 && cb == 0 && rowt < KK && half == 0;
            const bool yvv = Y != nullptr && conv_ok && tid < vcols;
#pragma unroll
            for (int j = 0; j < TC; ++j) {
                const QT yq = sconv_token(zq, wq, lq, bq, xq, cp.KW, cp.silu, j);
                const QT yk = sconv_token(zk, wk, lk, bk, xk, cp.KW, cp.silu, j);
                const QT yw = sconv_token(zv, wv, lv, bv, xv, cp.KW, cp.silu, j);
                qraw[j] = (RT)yq;
                kraw[j] = (RT)yk;
                vraw[j] = (RT)yw;
                if (j < tc) {  // one writer of each y
                    const int64_t tok = (int64_t)tb + t0 + j;
                    if (yqk) {
                        Y[tok * cp.C + qc] = yq;
                        Y[tok * cp.C + kc] = yk;
                    }
                    if (yvv) Y[tok * cp.C + vc] = yw;
                }
            }
        } else {
            const QT* qp = static_cast<const QT*>(p.q);
            const QT* kp = static_cast<const QT*>(p.kk);
            const QT* vp = static_cast<const QT*>(p.vv);
#pragma unroll
            for (int j = 0; j < TC; ++j) {
                const int64_t tok = (int64_t)tb + t0 + min(j, tc - 1);
                const int64_t rq = (tok * p.hqk + hq) * KK + row, rt = tok * p.hv + h;
                kraw[j] = (RT)kp[rq];
                qraw[j] = (RT)qp[rq];
                araw[j] = __ldg(p.a + rt * KK + row);
                vraw[j] = (RT)vp[rt * p.v + (int64_t)cb * BV + col];
            }
        }
    };

    // Programmatic dependent launch: as in the decode kernel, only the slot ids
    // and the state may be read before the previous kernel completes, and only
    // when the caller vouches for it (KDA_LAUNCH_PDL_EARLY_STATE).  The first
    // chunk's inputs are requested as soon as that allows.
    cudaTriggerProgrammaticLaunchCompletion();
    const bool early = (p.flags & LAUNCH_PDL_EARLY_STATE) != 0;
    if (tid == 0) {
        mbar_init(bar_st, 1);
        fence_mbar_init();
    }
    if (!early) cudaGridDependencySynchronize();
    // The index metadata (token range, accepted column, slot ids) is requested
    // first, the inputs while it is in flight.  Request n owns tokens
    // tb .. tb + Tn - 1; its initial slot is column accepted[n] - 1 (or 0) of
    // its row of init_slot, and token j's snapshot goes to column j of its row
    // of snap_slot.
    if (p.cu != nullptr) {
        tb = p.cu[n];
        Tn = p.cu[n + 1] - tb;
    }
    const bool range_ok = tb >= 0 && Tn >= 0 && Tn <= T && (int64_t)tb + Tn <= p.total;
    int col = 0;
    if (p.accepted != nullptr) col = p.accepted[n] - 1;
    const bool arg_ok = range_ok && col >= 0 && col < p.num_cols;
    const int32_t slot = arg_ok ? p.init_slot[(int64_t)n * p.init_stride + col] : 0;
    const bool final_mode = p.final_slot != nullptr;  // prefill: no snapshots, one final store
    const int32_t snap0 = !final_mode && arg_ok && lane < Tn ? p.snap_slot[(int64_t)n * p.snap_stride + lane] : 0;
    const int32_t fin = final_mode ? p.final_slot[n] : -1;
    const bool issued = arg_ok && Tn > 0;  // the first chunk's inputs are requested
    // CONV: the window slot and the geometry of its update (history at the
    // accepted index acc = col; m = acc + KW - 1 entries before the inputs,
    // kept = max(0, L - Tn) of them kept)
    bool conv_geom = true, conv_slot_ok = true;
    if constexpr (CONV) {
        const auto& cp = p.conv;
        cslot = arg_ok ? cp.slot[n] : 0;
        cacc = col;
        const int m = col + cp.KW - 1, kept = max(0, cp.L - Tn);
        conv_geom = m <= cp.L && kept <= m;
        conv_slot_ok = cslot >= 0 && cslot < cp.num_slots;
        conv_ok = arg_ok && conv_geom && conv_slot_ok;
        if (issued) {  // no window read unless valid (zero history otherwise)
            const bool rs = !conv_ok || (p.reset != nullptr && p.reset[n] != 0);
            const QT* W = static_cast<const QT*>(cp.window) + (int64_t)(conv_ok ? cslot : 0) * cp.slot_stride;
            const int row = rowt < KK ? rowt : 0, vcol = tid < vcols ? tid : 0;
            const int qc = hq * KK + row, kc = (p.hqk + hq) * KK + row, vc = 2 * p.hqk * KK + h * p.v + cb * BV + vcol;
            sconv_load(zq, wq, lq, bq, W + qc, cp.C, cp.KW, cacc, rs, cp.w + (int64_t)qc * cp.KW,
                       cp.bias != nullptr ? cp.bias + qc : nullptr);
            sconv_load(zk, wk, lk, bk, W + kc, cp.C, cp.KW, cacc, rs, cp.w + (int64_t)kc * cp.KW,
                       cp.bias != nullptr ? cp.bias + kc : nullptr);
            sconv_load(zv, wv, lv, bv, W + vc, cp.C, cp.KW, cacc, rs, cp.w + (int64_t)vc * cp.KW,
                       cp.bias != nullptr ? cp.bias + vc : nullptr);
        }
    }
    // The first chunk's inputs: in the prologue, under the slot-id loads,
    // when the registers allow it (128-thread tiles); else with the chunk.
    constexpr bool PRO_INPUTS = SH::NT <= 128;
    if (PRO_INPUTS && !early && issued) load_inputs(0, min(TC, Tn));
    const bool padding = (p.mode & MODE_PADDING) != 0;
    auto slot_bad = [&](int32_t s) { return s >= p.num_slots || (s < 0 && !padding); };
    bool bad = !arg_ok || slot_bad(slot) || slot_bad(snap0) || fin >= p.num_slots;
    const bool conv_bad = CONV && arg_ok && Tn > 0 && !(slot < 0 && padding) && !(conv_geom && conv_slot_ok);
    bad |= conv_bad;
    for (int t = lane + 32; !final_mode && arg_ok && t < Tn; t += 32)
        bad |= slot_bad(p.snap_slot[(int64_t)n * p.snap_stride + t]);
    bad = __any_sync(0xffffffffu, bad);  // the same answer in every warp
    const bool pad = !bad && slot < 0;     // a padding request
    const bool rst = !bad && p.reset != nullptr && p.reset[n] != 0;
    // A prefill request with no tokens still stores its initial state (zero on
    // a reset) to its final slot: the state after its last token.
    const bool need_state = Tn > 0 || (final_mode && fin >= 0);
    if (tid == 0 && !bad && !pad && !rst && need_state) {
        prefetch_tmap(&tmap);
        mbar_arrive_expect_tx(bar_st, (uint32_t)KK * SH::ROWBYTES);
        if (!(p.flags & LAUNCH_TEST_WITHHOLD_STATE))  // the test hook: the wait runs out
            tma_load_3d(smem, &tmap, bar_st, cb * BV, h * KK, slot);
    }
    if (early) {
        cudaGridDependencySynchronize();
        if (PRO_INPUTS && issued) load_inputs(0, min(TC, Tn));
    }
    if (bad || pad || !need_state) {
        if (pad)  // padding: this tile's outputs of every token are zero
            for (int e = tid; e < Tn * vcols; e += SH::NT)
                p.o[((int64_t)(tb + e / vcols) * p.hv + h) * p.v + cb * BV + e % vcols] = 0.f;
        if constexpr (CONV) {  // ... and so are its conv outputs (its window is left alone)
            if (pad && p.conv.y != nullptr) {
                const auto& cp = p.conv;
                QT* Y = static_cast<QT*>(cp.y);
                QT zero;
                conv_round(0.f, zero);
                const int qc = hq * KK + rowt, kc = (p.hqk + hq) * KK + rowt, vc = 2 * p.hqk * KK + h * p.v + cb * BV + tid;
                for (int j = 0; j < Tn; ++j) {
                    const int64_t row0 = ((int64_t)tb + j) * cp.C;
                    if (h % (p.hv / p.hqk) == 0 && cb == 0 && rowt < KK && half == 0) {
                        Y[row0 + qc] = zero;
                        Y[row0 + kc] = zero;
                    }
                    if (tid < vcols) Y[row0 + vc] = zero;
                }
            }
        }
        if (tid == 0 && bad) atomicCAS(p.status, 0, arg_ok && conv_geom ? STATUS_SLOT_RANGE : STATUS_ARG);
        return;  // uniform; no state copy was issued
    }
    __syncthreads();  // barriers initialised
    // CONV: a value column's window belongs to this CTA alone: rewrite it from
    // the registers, once the request is known valid (the inputs' registers
    // hold it from here: 128-thread tiles load the first chunk in the
    // prologue; the 256-thread ones do so in the loop, and rewrite it there)
    auto conv_v_store = [&]() {
        if constexpr (CONV) {
            if (tid < vcols) {
                const auto& cp = p.conv;
                const int vc = 2 * p.hqk * KK + h * p.v + cb * BV + tid;
                sconv_window_store_regs(static_cast<QT*>(cp.window) + (int64_t)cslot * cp.slot_stride + vc, cp.C,
                                        cp.L, cp.KW, cacc + cp.KW - 1, Tn, rst, zv, xv);
            }
        }
    };
    if constexpr (PRO_INPUTS) conv_v_store();

    // the carry as pairs of adjacent columns: each pair's update is one packed
    // fp32 FMA (two fmaf with their own rounding, the same results)
    constexpr int VP = VEC / 2;
    float2 x[ROWS][VP];
    bool state_in = false;
    bool alive = true;
    int conv_prev = -1;  // CONV: this CTA's read count before its own, once counted
    if (Tn == 0) {  // prefill, empty prompt: the loaded tile (or zeros) goes to the final slot as is
        const bool ok = rst || mbar_wait(bar_st, 0);
        if (__syncthreads_or(ok ? 0 : 1)) {
            alive = false;
        } else {
            if (rst) {
                for (int e = tid; e < KK * (SH::ROWBYTES / 16); e += SH::NT)
                    sts128(tile_base + e * 16, make_uint4(0u, 0u, 0u, 0u));
                fence_proxy_async_smem();
            }
            __syncthreads();
            if (tid == 0) {
                tma_store_3d(&tmap, smem, cb * BV, h * KK, fin);
                bulk_commit();
            }
        }
    }
    const bool scaled = p.a_log != nullptr;
    const float gscale = scaled ? expf(__ldg(p.a_log + h)) : 1.f;
    const float gbias = p.dt_bias != nullptr && rowt < KK ? __ldg(p.dt_bias + (int64_t)h * KK + rowt) : 0.f;
    for (int t0 = 0; t0 < Tn; t0 += TC) {
        const int tc = min(TC, Tn - t0);
        // CONV: one chunk (the host refuses longer requests), so the conv's
        // history and weights die with the first call
        if (CONV ? (t0 == 0 && !PRO_INPUTS) : (t0 > 0 || !PRO_INPUTS)) load_inputs(t0, tc);
        if constexpr (!PRO_INPUTS) {
            if (t0 == 0) conv_v_store();
        }
        if (tid < tc) {
            bsm[tid] = __ldg(p.b + ((int64_t)tb + t0 + tid) * p.hv + h);
            snaps[tid] = final_mode ? -1 : p.snap_slot[(int64_t)n * p.snap_stride + t0 + tid];
        }

        // (1) row tid of every token, in one pass: alpha; the gates
        // {c k, c q, alpha, k} and v into shared memory; this row's terms of
        // the 64 raw sums A and B and of the squared norms, summed over the
        // warp's rows (reduce-scatters: lane pair 2m holds norm value m, lane
        // L sum L of each half of A and B) and stored per warp
        {
            float kt[TC], qt[TC], at[TC];
#pragma unroll
            for (int j = 0; j < TC; ++j) {
                const bool in_row = j < tc && rowt < KK;
                kt[j] = in_row ? to_f32(kraw[j]) : 0.f;
                qt[j] = in_row ? to_f32(qraw[j]) : 0.f;
                at[j] = in_row ? araw[j] : 0.f;
            }
            if (tid < BV)
#pragma unroll
                for (int j = 0; j < TC; ++j)
                    if (j < tc)
                        reinterpret_cast<float*>(gts + j * SH::G_TOK + SH::G_V)[tid] =
                            tid < vcols ? to_f32(vraw[j]) : 0.f;
            // the decay, one branch for all tokens
            if (scaled) {
#pragma unroll
                for (int j = 0; j < TC; ++j) at[j] = j < tc && rowt < KK ? gate_alpha(at[j], true, gscale, gbias) : 0.f;
            } else {
#pragma unroll
                for (int j = 0; j < TC; ++j) at[j] = j < tc && rowt < KK ? gate_alpha(at[j], false, gscale, gbias) : 0.f;
            }
            // the first chunk of an fp16 pool at K = KMAX takes its column sums
            // on the tensor cores: rows 2 j (c k) and 2 j + 1 (c q) of the gate
            // matrix, each value split into three fp16 parts g = h0 + h1 2^-11 +
            // h2 2^-22 (exact differences; the rest is below 2^-33 |g|)
            const bool mma_cs = SH::MMA_CS && t0 == 0 && !rst && KK == KMAX;
            float2 gpair[TC];  // {c k, c q} of token j: gate-matrix rows 2 j and 2 j + 1
            float cdec = 1.f;
#pragma unroll
            for (int j = 0; j < TC; ++j) {
                cdec *= at[j];  // c_j: alpha of tokens 0 .. j
                gpair[j] = make_float2(cdec * kt[j], cdec * qt[j]);
                if (j < tc && tid < KK)
                    reinterpret_cast<float4*>(gts + j * SH::G_TOK)[tid] = make_float4(gpair[j].x, gpair[j].y, at[j], kt[j]);
            }
            if constexpr (SH::MMA_CS) {
                // past tc the raw k and q are zero, so are those rows; thread
                // tid < KMAX = NT writes key row tid of each part
                if (mma_cs) {
                    uint32_t part[3][TC];
#pragma unroll
                    for (int j = 0; j < TC; ++j) {
                        const float2 g = gpair[j];
                        const __half2 h0 = __float22half2_rn(g);
                        const float2 f0 = __half22float2(h0);
                        const float2 r1 = make_float2((g.x - f0.x) * 2048.f, (g.y - f0.y) * 2048.f);
                        const __half2 h1 = __float22half2_rn(r1);
                        const float2 f1 = __half22float2(h1);
                        const __half2 h2 = __float22half2_rn(make_float2((r1.x - f1.x) * 2048.f, (r1.y - f1.y) * 2048.f));
                        part[0][j] = *reinterpret_cast<const uint32_t*>(&h0);
                        part[1][j] = *reinterpret_cast<const uint32_t*>(&h1);
                        part[2][j] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    const uint32_t lo = smem_u32(g16) + g16_half(tid, 0), hi = smem_u32(g16) + g16_half(tid, 1);
#pragma unroll
                    for (int q = 0; q < 3; ++q) {
                        sts128(lo + q * SH::G16_ARRAY, make_uint4(part[q][0], part[q][1], part[q][2], part[q][3]));
                        sts128(hi + q * SH::G16_ARRAY, make_uint4(part[q][4], part[q][5], part[q][6], part[q][7]));
                    }
                }
            }
            if (half == 0) {  // the first RW warps: the squared norms
                float sq[2 * TC];
#pragma unroll
                for (int j = 0; j < TC; ++j) { sq[2 * j] = kt[j] * kt[j]; sq[2 * j + 1] = qt[j] * qt[j]; }
                const float s = warp_reduce_scatter<2 * TC>(sq, lane);
                if ((lane & 1) == 0) {
                    const int m = lane >> 1;  // token m >> 1, k (even) or q (odd)
                    nrm[((m >> 1) * SH::RW + warp) * 2 + (m & 1)] = s;
                }
            }
            float part[32];
            if (!SH::SPLIT || half == 0) {
                ab_terms<0, TC>(part, kt, kt, qt, at);
                abw[(warp % SH::RW) * 64 + lane] = warp_reduce_scatter<32>(part, lane);
            }
            if (!SH::SPLIT || half == 1) {
                ab_terms<32, TC>(part, kt, kt, qt, at);
                abw[(warp % SH::RW) * 64 + 32 + lane] = warp_reduce_scatter<32>(part, lane);
            }
        }
        {  // the initial state arrives (first chunk) while the rows are summed
            bool ok = true;
            if (!state_in) ok = rst || mbar_wait(bar_st, 0);
            if (__syncthreads_or(ok ? 0 : 1)) {
                alive = false;
                break;
            }
        }
        if constexpr (CONV) {
            // every thread has used the window values it read (they fed the
            // row pass, before the barrier above): thread 0 counts the CTA's
            // read of its q/k windows; the result is needed only at the end
            if (tid == 0 && t0 == 0 && (p.hv / p.hqk) * vt > 1)
                conv_prev = atomicAdd(p.conv.counters + (int64_t)n * p.hqk + hq, 1);
        }
        if (!state_in) {
#pragma unroll
            for (int rr = 0; rr < ROWS; ++rr) {
                const int row = lane + 32 * rr;
                if (!rst && row < KK) SV::widen2(lds128(tile_base + swz<SH::ROWBYTES>(row, chunk)), x[rr]);
                else
#pragma unroll
                    for (int c = 0; c < VP; ++c) x[rr][c] = make_float2(0.f, 0.f);
            }
            state_in = true;
        }
        // (2) the scalars, beside the column sums: thread e < 64 finishes sum e
        // of A and B, scaled by beta_s / (|k_s| |k_t|) or beta_s / (|k_s| |q_t|);
        // threads 64 .. 64 + tc - 1 keep {beta, 1/|k|, 1/|q|} of their token
        if (tid < 64) {
            const bool is_a = tid < 28;
            int t = is_a ? 1 : 0, s = 0;
            if (is_a) {
#pragma unroll
                for (int u = 2; u < TC; ++u) t += idx_a(u, 0) <= tid ? 1 : 0;
                s = tid - idx_a(t, 0);
            } else {
#pragma unroll
                for (int u = 1; u < TC; ++u) t += idx_b(u, 0) <= tid ? 1 : 0;
                s = tid - idx_b(t, 0);
            }
            float v = 0.f;
            if (t < tc) {
                float ks = 0.f, rt = 0.f;
#pragma unroll
                for (int w = 0; w < SH::RW; ++w) {
                    v += abw[w * 64 + tid];
                    ks += nrm[(s * SH::RW + w) * 2 + 0];
                    rt += nrm[(t * SH::RW + w) * 2 + (is_a ? 0 : 1)];
                }
                const float beta = sigmoid_neg(-bsm[s]);  // sigmoid(b_s)
                v *= beta * __frsqrt_rn(ks + L2_EPS) * __frsqrt_rn(rt + L2_EPS);
            }
            ab[tid] = v;
        } else if (tid < 64 + tc) {
            const int t = tid - 64;
            float kk2 = 0.f, qq2 = 0.f;
#pragma unroll
            for (int w = 0; w < SH::RW; ++w) {
                kk2 += nrm[(t * SH::RW + w) * 2 + 0];
                qq2 += nrm[(t * SH::RW + w) * 2 + 1];
            }
            scal[t] = make_float4(sigmoid_neg(-bsm[t]), __frsqrt_rn(kk2 + L2_EPS),
                                  __frsqrt_rn(qq2 + L2_EPS), 0.f);
        }

        // (3) the column sums of the chunk's initial state against c k and
        // c q of every token.  Tensor cores where the first chunk's state is
        // the fp16 tile itself: warp w multiplies the 16 x 128 gate matrix by
        // its 128 x 8 slice of the tile, once per fp16 part, and adds the
        // parts' fp32 sums at their scales (rows and columns of the products:
        // lane l holds rows l / 4 and l / 4 + 8, columns 2 (l % 4) and + 1)
        if constexpr (SH::MMA_CS) {
            if (t0 == 0 && !rst && KK == KMAX) {
                float acc[3][4] = {};
                // lane l addresses row r = l % 8 of 8 x 8 block l / 8 of the A
                // fragment (m 0-7 | 8-15 by l / 8 odd, k 0-7 | 8-15 by l / 16),
                // stored k-major: key row kb + (l / 16) 8 + r, half (l / 8) % 2.
                // kb is a multiple of 16, so the swap of the halves depends on
                // r alone and row kb adds kb * 32 bytes
                const uint32_t gb16 = smem_u32(g16) + g16_half((lane >> 4) * 8 + (lane & 7), (lane >> 3) & 1);
#pragma unroll
                for (int kb = 0; kb < KMAX; kb += 16) {
                    uint32_t b0, b1;  // rows kb .. kb + 15 of this warp's 8 columns
                    ldsm_x2_trans(tile_base + swz<SH::ROWBYTES>(kb + (lane & 15), chunk), b0, b1);
#pragma unroll
                    for (int part = 0; part < 3; ++part) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_trans(gb16 + part * SH::G16_ARRAY + kb * 32, a0, a1, a2, a3);
                        mma_16816_f16(acc[part], a0, a1, a2, a3, b0, b1);
                    }
                }
                const int m = lane >> 2, c = (lane & 3) * 2;
                float* r0 = res + m * BV + chunk * VEC + c;
                float* r8 = res + (m + 8) * BV + chunk * VEC + c;
                constexpr float S1 = 1.f / 2048.f, S2 = 1.f / (2048.f * 2048.f);
                r0[0] = fmaf(acc[2][0], S2, fmaf(acc[1][0], S1, acc[0][0]));
                r0[1] = fmaf(acc[2][1], S2, fmaf(acc[1][1], S1, acc[0][1]));
                r8[0] = fmaf(acc[2][2], S2, fmaf(acc[1][2], S1, acc[0][2]));
                r8[1] = fmaf(acc[2][3], S2, fmaf(acc[1][3], S1, acc[0][3]));
            }
        }
        // Otherwise on the CUDA cores from the fp32 carry, G tokens (32 values
        // per lane) at a time; the groups run as a loop (fewer instructions to
        // fetch)
        const bool fma_cs = !(SH::MMA_CS && t0 == 0 && !rst && KK == KMAX);
#pragma unroll 1
        for (int g0 = 0; fma_cs && g0 < TC; g0 += G) {
            if (g0 < tc) {
                float2 acc2[G * VEC];  // token jj: pairs jj VEC .. (c k), jj VEC + VP .. (c q)
#pragma unroll
                for (int i = 0; i < G * VEC; ++i) acc2[i] = make_float2(0.f, 0.f);
#pragma unroll
                for (int jj = 0; jj < G; ++jj) {
                    if (g0 + jj < tc) {
                        const uint32_t gb = gate_base + (g0 + jj) * SH::G_TOK;
#pragma unroll
                        for (int rr = 0; rr < ROWS; ++rr) {
                            const int row = lane + 32 * rr;
                            if (row < KK) {
                                const uint4 gq = lds128(gb + row * 16);
                                const float w = __uint_as_float(gq.x), z = __uint_as_float(gq.y);
                                const float2 w2 = make_float2(w, w), z2 = make_float2(z, z);
#pragma unroll
                                for (int c = 0; c < VP; ++c) {
                                    acc2[jj * VEC + c] = __ffma2_rn(x[rr][c], w2, acc2[jj * VEC + c]);
                                    acc2[jj * VEC + VP + c] = __ffma2_rn(x[rr][c], z2, acc2[jj * VEC + VP + c]);
                                }
                            }
                        }
                    }
                }
                float acc[2 * G * VEC];
#pragma unroll
                for (int i = 0; i < G * VEC; ++i) {
                    acc[2 * i] = acc2[i].x;
                    acc[2 * i + 1] = acc2[i].y;
                }
                const float sum = warp_reduce_scatter<2 * G * VEC>(acc, lane);  // entry `lane`
                const int jj = lane / (2 * VEC), kind = (lane / VEC) & 1, c = lane % VEC;
                res[((g0 + jj) * 2 + kind) * BV + chunk * VEC + c] = sum;
            }
        }
        __syncthreads();

        // (4) per column (lane j): forward substitution for d, and the
        // outputs.  Warp w keeps tokens TPW w .. TPW w + TPW - 1: it solves
        // up to its last token and writes only its own tokens' outputs and d,
        // so no warp carries all the outputs and stores.  d is kept scaled by
        // beta_t / |k_t| for the snapshots, which add raw k_t times it; the
        // columns past V get d = 0.
        {
            constexpr int TPW = TC / NW;
            const int j = lane, tlo = warp * TPW, thi = tlo + TPW;
            const bool col_ok = j < vcols;
            float d[TC];
#pragma unroll
            for (int t = 0; t < TC; ++t) {
                d[t] = 0.f;
                if (t < tc && t < thi) {
                    const float4 sc = scal[t];
                    if (col_ok) {
                        const float* g = reinterpret_cast<const float*>(gts + t * SH::G_TOK + SH::G_V);
                        float u = sc.y * res[(t * 2 + 0) * BV + j];
#pragma unroll
                        for (int s = 0; s < t; ++s) u = fmaf(ab[idx_a(t, s)], d[s], u);
                        d[t] = g[j] - u;  // d_t = v_t - (D_t S_(t-1))^T khat_t
                        if (t >= tlo) {
                            float o = sc.z * res[(t * 2 + 1) * BV + j];
#pragma unroll
                            for (int s = 0; s <= t; ++s) o = fmaf(ab[idx_b(t, s)], d[s], o);
                            p.o[(((int64_t)tb + t0 + t) * p.hv + h) * p.v + cb * BV + j] = o * p.inv_sqrt_k;
                        }
                    }
                    if (t >= tlo) dsm[t * BV + j] = d[t] * (sc.x * sc.y);
                }
            }
        }
        __syncthreads();

        // (5) the snapshots: S_t = alpha_t S_(t-1) + (beta_t khat_t) d_t^T,
        // staged rounded in a swizzled tile, then stored.  Prefill keeps
        // only the carry: the same update, nothing staged or stored.
        for (int j = 0; final_mode && j < tc; ++j) {
            float2 d[VP];
#pragma unroll
            for (int c = 0; c < VP; c += 2) {
                const float4 d4 = *reinterpret_cast<const float4*>(dsm + j * BV + chunk * VEC + 2 * c);
                d[c] = make_float2(d4.x, d4.y);
                d[c + 1] = make_float2(d4.z, d4.w);
            }
            const uint32_t gb = gate_base + j * SH::G_TOK;
#pragma unroll
            for (int rr = 0; rr < ROWS; ++rr) {
                const int row = lane + 32 * rr;
                if (row < KK) {
                    const uint4 gq = lds128(gb + row * 16);
                    const float2 al2 = make_float2(__uint_as_float(gq.z), __uint_as_float(gq.z));
                    const float2 bk2 = make_float2(__uint_as_float(gq.w), __uint_as_float(gq.w));
#pragma unroll
                    for (int c = 0; c < VP; ++c) x[rr][c] = __ffma2_rn(al2, x[rr][c], __fmul2_rn(bk2, d[c]));
                }
            }
        }
        for (int j = 0; !final_mode && j < tc; ++j) {
            float2 d[VP];
#pragma unroll
            for (int c = 0; c < VP; c += 2) {
                const float4 d4 = *reinterpret_cast<const float4*>(dsm + j * BV + chunk * VEC + 2 * c);
                d[c] = make_float2(d4.x, d4.y);
                d[c + 1] = make_float2(d4.z, d4.w);
            }
            const uint32_t gb = gate_base + j * SH::G_TOK;
            const int b = (t0 + j) % SH::NSTAGE;
            const uint32_t stage = tile_base + b * SH::TILE_BYTES;
#pragma unroll
            for (int rr = 0; rr < ROWS; ++rr) {
                const int row = lane + 32 * rr;
                if (row < KK) {
                    const uint4 gq = lds128(gb + row * 16);
                    const float2 al2 = make_float2(__uint_as_float(gq.z), __uint_as_float(gq.z));
                    const float2 bk2 = make_float2(__uint_as_float(gq.w), __uint_as_float(gq.w));
#pragma unroll
                    for (int c = 0; c < VP; ++c) x[rr][c] = __ffma2_rn(al2, x[rr][c], __fmul2_rn(bk2, d[c]));
                    sts128(stage + swz<SH::ROWBYTES>(row, chunk), SV::narrow2(x[rr]));
                }
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0 && snaps[j] >= 0) {  // a negative slot: this snapshot is not kept
                tma_store_3d(&tmap, smem + b * SH::TILE_BYTES, cb * BV, h * KK, snaps[j]);
                bulk_commit();
                // the store of token t - 1 may still read its buffer; the one
                // token t + 1 rewrites is free
                bulk_wait_read<SH::NSTAGE - 2>();
            }
        }
        // the next chunk rewrites the gates, d and the token scalars
        __syncthreads();
    }
    // CONV: the q/k windows' update, all threads together (the value
    // columns' were rewritten after the prologue).  A q/k channel's window is
    // read by every CTA of the request's value heads sharing the q/k head, and
    // the one whose count completes it writes the new entries and puts the
    // count back to zero.  No CTA waits for another.  conv_prev < 0: not
    // counted yet (a wait that ran out before the count).
    if constexpr (CONV) {
        const auto& cp = p.conv;
        const int m = col + cp.KW - 1, readers = (p.hv / p.hqk) * vt;
        QT* W = static_cast<QT*>(cp.window) + (int64_t)cslot * cp.slot_stride;
        const QT* X = static_cast<const QT*>(cp.x) + (int64_t)tb * cp.C;
        bool last = true;
        if (readers > 1) {
            int* flag = snaps + TC - 1;  // the last token's snapshot id is no longer needed
            __syncthreads();
            if (tid == 0) {
                int* cnt = cp.counters + (int64_t)n * p.hqk + hq;
                const bool done = (conv_prev >= 0 ? conv_prev : atomicAdd(cnt, 1)) == readers - 1;
                if (done) atomicExch(cnt, 0);
                *flag = done ? 1 : 0;
            }
            __syncthreads();
            last = *flag != 0;
        }
        if (last && rowt < KK && half == 0)
            sconv_window_store2(W, X, hq * KK + rowt, (p.hqk + hq) * KK + rowt, cp.C, cp.L, m, Tn, rst);
    }
    // prefill: the state after the last token, staged rounded in buffer 0 (free:
    // no snapshot store used it) and stored as one box
    if (final_mode && alive && state_in && fin >= 0) {
#pragma unroll
        for (int rr = 0; rr < ROWS; ++rr) {
            const int row = lane + 32 * rr;
            if (row < KK) sts128(tile_base + swz<SH::ROWBYTES>(row, chunk), SV::narrow2(x[rr]));
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&tmap, smem, cb * BV, h * KK, fin);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait<0>();  // the stores are complete
    if (!alive) {
        if (tid == 0) {
            atomicExch(p.status, STATUS_TIMEOUT);
            if (!rst) mbar_wait(bar_st, 0);  // bounded: no copy may still target this CTA's memory
        }
    }
}
#undef KK

}  // namespace kda
