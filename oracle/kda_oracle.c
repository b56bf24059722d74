/*
 * KDA recurrent-state oracle: TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of the Kimi Delta Attention (KDA) gated
 * delta-rule recurrent-state update at decode and speculative-verify time.
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this file's library; the product path never does, and this file
 * shares no code, header or table with the CUDA library.
 *
 * Sources (three ROCm/ATOM pull-request pages; cited by number and section):
 *  - ATOM pull request 2945 (the mono decode kernel K1 takes an fp16 state
 *    pool), Summary and Changes: a loaded state is widened to fp32, the
 *    recurrence runs in fp32, a stored state is rounded to fp16 to nearest
 *    even; one address function state_at(c, slot) serves the initial state
 *    and each token's snapshot slot.  Limitations: the norm bound -- with a
 *    unit-norm k, 0 < beta < 1 and alpha <= 1, one token can grow the squared
 *    norm of state column j by no more than v_j^2.
 *  - ATOM pull request 2130, "perf(kimi-k3): make the KDA temporal state dtype
 *    configurable", What: the state of one layer and slot is [HV=12, K=128,
 *    V=128]; q and k are L2-normalised inside the kernel; the kernel is a
 *    fused sigmoid-gating delta-rule update.
 *  - The order of operations (decay, then u = S^T k, then the delta update,
 *    then o = S^T q / sqrt(K)) and the gate form g = -softplus(a), alpha =
 *    exp(g), beta = sigmoid(b) are the plainest reading of the method's
 *    statement; the pages never print the recurrence as an equation.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes): L2 norm x / sqrt(sum x^2 + 1e-6); softplus written in
 * its overflow-free form; the fp64 carry across speculative tokens is never
 * rounded, only each stored snapshot is; an fp32 pool is stored with the
 * ordinary fp64 -> fp32 conversion (round to nearest even).
 *
 * Everything here is fp64.  The one rounding it performs is the store into the
 * pool's own element type.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_L2_EPS 1e-6

enum { ORACLE_F32 = 0, ORACLE_F16 = 1 };

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16, written from the format's definition:                  */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormal        */
/* quantum 2^-24; largest finite value 65504.                                */
/* ------------------------------------------------------------------------ */

double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0x1f) {
        mag = frac ? NAN : INFINITY;
    } else if (expo == 0) {
        mag = ldexp((double)frac, -24);                 /* subnormal or zero */
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25);  /* (1 + f/1024) 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* Round an fp64 value to binary16, to nearest, ties to even.  The quantum of
 * the binade |x| falls in is a power of two, so |x| / quantum is exact, and
 * rint() (the default rounding mode is nearest-even) does the one rounding. */
uint16_t oracle_f64_to_f16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    /* Halfway between 65504 and 65536 (the first value past the format)
     * ties to 65536, whose significand is even: that, and above, is inf. */
    if (ax >= 65520.0) return (uint16_t)(sign | 0x7c00);

    double quantum;
    if (ax < ldexp(1.0, -14)) {
        quantum = ldexp(1.0, -24);
    } else {
        int e2;
        frexp(ax, &e2);                     /* ax = f 2^e2, f in [0.5, 1) */
        quantum = ldexp(1.0, (e2 - 1) - 10);
    }
    double r = rint(ax / quantum) * quantum;  /* the rounded magnitude, exact */

    if (r < ldexp(1.0, -14)) {
        /* subnormal (or zero): the integer count of 2^-24 quanta */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
    }
    int e2;
    frexp(r, &e2);
    int E = e2 - 1;                                   /* r in [2^E, 2^(E+1)) */
    uint16_t frac = (uint16_t)(r / ldexp(1.0, E - 10) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | frac);
}

void oracle_f64_to_f16_rne_array(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_f16_rne(x[i]);
}

void oracle_f16_to_f64_array(const uint16_t* h, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f64(h[i]);
}

/* ------------------------------------------------------------------------ */
/* The pool and its one address function                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    void* base;           /* element 0 of slot 0 */
    int dtype;            /* ORACLE_F32 or ORACLE_F16 */
    int64_t num_slots;
    int hv, k, v;
    int64_t slot_stride;  /* elements from one slot to the next */
} oracle_pool;

/* state_at(slot, head): element offset of S[0][0] of one head's [K][V] state
 * (ATOM PR 2945, Changes: one address function for every state access). */
static int64_t state_at(const oracle_pool* p, int64_t slot, int h)
{
    return slot * p->slot_stride + (int64_t)h * p->k * p->v;
}

static void load_state(const oracle_pool* p, int64_t slot, int h, double* S)
{
    int64_t off = state_at(p, slot, h);
    int64_t kv = (int64_t)p->k * p->v;
    if (p->dtype == ORACLE_F32) {
        const float* src = (const float*)p->base + off;
        for (int64_t e = 0; e < kv; ++e) S[e] = (double)src[e];
    } else {
        const uint16_t* src = (const uint16_t*)p->base + off;
        for (int64_t e = 0; e < kv; ++e) S[e] = oracle_f16_to_f64(src[e]);
    }
}

static void store_state(const oracle_pool* p, int64_t slot, int h, const double* S)
{
    int64_t off = state_at(p, slot, h);
    int64_t kv = (int64_t)p->k * p->v;
    if (p->dtype == ORACLE_F32) {
        float* dst = (float*)p->base + off;
        for (int64_t e = 0; e < kv; ++e) dst[e] = (float)S[e];
    } else {
        uint16_t* dst = (uint16_t*)p->base + off;
        for (int64_t e = 0; e < kv; ++e) dst[e] = oracle_f64_to_f16_rne(S[e]);
    }
}

/* ------------------------------------------------------------------------ */
/* One token of the recurrence on one head's fp64 state S[K][V]              */
/* ------------------------------------------------------------------------ */

static double softplus(double a)
{
    /* log(1 + e^a), in the form that never overflows */
    return a > 0 ? a + log1p(exp(-a)) : log1p(exp(a));
}

/*
 * q, k, a: [K]; v: [V]; b: scalar; o: [V] (out).  Work arrays qh, kh, u: [K or V].
 *   khat = k / sqrt(sum k^2 + eps), qhat likewise        (L2 norm, in-kernel)
 *   beta = sigmoid(b); alpha_i = exp(-softplus(a_i))      (fused gating)
 *   S <- diag(alpha) S                                    (per-key-channel decay)
 *   u  = S^T khat                                         (what S recalls for k)
 *   S <- S + beta khat (v - u)^T                          (delta update)
 *   o  = S^T qhat / sqrt(K)                               (read-out, updated S)
 */
static void recur_token_gated(int K, int V, double* S,
                              const double* q, const double* k, const double* v,
                              const double* a, double b, double scale, const double* bias,
                              double* o, double* qh, double* kh, double* u);

static void recur_token(int K, int V, double* S,
                        const double* q, const double* k, const double* v,
                        const double* a, double b, double* o,
                        double* qh, double* kh, double* u)
{
    recur_token_gated(K, V, S, q, k, v, a, b, 1.0, NULL, o, qh, kh, u);
}

/*
 * The same token with the learned gate scale of the KDA layer:
 *   alpha_i = exp(-scale * softplus(a_i + bias_i)),  scale = exp(A_log) of the head.
 * scale = 1 and bias = NULL is the plain gate exp(-softplus(a_i)) above, to the bit.
 */
static void recur_token_gated(int K, int V, double* S,
                              const double* q, const double* k, const double* v,
                              const double* a, double b, double scale, const double* bias,
                              double* o, double* qh, double* kh, double* u)
{
    double qq = 0.0, kk = 0.0;
    for (int i = 0; i < K; ++i) { qq += q[i] * q[i]; kk += k[i] * k[i]; }
    double qn = sqrt(qq + ORACLE_L2_EPS), kn = sqrt(kk + ORACLE_L2_EPS);
    for (int i = 0; i < K; ++i) { qh[i] = q[i] / qn; kh[i] = k[i] / kn; }

    double beta = 1.0 / (1.0 + exp(-b));

    for (int i = 0; i < K; ++i) {
        double alpha = exp(-(scale * softplus(bias ? a[i] + bias[i] : a[i])));
        for (int j = 0; j < V; ++j) S[(int64_t)i * V + j] *= alpha;
    }
    for (int j = 0; j < V; ++j) {
        double s = 0.0;
        for (int i = 0; i < K; ++i) s += S[(int64_t)i * V + j] * kh[i];
        u[j] = s;
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            S[(int64_t)i * V + j] += beta * kh[i] * (v[j] - u[j]);
    double inv_sqrt_k = 1.0 / sqrt((double)K);
    for (int j = 0; j < V; ++j) {
        double s = 0.0;
        for (int i = 0; i < K; ++i) s += S[(int64_t)i * V + j] * qh[i];
        o[j] = s * inv_sqrt_k;
    }
}

/*
 * The whole step for requests n = 0..N-1, heads h = 0..HV-1, tokens t = 0..T-1.
 * Inputs are fp64, already widened exactly from whatever type the caller used:
 *   q, k, a: [N][T][HV][K];  v: [N][T][HV][V];  b: [N][T][HV];  o: [N][T][HV][V].
 * init_slot[n]: the slot the request's state is read from (unless reset[n]).
 * snap_slot == NULL (decode, T must be 1): the state is written back in place
 *   to init_slot[n].
 * snap_slot != NULL ([N][T], speculative verify): the state after token t is
 *   written to snap_slot[n*T + t]; init_slot[n] is not written.
 * reset (may be NULL): reset[n] != 0 starts request n from a zero state.
 * Returns 0, or -1 when a slot id lies outside [0, num_slots).
 */
static int run(const oracle_pool* p, int n_req, int T,
               const int32_t* init_slot, const int32_t* snap_slot, const uint8_t* reset,
               const double* q, const double* k, const double* v,
               const double* a, const double* b, double* o, int nthreads)
{
    const int HV = p->hv, K = p->k, V = p->v;
    for (int n = 0; n < n_req; ++n) {
        if (init_slot[n] < 0 || init_slot[n] >= p->num_slots) return -1;
        if (snap_slot)
            for (int t = 0; t < T; ++t)
                if (snap_slot[(int64_t)n * T + t] < 0 ||
                    snap_slot[(int64_t)n * T + t] >= p->num_slots) return -1;
    }
    int64_t pairs = (int64_t)n_req * HV;
    int bad = 0;
#if defined(_OPENMP)
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) if (nthreads > 1)
#endif
    for (int64_t nh = 0; nh < pairs; ++nh) {
        int n = (int)(nh / HV), h = (int)(nh % HV);
        double* S = (double*)malloc(sizeof(double) * ((size_t)K * V + 2 * (size_t)K + (size_t)V));
        if (!S) { bad = 1; continue; }
        double* qh = S + (int64_t)K * V;
        double* kh = qh + K;
        double* u = kh + K;
        if (reset && reset[n]) memset(S, 0, sizeof(double) * (size_t)K * V);
        else load_state(p, init_slot[n], h, S);
        for (int t = 0; t < T; ++t) {
            int64_t row = ((int64_t)n * T + t) * HV + h;
            recur_token(K, V, S, q + row * K, k + row * K, v + row * V,
                        a + row * K, b[row], o + row * V, qh, kh, u);
            if (snap_slot) store_state(p, snap_slot[(int64_t)n * T + t], h, S);
        }
        if (!snap_slot) store_state(p, init_slot[n], h, S);
        free(S);
    }
    (void)nthreads;
    return bad ? -2 : 0;
}

int oracle_decode_step(void* base, int dtype, int64_t num_slots, int hv, int k, int v,
                       int64_t slot_stride, int n_req, const int32_t* slot_ids,
                       const uint8_t* reset, const double* q, const double* kk,
                       const double* vv, const double* a, const double* b, double* o,
                       int nthreads)
{
    oracle_pool p = {base, dtype, num_slots, hv, k, v, slot_stride};
    return run(&p, n_req, 1, slot_ids, NULL, reset, q, kk, vv, a, b, o, nthreads);
}

int oracle_spec_verify(void* base, int dtype, int64_t num_slots, int hv, int k, int v,
                       int64_t slot_stride, int n_req, int T, const int32_t* init_slot,
                       const int32_t* snap_slot, const uint8_t* reset, const double* q,
                       const double* kk, const double* vv, const double* a, const double* b,
                       double* o, int nthreads)
{
    oracle_pool p = {base, dtype, num_slots, hv, k, v, slot_stride};
    return run(&p, n_req, T, init_slot, snap_slot, reset, q, kk, vv, a, b, o, nthreads);
}

/*
 * The general step: accepted-length speculative decode over packed,
 * variable-length requests (the address function state_at(c, slot) of ATOM
 * pull request 2945, Changes, serving a request's initial state and each of
 * its tokens' snapshot slots; the number of tokens a step keeps varies with
 * the drafts accepted, ATOM pull request 2945, Performance).
 *
 *   tokens are packed: request r owns tokens cu[r] .. cu[r+1]-1 (T_r of them);
 *     cu == NULL means T_r = t_uniform and request r owns r*t_uniform ..
 *   q, k: [total][H][K] (value head h reads q/k head h / (HV / H));
 *   v: [total][HV][V];  a: [total][HV][K];  b: [total][HV];  o: [total][HV][V]
 *   slot_table[r][c], c < num_cols: the request's slots, column c = token c
 *   initial column c0 = accepted ? accepted[r] - 1 : 0, which must lie in
 *     [0, num_cols); the initial slot is slot_table[r][c0]
 *   a negative initial slot marks a padding request: nothing is read or
 *     stored and its output rows are zero
 *   in_place (decode): T_r must be 1 and the state goes back to the initial
 *     slot; otherwise the state after token j goes to slot_table[r][j], and a
 *     negative entry there means that snapshot is not kept
 *   reset[r] != 0 starts request r from a zero state
 *   a_log ([HV]) and dt_bias ([HV][K]) may be NULL: scale 1, bias 0
 * Returns 0; -1 for a slot id >= num_slots; -3 for an inconsistent layout
 * (initial column outside the table, T_r > num_cols, T_r != 1 in place,
 * H not dividing HV, cu not non-decreasing).
 */
int oracle_step(void* base, int dtype, int64_t num_slots, int hv, int k, int v,
                int64_t slot_stride, int n_req, int h_qk, const int32_t* cu, int t_uniform,
                const int32_t* slot_table, int num_cols, const int32_t* accepted, int in_place,
                const uint8_t* reset, const double* q, const double* kk, const double* vv,
                const double* a, const double* b, const double* a_log, const double* dt_bias,
                double* o, int nthreads)
{
    oracle_pool p = {base, dtype, num_slots, hv, k, v, slot_stride};
    const int HV = hv, K = k, V = v;
    if (h_qk <= 0 || HV % h_qk != 0) return -3;
    const int group = HV / h_qk;
    for (int r = 0; r < n_req; ++r) {
        int64_t t0 = cu ? cu[r] : (int64_t)r * t_uniform;
        int64_t tr = cu ? (int64_t)cu[r + 1] - cu[r] : t_uniform;
        if (tr < 0 || tr > num_cols || (in_place && tr != 1) || t0 < 0) return -3;
        int c0 = accepted ? accepted[r] - 1 : 0;
        if (c0 < 0 || c0 >= num_cols) return -3;
        const int32_t* row = slot_table + (int64_t)r * num_cols;
        if (row[c0] >= num_slots) return -1;
        if (row[c0] < 0) continue;
        if (!in_place)
            for (int64_t j = 0; j < tr; ++j)
                if (row[j] >= num_slots) return -1;
    }
    int64_t pairs = (int64_t)n_req * HV;
    int bad = 0;
#if defined(_OPENMP)
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) if (nthreads > 1)
#endif
    for (int64_t nh = 0; nh < pairs; ++nh) {
        int r = (int)(nh / HV), h = (int)(nh % HV);
        int64_t t0 = cu ? cu[r] : (int64_t)r * t_uniform;
        int64_t tr = cu ? (int64_t)cu[r + 1] - cu[r] : t_uniform;
        const int32_t* row = slot_table + (int64_t)r * num_cols;
        int32_t s0 = row[accepted ? accepted[r] - 1 : 0];
        if (s0 < 0) {  /* padding request */
            for (int64_t j = 0; j < tr; ++j)
                memset(o + ((t0 + j) * HV + h) * V, 0, sizeof(double) * (size_t)V);
            continue;
        }
        double* S = (double*)malloc(sizeof(double) * ((size_t)K * V + 2 * (size_t)K + (size_t)V));
        if (!S) { bad = 1; continue; }
        double* qh = S + (int64_t)K * V;
        double* kh = qh + K;
        double* u = kh + K;
        if (reset && reset[r]) memset(S, 0, sizeof(double) * (size_t)K * V);
        else load_state(&p, s0, h, S);
        double scale = a_log ? exp(a_log[h]) : 1.0;
        const double* bias = dt_bias ? dt_bias + (int64_t)h * K : NULL;
        int hq = h / group;
        for (int64_t j = 0; j < tr; ++j) {
            int64_t tok = t0 + j;
            int64_t vrow = tok * HV + h, qrow = tok * h_qk + hq;
            recur_token_gated(K, V, S, q + qrow * K, kk + qrow * K, vv + vrow * V, a + vrow * K,
                              b[vrow], scale, bias, o + vrow * V, qh, kh, u);
            if (!in_place && row[j] >= 0) store_state(&p, row[j], h, S);
        }
        if (in_place) store_state(&p, s0, h, S);
        free(S);
    }
    (void)nthreads;
    return bad ? -2 : 0;
}

/* ------------------------------------------------------------------------ */
/* bfloat16 (1 sign, 8 exponent bits with bias 127, 7 fraction bits): the    */
/* fp32 exponent range with a 7-bit fraction.                                 */
/* ------------------------------------------------------------------------ */

double oracle_bf16_to_f64(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);  /* the bf16 value is the fp32 value with these top bits */
    return (double)f;
}

/* fp64 -> bf16, to nearest, ties to even, in one rounding: the quantum of the
 * binade is 2^(e - 7); below 2^-126 the quantum is the subnormal one, 2^-133. */
uint16_t oracle_f64_to_bf16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7fc0);
    /* the largest finite bf16 is (2 - 2^-7) 2^127; halfway to 2^128 rounds up */
    if (ax >= ldexp(2.0 - ldexp(1.0, -8), 127)) return (uint16_t)(sign | 0x7f80);
    double quantum;
    if (ax < ldexp(1.0, -126)) {
        quantum = ldexp(1.0, -133);
    } else {
        int e2;
        frexp(ax, &e2);
        quantum = ldexp(1.0, (e2 - 1) - 7);
    }
    double r = rint(ax / quantum) * quantum;
    float f = (float)r;  /* exact: r has at most 8 significant bits inside the fp32 range */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

void oracle_f64_to_bf16_rne_array(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16_rne(x[i]);
}

/*
 * The causal short convolution in front of the recurrence, with its paged
 * window (ATOM pull request 2894, review thread: the conv pool keeps the last
 * kernel - 1 + num_spec inputs of a request; a step reads its kernel - 1
 * history entries starting at the accepted index acc_idx, and writes back the
 * kept old entries followed by the step's inputs).
 *
 * Window of slot s: W[s][e][c], e = 0 .. L-1 oldest first, c < C channels
 * (channel innermost).  Request r: tokens cu[r] .. cu[r+1]-1 (or r*t_uniform ..),
 * window slot conv_slot[r] (negative: padding, nothing read or stored, output
 * rows zero), acc = accepted ? accepted[r] - 1 : 0.
 *   history h_i = W[acc + i], i < KW - 1 (zero when reset[r]);
 *   z = h ++ x;  y_t[c] = act(bias[c] + sum_{i<KW} w[c][i] z[t + i])
 *   (w[c][KW-1] weighs the newest input; act = SiLU x sigmoid(x), or none);
 *   with m = acc + KW - 1 valid entries and kept = max(0, L - T) old ones,
 *   the new window is W[m - kept .. m - 1] (zero when reset) followed by the
 *   last min(T, L) inputs.  T = 0 leaves the window alone.
 * x, y and the window share dtype (0 fp32, 1 fp16, 2 bf16); y is rounded to it.
 * Returns 0; -1 slot >= num_slots; -3 layout (m > L, m < kept, acc < 0).
 */
static double conv_load(int dtype, const void* p, int64_t i)
{
    if (dtype == 0) return (double)((const float*)p)[i];
    uint16_t h = ((const uint16_t*)p)[i];
    return dtype == 1 ? oracle_f16_to_f64(h) : oracle_bf16_to_f64(h);
}

static void conv_store(int dtype, void* p, int64_t i, double v)
{
    if (dtype == 0) ((float*)p)[i] = (float)v;
    else ((uint16_t*)p)[i] = dtype == 1 ? oracle_f64_to_f16_rne(v) : oracle_f64_to_bf16_rne(v);
}

int oracle_conv_step(void* wbase, int dtype, int64_t num_slots, int C, int L, int64_t slot_stride,
                     int n_req, const int32_t* cu, int t_uniform, const int32_t* conv_slot,
                     const int32_t* accepted, const uint8_t* reset, int KW, int silu,
                     const void* x, const double* w, const double* bias, void* y)
{
    for (int r = 0; r < n_req; ++r) {
        int64_t T = cu ? (int64_t)cu[r + 1] - cu[r] : t_uniform;
        int acc = accepted ? accepted[r] - 1 : 0;
        if (conv_slot[r] >= num_slots) return -1;
        if (conv_slot[r] < 0 || T == 0) continue;
        int m = acc + KW - 1;
        int64_t kept = L - T > 0 ? L - T : 0;
        if (acc < 0 || m > L || m < kept || T < 0) return -3;
    }
    double* old = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double* z = (double*)malloc(sizeof(double) * (size_t)(KW + 1));
    if (!old || !z) { free(old); free(z); return -2; }
    for (int r = 0; r < n_req; ++r) {
        int64_t t0 = cu ? cu[r] : (int64_t)r * t_uniform;
        int64_t T = cu ? (int64_t)cu[r + 1] - cu[r] : t_uniform;
        int32_t s = conv_slot[r];
        if (s < 0) {
            for (int64_t t = 0; t < T; ++t)
                for (int c = 0; c < C; ++c) conv_store(dtype, y, (t0 + t) * C + c, 0.0);
            continue;
        }
        if (T == 0) continue;
        int acc = accepted ? accepted[r] - 1 : 0;
        int m = acc + KW - 1;
        int64_t kept = L - T > 0 ? L - T : 0;
        int rst = reset && reset[r];
        int64_t wofs = (int64_t)s * slot_stride;
        for (int c = 0; c < C; ++c) {
            /* history and kept entries, read before anything is written */
            for (int i = 0; i < KW - 1; ++i)
                z[i] = rst ? 0.0 : conv_load(dtype, wbase, wofs + (int64_t)(acc + i) * C + c);
            for (int64_t e = 0; e < kept; ++e)
                old[e] = rst ? 0.0 : conv_load(dtype, wbase, wofs + (m - kept + e) * C + c);
            for (int64_t t = 0; t < T; ++t) {
                z[KW - 1] = conv_load(dtype, x, (t0 + t) * C + c);
                double s_ = bias ? bias[c] : 0.0;
                for (int i = 0; i < KW; ++i) s_ += w[(int64_t)c * KW + i] * z[i];
                double out = silu ? s_ / (1.0 + exp(-s_)) : s_;
                conv_store(dtype, y, (t0 + t) * C + c, out);
                for (int i = 0; i < KW - 1; ++i) z[i] = z[i + 1];
            }
            for (int64_t e = 0; e < kept; ++e)
                conv_store(dtype, wbase, wofs + e * C + c, old[e]);
            int64_t nin = T < L ? T : L;
            for (int64_t e = 0; e < nin; ++e)
                conv_store(dtype, wbase, wofs + (kept + e) * C + c,
                           conv_load(dtype, x, (t0 + T - nin + e) * C + c));
        }
    }
    free(old);
    free(z);
    return 0;
}

/*
 * Checkpoint flush and load through the address function (ATOM pull request
 * 2945, Changes: under ReplaySSM the checkpoint load and the flush go through
 * state_at; pull request 2130, What: the checkpoint plane shapes and layout id
 * derive from the state dtype).  A plane holds entries of one slot's state
 * ([HV][K][V], the pool's element type).  flush: plane[entry[i]] <- pool[slot[i]];
 * load: pool[slot[i]] <- plane[entry[i]].  A negative slot or entry skips i.
 * Element copies only: nothing is converted.  Returns 0, or -1 for an index
 * past its buffer.
 */
int oracle_ckpt_transfer(void* pool_base, int64_t num_slots, int64_t slot_stride,
                         void* plane_base, int64_t num_entries, int64_t entry_stride,
                         int64_t state_elems, int elem_bytes, int n, const int32_t* slot,
                         const int32_t* entry, int load)
{
    for (int i = 0; i < n; ++i) {
        if (slot[i] >= num_slots || entry[i] >= num_entries) return -1;
    }
    for (int i = 0; i < n; ++i) {
        if (slot[i] < 0 || entry[i] < 0) continue;
        char* p = (char*)pool_base + (int64_t)slot[i] * slot_stride * elem_bytes;
        char* c = (char*)plane_base + (int64_t)entry[i] * entry_stride * elem_bytes;
        if (load) memcpy(p, c, (size_t)(state_elems * elem_bytes));
        else memcpy(c, p, (size_t)(state_elems * elem_bytes));
    }
    return 0;
}

/*
 * Prefill: the same recurrence over each request's prompt (the second
 * workload of ATOM pull request 2130, What: prefill reads and writes the state
 * through the destination's element type like every other path).  Request r
 * owns tokens cu[r] .. cu[r+1]-1 (or r*t_uniform ..); its state starts from
 * init_slot[r] (zero when reset[r]; a negative init_slot is a padding request:
 * nothing read or stored, outputs zero) and only the state after its last
 * token is stored, to final_slot[r] (negative: not stored; may equal
 * init_slot[r]).  A request with no tokens stores its initial state (zero
 * when reset[r]) to final_slot[r]: the state after its last token is the state
 * it started from, so splitting a prompt into an empty part and the rest
 * changes nothing.
 * Heads, gate and layouts as in oracle_step.  Returns 0, -1 slot out of range,
 * -3 layout.
 */
int oracle_prefill(void* base, int dtype, int64_t num_slots, int hv, int k, int v,
                   int64_t slot_stride, int n_req, int h_qk, const int32_t* cu, int t_uniform,
                   const int32_t* init_slot, const int32_t* final_slot, const uint8_t* reset,
                   const double* q, const double* kk, const double* vv, const double* a,
                   const double* b, const double* a_log, const double* dt_bias, double* o,
                   int nthreads)
{
    oracle_pool p = {base, dtype, num_slots, hv, k, v, slot_stride};
    const int HV = hv, K = k, V = v;
    if (h_qk <= 0 || HV % h_qk != 0) return -3;
    const int group = HV / h_qk;
    for (int r = 0; r < n_req; ++r) {
        int64_t tr = cu ? (int64_t)cu[r + 1] - cu[r] : t_uniform;
        if (tr < 0) return -3;
        if (init_slot[r] >= num_slots || final_slot[r] >= num_slots) return -1;
    }
    int64_t pairs = (int64_t)n_req * HV;
    int bad = 0;
#if defined(_OPENMP)
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) if (nthreads > 1)
#endif
    for (int64_t nh = 0; nh < pairs; ++nh) {
        int r = (int)(nh / HV), h = (int)(nh % HV);
        int64_t t0 = cu ? cu[r] : (int64_t)r * t_uniform;
        int64_t tr = cu ? (int64_t)cu[r + 1] - cu[r] : t_uniform;
        if (init_slot[r] < 0) {  /* padding request */
            for (int64_t j = 0; j < tr; ++j)
                memset(o + ((t0 + j) * HV + h) * V, 0, sizeof(double) * (size_t)V);
            continue;
        }
        double* S = (double*)malloc(sizeof(double) * ((size_t)K * V + 2 * (size_t)K + (size_t)V));
        if (!S) { bad = 1; continue; }
        double* qh = S + (int64_t)K * V;
        double* kh = qh + K;
        double* u = kh + K;
        if (reset && reset[r]) memset(S, 0, sizeof(double) * (size_t)K * V);
        else load_state(&p, init_slot[r], h, S);
        double scale = a_log ? exp(a_log[h]) : 1.0;
        const double* bias = dt_bias ? dt_bias + (int64_t)h * K : NULL;
        int hq = h / group;
        for (int64_t j = 0; j < tr; ++j) {
            int64_t tok = t0 + j;
            int64_t vrow = tok * HV + h, qrow = tok * h_qk + hq;
            recur_token_gated(K, V, S, q + qrow * K, kk + qrow * K, vv + vrow * V, a + vrow * K,
                              b[vrow], scale, bias, o + vrow * V, qh, kh, u);
        }
        if (final_slot[r] >= 0) store_state(&p, final_slot[r], h, S);
        free(S);
    }
    (void)nthreads;
    return bad ? -2 : 0;
}
