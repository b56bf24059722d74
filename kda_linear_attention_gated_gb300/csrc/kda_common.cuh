// Shared device helpers of the KDA kernels: parameters, element conversion,
// the state address function, and the PTX wrappers for TMA (cp.async.bulk),
// mbarriers and proxy fences used by the pipelined kernels (sm_90+ PTX, valid
// on sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kda {

constexpr int KMAX = 128;        // largest K (and V) a launch accepts
constexpr float L2_EPS = 1e-6f;  // L2-norm epsilon: x / sqrt(sum x^2 + eps)
constexpr int32_t STATUS_SLOT_RANGE = 8;   // KDA_ERR_SLOT_RANGE in kda.h
constexpr int32_t STATUS_TIMEOUT = 10;     // KDA_ERR_TIMEOUT in kda.h
constexpr int32_t STATUS_SMEM_ALIGN = 6;   // KDA_ERR_ALIGN in kda.h (shared-memory base)
constexpr int32_t STATUS_ARG = 9;          // KDA_ERR_ARG in kda.h (bad accepted column or token offsets)
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // a pipeline wait gives up after 1 s

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
    uint32_t flags;           // KDA_LAUNCH_* bits
    // The general step; the values make_params sets reproduce plain decode and verify.
    int hqk;                  // q/k heads: value head h reads q/k head h / (hv / hqk)
    int init_stride;          // elements between two requests' rows of init_slot
    int snap_stride;          // ... of snap_slot
    int num_cols;             // columns of a slot-table row (bounds the accepted column)
    const int32_t* accepted;  // [n] or nullptr: request n's initial slot is column accepted[n] - 1
    const int32_t* cu;        // [n + 1] or nullptr: request n owns tokens cu[n] .. cu[n+1] - 1
                              // (else n t .. n t + t - 1); t bounds cu[n+1] - cu[n]
    const float* a_log;       // [hv] or nullptr: gate scale exp(a_log[h])
    const float* dt_bias;     // [hv][k] or nullptr: gate bias
    uint32_t mode;            // MODE_* bits
    int total;                // rows of the packed token arrays (bounds cu)
    const int32_t* final_slot; // [n] or nullptr: prefill, only the state after the last token is
                              // stored, to final_slot[n] (negative: not stored); no snapshots
    // The fused short convolution of a decode step (the conv-decode kernel only):
    // q, k and v are its outputs y, of QT, computed from x and the window.
    struct Conv {
        void* window;             // [num_slots] x [L][C] of QT, slot_stride apart
        int64_t num_slots;
        int64_t slot_stride;      // elements
        int C, L, KW;             // channels, window entries, kernel width
        int silu;
        const int32_t* slot;      // [n]: window slot of request n
        const void* x;            // [n][C] of QT
        const float* w;           // [C][KW]
        const float* bias;        // [C] or nullptr
        void* y;                  // [n][C] of QT or nullptr
        int32_t* counters;        // [n][hqk]: reads of a q/k head's window so far
    } conv;
};

// A negative initial slot marks a padding request (nothing read or stored,
// output rows zero); a negative snapshot slot marks a snapshot not kept.
// Without this bit a negative slot is out of range.
constexpr uint32_t MODE_PADDING = 1u;

__device__ __forceinline__ float softplus_f(float x) {
    return x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

// sigmoid(-x) = 1 / (1 + e^x): the fast reciprocal refined by one
// Newton-Raphson step, r <- r + r (1 - y r), which brings its error to about
// half an ulp at a fraction of the cost of the correctly rounded reciprocal.
// Past x = 88 (e^x overflows) the result is exactly 0; between 87.3 and 88
// (y > 2^126) the fast reciprocal gives 0, and the step keeps it: the true
// value there is below 1.2e-38.  x = -inf gives exactly 1; a NaN passes through.
__device__ __forceinline__ float sigmoid_neg(float x) {
    if (x > 88.f) return 0.f;
    const float y = 1.0f + expf(x);
    const float r = __fdividef(1.0f, y);
    return fmaf(r, fmaf(-y, r, 1.0f), r);
}

// The per-key-channel decay alpha_i of one row.  Plain gate: exp(-softplus(a))
// = 1 / (1 + e^a) (one exponential, no logarithm).  Learned scale (the KDA
// layer's A_log, dt_bias): exp(-exp(A_log) softplus(a + dt_bias)).
__device__ __forceinline__ float gate_alpha(float a, bool scaled, float scale, float bias) {
    return scaled ? expf(-scale * softplus_f(a + bias)) : sigmoid_neg(a);
}

constexpr uint32_t LAUNCH_PDL = 1u;               // KDA_LAUNCH_PDL in kda.h
constexpr uint32_t LAUNCH_PDL_EARLY_STATE = 2u;   // KDA_LAUNCH_PDL_EARLY_STATE in kda.h
constexpr uint32_t LAUNCH_TEST_WITHHOLD_STATE = 1u << 30;  // KDA_LAUNCH_TEST_WITHHOLD_STATE in kda.h

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// A 16-byte vector of state elements <-> fp32 registers.
template <typename ST> struct StateVec;

// Float pairs for the packed fp32 FMA of sm_100 and later (one FFMA2 does two
// fmaf with the same rounding each): widen2 / narrow2 move a 16-byte vector
// as VEC / 2 pairs of adjacent elements.
template <> struct StateVec<float> {
    static constexpr int VEC = 4;
    static __device__ __forceinline__ void widen2(const uint4& r, float2 (&x)[VEC / 2]) {
        x[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
        x[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
    }
    static __device__ __forceinline__ uint4 narrow2(const float2 (&x)[VEC / 2]) {
        return make_uint4(__float_as_uint(x[0].x), __float_as_uint(x[0].y),
                          __float_as_uint(x[1].x), __float_as_uint(x[1].y));
    }
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
    static __device__ __forceinline__ void widen2(const uint4& r, float2 (&x)[VEC / 2]) {
        x[0] = w2(r.x); x[1] = w2(r.y); x[2] = w2(r.z); x[3] = w2(r.w);
    }
    static __device__ __forceinline__ uint4 narrow2(const float2 (&x)[VEC / 2]) {
        return make_uint4(n2(x[0].x, x[0].y), n2(x[1].x, x[1].y), n2(x[2].x, x[2].y), n2(x[3].x, x[3].y));
    }
};

// state_at(slot, h): the one address function for every state access
// (ROCm/ATOM pull request 2945, Changes), in elements from the pool base.
__device__ __forceinline__ int64_t state_at(const StepParams& p, int64_t slot, int h) {
    return slot * p.slot_stride + (int64_t)h * p.k * p.v;
}

// ---------------------------------------------------------------------------
// PTX: shared-memory addresses, mbarriers, TMA, proxy fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Add `bytes` to the phase's expected transaction count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One bounded test of a phase.  With the suspend-time hint the waiting warp is
// parked by the hardware until the phase completes or about 1 ms passes, so
// waiting warps do not take issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete; false if it
// has not completed within WAIT_LIMIT_NS (the caller reports a timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
    return true;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 3-D tiled TMA load global -> shared, completing `bytes` on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 1-D bulk copy global -> shared of `bytes` (a multiple of 16; both addresses
// 16-byte aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled TMA store shared -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src,
                                             int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
        ::"l"(map), "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// All but the N most recent bulk groups have finished reading shared memory.
template <int N> __device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// All but the N most recent bulk groups have completed (writes performed).
template <int N> __device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Warp-level tensor-core pieces (PTX ISA: ldmatrix, mma.sync m16n8k16 with
// fp16 operands and fp32 accumulation).  Every address is a shared-memory
// address of a 16-byte aligned 8-element row.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}
// d += A B for a 16 x 16 fp16 A (row-major fragment) and a 16 x 8 fp16 B
// (column fragment), fp32 accumulators.
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
// d += A B for a 16 x 16 bf16 A (row-major fragment) and a 16 x 8 bf16 B
// (column fragment), fp32 accumulators.
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// x = p0 + p1 + p2 exactly, each part a bf16 value (8 significant bits): p0
// is x rounded to bf16, p1 the remainder rounded, p2 what is left (at most 8
// significant bits, so exact).  Both differences are exact in fp32.  Two
// values at a time, packed as the bf16x2 words an mma fragment takes (the
// first value in the low half).
__device__ __forceinline__ void split3_bf16x2(float x, float y, uint32_t& p0, uint32_t& p1, uint32_t& p2) {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(x, y);
    const float2 b0 = __bfloat1622float2(h0);
    const float rx = x - b0.x, ry = y - b0.y;
    const __nv_bfloat162 h1 = __floats2bfloat162_rn(rx, ry);
    const float2 b1 = __bfloat1622float2(h1);
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(rx - b1.x, ry - b1.y);
    p0 = *reinterpret_cast<const uint32_t*>(&h0);
    p1 = *reinterpret_cast<const uint32_t*>(&h1);
    p2 = *reinterpret_cast<const uint32_t*>(&h2);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr) : "memory");
    return r;
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4& r) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(r.x), "r"(r.y), "r"(r.z), "r"(r.w) : "memory");
}

// Byte offset of (row, 16-byte chunk) inside a tile that TMA wrote with the
// swizzle mode matching ROWBYTES (128 B -> SWIZZLE_128B, 64 B -> SWIZZLE_64B,
// 32 B -> SWIZZLE_32B): the chunk index is XORed with address bits 7.. of the
// row, which spreads the 8 rows a quarter-warp reads over all 32 banks.  The
// tile base must be aligned to the pattern's period (1024 B suffices).
template <int ROWBYTES>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    static_assert(ROWBYTES == 128 || ROWBYTES == 64 || ROWBYTES == 32, "row bytes");
    if constexpr (ROWBYTES == 128) return row * 128 + ((chunk ^ (row & 7)) << 4);
    else if constexpr (ROWBYTES == 64) return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
    else return row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4);
}

// Reduce NV values per lane over the 32 lanes of a warp, scattering the
// results: afterwards lane l holds the full sum of value (l >> (5 - log2 NV))
// (lanes sharing that index hold the same sum).  Each step sends the half of
// the values the lane does not keep, so the whole reduction costs
// NV/2 + NV/4 + ... + 1 shuffles plus one per remaining lane bit, instead of
// 5 NV for NV separate butterflies.
template <int NV>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NV], int lane) {
    static_assert(NV >= 1 && NV <= 32 && (NV & (NV - 1)) == 0, "power of two");
    int m = 16;
#pragma unroll
    for (int cnt = NV; cnt > 1; cnt >>= 1, m >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < cnt / 2; ++k) {
            const float send = upper ? v[k] : v[k + cnt / 2];
            const float keep = upper ? v[k + cnt / 2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    float s = v[0];
#pragma unroll
    for (; m >= 1; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    return s;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

}  // namespace kda
