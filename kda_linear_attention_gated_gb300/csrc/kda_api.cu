// C ABI of the KDA recurrent-state library (declared in include/kda.h).
//
// This translation unit is compiled once per state-pool dtype:
//   -DKDA_STATE16=0 -> libkda_h0.so (fp32 pool)
//   -DKDA_STATE16=1 -> libkda_h1.so (fp16 pool)
// following ROCm/ATOM pull request 2945 (Changes): the pool's dtype is a build
// constant, and a pool of the other dtype is refused at call time.
//
// Host side: validate every argument synchronously, pick the column tile by
// element size, and enqueue exactly one kernel on the caller's stream.
#include <cuda_runtime.h>

#include <cstdint>

#include "kda.h"
#include "kda_kernels.cuh"

#ifndef KDA_STATE16
#error "build with -DKDA_STATE16=0 (fp32 pool) or -DKDA_STATE16=1 (fp16 pool)"
#endif

// Column tile (BV) and threads per CTA.  A 2-byte state takes twice the
// columns of a 4-byte one so that a CTA moves the same bytes (the element-size
// rule of ROCm/ATOM pull request 2130, What); the values are tuned on GB300.
#if KDA_STATE16
using state_t = __half;
static constexpr int kBuildDtype = KDA_F16;
#ifndef KDA_DEC_BV
#define KDA_DEC_BV 64
#endif
#ifndef KDA_DEC_NT
#define KDA_DEC_NT 256
#endif
#ifndef KDA_VER_BV
#define KDA_VER_BV 32
#endif
#ifndef KDA_VER_NT
#define KDA_VER_NT 128
#endif
#else
using state_t = float;
static constexpr int kBuildDtype = KDA_F32;
#ifndef KDA_DEC_BV
#define KDA_DEC_BV 32
#endif
#ifndef KDA_DEC_NT
#define KDA_DEC_NT 128
#endif
#ifndef KDA_VER_BV
#define KDA_VER_BV 32
#endif
#ifndef KDA_VER_NT
#define KDA_VER_NT 128
#endif
#endif

namespace {

int elem_size(int32_t dtype) {
    switch (dtype) {
        case KDA_F32: return 4;
        case KDA_F16: return 2;
        case KDA_BF16: return 2;
        default: return 0;
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape, alignment and dtype of one pool, without the build-dtype rule.
int check_pool_self(const kda_pool* p) {
    if (p == nullptr) return KDA_ERR_NULL;
    if (p->dtype != KDA_F32 && p->dtype != KDA_F16) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (p->base == nullptr) return KDA_ERR_NULL;
    if (p->hv < 1 || p->num_slots < 1) return KDA_ERR_SHAPE;
    if (p->k < 16 || p->k > kda::KMAX || p->k % 16 != 0) return KDA_ERR_SHAPE;
    if (p->v < 16 || p->v > kda::KMAX || p->v % 16 != 0) return KDA_ERR_SHAPE;
    const int64_t per_slot = (int64_t)p->hv * p->k * p->v;
    if (p->slot_stride < per_slot) return KDA_ERR_SHAPE;
    const int es = elem_size(p->dtype);
    if (!aligned(p->base, 16) || (p->slot_stride * es) % 16 != 0) return KDA_ERR_ALIGN;
    return KDA_OK;
}

int check_pool_for_build(const kda_pool* p) {
    const int rc = check_pool_self(p);
    if (rc != KDA_OK) return rc;
    if (p->dtype != kBuildDtype) return KDA_ERR_DTYPE_MISMATCH;
    return KDA_OK;
}

template <int BV, int NT, bool VERIFY, typename QT>
int launch_typed(const kda::StepParams& prm, cudaStream_t stream) {
    const int64_t vt = (prm.v + BV - 1) / BV;
    const int64_t blocks = (int64_t)prm.n * prm.hv * vt;
    if (blocks > 0x7fffffffLL) return KDA_ERR_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kda::kda_step_kernel<state_t, QT, BV, NT, VERIFY>, prm);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

template <int BV, int NT, bool VERIFY>
int launch(const kda::StepParams& prm, int32_t qkv_dtype, cudaStream_t stream) {
    switch (qkv_dtype) {
        case KDA_F32: return launch_typed<BV, NT, VERIFY, float>(prm, stream);
        case KDA_F16: return launch_typed<BV, NT, VERIFY, __half>(prm, stream);
        case KDA_BF16: return launch_typed<BV, NT, VERIFY, __nv_bfloat16>(prm, stream);
        default: return KDA_ERR_DTYPE_UNSUPPORTED;
    }
}

// Shared argument checks of the two step entry points.
int check_step_args(const kda_pool* pool, const int32_t* init_slot, int32_t n, int32_t t,
                    const void* q, const void* k, const void* v, int32_t qkv_dtype,
                    const float* a, const float* b, const float* o, const int32_t* dev_status) {
    int rc = check_pool_for_build(pool);
    if (rc != KDA_OK) return rc;
    if (n < 0 || t < 0) return KDA_ERR_ARG;
    const int qs = elem_size(qkv_dtype);
    if (qs == 0) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (n == 0 || t == 0) return KDA_OK;  // nothing to do; empty buffers may be NULL
    if (!init_slot || !q || !k || !v || !a || !b || !o || !dev_status) return KDA_ERR_NULL;
    if (!aligned(init_slot, 4) || !aligned(dev_status, 4) || !aligned(a, 4) || !aligned(b, 4) ||
        !aligned(o, 4) || !aligned(q, qs) || !aligned(k, qs) || !aligned(v, qs))
        return KDA_ERR_ALIGN;
    return KDA_OK;
}

kda::StepParams make_params(const kda_pool* pool, const int32_t* init_slot,
                            const int32_t* snap_slot, const uint8_t* reset, int32_t n,
                            int32_t t, const void* q, const void* k, const void* v,
                            const float* a, const float* b, float* o, int32_t* dev_status) {
    kda::StepParams prm;
    prm.pool = pool->base;
    prm.num_slots = pool->num_slots;
    prm.slot_stride = pool->slot_stride;
    prm.hv = pool->hv;
    prm.k = pool->k;
    prm.v = pool->v;
    prm.n = n;
    prm.t = t;
    prm.init_slot = init_slot;
    prm.snap_slot = snap_slot;
    prm.reset = reset;
    prm.q = q;
    prm.kk = k;
    prm.vv = v;
    prm.a = a;
    prm.b = b;
    prm.o = o;
    prm.status = dev_status;
    prm.inv_sqrt_k = 1.0f / sqrtf((float)pool->k);
    return prm;
}

}  // namespace

extern "C" {

int kda_build_state_dtype(void) { return kBuildDtype; }

int kda_pool_check(const kda_pool* pools, int32_t n_layers) {
    if (pools == nullptr) return KDA_ERR_NULL;
    if (n_layers < 1) return KDA_ERR_ARG;
    // Every pool must be a valid fp32/fp16 pool on its own first.
    for (int32_t l = 0; l < n_layers; ++l) {
        const int rc = check_pool_self(&pools[l]);
        if (rc != KDA_OK) return rc;
    }
    // One dtype and one head shape across every layer.
    for (int32_t l = 1; l < n_layers; ++l) {
        if (pools[l].dtype != pools[0].dtype || pools[l].hv != pools[0].hv ||
            pools[l].k != pools[0].k || pools[l].v != pools[0].v)
            return KDA_ERR_LAYERS_DISAGREE;
    }
    return pools[0].dtype == kBuildDtype ? KDA_OK : KDA_ERR_DTYPE_MISMATCH;
}

int kda_state_bytes(const kda_pool* pool, int64_t* bytes_per_slot) {
    if (pool == nullptr || bytes_per_slot == nullptr) return KDA_ERR_NULL;
    if (pool->dtype != KDA_F32 && pool->dtype != KDA_F16) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (pool->hv < 1 || pool->k < 1 || pool->v < 1) return KDA_ERR_SHAPE;
    *bytes_per_slot = (int64_t)pool->hv * pool->k * pool->v * elem_size(pool->dtype);
    return KDA_OK;
}

int kda_decode_step(const kda_pool* pool, const int32_t* slot_ids, const uint8_t* reset,
                    int32_t n, const void* q, const void* k, const void* v, int32_t qkv_dtype,
                    const float* a, const float* b, float* o, int32_t* dev_status,
                    void* stream) {
    const int rc = check_step_args(pool, slot_ids, n, 1, q, k, v, qkv_dtype, a, b, o, dev_status);
    if (rc != KDA_OK) return rc;
    if (n == 0) return KDA_OK;
    const kda::StepParams prm =
        make_params(pool, slot_ids, nullptr, reset, n, 1, q, k, v, a, b, o, dev_status);
    return launch<KDA_DEC_BV, KDA_DEC_NT, false>(prm, qkv_dtype, static_cast<cudaStream_t>(stream));
}

int kda_spec_verify(const kda_pool* pool, const int32_t* init_slot, const int32_t* snap_slot,
                    const uint8_t* reset, int32_t n, int32_t t, const void* q, const void* k,
                    const void* v, int32_t qkv_dtype, const float* a, const float* b,
                    float* o, int32_t* dev_status, void* stream) {
    const int rc = check_step_args(pool, init_slot, n, t, q, k, v, qkv_dtype, a, b, o, dev_status);
    if (rc != KDA_OK) return rc;
    if (n == 0 || t == 0) return KDA_OK;
    if (snap_slot == nullptr) return KDA_ERR_NULL;
    if (!aligned(snap_slot, 4)) return KDA_ERR_ALIGN;
    const kda::StepParams prm =
        make_params(pool, init_slot, snap_slot, reset, n, t, q, k, v, a, b, o, dev_status);
    return launch<KDA_VER_BV, KDA_VER_NT, true>(prm, qkv_dtype, static_cast<cudaStream_t>(stream));
}

const char* kda_strerror(int32_t code) {
    switch (code) {
        case KDA_OK: return "ok";
        case KDA_ERR_NULL: return "a required pointer is NULL";
        case KDA_ERR_DTYPE_MISMATCH: return "state pool dtype differs from the library's build dtype";
        case KDA_ERR_DTYPE_UNSUPPORTED: return "unsupported dtype (state pools are fp32 or fp16 only; q/k/v fp32, fp16 or bf16)";
        case KDA_ERR_LAYERS_DISAGREE: return "layers disagree on the state dtype or head shape";
        case KDA_ERR_SHAPE: return "bad shape (K and V must be multiples of 16 in 16..128; slot stride >= hv*k*v)";
        case KDA_ERR_ALIGN: return "misaligned pointer or stride (pool 16-byte aligned; inputs naturally aligned)";
        case KDA_ERR_LAUNCH: return "CUDA kernel launch failed";
        case KDA_ERR_SLOT_RANGE: return "a slot id lies outside [0, num_slots); its tiles were skipped";
        case KDA_ERR_ARG: return "bad argument";
        default: return "unknown kda status code";
    }
}

}  // extern "C"
