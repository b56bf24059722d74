// C ABI of the KDA recurrent-state library (declared in include/kda.h).
//
// This translation unit is compiled once per state-pool dtype:
//   -DKDA_STATE16=0 -> libkda_h0.so (fp32 pool)
//   -DKDA_STATE16=1 -> libkda_h1.so (fp16 pool)
// following ROCm/ATOM pull request 2945 (Changes): the pool's dtype is a build
// constant, and a pool of the other dtype is refused at call time.
//
// Host side: validate every argument synchronously, encode the pool's TMA
// tensor map, and enqueue exactly one kernel on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "kda.h"
#include "kda_decode_tma.cuh"
#include "kda_verify_tma.cuh"
#include "kda_conv.cuh"
#include "kda_ckpt.cuh"
#include "kda_prefill_chunk.cuh"
#include "kda_stage.cuh"

#ifndef KDA_STATE16
#error "build with -DKDA_STATE16=0 (fp32 pool) or -DKDA_STATE16=1 (fp16 pool)"
#endif

// Tile shapes.  A tile is BV state columns x all K rows; BV * element size is
// 128 bytes, one TMA box row and one swizzle span, so a 2-byte state takes
// twice the columns of a 4-byte one and a tile moves the same bytes (the
// element-size rule of ROCm/ATOM pull request 2130, What).  Decode runs one
// CTA of DEC_NT threads per tile, at least DEC_MINB resident per SM; the values
// are tuned on GB300.
// Verify carries the state in registers across tokens and runs its tokens in
// sequence, so its tiles are 32 columns wide (128-byte rows for fp32, 64-byte
// rows for fp16), for registers and for parallelism.
#if KDA_STATE16
using state_t = __half;
static constexpr int kBuildDtype = KDA_F16;
#ifndef KDA_DEC_BV
#define KDA_DEC_BV 64
#endif
#ifndef KDA_VER_BV
#define KDA_VER_BV 32
#endif
#else
using state_t = float;
static constexpr int kBuildDtype = KDA_F32;
#ifndef KDA_DEC_BV
#define KDA_DEC_BV 32
#endif
#ifndef KDA_VER_BV
#define KDA_VER_BV 32
#endif
#endif

#ifndef KDA_DEC_NT
#define KDA_DEC_NT 128
#endif
#ifndef KDA_DEC_MINB
#if KDA_STATE16
#define KDA_DEC_MINB 8
#else
#define KDA_DEC_MINB 11
#endif
#endif
// Decode tiles per CTA for launches past one wave: an fp16 pool's two
// 64-column tiles of a head then share one CTA (768 CTAs at N = 64, all
// resident); an fp32 pool's stay one per CTA (two would leave 6 CTAs per SM
// for 3072 tiles).  Launches within one wave keep one tile per CTA, for the
// parallelism.
#ifndef KDA_DEC_TPC
#if KDA_STATE16
#define KDA_DEC_TPC 2
#else
#define KDA_DEC_TPC 1
#endif
#endif
// Warps per 16-column block of the prefill scan: KDA_PSCAN_KS_MID when the
// grid has a CTA per SM or more only with one or two blocks per CTA, and
// KDA_PSCAN_KS_FEW when it has fewer CTAs than SMs (few long prompts).
#ifndef KDA_PSCAN_KS_MID
#define KDA_PSCAN_KS_MID 1
#endif
#ifndef KDA_PSCAN_KS_FEW
#define KDA_PSCAN_KS_FEW 2
#endif
#ifndef KDA_DEC_KEEP
#define KDA_DEC_KEEP 0
#endif
// The same two settings for the kernel with more than one tile per CTA.  Its
// shared memory (two state tiles) allows 6 CTAs per SM, so 6 sets the register
// cap (80), and the rows' raw 16-byte words from the sums pass stay in
// registers for the update pass (32 registers) instead of being read again.
#ifndef KDA_DEC_KEEP2
#define KDA_DEC_KEEP2 1
#endif
#ifndef KDA_DEC_MINB2
#define KDA_DEC_MINB2 6
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
    if (p->num_slots > 0x7fffffffLL) return KDA_ERR_SHAPE;  // slot ids are int32
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Tensor map of the pool as a 3-D tensor [num_slots][hv * k][v] (v innermost),
// box [1][k][bv]: one tile of one head of one slot, swizzled to match the row
// bytes.  Out-of-range columns of a partial last tile load as zeros and are
// not stored.
int make_pool_map(const kda_pool* pool, int bv, CUtensorMap* map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return KDA_ERR_LAUNCH;
    const int es = elem_size(pool->dtype);
    const cuuint64_t dims[3] = {(cuuint64_t)pool->v, (cuuint64_t)pool->hv * (cuuint64_t)pool->k,
                                (cuuint64_t)pool->num_slots};
    const cuuint64_t strides[2] = {(cuuint64_t)pool->v * es, (cuuint64_t)pool->slot_stride * es};
    const cuuint32_t box[3] = {(cuuint32_t)bv, (cuuint32_t)pool->k, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const int rowbytes = bv * es;
    const CUtensorMapSwizzle sw = rowbytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : rowbytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_32B;
    const CUresult r = enc(map, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           3, pool->base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KDA_OK : KDA_ERR_LAUNCH;
}

// Resident CTAs per SM of `kernel` with `smem` dynamic bytes (also raises the
// kernel's dynamic shared-memory limit); cached per (kernel, device).
int occupancy(const void* kernel, int threads, size_t smem, int* blocks_per_sm, int* sms) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, std::pair<int, int>> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({kernel, dev});
    if (it == cache.end()) {
        int occ = 0, count = 0;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            occ < 1)
            return KDA_ERR_LAUNCH;
        it = cache.emplace(std::make_pair(kernel, dev), std::make_pair(occ, count)).first;
    }
    *blocks_per_sm = it->second.first;
    *sms = it->second.second;
    return KDA_OK;
}

// The scratch of kda_prefill_chunked_noalloc: a file-scope device array, so
// that the call allocates nothing.  Its address is looked up once per device.
static __device__ __align__(256) float g_prefill_scratch[KDA_PREFILL_SCRATCH_BYTES / 4];

void* prefill_scratch() {
    static std::mutex mu;
    static std::map<int, void*> addr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find(dev);
    if (it == addr.end()) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess) return nullptr;
        it = addr.emplace(dev, p).first;
    }
    return it->second;
}

// Programmatic dependent launch attribute when the caller asked for it.
void set_pdl(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, uint32_t flags) {
    if (flags & KDA_LAUNCH_PDL) {
        attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr->val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
}

// The prefill scan pass with WPC column blocks of 16 value columns per CTA,
// KS warps per block, launched with programmatic dependent launch so that it
// starts while the first pass drains.
template <int WPC, int KS>
int launch_scan(const kda::StepParams& prm, const uint8_t* ws, int64_t heads, int v, cudaStream_t st) {
    constexpr size_t smem = kda::PrefillScanSmem<WPC, KS>::BYTES;
    // K = 128 (the configured models' key dimension) gets a build whose row
    // loops have compile-time bounds
    auto scan = prm.k == kda::KMAX ? kda::kda_prefill_scan_kernel<state_t, WPC, KS, true>
                                   : kda::kda_prefill_scan_kernel<state_t, WPC, KS, false>;
    int occ = 0, sms = 0;
    const int rc = occupancy(reinterpret_cast<const void*>(scan), WPC * KS * 32, smem, &occ, &sms);
    if (rc != KDA_OK) return rc;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    cfg.gridDim = dim3((unsigned)(heads * ((v + 16 * WPC - 1) / (16 * WPC))), 1, 1);
    cfg.blockDim = dim3(WPC * KS * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    set_pdl(cfg, &attr, KDA_LAUNCH_PDL);
    return cudaLaunchKernelEx(&cfg, scan, prm, ws) == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

template <typename QT, bool FULLK, int TPC, bool CONV>
int launch_decode_k(const kda_pool* pool, const kda::StepParams& prm, cudaStream_t stream) {
    constexpr int BV = KDA_DEC_BV, NT = KDA_DEC_NT;
    constexpr size_t smem = kda::decode_smem_bytes<state_t, BV, NT, (int)sizeof(QT), TPC>();
    constexpr int MINB = TPC > 1 ? KDA_DEC_MINB2 : KDA_DEC_MINB;
    constexpr bool KEEP = (TPC > 1 ? KDA_DEC_KEEP2 : KDA_DEC_KEEP) != 0;
    auto kernel = kda::kda_decode_kernel<state_t, QT, BV, NT, MINB, KEEP, FULLK, TPC, CONV>;
    // CTAs: TPC column blocks each
    const int64_t tiles = (int64_t)prm.n * prm.hv * (((prm.v + BV - 1) / BV + TPC - 1) / TPC);
    if (tiles > 0x7fffffffLL) return KDA_ERR_SHAPE;
    CUtensorMap map;
    int rc = make_pool_map(pool, BV, &map);
    if (rc != KDA_OK) return rc;
    int occ = 0, sms = 0;
    rc = occupancy(reinterpret_cast<const void*>(kernel), NT, smem, &occ, &sms);
    if (rc != KDA_OK) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    set_pdl(cfg, &attr, prm.flags);
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, map, prm);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

// K = 128 (the configured models' key dimension) gets a build without the
// per-row bound checks.
template <typename QT, int TPC, bool CONV>
int launch_decode_t(const kda_pool* pool, const kda::StepParams& prm, cudaStream_t stream) {
    return prm.k == kda::KMAX ? launch_decode_k<QT, true, TPC, CONV>(pool, prm, stream)
                              : launch_decode_k<QT, false, TPC, CONV>(pool, prm, stream);
}

// KDA_DEC_TPC tiles per CTA when the one-tile grid is more than one wave of
// the one-tile kernel, else one.  CONV: the decode with the fused
// convolution, two tiles a CTA on either pool past one wave: each CTA forms
// its q/k head's 2 K conv outputs, so fewer CTAs a head form them fewer times
// and share each q/k window among fewer readers.
template <typename QT, bool CONV = false>
int launch_decode(const kda_pool* pool, const kda::StepParams& prm, cudaStream_t stream) {
    constexpr int TPC = CONV ? 2 : KDA_DEC_TPC;
    if constexpr (TPC > 1) {
        constexpr int BV = KDA_DEC_BV, NT = KDA_DEC_NT;
        constexpr size_t smem = kda::decode_smem_bytes<state_t, BV, NT, (int)sizeof(QT)>();
        const int64_t tiles = (int64_t)prm.n * prm.hv * ((prm.v + BV - 1) / BV);
        int occ = 0, sms = 0;
        const int rc = occupancy(reinterpret_cast<const void*>(
                                     kda::kda_decode_kernel<state_t, QT, BV, NT, KDA_DEC_MINB, KDA_DEC_KEEP != 0, true>),
                                 NT, smem, &occ, &sms);
        if (rc != KDA_OK) return rc;
        if (tiles > (int64_t)occ * sms) return launch_decode_t<QT, TPC, CONV>(pool, prm, stream);
    }
    return launch_decode_t<QT, 1, CONV>(pool, prm, stream);
}

template <typename QT, bool WIDE, bool CONV>
int launch_verify_shape(const kda_pool* pool, const kda::StepParams& prm, cudaStream_t stream, int64_t tiles) {
    constexpr int BV = KDA_VER_BV;
    using SH = kda::VerifyShape<state_t, BV, (int)sizeof(QT), WIDE>;
    constexpr size_t smem = kda::verify_smem_bytes<state_t, BV, (int)sizeof(QT), WIDE>();
    // an fp16 pool at K = 128 gets the build with compile-time row loops; an
    // fp32 pool's 256-thread tiles have no register room for it (it spills)
    // (the fused convolution's wide shape exists for K = 128 only: see launch_verify)
    constexpr bool kFullkOk = sizeof(state_t) == 2;
    auto kernel = (kFullkOk && prm.k == kda::KMAX) || (CONV && WIDE)
                      ? kda::kda_verify_kernel<state_t, QT, BV, kFullkOk, WIDE, CONV>
                      : kda::kda_verify_kernel<state_t, QT, BV, false, WIDE && !CONV, CONV>;
    CUtensorMap map;
    int rc = make_pool_map(pool, BV, &map);
    if (rc != KDA_OK) return rc;
    int occ = 0, sms = 0;
    rc = occupancy(reinterpret_cast<const void*>(kernel), SH::NT, smem, &occ, &sms);
    if (rc != KDA_OK) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, 1, 1);
    cfg.blockDim = dim3(SH::NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    set_pdl(cfg, &attr, prm.flags);
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, map, prm);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

// A launch that fits in one wave of the default shape runs it; a larger one,
// on an fp16 pool with 16-bit inputs, runs the wide shape (4 CTAs per SM).
// CONV: the step with the short convolution fused in front.
template <typename QT, bool CONV = false>
int launch_verify(const kda_pool* pool, const kda::StepParams& prm, cudaStream_t stream) {
    constexpr int BV = KDA_VER_BV;
    const int64_t tiles = (int64_t)prm.n * prm.hv * ((prm.v + BV - 1) / BV);
    if (tiles > 0x7fffffffLL) return KDA_ERR_SHAPE;
    constexpr bool kWideOk = sizeof(state_t) == 2 && sizeof(QT) == 2;
    if constexpr (kWideOk) {
        using SH = kda::VerifyShape<state_t, BV, (int)sizeof(QT)>;
        constexpr size_t smem = kda::verify_smem_bytes<state_t, BV, (int)sizeof(QT)>();
        int occ = 0, sms = 0;
        const int rc = occupancy(reinterpret_cast<const void*>(kda::kda_verify_kernel<state_t, QT, BV, false>),
                                 SH::NT, smem, &occ, &sms);
        if (rc != KDA_OK) return rc;
        // the fused convolution's wide build at K < 128 has no register room:
        // those launches keep the default shape, in more waves
        if (tiles > (int64_t)occ * sms && (!CONV || prm.k == kda::KMAX))
            return launch_verify_shape<QT, kWideOk, CONV>(pool, prm, stream, tiles);
    }
    return launch_verify_shape<QT, false, CONV>(pool, prm, stream, tiles);
}

template <bool VERIFY>
int launch(const kda_pool* pool, const kda::StepParams& prm, int32_t qkv_dtype, cudaStream_t stream) {
    switch (qkv_dtype) {
        case KDA_F32:
            return VERIFY ? launch_verify<float>(pool, prm, stream) : launch_decode<float>(pool, prm, stream);
        case KDA_F16:
            return VERIFY ? launch_verify<__half>(pool, prm, stream) : launch_decode<__half>(pool, prm, stream);
        case KDA_BF16:
            return VERIFY ? launch_verify<__nv_bfloat16>(pool, prm, stream)
                          : launch_decode<__nv_bfloat16>(pool, prm, stream);
        default: return KDA_ERR_DTYPE_UNSUPPORTED;
    }
}

// Shared argument checks of the two step entry points.
int check_step_args(const kda_pool* pool, const int32_t* init_slot, int32_t n, int32_t t,
                    const void* q, const void* k, const void* v, int32_t qkv_dtype,
                    const float* a, const float* b, const float* o, const int32_t* dev_status,
                    uint32_t flags) {
    int rc = check_pool_for_build(pool);
    if (rc != KDA_OK) return rc;
    if (n < 0 || t < 0) return KDA_ERR_ARG;
    if (flags & ~(uint32_t)(KDA_LAUNCH_PDL | KDA_LAUNCH_PDL_EARLY_STATE | KDA_LAUNCH_TEST_WITHHOLD_STATE))
        return KDA_ERR_ARG;
    const int qs = elem_size(qkv_dtype);
    if (qs == 0) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (n == 0 || t == 0) return KDA_OK;  // nothing to do; empty buffers may be NULL
    if (!init_slot || !q || !k || !v || !a || !b || !o || !dev_status) return KDA_ERR_NULL;
    // q, k, v and a rows are moved by 16-byte bulk copies
    if (!aligned(init_slot, 4) || !aligned(dev_status, 4) || !aligned(b, 4) || !aligned(o, 4) ||
        !aligned(a, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))
        return KDA_ERR_ALIGN;
    return KDA_OK;
}

kda::StepParams make_params(const kda_pool* pool, const int32_t* init_slot,
                            const int32_t* snap_slot, const uint8_t* reset, int32_t n,
                            int32_t t, const void* q, const void* k, const void* v,
                            const float* a, const float* b, float* o, int32_t* dev_status,
                            uint32_t flags) {
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
    prm.flags = flags;
    // plain decode / verify: one q/k head per value head, one slot per request
    // row (init), t snapshot columns, no accepted column, no offsets, plain gate
    prm.hqk = pool->hv;
    prm.init_stride = 1;
    prm.snap_stride = t;
    prm.num_cols = 1;
    prm.accepted = nullptr;
    prm.cu = nullptr;
    prm.a_log = nullptr;
    prm.dt_bias = nullptr;
    prm.mode = 0;
    prm.total = n * t;
    prm.final_slot = nullptr;
    prm.conv = kda::StepParams::Conv{};
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
                    uint32_t flags, void* stream) {
    const int rc = check_step_args(pool, slot_ids, n, 1, q, k, v, qkv_dtype, a, b, o, dev_status, flags);
    if (rc != KDA_OK) return rc;
    if (n == 0) return KDA_OK;
    const kda::StepParams prm =
        make_params(pool, slot_ids, nullptr, reset, n, 1, q, k, v, a, b, o, dev_status, flags);
    return launch<false>(pool, prm, qkv_dtype, static_cast<cudaStream_t>(stream));
}

int kda_spec_verify(const kda_pool* pool, const int32_t* init_slot, const int32_t* snap_slot,
                    const uint8_t* reset, int32_t n, int32_t t, const void* q, const void* k,
                    const void* v, int32_t qkv_dtype, const float* a, const float* b,
                    float* o, int32_t* dev_status, uint32_t flags, void* stream) {
    const int rc = check_step_args(pool, init_slot, n, t, q, k, v, qkv_dtype, a, b, o, dev_status, flags);
    if (rc != KDA_OK) return rc;
    if (n == 0 || t == 0) return KDA_OK;
    if (snap_slot == nullptr) return KDA_ERR_NULL;
    if (!aligned(snap_slot, 4)) return KDA_ERR_ALIGN;
    const kda::StepParams prm =
        make_params(pool, init_slot, snap_slot, reset, n, t, q, k, v, a, b, o, dev_status, flags);
    return launch<true>(pool, prm, qkv_dtype, static_cast<cudaStream_t>(stream));
}

int kda_step(const kda_pool* pool, const kda_step_args* args, int32_t* dev_status, uint32_t flags,
             void* stream) {
    if (args == nullptr) return KDA_ERR_NULL;
    const kda_step_args& g = *args;
    int rc = check_pool_for_build(pool);
    if (rc != KDA_OK) return rc;
    if (g.n < 0 || g.total < 0 || g.max_t < 0 || g.reserved != 0) return KDA_ERR_ARG;
    if (flags & ~(uint32_t)(KDA_LAUNCH_PDL | KDA_LAUNCH_PDL_EARLY_STATE | KDA_LAUNCH_TEST_WITHHOLD_STATE))
        return KDA_ERR_ARG;
    if (elem_size(g.qkv_dtype) == 0) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (g.h_qk < 1 || pool->hv % g.h_qk != 0 || g.num_cols < 1) return KDA_ERR_SHAPE;
    if (g.in_place) {
        if (g.cu_seqlens != nullptr || g.total != g.n || (g.n > 0 && g.max_t != 1)) return KDA_ERR_SHAPE;
    } else {
        if (g.max_t > g.num_cols) return KDA_ERR_SHAPE;
        if (g.cu_seqlens == nullptr && (int64_t)g.total != (int64_t)g.n * g.max_t) return KDA_ERR_SHAPE;
    }
    if (g.n == 0 || g.total == 0 || g.max_t == 0) return KDA_OK;
    if (!g.slot_table || !g.q || !g.k || !g.v || !g.a || !g.b || !g.o || !dev_status) return KDA_ERR_NULL;
    if (!aligned(g.slot_table, 4) || !aligned(dev_status, 4) || !aligned(g.b, 4) || !aligned(g.o, 4) ||
        !aligned(g.a, 16) || !aligned(g.q, 16) || !aligned(g.k, 16) || !aligned(g.v, 16) ||
        (g.cu_seqlens && !aligned(g.cu_seqlens, 4)) || (g.accepted && !aligned(g.accepted, 4)) ||
        (g.a_log && !aligned(g.a_log, 4)) || (g.dt_bias && !aligned(g.dt_bias, 4)))
        return KDA_ERR_ALIGN;
    kda::StepParams prm = make_params(pool, g.slot_table, g.in_place ? nullptr : g.slot_table, g.reset, g.n,
                                      g.in_place ? 1 : g.max_t, g.q, g.k, g.v, g.a, g.b, g.o, dev_status, flags);
    prm.hqk = g.h_qk;
    prm.init_stride = g.num_cols;
    prm.snap_stride = g.num_cols;
    prm.num_cols = g.num_cols;
    prm.accepted = g.accepted;
    prm.cu = g.in_place ? nullptr : g.cu_seqlens;
    prm.total = g.total;
    prm.a_log = g.a_log;
    prm.dt_bias = g.dt_bias;
    prm.mode = kda::MODE_PADDING;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return g.in_place ? launch<false>(pool, prm, g.qkv_dtype, st) : launch<true>(pool, prm, g.qkv_dtype, st);
}

int kda_prefill(const kda_pool* pool, const kda_prefill_args* args, int32_t* dev_status, uint32_t flags,
                void* stream) {
    if (args == nullptr) return KDA_ERR_NULL;
    const kda_prefill_args& g = *args;
    int rc = check_pool_for_build(pool);
    if (rc != KDA_OK) return rc;
    if (g.n < 0 || g.total < 0 || g.max_t < 0 || g.reserved != 0) return KDA_ERR_ARG;
    if (flags & ~(uint32_t)(KDA_LAUNCH_PDL | KDA_LAUNCH_PDL_EARLY_STATE)) return KDA_ERR_ARG;
    if (elem_size(g.qkv_dtype) == 0) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (g.h_qk < 1 || pool->hv % g.h_qk != 0) return KDA_ERR_SHAPE;
    if (g.cu_seqlens == nullptr && (int64_t)g.total != (int64_t)g.n * g.max_t) return KDA_ERR_SHAPE;
    // with no tokens at all there is still work: each request's initial state
    // goes to its final slot (the token buffers may then be NULL)
    if (g.n == 0) return KDA_OK;
    if (!g.init_slot || !g.final_slot || !dev_status) return KDA_ERR_NULL;
    if (g.total > 0 && (!g.q || !g.k || !g.v || !g.a || !g.b || !g.o)) return KDA_ERR_NULL;
    if (!aligned(g.init_slot, 4) || !aligned(g.final_slot, 4) || !aligned(dev_status, 4) || !aligned(g.b, 4) ||
        !aligned(g.o, 4) || !aligned(g.a, 16) || !aligned(g.q, 16) || !aligned(g.k, 16) || !aligned(g.v, 16) ||
        (g.cu_seqlens && !aligned(g.cu_seqlens, 4)) || (g.a_log && !aligned(g.a_log, 4)) ||
        (g.dt_bias && !aligned(g.dt_bias, 4)))
        return KDA_ERR_ALIGN;
    kda::StepParams prm = make_params(pool, g.init_slot, nullptr, g.reset, g.n, g.max_t, g.q, g.k, g.v, g.a, g.b,
                                      g.o, dev_status, flags);
    prm.hqk = g.h_qk;
    prm.cu = g.cu_seqlens;
    prm.total = g.total;
    prm.a_log = g.a_log;
    prm.dt_bias = g.dt_bias;
    prm.mode = kda::MODE_PADDING;
    prm.final_slot = g.final_slot;
    return launch<true>(pool, prm, g.qkv_dtype, static_cast<cudaStream_t>(stream));
}

int kda_prefill_workspace_bytes(const kda_pool* pool, int32_t n, int32_t total, int64_t* bytes) {
    if (pool == nullptr || bytes == nullptr) return KDA_ERR_NULL;
    if (n < 0 || total < 0) return KDA_ERR_ARG;
    // one block per (chunk slot, head); chunk slots stay below total / 16 + n
    *bytes = ((int64_t)total / kda::PCH + n) * pool->hv * (int64_t)kda::PCH_BYTES;
    return KDA_OK;
}

int kda_prefill_chunked(const kda_pool* pool, const kda_prefill_args* args, void* workspace,
                        int64_t workspace_bytes, int32_t* dev_status, uint32_t flags, void* stream) {
    if (args == nullptr) return KDA_ERR_NULL;
    const kda_prefill_args& g = *args;
    int rc = check_pool_for_build(pool);
    if (rc != KDA_OK) return rc;
    if (g.n < 0 || g.total < 0 || g.max_t < 0 || g.reserved != 0) return KDA_ERR_ARG;
    if (flags & ~(uint32_t)(KDA_LAUNCH_PDL | KDA_LAUNCH_PDL_EARLY_STATE)) return KDA_ERR_ARG;
    if (elem_size(g.qkv_dtype) == 0) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (g.h_qk < 1 || pool->hv % g.h_qk != 0) return KDA_ERR_SHAPE;
    if (g.cu_seqlens == nullptr && (int64_t)g.total != (int64_t)g.n * g.max_t) return KDA_ERR_SHAPE;
    // as in kda_prefill: with no tokens the scan pass alone stores the initial states
    if (g.n == 0) return KDA_OK;
    if (!g.init_slot || !g.final_slot || !dev_status || !workspace) return KDA_ERR_NULL;
    if (g.total > 0 && (!g.q || !g.k || !g.v || !g.a || !g.b || !g.o)) return KDA_ERR_NULL;
    int64_t need = 0;
    kda_prefill_workspace_bytes(pool, g.n, g.total, &need);
    if (workspace_bytes < need) return KDA_ERR_ARG;
    if (!aligned(workspace, 256) || !aligned(g.init_slot, 4) || !aligned(g.final_slot, 4) ||
        !aligned(dev_status, 4) || !aligned(g.b, 4) || !aligned(g.o, 4) || !aligned(g.a, 4) ||
        !aligned(g.q, 4) || !aligned(g.k, 4) || !aligned(g.v, 4) || (g.cu_seqlens && !aligned(g.cu_seqlens, 4)) ||
        (g.a_log && !aligned(g.a_log, 4)) || (g.dt_bias && !aligned(g.dt_bias, 4)))
        return KDA_ERR_ALIGN;
    kda::StepParams prm = make_params(pool, g.init_slot, nullptr, g.reset, g.n, g.max_t, g.q, g.k, g.v, g.a, g.b,
                                      g.o, dev_status, flags);
    prm.hqk = g.h_qk;
    prm.cu = g.cu_seqlens;
    prm.total = g.total;
    prm.a_log = g.a_log;
    prm.dt_bias = g.dt_bias;
    prm.mode = kda::MODE_PADDING;
    prm.final_slot = g.final_slot;
    const int max_chunks = (g.max_t + kda::PCH - 1) / kda::PCH;
    const int vtiles = (pool->v + 15) / 16;  // the narrowest scan tiling bounds the grid
    if ((int64_t)g.n * max_chunks > 0x7fffffffLL || (int64_t)g.n * pool->hv * vtiles > 0x7fffffffLL ||
        pool->hv > 65535)
        return KDA_ERR_SHAPE;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    cfg.gridDim = dim3((unsigned)(g.n * max_chunks), (unsigned)pool->hv, 1);
    cfg.blockDim = dim3(kda::KMAX, 1, 1);
    cfg.stream = st;
    set_pdl(cfg, &attr, flags);
    cudaError_t err = cudaSuccess;
    if (max_chunks > 0) {  // no chunk at all (max_t == 0): only the scan pass runs
        switch (g.qkv_dtype) {
            case KDA_F32: err = cudaLaunchKernelEx(&cfg, kda::kda_prefill_prep_kernel<float>, prm, ws, max_chunks); break;
            case KDA_F16: err = cudaLaunchKernelEx(&cfg, kda::kda_prefill_prep_kernel<__half>, prm, ws, max_chunks); break;
            default: err = cudaLaunchKernelEx(&cfg, kda::kda_prefill_prep_kernel<__nv_bfloat16>, prm, ws, max_chunks); break;
        }
    }
    if (err != cudaSuccess) return KDA_ERR_LAUNCH;
    // The most column blocks per scan CTA (they share each chunk's operand
    // copy) whose grid still covers the SMs.  When even one block per CTA
    // leaves SMs idle (few long prompts), each block's rows are split over
    // KS warps, which shortens every chunk step.
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KDA_ERR_LAUNCH;
    const int64_t heads = (int64_t)g.n * pool->hv;
    auto ctas = [&](int wpc) { return heads * ((pool->v + 16 * wpc - 1) / (16 * wpc)); };
    if (ctas(8) >= sms) return launch_scan<8, 1>(prm, ws, heads, pool->v, st);
    if (ctas(4) >= sms) return launch_scan<4, 1>(prm, ws, heads, pool->v, st);
    if (ctas(2) >= sms) return launch_scan<2, KDA_PSCAN_KS_MID>(prm, ws, heads, pool->v, st);
    if (ctas(1) >= sms) return launch_scan<1, KDA_PSCAN_KS_MID>(prm, ws, heads, pool->v, st);
    return launch_scan<1, KDA_PSCAN_KS_FEW>(prm, ws, heads, pool->v, st);
}

int kda_prefill_chunked_noalloc(const kda_pool* pool, const kda_prefill_args* args, int32_t* dev_status,
                                uint32_t flags, void* stream) {
    if (pool == nullptr || args == nullptr) return KDA_ERR_NULL;
    int64_t need = 0;
    const int rc = kda_prefill_workspace_bytes(pool, args->n, args->total, &need);
    if (rc != KDA_OK) return rc;
    if (need > KDA_PREFILL_SCRATCH_BYTES) return KDA_ERR_SHAPE;
    void* ws = prefill_scratch();
    if (ws == nullptr) return KDA_ERR_LAUNCH;
    return kda_prefill_chunked(pool, args, ws, KDA_PREFILL_SCRATCH_BYTES, dev_status, flags, stream);
}

int kda_conv_step(const kda_conv_window* win, const kda_conv_args* args, int32_t* dev_status,
                  uint32_t flags, void* stream) {
    if (win == nullptr || args == nullptr) return KDA_ERR_NULL;
    const kda_conv_args& g = *args;
    const int es = elem_size(win->dtype);
    if (es == 0) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (win->reserved != 0 || g.reserved != 0 || g.n < 0 || g.total < 0 || g.max_t < 0 ||
        (g.activation != 0 && g.activation != 1))
        return KDA_ERR_ARG;
    if (flags & ~(uint32_t)(KDA_LAUNCH_PDL | KDA_LAUNCH_PDL_EARLY_STATE)) return KDA_ERR_ARG;
    if (win->channels < 1 || g.kernel_width < 1 || g.kernel_width > kda::CONV_KW_MAX ||
        win->state_len < g.kernel_width - 1 || win->state_len > kda::CONV_L_MAX || win->num_slots < 1 ||
        win->slot_stride < (int64_t)win->state_len * win->channels)
        return KDA_ERR_SHAPE;
    if (g.cu_seqlens == nullptr && (int64_t)g.total != (int64_t)g.n * g.max_t) return KDA_ERR_SHAPE;
    if (g.n == 0 || g.total == 0 || g.max_t == 0) return KDA_OK;
    if (!win->base || !g.conv_slot || !g.x || !g.weight || !g.y || !dev_status) return KDA_ERR_NULL;
    if (!aligned(win->base, es) || !aligned(g.x, es) || !aligned(g.y, es) || !aligned(g.conv_slot, 4) ||
        !aligned(g.weight, 4) || !aligned(dev_status, 4) || (g.bias && !aligned(g.bias, 4)) ||
        (g.cu_seqlens && !aligned(g.cu_seqlens, 4)) || (g.accepted && !aligned(g.accepted, 4)))
        return KDA_ERR_ALIGN;
    // four channels a thread when the kernel is at most 4 wide and the channel
    // count and every address allow 4-element accesses, else one
    const int64_t vb = 4LL * es;
    const bool vec4 = g.kernel_width <= kda::CONV_VEC_KW_MAX && win->channels % 4 == 0 &&
                      win->slot_stride % 4 == 0 && aligned(win->base, vb) && aligned(g.x, vb) && aligned(g.y, vb);
    const int vc = vec4 ? 4 : 1, ct = vec4 ? kda::CONV_VEC_THREADS : kda::CONV_THREADS;
    const int64_t cblocks = (win->channels / vc + ct - 1) / ct;
    if (cblocks * g.n > 0x7fffffffLL) return KDA_ERR_SHAPE;
    kda::ConvParams prm;
    prm.window = win->base;
    prm.num_slots = win->num_slots;
    prm.slot_stride = win->slot_stride;
    prm.C = win->channels;
    prm.L = win->state_len;
    prm.KW = g.kernel_width;
    prm.n = g.n;
    prm.t = g.max_t;
    prm.total = g.total;
    prm.cu = g.cu_seqlens;
    prm.conv_slot = g.conv_slot;
    prm.accepted = g.accepted;
    prm.reset = g.reset;
    prm.x = g.x;
    prm.w = g.weight;
    prm.bias = g.bias;
    prm.y = g.y;
    prm.silu = g.activation;
    prm.flags = flags;
    prm.status = dev_status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cblocks * g.n), 1, 1);
    cfg.blockDim = dim3((unsigned)ct, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    set_pdl(cfg, &attr, flags);
    cudaError_t err;
    using namespace kda;
    constexpr int C1 = CONV_THREADS, C4 = CONV_VEC_THREADS, K1 = CONV_KW_MAX, K4 = CONV_VEC_KW_MAX;
    switch (win->dtype) {
        case KDA_F32:
            err = vec4 ? (g.kernel_width == 4 ? cudaLaunchKernelEx(&cfg, kda_conv_kernel<float, 4, C4, K4, 4>, prm)
                                               : cudaLaunchKernelEx(&cfg, kda_conv_kernel<float, 4, C4, K4, 0>, prm))
                       : cudaLaunchKernelEx(&cfg, kda_conv_kernel<float, 1, C1, K1, 0>, prm);
            break;
        case KDA_F16:
            err = vec4 ? (g.kernel_width == 4 ? cudaLaunchKernelEx(&cfg, kda_conv_kernel<__half, 4, C4, K4, 4>, prm)
                                               : cudaLaunchKernelEx(&cfg, kda_conv_kernel<__half, 4, C4, K4, 0>, prm))
                       : cudaLaunchKernelEx(&cfg, kda_conv_kernel<__half, 1, C1, K1, 0>, prm);
            break;
        default:
            err = vec4 ? (g.kernel_width == 4 ? cudaLaunchKernelEx(&cfg, kda_conv_kernel<__nv_bfloat16, 4, C4, K4, 4>, prm)
                                               : cudaLaunchKernelEx(&cfg, kda_conv_kernel<__nv_bfloat16, 4, C4, K4, 0>, prm))
                       : cudaLaunchKernelEx(&cfg, kda_conv_kernel<__nv_bfloat16, 1, C1, K1, 0>, prm);
            break;
    }
    return err == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

int kda_decode_conv_step(const kda_pool* pool, const kda_conv_window* win, const kda_decode_conv_args* args,
                         int32_t* dev_status, uint32_t flags, void* stream) {
    if (win == nullptr || args == nullptr) return KDA_ERR_NULL;
    const kda_decode_conv_args& g = *args;
    int rc = check_pool_for_build(pool);
    if (rc != KDA_OK) return rc;
    const int es = elem_size(win->dtype);
    if (es == 0) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (win->reserved != 0 || g.n < 0 || (g.activation != 0 && g.activation != 1)) return KDA_ERR_ARG;
    if (flags & ~(uint32_t)(KDA_LAUNCH_PDL | KDA_LAUNCH_PDL_EARLY_STATE)) return KDA_ERR_ARG;
    // one token a request keeps state_len - 1 old entries, all within the
    // kernel_width - 1 history it reads
    if (g.h_qk < 1 || pool->hv % g.h_qk != 0 || g.kernel_width < 1 || g.kernel_width > kda::DCONV_KW_MAX ||
        win->state_len < g.kernel_width - 1 || win->state_len > g.kernel_width || win->num_slots < 1 ||
        (int64_t)win->channels != 2LL * g.h_qk * pool->k + (int64_t)pool->hv * pool->v ||
        win->slot_stride < (int64_t)win->state_len * win->channels)
        return KDA_ERR_SHAPE;
    if (g.n == 0) return KDA_OK;
    if (!win->base || !g.slot_ids || !g.conv_slot || !g.x || !g.weight || !g.a || !g.b || !g.o ||
        !g.counters || !dev_status)
        return KDA_ERR_NULL;
    if (!aligned(win->base, es) || !aligned(g.x, es) || (g.y && !aligned(g.y, es)) || !aligned(g.slot_ids, 4) ||
        !aligned(g.conv_slot, 4) || !aligned(g.weight, 4) || (g.bias && !aligned(g.bias, 4)) ||
        !aligned(g.a, 16) || !aligned(g.b, 4) || !aligned(g.o, 4) || !aligned(g.counters, 4) ||
        !aligned(dev_status, 4) || (g.a_log && !aligned(g.a_log, 4)) || (g.dt_bias && !aligned(g.dt_bias, 4)))
        return KDA_ERR_ALIGN;
    kda::StepParams prm = make_params(pool, g.slot_ids, nullptr, g.reset, g.n, 1, nullptr, nullptr, nullptr,
                                      g.a, g.b, g.o, dev_status, flags);
    prm.hqk = g.h_qk;
    prm.a_log = g.a_log;
    prm.dt_bias = g.dt_bias;
    prm.conv.window = win->base;
    prm.conv.num_slots = win->num_slots;
    prm.conv.slot_stride = win->slot_stride;
    prm.conv.C = win->channels;
    prm.conv.L = win->state_len;
    prm.conv.KW = g.kernel_width;
    prm.conv.silu = g.activation;
    prm.conv.slot = g.conv_slot;
    prm.conv.x = g.x;
    prm.conv.w = g.weight;
    prm.conv.bias = g.bias;
    prm.conv.y = g.y;
    prm.conv.counters = g.counters;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (win->dtype) {
        case KDA_F32: return launch_decode<float, true>(pool, prm, st);
        case KDA_F16: return launch_decode<__half, true>(pool, prm, st);
        default: return launch_decode<__nv_bfloat16, true>(pool, prm, st);
    }
}

int kda_step_conv(const kda_pool* pool, const kda_step_args* args, const kda_conv_window* win,
                  const kda_step_conv_args* cv, int32_t* dev_status, uint32_t flags, void* stream) {
    if (args == nullptr || win == nullptr || cv == nullptr) return KDA_ERR_NULL;
    const kda_step_args& g = *args;
    int rc = check_pool_for_build(pool);
    if (rc != KDA_OK) return rc;
    const int es = elem_size(win->dtype);
    if (es == 0) return KDA_ERR_DTYPE_UNSUPPORTED;
    if (g.n < 0 || g.total < 0 || g.max_t < 0 || g.reserved != 0 || win->reserved != 0 || g.in_place != 0 ||
        g.q != nullptr || g.k != nullptr || g.v != nullptr || g.qkv_dtype != win->dtype ||
        (cv->activation != 0 && cv->activation != 1))
        return KDA_ERR_ARG;
    if (flags & ~(uint32_t)(KDA_LAUNCH_PDL | KDA_LAUNCH_PDL_EARLY_STATE)) return KDA_ERR_ARG;
    if (g.h_qk < 1 || pool->hv % g.h_qk != 0 || g.num_cols < 1 || g.max_t > g.num_cols ||
        g.max_t > kda::VerifyShape<state_t, KDA_VER_BV, 2>::TC)
        return KDA_ERR_SHAPE;
    if (g.cu_seqlens == nullptr && (int64_t)g.total != (int64_t)g.n * g.max_t) return KDA_ERR_SHAPE;
    if (cv->kernel_width < 1 || cv->kernel_width > kda::DCONV_KW_MAX || win->state_len < cv->kernel_width - 1 ||
        win->state_len > kda::CONV_L_MAX || win->num_slots < 1 ||
        (int64_t)win->channels != 2LL * g.h_qk * pool->k + (int64_t)pool->hv * pool->v ||
        win->slot_stride < (int64_t)win->state_len * win->channels)
        return KDA_ERR_SHAPE;
    if (g.n == 0 || g.total == 0 || g.max_t == 0) return KDA_OK;
    if (!g.slot_table || !g.a || !g.b || !g.o || !dev_status || !win->base || !cv->conv_slot || !cv->x ||
        !cv->weight || !cv->counters)
        return KDA_ERR_NULL;
    if (!aligned(g.slot_table, 4) || !aligned(dev_status, 4) || !aligned(g.a, 4) || !aligned(g.b, 4) ||
        !aligned(g.o, 4) || (g.cu_seqlens && !aligned(g.cu_seqlens, 4)) || (g.accepted && !aligned(g.accepted, 4)) ||
        (g.a_log && !aligned(g.a_log, 4)) || (g.dt_bias && !aligned(g.dt_bias, 4)) || !aligned(win->base, es) ||
        !aligned(cv->x, es) || (cv->y && !aligned(cv->y, es)) || !aligned(cv->conv_slot, 4) ||
        !aligned(cv->weight, 4) || (cv->bias && !aligned(cv->bias, 4)) || !aligned(cv->counters, 4))
        return KDA_ERR_ALIGN;
    kda::StepParams prm = make_params(pool, g.slot_table, g.slot_table, g.reset, g.n, g.max_t, nullptr, nullptr,
                                      nullptr, g.a, g.b, g.o, dev_status, flags);
    prm.hqk = g.h_qk;
    prm.init_stride = g.num_cols;
    prm.snap_stride = g.num_cols;
    prm.num_cols = g.num_cols;
    prm.accepted = g.accepted;
    prm.cu = g.cu_seqlens;
    prm.total = g.total;
    prm.a_log = g.a_log;
    prm.dt_bias = g.dt_bias;
    prm.mode = kda::MODE_PADDING;
    prm.conv.window = win->base;
    prm.conv.num_slots = win->num_slots;
    prm.conv.slot_stride = win->slot_stride;
    prm.conv.C = win->channels;
    prm.conv.L = win->state_len;
    prm.conv.KW = cv->kernel_width;
    prm.conv.silu = cv->activation;
    prm.conv.slot = cv->conv_slot;
    prm.conv.x = cv->x;
    prm.conv.w = cv->weight;
    prm.conv.bias = cv->bias;
    prm.conv.y = cv->y;
    prm.conv.counters = cv->counters;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (win->dtype) {
        case KDA_F32: return launch_verify<float, true>(pool, prm, st);
        case KDA_F16: return launch_verify<__half, true>(pool, prm, st);
        default: return launch_verify<__nv_bfloat16, true>(pool, prm, st);
    }
}

static_assert(kda::STAGE_MAX_COPIES == KDA_STAGE_MAX_COPIES, "staging copies per launch");

int kda_stage_host(const kda_host_copy* copies, int32_t n, uint32_t flags, void* stream) {
    if (n < 0 || n > KDA_STAGE_MAX_COPIES) return KDA_ERR_ARG;
    if (flags & ~(uint32_t)KDA_LAUNCH_PDL) return KDA_ERR_ARG;
    if (n == 0) return KDA_OK;
    if (copies == nullptr) return KDA_ERR_NULL;
    kda::StageParams prm = {};
    int64_t total = 0;
    for (int32_t i = 0; i < n; ++i) {
        const kda_host_copy& c = copies[i];
        if (c.bytes < 0 || c.bytes % 16 != 0) return KDA_ERR_ARG;
        if (c.bytes > 0 && (c.dst == nullptr || c.src == nullptr)) return KDA_ERR_NULL;
        if (!aligned(c.dst, 16) || !aligned(c.src, 16)) return KDA_ERR_ALIGN;
        const void* dev_src = c.src;
        if (c.bytes > 0) {
            // the source: pinned host memory the device can address; the
            // destination: device memory
            cudaPointerAttributes a;
            if (cudaPointerGetAttributes(&a, c.src) != cudaSuccess || a.type != cudaMemoryTypeHost ||
                a.devicePointer == nullptr) {
                cudaGetLastError();  // clear the error an unregistered pointer may leave
                return KDA_ERR_ARG;
            }
            dev_src = a.devicePointer;
            if (cudaPointerGetAttributes(&a, c.dst) != cudaSuccess || a.type != cudaMemoryTypeDevice) {
                cudaGetLastError();
                return KDA_ERR_ARG;
            }
            if (!aligned(dev_src, 16)) return KDA_ERR_ALIGN;
        }
        prm.dst[i] = static_cast<uint4*>(c.dst);
        prm.src[i] = static_cast<const uint4*>(dev_src);
        total += c.bytes / 16;
        prm.end[i] = total;
    }
    prm.n = n;
    prm.flags = flags;
    if (total == 0) return KDA_OK;
    const int64_t blocks = (total + kda::STAGE_THREADS - 1) / kda::STAGE_THREADS;
    if (blocks > 0x7fffffffLL) return KDA_ERR_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(kda::STAGE_THREADS, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    set_pdl(cfg, &attr, flags);
    return cudaLaunchKernelEx(&cfg, kda::kda_stage_kernel, prm) == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

uint32_t kda_layout_id(const kda_pool* pool) {
    if (pool == nullptr) return 0u;
    const int32_t words[5] = {1, pool->dtype, pool->hv, pool->k, pool->v};
    uint32_t h = 2166136261u;  // FNV-1a, 32-bit
    for (int32_t w : words)
        for (int b = 0; b < 4; ++b) {
            h ^= (uint32_t)((uint32_t)w >> (8 * b)) & 0xffu;
            h *= 16777619u;
        }
    return h;
}

}  // extern "C"

namespace {

int ckpt_transfer(const kda_pool* pool, const kda_ckpt_plane* plane, const int32_t* slots,
                  const int32_t* entries, int32_t n, int32_t* dev_status, uint32_t flags, void* stream,
                  int load) {
    int rc = check_pool_for_build(pool);
    if (rc != KDA_OK) return rc;
    if (plane == nullptr) return KDA_ERR_NULL;
    if (n < 0 || plane->reserved != 0) return KDA_ERR_ARG;
    if (flags & ~(uint32_t)(KDA_LAUNCH_PDL | KDA_LAUNCH_PDL_EARLY_STATE)) return KDA_ERR_ARG;
    if (plane->layout_id != kda_layout_id(pool)) return KDA_ERR_LAYOUT;
    const int es = elem_size(pool->dtype);
    const int64_t state = (int64_t)pool->hv * pool->k * pool->v;
    if (plane->num_entries < 1 || plane->entry_stride < state) return KDA_ERR_SHAPE;
    if (n == 0) return KDA_OK;
    if (!plane->base || !slots || !entries || !dev_status) return KDA_ERR_NULL;
    if (!aligned(plane->base, 16) || (plane->entry_stride * es) % 16 != 0 || !aligned(slots, 4) ||
        !aligned(entries, 4) || !aligned(dev_status, 4))
        return KDA_ERR_ALIGN;
    kda::CkptParams prm;
    prm.pool = static_cast<char*>(pool->base);
    prm.num_slots = pool->num_slots;
    prm.slot_bytes = pool->slot_stride * es;
    prm.plane = static_cast<char*>(plane->base);
    prm.num_entries = plane->num_entries;
    prm.entry_bytes = plane->entry_stride * es;
    prm.state_bytes = state * es;
    prm.n = n;
    prm.slots = slots;
    prm.entries = entries;
    prm.load = load;
    prm.status = dev_status;
    const int64_t pieces = (prm.state_bytes + kda::CKPT_PIECE - 1) / kda::CKPT_PIECE;
    if (pieces * n > 0x7fffffffLL) return KDA_ERR_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(pieces * n), 1, 1);
    cfg.blockDim = dim3(kda::CKPT_THREADS, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    set_pdl(cfg, &attr, flags);
    return cudaLaunchKernelEx(&cfg, kda::kda_ckpt_kernel, prm) == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int kda_ckpt_flush(const kda_pool* pool, const kda_ckpt_plane* plane, const int32_t* slots,
                   const int32_t* entries, int32_t n, int32_t* dev_status, uint32_t flags, void* stream) {
    return ckpt_transfer(pool, plane, slots, entries, n, dev_status, flags, stream, 0);
}

int kda_ckpt_load(const kda_pool* pool, const kda_ckpt_plane* plane, const int32_t* slots,
                  const int32_t* entries, int32_t n, int32_t* dev_status, uint32_t flags, void* stream) {
    return ckpt_transfer(pool, plane, slots, entries, n, dev_status, flags, stream, 1);
}

const char* kda_strerror(int32_t code) {
    switch (code) {
        case KDA_OK: return "ok";
        case KDA_ERR_NULL: return "a required pointer is NULL";
        case KDA_ERR_DTYPE_MISMATCH: return "state pool dtype differs from the library's build dtype";
        case KDA_ERR_DTYPE_UNSUPPORTED: return "unsupported dtype (state pools are fp32 or fp16 only; q/k/v fp32, fp16 or bf16)";
        case KDA_ERR_LAYERS_DISAGREE: return "layers disagree on the state dtype or head shape";
        case KDA_ERR_SHAPE: return "bad shape (K and V must be multiples of 16 in 16..128; slot stride >= hv*k*v)";
        case KDA_ERR_ALIGN: return "misaligned pointer or stride (pool, q, k, v, a 16-byte aligned; b, o, ids 4-byte)";
        case KDA_ERR_LAUNCH: return "CUDA kernel launch failed";
        case KDA_ERR_SLOT_RANGE: return "a slot id lies outside [0, num_slots); its tiles were skipped";
        case KDA_ERR_ARG: return "bad argument (on the device: an accepted column or token offsets out of range)";
        case KDA_ERR_TIMEOUT: return "a device-side pipeline wait ran out (1 s); the call's results are incomplete";
        case KDA_ERR_LAYOUT: return "the checkpoint plane was written under another state layout (dtype or shape)";
        default: return "unknown kda status code";
    }
}

}  // extern "C"
