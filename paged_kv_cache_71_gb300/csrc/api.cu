// api.cu -- the extern "C" entry points of libpkv.so: argument validation,
// launch planning (grid, pipeline depth, workspace), TMA descriptor encoding
// and dispatch to the kernel instantiations.  No entry point allocates,
// frees or synchronises device memory.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "cache_ops.cuh"
#include "decode.cuh"
#include "decode_mma.cuh"
#include "mixed.cuh"
#include "prefill.cuh"

namespace pkv {

// The kernel instantiations live in decode_{f32,bf16,fp8,i8}_s{4,8,16,32}.cu.
#define PKV_EXTERN(G_, D_, S_, KV_, QT_)                                                                    \
    extern template cudaError_t launch_paged_decode<G_, D_, S_, KV_, QT_>(                                   \
        const CUtensorMap&, const CUtensorMap&, const DecodeArgs&, int, int, size_t, cudaStream_t);
#define PKV_EXTERN_GD(S_, KV_, QT_)                                                                         \
    PKV_EXTERN(1, 64, S_, KV_, QT_) PKV_EXTERN(2, 64, S_, KV_, QT_) PKV_EXTERN(4, 64, S_, KV_, QT_)          \
    PKV_EXTERN(8, 64, S_, KV_, QT_) PKV_EXTERN(1, 128, S_, KV_, QT_) PKV_EXTERN(2, 128, S_, KV_, QT_)        \
    PKV_EXTERN(4, 128, S_, KV_, QT_) PKV_EXTERN(8, 128, S_, KV_, QT_)
#define PKV_EXTERN_ALL(KV_, QT_)                                                                            \
    PKV_EXTERN_GD(4, KV_, QT_) PKV_EXTERN_GD(8, KV_, QT_) PKV_EXTERN_GD(16, KV_, QT_) PKV_EXTERN_GD(32, KV_, QT_)
PKV_EXTERN_ALL(KvF32, KvF32)
PKV_EXTERN_ALL(KvBF16, KvBF16)
PKV_EXTERN_ALL(KvE4M3, KvBF16)
PKV_EXTERN_ALL(KvI8, KvBF16)
#undef PKV_EXTERN_ALL
#undef PKV_EXTERN_GD
#undef PKV_EXTERN
// The tensor-core form's instantiations live in decode_mma_{bf16,fp8,i8}_s{4,8,16,32}.cu.
#define PKV_EXTERN_MMA(S_, KV_, G_, HP_)                                                                    \
    extern template cudaError_t launch_paged_decode_mma<G_, S_, KV_, HP_>(                                  \
        const CUtensorMap&, const CUtensorMap&, const DecodeArgs&, int, int, size_t, cudaStream_t);
#define PKV_EXTERN_MMA_GH(S_, KV_)                                                                          \
    PKV_EXTERN_MMA(S_, KV_, 1, 1) PKV_EXTERN_MMA(S_, KV_, 2, 1) PKV_EXTERN_MMA(S_, KV_, 4, 1)                \
    PKV_EXTERN_MMA(S_, KV_, 8, 1) PKV_EXTERN_MMA(S_, KV_, 1, 2) PKV_EXTERN_MMA(S_, KV_, 2, 2)                \
    PKV_EXTERN_MMA(S_, KV_, 4, 2) PKV_EXTERN_MMA(S_, KV_, 8, 2)
#define PKV_EXTERN_MMA_ALL(KV_)                                                                             \
    PKV_EXTERN_MMA_GH(4, KV_) PKV_EXTERN_MMA_GH(8, KV_) PKV_EXTERN_MMA_GH(16, KV_) PKV_EXTERN_MMA_GH(32, KV_)
PKV_EXTERN_MMA_ALL(KvBF16)
PKV_EXTERN_MMA_ALL(KvE4M3)
PKV_EXTERN_MMA_ALL(KvI8)
#undef PKV_EXTERN_MMA_ALL
#undef PKV_EXTERN_MMA_GH
#undef PKV_EXTERN_MMA
// The mixed-step kernel's instantiations live in mixed_{bf16,fp8,i8}.cu.
#define PKV_EXTERN_MIX(N_, KV_, G_)                                                                         \
    extern template cudaError_t launch_paged_mixed<N_, G_, KV_>(const CUtensorMap&, const CUtensorMap&,        \
                                                                const CUtensorMap&, const PrefillArgs&,         \
                                                                const DecodeArgs&, const MixedArgs&, int,       \
                                                                size_t, cudaStream_t);
#define PKV_EXTERN_MIX_G(N_, KV_) PKV_EXTERN_MIX(N_, KV_, 1) PKV_EXTERN_MIX(N_, KV_, 2) PKV_EXTERN_MIX(N_, KV_, 4) PKV_EXTERN_MIX(N_, KV_, 8)
PKV_EXTERN_MIX_G(0, KvBF16)
PKV_EXTERN_MIX_G(1, KvE4M3)
PKV_EXTERN_MIX_G(2, KvI8)
#undef PKV_EXTERN_MIX_G
#undef PKV_EXTERN_MIX

// ------------------------------------------------------------------ error detail

static thread_local char g_detail[512] = "";

static pkv_status fail(pkv_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
static pkv_status fail(pkv_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
    return st;
}

void set_last_error(const char* msg) { snprintf(g_detail, sizeof g_detail, "%s", msg); }

static pkv_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ device properties

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
};

static DeviceInfo g_dev[64];
static std::mutex g_dev_mu;

static pkv_status device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev[dev].sms == 0) {
        int sms = 0, smem = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(shared memory)");
        g_dev[dev].sms = sms;
        g_dev[dev].smem_optin = smem;
    }
    *out = g_dev[dev];
    return PKV_OK;
}

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// L2 fetch size for rows of `row_bytes` contiguous bytes: the row itself, never more.  The row of the next KV head
// follows in memory, and a wider promotion fetches it from DRAM for a warp that does not need it (at 128-byte rows
// 256-byte promotion read 1.42x the bytes of an INT8 decode, the neighbour head's rows mostly evicted before use).
static CUtensorMapL2promotion promotion_for_row(uint64_t row_bytes) {
    return row_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
           : row_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                              : CU_TENSOR_MAP_L2_PROMOTION_L2_64B;
}

// A [NB*S][Hkv][D] view of one cache tensor, box = one (block, head) tile [S][1][D].
static pkv_status cache_tensor_map(CUtensorMap* map, const void* base, const pkv_cache_desc& c) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int es = c.dtype == PKV_F32 ? 4 : c.dtype == PKV_BF16 ? 2 : 1;
    const CUtensorMapDataType dt = c.dtype == PKV_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : c.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(c.head_dim), static_cast<cuuint64_t>(c.num_kv_heads),
                          static_cast<cuuint64_t>(c.num_blocks) * c.block_size};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(c.head_dim) * es,
                             static_cast<cuuint64_t>(c.num_kv_heads) * c.head_dim * es};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(c.head_dim), 1u, static_cast<cuuint32_t>(c.block_size)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, promotion_for_row(static_cast<uint64_t>(c.head_dim) * es),
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return PKV_OK;
}

// A 3-D tiled map with 128-byte swizzle; the inner box is 128 bytes (64 bf16 or 128 FP8 codes).  fetch_bytes: the L2
// promotion size (0: the inner row itself).
static pkv_status tensor_map_sw128(CUtensorMap* map, const void* base, bool fp8, uint64_t d0, uint64_t d1, uint64_t d2,
                                   uint32_t b1, uint32_t b2, uint64_t fetch_bytes = 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {d0, d1, d2};
    const uint64_t es = fp8 ? 1 : 2;
    cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
    cuuint32_t box[3] = {fp8 ? 128u : 64u, b1, b2};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     promotion_for_row(fetch_bytes ? fetch_bytes : d0 * es),
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (swizzled) failed (%d)", static_cast<int>(r));
    return PKV_OK;
}

// ------------------------------------------------------------------ validation helpers

static int elem_bytes(int dt) {
    return dt == PKV_F32 ? 4 : dt == PKV_BF16 ? 2 : (dt == PKV_FP8_E4M3 || dt == PKV_INT8) ? 1 : 0;
}
static bool narrow(int dt) { return dt == PKV_FP8_E4M3 || dt == PKV_INT8; }

static pkv_status check_cache(const pkv_cache_desc* c) {
    if (!c) return fail(PKV_ERR_INVALID_ARG, "cache descriptor is NULL");
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0)
        return fail(PKV_ERR_INVALID_ARG, "cache sizes must be positive (NB=%d S=%d Hkv=%d D=%d)", c->num_blocks,
                    c->block_size, c->num_kv_heads, c->head_dim);
    if (elem_bytes(c->dtype) == 0) return fail(PKV_ERR_INVALID_ARG, "unknown cache dtype %d", c->dtype);
    if (c->block_size != 4 && c->block_size != 8 && c->block_size != 16 && c->block_size != 32)
        return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 4, 8, 16, 32)", c->block_size);
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", c->head_dim);
    if (static_cast<int64_t>(c->num_blocks) * c->block_size > INT32_MAX)
        return fail(PKV_ERR_OUT_OF_RANGE, "num_blocks * block_size exceeds 2^31-1");
    if (narrow(c->dtype) &&
        !(c->k_scale > 0.f && c->v_scale > 0.f && c->k_scale < 3.0e38f && c->v_scale < 3.0e38f))
        return fail(PKV_ERR_INVALID_ARG, "FP8 / INT8 caches need finite positive k_scale / v_scale");
    if ((c->k_head_scales || c->v_head_scales) && !narrow(c->dtype))
        return fail(PKV_ERR_INVALID_ARG, "per-head scales apply to FP8 / INT8 caches only");
    if ((reinterpret_cast<uintptr_t>(c->k_head_scales) | reinterpret_cast<uintptr_t>(c->v_head_scales)) & 3u)
        return fail(PKV_ERR_INVALID_ARG, "per-head scale arrays must be 4-byte aligned");
    return PKV_OK;
}

static int policy_warps(int G, int D) {
    switch (G * 1000 + D) {
        case 1064: return DecodePolicy<1, 64>::warps;
        case 2064: return DecodePolicy<2, 64>::warps;
        case 4064: return DecodePolicy<4, 64>::warps;
        case 8064: return DecodePolicy<8, 64>::warps;
        case 1128: return DecodePolicy<1, 128>::warps;
        case 2128: return DecodePolicy<2, 128>::warps;
        case 4128: return DecodePolicy<4, 128>::warps;
        default: return DecodePolicy<8, 128>::warps;
    }
}

// Smallest GQA group that a bf16 cache decodes on the tensor-core form; below it the CUDA cores keep up with HBM
// (measured on GB300), at and above it their fp32 FMA issue is the limit.
#ifndef PKV_BF16_MMA_MIN_G
#define PKV_BF16_MMA_MIN_G 8
#endif
// Largest GQA group for which the tensor-core form takes two KV heads per work unit (when the head count is even).
#ifndef PKV_MMA_PAIR_MAX_G
#define PKV_MMA_PAIR_MAX_G 4
#endif

// Which decode form runs: the tensor-core form for FP8 / INT8 caches and bf16 caches from PKV_BF16_MMA_MIN_G up
// (128-dim heads), the CUDA-core form otherwise.  The shared-block form (batches whose tables share physical
// blocks, re-read from L2) takes every bf16 cache of 128-dim heads to the tensor-core form, with one KV head per
// work unit (its 8 KB stages keep 8 warps per SM; a bf16 head pair's 16 KB stages leave room for 4).
static bool uses_tensor_core(int dtype, int G, int D, bool shared = false) {
    return D == 128 && (narrow(dtype) || (dtype == PKV_BF16 && (shared || G >= PKV_BF16_MMA_MIN_G)));
}
static int mma_heads_per_unit(int G, int Hkv, int dtype, bool shared = false) {
    if (shared && dtype == PKV_BF16) return 1;
    return (G <= PKV_MMA_PAIR_MAX_G && Hkv % 2 == 0) ? 2 : 1;
}

// Split-KV scratch: one completion counter per (sequence, KV head), then two partial (O, m, l) records per worker
// warp, each over the query heads of one work unit (G, or 2G when the tensor-core form pairs KV heads).
static size_t workspace_bytes_for(int sms, int B, int Hkv, int G, int D, int dtype, bool shared = false) {
    const size_t tickets = ((static_cast<size_t>(B) * Hkv * 4 + 255) / 256) * 256;
    const bool tc = uses_tensor_core(dtype, G, D, shared);
    const size_t W = static_cast<size_t>(sms) * (tc ? kMmaWarps : policy_warps(G, D));
    const size_t rows = static_cast<size_t>(G) * (tc ? mma_heads_per_unit(G, Hkv, dtype, shared) : 1);
    return tickets + W * 2 * rows * (D + 2) * 4;
}

template <int D, int S, class KV, class QT>
static cudaError_t dispatch_g(int G, const CUtensorMap& km, const CUtensorMap& vm, const DecodeArgs& a, int grid,
                              int block, size_t smem, cudaStream_t s) {
    switch (G) {
        case 1: return launch_paged_decode<1, D, S, KV, QT>(km, vm, a, grid, block, smem, s);
        case 2: return launch_paged_decode<2, D, S, KV, QT>(km, vm, a, grid, block, smem, s);
        case 4: return launch_paged_decode<4, D, S, KV, QT>(km, vm, a, grid, block, smem, s);
        case 8: return launch_paged_decode<8, D, S, KV, QT>(km, vm, a, grid, block, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int S, class KV, class QT>
static cudaError_t dispatch_d(int D, int G, const CUtensorMap& km, const CUtensorMap& vm, const DecodeArgs& a,
                              int grid, int block, size_t smem, cudaStream_t s) {
    if (D == 64) return dispatch_g<64, S, KV, QT>(G, km, vm, a, grid, block, smem, s);
    return dispatch_g<128, S, KV, QT>(G, km, vm, a, grid, block, smem, s);
}

template <class KV, class QT>
static cudaError_t dispatch_s(int S, int D, int G, const CUtensorMap& km, const CUtensorMap& vm, const DecodeArgs& a,
                              int grid, int block, size_t smem, cudaStream_t s) {
    switch (S) {
        case 4: return dispatch_d<4, KV, QT>(D, G, km, vm, a, grid, block, smem, s);
        case 8: return dispatch_d<8, KV, QT>(D, G, km, vm, a, grid, block, smem, s);
        case 16: return dispatch_d<16, KV, QT>(D, G, km, vm, a, grid, block, smem, s);
        case 32: return dispatch_d<32, KV, QT>(D, G, km, vm, a, grid, block, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv

#define PKV_API extern "C" __attribute__((visibility("default")))

using namespace pkv;

// ------------------------------------------------------------------ entry points

PKV_API const char* pkv_status_string(pkv_status st) {
    switch (st) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_OUT_OF_RANGE: return "PKV_ERR_OUT_OF_RANGE";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    }
    return "PKV_ERR_UNKNOWN";
}

PKV_API const char* pkv_last_error(void) { return g_detail; }

PKV_API int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

PKV_API pkv_status pkv_reshape_and_cache(const void* k_new, const void* v_new, int32_t src_dtype,
                                         const int64_t* slot_mapping, int32_t num_tokens, void* k_cache,
                                         void* v_cache, const pkv_cache_desc* cache, int32_t* device_error,
                                         void* stream) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
        return fail(PKV_ERR_INVALID_ARG, "null tensor pointer");
    if (src_dtype != PKV_F32 && src_dtype != PKV_BF16)
        return fail(PKV_ERR_UNSUPPORTED, "source dtype %d (supported: f32, bf16)", src_dtype);
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PKV_ERR_INVALID_ARG, "k_new, v_new and the caches must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return fail(PKV_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
    DeviceInfo di;
    if ((st = device_info(&di)) != PKV_OK) return st;
    const int64_t pool_slots = static_cast<int64_t>(cache->num_blocks) * cache->block_size;
    const int row = cache->num_kv_heads * cache->head_dim;
    cudaError_t e = launch_reshape_and_cache(k_new, v_new, src_dtype, slot_mapping, num_tokens, k_cache, v_cache,
                                             cache->dtype, pool_slots, row, cache->head_dim, cache->k_scale,
                                             cache->v_scale, cache->k_head_scales, cache->v_head_scales,
                                             device_error, di.sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
    return PKV_OK;
}

PKV_API pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                   const int64_t* block_mapping, int32_t num_pairs, int32_t* device_error,
                                   void* stream) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return fail(PKV_ERR_INVALID_ARG, "num_pairs %d < 0", num_pairs);
    if (num_pairs == 0) return PKV_OK;
    // one CTA per (pair, tensor): the grid of 2 * num_pairs CTAs must stay below 2^31
    if (num_pairs >= (1 << 30)) return fail(PKV_ERR_OUT_OF_RANGE, "num_pairs %d >= 2^30", num_pairs);
    if (!k_cache || !v_cache || !block_mapping) return fail(PKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(PKV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(block_mapping) & 7u) != 0)
        return fail(PKV_ERR_INVALID_ARG, "block_mapping must be 8-byte aligned");
    const int64_t block_bytes = static_cast<int64_t>(cache->block_size) * cache->num_kv_heads * cache->head_dim *
                                elem_bytes(cache->dtype);
    cudaError_t e = launch_copy_blocks(k_cache, v_cache, block_mapping, num_pairs, cache->num_blocks, block_bytes,
                                       device_error, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
    return PKV_OK;
}

// True when the device can dereference p (device, managed or mapped host memory, or any host
// memory on a device with pageable-memory access such as a Grace-attached GPU).
static bool device_accessible(const void* p, int dev) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return true;
    if (at.type == cudaMemoryTypeHost) return at.devicePointer == p;
    int pageable = 0;
    cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
    return pageable != 0;
}

PKV_API pkv_status pkv_swap_blocks(const void* src_k, const void* src_v, int32_t src_num_blocks, void* dst_k,
                                   void* dst_v, int32_t dst_num_blocks, const pkv_cache_desc* cache,
                                   const int64_t* block_mapping, int32_t num_pairs, int32_t* device_error,
                                   void* stream) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes (num_pairs=%d src_num_blocks=%d dst_num_blocks=%d)", num_pairs,
                    src_num_blocks, dst_num_blocks);
    if (num_pairs == 0) return PKV_OK;
    if (num_pairs >= (1 << 30)) return fail(PKV_ERR_OUT_OF_RANGE, "num_pairs %d >= 2^30", num_pairs);
    if (!src_k || !src_v || !dst_k || !dst_v || !block_mapping) return fail(PKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
        return fail(PKV_ERR_INVALID_ARG, "pools must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(block_mapping) & 7u) != 0)
        return fail(PKV_ERR_INVALID_ARG, "block_mapping must be 8-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const void* ptrs[5] = {src_k, src_v, dst_k, dst_v, block_mapping};
    for (const void* p : ptrs)
        if (!device_accessible(p, dev))
            return fail(PKV_ERR_INVALID_ARG, "pointer %p is not accessible from the device (pin or register it)", p);
    const int64_t block_bytes = static_cast<int64_t>(cache->block_size) * cache->num_kv_heads * cache->head_dim *
                                elem_bytes(cache->dtype);
    e = launch_swap_blocks(src_k, src_v, src_num_blocks, dst_k, dst_v, dst_num_blocks, block_mapping, num_pairs,
                           block_bytes, device_error, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "swap_blocks launch");
    return PKV_OK;
}

PKV_API pkv_status pkv_block_hashes(const int32_t* token_ids, const int64_t* cu_tokens, int32_t num_seqs,
                                    int32_t block_size, const int64_t* out_offsets, uint64_t* hashes,
                                    int64_t hashes_capacity, int32_t* device_error, void* stream) {
    g_detail[0] = 0;
    if (num_seqs < 0 || block_size <= 0 || hashes_capacity < 0)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes (num_seqs=%d block_size=%d capacity=%lld)", num_seqs, block_size,
                    static_cast<long long>(hashes_capacity));
    if (num_seqs == 0) return PKV_OK;
    if (!token_ids || !cu_tokens || !out_offsets || !hashes) return fail(PKV_ERR_INVALID_ARG, "null pointer");
    if ((reinterpret_cast<uintptr_t>(cu_tokens) & 7u) || (reinterpret_cast<uintptr_t>(out_offsets) & 7u) ||
        (reinterpret_cast<uintptr_t>(hashes) & 7u) || (reinterpret_cast<uintptr_t>(token_ids) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "misaligned pointer");
    DeviceInfo di;
    pkv_status st = device_info(&di);
    if (st != PKV_OK) return st;
    cudaError_t e = launch_block_hashes(token_ids, cu_tokens, num_seqs, block_size, out_offsets, hashes,
                                        hashes_capacity, device_error, di.sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "block_hashes launch");
    return PKV_OK;
}

template <class KV>
static cudaError_t dispatch_mma(int S, int G, int HP, const CUtensorMap& km, const CUtensorMap& vm,
                                const DecodeArgs& a, int grid, int block, size_t smem, cudaStream_t s) {
#define PKV_MMA_G(S_)                                                                                         \
    switch (G * 10 + HP) {                                                                                    \
        case 11: return launch_paged_decode_mma<1, S_, KV, 1>(km, vm, a, grid, block, smem, s);               \
        case 21: return launch_paged_decode_mma<2, S_, KV, 1>(km, vm, a, grid, block, smem, s);               \
        case 41: return launch_paged_decode_mma<4, S_, KV, 1>(km, vm, a, grid, block, smem, s);               \
        case 81: return launch_paged_decode_mma<8, S_, KV, 1>(km, vm, a, grid, block, smem, s);               \
        case 12: return launch_paged_decode_mma<1, S_, KV, 2>(km, vm, a, grid, block, smem, s);               \
        case 22: return launch_paged_decode_mma<2, S_, KV, 2>(km, vm, a, grid, block, smem, s);               \
        case 42: return launch_paged_decode_mma<4, S_, KV, 2>(km, vm, a, grid, block, smem, s);               \
        case 82: return launch_paged_decode_mma<8, S_, KV, 2>(km, vm, a, grid, block, smem, s);               \
        default: return cudaErrorInvalidValue;                                                                \
    }
    switch (S) {
        case 4: PKV_MMA_G(4)
        case 8: PKV_MMA_G(8)
        case 16: PKV_MMA_G(16)
        case 32: PKV_MMA_G(32)
        default: return cudaErrorInvalidValue;
    }
#undef PKV_MMA_G
}

// Decode on the tensor-core form of the kernel (decode_mma.cuh): FP8 / INT8 caches, and bf16 caches from
// PKV_BF16_MMA_MIN_G up, 128-dim heads.  Its stages hold 128-byte swizzled K and V tiles only (two 64-dim halves per
// bf16 row), each half starting on a 1024-byte boundary; `a` arrives with everything but the shared-memory plan.
static pkv_status decode_tensor_core(DecodeArgs a, const pkv_cache_desc& c, int G, int num_seqs, const void* k_cache,
                                     const void* v_cache, const DeviceInfo& di, bool shared, cudaStream_t s) {
    const int S = c.block_size, Hkv = c.num_kv_heads;
    const bool b16 = c.dtype == PKV_BF16;
    const int HP = mma_heads_per_unit(G, Hkv, c.dtype, shared);  // KV heads per work unit
    const uint32_t tile = static_cast<uint32_t>((b16 ? 2 : 1) * std::max(S * 128, 1024));
    a.kv_bytes = static_cast<uint32_t>(S * 128 * (b16 ? 2 : 1));  // one K (or V) tile of one head
    a.q_bytes = 0;  // the query rows are read straight into registers
    a.stage_bytes = 2 * HP * tile;
    a.prefix_bytes = static_cast<uint32_t>(((static_cast<size_t>(num_seqs) + 1) * 4 + 1023) / 1024 * 1024);
    const size_t budget = static_cast<size_t>(di.smem_optin) - 256 - 1024;  // static shared memory, alignment slack
    int nw = kMmaWarps, depth = 0;
    while (nw >= 1) {
        const size_t avail = budget > a.prefix_bytes ? budget - a.prefix_bytes : 0;
        const size_t per_warp_avail = avail / nw;
        depth = 6;  // the deepest pipeline whose region, rounded to 1024 bytes, fits
        while (depth >= 2 && (static_cast<size_t>(depth) * a.stage_bytes + 8 * depth + 1023) / 1024 * 1024 > per_warp_avail)
            --depth;
        if (depth >= 2) break;
        nw >>= 1;
    }
    if (depth < 2) return fail(PKV_ERR_UNSUPPORTED, "shared memory too small for this block size and batch");
    a.depth = depth;
    a.warp_bytes = static_cast<uint32_t>((static_cast<size_t>(depth) * a.stage_bytes + 8 * depth + 1023) / 1024 * 1024);
    const size_t smem = a.prefix_bytes + static_cast<size_t>(nw) * a.warp_bytes + 1024;
    const uint64_t rows = static_cast<uint64_t>(c.num_blocks) * S;
    CUtensorMap km, vm;
    pkv_status st;
    // a unit's HP heads are read together, so a one-byte row pair (256 contiguous bytes) is fetched as one
    const uint64_t fetch = static_cast<uint64_t>(b16 ? 256 : 128 * HP);
    if ((st = tensor_map_sw128(&km, k_cache, !b16, 128, Hkv, rows, 1, S, fetch)) != PKV_OK) return st;
    if ((st = tensor_map_sw128(&vm, v_cache, !b16, 128, Hkv, rows, 1, S, fetch)) != PKV_OK) return st;
    if (a.tickets) {
        cudaError_t e = cudaMemsetAsync(a.tickets, 0, static_cast<size_t>(num_seqs) * Hkv * 4, s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing split-KV counters");
    }
    const cudaError_t e =
        b16                       ? dispatch_mma<KvBF16>(S, G, HP, km, vm, a, di.sms, nw * 32, smem, s)
        : c.dtype == PKV_FP8_E4M3 ? dispatch_mma<KvE4M3>(S, G, HP, km, vm, a, di.sms, nw * 32, smem, s)
                                  : dispatch_mma<KvI8>(S, G, HP, km, vm, a, di.sms, nw * 32, smem, s);
    if (e != cudaSuccess) return cuda_fail(e, "paged_attention_decode launch");
    return PKV_OK;
}

PKV_API pkv_status pkv_paged_attention_workspace_size(const pkv_cache_desc* cache, int32_t num_seqs,
                                                      int32_t num_q_heads, int32_t num_splits, size_t* bytes) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (!bytes) return fail(PKV_ERR_INVALID_ARG, "bytes is NULL");
    if (num_seqs < 0 || num_q_heads <= 0 || num_splits < 0)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes (num_seqs=%d num_q_heads=%d num_splits=%d)", num_seqs,
                    num_q_heads, num_splits);
    if (num_q_heads % cache->num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads,
                    cache->num_kv_heads);
    if (num_splits == 1) {
        *bytes = 0;
        return PKV_OK;
    }
    DeviceInfo di;
    if ((st = device_info(&di)) != PKV_OK) return st;
    *bytes = workspace_bytes_for(di.sms, num_seqs, cache->num_kv_heads, num_q_heads / cache->num_kv_heads,
                                 cache->head_dim, cache->dtype);
    return PKV_OK;
}

// The decode entry points: `shared` selects the shared-block form (pkv_paged_attention_decode_shared).
static pkv_status decode_entry(void* out, const void* q, int32_t q_dtype, const void* k_cache, const void* v_cache,
                               const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, float scale,
                               int32_t num_splits, int32_t max_context_len, void* workspace, size_t workspace_bytes,
                               int32_t* device_error, void* stream, bool shared) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    const int Hkv = cache->num_kv_heads, D = cache->head_dim, S = cache->block_size;
    if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_splits < 0 || max_context_len < 0)
        return fail(PKV_ERR_INVALID_ARG,
                    "bad sizes (num_seqs=%d num_q_heads=%d max_blocks_per_seq=%d num_splits=%d max_context_len=%d)",
                    num_seqs, num_q_heads, max_blocks_per_seq, num_splits, max_context_len);
    if (num_q_heads % Hkv != 0)
        return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads, Hkv);
    const int G = num_q_heads / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PKV_ERR_UNSUPPORTED, "GQA group size %d (supported: 1, 2, 4, 8)", G);
    if (num_seqs > 8192) return fail(PKV_ERR_UNSUPPORTED, "num_seqs %d > 8192", num_seqs);
    if (Hkv > 1024) return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads %d > 1024", Hkv);
    if (static_cast<int64_t>(num_seqs) * max_blocks_per_seq * Hkv > INT32_MAX - 64)
        return fail(PKV_ERR_OUT_OF_RANGE, "num_seqs * max_blocks_per_seq * num_kv_heads must stay below 2^31");
    if (!(scale == scale) || scale == 0.f) return fail(PKV_ERR_INVALID_ARG, "scale must be finite and non-zero");
    const bool combo_ok = (q_dtype == PKV_F32 && cache->dtype == PKV_F32) ||
                          (q_dtype == PKV_BF16 && (cache->dtype == PKV_BF16 || narrow(cache->dtype)));
    if (!combo_ok)
        return fail(PKV_ERR_UNSUPPORTED, "q dtype %d with cache dtype %d (supported: f32/f32, bf16/bf16|fp8|int8)",
                    q_dtype, cache->dtype);
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PKV_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PKV_ERR_INVALID_ARG, "q, out and the caches must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "block_tables / context_lens must be 4-byte aligned");

    DeviceInfo di;
    if ((st = device_info(&di)) != PKV_OK) return st;

    // ---- work split
    int part_blocks;
    if (num_splits == 0) {
        part_blocks = 1;
    } else if (num_splits == 1) {
        part_blocks = 1 << 30;
    } else {
        const int64_t maxlen = max_context_len > 0 ? max_context_len : static_cast<int64_t>(max_blocks_per_seq) * S;
        const int64_t mb = (maxlen + S - 1) / S;
        part_blocks = static_cast<int>(std::max<int64_t>(1, (mb + num_splits - 1) / num_splits));
    }
    int32_t* tickets = nullptr;
    float* partials = nullptr;
    if (num_splits != 1) {
        const size_t need = workspace_bytes_for(di.sms, num_seqs, Hkv, G, D, cache->dtype, shared);
        if (!workspace || workspace_bytes < need)
            return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                        workspace ? workspace_bytes : static_cast<size_t>(0));
        if (!aligned16(workspace)) return fail(PKV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
        tickets = static_cast<int32_t*>(workspace);
        const size_t tb = ((static_cast<size_t>(num_seqs) * Hkv * 4 + 255) / 256) * 256;
        partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + tb);
    }

    // ---- shared-memory plan
    const int kv_es = elem_bytes(cache->dtype), q_es = elem_bytes(q_dtype);
    DecodeArgs a;
    a.out = out;
    a.q = q;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.tickets = tickets;
    a.partials = partials;
    a.err = device_error;
    a.B = num_seqs;
    a.Hq = num_q_heads;
    a.Hkv = Hkv;
    a.S = S;
    a.MB = max_blocks_per_seq;
    a.NB = cache->num_blocks;
    a.part_blocks = part_blocks;
    const float kLog2e = 1.4426950408889634f;
    a.q_mul = scale * kLog2e * (narrow(cache->dtype) ? cache->k_scale : 1.f);
    a.o_mul = narrow(cache->dtype) ? cache->v_scale : 1.f;
    a.q_base = scale * kLog2e;
    a.k_head = cache->k_head_scales;
    a.v_head = cache->v_head_scales;
    a.kv_bytes = static_cast<uint32_t>(S * D * kv_es);
    a.q_bytes = static_cast<uint32_t>(G * D * q_es);
    a.stage_bytes = ((2 * a.kv_bytes + a.q_bytes + 127) / 128) * 128;
    a.prefix_bytes = static_cast<uint32_t>(((static_cast<size_t>(num_seqs) + 1) * 4 + 127) / 128 * 128);
    a.timeout_ns = 2000000000ull;
    if (uses_tensor_core(cache->dtype, G, D, shared))
        return decode_tensor_core(a, *cache, G, num_seqs, k_cache, v_cache, di, shared,
                                  static_cast<cudaStream_t>(stream));
    const size_t budget = static_cast<size_t>(di.smem_optin) - 256;  // static shared memory of the kernel
    int nw = policy_warps(G, D), depth = 0;
    while (nw >= 1) {
        const size_t fixed = 16 * G * 8 + G * 8 + 8 * 8;  // pbuf, abuf, up to 8 barriers
        const size_t avail = budget > a.prefix_bytes ? budget - a.prefix_bytes : 0;
        const size_t per_warp_avail = avail / nw;
        depth = per_warp_avail > fixed ? static_cast<int>((per_warp_avail - fixed) / a.stage_bytes) : 0;
        if (depth > 6) depth = 6;
        if (depth >= 2) break;
        nw >>= 1;
    }
    if (depth < 2) return fail(PKV_ERR_UNSUPPORTED, "shared memory too small for this block/head size");
    a.depth = depth;
    const size_t fixed = 16 * G * 8 + G * 8 + 8 * static_cast<size_t>(depth);
    a.warp_bytes = static_cast<uint32_t>(((static_cast<size_t>(depth) * a.stage_bytes + fixed + 127) / 128) * 128);
    const size_t smem = a.prefix_bytes + static_cast<size_t>(nw) * a.warp_bytes;

    CUtensorMap km, vm;
    if ((st = cache_tensor_map(&km, k_cache, *cache)) != PKV_OK) return st;
    if ((st = cache_tensor_map(&vm, v_cache, *cache)) != PKV_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (tickets) {
        cudaError_t e = cudaMemsetAsync(tickets, 0, static_cast<size_t>(num_seqs) * Hkv * 4, s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing split-KV counters");
    }
    cudaError_t e;
    if (cache->dtype == PKV_F32)
        e = dispatch_s<KvF32, KvF32>(S, D, G, km, vm, a, di.sms, nw * 32, smem, s);
    else if (cache->dtype == PKV_BF16)
        e = dispatch_s<KvBF16, KvBF16>(S, D, G, km, vm, a, di.sms, nw * 32, smem, s);
    else if (cache->dtype == PKV_FP8_E4M3)
        e = dispatch_s<KvE4M3, KvBF16>(S, D, G, km, vm, a, di.sms, nw * 32, smem, s);
    else
        e = dispatch_s<KvI8, KvBF16>(S, D, G, km, vm, a, di.sms, nw * 32, smem, s);
    if (e != cudaSuccess) return cuda_fail(e, "paged_attention_decode launch");
    return PKV_OK;
}

PKV_API pkv_status pkv_paged_attention_decode(void* out, const void* q, int32_t q_dtype, const void* k_cache,
                                              const void* v_cache, const pkv_cache_desc* cache,
                                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                                              const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                              float scale, int32_t num_splits, int32_t max_context_len,
                                              void* workspace, size_t workspace_bytes, int32_t* device_error,
                                              void* stream) {
    return decode_entry(out, q, q_dtype, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                        num_seqs, num_q_heads, scale, num_splits, max_context_len, workspace, workspace_bytes,
                        device_error, stream, false);
}

PKV_API pkv_status pkv_paged_attention_decode_shared(void* out, const void* q, int32_t q_dtype, const void* k_cache,
                                                     const void* v_cache, const pkv_cache_desc* cache,
                                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                     const int32_t* context_lens, int32_t num_seqs,
                                                     int32_t num_q_heads, float scale, int32_t num_splits,
                                                     int32_t max_context_len, void* workspace, size_t workspace_bytes,
                                                     int32_t* device_error, void* stream) {
    return decode_entry(out, q, q_dtype, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                        num_seqs, num_q_heads, scale, num_splits, max_context_len, workspace, workspace_bytes,
                        device_error, stream, true);
}

PKV_API pkv_status pkv_paged_prefill_chunk(void* out, const void* q, int32_t q_dtype, int32_t num_q_tokens,
                                           int32_t q_start_pos, const void* k_cache, const void* v_cache,
                                           const pkv_cache_desc* cache, const int32_t* block_table, int32_t kv_len,
                                           int32_t num_q_heads, float scale, int32_t* device_error, void* stream) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    const int Hkv = cache->num_kv_heads, D = cache->head_dim, S = cache->block_size;
    if (num_q_tokens < 0 || q_start_pos < 0 || num_q_heads <= 0 || kv_len < 0)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes (num_q_tokens=%d q_start_pos=%d num_q_heads=%d kv_len=%d)",
                    num_q_tokens, q_start_pos, num_q_heads, kv_len);
    if (static_cast<int64_t>(q_start_pos) + num_q_tokens > kv_len)
        return fail(PKV_ERR_INVALID_ARG, "kv_len %d < q_start_pos + num_q_tokens (the chunk's own keys must be cached)",
                    kv_len);
    if (num_q_heads % Hkv != 0)
        return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads, Hkv);
    const int G = num_q_heads / Hkv;
    if (q_dtype != PKV_BF16 || (cache->dtype != PKV_BF16 && !narrow(cache->dtype)))
        return fail(PKV_ERR_UNSUPPORTED, "prefill chunk supports bf16 queries with a bf16, FP8 or INT8 cache");
    const bool fp8 = narrow(cache->dtype);
    if (D != 128) return fail(PKV_ERR_UNSUPPORTED, "prefill chunk supports head_dim 128");
    if (S < 8) return fail(PKV_ERR_UNSUPPORTED, "prefill chunk supports block_size 8, 16, 32");
    if (G > 128 || 128 % G != 0) return fail(PKV_ERR_UNSUPPORTED, "GQA group %d must divide 128", G);
    if (num_q_tokens == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table) return fail(PKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PKV_ERR_INVALID_ARG, "q, out and the caches must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(block_table) & 3u) return fail(PKV_ERR_INVALID_ARG, "block_table alignment");
    if (!(scale > 0.f && scale < 3.0e38f)) return fail(PKV_ERR_INVALID_ARG, "scale must be finite and positive");
    DeviceInfo di;
    if ((st = device_info(&di)) != PKV_OK) return st;
    CUtensorMap qm, km, vm;
    if ((st = tensor_map_sw128(&qm, q, false, 128, num_q_heads, num_q_tokens, G, 128 / G)) != PKV_OK) return st;
    const uint64_t rows = static_cast<uint64_t>(cache->num_blocks) * S;
    if ((st = tensor_map_sw128(&km, k_cache, fp8, 128, Hkv, rows, 1, S)) != PKV_OK) return st;
    if ((st = tensor_map_sw128(&vm, v_cache, fp8, 128, Hkv, rows, 1, S)) != PKV_OK) return st;
    PrefillArgs a;
    a.out = out;
    a.block_table = block_table;
    a.err = device_error;
    a.NQ = num_q_tokens;
    a.q_start = q_start_pos;
    a.kv_len = kv_len;
    a.Hq = num_q_heads;
    a.Hkv = Hkv;
    a.G = G;
    a.S = S;
    a.NB = cache->num_blocks;
    a.n_table = (kv_len + S - 1) / S;
    a.sm_log2 = scale * 1.4426950408889634f * (fp8 ? cache->k_scale : 1.f);
    a.out_mul = fp8 ? cache->v_scale : 1.f;
    a.sm_base = scale * 1.4426950408889634f;
    a.k_head = cache->k_head_scales;
    a.v_head = cache->v_head_scales;
    a.timeout_ns = 2000000000ull;
    const int nk = cache->dtype == PKV_INT8 ? 2 : fp8 ? 1 : 0;
    if (static_cast<size_t>(di.smem_optin) < prefill_ws_smem_bytes(nk))
        return fail(PKV_ERR_UNSUPPORTED, "device shared memory too small for the prefill tile");
    cudaError_t e = launch_paged_prefill_ws(qm, km, vm, a, nk, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged_prefill_chunk launch");
    return PKV_OK;
}

PKV_API pkv_status pkv_paged_prefill_varlen(void* out, const void* q, int32_t q_dtype, int32_t total_q_tokens,
                                            const int32_t* cu_q, const int32_t* q_starts, const int32_t* kv_lens,
                                            const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                                            int32_t num_seqs, int32_t num_q_heads, float scale,
                                            int32_t* device_error, void* stream) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    const int Hkv = cache->num_kv_heads, D = cache->head_dim, S = cache->block_size;
    if (total_q_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes (total_q_tokens=%d num_seqs=%d num_q_heads=%d MB=%d)",
                    total_q_tokens, num_seqs, num_q_heads, max_blocks_per_seq);
    if (num_q_heads % Hkv != 0)
        return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads, Hkv);
    const int G = num_q_heads / Hkv;
    if (q_dtype != PKV_BF16 || (cache->dtype != PKV_BF16 && !narrow(cache->dtype)))
        return fail(PKV_ERR_UNSUPPORTED, "varlen prefill supports bf16 queries with a bf16, FP8 or INT8 cache");
    const bool fp8 = narrow(cache->dtype);
    const int nk = cache->dtype == PKV_INT8 ? 2 : fp8 ? 1 : 0;
    if (D != 128) return fail(PKV_ERR_UNSUPPORTED, "prefill supports head_dim 128");
    if (S < 8) return fail(PKV_ERR_UNSUPPORTED, "prefill supports block_size 8, 16, 32");
    if (G > 128 || 128 % G != 0) return fail(PKV_ERR_UNSUPPORTED, "GQA group %d must divide 128", G);
    if (num_seqs > prefill_ws_max_seqs())
        return fail(PKV_ERR_UNSUPPORTED, "num_seqs %d > %d chunks per call", num_seqs, prefill_ws_max_seqs());
    if (static_cast<int64_t>(num_seqs) * max_blocks_per_seq > INT32_MAX)
        return fail(PKV_ERR_OUT_OF_RANGE, "block table larger than 2^31-1 entries");
    if (num_seqs == 0 || total_q_tokens == 0) return PKV_OK;
    if (!out || !q || !cu_q || !q_starts || !kv_lens || !k_cache || !v_cache || !block_tables)
        return fail(PKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PKV_ERR_INVALID_ARG, "q, out and the caches must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(cu_q) | reinterpret_cast<uintptr_t>(q_starts) |
         reinterpret_cast<uintptr_t>(kv_lens) | reinterpret_cast<uintptr_t>(block_tables)) & 3u)
        return fail(PKV_ERR_INVALID_ARG, "index arrays must be 4-byte aligned");
    if (!(scale > 0.f && scale < 3.0e38f)) return fail(PKV_ERR_INVALID_ARG, "scale must be finite and positive");
    DeviceInfo di;
    if ((st = device_info(&di)) != PKV_OK) return st;
    if (static_cast<size_t>(di.smem_optin) < prefill_ws_smem_bytes(nk))
        return fail(PKV_ERR_UNSUPPORTED, "device shared memory too small for the prefill tile");
    CUtensorMap qm, km, vm;
    if ((st = tensor_map_sw128(&qm, q, false, 128, num_q_heads, total_q_tokens, G, 128 / G)) != PKV_OK) return st;
    const uint64_t rows = static_cast<uint64_t>(cache->num_blocks) * S;
    if ((st = tensor_map_sw128(&km, k_cache, fp8, 128, Hkv, rows, 1, S)) != PKV_OK) return st;
    if ((st = tensor_map_sw128(&vm, v_cache, fp8, 128, Hkv, rows, 1, S)) != PKV_OK) return st;
    PrefillArgs a;
    a.out = out;
    a.block_table = block_tables;
    a.err = device_error;
    a.NQ = total_q_tokens;
    a.q_start = 0;
    a.kv_len = 0;
    a.Hq = num_q_heads;
    a.Hkv = Hkv;
    a.G = G;
    a.S = S;
    a.NB = cache->num_blocks;
    a.n_table = max_blocks_per_seq;
    a.sm_log2 = scale * 1.4426950408889634f * (fp8 ? cache->k_scale : 1.f);
    a.out_mul = fp8 ? cache->v_scale : 1.f;
    a.sm_base = scale * 1.4426950408889634f;
    a.k_head = cache->k_head_scales;
    a.v_head = cache->v_head_scales;
    a.timeout_ns = 2000000000ull;
    a.nseq = num_seqs;
    a.MB = max_blocks_per_seq;
    a.cu_q = cu_q;
    a.q_starts = q_starts;
    a.kv_lens = kv_lens;
    cudaError_t e = launch_paged_prefill_ws(qm, km, vm, a, nk, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged_prefill_varlen launch");
    return PKV_OK;
}

// ------------------------------------------------------------------ mixed step

// Split-KV scratch of the mixed step's decode: one completion counter per (decode token, KV head), then two partial
// records per worker warp (8 per SM, one KV head per work unit).
static size_t mixed_workspace_bytes(int sms, int num_decode, int Hkv, int G) {
    if (num_decode == 0) return 0;
    const size_t tickets = ((static_cast<size_t>(num_decode) * Hkv * 4 + 255) / 256) * 256;
    return tickets + static_cast<size_t>(sms) * kMmaWarps * 2 * G * (128 + 2) * 4;
}

PKV_API pkv_status pkv_paged_attention_mixed_workspace_size(const pkv_cache_desc* cache, int32_t num_decode,
                                                            int32_t num_q_heads, size_t* bytes) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (!bytes) return fail(PKV_ERR_INVALID_ARG, "bytes is NULL");
    if (num_decode < 0 || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes (num_decode=%d num_q_heads=%d)", num_decode, num_q_heads);
    DeviceInfo di;
    if ((st = device_info(&di)) != PKV_OK) return st;
    *bytes = mixed_workspace_bytes(di.sms, num_decode, cache->num_kv_heads, num_q_heads / cache->num_kv_heads);
    return PKV_OK;
}

template <int N, class KV>
static cudaError_t dispatch_mixed(int G, const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                                  const PrefillArgs& pa, const DecodeArgs& da, const MixedArgs& ma, int grid,
                                  size_t smem, cudaStream_t s) {
    switch (G) {
        case 1: return launch_paged_mixed<N, 1, KV>(qm, km, vm, pa, da, ma, grid, smem, s);
        case 2: return launch_paged_mixed<N, 2, KV>(qm, km, vm, pa, da, ma, grid, smem, s);
        case 4: return launch_paged_mixed<N, 4, KV>(qm, km, vm, pa, da, ma, grid, smem, s);
        case 8: return launch_paged_mixed<N, 8, KV>(qm, km, vm, pa, da, ma, grid, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

PKV_API pkv_status pkv_paged_attention_mixed(void* out, const void* q, int32_t q_dtype, int32_t total_q_tokens,
                                             const int32_t* cu_q, const int32_t* q_starts, const int32_t* kv_lens,
                                             const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                                             int32_t num_seqs, int32_t num_decode, int32_t num_q_heads, float scale,
                                             void* workspace, size_t workspace_bytes, int32_t* device_error,
                                             void* stream) {
    g_detail[0] = 0;
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    const int Hkv = cache->num_kv_heads, D = cache->head_dim, S = cache->block_size;
    if (total_q_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_decode < 0 ||
        num_decode > num_seqs || num_decode > total_q_tokens)
        return fail(PKV_ERR_INVALID_ARG,
                    "bad sizes (total_q_tokens=%d num_seqs=%d num_decode=%d num_q_heads=%d max_blocks_per_seq=%d)",
                    total_q_tokens, num_seqs, num_decode, num_q_heads, max_blocks_per_seq);
    if (num_q_heads % Hkv != 0)
        return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads, Hkv);
    const int G = num_q_heads / Hkv;
    if (q_dtype != PKV_BF16 || (cache->dtype != PKV_BF16 && !narrow(cache->dtype)))
        return fail(PKV_ERR_UNSUPPORTED, "the mixed step supports bf16 queries with a bf16, FP8 or INT8 cache");
    if (D != 128 || S != 16) return fail(PKV_ERR_UNSUPPORTED, "the mixed step supports head_dim 128, block_size 16");
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PKV_ERR_UNSUPPORTED, "GQA group size %d (supported: 1, 2, 4, 8)", G);
    if (num_seqs > prefill_ws_max_seqs())
        return fail(PKV_ERR_UNSUPPORTED, "num_seqs %d > %d chunks per call", num_seqs, prefill_ws_max_seqs());
    if (num_decode > 8192) return fail(PKV_ERR_UNSUPPORTED, "num_decode %d > 8192", num_decode);
    if (static_cast<int64_t>(num_seqs) * max_blocks_per_seq * Hkv > INT32_MAX - 64)
        return fail(PKV_ERR_OUT_OF_RANGE, "num_seqs * max_blocks_per_seq * num_kv_heads must stay below 2^31");
    if (num_seqs == 0 || total_q_tokens == 0) return PKV_OK;
    if (!out || !q || !cu_q || !q_starts || !kv_lens || !k_cache || !v_cache || !block_tables)
        return fail(PKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PKV_ERR_INVALID_ARG, "q, out and the caches must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(cu_q) | reinterpret_cast<uintptr_t>(q_starts) |
         reinterpret_cast<uintptr_t>(kv_lens) | reinterpret_cast<uintptr_t>(block_tables)) & 3u)
        return fail(PKV_ERR_INVALID_ARG, "index arrays must be 4-byte aligned");
    if (!(scale > 0.f && scale < 3.0e38f)) return fail(PKV_ERR_INVALID_ARG, "scale must be finite and positive");
    DeviceInfo di;
    if ((st = device_info(&di)) != PKV_OK) return st;
    if (di.sms > 256) return fail(PKV_ERR_UNSUPPORTED, "the mixed step's work split takes at most 256 SMs");
    const size_t need = mixed_workspace_bytes(di.sms, num_decode, Hkv, G);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : static_cast<size_t>(0));
    if (need > 0 && !aligned16(workspace)) return fail(PKV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    const bool fp8 = narrow(cache->dtype);
    const int nk = cache->dtype == PKV_INT8 ? 2 : fp8 ? 1 : 0;
    const bool b16 = cache->dtype == PKV_BF16;
    const float kLog2e = 1.4426950408889634f;

    // ---- prefill chunks: [num_decode, num_seqs)
    PrefillArgs pa;
    pa.out = out;
    pa.block_table = block_tables;
    pa.err = device_error;
    pa.NQ = total_q_tokens;
    pa.q_start = 0;
    pa.kv_len = 0;
    pa.Hq = num_q_heads;
    pa.Hkv = Hkv;
    pa.G = G;
    pa.S = S;
    pa.NB = cache->num_blocks;
    pa.n_table = max_blocks_per_seq;
    pa.sm_log2 = scale * kLog2e * (fp8 ? cache->k_scale : 1.f);
    pa.out_mul = fp8 ? cache->v_scale : 1.f;
    pa.sm_base = scale * kLog2e;
    pa.k_head = cache->k_head_scales;
    pa.v_head = cache->v_head_scales;
    pa.timeout_ns = 2000000000ull;
    pa.nseq = num_seqs;
    pa.MB = max_blocks_per_seq;
    pa.cu_q = cu_q;
    pa.q_starts = q_starts;
    pa.kv_lens = kv_lens;
    pa.first_chunk = num_decode;
    const int cta_q = 2 * (128 / G);
    MixedArgs ma;
    ma.num_decode = num_decode;
    ma.slots_x = num_seqs > num_decode ? (total_q_tokens - num_decode) / cta_q + (num_seqs - num_decode) : 0;
    // a prefill key tile's weight in decode stream items (one block of one KV head, K and V)
    ma.tile_cost = kDecodeBytesPerKeyTile * kCostUnit / (S * 128 * (b16 ? 2 : 1) * 2);

    // ---- decode tokens: chunks [0, num_decode), one query each at position kv_len - 1 (the tensor-core decode, one
    // KV head per work unit)
    DecodeArgs da;
    da.out = out;
    da.q = q;
    da.block_tables = block_tables;
    da.context_lens = kv_lens;
    da.err = device_error;
    da.B = num_decode;
    da.Hq = num_q_heads;
    da.Hkv = Hkv;
    da.S = S;
    da.MB = max_blocks_per_seq;
    da.NB = cache->num_blocks;
    da.part_blocks = 1;
    da.q_mul = scale * kLog2e * (fp8 ? cache->k_scale : 1.f);
    da.o_mul = fp8 ? cache->v_scale : 1.f;
    da.q_base = scale * kLog2e;
    da.k_head = cache->k_head_scales;
    da.v_head = cache->v_head_scales;
    da.timeout_ns = 2000000000ull;
    da.tickets = nullptr;
    da.partials = nullptr;
    if (need > 0) {
        da.tickets = static_cast<int32_t*>(workspace);
        const size_t tb = ((static_cast<size_t>(num_decode) * Hkv * 4 + 255) / 256) * 256;
        da.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + tb);
    }
    const uint32_t tile = static_cast<uint32_t>((b16 ? 2 : 1) * std::max(S * 128, 1024));
    da.kv_bytes = static_cast<uint32_t>(S * 128 * (b16 ? 2 : 1));
    da.q_bytes = 0;
    da.stage_bytes = 2 * tile;
    // the sequence prefix of the decode tokens, and before it the slot prefix of the prefill chunks
    const size_t n_prefix = static_cast<size_t>(std::max(num_decode, num_seqs - num_decode)) + 1;
    da.prefix_bytes = static_cast<uint32_t>((n_prefix * 4 + 1023) / 1024 * 1024);
    // CTA costs and cut points of the weighted split
    const size_t cost_bytes = ((2 * static_cast<size_t>(di.sms) + 1) * 4 + 1023) / 1024 * 1024;
    const size_t budget = static_cast<size_t>(di.smem_optin) - 1024 - 1024 - cost_bytes;  // static smem, slack
    const size_t per_warp = budget > da.prefix_bytes ? (budget - da.prefix_bytes) / kMmaWarps : 0;
    int depth = 6;
    while (depth >= 2 && (static_cast<size_t>(depth) * da.stage_bytes + 8 * depth + 1023) / 1024 * 1024 > per_warp)
        --depth;
    if (depth < 2) return fail(PKV_ERR_UNSUPPORTED, "shared memory too small for the mixed step's decode");
    da.depth = depth;
    da.warp_bytes = static_cast<uint32_t>((static_cast<size_t>(depth) * da.stage_bytes + 8 * depth + 1023) / 1024 * 1024);
    ma.cost_off = static_cast<uint32_t>(da.prefix_bytes + static_cast<size_t>(kMmaWarps) * da.warp_bytes);
    const size_t smem_dec = ma.cost_off + cost_bytes + 1024;
    const size_t smem = std::max(smem_dec, prefill_ws_smem_bytes(nk));
    if (smem > static_cast<size_t>(di.smem_optin) - 1024)
        return fail(PKV_ERR_UNSUPPORTED, "device shared memory too small for the mixed step");

    CUtensorMap qm, km, vm;
    if ((st = tensor_map_sw128(&qm, q, false, 128, num_q_heads, total_q_tokens, G, 128 / G)) != PKV_OK) return st;
    const uint64_t rows = static_cast<uint64_t>(cache->num_blocks) * S;
    if ((st = tensor_map_sw128(&km, k_cache, fp8, 128, Hkv, rows, 1, S)) != PKV_OK) return st;
    if ((st = tensor_map_sw128(&vm, v_cache, fp8, 128, Hkv, rows, 1, S)) != PKV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (da.tickets) {
        cudaError_t e = cudaMemsetAsync(da.tickets, 0, static_cast<size_t>(num_decode) * Hkv * 4, s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing split-KV counters");
    }
    const cudaError_t e =
        nk == 0   ? dispatch_mixed<0, KvBF16>(G, qm, km, vm, pa, da, ma, di.sms, smem, s)
        : nk == 1 ? dispatch_mixed<1, KvE4M3>(G, qm, km, vm, pa, da, ma, di.sms, smem, s)
                  : dispatch_mixed<2, KvI8>(G, qm, km, vm, pa, da, ma, di.sms, smem, s);
    if (e != cudaSuccess) return cuda_fail(e, "paged_attention_mixed launch");
    return PKV_OK;
}
