// cache_ops.cu -- the cache write (reshape_and_cache) and the block copy
// (copy_blocks) kernels.  Both are pure data movement: 16-byte vectors,
// coalesced, one pass, grid sized in multiples of the SM count.
#include "cache_ops.cuh"

namespace pkv {

// ------------------------------------------------------------------ reshape_and_cache
//
// New token i goes to slot[i] = block * S + offset ("3.3 批处理与内存管理",
// "PagedAttention：块表"): k_cache[slot / S][slot % S][:, :] = convert(k_new[i]).
// In the [NB][S][Hkv][D] layout one token's Hkv*D elements are contiguous in
// both source and destination, so a token is one contiguous run per tensor.
// Each thread moves 8 elements.

template <int SRC, int DST>
__device__ __forceinline__ void convert8(const uint8_t* src, uint8_t* dst, float scale) {
    float f[8];
    if constexpr (SRC == PKV_F32) {
        const float4 a = reinterpret_cast<const float4*>(src)[0];
        const float4 b = reinterpret_cast<const float4*>(src)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p = bf16x2_to_float2(w[i]);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
    if constexpr (DST == PKV_F32) {
        reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
    } else if constexpr (DST == PKV_BF16) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = static_cast<uint32_t>(float_to_bf16_bits(f[2 * i])) |
                   (static_cast<uint32_t>(float_to_bf16_bits(f[2 * i + 1])) << 16);
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (DST == PKV_INT8) {
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y = f[i] / scale;  // IEEE fp32 division, then RNE to an integer, clamped to +-127
            w[i / 4] |= static_cast<uint32_t>(float_to_s8_sym(y)) << (8 * (i % 4));
        }
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else {
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y = f[i] / scale;  // IEEE fp32 division, then RNE to E4M3 with saturation
            w[i / 4] |= static_cast<uint32_t>(float_to_e4m3_sat(y)) << (8 * (i % 4));
        }
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    }
}

template <int SRC, int DST>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const uint8_t* __restrict__ k_new,
                                                                const uint8_t* __restrict__ v_new,
                                                                const int64_t* __restrict__ slots, int T,
                                                                uint8_t* __restrict__ k_cache,
                                                                uint8_t* __restrict__ v_cache, int64_t pool_slots,
                                                                int row_elems, int head_dim, float k_scale,
                                                                float v_scale, const float* __restrict__ k_head,
                                                                const float* __restrict__ v_head, int32_t* err) {
    constexpr int SES = (SRC == PKV_F32) ? 4 : 2;
    constexpr int DES = (DST == PKV_F32) ? 4 : (DST == PKV_BF16) ? 2 : 1;  // FP8 and INT8: one byte
    const int vec_per_row = row_elems / 8;
    const long long total = static_cast<long long>(T) * 2 * vec_per_row;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int vec = static_cast<int>(idx % vec_per_row);
        const long long rest = idx / vec_per_row;
        const int kv = static_cast<int>(rest & 1);
        const int i = static_cast<int>(rest >> 1);
        const int64_t slot = slots[i];
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (kv == 0 && vec == 0) raise_error(err, PKV_DEVERR_BAD_SLOT);
            continue;
        }
        const uint8_t* src = (kv ? v_new : k_new) + (static_cast<size_t>(i) * row_elems + vec * 8) * SES;
        uint8_t* dst = (kv ? v_cache : k_cache) + (static_cast<size_t>(slot) * row_elems + vec * 8) * DES;
        // per-head scales (when given) replace the per-tensor ones: the 8 elements lie in head (vec * 8) / D
        const float* hs = kv ? v_head : k_head;
        convert8<SRC, DST>(src, dst, hs ? __ldg(hs + (vec * 8) / head_dim) : (kv ? v_scale : k_scale));
    }
}

cudaError_t launch_reshape_and_cache(const void* k_new, const void* v_new, int src_dtype, const int64_t* slots,
                                     int T, void* k_cache, void* v_cache, int dst_dtype, int64_t pool_slots,
                                     int row_elems, int head_dim, float k_scale, float v_scale,
                                     const float* k_head, const float* v_head, int32_t* err, int num_sms,
                                     cudaStream_t stream) {
    const long long total = static_cast<long long>(T) * 2 * (row_elems / 8);
    const int block = 256;
    long long want = (total + block - 1) / block;
    const long long cap = static_cast<long long>(num_sms) * 8;
    const int grid = static_cast<int>(want < cap ? (want < 1 ? 1 : want) : cap);
    auto* kn = static_cast<const uint8_t*>(k_new);
    auto* vn = static_cast<const uint8_t*>(v_new);
    auto* kc = static_cast<uint8_t*>(k_cache);
    auto* vc = static_cast<uint8_t*>(v_cache);
#define PKV_RC(S_, D_)                                                                                          \
    if (src_dtype == S_ && dst_dtype == D_) {                                                                   \
        reshape_and_cache_kernel<S_, D_><<<grid, block, 0, stream>>>(kn, vn, slots, T, kc, vc, pool_slots,      \
                                                                    row_elems, head_dim, k_scale, v_scale,      \
                                                                    k_head, v_head, err);                       \
        return cudaGetLastError();                                                                              \
    }
    PKV_RC(PKV_F32, PKV_F32)
    PKV_RC(PKV_F32, PKV_BF16)
    PKV_RC(PKV_F32, PKV_FP8_E4M3)
    PKV_RC(PKV_BF16, PKV_F32)
    PKV_RC(PKV_BF16, PKV_BF16)
    PKV_RC(PKV_BF16, PKV_FP8_E4M3)
    PKV_RC(PKV_F32, PKV_INT8)
    PKV_RC(PKV_BF16, PKV_INT8)
#undef PKV_RC
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ copy_blocks
//
// Copy-on-write data copy ("3.3 批处理与内存管理", "共享与写时复制"): whole
// physical blocks, K and V, src -> dst.  One CTA per (pair, tensor); a block
// of bf16 S=16, Hkv=8, D=128 is 32 KB = 2048 vectors of 16 B.

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint8_t* __restrict__ k_cache,
                                                          uint8_t* __restrict__ v_cache,
                                                          const int64_t* __restrict__ mapping, int num_pairs,
                                                          int num_blocks, int64_t block_bytes, int32_t* err) {
    const int pair = blockIdx.x >> 1;
    const int kv = blockIdx.x & 1;
    if (pair >= num_pairs) return;
    const int64_t src = mapping[2 * pair];
    const int64_t dst = mapping[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (kv == 0 && threadIdx.x == 0) raise_error(err, PKV_DEVERR_BAD_BLOCK);
        return;
    }
    uint8_t* base = kv ? v_cache : k_cache;
    const uint4* s = reinterpret_cast<const uint4*>(base + src * block_bytes);
    uint4* d = reinterpret_cast<uint4*>(base + dst * block_bytes);
    const int64_t nvec = block_bytes / 16;
    constexpr int U = 4;
    for (int64_t i = threadIdx.x; i < nvec; i += static_cast<int64_t>(blockDim.x) * U) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t j = i + static_cast<int64_t>(u) * blockDim.x;
            if (j < nvec) r[u] = __ldcs(s + j);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t j = i + static_cast<int64_t>(u) * blockDim.x;
            if (j < nvec) __stcs(d + j, r[u]);
        }
    }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* mapping, int num_pairs, int num_blocks,
                               int64_t block_bytes, int32_t* err, cudaStream_t stream) {
    copy_blocks_kernel<<<2u * static_cast<unsigned>(num_pairs), 256, 0, stream>>>(static_cast<uint8_t*>(k_cache),
                                                         static_cast<uint8_t*>(v_cache), mapping, num_pairs,
                                                         num_blocks, block_bytes, err);
    return cudaGetLastError();
}

}  // namespace pkv

namespace pkv {

// ------------------------------------------------------------------ swap_blocks
//
// Preemption by swapping ("从 PagedAttention 到 Chunked Prefill" §3.1): a
// preempted sequence's blocks move to CPU memory and back.  On GB300 the
// Grace memory is reachable from the GPU over NVLink-C2C, so one kernel
// gathers all pairs with 16-byte loads and stores, whichever side is host
// memory.  One CTA per (pair, tensor).

__global__ void __launch_bounds__(256) swap_blocks_kernel(const uint8_t* __restrict__ src_k,
                                                          const uint8_t* __restrict__ src_v,
                                                          uint8_t* __restrict__ dst_k, uint8_t* __restrict__ dst_v,
                                                          const int64_t* __restrict__ mapping, int num_pairs,
                                                          int src_nb, int dst_nb, int64_t block_bytes, int32_t* err) {
    const int pair = blockIdx.x >> 1;
    const int kv = blockIdx.x & 1;
    if (pair >= num_pairs) return;
    const int64_t src = mapping[2 * pair];
    const int64_t dst = mapping[2 * pair + 1];
    if (src < 0 || src >= src_nb || dst < 0 || dst >= dst_nb) {
        if (kv == 0 && threadIdx.x == 0) raise_error(err, PKV_DEVERR_BAD_BLOCK);
        return;
    }
    const uint4* s = reinterpret_cast<const uint4*>((kv ? src_v : src_k) + src * block_bytes);
    uint4* d = reinterpret_cast<uint4*>((kv ? dst_v : dst_k) + dst * block_bytes);
    const int64_t nvec = block_bytes / 16;
    constexpr int U = 8;
    for (int64_t i = threadIdx.x; i < nvec; i += static_cast<int64_t>(blockDim.x) * U) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t j = i + static_cast<int64_t>(u) * blockDim.x;
            if (j < nvec) r[u] = __ldcs(s + j);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t j = i + static_cast<int64_t>(u) * blockDim.x;
            if (j < nvec) __stcs(d + j, r[u]);
        }
    }
}

cudaError_t launch_swap_blocks(const void* src_k, const void* src_v, int src_nb, void* dst_k, void* dst_v,
                               int dst_nb, const int64_t* mapping, int num_pairs, int64_t block_bytes, int32_t* err,
                               cudaStream_t stream) {
    swap_blocks_kernel<<<2u * static_cast<unsigned>(num_pairs), 256, 0, stream>>>(
        static_cast<const uint8_t*>(src_k), static_cast<const uint8_t*>(src_v), static_cast<uint8_t*>(dst_k),
        static_cast<uint8_t*>(dst_v), mapping, num_pairs, src_nb, dst_nb, block_bytes, err);
    return cudaGetLastError();
}

}  // namespace pkv
