// prefill_ws.cu -- the chunked-prefill kernels: one chunk (pkv_paged_prefill_chunk) or several chunks of different
// sequences (pkv_paged_prefill_varlen) over bf16, FP8 or INT8 caches, one CTA per tile of prefill_tile.cuh.
#include "prefill_tile.cuh"

namespace pkv {

template <int NARROW, bool ADAPT>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_ws_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    prefill_tile<NARROW, ADAPT, false>(qmap, kmap, vmap, a, blockIdx.x, blockIdx.y, gridDim.x, smem_raw);
}

template <int NARROW>
static size_t ws_smem_bytes() {
    return static_cast<size_t>(Plan<NARROW>::kOffMeta) + kMetaCount + 4 * (kMaxSeqs + 1) + 1024;
}

size_t prefill_ws_smem_bytes(int narrow) {
    return narrow == 2 ? ws_smem_bytes<2>() : narrow == 1 ? ws_smem_bytes<1>() : ws_smem_bytes<0>();
}

int prefill_ws_max_seqs() { return kMaxSeqs; }

template <int NARROW>
static cudaError_t launch_ws(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const PrefillArgs& a, cudaStream_t stream) {
    const size_t smem = ws_smem_bytes<NARROW>();
    constexpr bool kAdapt = NARROW == 2;
    const bool adapt = kAdapt && a.cu_q != nullptr;
    cudaError_t e = cudaFuncSetAttribute(
        adapt ? paged_prefill_ws_kernel<NARROW, kAdapt> : paged_prefill_ws_kernel<NARROW, false>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // CTAs: one per 2 * 128 / G tokens of each chunk; in the varlen form an upper bound (each chunk adds at
    // most one partial CTA), the CTAs past the chunks' total leave at once
    const int cta_q = 2 * (128 / a.G);
    const int grid_x = a.cu_q == nullptr ? (a.NQ + cta_q - 1) / cta_q : a.NQ / cta_q + a.nseq;
    if (grid_x <= 0) return cudaSuccess;
    dim3 grid(grid_x, a.Hkv);
    if (adapt)
        paged_prefill_ws_kernel<NARROW, kAdapt><<<grid, kThreads, smem, stream>>>(qmap, kmap, vmap, a);
    else
        paged_prefill_ws_kernel<NARROW, false><<<grid, kThreads, smem, stream>>>(qmap, kmap, vmap, a);
    return cudaGetLastError();
}

cudaError_t launch_paged_prefill_ws(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                    const PrefillArgs& a, int narrow, cudaStream_t stream) {
    switch (narrow) {
        case 0: return launch_ws<0>(qmap, kmap, vmap, a, stream);
        case 1: return launch_ws<1>(qmap, kmap, vmap, a, stream);
        case 2: return launch_ws<2>(qmap, kmap, vmap, a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
