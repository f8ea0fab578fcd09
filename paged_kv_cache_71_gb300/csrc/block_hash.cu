// block_hash.cu -- content hashes of full KV blocks, for hash-based prefix caching.
//
// "3.3 批处理与内存管理", section "前缀缓存与 RadixAttention": every full block
// is identified by its tokens together with the hash of all blocks before it,
// and a new request reuses every leading block whose hash is already cached.
// Definition (FNV-1a, 64-bit, bytes little-endian):
//   d_j = FNV-1a over the block's S token ids (4 bytes each)
//   h_j = FNV-1a over (h_{j-1}, 8 bytes; 0 for the first block) ++ (d_j, 8 bytes)
// One warp per sequence: lanes hash 32 blocks' tokens in parallel, then the
// chain over those 32 digests runs in every lane in lock step and lane i
// keeps the hash of its block.
#include "cache_ops.cuh"

namespace pkv {

namespace {

constexpr uint64_t kFnvBasis = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

__device__ __forceinline__ uint64_t fnv_byte(uint64_t h, uint32_t byte) { return (h ^ byte) * kFnvPrime; }

__device__ __forceinline__ uint64_t fnv_u32(uint64_t h, uint32_t v) {
    h = fnv_byte(h, v & 0xffu);
    h = fnv_byte(h, (v >> 8) & 0xffu);
    h = fnv_byte(h, (v >> 16) & 0xffu);
    return fnv_byte(h, v >> 24);
}

__device__ __forceinline__ uint64_t fnv_u64(uint64_t h, uint64_t v) {
    h = fnv_u32(h, static_cast<uint32_t>(v));
    return fnv_u32(h, static_cast<uint32_t>(v >> 32));
}

}  // namespace

__global__ void __launch_bounds__(256) block_hash_kernel(const int32_t* __restrict__ tokens,
                                                         const int64_t* __restrict__ cu_tokens, int num_seqs,
                                                         int block_size, const int64_t* __restrict__ out_offsets,
                                                         uint64_t* __restrict__ out, int64_t capacity, int32_t* err) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int s = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; s < num_seqs; s += warps) {
        const int64_t t0 = cu_tokens[s];
        const int64_t L = cu_tokens[s + 1] - t0;
        if (L < 0) {
            if (lane == 0) raise_error(err, PKV_DEVERR_BAD_LENGTH);
            continue;
        }
        const int64_t nfull = L / block_size;
        const int64_t off = out_offsets[s];
        if (off < 0 || off + nfull > capacity) {
            if (lane == 0) raise_error(err, PKV_DEVERR_BAD_SLOT);
            continue;
        }
        uint64_t prev = 0;
        for (int64_t j0 = 0; j0 < nfull; j0 += 32) {
            const int64_t j = j0 + lane;
            uint64_t d = kFnvBasis;
            if (j < nfull) {
                const int32_t* tb = tokens + t0 + j * block_size;
                for (int t = 0; t < block_size; ++t) d = fnv_u32(d, static_cast<uint32_t>(tb[t]));
            }
            const int n = static_cast<int>(nfull - j0 < 32 ? nfull - j0 : 32);
            uint64_t mine = 0;
            for (int i = 0; i < n; ++i) {
                const uint64_t di = __shfl_sync(kFull, d, i);
                prev = fnv_u64(fnv_u64(kFnvBasis, prev), di);
                if (lane == i) mine = prev;
            }
            if (j < nfull) out[off + j] = mine;
        }
    }
}

cudaError_t launch_block_hashes(const int32_t* tokens, const int64_t* cu_tokens, int num_seqs, int block_size,
                                const int64_t* out_offsets, uint64_t* out, int64_t capacity, int32_t* err,
                                int num_sms, cudaStream_t stream) {
    const int warps_needed = num_seqs;
    int grid = (warps_needed + 7) / 8;
    if (grid > num_sms * 8) grid = num_sms * 8;
    if (grid < 1) grid = 1;
    block_hash_kernel<<<grid, 256, 0, stream>>>(tokens, cu_tokens, num_seqs, block_size, out_offsets, out, capacity,
                                                err);
    return cudaGetLastError();
}

}  // namespace pkv
