// cache_ops.cuh -- launchers of the cache write and block copy kernels.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

cudaError_t launch_reshape_and_cache(const void* k_new, const void* v_new, int src_dtype, const int64_t* slots,
                                     int T, void* k_cache, void* v_cache, int dst_dtype, int64_t pool_slots,
                                     int row_elems, int head_dim, float k_scale, float v_scale,
                                     const float* k_head, const float* v_head, int32_t* err, int num_sms,
                                     cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* mapping, int num_pairs, int num_blocks,
                               int64_t block_bytes, int32_t* err, cudaStream_t stream);

cudaError_t launch_swap_blocks(const void* src_k, const void* src_v, int src_nb, void* dst_k, void* dst_v,
                               int dst_nb, const int64_t* mapping, int num_pairs, int64_t block_bytes, int32_t* err,
                               cudaStream_t stream);

cudaError_t launch_block_hashes(const int32_t* tokens, const int64_t* cu_tokens, int num_seqs, int block_size,
                                const int64_t* out_offsets, uint64_t* out, int64_t capacity, int32_t* err,
                                int num_sms, cudaStream_t stream);

}  // namespace pkv
