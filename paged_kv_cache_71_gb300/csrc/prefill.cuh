// prefill.cuh -- arguments and launcher of the chunked-prefill tile kernel.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

struct PrefillArgs {
    void* out;                   // [NQ][Hq][128] bf16
    const int32_t* block_table;  // one sequence, n_table entries
    int32_t* err;                // nullable
    int NQ, q_start, kv_len, Hq, Hkv, G, S, NB, n_table;
    float sm_log2;               // scale * log2(e) (* k_scale for FP8 / INT8 caches)
    float out_mul;               // v_scale for FP8 / INT8 caches, else 1
    uint64_t timeout_ns;
};

size_t prefill_smem_bytes(bool fp8);

cudaError_t launch_paged_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const PrefillArgs& a, int narrow, cudaStream_t stream);  // 0 bf16, 1 FP8, 2 INT8

}  // namespace pkv
