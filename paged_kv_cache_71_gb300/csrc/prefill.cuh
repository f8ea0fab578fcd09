// prefill.cuh -- arguments and launcher of the chunked-prefill tile kernel.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

struct PrefillArgs {
    void* out;                   // [NQ][Hq][128] bf16 (varlen: [total_q][Hq][128])
    const int32_t* block_table;  // one sequence, n_table entries (varlen: [nseq][MB])
    int32_t* err;                // nullable
    int NQ, q_start, kv_len, Hq, Hkv, G, S, NB, n_table;
    // varlen (nseq > 1): per-chunk query offsets / start positions / key counts, device arrays
    int nseq = 1, MB = 0;
    const int32_t* cu_q = nullptr;
    const int32_t* q_starts = nullptr;
    const int32_t* kv_lens = nullptr;
    float sm_log2;               // scale * log2(e) (* k_scale for FP8 / INT8 caches)
    float out_mul;               // v_scale for FP8 / INT8 caches, else 1
    uint64_t timeout_ns;
};

size_t prefill_smem_bytes(bool fp8);
size_t prefill_ws_smem_bytes();
int prefill_ws_max_seqs();

// bf16 caches, warp-specialised, one or several chunks (prefill_ws.cu)
cudaError_t launch_paged_prefill_ws(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                    const PrefillArgs& a, cudaStream_t stream);

cudaError_t launch_paged_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const PrefillArgs& a, int narrow, cudaStream_t stream);  // 0 bf16, 1 FP8, 2 INT8

}  // namespace pkv
