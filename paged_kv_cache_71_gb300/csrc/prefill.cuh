// prefill.cuh -- arguments and launcher of the chunked-prefill tile kernel (prefill_ws.cu).
#pragma once

#include "pkv_device.cuh"

namespace pkv {

struct PrefillArgs {
    void* out;                   // [NQ][Hq][128] bf16 (varlen: [total_q][Hq][128])
    const int32_t* block_table;  // one sequence, n_table entries (varlen: [nseq][MB])
    int32_t* err;                // nullable
    int NQ, q_start, kv_len, Hq, Hkv, G, S, NB, n_table;
    // varlen (cu_q set): per-chunk query offsets / start positions / key counts, device arrays
    int nseq = 1, MB = 0;
    int first_chunk = 0;         // chunks below it are not prefill chunks (a mixed step's decode tokens)
    const int32_t* cu_q = nullptr;
    const int32_t* q_starts = nullptr;
    const int32_t* kv_lens = nullptr;
    float sm_log2;               // scale * log2(e) (* k_scale for FP8 / INT8 caches)
    float out_mul;               // v_scale for FP8 / INT8 caches, else 1
    float sm_base = 0.f;         // scale * log2(e)
    const float* k_head = nullptr;  // per-KV-head scales replacing k_scale / v_scale (nullable)
    const float* v_head = nullptr;
    uint64_t timeout_ns;
};

size_t prefill_ws_smem_bytes(int narrow);
int prefill_ws_max_seqs();

// warp-specialised tile, one or several chunks (prefill_ws.cu); narrow: 0 bf16, 1 FP8 E4M3, 2 INT8 cache
cudaError_t launch_paged_prefill_ws(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                    const PrefillArgs& a, int narrow, cudaStream_t stream);


}  // namespace pkv
