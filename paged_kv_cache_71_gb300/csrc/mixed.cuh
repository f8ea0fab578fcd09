// mixed.cuh -- one launch for a mixed serving step: decode tokens and prefill chunks of different sequences
// ("从 PagedAttention 到 Chunked Prefill" §3.2: chunked prefill and decode share one step; "3.3 批处理与内存管理",
// section "分块预填充").
//
// One CTA per SM, 384 threads.  Each CTA first runs its prefill tiles (prefill_tile.cuh: the tcgen05/TMEM tile, all
// 12 warps), then joins the decode of the step's decode tokens (decode_mma.cuh: the per-warp tensor-core decode, 8
// worker warps) -- the 4 remaining warps give their registers back (setmaxnreg) so that the workers get the 232 a
// thread they need.  The decode stream is cut by weight: a CTA that spent the first part of the launch on prefill
// tiles gets a smaller part of the stream, so that all CTAs finish together.  The weight of a prefill key tile, in
// decode stream items, comes from measurements on GB300: one 64-key tile of a two-query-tile CTA takes as long as an
// SM needs to stream about kDecodeBytesPerKeyTile bytes of decode K/V.
#pragma once

#include "decode_mma.cuh"
#include "prefill_tile.cuh"

namespace pkv {

// Decode K/V bytes one SM streams in the time of one 64-key prefill tile of a CTA holding two 128-row query tiles
// (GB300: bf16 tile 0.87 us per key tile against 39 KB/us of decode per SM; FP8 1.04 us against 34 KB/us)
constexpr int kDecodeBytesPerKeyTile = 36 * 1024;

struct MixedArgs {
    int num_decode;   // chunks [0, num_decode) are decode tokens, [num_decode, nseq) prefill chunks
    int slots_x;      // prefill tile slots per KV head (an upper bound of the CTAs the chunks need)
    int item_bytes;   // bytes of one decode stream item (a block of one KV head, K and V)
    uint32_t cost_off;  // offset of the cost / cut-point arrays in dynamic shared memory (past the decode plan)
};

template <int NARROW, int G, class KV>
__global__ void __launch_bounds__(384, 1)
    paged_mixed_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const PrefillArgs pa, const DecodeArgs da,
                       const MixedArgs ma) {
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ncta = gridDim.x, cta = blockIdx.x;
    const int n_slots = ma.slots_x * pa.Hkv;

    // ---- phase 1: this CTA's prefill tile slots (slot -> query-tile slot x, KV head h)
    for (int sl = cta; sl < n_slots; sl += ncta)
        prefill_tile<NARROW, NARROW == 2, true>(qmap, kmap, vmap, pa, sl % ma.slots_x, sl / ma.slots_x, ma.slots_x,
                                                smem_raw);

    // ---- phase 2: decode; warps 8-11 leave and hand their registers to the 8 worker warps
    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 24;");
        return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
    if (ma.num_decode == 0) return;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* pcost = reinterpret_cast<int*>(base + ma.cost_off);  // ncta entries
    int* cb = pcost + ncta;                                   // ncta + 1 entries
    if (warp == 0) {
        // every CTA's prefill work in decode stream items: the key tiles of the slots it ran (the same arithmetic
        // as the tile's own: chunk from the CTA-count prefix, tokens heaviest first, keys up to the causal limit)
        const int cta_q = 2 * (128 / pa.G);
        for (int c = lane; c < ncta; c += 32) pcost[c] = 0;
        __syncwarp();
        int run = 0;  // CTA slots of the chunks before the current group of 32
        for (int c0 = ma.num_decode; c0 < pa.nseq; c0 += 32) {
            const int c = c0 + lane;
            int nt = 0, kv_len = 0, q_start = 0, nq = 0;
            if (c < pa.nseq) {
                const int q0 = pa.cu_q[c], q1 = pa.cu_q[c + 1];
                if (q0 >= 0 && q1 >= q0 && q1 <= pa.NQ) {
                    nq = q1 - q0;
                    nt = (nq + cta_q - 1) / cta_q;
                    kv_len = pa.kv_lens[c];
                    q_start = pa.q_starts[c];
                }
            }
            int incl = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            const int first = run + incl - nt;
            for (int xi = 0; xi < nt; ++xi) {  // slot x = first + xi holds tokens from (nt - 1 - xi) * cta_q
                const int i0 = (nt - 1 - xi) * cta_q;
                const int last_q = min(i0 + cta_q, nq) - 1;
                const int max_key = min(kv_len - 1, q_start + last_q);
                const int kt = max_key >= 0 ? max_key / 64 + 1 : 0;
                const int x = first + xi;
                if (x >= ma.slots_x) continue;
                const long long items = (static_cast<long long>(kt) * kDecodeBytesPerKeyTile) / ma.item_bytes;
                for (int h = 0; h < pa.Hkv; ++h) atomicAdd(&pcost[(h * ma.slots_x + x) % ncta], static_cast<int>(items));
            }
            run += __shfl_sync(kFull, incl, 31);
            __syncwarp();
        }
        // decode tokens must be chunks of one query at position kv_len - 1
        if (cta == 0)
            for (int s = lane; s < ma.num_decode; s += 32)
                if (pa.cu_q[s] != s || pa.cu_q[s + 1] != s + 1 || pa.q_starts[s] != pa.kv_lens[s] - 1)
                    raise_error(pa.err, PKV_DEVERR_BAD_LENGTH);
    }
    threads_sync(256);
    decode_mma_body<G, 16, KV, 1, true>(kmap, vmap, da, smem_raw, cta, ncta, 256, pcost, cb);
}

template <int NARROW, int G, class KV>
cudaError_t launch_paged_mixed(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               const PrefillArgs& pa, const DecodeArgs& da, const MixedArgs& ma, int grid,
                               size_t smem, cudaStream_t stream) {
    auto kern = paged_mixed_kernel<NARROW, G, KV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, 384, smem, stream>>>(qmap, kmap, vmap, pa, da, ma);
    return cudaGetLastError();
}

}  // namespace pkv
