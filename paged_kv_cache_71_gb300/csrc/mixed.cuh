// mixed.cuh -- one launch for a mixed serving step: decode tokens and prefill chunks of different sequences
// ("从 PagedAttention 到 Chunked Prefill" §3.2: chunked prefill and decode share one step; "3.3 批处理与内存管理",
// section "分块预填充").
//
// One CTA per SM, 384 threads.  Each CTA first runs its prefill tiles (prefill_tile.cuh: the tcgen05/TMEM tile, all
// 12 warps), then joins the decode of the step's decode tokens (decode_mma.cuh: the per-warp tensor-core decode, 8
// worker warps) -- the 4 remaining warps give their registers back (setmaxnreg) so that the workers get 240 a thread
// (the whole register file: 4 x 24 + 8 x 240 = 12 x 168).  The decode stream is cut by weight: a CTA that spent the
// first part of the launch on prefill tiles gets a smaller part of the stream, so that all CTAs finish together.  The
// weight of a prefill key tile, in decode stream items, comes from measurements on GB300: one 64-key tile of a
// two-query-tile CTA takes as long as an SM needs to stream about kDecodeBytesPerKeyTile bytes of decode K/V.
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
    int tile_cost;    // one prefill key tile in 1/kCostUnit decode stream items
    uint32_t cost_off;  // offset of the cost and cut-point arrays in dynamic shared memory (past the decode plan)
};

// This CTA's prefill tile slots (slot -> query-tile slot x, KV head h).  Kept out of line: inlined, it changed how
// the decode that follows was compiled, and the FP8 decode ran 4% slower (Llama-70B step, GB300).
template <int NARROW>
__device__ __noinline__ void mixed_prefill_slots(const CUtensorMap& qmap, const CUtensorMap& kmap,
                                                 const CUtensorMap& vmap, const PrefillArgs& pa, int slots_x,
                                                 uint8_t* smem_raw) {
    const int n_slots = slots_x * pa.Hkv;
    for (int sl = blockIdx.x; sl < n_slots; sl += gridDim.x)
        prefill_tile<NARROW, NARROW == 2, true>(qmap, kmap, vmap, pa, sl % slots_x, sl / slots_x, slots_x, smem_raw);
}

template <int NARROW, int G, class KV>
__global__ void __launch_bounds__(384, 1)
    paged_mixed_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const PrefillArgs pa, const DecodeArgs da,
                       const MixedArgs ma) {
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ncta = gridDim.x, cta = blockIdx.x;
    const int n_slots = ma.slots_x * pa.Hkv;

    // ---- phase 1: this CTA's prefill tile slots
    mixed_prefill_slots<NARROW>(qmap, kmap, vmap, pa, ma.slots_x, smem_raw);

    // ---- phase 2: decode; warps 8-11 leave and hand their registers to the 8 worker warps
    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 24;");
        return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 240;");
    if (ma.num_decode == 0) return;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* pcost = reinterpret_cast<int*>(base + ma.cost_off);  // ncta entries
    int* cb = pcost + ncta;                                   // cut points (ncta + 1; 8 of them scratch here)
    // Every CTA's prefill work in 1/kCostUnit decode stream items: the key tiles of the slots it ran, with the tile's
    // own arithmetic (chunk from the prefix of slot counts, tokens heaviest first, keys up to the causal limit).
    // All 256 threads: (1) slot counts of the prefill chunks and their exclusive prefix, in the decode plan's
    // sequence-prefix region (the decode rewrites it after the barrier below); (2) one thread per CTA sums its slots.
    const int cta_q = 2 * (128 / pa.G);
    const int nch = pa.nseq - ma.num_decode;
    int* cpre = reinterpret_cast<int*>(base);  // nch + 1 entries
    auto chunk_geom = [&](int c, int& nq, int& q_start, int& kv_len) {  // chunk c's query count (0 if malformed)
        const int q0 = pa.cu_q[c], q1 = pa.cu_q[c + 1];
        nq = (q0 >= 0 && q1 >= q0 && q1 <= pa.NQ) ? q1 - q0 : 0;
        q_start = pa.q_starts[c];
        kv_len = pa.kv_lens[c];
    };
    {
        const int per = (nch + 255) / 256;
        const int i_lo = min(tid * per, nch), i_hi = min(i_lo + per, nch);
        int sum = 0;
        for (int i = i_lo; i < i_hi; ++i) {
            const int q0 = pa.cu_q[ma.num_decode + i], q1 = pa.cu_q[ma.num_decode + i + 1];
            const int nt = (q0 >= 0 && q1 >= q0 && q1 <= pa.NQ) ? (q1 - q0 + cta_q - 1) / cta_q : 0;
            cpre[i + 1] = nt;
            sum += nt;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) cb[warp] = incl;
        threads_sync(256);
        int run = incl - sum;
        for (int k = 0; k < warp; ++k) run += cb[k];
        for (int i = i_lo; i < i_hi; ++i) {
            run += cpre[i + 1];
            cpre[i + 1] = run;
        }
        if (tid == 0) cpre[0] = 0;
        threads_sync(256);
    }
    const int n_used = cpre[nch];  // slot columns holding a chunk
    for (int c = tid; c < ncta; c += 256) {
        int cost = 0;
        for (int sl = c; sl < n_slots; sl += ncta) {
            const int x = sl % ma.slots_x;
            if (x >= n_used) continue;
            int lo = 0, hi = nch - 1;  // the chunk whose slots hold x
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (cpre[mid] <= x) lo = mid; else hi = mid - 1;
            }
            int nq, q_start, kv_len;
            chunk_geom(ma.num_decode + lo, nq, q_start, kv_len);
            const int nt = cpre[lo + 1] - cpre[lo];
            const int i0 = (nt - 1 - (x - cpre[lo])) * cta_q;  // slot x's first token
            const int last_q = min(i0 + cta_q, nq) - 1;
            const int max_key = min(kv_len - 1, q_start + last_q);
            if (max_key >= 0) cost += (max_key / 64 + 1) * ma.tile_cost;
        }
        pcost[c] = cost;
    }
    // decode tokens must be chunks of one query at position kv_len - 1
    if (cta == 0)
        for (int s = tid; s < ma.num_decode; s += 256)
            if (pa.cu_q[s] != s || pa.cu_q[s + 1] != s + 1 || pa.q_starts[s] != pa.kv_lens[s] - 1)
                raise_error(pa.err, PKV_DEVERR_BAD_LENGTH);
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
