// prefill.cu -- one chunk of a chunked prefill on the 5th-generation tensor cores.
//
// Method ("3.3 批处理与内存管理", section "分块预填充"): the queries of one
// chunk attend to the sequence's KV cache, which already holds the earlier
// chunks and (written first) this chunk's own keys; query i sits at
// position q_start + i and sees keys 0 .. q_start + i (causal).  This is the
// one place of the decode step that is a real dense contraction, so it runs
// on tcgen05:
//   * a CTA owns 128 query rows = (128 / G) consecutive query tokens x the G
//     query heads that share one KV head, so every row of the tile reads
//     the same paged K/V;
//   * Q (128 x 128 bf16) and each 128-key tile of K and V are fetched by TMA
//     with 128-byte swizzle, block by block through the block table
//     (block = table[p / S]); K/V tiles are double-buffered;
//   * S = Q K^T and O += P V are tcgen05.mma kind::f16 (bf16 in, fp32
//     accumulate) issued by one thread, with S and O in tensor memory;
//   * the 128 threads each own one row: online softmax on S (max, exp2,
//     sum) in fp32, P written back to shared memory as bf16 in the swizzled
//     K-major layout the next MMA reads; the O accumulator in TMEM is only
//     rescaled when a row's running max grows by more than 8 (log2 units);
//   * every wait is bounded: on timeout the CTA records the error, leaves
//     the loop together, waits (bounded) for its own MMAs and frees TMEM.
#include "prefill.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;     // query rows per CTA (M)
constexpr int kKeys = 128;     // keys per tile (N of S, K of P.V)
constexpr int kHalf = 16384;   // 128 rows x 64 bf16, one 128-byte-swizzled half tile
constexpr int kOffQ = 0;                       // 2 halves
constexpr int kOffK = kOffQ + 2 * kHalf;       // 2 stages x 2 halves
constexpr int kOffV = kOffK + 4 * kHalf;       // 2 stages x 2 halves
constexpr int kOffP = kOffV + 4 * kHalf;       // 2 halves
constexpr int kOffBar = kOffP + 2 * kHalf;     // mbarriers, TMEM address, abort flag
constexpr int kTmemCols = 256;                 // S: columns 0..127, O: 128..255
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);   // S = Q K^T, both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, true);   // O = P V, V is N (d) major

// mbarrier slots
constexpr int kBarKV0 = 0, kBarQ = 2, kBarS = 3, kBarO = 4;  // kBarKV0 + stage: K/V copies

__device__ __forceinline__ void tma_load_3d_plain(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                  uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(float_to_bf16_bits(lo)) | (static_cast<uint32_t>(float_to_bf16_bits(hi)) << 16);
}

__device__ __forceinline__ float bf16_round(float x) {
    return __uint_as_float(static_cast<uint32_t>(float_to_bf16_bits(x)) << 16);
}

}  // namespace

__global__ void __launch_bounds__(128, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int h = blockIdx.y;
    const int rows_q = kRows / a.G;                                   // query tokens per CTA
    const int i0 = (gridDim.x - 1 - blockIdx.x) * rows_q;             // heaviest (latest) tiles first
    const uint32_t bar = sb + kOffBar;                                // 8 bytes per mbarrier
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 72);

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(bar + 8 * i, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 128;
    const uint32_t trow = static_cast<uint32_t>(warp * 32) << 16;    // this warp's TMEM lanes

    const int r = tid;                        // this thread's row of the tile
    const int qi = i0 + r / a.G;              // its query token
    const int qpos = a.q_start + qi;          // its position
    const int last_q = min(i0 + rows_q, a.NQ) - 1;
    const int max_key = min(a.kv_len - 1, a.q_start + last_q);
    const int n_tiles = max_key / kKeys + 1;
    const int blocks_per_tile = kKeys / a.S;

    // thread 0: copy the K and V tiles of key tile j into stage j & 1
    auto load_kv = [&](int j) {
        const int st = j & 1;
        const uint32_t b = bar + 8 * (kBarKV0 + st);
        mbar_arrive_expect_tx(b, 4 * kHalf);
        for (int bi = 0; bi < blocks_per_tile; ++bi) {
            const int idx = j * blocks_per_tile + bi;
            int c2 = a.NB * a.S;  // beyond the pool: the copy fills zeros
            if (idx < a.n_table) {
                const int phys = a.block_table[idx];
                if (phys >= 0 && phys < a.NB) c2 = phys * a.S;
                else raise_error(a.err, PKV_DEVERR_BAD_BLOCK);
            }
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint32_t off = st * 2 * kHalf + hf * kHalf + bi * a.S * 128;
                tma_load_3d_plain(sb + kOffK + off, &kmap, hf * 64, h, c2, b);
                tma_load_3d_plain(sb + kOffV + off, &vmap, hf * 64, h, c2, b);
            }
        }
    };

    if (tid == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        mbar_arrive_expect_tx(bar + 8 * kBarQ, 2 * kHalf);
        tma_load_3d_plain(sb + kOffQ, &qmap, 0, h * a.G, i0, bar + 8 * kBarQ);
        tma_load_3d_plain(sb + kOffQ + kHalf, &qmap, 64, h * a.G, i0, bar + 8 * kBarQ);
        load_kv(0);
        if (n_tiles > 1) load_kv(1);
    }
    if (!mbar_wait_bounded(bar + 8 * kBarQ, 0, a.timeout_ns)) *abort_flag = 1;

    float m_ref = -INFINITY;  // running max of this row (log2 units)
    float l_run = 0.f;        // running sum of this row's (bf16-rounded) probabilities
    int issued_s = 0;         // S = Q K^T groups committed so far
    int issued_o = 0;         // P.V groups committed so far
    int kv_waited = 0;        // key tiles whose copies were waited for
    int kv_loaded = n_tiles < 2 ? n_tiles : 2;  // key tiles whose copies were issued

    for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        const int tile0 = j * kKeys;
        // ---- K/V of this tile landed; zero V rows of keys past the end (their slots are not data)
        if (!mbar_wait_bounded(bar + 8 * (kBarKV0 + st), (j >> 1) & 1, a.timeout_ns)) *abort_flag = 1;
        kv_waited = j + 1;
        const int nvalid = min(kKeys, a.kv_len - tile0);
        if (nvalid < kKeys) {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int idx = tid; idx < (kKeys - nvalid) * 16; idx += blockDim.x) {
                const int row = nvalid + idx / 16, hf = (idx / 8) & 1, ch = idx & 7;
                *reinterpret_cast<uint4*>(smem + kOffV + st * 2 * kHalf + hf * kHalf + row * 128 + ch * 16) = z;
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        if (*abort_flag) break;
        tc_fence_after();

        // ---- S = Q K^T (8 MMAs of K = 16 over the two 64-wide halves of d)
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t hf = kk >> 2, koff = (kk & 3) * 32;
                const uint64_t ad = smem_desc_sw128(sb + kOffQ + hf * kHalf + koff, 16, 1024);
                const uint64_t bd = smem_desc_sw128(sb + kOffK + st * 2 * kHalf + hf * kHalf + koff, 16, 1024);
                tc_mma_f16(tS, ad, bd, kIdescS, kk > 0);
            }
            tc_commit(bar + 8 * kBarS);
        }
        issued_s = j + 1;
        if (!mbar_wait_bounded(bar + 8 * kBarS, j & 1, a.timeout_ns)) *abort_flag = 1;
        tc_fence_after();

        // ---- pass 1: this row's maximum over the tile (masked keys excluded)
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKeys; c += 32) {
            float v[32];
            tmem_ld32(tS + trow + c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int key = tile0 + c + i;
                if (key < a.kv_len && key <= qpos) mt = fmaxf(mt, v[i] * a.sm_log2);
            }
        }

        // ---- the previous P.V has finished: O may be rescaled and P overwritten
        if (j > 0) {
            if (!mbar_wait_bounded(bar + 8 * kBarO, (j - 1) & 1, a.timeout_ns)) *abort_flag = 1;
            tc_fence_after();
            if (j + 1 < n_tiles) {
                if (tid == 0) load_kv(j + 1);  // its stage was read by tile j - 1
                kv_loaded = j + 2;
            }
        }
        const bool need = mt > m_ref + 8.f;
        if (j > 0 && __any_sync(kFull, need)) {
            const float m_new = need ? mt : m_ref;
            const float alpha = exp2f(m_ref - m_new);
#pragma unroll
            for (int c = 0; c < 128; c += 32) {
                float o[32];
                tmem_ld32(tO + trow + c, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] *= alpha;
                tmem_st32(tO + trow + c, o);
            }
            l_run *= alpha;
            m_ref = m_new;
        } else if (need) {
            m_ref = mt;
        }

        // ---- pass 2: probabilities as bf16 into the swizzled K-major P tile, and the row sum
        float ls = 0.f;
#pragma unroll
        for (int c = 0; c < kKeys; c += 32) {
            float v[32];
            tmem_ld32(tS + trow + c, v);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float p0 = 0.f, p1 = 0.f;
                const int k0 = tile0 + c + i;
                if (k0 < a.kv_len && k0 <= qpos) p0 = bf16_round(exp2f(v[i] * a.sm_log2 - m_ref));
                if (k0 + 1 < a.kv_len && k0 + 1 <= qpos) p1 = bf16_round(exp2f(v[i + 1] * a.sm_log2 - m_ref));
                ls += p0 + p1;
                pk[i / 2] = pack_bf16x2(p0, p1);
            }
            const int hf = c >> 6;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int chunk = ((c & 63) >> 3) + q4;
                const int phys = chunk ^ (r & 7);
                *reinterpret_cast<uint4*>(smem + kOffP + hf * kHalf + r * 128 + phys * 16) =
                    make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            }
        }
        l_run += ls;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*abort_flag) break;
        tc_fence_after();

        // ---- O += P V (8 MMAs of K = 16 keys); V rows are keys, d contiguous (N-major)
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t hf = kk >> 2, koff = (kk & 3) * 32;
                const uint64_t ad = smem_desc_sw128(sb + kOffP + hf * kHalf + koff, 16, 1024);
                const uint64_t bd = smem_desc_sw128(sb + kOffV + st * 2 * kHalf + kk * 2048, kHalf, 1024);
                tc_mma_f16(tO, ad, bd, kIdescPV, (j > 0) || (kk > 0));
            }
            tc_commit(bar + 8 * kBarO);
        }
        issued_o = j + 1;
    }

    const bool aborted = *abort_flag != 0;
    // ---- the last P.V (bounded wait; also on abort, so no MMA is left running)
    if (issued_o > 0) {
        if (!mbar_wait_bounded(bar + 8 * kBarO, (issued_o - 1) & 1, a.timeout_ns)) *abort_flag = 1;
        tc_fence_after();
    }
    if (aborted) {
        // leave nothing in flight: the last S = Q K^T and every issued key-tile copy (all bounded)
        if (issued_s > 0) mbar_wait_bounded(bar + 8 * kBarS, (issued_s - 1) & 1, a.timeout_ns);
        for (int t = kv_waited; t < kv_loaded; ++t)
            mbar_wait_bounded(bar + 8 * (kBarKV0 + (t & 1)), (t >> 1) & 1, a.timeout_ns);
    }
    if (aborted || *abort_flag) {
        if (tid == 0) raise_error(a.err, PKV_DEVERR_TIMEOUT);
    } else {
        // ---- out = O / l for this row
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const int g = r % a.G;
        uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) +
                        ((static_cast<size_t>(qi) * a.Hq + static_cast<size_t>(h) * a.G + g) * 128) * 2;
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
            float o[32];
            tmem_ld32(tO + trow + c, o);  // warp-collective: every lane loads, valid rows store
            if (qi < a.NQ) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 w;
                    w.x = pack_bf16x2(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
                    w.y = pack_bf16x2(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
                    w.z = pack_bf16x2(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
                    w.w = pack_bf16x2(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
                    *reinterpret_cast<uint4*>(orow + (c + 8 * q4) * 2) = w;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

size_t prefill_smem_bytes() { return static_cast<size_t>(kOffBar) + 128 + 1024; }

cudaError_t launch_paged_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const PrefillArgs& a, cudaStream_t stream) {
    const size_t smem = prefill_smem_bytes();
    cudaError_t e =
        cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int rows_q = kRows / a.G;
    dim3 grid((a.NQ + rows_q - 1) / rows_q, a.Hkv);
    paged_prefill_kernel<<<grid, 128, smem, stream>>>(qmap, kmap, vmap, a);
    return cudaGetLastError();
}

}  // namespace pkv
