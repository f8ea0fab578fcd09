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
constexpr int kOffStage = kOffP + 2 * kHalf;   // FP8 caches only: K and V codes of one key tile (32 KB)
template <bool FP8>
constexpr int off_bar() { return kOffStage + (FP8 ? 2 * kHalf : 0); }  // mbarriers, TMEM address, abort flag
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

// Two floats -> packed bf16x2 (round to nearest even), low half first.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace

// NARROW: 0 = bf16 cache; 1 = FP8 E4M3 codes; 2 = INT8 codes (both widened to bf16 on chip).
// 256 threads: warp w works on TMEM lanes 32 (w % 4) .. + 31 (rows of the tile) and on the
// half w / 4 of the columns -- keys 64 (w / 4) .. + 63 of S, head dims of O likewise.
template <int NARROW>
__global__ void __launch_bounds__(256, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
    constexpr bool FP8 = NARROW != 0;  // a one-byte cache, staged and widened
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int h = blockIdx.y;
    const int rows_q = kRows / a.G;                                   // query tokens per CTA
    const int i0 = (gridDim.x - 1 - blockIdx.x) * rows_q;             // heaviest (latest) tiles first
    constexpr int kOffBar = off_bar<FP8>();
    const uint32_t bar = sb + kOffBar;                                // 8 bytes per mbarrier
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 72);
    float* row_x = reinterpret_cast<float*>(smem + kOffBar + 128);   // [2][128] per-half row maxima / sums

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
    const uint32_t trow = static_cast<uint32_t>(quad * 32) << 16;    // this warp's TMEM lanes
    const int col0 = half * 64;                                       // this thread's 64 columns

    const int r = quad * 32 + lane;           // this thread's row of the tile
    const int qi = i0 + r / a.G;              // its query token
    const int qpos = a.q_start + qi;          // its position
    const int last_q = min(i0 + rows_q, a.NQ) - 1;
    const int max_key = min(a.kv_len - 1, a.q_start + last_q);
    const int n_tiles = max_key / kKeys + 1;
    const int blocks_per_tile = kKeys / a.S;

    // Thread 0: copy the K and V tiles of key tile j (bf16: into stage j & 1; FP8/INT8: into the code
    // staging area).  The tile's block-table entries are read first, all at once, so their latencies overlap.
    auto load_kv = [&](int j) {
        const int st = FP8 ? 0 : (j & 1);
        const uint32_t b = bar + 8 * (kBarKV0 + st);
        int c2s[kKeys / 8];
#pragma unroll
        for (int bi = 0; bi < kKeys / 8; ++bi) {
            const int idx = j * blocks_per_tile + bi;
            c2s[bi] = (bi < blocks_per_tile && idx < a.n_table) ? a.block_table[idx] : -1;
        }
        mbar_arrive_expect_tx(b, FP8 ? 2 * kHalf : 4 * kHalf);
        for (int bi = 0; bi < blocks_per_tile; ++bi) {
            const int idx = j * blocks_per_tile + bi;
            const int phys = c2s[bi];
            int c2 = a.NB * a.S;  // beyond the pool: the copy fills zeros
            if (idx < a.n_table) {
                if (phys >= 0 && phys < a.NB) c2 = phys * a.S;
                else raise_error(a.err, PKV_DEVERR_BAD_BLOCK);
            }
            if constexpr (FP8) {
                const uint32_t off = bi * a.S * 128;  // 128 one-byte codes per key row
                tma_load_3d_plain(sb + kOffStage + off, &kmap, 0, h, c2, b);
                tma_load_3d_plain(sb + kOffStage + kHalf + off, &vmap, 0, h, c2, b);
            } else {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const uint32_t off = st * 2 * kHalf + hf * kHalf + bi * a.S * 128;
                    tma_load_3d_plain(sb + kOffK + off, &kmap, hf * 64, h, c2, b);
                    tma_load_3d_plain(sb + kOffV + off, &vmap, hf * 64, h, c2, b);
                }
            }
        }
    };

    // FP8 / INT8: widen the staged codes of one key tile into the bf16 stage st (exact; the
    // per-tensor scales are applied to the scores and to the output instead).
    // Thread t converts key row t % 128 of K (t < 128) or of V; V rows of keys past the end become 0.
    auto widen_fp8 = [&](int st, int nvalid) {
        const int t = tid & 127, kv = tid >> 7;
        const uint8_t* src = smem + kOffStage + kv * kHalf + t * 128;
        uint8_t* dst0 = smem + (kv ? kOffV : kOffK) + st * 2 * kHalf + t * 128;
        const bool zero = kv == 1 && t >= nvalid;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // logical 16-code chunk: head dims 16c .. 16c + 15
            uint32_t o[8];
            if (zero) {
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = 0u;
            } else {
                const uint4 wv = *reinterpret_cast<const uint4*>(src + ((c ^ (t & 7)) * 16));
                const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 f0, f1;
                    if constexpr (NARROW == 2) {
                        f0 = s8x2_to_float2(ws[i], 0);
                        f1 = s8x2_to_float2(ws[i], 2);
                    } else {
                        f0 = e4m3x2_to_float2(static_cast<uint16_t>(ws[i] & 0xffffu));
                        f1 = e4m3x2_to_float2(static_cast<uint16_t>(ws[i] >> 16));
                    }
                    o[2 * i] = pack_bf16x2_rn(f0.x, f0.y);
                    o[2 * i + 1] = pack_bf16x2_rn(f1.x, f1.y);
                }
            }
            uint8_t* dst = dst0 + (c >> 2) * kHalf;
            const int lc = 2 * (c & 3);
            *reinterpret_cast<uint4*>(dst + ((lc ^ (t & 7)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + (((lc + 1) ^ (t & 7)) * 16)) = make_uint4(o[4], o[5], o[6], o[7]);
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
        if (!FP8 && n_tiles > 1) load_kv(1);
    }
    if (!mbar_wait_bounded(bar + 8 * kBarQ, 0, a.timeout_ns)) *abort_flag = 1;

    float m_ref = -INFINITY;  // running max of this row (log2 units), same in both halves
    float l_run = 0.f;        // running sum of this thread's half of the row's probabilities
    int issued_s = 0;         // S = Q K^T groups committed so far
    int issued_o = 0;         // P.V groups committed so far
    int kv_waited = 0;        // key tiles whose copies were waited for
    int kv_loaded = FP8 ? 1 : (n_tiles < 2 ? n_tiles : 2);  // key tiles whose copies were issued

    for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        const int tile0 = j * kKeys;
        // ---- K/V of this tile landed; zero V rows of keys past the end (their slots are not data)
        const int nvalid = min(kKeys, a.kv_len - tile0);
        if constexpr (FP8) {
            if (!mbar_wait_bounded(bar + 8 * kBarKV0, j & 1, a.timeout_ns)) *abort_flag = 1;
            kv_waited = j + 1;
            widen_fp8(st, nvalid);
            fence_proxy_async_smem();
            __syncthreads();
            if (j + 1 < n_tiles) {
                if (tid == 0 && !*abort_flag) load_kv(j + 1);  // the staging area is free again
                kv_loaded = j + 2;
            }
        } else {
            if (!mbar_wait_bounded(bar + 8 * (kBarKV0 + st), (j >> 1) & 1, a.timeout_ns)) *abort_flag = 1;
            kv_waited = j + 1;
            if (nvalid < kKeys) {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                for (int idx = tid; idx < (kKeys - nvalid) * 16; idx += blockDim.x) {
                    const int row = nvalid + idx / 16, hf = (idx / 8) & 1, ch = idx & 7;
                    *reinterpret_cast<uint4*>(smem + kOffV + st * 2 * kHalf + hf * kHalf + row * 128 + ch * 16) = z;
                }
                fence_proxy_async_smem();
            }
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

        // ---- this thread's 64 scores; keys <= q_start + i0 are visible to every row of the CTA,
        // so only tiles past that point (or past kv_len) need per-key masks
        float v[64];
        tmem_ld64(tS + trow + col0, v);
        const bool masked = (tile0 + kKeys - 1 > a.q_start + i0) || (tile0 + kKeys > a.kv_len);
        const int lim = min(a.kv_len, qpos + 1) - tile0 - col0;  // visible keys of this row in these columns
        float mraw = -INFINITY;
        if (!masked) {
#pragma unroll
            for (int i = 0; i < 64; ++i) mraw = fmaxf(mraw, v[i]);
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) mraw = fmaxf(mraw, (i < lim) ? v[i] : -INFINITY);
        }
        row_x[half * 128 + r] = mraw;
        __syncthreads();
        // the scale is positive, so it keeps the order of the maxima
        const float mt = fmaxf(mraw, row_x[(1 - half) * 128 + r]) * a.sm_log2;

        // ---- the previous P.V has finished: O may be rescaled and P overwritten
        if (j > 0) {
            if (!mbar_wait_bounded(bar + 8 * kBarO, (j - 1) & 1, a.timeout_ns)) *abort_flag = 1;
            tc_fence_after();
            if (!FP8 && j + 1 < n_tiles) {
                if (tid == 0) load_kv(j + 1);  // its stage was read by tile j - 1
                kv_loaded = j + 2;
            }
        }
        const bool need = mt > m_ref + 8.f;
        if (j > 0 && __any_sync(kFull, need)) {
            const float m_new = need ? mt : m_ref;
            const float alpha = ex2_approx(m_ref - m_new);
            float o[64];
            tmem_ld64(tO + trow + col0, o);
#pragma unroll
            for (int i = 0; i < 64; ++i) o[i] *= alpha;
            tmem_st64(tO + trow + col0, o);
            l_run *= alpha;
            m_ref = m_new;
        } else if (need) {
            m_ref = mt;
        }

        // ---- probabilities as bf16 into this thread's swizzled 128-byte row of P half `half`
        float ls = 0.f;
        const float neg_m = -m_ref;
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
            float p0 = ex2_approx(fmaf(v[i], a.sm_log2, neg_m));
            float p1 = ex2_approx(fmaf(v[i + 1], a.sm_log2, neg_m));
            if (masked) {
                p0 = (i < lim) ? p0 : 0.f;
                p1 = (i + 1 < lim) ? p1 : 0.f;
            }
            ls += p0 + p1;
            pk[i / 2] = pack_bf16x2_rn(p0, p1);
        }
        uint8_t* prow = smem + kOffP + half * kHalf + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) * 16)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
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
            mbar_wait_bounded(bar + 8 * (kBarKV0 + (FP8 ? 0 : (t & 1))), FP8 ? (t & 1) : ((t >> 1) & 1), a.timeout_ns);
    }
    // ---- the row sum from both halves
    row_x[half * 128 + r] = l_run;
    __syncthreads();
    const float l_row = l_run + row_x[(1 - half) * 128 + r];
    if (aborted || *abort_flag) {
        if (tid == 0) raise_error(a.err, PKV_DEVERR_TIMEOUT);
    } else {
        // ---- out = O / l for this row's 64 head dims
        const float inv = l_row > 0.f ? a.out_mul / l_row : 0.f;
        const int g = r % a.G;
        uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) +
                        ((static_cast<size_t>(qi) * a.Hq + static_cast<size_t>(h) * a.G + g) * 128 + col0) * 2;
        float o[64];
        tmem_ld64(tO + trow + col0, o);  // warp-collective: every lane loads, valid rows store
        if (qi < a.NQ) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                uint4 w;
                w.x = pack_bf16x2_rn(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
                w.y = pack_bf16x2_rn(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
                w.z = pack_bf16x2_rn(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
                w.w = pack_bf16x2_rn(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
                *reinterpret_cast<uint4*>(orow + q4 * 16) = w;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

size_t prefill_smem_bytes(bool fp8) {
    return static_cast<size_t>(fp8 ? off_bar<true>() : off_bar<false>()) + 128 + 1024 + 1024;
}

cudaError_t launch_paged_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const PrefillArgs& a, int narrow, cudaStream_t stream) {
    const size_t smem = prefill_smem_bytes(narrow != 0);
    auto kern = narrow == 2 ? paged_prefill_kernel<2> : (narrow == 1 ? paged_prefill_kernel<1> : paged_prefill_kernel<0>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int rows_q = kRows / a.G;
    dim3 grid((a.NQ + rows_q - 1) / rows_q, a.Hkv);
    kern<<<grid, 256, smem, stream>>>(qmap, kmap, vmap, a);
    return cudaGetLastError();
}

}  // namespace pkv
