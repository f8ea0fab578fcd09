// prefill_ws.cu -- chunked-prefill attention over bf16 caches, warp-specialised.
//
// Method ("3.3 批处理与内存管理", section "分块预填充"): the query tokens of a
// chunk attend causally to the sequence's paged KV cache, which already holds
// the earlier chunks and (written first) the chunk's own keys.  Several
// chunks of different sequences can go in one launch (varlen): chunk s has
// query tokens [cu_q[s], cu_q[s+1]) at positions q_start[s] + i and kv_len[s]
// cached keys.
//
// A CTA owns 128 query rows (128 / G tokens x the G query heads of one KV
// head) of one chunk and walks the chunk's keys in tiles of 128:
//   * warp 8 (producer) copies K and V tiles with TMA (128-byte swizzle,
//     one block of the block table per copy) into separate rings (K three
//     deep, V two deep), reading the block table one tile ahead;
//   * warp 9 (one thread) issues the tcgen05 MMAs: S(j+1) = Q K(j+1)^T into
//     the other of two TMEM S buffers as soon as its keys land, then
//     O += P(j) V(j) with P read from TMEM once the softmax of tile j is done
//     -- so the tensor pipe computes the next scores while the softmax works;
//   * warps 0-7 (softmax) each own 64 columns of 32 rows: row maximum over
//     the two halves of a row (pair barrier), exp2, bf16 P written to one of
//     two TMEM P buffers, running sums.  O in TMEM is rescaled only when a
//     row's maximum grows by more than 8 (log2 units); only then does the
//     softmax wait for the previous P.V.
// Hand-offs are mbarriers (no CTA-wide barrier inside the loop).  Every wait
// is bounded; on timeout a role records the error and leaves its loop, the
// CTA drains its own MMAs and copies (bounded) and frees TMEM.
#include "prefill.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128, kKeys = 128, kHalf = 16384;
constexpr int kKStages = 3, kVStages = 2;
constexpr int kOffQ = 0;                                  // 2 halves of 64 head dims
constexpr int kOffK = kOffQ + 2 * kHalf;                  // kKStages x 2 halves
constexpr int kOffV = kOffK + kKStages * 2 * kHalf;       // kVStages x 2 halves
constexpr int kOffMeta = kOffV + kVStages * 2 * kHalf;    // barriers, TMEM address, flags, row exchange, tile counts
constexpr int kTmemCols = 512;  // S0: 0..127, S1: 128..255, O: 256..383, P0: 384..447, P1: 448..511
constexpr int kColO = 256, kColP = 384;
constexpr int kSoftmax = 256;   // softmax threads (warps 0-7)
constexpr int kThreads = 320;   // + producer warp 8 + MMA warp 9
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, true);

// mbarrier slots (8 bytes each)
constexpr int kBarKFull = 0;    // + stage (3): K copies landed (producer, expect_tx)
constexpr int kBarKEmpty = 3;   // + stage (3): S of the tile in that stage done (MMA commit)
constexpr int kBarVFull = 6;    // + stage (2): V copies landed
constexpr int kBarVEmpty = 8;   // + stage (2): P.V of the tile in that stage done (MMA commit)
constexpr int kBarSFull = 10;   // + buffer: S written (MMA commit)
constexpr int kBarSEmpty = 12;  // + buffer: S read by all softmax threads (256 arrivals)
constexpr int kBarPFull = 14;   // + buffer: P written (and O rescaled) by all softmax threads (256 arrivals)
constexpr int kBarODone = 16;   // + buffer: O += P V of the tile using that P buffer done (MMA commit)
constexpr int kBarQFull = 18;   // Q landed
constexpr int kBarPair = 19;    // + 2 * quad + parity: the two warps of a row quadrant exchanged (64 arrivals)
constexpr int kBarDrain = 27;   // final commit of the MMA thread
constexpr int kNumBars = 28;
constexpr int kMaxSeqs = 2048;  // chunks per launch (tile counts are kept in shared memory)
static_assert(8 * kNumBars <= 232, "barrier slots overlap the TMEM address slot");

__device__ __forceinline__ void tma_load_3d_nohint(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                   uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}


}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_ws_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int rows_q = kRows / a.G;

    const uint32_t bar = sb + kOffMeta;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMeta + 232);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMeta + 236);
    int* tile_info = reinterpret_cast<int*>(smem + kOffMeta + 240);   // s, i0 of this CTA (or -1)
    float* row_x = reinterpret_cast<float*>(smem + kOffMeta + 256);    // [2 parity][2 half][128]
    int* tcount = reinterpret_cast<int*>(smem + kOffMeta + 256 + 2048);  // prefix of tiles per chunk

    // ---- which chunk and which 128 rows: chunk s covers tiles [tcount[s], tcount[s+1]) of the grid
    const bool single = a.cu_q == nullptr;  // one chunk described by the scalar fields
    if (single) {
        if (tid == 0) {
            const int nt = (a.NQ + rows_q - 1) / rows_q;
            const int t = blockIdx.x;
            tile_info[0] = t < nt ? 0 : -1;
            tile_info[1] = (nt - 1 - t) * rows_q;  // heaviest (latest) tiles first
        }
    } else {
        // tiles per chunk, then an exclusive prefix over the chunks: each thread takes a contiguous run
        // of chunks, a warp scan joins the runs, a second pass writes the prefix
        int* part = reinterpret_cast<int*>(row_x);  // per-warp totals (row_x is free until the main loop)
        const int per = (a.nseq + kThreads - 1) / kThreads;
        const int c_lo = min(tid * per, a.nseq), c_hi = min(c_lo + per, a.nseq);
        int sum = 0;
        for (int c = c_lo; c < c_hi; ++c) {
            const int q0 = a.cu_q[c], q1 = a.cu_q[c + 1];
            const bool bad = q0 < 0 || q1 < q0 || q1 > a.NQ;
            if (bad) raise_error(a.err, PKV_DEVERR_BAD_LENGTH);
            const int nt = bad ? 0 : (q1 - q0 + rows_q - 1) / rows_q;
            tcount[c + 1] = nt;
            sum += nt;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) part[warp] = incl;
        __syncthreads();
        int run = incl - sum;
        for (int w = 0; w < warp; ++w) run += part[w];
        for (int c = c_lo; c < c_hi; ++c) {
            run += tcount[c + 1];
            tcount[c + 1] = run;
        }
        if (tid == 0) tcount[0] = 0;
        __syncthreads();
        if (tid == 0) {
            const int t = blockIdx.x;
            if (t == 0 && tcount[a.nseq] > static_cast<int>(gridDim.x)) raise_error(a.err, PKV_DEVERR_BAD_LENGTH);
            int s = -1;
            if (t < tcount[a.nseq]) {
                int lo = 0, hi = a.nseq - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (tcount[mid] <= t) lo = mid; else hi = mid - 1;
                }
                s = lo;
            }
            tile_info[0] = s;
            if (s >= 0) {
                const int nt = tcount[s + 1] - tcount[s];
                tile_info[1] = (nt - 1 - (t - tcount[s])) * rows_q;
            }
        }
    }
    __syncthreads();
    const int s = tile_info[0];
    if (s < 0) return;  // the whole CTA leaves together, before any TMEM or barrier work
    const int i0 = tile_info[1];

    // this chunk's geometry
    const int q_base = single ? 0 : a.cu_q[s];
    const int NQ = single ? a.NQ : a.cu_q[s + 1] - q_base;
    const int q_start = single ? a.q_start : a.q_starts[s];
    const int kv_len = single ? a.kv_len : a.kv_lens[s];
    const int32_t* table = single ? a.block_table : a.block_table + static_cast<size_t>(s) * a.MB;
    const int n_table = (kv_len + a.S - 1) / a.S;
    if (kv_len < q_start + NQ || q_start < 0 || n_table > (single ? a.n_table : a.MB)) {
        if (tid == 0) raise_error(a.err, PKV_DEVERR_BAD_LENGTH);
        return;
    }
    const int last_q = min(i0 + rows_q, NQ) - 1;
    const int max_key = min(kv_len - 1, q_start + last_q);
    const int n_tiles = max_key / kKeys + 1;
    const int blocks_per_tile = kKeys / a.S;

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool many = (i >= kBarSEmpty && i < kBarSEmpty + 2) || (i >= kBarPFull && i < kBarPFull + 2);
            const bool pair = i >= kBarPair && i < kBarPair + 8;
            mbar_init(bar + 8 * i, many ? kSoftmax : (pair ? 64 : 1));
        }
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
    const uint32_t tO = tmem + kColO;

    if (warp == 8) {
        // ------------------------------------------------ producer: Q, then K and V tiles ahead of use
        if (lane == 0) {
            prefetch_tensormap(&qmap);
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            mbar_arrive_expect_tx(bar + 8 * kBarQFull, 2 * kHalf);
            tma_load_3d_nohint(sb + kOffQ, &qmap, 0, h * a.G, q_base + i0, bar + 8 * kBarQFull);
            tma_load_3d_nohint(sb + kOffQ + kHalf, &qmap, 64, h * a.G, q_base + i0, bar + 8 * kBarQFull);
            // rows of the pool for the blocks of one tile (beyond the pool: the copy fills zeros)
            auto tile_rows = [&](int j, int (&c2)[kKeys / 8]) {
#pragma unroll
                for (int bi = 0; bi < kKeys / 8; ++bi) {
                    const int idx = j * blocks_per_tile + bi;
                    c2[bi] = (bi < blocks_per_tile && idx < n_table) ? table[idx] : -1;
                }
#pragma unroll
                for (int bi = 0; bi < kKeys / 8; ++bi) {
                    const int idx = j * blocks_per_tile + bi;
                    int r = a.NB * a.S;
                    if (bi < blocks_per_tile && idx < n_table) {
                        if (c2[bi] >= 0 && c2[bi] < a.NB) r = c2[bi] * a.S;
                        else raise_error(a.err, PKV_DEVERR_BAD_BLOCK);
                    }
                    c2[bi] = r;
                }
            };
            int rows[kKeys / 8];
            tile_rows(0, rows);
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int ks = j % kKStages, vs = j % kVStages;
                if (j >= kKStages &&
                    !mbar_wait_bounded(bar + 8 * (kBarKEmpty + ks), (j / kKStages - 1) & 1, a.timeout_ns)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const uint32_t kb = bar + 8 * (kBarKFull + ks);
                mbar_arrive_expect_tx(kb, 2 * kHalf);
                for (int bi = 0; bi < blocks_per_tile; ++bi) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_3d_nohint(sb + kOffK + ks * 2 * kHalf + hf * kHalf + bi * a.S * 128, &kmap, hf * 64,
                                           h, rows[bi], kb);
                }
                k_issued = j + 1;
                if (j >= kVStages &&
                    !mbar_wait_bounded(bar + 8 * (kBarVEmpty + vs), (j / kVStages - 1) & 1, a.timeout_ns)) {
                    *abort_flag = 1;
                    break;
                }
                const uint32_t vb = bar + 8 * (kBarVFull + vs);
                mbar_arrive_expect_tx(vb, 2 * kHalf);
                for (int bi = 0; bi < blocks_per_tile; ++bi) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_3d_nohint(sb + kOffV + vs * 2 * kHalf + hf * kHalf + bi * a.S * 128, &vmap, hf * 64,
                                           h, rows[bi], vb);
                }
                v_issued = j + 1;
                if (j + 1 < n_tiles) tile_rows(j + 1, rows);  // the table read overlaps the next waits
            }
            // its own copies have landed before the CTA may finish (bounded)
            for (int t = k_issued - kKStages < 0 ? 0 : k_issued - kKStages; t < k_issued; ++t)
                mbar_wait_bounded(bar + 8 * (kBarKFull + t % kKStages), (t / kKStages) & 1, a.timeout_ns);
            for (int t = v_issued - kVStages < 0 ? 0 : v_issued - kVStages; t < v_issued; ++t)
                mbar_wait_bounded(bar + 8 * (kBarVFull + t % kVStages), (t / kVStages) & 1, a.timeout_ns);
            mbar_wait_bounded(bar + 8 * kBarQFull, 0, a.timeout_ns);
        }
    } else if (warp == 9) {
        // ------------------------------------------------ MMA issuer (one thread)
        if (lane == 0) {
            auto issue_s = [&](int j) {
                const int ks = j % kKStages;
                const uint32_t tS = tmem + 128 * (j & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t hf = kk >> 2, koff = (kk & 3) * 32;
                    const uint64_t ad = smem_desc_sw128(sb + kOffQ + hf * kHalf + koff, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(sb + kOffK + ks * 2 * kHalf + hf * kHalf + koff, 16, 1024);
                    tc_mma_f16(tS, ad, bd, kIdescS, kk > 0);
                }
                tc_commit(bar + 8 * (kBarSFull + (j & 1)));
                tc_commit(bar + 8 * (kBarKEmpty + ks));
            };
            bool ok = mbar_wait_bounded(bar + 8 * kBarQFull, 0, a.timeout_ns) &&
                      mbar_wait_bounded(bar + 8 * kBarKFull, 0, a.timeout_ns);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles) {
                    const int n = j + 1, b = n & 1;
                    ok = mbar_wait_bounded(bar + 8 * (kBarKFull + n % kKStages), (n / kKStages) & 1, a.timeout_ns) &&
                         (n < 2 || mbar_wait_bounded(bar + 8 * (kBarSEmpty + b), ((n - 2) >> 1) & 1, a.timeout_ns));
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(n);
                }
                const int b = j & 1, vs = j % kVStages;
                ok = mbar_wait_bounded(bar + 8 * (kBarPFull + b), (j >> 1) & 1, a.timeout_ns) &&
                     mbar_wait_bounded(bar + 8 * (kBarVFull + vs), (j / kVStages) & 1, a.timeout_ns);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t bd = smem_desc_sw128(sb + kOffV + vs * 2 * kHalf + kk * 2048, kHalf, 1024);
                    tc_mma_f16_ts(tO, tmem + kColP + 64 * b + 8 * kk, bd, kIdescPV, (j > 0) || (kk > 0));
                }
                tc_commit(bar + 8 * (kBarODone + b));
                tc_commit(bar + 8 * (kBarVEmpty + vs));
            }
            if (!ok) *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------ softmax warps 0-7
        const int quad = warp & 3, half = warp >> 2;
        const int r = quad * 32 + lane;
        const int qi = i0 + r / a.G;
        const int qpos = q_start + qi;
        const uint32_t trow = static_cast<uint32_t>(quad * 32) << 16;
        const int col0 = half * 64;
        float m_ref = -INFINITY, l_run = 0.f;
        int done = 0;  // tiles whose P was handed over
        // exchange a value with the other warp of this row quadrant (bounded wait)
        auto exchange = [&](int k, float mine, float* rx) -> float {
            rx[half * 128 + r] = mine;
            const uint32_t pb = bar + 8 * (kBarPair + 2 * quad + (k & 1));
            mbar_arrive(pb);
            if (!__all_sync(kFull, mbar_wait_bounded(pb, (k >> 1) & 1, a.timeout_ns))) *abort_flag = 1;
            return rx[(1 - half) * 128 + r];
        };
        // P.V of tile t (which used P buffer t & 1) has completed
        auto wait_pv = [&](int t) -> bool {
            return __all_sync(kFull, mbar_wait_bounded(bar + 8 * (kBarODone + (t & 1)), (t >> 1) & 1, a.timeout_ns));
        };
        for (int j = 0; j < n_tiles; ++j) {
            if (__any_sync(kFull, *abort_flag != 0)) break;
            const int b = j & 1;
            const int tile0 = j * kKeys;
            if (!__all_sync(kFull, mbar_wait_bounded(bar + 8 * (kBarSFull + b), (j >> 1) & 1, a.timeout_ns))) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            float v[64];
            tmem_ld64(tmem + 128 * b + trow + col0, v);
            tc_fence_before();
            mbar_arrive(bar + 8 * (kBarSEmpty + b));
            const bool masked = (tile0 + kKeys - 1 > q_start + i0) || (tile0 + kKeys > kv_len);
            const int lim = min(kv_len, qpos + 1) - tile0 - col0;
            float mraw = -INFINITY;
            if (!masked) {
#pragma unroll
                for (int i = 0; i < 64; ++i) mraw = fmaxf(mraw, v[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) mraw = fmaxf(mraw, (i < lim) ? v[i] : -INFINITY);
            }
            const float other = exchange(j, mraw, row_x + (j & 1) * 256);
            const float mt = fmaxf(mraw, other) * a.sm_log2;
            const bool need = mt > m_ref + 8.f;
            if (j > 0 && __any_sync(kFull, need)) {
                // O may be rescaled only once the previous P.V is done (none is in flight then)
                if (!wait_pv(j - 1)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
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
                pk[i / 2] = bf16x2_rn(p0, p1);
            }
            l_run += ls;
            // P buffer b is free once P.V of tile j - 2 is done
            if (j >= 2 && !wait_pv(j - 2)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            tmem_st32u(tmem + kColP + 64 * b + trow + half * 32, pk);
            // keys past kv_len in this tile: their V rows are not data, make them zero once they have landed
            const int nvalid = min(kKeys, kv_len - tile0);
            if (nvalid < kKeys) {
                const int vs = j % kVStages;
                if (!__all_sync(kFull, mbar_wait_bounded(bar + 8 * (kBarVFull + vs), (j / kVStages) & 1,
                                                         a.timeout_ns))) {
                    *abort_flag = 1;
                    break;
                }
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                for (int idx = tid; idx < (kKeys - nvalid) * 16; idx += kSoftmax) {
                    const int row = nvalid + idx / 16, hf = (idx / 8) & 1, ch = idx & 7;
                    *reinterpret_cast<uint4*>(smem + kOffV + vs * 2 * kHalf + hf * kHalf + row * 128 + ch * 16) = z;
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(bar + 8 * (kBarPFull + b));
            done = j + 1;
        }
        // ---- the last P.V, the row sum over both halves, out = O / l
        bool ok = !__any_sync(kFull, *abort_flag != 0) && done == n_tiles && wait_pv(n_tiles - 1);
        tc_fence_after();
        const float l_row = l_run + (ok ? exchange(n_tiles, l_run, row_x + (n_tiles & 1) * 256) : 0.f);
        float o[64];
        tmem_ld64(tO + trow + col0, o);  // warp-collective: every lane loads, valid rows store
        if (ok && qi < NQ) {
            const float inv = l_row > 0.f ? a.out_mul / l_row : 0.f;
            const int g = r % a.G;
            uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) +
                            ((static_cast<size_t>(q_base + qi) * a.Hq + static_cast<size_t>(h) * a.G + g) * 128 + col0) * 2;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                uint4 w;
                w.x = bf16x2_rn(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
                w.y = bf16x2_rn(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
                w.z = bf16x2_rn(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
                w.w = bf16x2_rn(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
                *reinterpret_cast<uint4*>(orow + q4 * 16) = w;
            }
        }
        if (!ok) *abort_flag = 1;
    }

    // ---- drain: nothing of this CTA may still be in flight when TMEM is freed and the CTA exits
    if (warp == 9 && lane == 0) {
        tc_commit(bar + 8 * kBarDrain);  // arrives once every MMA issued so far has completed
        mbar_wait_bounded(bar + 8 * kBarDrain, 0, a.timeout_ns);
    }
    __syncthreads();
    if (*abort_flag && tid == 0) raise_error(a.err, PKV_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

size_t prefill_ws_smem_bytes() { return static_cast<size_t>(kOffMeta) + 256 + 2048 + 4 * (kMaxSeqs + 1) + 1024; }

int prefill_ws_max_seqs() { return kMaxSeqs; }

cudaError_t launch_paged_prefill_ws(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                    const PrefillArgs& a, int grid_x, cudaStream_t stream) {
    const size_t smem = prefill_ws_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(grid_x, a.Hkv);
    paged_prefill_ws_kernel<<<grid, kThreads, smem, stream>>>(qmap, kmap, vmap, a);
    return cudaGetLastError();
}

}  // namespace pkv
