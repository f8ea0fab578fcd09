// prefill_tile.cuh -- the chunked-prefill tile (warp-specialised, tcgen05/TMEM) as a device function, shared by
// the prefill kernels (prefill_ws.cu) and the mixed-step kernel (mixed_*.cu).
//
// Method ("3.3 批处理与内存管理", section "分块预填充"): the query tokens of a
// chunk attend causally to the sequence's paged KV cache, which already holds
// the earlier chunks and (written first) the chunk's own keys.  Several
// chunks of different sequences can go in one launch (varlen): chunk s has
// query tokens [cu_q[s], cu_q[s+1]) at positions q_start[s] + i and kv_len[s]
// cached keys.
//
// A CTA owns two tiles of 128 query rows (each 128 / G tokens x the G query
// heads of one KV head) of one chunk, A and B, and walks the chunk's keys in
// tiles of 64, each K/V tile serving both query tiles.  TMEM holds, per
// query tile, two score buffers (fp32, 64 keys; the bf16 P of a key tile is
// written over the first half of its own score buffer) and the output
// accumulator O (fp32, 128 dims):
//   * warps 8 and 10 (producers) copy Q once and the K tiles (warp 8) and the
//     V tiles (warp 10) with TMA (128-byte swizzle, one block of the block
//     table per copy, one lane per block) into two 4-deep rings; block-table
//     entries are read 32 at a time, a batch ahead.  FP8 codes go the same way
//     into 6-deep rings of 128-byte lines and feed 8-bit MMAs directly (query
//     rows and probabilities split into two E4M3 parts).  INT8 codes go to a
//     two-slot staging ring per operand and are widened to f16 into a 3-deep
//     ring: by the producer alone when both query tiles are live, else half
//     the rows by the producer and half by the MMA warp that consumes the
//     operand; their MMAs run on f16 operands (Q converted in place once, P
//     packed as f16);
//   * warps 9 and 11 issue the tcgen05 MMAs (each warp runs its loop, one
//     elected lane issues): warp 9 S_A(j), S_B(j) into the buffers that
//     P(j-2) was read from, as soon as P(j-2).V has completed; warp 11
//     P_A(j).V(j), P_B(j).V(j) once the softmax of tile j is done.  So the
//     scores of the next tile are computed while the softmax works, and
//     neither kind of MMA waits behind the other's issue;
//   * warps 0-3 (query tile A) and 4-7 (tile B): one thread per row reads its
//     64 scores, keeps the running maximum and sum, writes bf16 P over them,
//     and rescales its O row (after the previous P.V has completed) only
//     when the row maximum grows by more than 8 (log2 units).
// Hand-offs are mbarriers, one per buffer where a phase could otherwise be
// overtaken; every wait is bounded; on timeout a role records the error and
// leaves its loop, the CTA drains its own MMAs and copies (bounded) and
// frees TMEM.
#pragma once

#include <type_traits>

#include "prefill.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128, kKeys = 64;
constexpr int kQHalf = kRows * 128;            // 64 head dims of 128 rows, bytes
constexpr int kKvHalf = kKeys * 128;           // 64 head dims of 64 keys, bytes (bf16)
constexpr int kStgSlot = kKeys * 128;          // one key tile of one-byte codes (128 head dims), bytes
constexpr int kOffQ = 0;                       // tile A: 2 halves, tile B: 2 halves

// Shared-memory plan per cache kind (NARROW: 0 bf16, 1 FP8 E4M3 codes, 2 INT8 codes).  bf16 tiles and FP8 codes
// go straight from TMA into the K and V rings that the MMAs read (FP8: one 128-byte line of codes per key, 8 KB
// per 64-key stage).  INT8 codes land in a two-slot staging ring per operand and are widened to f16 by the
// producer (and MMA) warps into the rings.
template <int NARROW>
struct Plan {
    static constexpr int kStages = NARROW == 0 ? 4 : NARROW == 1 ? 6 : 3;  // K and V ring depth
    static constexpr int kStage = NARROW == 1 ? kStgSlot : 2 * kKvHalf;   // bytes of one ring stage
    static constexpr int kOffK = kOffQ + 4 * kQHalf;
    static constexpr int kOffV = kOffK + kStages * kStage;
    static constexpr int kOffStg = kOffV + kStages * kStage;            // INT8: K 2 slots, then V 2 slots
    static constexpr int kOffMeta = kOffStg + (NARROW == 2 ? 4 * kStgSlot : 0);
};
constexpr int kMaxStages = 6;
constexpr int kTmemCols = 512;
constexpr int kColS = 0;     // + 128 * tile + 64 * buffer: scores (fp32, 64 keys); P over the first 32 columns
constexpr int kColO = 256;   // + 128 * tile: output accumulator (fp32, 128 dims)
constexpr int kSoftmax = 256;
constexpr int kThreads = 384;  // + producer warps 8 (K) and 10 (V), MMA warps 9 (S) and 11 (P.V)
// Instruction descriptor for kind::f16 with f16 A and B (bits 7-9 = 0, 10-12 = 0; bf16 sets both to 1), fp32
// accumulator, A K-major, B K- or MN-major (bit 16), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t idesc_f16_f32(int M, int N, bool b_mn_major) {
    return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
// MMA operand types: bf16 for bf16 caches; f16 for one-byte caches (their codes widen to f16 in one step, and Q
// and P are taken to f16 to match)
template <int NARROW>
constexpr uint32_t kIdescS = NARROW ? idesc_f16_f32(128, kKeys, false) : idesc_bf16_f32(128, kKeys, false);
template <int NARROW>
constexpr uint32_t kIdescPV = NARROW ? idesc_f16_f32(128, 128, true) : idesc_bf16_f32(128, 128, true);
// kind::f8f6f4 with E4M3 A and B (type fields 0): the same bit pattern as the f16 descriptor above
constexpr uint32_t kIdescS8 = idesc_f16_f32(128, kKeys, false);
constexpr uint32_t kIdescPV8 = idesc_f16_f32(128, 128, true);
// FP8 caches: the running maximum is set 4 (log2 units) below a new row maximum, so that the probabilities reach
// up to 2^4..2^8 and their two E4M3 parts keep full precision for smaller values
constexpr float kP8Shift = 4.f;

// mbarrier slots (8 bytes each); "tb" = 2 * tile + buffer
constexpr int kBarKFull = 0;                         // + stage: K in the bf16 ring (copies landed / widened)
constexpr int kBarKEmpty = kBarKFull + kMaxStages;   // + stage: the S MMAs that read it done
constexpr int kBarVFull = kBarKEmpty + kMaxStages;   // + stage: V in the bf16 ring
constexpr int kBarVEmpty = kBarVFull + kMaxStages;   // + stage: the P.V MMAs that read it done
constexpr int kBarSFull = kBarVEmpty + kMaxStages;   // + tb: S written
constexpr int kBarPFull = kBarSFull + 4;          // + tb: P written, O rescaled (128 arrivals)
constexpr int kBarPVDone = kBarPFull + 4;         // + tb: P.V of the key tile that used buffer b done
constexpr int kBarQFull = kBarPVDone + 4;
constexpr int kBarFinal = kBarQFull + 1;          // every MMA done
constexpr int kBarDrain = kBarFinal + 1;          // after an abort: every MMA issued so far done
constexpr int kBarStg = kBarDrain + 1;            // + 2 * (V ? 1 : 0) + slot: one-byte codes landed in staging
constexpr int kBarStgFree = kBarStg + 4;          // + 2 * (V ? 1 : 0) + slot: the MMA warp's half of it widened
constexpr int kBarQConv = kBarStgFree + 4;        // one-byte caches: Q converted to f16 (8 softmax warps)
constexpr int kNumBars = kBarQConv + 1;
constexpr int kMetaTmem = 8 * kNumBars;           // TMEM base address
constexpr int kMetaAbort = kMetaTmem + 4;
constexpr int kMetaTile = kMetaAbort + 4;         // chunk, first token (or -1)
constexpr int kMetaPart = kMetaTile + 8;          // per-warp partial sums of the CTA-count scan
constexpr int kMetaCount = 512;                   // CTAs per chunk, prefix
constexpr int kMaxSeqs = 2048;                    // chunks per launch
static_assert(kMetaPart + 4 * (kThreads / 32) <= kMetaCount, "meta slots overlap");

__device__ __forceinline__ void tma_load_3d_nohint(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                   uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// two E4M3 codes in the low 16 bits of w (low byte first) -> f16x2, exactly
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_u(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(w)));
    return r;
}

// f16x2 -> two floats (exact)
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
    float lo, hi;
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
    return make_float2(lo, hi);
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// f16x2 -> two E4M3 codes (low half to the low byte), round to nearest even, saturating to +-448
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
    return r;
}

// two floats -> two E4M3 codes (lo to the low byte), round to nearest even, saturating
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// A value x split into two E4M3 codes, hi = E4M3(x) and lo = E4M3(x - hi): hi + lo carries about 8 significant
// bits (a bf16 value exactly, when lo stays in E4M3's normal range).  Four f16 values (two f16x2 words, lowest
// first) give one 32-bit word of four hi codes and one of four lo codes.
__device__ __forceinline__ void split_e4m3x4(uint32_t h01, uint32_t h23, uint32_t& hi, uint32_t& lo) {
    const uint32_t a = f16x2_to_e4m3x2(h01), b = f16x2_to_e4m3x2(h23);
    uint32_t ra, rb;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(ra) : "r"(h01), "r"(e4m3x2_to_f16x2_u(a)));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(rb) : "r"(h23), "r"(e4m3x2_to_f16x2_u(b)));
    hi = a | (b << 16);
    lo = f16x2_to_e4m3x2(ra) | (f16x2_to_e4m3x2(rb) << 16);
}


// Signed bytes i0, i0 + 1 of w -> f16x2, exactly.  f = w ^ 0x80808080 holds u = byte + 128; u placed in the low
// mantissa bits of 0x6400 (1024) reads 1024 + u, and one packed subtraction of 1152 leaves the byte's value.
__device__ __forceinline__ uint32_t s8x2_to_f16x2(uint32_t f, int i0) {
    const uint32_t h = __byte_perm(f, 0x64646464u, 0x5040u | (static_cast<uint32_t>(i0 + 1) << 8) |
                                                        static_cast<uint32_t>(i0));
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}

}  // namespace

// One tile of the warp-specialised chunked-prefill kernel, run by all 384 threads of a CTA: query-tile slot tile_x
// (of grid_x slots; the varlen form maps slots to chunks) of KV head h, with the CTA's dynamic shared memory at
// smem_raw.  ADAPT (INT8 caches, varlen launches): each CTA chooses split widening when only its query tile A is
// live.  REUSE: the CTA goes on to other work afterwards, so the tile's mbarriers are invalidated before it returns.
template <int NARROW, bool ADAPT, bool REUSE>
__device__ __forceinline__ void prefill_tile(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                             const PrefillArgs& a, int tile_x, int h, int grid_x, uint8_t* smem_raw) {
    constexpr int kStages = Plan<NARROW>::kStages, kOffK = Plan<NARROW>::kOffK, kOffV = Plan<NARROW>::kOffV;
    constexpr int kOffStg = Plan<NARROW>::kOffStg, kOffMeta = Plan<NARROW>::kOffMeta, kStage = Plan<NARROW>::kStage;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows_q = kRows / a.G;    // tokens per query tile
    const int cta_q = 2 * rows_q;      // tokens per CTA

    const uint32_t bar = sb + kOffMeta;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMeta + kMetaTmem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMeta + kMetaAbort);
    int* tile_info = reinterpret_cast<int*>(smem + kOffMeta + kMetaTile);
    int* part = reinterpret_cast<int*>(smem + kOffMeta + kMetaPart);
    int* tcount = reinterpret_cast<int*>(smem + kOffMeta + kMetaCount);

    // ---- which chunk and which tokens: chunk s covers CTAs [tcount[s], tcount[s+1]) of the grid
    const bool single = a.cu_q == nullptr;  // one chunk described by the scalar fields
    if (single) {
        if (tid == 0) {
            const int nt = (a.NQ + cta_q - 1) / cta_q;
            const int t = tile_x;
            tile_info[0] = t < nt ? 0 : -1;
            tile_info[1] = (nt - 1 - t) * cta_q;  // heaviest (latest) tokens first
        }
    } else {
        // CTAs per chunk, then an exclusive prefix over the chunks: each thread takes a contiguous run
        // of chunks, a warp scan joins the runs, a second pass writes the prefix
        const int per = (a.nseq + kThreads - 1) / kThreads;
        const int c_lo = min(tid * per, a.nseq), c_hi = min(c_lo + per, a.nseq);
        int sum = 0;
        for (int c = c_lo; c < c_hi; ++c) {
            const int q0 = a.cu_q[c], q1 = a.cu_q[c + 1];
            const bool bad = q0 < 0 || q1 < q0 || q1 > a.NQ;
            if (bad) raise_error(a.err, PKV_DEVERR_BAD_LENGTH);
            const int nt = (bad || c < a.first_chunk) ? 0 : (q1 - q0 + cta_q - 1) / cta_q;
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
            const int t = tile_x;
            if (t == 0 && tcount[a.nseq] > grid_x) raise_error(a.err, PKV_DEVERR_BAD_LENGTH);
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
                tile_info[1] = (nt - 1 - (t - tcount[s])) * cta_q;
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
    const bool has_b = i0 + rows_q < NQ;  // query tile B holds at least one token of the chunk
    const int last_q = min(i0 + cta_q, NQ) - 1;
    const int max_key = min(kv_len - 1, q_start + last_q);
    const int n_tiles = max_key / kKeys + 1;
    const int blocks_per_tile = kKeys / a.S;
    // One-byte caches: with both query tiles live the tensor pipe has work enough to hide the widening and the
    // producer widens every row, leaving the MMA warps to issue; in a varlen launch a CTA with tile A alone (a
    // decode token) has the MMA warps also widen half of the rows of the operand they consume.  Single-chunk
    // launches compile the producer-only form alone.
    const bool split = NARROW == 2 && ADAPT && !has_b;

    if (tid == 0) {
        // the bf16 instance never waits on the staging-free barriers
        for (int i = 0; i < (NARROW ? kNumBars : kBarStgFree); ++i) {
            int count = (i >= kBarPFull && i < kBarPFull + 4) ? kSoftmax / 2 : i == kBarDrain ? 2 : 1;
            if (i == kBarQConv) count = kSoftmax / 32;
            // split widening: an f16 K or V stage is complete when both warps widened their halves
            if (split && ((i >= kBarKFull && i < kBarKFull + kMaxStages) || (i >= kBarVFull && i < kBarVFull + kMaxStages)))
                count = 2;
            mbar_init(bar + 8 * i, count);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        if constexpr (!REUSE) tmem_relinquish();  // a reused CTA allocates again for its next tile
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // INT8 caches: widen rows rr * 32 + lane of key tile `slot` of the K (or V) staging ring into f16 stage st
    // (exact: every INT8 code is an f16 value; the per-tensor or per-head scales go to the scores and the
    // output).  128 codes per key row, in 128-byte swizzled lines like the 16-bit halves.  With split widening
    // each of the two warps that serve an operand (its producer and its MMA warp) widens one half of the rows.
    auto widen_rows = [&](bool is_v, int slot, int st, int rr) {
        const uint8_t* src = smem + kOffStg + ((is_v ? 2 : 0) + slot) * kStgSlot;
        uint8_t* dstb = smem + (is_v ? kOffV : kOffK) + st * kStage;
        const int r = lane + 32 * rr, sw = r & 7;
        src += r * 128;
        uint8_t* dst = dstb + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16 codes: head dims 16c .. 16c + 15
            const uint4 wv = *reinterpret_cast<const uint4*>(src + ((c ^ sw) * 16));
            const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t f = ws[i] ^ 0x80808080u;
                o[2 * i] = s8x2_to_f16x2(f, 0);
                o[2 * i + 1] = s8x2_to_f16x2(f, 2);
            }
            uint8_t* dh = dst + (c >> 2) * kKvHalf;
            const int lc = 2 * (c & 3);
            *reinterpret_cast<uint4*>(dh + ((lc ^ sw) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dh + (((lc + 1) ^ sw) * 16)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
    };

    if (warp == 8 || warp == 10) {
        // ------------------------------------------------ producer warps: warp 8 copies Q and the K tiles,
        // warp 10 the V tiles.  Block-table entries come 32 at a time (one per lane, the next batch loaded a
        // batch ahead) and are handed out by shuffle; lane bi issues the copies of block bi of a key tile.
        const bool is_v = warp == 10;
        if (!is_v && lane == 0) {
            prefetch_tensormap(&qmap);
            prefetch_tensormap(&kmap);
            const uint32_t qb = bar + 8 * kBarQFull;
            mbar_arrive_expect_tx(qb, (has_b ? 4 : 2) * kQHalf);
            for (int t = 0; t < (has_b ? 2 : 1); ++t)
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_3d_nohint(sb + kOffQ + (2 * t + hf) * kQHalf, &qmap, hf * 64, h * a.G,
                                       q_base + i0 + t * rows_q, qb);
        }
        if (is_v && lane == 0) prefetch_tensormap(&vmap);
        const CUtensorMap* map = is_v ? &vmap : &kmap;
        const int full = is_v ? kBarVFull : kBarKFull, empty = is_v ? kBarVEmpty : kBarKEmpty;
        const uint32_t dst0 = sb + (is_v ? kOffV : kOffK);
        auto entry = [&](int idx) { return idx < n_table ? __ldg(table + idx) : -1; };
        int cur_c = 0, cur = entry(lane), nxt = entry(32 + lane);
        // this lane's pool row for block `lane` of key tile jj (tiles asked for in increasing order)
        auto tile_row = [&](int jj) {
            const int idx0 = jj * blocks_per_tile;  // blocks_per_tile divides 32: a tile stays in one batch
            if ((idx0 >> 5) != cur_c) {
                cur = nxt;
                cur_c = idx0 >> 5;
                nxt = entry((cur_c + 1) * 32 + lane);
            }
            const int e = __shfl_sync(kFull, cur, (idx0 + lane) & 31);
            int row = a.NB * a.S;  // beyond the pool: the copy fills zeros
            if (lane < blocks_per_tile && idx0 + lane < n_table) {
                if (e >= 0 && e < a.NB) row = e * a.S;
                else if (!is_v) raise_error(a.err, PKV_DEVERR_BAD_BLOCK);
            }
            return row;
        };
        // a free stage of the bf16 ring for key tile j
        auto wait_free = [&](int j) {
            return j < kStages || __all_sync(kFull, mbar_spin_bounded(bar + 8 * (empty + j % kStages),
                                                                     (j / kStages - 1) & 1, a.timeout_ns));
        };
        int issued = 0, staged = 0, widened = 0;
        if constexpr (NARROW != 2) {
            // bf16 tiles (two 64-dim halves per key) or FP8 codes (one 128-byte line per key) straight into the ring
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % kStages;
                const int row = tile_row(j);
                if (!wait_free(j)) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
                if (__any_sync(kFull, *abort_flag != 0)) break;
                const uint32_t fb = bar + 8 * (full + st);
                if (lane == 0) mbar_arrive_expect_tx(fb, kStage);
                __syncwarp();
                if (lane < blocks_per_tile) {
                    if constexpr (NARROW == 0) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
                            tma_load_3d_nohint(dst0 + st * kStage + hf * kKvHalf + lane * a.S * 128, map, hf * 64, h,
                                               row, fb);
                    } else {
                        tma_load_3d_nohint(dst0 + st * kStage + lane * a.S * 128, map, 0, h, row, fb);
                    }
                }
                issued = j + 1;
            }
        } else {
            // one-byte codes: copy tile j+1 into its staging slot (once tile j-1 has been widened from there: by this
            // warp, and with split widening by the MMA warp too), then widen the rows of tile j (split widening: the
            // first half) into the f16 ring
            const int sbar = kBarStg + (is_v ? 2 : 0), fbar = kBarStgFree + (is_v ? 2 : 0);
            const uint32_t stg0 = sb + kOffStg + (is_v ? 2 : 0) * kStgSlot;
            auto stage = [&](int jj, int row) {
                const uint32_t fb = bar + 8 * (sbar + (jj & 1));
                if (lane == 0) mbar_arrive_expect_tx(fb, kStgSlot);
                __syncwarp();
                if (lane < blocks_per_tile)
                    tma_load_3d_nohint(stg0 + (jj & 1) * kStgSlot + lane * a.S * 128, map, 0, h, row, fb);
            };
            stage(0, tile_row(0));
            staged = 1;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % kStages;
                if (j + 1 < n_tiles) {
                    // slot (j+1) & 1 last held tile j-1: this warp widened its rows at j-1 (and fenced)
                    if (split && j >= 1 && !__all_sync(kFull, mbar_spin_bounded(bar + 8 * (fbar + ((j - 1) & 1)),
                                                                      ((j - 1) >> 1) & 1, a.timeout_ns))) {
                        if (lane == 0) *abort_flag = 1;
                        break;
                    }
                    stage(j + 1, tile_row(j + 1));
                    staged = j + 2;
                }
                if (!__all_sync(kFull, mbar_spin_bounded(bar + 8 * (sbar + (j & 1)), (j >> 1) & 1, a.timeout_ns)) ||
                    !wait_free(j)) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
                widened = j + 1;
                if (__any_sync(kFull, *abort_flag != 0)) break;
                widen_rows(is_v, j & 1, st, 0);
                if (!split) widen_rows(is_v, j & 1, st, 1);
                fence_proxy_async_smem();  // the MMA (async proxy) reads what was written; the next copy overwrites
                __syncwarp();
                if (lane == 0) mbar_arrive(bar + 8 * (full + st));
            }
        }
        // its own copies have landed before the CTA may finish (bounded)
        if (lane == 0) {
            for (int t = issued - kStages < 0 ? 0 : issued - kStages; t < issued; ++t)
                mbar_wait_bounded(bar + 8 * (full + t % kStages), (t / kStages) & 1, a.timeout_ns);
            for (int t = widened; t < staged; ++t)
                mbar_wait_bounded(bar + 8 * (kBarStg + (is_v ? 2 : 0) + (t & 1)), (t >> 1) & 1, a.timeout_ns);
            if (!is_v) mbar_wait_bounded(bar + 8 * kBarQFull, 0, a.timeout_ns);
        }
    } else if (warp == 9 || warp == 11) {
        // ------------------------------------------------ MMA warps: warp 9 issues the S MMAs, warp 11 the P.V
        // MMAs; each warp runs its loop as a whole and one elected lane issues (operands stay warp-uniform)
        // descriptors are built once; an operand at byte offset x from the tile base is base + (x >> 4)
        // (the 14-bit start-address field cannot carry: shared addresses stay below 256 KB)
        const uint64_t d_kmaj = smem_desc_sw128(sb, 16, 1024);       // Q and K: K-major rows of 128 B
        const uint64_t d_v = smem_desc_sw128(sb, kKvHalf, 1024);     // V: N-major, d-halves kKvHalf apart
        bool ok = true;
        // one-byte caches: this warp widens the second half of the rows of key tile jj of its operand (K for the
        // S warp, V for the P.V warp) once its codes landed and its bf16 stage is free, then frees the staging slot
        auto widen_half = [&](bool is_v, int jj) -> bool {
            const int full = is_v ? kBarVFull : kBarKFull, empty = is_v ? kBarVEmpty : kBarKEmpty;
            const int stg = kBarStg + (is_v ? 2 : 0), stf = kBarStgFree + (is_v ? 2 : 0);
            const int st = jj % kStages;
            if (!__all_sync(kFull, mbar_spin_bounded(bar + 8 * (stg + (jj & 1)), (jj >> 1) & 1, a.timeout_ns)))
                return false;
            if (jj >= kStages && !__all_sync(kFull, mbar_spin_bounded(bar + 8 * (empty + st), (jj / kStages - 1) & 1,
                                                                      a.timeout_ns)))
                return false;
            widen_rows(is_v, jj & 1, st, 1);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar + 8 * (full + st));
                mbar_arrive(bar + 8 * (stf + (jj & 1)));
            }
            return true;
        };
        if (warp == 9) {
            // S(j) of both query tiles into buffer j & 1, which P(j-2) was read from
            auto issue_s = [&](int t, int j) {
                const uint64_t a0 = d_kmaj + ((kOffQ + 2 * t * kQHalf) >> 4);
                const uint64_t b0 = d_kmaj + ((kOffK + (j % kStages) * kStage) >> 4);
                const uint32_t d = tmem + kColS + 128 * t + 64 * (j & 1);
                if constexpr (NARROW == 1) {
                    // E4M3: the query row's hi codes in the tile's first 16 KB, its lo codes in the second; the key
                    // codes one 128-byte line per key; 32 head dims (32 bytes) per MMA
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        tc_mma_f8_warp(d, a0 + 2 * kk, b0 + 2 * kk, kIdescS8, kk > 0);
                        tc_mma_f8_warp(d, a0 + (kQHalf >> 4) + 2 * kk, b0 + 2 * kk, kIdescS8, 1u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off_a = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
                        const uint32_t off_b = ((kk >> 2) * kKvHalf + (kk & 3) * 32) >> 4;
                        tc_mma_f16_warp(d, a0 + off_a, b0 + off_b, kIdescS<NARROW>, kk > 0);
                    }
                }
                tc_commit_warp(bar + 8 * (kBarSFull + 2 * t + (j & 1)));
            };
            // Q landed (bf16 caches) or converted to f16 by the softmax warps (one-byte caches)
            const uint32_t qb = bar + 8 * (NARROW ? kBarQConv : kBarQFull);
            if (split) ok = widen_half(false, 0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                const uint32_t kb = bar + 8 * (kBarKFull + j % kStages), kph = (j / kStages) & 1;
                for (int t = 0; t < (has_b ? 2 : 1); ++t) {
                    // query tile t: Q and K(j) landed, and P_t(j-2).V done with the buffer
                    ok = j < 2 ? __all_sync(kFull, mbar_spin2_bounded(qb, 0, kb, kph, a.timeout_ns))
                               : __all_sync(kFull, mbar_spin2_bounded(bar + 8 * (kBarPVDone + 2 * t + (j & 1)),
                                                                      ((j - 2) >> 1) & 1, kb, kph, a.timeout_ns));
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(t, j);
                }
                if (!ok) break;
                tc_commit_warp(bar + 8 * (kBarKEmpty + j % kStages));
                // the next tile's half of K, while the tensor pipe works on S(j)
                if (split && j + 1 < n_tiles) ok = widen_half(false, j + 1);
            }
        } else {
            // P(j).V(j) of both query tiles once their softmax is done
            auto issue_pv = [&](int t, int j) {
                const uint64_t b0 = d_v + ((kOffV + (j % kStages) * kStage) >> 4);
                const uint32_t d = tmem + kColO + 128 * t, p = tmem + kColS + 128 * t + 64 * (j & 1);
                const uint32_t acc0 = j > 0;
                if constexpr (NARROW == 1) {
                    // E4M3: P's hi codes of the 64 keys in 16 columns (four per column), its lo codes in the next
                    // 16; V codes N-major, 128 head dims per 128-byte line, 32 keys (four 1024-byte groups) per MMA
#pragma unroll
                    for (int kc = 0; kc < kKeys / 32; ++kc) {
                        tc_mma_f8_ts_warp(d, p + 8 * kc, b0 + ((kc * 4096) >> 4), kIdescPV8, kc > 0 ? 1u : acc0);
                        tc_mma_f8_ts_warp(d, p + 16 + 8 * kc, b0 + ((kc * 4096) >> 4), kIdescPV8, 1u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk)
                        tc_mma_f16_ts_warp(d, p + 8 * kk, b0 + ((kk * 2048) >> 4), kIdescPV<NARROW>,
                                           kk > 0 ? 1u : acc0);
                }
                tc_commit_warp(bar + 8 * (kBarPVDone + 2 * t + (j & 1)));
            };
            if (split) ok = widen_half(true, 0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int st = j % kStages, b = j & 1;
                const uint32_t ph = (j >> 1) & 1, vb = bar + 8 * (kBarVFull + st), vph = (j / kStages) & 1;
                for (int t = 0; t < (has_b ? 2 : 1); ++t) {
                    // query tile t: its softmax of tile j done and V(j) landed
                    ok = __all_sync(kFull, mbar_spin2_bounded(bar + 8 * (kBarPFull + 2 * t + b), ph, vb, vph,
                                                              a.timeout_ns));
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(t, j);
                }
                if (!ok) break;
                tc_commit_warp(bar + 8 * (kBarVEmpty + st));
                // the next tile's half of V, while the tensor pipe works on P(j).V
                if (split && j + 1 < n_tiles) ok = widen_half(true, j + 1);
            }
            // the last P.V follows every S MMA (it needed that tile's softmax), so this covers all MMAs
            if (ok) tc_commit_warp(bar + 8 * kBarFinal);
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else {
        // ------------------------------------------------ softmax: warps 0-3 query tile A, 4-7 tile B
        const int t = warp >> 2, quad = warp & 3;
        const int r = quad * 32 + lane;
        const int qt0 = i0 + t * rows_q;  // first token of this query tile
        const int qi = qt0 + r / a.G;
        const int qpos = q_start + qi;
        const uint32_t trow = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tO = tmem + kColO + 128 * t + trow;
        float m_ref = -INFINITY, l_run = 0.f;
        int done = 0;
        const bool active = t == 0 || has_b;
        // score scale (log2 units) and output factor of this KV head: per-head scales when given
        float sm_log2 = a.k_head ? a.sm_base * __ldg(a.k_head + h) : a.sm_log2;
        const float out_mul = a.v_head ? __ldg(a.v_head + h) : a.out_mul;
        bool s_ready = false;  // the next tile's scores were seen complete ahead of time
        if constexpr (NARROW == 1) {
            // FP8 caches: the S MMAs run on E4M3 operands.  This thread's query row r (bf16, landed by TMA: dims
            // 0-63 in the tile's first 16 KB, 64-127 in the second) is scaled by 2^e, e chosen so that its largest
            // magnitude lies in [128, 256), and split into hi = E4M3(x) and lo = E4M3(x - hi), written over the row
            // (hi codes in the first 16 KB, lo codes in the second, 128 codes per 128-byte swizzled line); hi + lo
            // is the scaled bf16 value exactly for elements within 2^-10 of the row's largest.  The scores are
            // multiplied back by 2^-e.  Non-finite query values raise Q_RANGE.
            bool ok_q = !active || __all_sync(kFull, mbar_spin_bounded(bar + 8 * kBarQFull, 0, a.timeout_ns));
            if (!ok_q) *abort_flag = 1;
            if (active && ok_q) {
                uint8_t* qt = smem + kOffQ + 2 * t * kQHalf + r * 128;
                const int sw = r & 7;
                auto chunk = [&](int hf, int k) -> uint4 {  // bf16 dims 64 hf + 8k .. + 7
                    return *reinterpret_cast<const uint4*>(qt + hf * kQHalf + ((k ^ sw) << 4));
                };
                auto amax4 = [](uint32_t m, const uint4& x) {  // |value| bits: ordered like the values
                    const uint32_t ws[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) m = max(m, max((ws[i] << 17) >> 1, ((ws[i] >> 16) & 0x7fffu) << 16));
                    return m;
                };
                // dims 64..127 are kept in registers: the lo codes of dims 0..63 are written over them
                uint4 w1[8];
                uint32_t amax_bits = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    w1[k] = chunk(1, k);
                    amax_bits = amax4(amax4(amax_bits, w1[k]), chunk(0, k));
                }
                if (amax_bits >= 0x7f800000u) raise_error(a.err, PKV_DEVERR_Q_RANGE);  // inf or NaN
                const int ex = static_cast<int>(amax_bits >> 23) - 127;        // floor(log2(max |x|))
                const int e = min(126, max(-126, 7 - ex));
                const float up = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
                sm_log2 *= __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
                for (int c = 0; c < 8; ++c) {  // output chunk c: head dims 16c .. 16c + 15
                    // bf16 chunks 2c, 2c + 1; for c < 4 read here (chunks 0 .. 2c - 1 of that half are consumed,
                    // and the chunk-c slots written below hold chunks already read or kept in w1)
                    const uint4 s0 = c < 4 ? chunk(0, 2 * c) : w1[2 * c - 8];
                    const uint4 s1 = c < 4 ? chunk(0, 2 * c + 1) : w1[2 * c - 7];
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {  // dims 16c + 4i .. 16c + 4i + 3
                        const uint4 src = (i >> 1) ? s1 : s0;
                        const uint32_t x01 = (i & 1) ? src.z : src.x, x23 = (i & 1) ? src.w : src.y;
                        const float2 f01 = bf16x2_to_float2(x01), f23 = bf16x2_to_float2(x23);
                        const float q0 = f01.x * up, q1 = f01.y * up, q2 = f23.x * up, q3 = f23.y * up;
                        const uint32_t h01 = f32x2_to_e4m3x2(q0, q1), h23 = f32x2_to_e4m3x2(q2, q3);
                        const float2 b01 = f16x2_to_float2(e4m3x2_to_f16x2_u(h01));
                        const float2 b23 = f16x2_to_float2(e4m3x2_to_f16x2_u(h23));
                        hw[i] = h01 | (h23 << 16);
                        lw[i] = f32x2_to_e4m3x2(q0 - b01.x, q1 - b01.y) | (f32x2_to_e4m3x2(q2 - b23.x, q3 - b23.y) << 16);
                    }
                    *reinterpret_cast<uint4*>(qt + ((c ^ sw) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(qt + kQHalf + ((c ^ sw) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
                fence_proxy_async_smem();  // the S MMAs (async proxy) read what was written
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + 8 * kBarQConv);
        }
        if constexpr (NARROW == 2) {
            // INT8 caches: the MMAs run on f16 operands, so Q (bf16, landed by TMA) is converted in place, each
            // query tile by its own four warps; exact for |q| in [2^-14, 65504], larger values raise Q_RANGE
            bool ok_q = !active || __all_sync(kFull, mbar_spin_bounded(bar + 8 * kBarQFull, 0, a.timeout_ns));
            if (!ok_q) *abort_flag = 1;
            if (active && ok_q) {
                uint8_t* qt = smem + kOffQ + 2 * t * kQHalf;
                bool in_range = true;
                for (int i = quad * 32 + lane; i < 2 * kQHalf / 16; i += kSoftmax / 2) {
                    uint4 w = *reinterpret_cast<const uint4*>(qt + i * 16);
                    uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 f = bf16x2_to_float2(ws[k]);
                        in_range = in_range && fabsf(f.x) < 65520.f && fabsf(f.y) < 65520.f;
                        ws[k] = f16x2_rn(f.x, f.y);
                    }
                    *reinterpret_cast<uint4*>(qt + i * 16) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
                }
                if (!in_range) raise_error(a.err, PKV_DEVERR_Q_RANGE);
                fence_proxy_async_smem();  // the S MMAs (async proxy) read what was written
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + 8 * kBarQConv);
        }
        for (int j = 0; active && j < n_tiles; ++j) {
            const int tile0 = j * kKeys, b = j & 1;
            const uint32_t tS = tmem + kColS + 128 * t + 64 * b + trow;
            if (!__all_sync(kFull, s_ready) &&
                !__all_sync(kFull, mbar_spin_bounded(bar + 8 * (kBarSFull + 2 * t + b), (j >> 1) & 1,
                                                     a.timeout_ns))) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            float v[64];
            tmem_ld64(tS, v);
            // test the next tile's scores now; the answer is used only when that tile starts
            s_ready = j + 1 < n_tiles && mbar_test(bar + 8 * (kBarSFull + 2 * t + (b ^ 1)), ((j + 1) >> 1) & 1);
            const bool masked = (tile0 + kKeys - 1 > q_start + qt0) || (tile0 + kKeys > kv_len);
            const int lim = min(kv_len, qpos + 1) - tile0;
            float mx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
            if (!masked) {
#pragma unroll
                for (int i = 0; i < 64; i += 2) mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], v[i], v[i + 1]);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) mx[i & 7] = fmaxf(mx[i & 7], (i < lim) ? v[i] : -INFINITY);
            }
            const float mraw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            const float mt = mraw * sm_log2;
            const bool need = mt > m_ref + 8.f;
            // O is rescaled (below) only when some row of the warp needs it; rows that do not keep alpha = 1
            const bool rescale = j > 0 && __any_sync(kFull, need);
            const float m_new = need ? (NARROW == 1 ? mt - kP8Shift : mt) : m_ref;
            const float alpha = ex2_approx(m_ref - m_new);
            m_ref = m_new;
            // exponent arguments and running sums on packed fp32 pairs (two elements per instruction); the
            // masked form (edge tiles only) is a separate instance so the common path carries no selects
            const float2 sc2 = make_float2(sm_log2, sm_log2), nm2 = make_float2(-m_ref, -m_ref);
            float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            uint32_t pk[32];  // bf16 / f16 pairs; FP8: 16 words of four hi codes, then 16 of four lo codes
            auto exp_pack = [&](auto with_mask) {
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    const float2 x = __ffma2_rn(make_float2(v[i], v[i + 1]), sc2, nm2);
                    float p0 = ex2_approx(x.x);
                    float p1 = ex2_approx(x.y);
                    if constexpr (decltype(with_mask)::value) {
                        p0 = (i < lim) ? p0 : 0.f;
                        p1 = (i + 1 < lim) ? p1 : 0.f;
                    }
                    ls2[(i >> 1) & 1] = __fadd2_rn(ls2[(i >> 1) & 1], make_float2(p0, p1));
                    if constexpr (NARROW != 0) pk[i / 2] = f16x2_rn(p0, p1);
                    else pk[i / 2] = bf16x2_rn(p0, p1);
                }
                if constexpr (NARROW == 1) {
                    // the f16 probabilities (at most 2^8) split into two E4M3 parts for the 8-bit P.V MMAs
                    uint32_t hl[32];
#pragma unroll
                    for (int k = 0; k < 16; ++k) split_e4m3x4(pk[2 * k], pk[2 * k + 1], hl[k], hl[16 + k]);
#pragma unroll
                    for (int k = 0; k < 32; ++k) pk[k] = hl[k];
                }
            };
            if (masked) exp_pack(std::true_type{});
            else exp_pack(std::false_type{});
            const float2 lsum = __fadd2_rn(ls2[0], ls2[1]);
            l_run = l_run * alpha + (lsum.x + lsum.y);
            tmem_st32u(tS, pk);  // P over the scores just read (this thread's lane only)
            if (rescale) {
                // O may be touched only once the previous P.V of this query tile has completed
                if (!__all_sync(kFull, mbar_wait_bounded(bar + 8 * (kBarPVDone + 2 * t + ((j - 1) & 1)),
                                                         ((j - 1) >> 1) & 1, a.timeout_ns))) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float o[64];
                    tmem_ld64(tO + 64 * c, o);
#pragma unroll
                    for (int i = 0; i < 64; ++i) o[i] *= alpha;
                    tmem_st64(tO + 64 * c, o);
                }
            }
            // keys past kv_len in this tile: their V rows are not data, make them zero once they have landed
            // (tile A's threads do it; P.V of tile B is issued after P.V of tile A)
            const int nvalid = min(kKeys, kv_len - tile0);
            if (t == 0 && nvalid < kKeys) {
                const int st = j % kStages;
                if (!__all_sync(kFull, mbar_wait_bounded(bar + 8 * (kBarVFull + st), (j / kStages) & 1,
                                                         a.timeout_ns))) {
                    *abort_flag = 1;
                    break;
                }
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                if constexpr (NARROW == 1) {  // one 128-byte line of codes per key
                    for (int idx = tid; idx < (kKeys - nvalid) * 8; idx += kSoftmax / 2) {
                        const int row = nvalid + idx / 8, ch = idx & 7;
                        *reinterpret_cast<uint4*>(smem + kOffV + st * kStage + row * 128 + ch * 16) = z;
                    }
                } else {
                    for (int idx = tid; idx < (kKeys - nvalid) * 16; idx += kSoftmax / 2) {
                        const int row = nvalid + idx / 16, hf = (idx / 8) & 1, ch = idx & 7;
                        *reinterpret_cast<uint4*>(smem + kOffV + st * kStage + hf * kKvHalf + row * 128 + ch * 16) = z;
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(bar + 8 * (kBarPFull + 2 * t + b));
            done = j + 1;
        }
        // ---- every MMA done, out = O / l
        const bool ok = active && !__any_sync(kFull, *abort_flag != 0) && done == n_tiles &&
                        __all_sync(kFull, mbar_wait_bounded(bar + 8 * kBarFinal, 0, a.timeout_ns));
        tc_fence_after();
        if (active) {
            const bool store = ok && qi < NQ;
            const float inv = l_run > 0.f ? out_mul / l_run : 0.f;
            uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) +
                            (static_cast<size_t>(q_base + qi) * a.Hq + static_cast<size_t>(h) * a.G + r % a.G) * 256;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float o[64];
                tmem_ld64(tO + 64 * c, o);  // warp-collective: every lane loads, valid rows store
                if (store) {
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        uint4 w;
                        w.x = bf16x2_rn(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
                        w.y = bf16x2_rn(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
                        w.z = bf16x2_rn(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
                        w.w = bf16x2_rn(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
                        *reinterpret_cast<uint4*>(orow + c * 128 + q4 * 16) = w;
                    }
                }
            }
            if (!ok) *abort_flag = 1;
        }
    }

    // ---- drain: nothing of this CTA may still be in flight when TMEM is freed and the CTA exits
    __syncthreads();
    if ((warp == 9 || warp == 11) && *abort_flag) {
        tc_commit_warp(bar + 8 * kBarDrain);  // arrives once every MMA this warp issued has completed
        mbar_wait_bounded(bar + 8 * kBarDrain, 0, a.timeout_ns);
    }
    __syncthreads();
    if (*abort_flag && tid == 0) raise_error(a.err, PKV_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    if constexpr (REUSE) {
        if (tid == 0)  // the barriers initialised above (the bf16 instance leaves the staging ones out)
            for (int i = 0; i < (NARROW ? kNumBars : kBarStgFree); ++i) mbar_inval(bar + 8 * i);
        __syncthreads();
    }
}


}  // namespace pkv
