// decode_mma.cuh -- paged decode attention with the per-warp tensor-core MMA: FP8 (E4M3) and INT8 K/V caches, and
// bf16 caches in GQA groups of 8 (128-dim heads, bf16 queries).
//
// Method: the same online-softmax recurrence over the blocks named by each sequence's block table as the CUDA-core
// decode kernel (decode.cuh; "从 PagedAttention 到 Chunked Prefill" §2.2, "PagedAttention：块表"), with the same
// work split, TMA pipeline per warp and split-KV records.  What changes is the arithmetic: on the CUDA cores these
// cases need 2·G fp32 multiply-adds per cached element, which at the HBM rate is two thirds of the fp32 peak (INT8
// at G = 4, bf16 at G = 8) or more than all of it (FP8 at G = 8).  Here each warp computes, per 16-token tile of one
// (sequence, KV head),
//   S = Q · Kᵀ   as 2 × 8 mma.sync.m16n8k16 (rows: the G query heads, padded to 16; columns: 8 tokens; k: 16 dims)
//   O += P · V  as 16 mma.sync.m16n8k16 (rows: the G heads; columns: 8 head dims; k: the 16 tokens)
// with fp32 accumulation.  One-byte caches run f16 operands: every E4M3 and INT8 code is exactly an f16 value, Q is
// converted from bf16 to f16 once per segment (exact for |q| in [2^-14, 65504]; larger values raise
// PKV_DEVERR_Q_RANGE), and the probabilities are rounded to f16 (relative 2^-11) before P·V.  bf16 caches run bf16
// operands on the cached values as they are, with the probabilities rounded to bf16.  The per-tensor or per-head
// scales are applied to the fp32 scores and to the output.  For groups up to 4 a warp takes two neighbouring KV heads
// together (HP = 2): the second head's query rows are MMA rows 8-15.
//
// Fragment layout (lane = 4 g + t): in S, thread (g, t) holds row g (query head g of the group; row g + 8 for the
// second head of a unit) and tokens 2t, 2t+1 of each 8-token column tile.  The k index of the S MMAs is a
// permutation of the head dimension chosen so that a thread's K operand is one contiguous run of its token's row
// (one-byte codes: dims 32t .. 32t + 31, four per k-step; bf16: dims 16t .. 16t + 15 of each 64-dim half), and Q is
// permuted the same way; the dot product does not depend on the order of its terms.  In P·V the k index is the token
// in natural order, so the probabilities of S's output fragment are P's input fragment as they stand, and each
// thread reads 16-byte runs of four token rows and pairs tokens with byte permutes.  K and V tiles arrive by TMA with
// the 128-byte swizzle (128-byte rows), which keeps all these 16-byte shared-memory reads free of bank conflicts.
#pragma once

#include "decode.cuh"

namespace pkv {

// Warps per CTA of the tensor-core decode (at most the CUDA-core policy's count, which sizes the split-KV
// workspace): few instructions per block leave the pipeline depth, not the warp count, as what hides latency.
constexpr int kMmaWarps = 8;

// one m16n8k16 MMA, f16 (or bf16: B16) operands, fp32 accumulate in place.  The operands are whole register quads
// (rows 8-15 of A are zero registers of the quad and rows 8-15 of C accumulate nothing of use), so no copies are
// needed around it.
// two INT8 codes (low bytes first, or the high half when HI) -> f16x2 of 1152 + code, exactly (one byte permute).
// The key operand takes the codes in this biased form: q.(1152 + k) = q.k + 1152 sum(q), and the decode subtracts
// 1152 sum(q) (one value per query row and segment) from the fp32 scores, which saves the f16 subtraction per two
// key codes; the cancellation costs about 2^-20 of the scores' magnitude.
template <bool HI>
__device__ __forceinline__ uint32_t s8x2_to_biased_f16x2(uint32_t w) {
    return __byte_perm(w ^ 0x80808080u, 0x64646464u, HI ? 0x7362u : 0x5140u);
}

template <bool B16>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (B16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// two one-byte codes (low byte first in the low 16 bits of w, or the high 16 bits when HI) -> f16x2, exactly
template <class KV, bool HI>
__device__ __forceinline__ uint32_t codes2_to_f16x2(uint32_t w) {
    if constexpr (KV::code == PKV_INT8) {
        // signed byte b: (b ^ 0x80) = b + 128 in the low mantissa bits of 1024.0 reads 1024 + b + 128; one packed
        // subtraction of 1152 leaves b
        const uint32_t f = w ^ 0x80808080u;
        const uint32_t h = __byte_perm(f, 0x64646464u, HI ? 0x7362u : 0x5140u);
        uint32_t r;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
        return r;
    } else {
        uint32_t r;
        const uint16_t c = static_cast<uint16_t>(HI ? (w >> 16) : (w & 0xffffu));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
        return r;
    }
}

template <bool B16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (B16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Byte offset of 16-byte chunk c (0..7) of row r in a tile of 128-byte rows stored with the 128-byte TMA swizzle
// (the tile starts on a 1024-byte boundary, so the chunk is c ^ (r & 7))
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// byte b (0..3) of word w, and of word x, interleaved: [w.b, x.b, w.b+1, x.b+1] for even b
template <int B>
__device__ __forceinline__ uint32_t pair_bytes(uint32_t w, uint32_t x) {
    static_assert(B == 0 || B == 2, "even byte");
    return __byte_perm(w, x, B == 0 ? 0x5140u : 0x7362u);
}

// Shared-memory plan of one warp stage: the K tiles of its HP KV heads, then their V tiles.  A tile is one half
// (one-byte codes: S rows of 128 codes) or two halves (bf16: head dims 0-63, then 64-127, S rows of 128 bytes each),
// every half padded to 1024 bytes so that it starts on the 128-byte swizzle's 1024-byte period.  The query rows do
// not pass through the stages: each thread loads its Q into registers once per segment, so every stage byte
// carries K or V.
template <int S, int ES, int HP>
struct MmaStage {
    static constexpr int kHalf = S * 128 < 1024 ? 1024 : S * 128;
    static constexpr int kTile = (ES == 2 ? 2 : 1) * kHalf;
    static constexpr int kBytes = 2 * HP * kTile;
};

// HP: KV heads per work unit.  With HP = 2 (GQA groups up to 8) a warp takes two neighbouring KV heads of the same
// blocks together: the second head's query rows are rows 8-15 of the MMAs (zero padding otherwise), its scores the
// second half of each S quad and its output the second half of each O quad.  The MMA count per byte is the same,
// the per-block work of the pipeline (waits, refills, metadata, softmax reductions) is shared by two heads, and the
// two heads' rows of a token, adjacent in the cache, are fetched together.
// Barrier over the first nthreads threads of the CTA (all of them: __syncthreads; fewer, when the rest of the CTA
// does other work or has left: named barrier 1).
__device__ __forceinline__ void threads_sync(int nthreads) {
    if (nthreads == static_cast<int>(blockDim.x)) __syncthreads();
    else asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// The decode, run by the first nthreads threads of a CTA (nthreads / 32 worker warps) as CTA cta of ncta CTAs that
// share the work stream; smem_raw is the dynamic shared memory the plan in `a` describes.  pcost (nullable, ncta
// entries) weights the split for CTAs that join the stream late: CTA c is taken to have pcost[c] stream items of
// other work before its decode starts (in 1/kCostUnit items), and the stream is cut so that every CTA finishes
// together; cb is shared memory for the cut points (ncta + 1 ints, ncta <= 256, nthreads / 32 a power of two).
// WEIGHTED selects this form at compile time.
constexpr int kCostUnit = 16;  // the weighted split's CTA costs are in 1/16 stream items

template <int G, int S, class KV, int HP, bool WEIGHTED>
__device__ __forceinline__ void decode_mma_body(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeArgs& a,
                                                uint8_t* smem_raw, int cta, int ncta, int nthreads,
                                                const int* pcost, int* cb) {
    constexpr int D = 128;
    constexpr int TS = S < 16 ? S : 16;   // tokens of a block per 16-row MMA tile
    constexpr int NT = S / TS;            // tiles per block
    constexpr bool B16 = KV::es == 2;  // bf16 cache: bf16 MMAs on the cached values as they are
    constexpr int kHalf = MmaStage<S, KV::es, HP>::kHalf, kTile = MmaStage<S, KV::es, HP>::kTile;
    constexpr int GU = HP * G;  // query heads of a work unit (rows of its split-KV records)
    static_assert(G <= 8 && (HP == 1 || HP == 2), "query rows of one MMA tile");
    static_assert(KV::es <= 2, "one-byte or bf16 caches");

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NW = nthreads >> 5;
    const int B = a.B, Hkv = a.Hkv;
    const int g = lane >> 2, t = lane & 3;  // fragment row (query head) and column pair
    // this thread's operand offsets inside a K or V half: K rows g and 8 + g (1024 bytes further, same swizzle),
    // chunks 2t and 2t + 1; V rows 2t, 2t + 1 and 2t + 8, 2t + 9 (1024 bytes further), chunk g.  One-byte codes:
    // the K chunks are head dims 32t .. 32t + 31, the V chunk dims 16g .. 16g + 15.  bf16: the same chunks of both
    // halves, K dims 16t .. 16t + 15 and 64 + 16t .. 64 + 16t + 15, V dims 8g .. 8g + 7 and 64 + 8g .. 64 + 8g + 7.
    const uint32_t kb0 = sw128_offset(g, 2 * t), kb1 = sw128_offset(g, 2 * t + 1);
    const uint32_t vb0 = sw128_offset(2 * t, g), vb1 = sw128_offset(2 * t + 1, g);
    uint32_t zr;  // a zero the compiler cannot fold: it fills rows 8-15 of the A quads in place
    asm volatile("mov.b32 %0, 0;" : "=r"(zr));

    // ---- 1. per-sequence block counts and their prefix sum (P[s] = blocks before s)
    int* P = reinterpret_cast<int*>(smem);
    {
        const int per = (B + nthreads - 1) / nthreads;
        const int s0 = tid * per;
        const int s1 = min(B, s0 + per);
        int local = 0;
        for (int s = s0; s < s1; ++s) {
            int L = a.context_lens[s];
            if (L < 0 || L > a.MB * S) {
                if (cta == 0) raise_error(a.err, PKV_DEVERR_BAD_LENGTH);
                L = 0;
            }
            local += (L + S - 1) / S;
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        __shared__ int warp_tot[32];
        if (lane == 31) warp_tot[warp] = incl;
        threads_sync(nthreads);
        int wbase = 0;
        for (int i = 0; i < warp; ++i) wbase += warp_tot[i];
        int run = wbase + incl - local;
        for (int s = s0; s < s1; ++s) {
            P[s] = run;
            int L = a.context_lens[s];
            if (L < 0 || L > a.MB * S) L = 0;
            run += (L + S - 1) / S;
        }
        if (tid == nthreads - 1) {
            int tot = 0;
            for (int i = 0; i < NW; ++i) tot += warp_tot[i];
            P[B] = tot;
        }
        threads_sync(nthreads);
    }

    // ---- 2. empty sequences get zero rows (spread over the CTAs)
    for (int s = cta; s < B; s += ncta) {
        if (P[s + 1] != P[s]) continue;
        const int n = a.Hq * D;
        for (int i = tid; i < n; i += nthreads) reinterpret_cast<uint16_t*>(a.out)[static_cast<size_t>(s) * n + i] = 0;
    }

    // ---- 3. this warp's stages and barriers, and its share of the work stream
    uint8_t* wreg = smem + a.prefix_bytes + static_cast<size_t>(warp) * a.warp_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(wreg + static_cast<size_t>(a.depth) * a.stage_bytes);
    const uint32_t wreg_u32 = smem_u32(wreg);
    const uint32_t bars_u32 = smem_u32(bars);
    if (lane == 0) {
        for (int i = 0; i < a.depth; ++i) mbar_init(bars_u32 + 8 * i, 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int Hu = Hkv / HP;  // work units per block: KV heads taken HP at a time
    const int T = Hu * P[B];
    if (T == 0) return;
    const int W = WEIGHTED ? ncta * NW : min(ncta * NW, T);
    const int w = cta * NW + warp;
    if constexpr (WEIGHTED) {
        // CTA c's part of the stream: E - pcost[c] items, E chosen so that the parts add up to T (CTAs whose other
        // work alone reaches E get none).  Warp 0 of every CTA computes the same cut points, each lane over a run of
        // up to 8 CTAs held in registers, in fp32 (GB300 has little FP64 throughput, and a 64-bit division goes
        // through it): E by levelling, then every CTA's part rounded to whole items and an exact integer prefix over
        // the parts, so that the cuts are monotone; the last is T.
        if (warp == 0) {
            constexpr int kPer = 8;  // CTAs per lane: ncta <= 256
            const int per = (ncta + 31) / 32;
            const int c_lo = lane * per;
            float pv[kPer];  // this lane's CTAs' costs in items (-1: no CTA)
#pragma unroll
            for (int k = 0; k < kPer; ++k)
                pv[k] = (k < per && c_lo + k < ncta) ? static_cast<float>(pcost[c_lo + k]) * (1.0f / kCostUnit) : -1.f;
            const float Tf = static_cast<float>(T);
            auto wsum = [](float v) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
                return v;
            };
            float own = 0.f;
#pragma unroll
            for (int k = 0; k < kPer; ++k) own += fmaxf(pv[k], 0.f);
            float E = (Tf + wsum(own)) / static_cast<float>(ncta);
            int n_prev = ncta;
            for (int it = 0; it < 4; ++it) {  // drop CTAs at or above E and re-level (a few steps at most)
                float t2 = 0.f;
                int n2 = 0;
#pragma unroll
                for (int k = 0; k < kPer; ++k)
                    if (pv[k] >= 0.f && pv[k] < E) {
                        t2 += pv[k];
                        ++n2;
                    }
                n2 = __reduce_add_sync(kFull, n2);
                t2 = wsum(t2);
                if (n2 == 0 || n2 == n_prev) break;  // uniform across the warp
                n_prev = n2;
                E = (Tf + t2) / static_cast<float>(n2);
            }
            float mine_f = 0.f;
#pragma unroll
            for (int k = 0; k < kPer; ++k) mine_f += pv[k] >= 0.f ? fmaxf(E - pv[k], 0.f) : 0.f;
            const float acc = wsum(mine_f);
            const float inv = acc > 0.f ? Tf / acc : 0.f;
            int part[kPer];
#pragma unroll
            for (int k = 0; k < kPer; ++k)
                part[k] = pv[k] < 0.f ? 0
                          : acc > 0.f ? static_cast<int>(rintf(fmaxf(E - pv[k], 0.f) * inv))
                                      : (c_lo + k == 0 ? T : 0);
            // exact prefix sums (64-bit adds: rounding may take the total a few items past T), clamped only where
            // written
            long long mine = 0;
#pragma unroll
            for (int k = 0; k < kPer; ++k) mine += part[k];
            long long incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            long long run = incl - mine;
            if (lane == 0) cb[0] = 0;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int c = c_lo + k;
                run += part[k];
                if (k < per && c < ncta) cb[c + 1] = c + 1 == ncta ? T : static_cast<int>(min(static_cast<long long>(T), run));
            }
        }
        threads_sync(nthreads);
    }
    WorkSplit split{P, B, Hu, T, a.part_blocks, W, T / W, T % W};
    if constexpr (WEIGHTED) {
        split.cb = cb;
        split.nw_shift = 31 - __clz(NW);  // NW is a power of two (8)
    }
    const int A0 = split.start(w);
    const int A1 = split.start(w + 1);
    if (A0 >= A1) return;
    if (lane == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    const uint64_t pol = policy_evict_first();

    // Stream position x -> packed metadata (computed by the lane that owns x).
    auto make_meta = [&](int x) -> Meta {
        Meta m{0, -1, 0};
        if (x >= A1) return m;
        const int s = find_seq(P, B, x / Hu);
        const int local = x - Hu * P[s];
        const int nb = P[s + 1] - P[s];
        const int u = local / nb;
        const int j = local - u * nb;
        const int L = a.context_lens[s];
        m.a = s * 1024 + u;
        m.b = a.block_tables[static_cast<size_t>(s) * a.MB + j];
        const int valid = min(S, L - j * S);
        m.c = valid | (j == 0 ? kMetaFirst : 0) | (j == nb - 1 ? kMetaLast : 0) |
              ((m.b >= 0 && m.b < a.NB) ? kMetaOk : 0);
        return m;
    };

    // Issue the copies of a stream index into stage st (by the lane holding the block's metadata).
    auto issue = [&](int st, const Meta& m) {
        const bool ok = (m.c & kMetaOk) != 0;
        if (!ok) raise_error(a.err, PKV_DEVERR_BAD_BLOCK);
        const uint32_t bar = bars_u32 + 8 * st;
        const uint32_t dst = wreg_u32 + st * a.stage_bytes;
        if (ok) {
            mbar_arrive_expect_tx(bar, 2u * HP * a.kv_bytes);
            const int h0 = (m.a & 1023) * HP;
#pragma unroll
            for (int hh = 0; hh < HP; ++hh)
#pragma unroll
                for (int hf = 0; hf < (B16 ? 2 : 1); ++hf) {
                    tma_load_3d(dst + hh * kTile + hf * kHalf, &kmap, hf * 64, h0 + hh, m.b * S, bar, pol);
                    tma_load_3d(dst + (HP + hh) * kTile + hf * kHalf, &vmap, hf * 64, h0 + hh, m.b * S, bar, pol);
                }
        } else {
            mbar_arrive(bar);
        }
    };

    const int n_blocks = A1 - A0;
    int wbase = A0;
    Meta cur = make_meta(wbase + lane);
    Meta nxt = make_meta(wbase + 32 + lane);
    if (lane < a.depth && lane < n_blocks) {
        fence_proxy_async_smem();
        issue(lane, cur);
    }

    // Bounded wait for stream index k in stage st (phase parity ph); on timeout record the error and drain the
    // copies still in flight (bounded).
    auto wait_stage = [&](int k, int st, uint32_t ph) -> bool {
        if (mbar_wait_bounded(bars_u32 + 8 * st, ph, a.timeout_ns)) return true;
        raise_error(a.err, PKV_DEVERR_TIMEOUT);
        for (int kk = k + 1; kk < k + a.depth && kk < n_blocks; ++kk)
            mbar_wait_bounded(bars_u32 + 8 * static_cast<int>(kk % a.depth),
                              static_cast<uint32_t>((kk / a.depth) & 1), a.timeout_ns);
        return false;
    };

    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
    // The query rows of the pair whose first block follows stream position x, when the metadata window holds it:
    // prefetched into L2 (HP G rows of 256 bytes, contiguous), so that the next segment's own loads hit L2 instead
    // of waiting on DRAM behind the K/V stream.
    auto prefetch_next_q = [&](int x) {
        const unsigned f0 = __ballot_sync(kFull, (cur.c & kMetaFirst) && wbase + lane > x);
        const unsigned f1 = __ballot_sync(kFull, (nxt.c & kMetaFirst) && wbase + 32 + lane > x);
        if ((f0 | f1) == 0) return;
        const int sl = f0 ? __ffs(f0) - 1 : __ffs(f1) - 1;
        const int na = __shfl_sync(kFull, f0 ? cur.a : nxt.a, sl);
        if (lane < HP * G * 2) {
            const uint8_t* q0 = reinterpret_cast<const uint8_t*>(a.q) +
                                (static_cast<size_t>(na >> 10) * a.Hq + static_cast<size_t>(na & 1023) * HP * G) * D * 2;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(q0 + lane * 128));
        }
    };
    // A cut pair's ticket: the atomic's result is read only at the next segment's end (or at the end of the
    // share), so that its round trip does not stall the stream; the last finisher then merges the pair.
    int pend_s = -1, pend_u = 0, pend_blocks = 0, pend_old = 0;

    // the 32 output dims of thread (g, t), in runs of 16 contiguous dims: one-byte caches 32t .. 32t+31; bf16
    // caches 16t .. 16t+15 and 64+16t .. 64+16t+15 (output tile n, column 2t / 2t+1 is dim 8 (2t) + n / 8 (2t+1)
    // + n for n < 8, and 64 + the same for tile 8 + n)
    auto dim_of = [&](int i) { return B16 ? (i < 16 ? 16 * t + i : 64 + 16 * t + i - 16) : 32 * t + i; };
    // head hh's O in dim_of order
    auto o_row = [&](const float (&o)[16][4], int hh, float (&v)[32]) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            if constexpr (B16) {
                v[n] = o[n][2 * hh];
                v[8 + n] = o[n][2 * hh + 1];
                v[16 + n] = o[8 + n][2 * hh];
                v[24 + n] = o[8 + n][2 * hh + 1];
            } else {
                v[n] = o[n][2 * hh];
                v[8 + n] = o[8 + n][2 * hh];
                v[16 + n] = o[n][2 * hh + 1];
                v[24 + n] = o[8 + n][2 * hh + 1];
            }
        }
    };
    // out[s][query head (u HP + hh) G + g][dim_of(i)], bf16
    auto store_row = [&](int s, int u, int hh, const float (&x)[32], float inv) {
        uint32_t wv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            wv[i] = static_cast<uint32_t>(float_to_bf16_bits(x[2 * i] * inv)) |
                    (static_cast<uint32_t>(float_to_bf16_bits(x[2 * i + 1] * inv)) << 16);
        uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) +
                        (static_cast<size_t>(s) * a.Hq + static_cast<size_t>(u * HP + hh) * G + g) * D * 2;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(orow + dim_of(8 * i) * 2) =
                make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
    };
    auto out_mul = [&](int u, int hh) { return a.v_head ? __ldg(a.v_head + u * HP + hh) : a.o_mul; };
    const size_t rec_floats = static_cast<size_t>(GU) * (D + 2);

    // Merge of pair (s, u) by its last finisher: the shares that hold a segment of it are found 32 workers at a
    // time (one per lane; shares are contiguous in worker order), and their records are combined in stream order.
    // Every lane works on the merge: lane (row r, part c) owns dims [c DPL, (c + 1) DPL) of record row r (query
    // head u GU + r), and the loads of two records are in flight together.
    auto merge_pair = [&](int s, int u) {
        constexpr int LPR = 32 / GU;    // lanes per record row
        constexpr int DPL = D / LPR;    // dims per lane
        constexpr int NV = DPL / 4;     // 16-byte runs per lane (8-byte pairs when GU is odd)
        constexpr int NBATCH = DPL <= 32 ? 2 : 1;
        const int r_row = lane / LPR, d0 = (lane % LPR) * DPL;
        __threadfence();
        const int nb = P[s + 1] - P[s];
        const int U0 = Hu * P[s] + u * nb;
        const int U1 = U0 + nb;
        int w_first = 0;  // the last worker at or before w whose share starts at or before the pair
        for (int base = w;; base -= 32) {
            const int cand = base - lane;
            const unsigned okm = __ballot_sync(kFull, cand < 0 || split.start(cand) <= U0);
            if (okm) {
                w_first = max(0, base - (__ffs(okm) - 1));
                break;
            }
        }
        float Mx = -INFINITY, Ls = 0.f, acc[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
        auto load_rec = [&](const float* r, float& m, float& l, float4 (&ov)[NV]) {
            m = __ldcg(r + GU * D + r_row);
            l = __ldcg(r + GU * D + GU + r_row);
            const float* o = r + r_row * D + d0;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if constexpr (GU % 2 == 0) {
                    ov[i] = __ldcg(reinterpret_cast<const float4*>(o) + i);
                } else {
                    const float2 a01 = __ldcg(reinterpret_cast<const float2*>(o) + 2 * i);
                    const float2 a23 = __ldcg(reinterpret_cast<const float2*>(o) + 2 * i + 1);
                    ov[i] = make_float4(a01.x, a01.y, a23.x, a23.y);
                }
            }
        };
        auto combine = [&](float m, float l, const float4 (&ov)[NV]) {
            const float mn = fmaxf(Mx, m);
            const float fo = (Mx == -INFINITY) ? 0.f : ex2_approx(Mx - mn);
            const float fr = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
            Ls = Ls * fo + l * fr;
            Mx = mn;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                acc[4 * i] = acc[4 * i] * fo + ov[i].x * fr;
                acc[4 * i + 1] = acc[4 * i + 1] * fo + ov[i].y * fr;
                acc[4 * i + 2] = acc[4 * i + 2] * fo + ov[i].z * fr;
                acc[4 * i + 3] = acc[4 * i + 3] * fo + ov[i].w * fr;
            }
        };
        for (int base = w_first; base < W; base += 32) {
            // lane i: worker base + i, whether its (non-empty) share holds a segment of the pair, and which slot
            const int cand = base + lane;
            const int c0 = cand < W ? split.start(cand) : T;
            const int c1 = cand < W ? split.start(cand + 1) : T;
            const unsigned cm = __ballot_sync(kFull, cand < W && c0 < U1 && c1 > c0);
            const int slot_l = c0 >= U0 ? 0 : 1;
            const unsigned long long rec_l = reinterpret_cast<unsigned long long>(
                a.partials + (static_cast<size_t>(cand < W ? cand : 0) * 2 + slot_l) * rec_floats);
            unsigned m = cm;
            while (m != 0) {
                const float* r0 = reinterpret_cast<const float*>(__shfl_sync(kFull, rec_l, __ffs(m) - 1));
                m &= m - 1;
                float m0, l0;
                float4 o0[NV];
                load_rec(r0, m0, l0, o0);
                if (NBATCH == 2 && m != 0) {
                    const float* r1 = reinterpret_cast<const float*>(__shfl_sync(kFull, rec_l, __ffs(m) - 1));
                    m &= m - 1;
                    float m1, l1;
                    float4 o1[NV];
                    load_rec(r1, m1, l1, o1);
                    combine(m0, l0, o0);
                    combine(m1, l1, o1);
                } else {
                    combine(m0, l0, o0);
                }
            }
            if (!(__ballot_sync(kFull, cand < W && c1 < U1) >> 31 & 1u)) break;  // the pair ends in this round
        }
        // out[s][query head u GU + r_row][d0 .. d0 + DPL), bf16
        const int hh = r_row / G;
        const float inv = Ls > 0.f ? out_mul(u, hh) / Ls : 0.f;
        uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) +
                        (static_cast<size_t>(s) * a.Hq + static_cast<size_t>(u) * GU + r_row) * D * 2 + d0 * 2;
        uint32_t wv[DPL / 2];
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e)
            wv[e] = static_cast<uint32_t>(float_to_bf16_bits(acc[2 * e] * inv)) |
                    (static_cast<uint32_t>(float_to_bf16_bits(acc[2 * e + 1] * inv)) << 16);
        if constexpr (DPL >= 8) {
#pragma unroll
            for (int i = 0; i < DPL / 8; ++i)
                *reinterpret_cast<uint4*>(orow + i * 16) = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
        } else {  // one query head per unit (GU = 1): 4 dims per lane
            *reinterpret_cast<uint2*>(orow) = make_uint2(wv[0], wv[1]);
        }
    };
    auto resolve_pending = [&]() {
        if (pend_s < 0) return;
        const int old = __shfl_sync(kFull, pend_old, 0);
        if (old + pend_blocks == P[pend_s + 1] - P[pend_s]) merge_pair(pend_s, pend_u);
        pend_s = -1;
    };
    int k = 0;
    int st = 0;       // stage of stream index k (k % depth)
    uint32_t ph = 0;  // its phase parity ((k / depth) & 1)
    while (k < n_blocks) {
        // ------------------------------------------------ one segment: consecutive blocks of one (s, unit) pair
        const int seg_x0 = A0 + k;
        // Q fragment quads per k-step: rows g (head 0 of the unit) and g + 8 (head 1, or zero), dims as this
        // thread's K operand holds them
        uint32_t qa[8][4];
        // O[g][dim] of head 0 in elements 0, 1 and of head 1 in elements 2, 3 of output tile n (dims: dim_of below)
        float o[16][4];
        float m_ref[HP], l_run[HP], qm[HP];
        float qoff[HP];  // INT8: 1152 times the row's query sum, taken off the scores of the biased key codes  // per head: running max of row g (log2 units), this thread's share of
                                             // the running sum, score scale
        int ma = 0, mc = 0, seg_first = 0;
        bool first = true;
        int x_last;

        // One 16-row MMA tile of the block for every head of the unit: head hh's K rows at kt + hh kTile, V rows
        // at vt + hh kTile (shared addresses of the tile's row 0), tv valid tokens (M: tv may be below the tile's
        // rows, the rest are stale and masked out).
        auto tile = [&](auto masked, uint32_t kt, uint32_t vt, int tv) {
            constexpr bool M = decltype(masked)::value;
            const int lim = M ? tv : TS;
            // K operand of one token row (at byte offset ro in each half of a K tile at kb): registers b0, b1 per
            // k-step
            auto k_frags = [&](uint32_t kb, uint32_t ro, bool present, uint32_t (&kf)[8][2]) {
                if constexpr (B16) {
                    const uint4 x0 = present ? lds128(kb + ro + kb0) : zero4;
                    const uint4 x1 = present ? lds128(kb + ro + kb1) : zero4;
                    const uint4 x2 = present ? lds128(kb + kHalf + ro + kb0) : zero4;
                    const uint4 x3 = present ? lds128(kb + kHalf + ro + kb1) : zero4;
                    const uint32_t w[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                            x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        kf[ks][0] = w[2 * ks];
                        kf[ks][1] = w[2 * ks + 1];
                    }
                } else {
                    const uint4 x0 = present ? lds128(kb + ro + kb0) : zero4;
                    const uint4 x1 = present ? lds128(kb + ro + kb1) : zero4;
                    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        if constexpr (KV::code == PKV_INT8) {
                            kf[ks][0] = s8x2_to_biased_f16x2<false>(w[ks]);
                            kf[ks][1] = s8x2_to_biased_f16x2<true>(w[ks]);
                        } else {
                            kf[ks][0] = codes2_to_f16x2<KV, false>(w[ks]);
                            kf[ks][1] = codes2_to_f16x2<KV, true>(w[ks]);
                        }
                    }
                }
            };
            const int t0 = 2 * t, t2 = 8 + 2 * t;
            uint32_t pq[HP][4];  // P quads: head 0 in rows 0-7, head 1 in rows 8-15
#pragma unroll
            for (int hh = 0; hh < HP; ++hh) {
                // ---- S = Q Kᵀ against head hh's keys: column tile 0 holds tokens 0-7, tile 1 tokens 8-15
                // (thread: tokens 2t, 2t+1 of each); head hh's scores are elements 2 hh, 2 hh + 1 of the quads
                float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    uint32_t kf[8][2];
                    k_frags(kt + hh * kTile, 0u, g < TS, kf);
                    float e0[4] = {0.f, 0.f, 0.f, 0.f};  // odd k-steps: a second accumulation chain
#pragma unroll
                    for (int ks = 0; ks < 8; ks += 2) {
                        mma_16816<B16>(s0, qa[ks], kf[ks][0], kf[ks][1]);
                        mma_16816<B16>(e0, qa[ks + 1], kf[ks + 1][0], kf[ks + 1][1]);
                    }
                    s0[2 * hh] += e0[2 * hh];
                    s0[2 * hh + 1] += e0[2 * hh + 1];
                    if constexpr (TS > 8) {
                        k_frags(kt + hh * kTile, 1024u, true, kf);
                        float e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int ks = 0; ks < 8; ks += 2) {
                            mma_16816<B16>(s1, qa[ks], kf[ks][0], kf[ks][1]);
                            mma_16816<B16>(e1, qa[ks + 1], kf[ks + 1][0], kf[ks + 1][1]);
                        }
                        s1[2 * hh] += e1[2 * hh];
                        s1[2 * hh + 1] += e1[2 * hh + 1];
                    }
                }
                // ---- online softmax of head hh's row g over the tile's tokens
                if constexpr (KV::code == PKV_INT8) {
                    s0[2 * hh] -= qoff[hh];
                    s0[2 * hh + 1] -= qoff[hh];
                    s1[2 * hh] -= qoff[hh];
                    s1[2 * hh + 1] -= qoff[hh];
                }
                const float sc0 = (t0 < lim) ? s0[2 * hh] * qm[hh] : -INFINITY;
                const float sc1 = (t0 + 1 < lim) ? s0[2 * hh + 1] * qm[hh] : -INFINITY;
                const float sc2 = (t2 < lim) ? s1[2 * hh] * qm[hh] : -INFINITY;
                const float sc3 = (t2 + 1 < lim) ? s1[2 * hh + 1] * qm[hh] : -INFINITY;
                float mb = fmaxf(fmaxf(sc0, sc1), fmaxf(sc2, sc3));
                mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 1));
                mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 2));
                const bool need = mb > m_ref[hh] + kLazyRescale;
                if (__any_sync(kFull, need)) {
                    const float m_new = need ? mb : m_ref[hh];
                    const float alpha = (m_new == m_ref[hh]) ? 1.f : ex2_approx(m_ref[hh] - m_new);
                    l_run[hh] *= alpha;
                    m_ref[hh] = m_new;
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        o[n][2 * hh] *= alpha;
                        o[n][2 * hh + 1] *= alpha;
                    }
                }
                const float p0 = ex2_approx(sc0 - m_ref[hh]), p1 = ex2_approx(sc1 - m_ref[hh]);
                const float p2 = ex2_approx(sc2 - m_ref[hh]), p3 = ex2_approx(sc3 - m_ref[hh]);
                l_run[hh] += (p0 + p1) + (p2 + p3);
                const uint32_t plo = pack2<B16>(p0, p1), phi = pack2<B16>(p2, p3);
                pq[hh][0] = hh == 0 ? plo : zr;
                pq[hh][1] = hh == 0 ? zr : plo;
                pq[hh][2] = hh == 0 ? phi : zr;
                pq[hh][3] = hh == 0 ? zr : phi;
            }
            // ---- O += P V per head: thread (g, t) supplies V rows 2t, 2t+1, 2t+8, 2t+9 of its chunk(s); rows
            // past the valid tokens are zero (stale rows may hold anything, and 0 * NaN would reach O)
#pragma unroll
            for (int hh = 0; hh < HP; ++hh)
#pragma unroll
                for (int hf = 0; hf < (B16 ? 2 : 1); ++hf) {
                    const uint32_t vh = vt + hh * kTile + hf * kHalf;
                    const uint4 v0 = (t0 < lim) ? lds128(vh + vb0) : zero4;
                    const uint4 v1 = (t0 + 1 < lim) ? lds128(vh + vb1) : zero4;
                    const uint4 v2 = (t2 < lim) ? lds128(vh + 1024 + vb0) : zero4;
                    const uint4 v3 = (t2 + 1 < lim) ? lds128(vh + 1024 + vb1) : zero4;
                    const uint32_t va[4] = {v0.x, v0.y, v0.z, v0.w}, vb[4] = {v1.x, v1.y, v1.z, v1.w};
                    const uint32_t vc[4] = {v2.x, v2.y, v2.z, v2.w}, vd[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if constexpr (B16) {
                            // word j holds dims 2j, 2j+1 of the chunk: output tiles 8 hf + 2j and 8 hf + 2j + 1
                            mma_16816<true>(o[8 * hf + 2 * j], pq[hh], __byte_perm(va[j], vb[j], 0x5410u),
                                            __byte_perm(vc[j], vd[j], 0x5410u));
                            mma_16816<true>(o[8 * hf + 2 * j + 1], pq[hh], __byte_perm(va[j], vb[j], 0x7632u),
                                            __byte_perm(vc[j], vd[j], 0x7632u));
                        } else {
                            // word j holds dims 4j .. 4j+3 of the chunk: output tiles 4j .. 4j+3
                            const uint32_t lo01 = pair_bytes<0>(va[j], vb[j]), lo23 = pair_bytes<0>(vc[j], vd[j]);
                            const uint32_t hi01 = pair_bytes<2>(va[j], vb[j]), hi23 = pair_bytes<2>(vc[j], vd[j]);
                            mma_16816<false>(o[4 * j], pq[hh], codes2_to_f16x2<KV, false>(lo01),
                                             codes2_to_f16x2<KV, false>(lo23));
                            mma_16816<false>(o[4 * j + 1], pq[hh], codes2_to_f16x2<KV, true>(lo01),
                                             codes2_to_f16x2<KV, true>(lo23));
                            mma_16816<false>(o[4 * j + 2], pq[hh], codes2_to_f16x2<KV, false>(hi01),
                                             codes2_to_f16x2<KV, false>(hi23));
                            mma_16816<false>(o[4 * j + 3], pq[hh], codes2_to_f16x2<KV, true>(hi01),
                                             codes2_to_f16x2<KV, true>(hi23));
                        }
                    }
                }
        };

        while (true) {
            const int x = A0 + k;
            if (x - wbase >= 32) {
                wbase += 32;
                cur = nxt;
                nxt = make_meta(wbase + 32 + lane);
            }
            const int src = x - wbase;
            ma = __shfl_sync(kFull, cur.a, src);
            mc = __shfl_sync(kFull, cur.c, src);
            if (!wait_stage(k, st, ph)) return;
            const uint32_t sp = wreg_u32 + static_cast<uint32_t>(st) * a.stage_bytes;
            if (first) {
                // Q of this (s, unit): for each head hh of the unit, row g, the head dims this thread's K operand
                // holds, in the same permuted k order (one-byte caches: dims 32t .. 32t+31, bf16 -> f16; bf16
                // caches: dims 16t .. 16t+15 and 64+16t .. 64+16t+15 as they are)
                prefetch_next_q(x);
                seg_first = mc & kMetaFirst;
                bool in_range = true;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) qa[ks][1] = qa[ks][3] = zr;
#pragma unroll
                for (int hh = 0; hh < HP; ++hh) {
                    const int hk = (ma & 1023) * HP + hh;  // the KV head
                    qm[hh] = a.k_head ? a.q_base * __ldg(a.k_head + hk) : a.q_mul;
                    m_ref[hh] = -INFINITY;
                    l_run[hh] = 0.f;
                    const uint4* qrow = reinterpret_cast<const uint4*>(
                        reinterpret_cast<const uint8_t*>(a.q) +
                        (static_cast<size_t>(ma >> 10) * a.Hq + static_cast<size_t>(hk) * G + g) * D * 2);
                    float qsum = 0.f;  // INT8: this thread's dims of row g
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int qi = B16 ? (i < 2 ? 2 * t + i : 8 + 2 * t + i - 2) : 4 * t + i;  // 16-byte units
                        const uint4 w4 = g < G ? __ldg(qrow + qi) : zero4;
                        uint32_t f[4];
                        if constexpr (B16) {
                            f[0] = w4.x;
                            f[1] = w4.y;
                            f[2] = w4.z;
                            f[3] = w4.w;
                        } else {
                            const float2 f0 = bf16x2_to_float2(w4.x), f1 = bf16x2_to_float2(w4.y);
                            const float2 f2 = bf16x2_to_float2(w4.z), f3 = bf16x2_to_float2(w4.w);
                            in_range = in_range &&
                                       fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y))) < 65520.f &&
                                       fmaxf(fmaxf(fabsf(f2.x), fabsf(f2.y)), fmaxf(fabsf(f3.x), fabsf(f3.y))) < 65520.f;
                            f[0] = pack2<false>(f0.x, f0.y);
                            f[1] = pack2<false>(f1.x, f1.y);
                            f[2] = pack2<false>(f2.x, f2.y);
                            f[3] = pack2<false>(f3.x, f3.y);
                            if constexpr (KV::code == PKV_INT8)
                                qsum += ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
                        }
                        // dims d, d+1 go to the k 2t register of the quad, d+2, d+3 to the k 2t+8 register; head 0
                        // in rows g (elements 0, 2), head 1 in rows g + 8 (elements 1, 3)
                        qa[2 * i][hh] = f[0];
                        qa[2 * i][2 + hh] = f[1];
                        qa[2 * i + 1][hh] = f[2];
                        qa[2 * i + 1][2 + hh] = f[3];
                    }
                    if constexpr (KV::code == PKV_INT8) {  // the row's sum over the 4 lanes that hold it
                        qsum += __shfl_xor_sync(kFull, qsum, 1);
                        qsum += __shfl_xor_sync(kFull, qsum, 2);
                        qoff[hh] = 1152.f * qsum;
                    }
                }
                if (!in_range) raise_error(a.err, PKV_DEVERR_Q_RANGE);
#pragma unroll
                for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
                first = false;
            }
            if (mc & kMetaOk) {
                const int valid = mc & 63;
#pragma unroll
                for (int ti = 0; ti < NT; ++ti) {
                    const int tv = valid - ti * TS;
                    if (tv <= 0) break;
                    const uint32_t kt = sp + ti * TS * 128, vt = sp + HP * kTile + ti * TS * 128;
                    if (tv >= TS) tile(std::false_type{}, kt, vt, TS);
                    else tile(std::true_type{}, kt, vt, tv);
                }
            }
            __syncwarp();

            // ---- refill this stage with stream index k + depth (issued by the lane holding its metadata)
            const int kn = k + a.depth;
            if (kn < n_blocks) {
                const int sn = A0 + kn - wbase;
                if (lane == (sn & 31)) {
                    fence_proxy_async_smem();
                    issue(st, sn < 32 ? cur : nxt);
                }
            }
            const bool last = (mc & kMetaLast) != 0 || x == A1 - 1;
            ++k;
            if (++st == a.depth) {
                st = 0;
                ph ^= 1u;
            }
            if (last) {
                x_last = x;
                break;
            }
        }

        // ------------------------------------------------ end of segment
        const int s = ma >> 10, u = ma & 1023;
        const int nb = P[s + 1] - P[s];
#pragma unroll
        for (int hh = 0; hh < HP; ++hh) {
            l_run[hh] += __shfl_xor_sync(kFull, l_run[hh], 1);
            l_run[hh] += __shfl_xor_sync(kFull, l_run[hh], 2);
        }
        const bool whole = seg_first && (mc & kMetaLast) && (x_last - seg_x0 + 1 == nb);
        if (whole) {
            if (g < G) {
#pragma unroll
                for (int hh = 0; hh < HP; ++hh) {
                    float v[32];
                    o_row(o, hh, v);
                    store_row(s, u, hh, v, l_run[hh] > 0.f ? out_mul(u, hh) / l_run[hh] : 0.f);
                }
            }
            resolve_pending();
            continue;
        }
        // partial record of this segment: O[GU][D], m[GU], l[GU] (row hh G + g for head hh).  A record is
        // GU * (D + 2) floats, so records are 16-byte aligned for even GU and only 8-byte aligned for GU = 1: the O
        // runs move as float4 or as float2 pairs.
        {
            const int slot = (seg_x0 == A0) ? 0 : 1;
            float* rec = a.partials + (static_cast<size_t>(w) * 2 + slot) * rec_floats;
            if (g < G) {
#pragma unroll
                for (int hh = 0; hh < HP; ++hh) {
                    float v[32];
                    o_row(o, hh, v);
                    const int row = hh * G + g;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float* dst = rec + row * D + dim_of(4 * i);
                        if constexpr (GU % 2 == 0) {
                            *reinterpret_cast<float4*>(dst) =
                                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        } else {
                            reinterpret_cast<float2*>(dst)[0] = make_float2(v[4 * i], v[4 * i + 1]);
                            reinterpret_cast<float2*>(dst)[1] = make_float2(v[4 * i + 2], v[4 * i + 3]);
                        }
                    }
                    if (t == 0) {
                        rec[GU * D + row] = m_ref[hh];
                        rec[GU * D + GU + row] = l_run[hh];
                    }
                }
            }
        }
        resolve_pending();  // the previous cut pair, whose ticket result has long arrived
        __threadfence();
        __syncwarp();
        pend_s = s;
        pend_u = u;
        pend_blocks = x_last - seg_x0 + 1;
        if (lane == 0) pend_old = atomicAdd(&a.tickets[static_cast<size_t>(s) * Hu + u], pend_blocks);
    }
    resolve_pending();
}
template <int G, int S, class KV, int HP>
__global__ void __launch_bounds__(32 * kMmaWarps, 1)
    paged_decode_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                            const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    decode_mma_body<G, S, KV, HP, false>(kmap, vmap, a, smem_raw, blockIdx.x, gridDim.x, blockDim.x, nullptr,
                                         nullptr);
}

// Host-side launch for one instantiation (defined in decode_mma_*.cu).
template <int G, int S, class KV, int HP>
cudaError_t launch_paged_decode_mma(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeArgs& a, int grid,
                                    int block, size_t smem, cudaStream_t stream) {
    auto kern = paged_decode_mma_kernel<G, S, KV, HP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, block, smem, stream>>>(kmap, vmap, a);
    return cudaGetLastError();
}

}  // namespace pkv
