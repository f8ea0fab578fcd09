// decode.cuh -- paged decode attention kernel (one query token per sequence).
//
// Method: for every (sequence s, KV head h) the kernel streams the K/V
// blocks named by the sequence's block table ("3.3 批处理与内存管理",
// "PagedAttention：块表": block = table[p / S], offset = p % S) and keeps the
// online-softmax state of "从 PagedAttention 到 Chunked Prefill" §2.2:
//   m_i = max(m_{i-1}, rowmax(S_i))
//   l_i = e^{m_{i-1}-m_i} l_{i-1} + rowsum(e^{S_i - m_i})
//   O_i = e^{m_{i-1}-m_i} O_{i-1} + e^{S_i - m_i} V_i          (out = O_N / l_N)
// (the page prints a stray inverse on the O rescale factor; the recurrence
// above is the one consistent with its l update and with exact softmax).
// The G query heads that share KV head h are processed together, so each
// K/V block is read from HBM once per KV head (GQA grouping).
//
// GB300 design:
//  * Persistent grid, one CTA of 8 warps per SM.  Each warp is an
//    independent worker with its own TMA pipeline of `depth` stages; a
//    stage holds one K tile and one V tile ([S][D] each, fetched by 3-D
//    bulk-tensor copies straight out of the [NB][S][Hkv][D] pool) plus, at
//    the start of a segment, the G query rows (1-D bulk copy).
//  * Work balance (split-KV): all (s, h) pairs are laid end to end, block
//    by block; the warps get equal contiguous shares of that stream.  A
//    pair cut by a share boundary yields partial (m, l, O) records, merged
//    by whichever worker finishes that pair last (block-count ticket, no
//    spinning).  `part_blocks` restricts where cuts may fall (1 = any
//    block boundary; >= every length = never cut).
//  * Math on CUDA cores in fp32: lanes split the head dimension (LPT lanes
//    per token, TP tokens at a time); QK^T partial dots use packed FFMA2 and
//    a reduce-scatter over the LPT lanes so each lane ends with one score;
//    the row max is a warp butterfly; probabilities reach the P.V lanes
//    through a small per-warp shared buffer.  The running max used for the
//    exponentials is only raised when a block's max exceeds it by more than
//    8 (log2 units), so the O rescale runs rarely; the result is the same
//    softmax up to rounding.
#pragma once

#include <type_traits>

#include "pkv_device.cuh"

namespace pkv {

// ------------------------------------------------------------------ element traits

struct KvF32 {
    static constexpr int es = 4;
    static constexpr int code = PKV_F32;
};
struct KvBF16 {
    static constexpr int es = 2;
    static constexpr int code = PKV_BF16;
};
struct KvE4M3 {
    static constexpr int es = 1;
    static constexpr int code = PKV_FP8_E4M3;
};
struct KvI8 {
    static constexpr int es = 1;
    static constexpr int code = PKV_INT8;
};

// Load CH bytes of KV elements from shared memory and widen to fp32 pairs.
template <class KV, int CH>
__device__ __forceinline__ void load_kv_chunk(const uint8_t* p, float2 (&x)[CH / KV::es / 2]) {
    if constexpr (KV::es == 4) {
        static_assert(CH == 16 || CH == 8, "f32 chunk");
        if constexpr (CH == 16) {
            float4 v = *reinterpret_cast<const float4*>(p);
            x[0] = make_float2(v.x, v.y);
            x[1] = make_float2(v.z, v.w);
        } else {
            x[0] = *reinterpret_cast<const float2*>(p);
        }
    } else if constexpr (KV::es == 2) {
        if constexpr (CH == 16) {
            uint4 v = *reinterpret_cast<const uint4*>(p);
            x[0] = bf16x2_to_float2(v.x);
            x[1] = bf16x2_to_float2(v.y);
            x[2] = bf16x2_to_float2(v.z);
            x[3] = bf16x2_to_float2(v.w);
        } else {
            uint2 v = *reinterpret_cast<const uint2*>(p);
            x[0] = bf16x2_to_float2(v.x);
            x[1] = bf16x2_to_float2(v.y);
        }
    } else if constexpr (KV::code == PKV_INT8) {
        if constexpr (CH == 16) {
            uint4 v = *reinterpret_cast<const uint4*>(p);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[2 * i] = s8x2_to_float2(w[i], 0);
                x[2 * i + 1] = s8x2_to_float2(w[i], 2);
            }
        } else {
            uint2 v = *reinterpret_cast<const uint2*>(p);
            x[0] = s8x2_to_float2(v.x, 0);
            x[1] = s8x2_to_float2(v.x, 2);
            x[2] = s8x2_to_float2(v.y, 0);
            x[3] = s8x2_to_float2(v.y, 2);
        }
    } else {
        if constexpr (CH == 16) {
            uint4 v = *reinterpret_cast<const uint4*>(p);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[2 * i] = e4m3x2_to_float2(static_cast<uint16_t>(w[i] & 0xffffu));
                x[2 * i + 1] = e4m3x2_to_float2(static_cast<uint16_t>(w[i] >> 16));
            }
        } else {
            uint2 v = *reinterpret_cast<const uint2*>(p);
            const uint32_t w[2] = {v.x, v.y};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                x[2 * i] = e4m3x2_to_float2(static_cast<uint16_t>(w[i] & 0xffffu));
                x[2 * i + 1] = e4m3x2_to_float2(static_cast<uint16_t>(w[i] >> 16));
            }
        }
    }
}

template <class QT>
__device__ __forceinline__ float load_q_elem(const uint8_t* base, int idx) {
    if constexpr (QT::es == 4) {
        return reinterpret_cast<const float*>(base)[idx];
    } else {
        const uint16_t b = reinterpret_cast<const uint16_t*>(base)[idx];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
}

// Store n consecutive fp32 values as QT (f32 or bf16) to global memory.
template <class QT, int N>
__device__ __forceinline__ void store_out(void* dst, const float (&v)[N]) {
    if constexpr (QT::es == 4) {
        static_assert(N % 4 == 0 || N == 2, "f32 store width");
        if constexpr (N % 4 == 0) {
#pragma unroll
            for (int i = 0; i < N; i += 4)
                reinterpret_cast<float4*>(dst)[i / 4] = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
            *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
        }
    } else {
        uint32_t w[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i)
            w[i] = static_cast<uint32_t>(float_to_bf16_bits(v[2 * i])) |
                   (static_cast<uint32_t>(float_to_bf16_bits(v[2 * i + 1])) << 16);
        if constexpr (N / 2 == 4) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        } else if constexpr (N / 2 == 2) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
        } else if constexpr (N / 2 == 1) {
            *reinterpret_cast<uint32_t*>(dst) = w[0];
        } else {
#pragma unroll
            for (int i = 0; i < N / 2; i += 4)
                reinterpret_cast<uint4*>(dst)[i / 4] = make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]);
        }
    }
}

// ------------------------------------------------------------------ shape of the lane mapping

// Launch policy per instantiation, chosen from measurements on GB300: the
// kernel is bound by instruction issue, so it trades query/accumulator
// registers (more lanes per token) for more resident warps when the GQA
// group is small, and keeps 8 warps with 64 query registers per lane for
// G * D >= 1024, where the extra reductions would cost more than the warps
// gain.  PKV_DECODE_QREGS / PKV_DECODE_WARPS override both (experiments).
template <int G, int D>
struct DecodePolicy {
#ifdef PKV_DECODE_QREGS
    static constexpr int qregs = PKV_DECODE_QREGS;
#else
    static constexpr int qregs = (G * D <= 512) ? 32 : 64;
#endif
#ifdef PKV_DECODE_WARPS
    static constexpr int warps = PKV_DECODE_WARPS;
#else
    static constexpr int warps = (qregs <= 32) ? 12 : 8;
#endif
};

template <int G, int D, class KV>
struct DecodeShape {
    static constexpr int LPT = (G * D / DecodePolicy<G, D>::qregs > 8) ? G * D / DecodePolicy<G, D>::qregs : 8;  // lanes per token
    static constexpr int TP = 32 / LPT;                              // tokens in flight per warp
    static constexpr int DPL = D / LPT;                              // head dims per lane
    static constexpr int RB = DPL * KV::es;                          // row bytes per lane
    static constexpr int CH = RB >= 16 ? 16 : RB;                    // bytes per chunk
    static constexpr int NCH = RB / CH;                              // chunks per lane and row
    static constexpr int EPC = CH / KV::es;                          // elements per chunk
    static constexpr int DUP = LPT / G;                              // lanes holding the same score
    // select-free score reduction (heads XOR-permuted per lane): measured 7% faster for G = 8, while the
    // HBM-bound G <= 4 instances ran 1-2% slower with it
    static constexpr bool XPERM = G >= 8;
    static_assert(LPT <= 32 && G <= LPT, "lane mapping");
    static_assert(EPC % 2 == 0 && DPL % 2 == 0, "pairs");
    static_assert(DPL == NCH * EPC, "chunking");
};

// ------------------------------------------------------------------ kernel arguments

struct DecodeArgs {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* tickets;     // [B * Hkv], zero on entry
    float* partials;      // [W][2][G*(D+2)]
    int32_t* err;         // nullable
    int B, Hq, Hkv, S, MB, NB;
    int part_blocks;      // atoms of the work split (>= 1)
    float q_mul;          // scale * log2(e) * k_scale
    float o_mul;          // v_scale
    float q_base;         // scale * log2(e)
    const float* k_head;  // per-KV-head scales replacing k_scale / v_scale (nullable)
    const float* v_head;
    int depth;            // pipeline stages per warp
    uint32_t kv_bytes;    // one K (or V) tile: S * D * es
    uint32_t q_bytes;     // G query rows: G * D * q_es
    uint32_t stage_bytes; // 2 * kv_bytes + q_bytes, rounded to 128
    uint32_t warp_bytes;  // per-warp shared region
    uint32_t prefix_bytes;
    uint64_t timeout_ns;
};

constexpr float kLazyRescale = 8.0f;   // log2 units: raise the running max only beyond this

// Largest s in [0, B) with P[s] <= key (P[0] = 0 <= key).
__device__ __forceinline__ int find_seq(const int* P, int B, int key) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P[mid] <= key) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The work split: the T = Hkv * sum(blocks) (sequence, KV head, block) items laid end to end,
// worker w owning [start(w), start(w + 1)).  Raw shares are floor(w * T / W), moved forward to
// the next allowed cut (a pair boundary, or a multiple of C blocks inside a pair).  All
// arithmetic is 32-bit: T < 2^31 is checked on the host, and floor(w * T / W) is formed as
// w * (T / W) + floor(w * (T % W) / W) with w * (T % W) < W^2.
// Optional weighting (a mixed step, where some CTAs start on the stream late): cb[c] .. cb[c + 1] is CTA c's part
// of the stream, split evenly among its 2^nw_shift workers before snapping.
struct WorkSplit {
    const int* P;
    int B, Hkv, T, C, W, tq, tr;
    const int* cb = nullptr;
    int nw_shift = 0;

    __device__ __forceinline__ int snap(int x) const {
        if (x >= T) return T;
        const int s = find_seq(P, B, x / Hkv);
        const int nb = P[s + 1] - P[s];
        const int local = x - Hkv * P[s];
        const int j = local % nb;
        if (j == 0) return x;
        const int up = (C >= nb) ? nb : ((j + C - 1) / C) * C;
        return x - j + (up < nb ? up : nb);
    }
    __device__ __forceinline__ int start(int w) const {
        if (w >= W) return T;
        if (cb != nullptr) {
            const int c = w >> nw_shift, i = w - (c << nw_shift);
            const int span = cb[c + 1] - cb[c];
            const float f = static_cast<float>(i) * (1.0f / static_cast<float>(1 << nw_shift));  // exact
            return snap(cb[c] + min(span, static_cast<int>(static_cast<float>(span) * f)));
        }
        return snap(w * tq + (w * tr) / W);
    }
};

// Reduce-scatter of V[0..N) over the lanes of an aligned LPT-lane group, afterwards each lane holding the full
// sum for head gl = lg / (LPT / G).
//   XPERM: the lanes keep their heads in XOR-permuted order, slot i of a lane holding head i ^ gl.  At every
//   halving step both partners then keep slots [0, N/2) and send slots [N/2, N) (the upper half of a lane's slots
//   is exactly the half of the heads its partner keeps), so no lane-dependent select is needed.
//   Otherwise slot i holds head i and the upper partner of each step swaps halves with two selects per value.
template <int N, int OFF, bool XPERM>
__device__ __forceinline__ float reduce_scatter(float* v, int lane) {
    if constexpr (OFF == 0) {
        return v[0];
    } else if constexpr (N > 1) {
        const bool upper = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            if constexpr (XPERM) {
                v[i] += __shfl_xor_sync(kFull, v[i + N / 2], OFF);
            } else {
                const float send = upper ? v[i] : v[i + N / 2];
                const float keep = upper ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(kFull, send, OFF);
            }
        }
        return reduce_scatter<N / 2, OFF / 2, XPERM>(v, lane);
    } else {
        v[0] += __shfl_xor_sync(kFull, v[0], OFF);
        return reduce_scatter<1, OFF / 2, XPERM>(v, lane);
    }
}

// ------------------------------------------------------------------ the kernel

// Packed per-block metadata, one block of the worker's stream per lane.
//   a = s * 1024 + h            (sequence, KV head)
//   b = physical block id
//   c = valid tokens | first << 6 (block 0 of its pair) | last << 7 (last block of its pair)
//       | ok << 8 (block id in range)
struct Meta {
    int a, b, c;
};
constexpr int kMetaFirst = 1 << 6, kMetaLast = 1 << 7, kMetaOk = 1 << 8;

template <int G, int D, int S, class KV, class QT>
__global__ void __launch_bounds__(32 * DecodePolicy<G, D>::warps, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const DecodeArgs a) {
    using SH = DecodeShape<G, D, KV>;
    constexpr int LPT = SH::LPT, TP = SH::TP, DPL = SH::DPL, CH = SH::CH, NCH = SH::NCH, EPC = SH::EPC;
    constexpr int DUP = SH::DUP;
    constexpr int HP = DPL / 2;              // float2 pairs per lane and head
    constexpr int TS = S < 16 ? S : 16;      // tokens per softmax tile
    constexpr int NT = S / TS;               // tiles per block
    constexpr int R = TS / TP;               // rounds per tile
    constexpr int ROW = D * KV::es;          // bytes of one token row of one head
    static_assert(TS % TP == 0 && S % TS == 0, "tiling");

    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NW = blockDim.x >> 5;
    const int B = a.B, Hkv = a.Hkv;

    // ---- 1. per-sequence block counts and their prefix sum (P[s] = blocks before s)
    int* P = reinterpret_cast<int*>(smem);
    {
        const int per = (B + blockDim.x - 1) / blockDim.x;
        const int s0 = tid * per;
        const int s1 = min(B, s0 + per);
        int local = 0;
        for (int s = s0; s < s1; ++s) {
            int L = a.context_lens[s];
            if (L < 0 || L > a.MB * S) {
                if (blockIdx.x == 0) raise_error(a.err, PKV_DEVERR_BAD_LENGTH);
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
        __syncthreads();
        int wbase = 0;
        for (int i = 0; i < warp; ++i) wbase += warp_tot[i];
        int run = wbase + incl - local;
        for (int s = s0; s < s1; ++s) {
            P[s] = run;
            int L = a.context_lens[s];
            if (L < 0 || L > a.MB * S) L = 0;
            run += (L + S - 1) / S;
        }
        if (tid == blockDim.x - 1) {
            int tot = 0;
            for (int i = 0; i < NW; ++i) tot += warp_tot[i];
            P[B] = tot;
        }
        __syncthreads();
    }

    // ---- 2. empty sequences get zero rows (spread over the CTAs)
    for (int s = blockIdx.x; s < B; s += gridDim.x) {
        if (P[s + 1] != P[s]) continue;
        const int n = a.Hq * D;
        for (int i = tid; i < n; i += blockDim.x) {
            if constexpr (QT::es == 4)
                reinterpret_cast<float*>(a.out)[static_cast<size_t>(s) * n + i] = 0.f;
            else
                reinterpret_cast<uint16_t*>(a.out)[static_cast<size_t>(s) * n + i] = 0;
        }
    }

    // ---- 3. this warp's shared region, barriers and share of the work stream
    uint8_t* wreg = smem + a.prefix_bytes + static_cast<size_t>(warp) * a.warp_bytes;
    float2* pbuf = reinterpret_cast<float2*>(wreg + static_cast<size_t>(a.depth) * a.stage_bytes);
    float2* abuf = pbuf + 16 * G;
    uint64_t* bars = reinterpret_cast<uint64_t*>(abuf + G);
    const uint32_t wreg_u32 = smem_u32(wreg);
    const uint32_t bars_u32 = smem_u32(bars);
    if (lane == 0) {
        for (int i = 0; i < a.depth; ++i) mbar_init(bars_u32 + 8 * i, 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int T = Hkv * P[B];
    if (T == 0) return;
    // never more shares than blocks, so that no share is empty when cuts may fall anywhere
    const int W = min(static_cast<int>(gridDim.x) * NW, T);
    const int w = blockIdx.x * NW + warp;
    const WorkSplit split{P, B, Hkv, T, a.part_blocks, W, T / W, T % W};
    const int A0 = split.start(w);
    const int A1 = split.start(w + 1);
    if (A0 >= A1) return;
    if (lane == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    const uint64_t pol = policy_evict_first();

    const int tp = lane / LPT, lg = lane % LPT;
    const int gl = lg / DUP;  // the query head whose score this lane holds

    // Stream position x -> packed metadata (computed by the lane that owns x).
    auto make_meta = [&](int x) -> Meta {
        Meta m{0, -1, 0};
        if (x >= A1) return m;
        const int s = find_seq(P, B, x / Hkv);
        const int local = x - Hkv * P[s];
        const int nb = P[s + 1] - P[s];
        const int h = local / nb;
        const int j = local - h * nb;
        const int L = a.context_lens[s];
        m.a = s * 1024 + h;
        m.b = a.block_tables[static_cast<size_t>(s) * a.MB + j];
        const int valid = min(S, L - j * S);
        m.c = valid | (j == 0 ? kMetaFirst : 0) | (j == nb - 1 ? kMetaLast : 0) |
              ((m.b >= 0 && m.b < a.NB) ? kMetaOk : 0);
        return m;
    };

    // Issue the copies of stream index k (position A0 + k) into stage k % depth.
    // Called by the one lane that holds the block's metadata.
    auto issue = [&](int k, const Meta& m) {
        const int st = static_cast<int>(k % a.depth);
        const bool seg_start = (m.c & kMetaFirst) || (k == 0);
        const bool ok = (m.c & kMetaOk) != 0;
        if (!ok) raise_error(a.err, PKV_DEVERR_BAD_BLOCK);
        const uint32_t tx = (ok ? 2u * a.kv_bytes : 0u) + (seg_start ? a.q_bytes : 0u);
        const uint32_t bar = bars_u32 + 8 * st;
        const uint32_t dst = wreg_u32 + st * a.stage_bytes;
        if (tx) mbar_arrive_expect_tx(bar, tx); else mbar_arrive(bar);
        const int s = m.a >> 10, h = m.a & 1023;
        if (ok) {
            tma_load_3d(dst, &kmap, 0, h, m.b * S, bar, pol);
            tma_load_3d(dst + a.kv_bytes, &vmap, 0, h, m.b * S, bar, pol);
        }
        if (seg_start) {
            const uint8_t* src = reinterpret_cast<const uint8_t*>(a.q) +
                                 (static_cast<size_t>(s) * a.Hq + static_cast<size_t>(h) * G) * D * QT::es;
            bulk_load(dst + 2 * a.kv_bytes, src, a.q_bytes, bar);
        }
    };

    const int n_blocks = A1 - A0;
    int wbase = A0;
    Meta cur = make_meta(wbase + lane);
    Meta nxt = make_meta(wbase + 32 + lane);

    // prologue: fill the pipeline (lane k issues stream index k)
    if (lane < a.depth && lane < n_blocks) {
        fence_proxy_async_smem();
        issue(lane, cur);
    }

    // Bounded wait for stage k; on timeout record the error and drain the
    // copies still in flight (also bounded) so the warp can leave safely.
    auto wait_stage = [&](int k) -> bool {
        const int st = static_cast<int>(k % a.depth);
        if (mbar_wait_bounded(bars_u32 + 8 * st, static_cast<uint32_t>((k / a.depth) & 1), a.timeout_ns))
            return true;
        raise_error(a.err, PKV_DEVERR_TIMEOUT);
        for (int kk = k + 1; kk < k + a.depth && kk < n_blocks; ++kk)
            mbar_wait_bounded(bars_u32 + 8 * static_cast<int>(kk % a.depth),
                              static_cast<uint32_t>((kk / a.depth) & 1), a.timeout_ns);
        return false;
    };

    const size_t rec_floats = static_cast<size_t>(G) * (D + 2);
    // out[s][h G + g], this lane's dims, scaled by inv (lanes with tp == 0 store)
    auto store_rows = [&](int s, int h, const float2 (&o)[G][HP], const float (&inv)[G]) {
        if (tp != 0) return;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) +
                            (static_cast<size_t>(s) * a.Hq + static_cast<size_t>(h) * G + g) * D * QT::es;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                float v[EPC];
#pragma unroll
                for (int e = 0; e < EPC / 2; ++e) {
                    v[2 * e] = o[g][c * (EPC / 2) + e].x * inv[g];
                    v[2 * e + 1] = o[g][c * (EPC / 2) + e].y * inv[g];
                }
                store_out<QT, EPC>(orow + static_cast<size_t>((c * LPT + lg) * EPC) * QT::es, v);
            }
        }
    };
    // Merge of pair (s, h) by its last finisher: the shares that hold a segment of it are found 32 workers at a
    // time (one per lane; shares are contiguous in worker order) and their records combined in stream order.
    // Every lane works on the merge: lane (head g, part c) owns dims [c MDP, (c + 1) MDP) of query head h G + g,
    // and the loads of two records are in flight together.
    auto merge_pair = [&](int s, int h) {
        constexpr int MLR = 32 / G;   // lanes per query head
        constexpr int MDP = D / MLR;  // dims per lane (8-byte pairs: records of one head are 8-byte aligned only)
        const int r_g = lane / MLR, d0 = (lane % MLR) * MDP;
        __threadfence();
        const int nb = P[s + 1] - P[s];
        const int U0 = Hkv * P[s] + h * nb;
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
        float Mx = -INFINITY, Ls = 0.f, acc[MDP];
#pragma unroll
        for (int i = 0; i < MDP; ++i) acc[i] = 0.f;
        auto load_rec = [&](const float* r, float& m, float& l, float2 (&ov)[MDP / 2]) {
            m = __ldcg(r + G * D + r_g);
            l = __ldcg(r + G * D + G + r_g);
#pragma unroll
            for (int i = 0; i < MDP / 2; ++i) ov[i] = __ldcg(reinterpret_cast<const float2*>(r + r_g * D + d0) + i);
        };
        auto combine = [&](float m, float l, const float2 (&ov)[MDP / 2]) {
            const float mn = fmaxf(Mx, m);
            const float fo = (Mx == -INFINITY) ? 0.f : ex2_approx(Mx - mn);
            const float fr = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
            Ls = Ls * fo + l * fr;
            Mx = mn;
#pragma unroll
            for (int i = 0; i < MDP / 2; ++i) {
                acc[2 * i] = acc[2 * i] * fo + ov[i].x * fr;
                acc[2 * i + 1] = acc[2 * i + 1] * fo + ov[i].y * fr;
            }
        };
        for (int base = w_first; base < W; base += 32) {
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
                float2 o0[MDP / 2];
                load_rec(r0, m0, l0, o0);
                if (m != 0) {
                    const float* r1 = reinterpret_cast<const float*>(__shfl_sync(kFull, rec_l, __ffs(m) - 1));
                    m &= m - 1;
                    float m1, l1;
                    float2 o1[MDP / 2];
                    load_rec(r1, m1, l1, o1);
                    combine(m0, l0, o0);
                    combine(m1, l1, o1);
                } else {
                    combine(m0, l0, o0);
                }
            }
            if (!(__ballot_sync(kFull, cand < W && c1 < U1) >> 31 & 1u)) break;  // the pair ends in this round
        }
        const float inv = (Ls > 0.f) ? (a.v_head ? __ldg(a.v_head + h) : a.o_mul) / Ls : 0.f;
#pragma unroll
        for (int i = 0; i < MDP; ++i) acc[i] *= inv;
        uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) +
                        (static_cast<size_t>(s) * a.Hq + static_cast<size_t>(h) * G + r_g) * D * QT::es;
        store_out<QT, MDP>(orow + static_cast<size_t>(d0) * QT::es, acc);
    };
    // A cut pair's ticket: the atomic's result is read only at the next segment's end (or at the end of the
    // share), so that its round trip does not stall the stream; the last finisher then merges the pair.
    int pend_s = -1, pend_h = 0, pend_blocks = 0, pend_old = 0;
    auto resolve_pending = [&]() {
        if (pend_s < 0) return;
        const int old = __shfl_sync(kFull, pend_old, 0);
        if (old + pend_blocks == P[pend_s + 1] - P[pend_s]) merge_pair(pend_s, pend_h);
        pend_s = -1;
    };

    int k = 0;
    while (k < n_blocks) {
        // ------------------------------------------------ one segment: consecutive blocks of one (s, h) pair
        const int seg_x0 = A0 + k;
        float2 q2[G][HP];
        float2 o2[G][HP];
        float m_ref = -INFINITY;  // running max of head gl (log2 units), uniform over lanes holding gl
        float l_run = 0.f;        // this lane's share of the running sum of head gl
        int ma = 0, mc = 0, seg_first = 0;
        bool first = true;
        int x_last;
            // One softmax tile (TS tokens) of the block in this stage; M = some tokens are past the end.
            auto tile = [&](auto masked, const uint8_t* sp, int ti, int tv) {
                constexpr bool M = decltype(masked)::value;
                    const uint8_t* Ks = sp + ti * TS * ROW + (lg * CH);
                    const uint8_t* Vs = sp + a.kv_bytes + ti * TS * ROW + (lg * CH);
                    // ---- scores of this tile
                    float sr[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int t = r * TP + tp;
                        float2 acc[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            float2 kx[EPC / 2];
                            load_kv_chunk<KV, CH>(Ks + t * ROW + c * LPT * CH, kx);
#pragma unroll
                            for (int e = 0; e < EPC / 2; ++e)
#pragma unroll
                                for (int g = 0; g < G; ++g)
                                    acc[g] = __ffma2_rn(q2[g][c * (EPC / 2) + e], kx[e], acc[g]);
                        }
                        float v[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) v[g] = acc[g].x + acc[g].y;
                        const float sc = reduce_scatter<G, LPT / 2, SH::XPERM>(v, lane);
                        sr[r] = (!M || t < tv) ? sc : -INFINITY;
                    }
                    // ---- tile max over all tokens (butterfly over the token groups)
                    float mb = sr[0];
#pragma unroll
                    for (int r = 1; r < R; ++r) mb = fmaxf(mb, sr[r]);
#pragma unroll
                    for (int o = LPT; o < 32; o <<= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o));
                    const bool need = mb > m_ref + kLazyRescale;
                    if (__any_sync(kFull, need)) {
                        const float m_new = need ? mb : m_ref;
                        const float alpha = (m_new == m_ref) ? 1.f : ex2_approx(m_ref - m_new);
                        l_run *= alpha;
                        m_ref = m_new;
                        if (tp == 0 && (lg % DUP) == 0) abuf[gl] = make_float2(alpha, alpha);
                        __syncwarp();
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float2 al = abuf[g];
#pragma unroll
                            for (int i = 0; i < HP; ++i) o2[g][i] = __fmul2_rn(o2[g][i], al);
                        }
                    }
                    // ---- probabilities relative to the running max
                    float lsum = 0.f;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float p = (!M || sr[r] != -INFINITY) ? ex2_approx(sr[r] - m_ref) : 0.f;
                        lsum += p;
                        if ((lg % DUP) == 0) pbuf[(r * TP + tp) * G + gl] = make_float2(p, p);
                    }
                    l_run += lsum;
                    __syncwarp();
                    // ---- P.V
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int t = r * TP + tp;
                        if (!M || t < tv) {
                            float2 pp[G];
#pragma unroll
                            for (int g = 0; g < G; ++g) pp[g] = pbuf[t * G + g];
#pragma unroll
                            for (int c = 0; c < NCH; ++c) {
                                float2 vx[EPC / 2];
                                load_kv_chunk<KV, CH>(Vs + t * ROW + c * LPT * CH, vx);
#pragma unroll
                                for (int e = 0; e < EPC / 2; ++e)
#pragma unroll
                                    for (int g = 0; g < G; ++g)
                                        o2[g][c * (EPC / 2) + e] = __ffma2_rn(pp[g], vx[e], o2[g][c * (EPC / 2) + e]);
                            }
                        }
                    }
                    __syncwarp();
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
            if (!wait_stage(k)) return;
            const uint8_t* sp = wreg + static_cast<size_t>(k % a.depth) * a.stage_bytes;
            if (first) {
                seg_first = mc & kMetaFirst;
                const uint8_t* qs = sp + 2 * a.kv_bytes;
                const float qm = a.k_head ? a.q_base * __ldg(a.k_head + (ma & 1023)) : a.q_mul;
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
#pragma unroll
                        for (int e = 0; e < EPC; e += 2) {
                            const int d = (c * LPT + lg) * EPC + e;
                            // with XPERM slot g holds head g ^ gl (the order the reduce-scatter of the scores expects)
                            const int hq = (SH::XPERM ? (g ^ gl) : g) * D + d;
                            q2[g][(c * EPC + e) / 2] = make_float2(load_q_elem<QT>(qs, hq) * qm,
                                                                   load_q_elem<QT>(qs, hq + 1) * qm);
                            o2[g][(c * EPC + e) / 2] = make_float2(0.f, 0.f);
                        }
                first = false;
            }
            if (mc & kMetaOk) {
                const int valid = mc & 63;
                if (valid == S) {
#pragma unroll
                    for (int ti = 0; ti < NT; ++ti) tile(std::false_type{}, sp, ti, TS);
                } else {
#pragma unroll
                    for (int ti = 0; ti < NT; ++ti) {
                        const int tv = valid - ti * TS;
                        if (tv <= 0) break;
                        if (tv >= TS) tile(std::false_type{}, sp, ti, TS);
                        else tile(std::true_type{}, sp, ti, tv);
                    }
                }
            }
            __syncwarp();

            // ---- refill this stage with stream index k + depth (issued by the lane holding its metadata)
            const int kn = k + a.depth;
            if (kn < n_blocks) {
                const int sn = A0 + kn - wbase;
                if (lane == (sn & 31)) {
                    fence_proxy_async_smem();
                    issue(kn, sn < 32 ? cur : nxt);
                }
            }
            const bool last = (mc & kMetaLast) != 0 || x == A1 - 1;
            ++k;
            if (last) {
                x_last = x;
                break;
            }
        }

        // ------------------------------------------------ end of segment
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int i = 0; i < HP; ++i) {
                    o2[g][i].x += __shfl_xor_sync(kFull, o2[g][i].x, o);
                    o2[g][i].y += __shfl_xor_sync(kFull, o2[g][i].y, o);
                }
            l_run += __shfl_xor_sync(kFull, l_run, o);
        }
        const int s = ma >> 10, h = ma & 1023;
        const int nb = P[s + 1] - P[s];
        const bool whole = seg_first && (mc & kMetaLast) && (x_last - seg_x0 + 1 == nb);
        if (whole) {
            float inv[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float l_all = __shfl_sync(kFull, l_run, g * DUP);
                inv[g] = (l_all > 0.f) ? (a.v_head ? __ldg(a.v_head + h) : a.o_mul) / l_all : 0.f;
            }
            store_rows(s, h, o2, inv);
            resolve_pending();
            continue;
        }
        // partial record of this segment: O[G][D], m[G], l[G]
        {
            const int slot = (seg_x0 == A0) ? 0 : 1;
            float* rec = a.partials + (static_cast<size_t>(w) * 2 + slot) * rec_floats;
            if (tp == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
#pragma unroll
                        for (int e = 0; e < EPC / 2; ++e)
                            *reinterpret_cast<float2*>(rec + g * D + (c * LPT + lg) * EPC + 2 * e) =
                                o2[g][c * (EPC / 2) + e];
            }
            if (tp == 0 && (lg % DUP) == 0) {
                rec[G * D + gl] = m_ref;
                rec[G * D + G + gl] = l_run;
            }
        }
        resolve_pending();  // the previous cut pair, whose ticket result has long arrived
        __threadfence();
        __syncwarp();
        pend_s = s;
        pend_h = h;
        pend_blocks = x_last - seg_x0 + 1;
        if (lane == 0) pend_old = atomicAdd(&a.tickets[static_cast<size_t>(s) * Hkv + h], pend_blocks);
    }
    resolve_pending();
}

// Host-side launch for one instantiation (defined in the per-dtype .cu files).
template <int G, int D, int S, class KV, class QT>
cudaError_t launch_paged_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeArgs& a, int grid,
                                int block, size_t smem, cudaStream_t stream) {
    auto kern = paged_decode_kernel<G, D, S, KV, QT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, block, smem, stream>>>(kmap, vmap, a);
    return cudaGetLastError();
}

}  // namespace pkv
