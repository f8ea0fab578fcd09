/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for paged KV-cache decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or constant table
 * with the CUDA library; it is written from the pages' statement of the
 * method, not from the kernels.
 *
 * Sources (web pages, cited by title and section):
 *   [BMM]  "3.3 批处理与内存管理" (Batching and Memory Management),
 *          llm-learning-path part 3 -- sections "PagedAttention：块表"
 *          (block table equation and the worked example "例子"),
 *          "共享与写时复制" (sharing and copy-on-write), "分块预填充"
 *          (chunked prefill), "代码" (block allocator listing).
 *   [PAC]  "从 PagedAttention 到 Chunked Prefill" (ybb.press) -- §2.2
 *          online-softmax equations.
 *   [KVO]  "大模型推理的KV Cache优化全解" teaser on the PagedAttention tag
 *          page (guijiagi.com) -- §1.1 attention definition, the KVBlock
 *          layout [n_layers, block_size, n_kv_heads, head_dim], the GQA row
 *          of the technique table, the FP8 KV-cache paragraph.
 *
 * What is computed (the plain definition the method reaches exactly):
 *   out[s][hq] = softmax(scale * q[s][hq] . K_s^T) V_s
 * where K_s, V_s are the sequence's keys/values gathered in logical order
 * through its block table ([BMM] block-table equation):
 *   physical block = table[p / S],  offset = p % S.
 * Everything is evaluated in double precision with a two-pass (max, then
 * exp-sum) softmax; no blocking, fusion or reordering beyond that.
 *
 * Readings taken where the pages are silent (also listed in the design notes):
 *   - cache layout per layer: [num_blocks][S][Hkv][D], K and V separate
 *     (the KVBlock layout of [KVO] without the layer axis);
 *   - GQA: query head hq uses KV head hq / G, G = Hq / Hkv (contiguous groups);
 *   - slot = physical_block * S + offset; a negative slot is a padding token;
 *   - context length L_s includes the token written in this step;
 *   - L_s == 0 gives an all-zero output row;
 *   - FP8 is OCP E4M3 (bias 7, no infinities, S.1111.111 is NaN), with one
 *     fp32 scale per tensor: code = sat(RNE(x / scale)), value = code * scale;
 *     x / scale is an fp32 division, the precision the kernel uses to decide
 *     the code;
 *   - INT8 is symmetric: code = clamp(RNE(x / scale), -127, 127), value =
 *     code * scale, one fp32 scale per tensor;
 *   - per-head scales (optional, FP8 and INT8): one fp32 scale per KV head
 *     replaces the per-tensor scale of that head, in the write and the read;
 *   - bf16 values widen exactly; fp32 -> bf16 is round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_I8 = 3 };

enum {
    ORC_OK = 0,
    ORC_BAD_ARG = 1,
    ORC_BAD_SLOT = 2,
    ORC_BAD_BLOCK = 3,
    ORC_NO_MEMORY = 4
};

/* ------------------------------------------------------------------ */
/* Element formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even.  The two candidates are the
 * bf16 values next to x (the truncation toward zero and the next one away
 * from zero); the nearer one wins, a tie goes to the even significand. */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u = f32_bits(x);
    if (isnan(x))
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t lo_bits = u & 0xFFFF0000u;
    uint32_t hi_bits = lo_bits + 0x10000u; /* next magnitude up (may be inf) */
    double lo = fabs((double)f32_from_bits(lo_bits));
    double hi = fabs((double)f32_from_bits(hi_bits));
    double a = fabs((double)x);
    double dlo = a - lo, dhi = hi - a;
    uint32_t pick;
    if (dlo < dhi)
        pick = lo_bits;
    else if (dhi < dlo)
        pick = hi_bits;
    else
        pick = (((lo_bits >> 16) & 1u) == 0) ? lo_bits : hi_bits;
    return (uint16_t)(pick >> 16);
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; the only
 * NaN encodings are S.1111.111; there are no infinities; max finite 448. */
double orc_e4m3_to_double(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Quantise an fp32 value to E4M3 with saturation: the nearest finite code
 * (searched over all 127 non-negative finite codes), ties to the code with
 * an even mantissa; magnitudes at or beyond 448 clamp to 448; the sign is
 * kept (so tiny negatives give negative zero).  NaN maps to 0x7F. */
uint8_t orc_f32_to_e4m3(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_to_double((uint8_t)c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* Symmetric INT8 with a per-tensor scale ("从 PagedAttention 到 Chunked
 * Prefill" §5.4; the INT8 row of "大模型推理的KV Cache优化全解"): the code is
 * x / scale (an fp32 division) rounded to the nearest integer, ties to even,
 * and clamped to [-127, 127]; the value is code * scale.  NaN maps to 0. */
int8_t orc_f32_to_i8(float y)
{
    if (isnan(y))
        return 0;
    double r = rint((double)y); /* default rounding mode: ties to even */
    if (r > 127.0)
        r = 127.0;
    if (r < -127.0)
        r = -127.0;
    return (int8_t)r;
}

static int narrow_dt(int dt)
{
    return dt == ORC_E4M3 || dt == ORC_I8;
}

static size_t elem_size(int dt)
{
    return dt == ORC_F32 ? 4 : dt == ORC_BF16 ? 2 : 1;
}

/* Read element i of an array of dtype dt as a double (fp8: code * scale). */
static double load_elem(const void *base, int dt, size_t i, double fp8_scale)
{
    if (dt == ORC_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * i, 4);
        return (double)f;
    }
    if (dt == ORC_BF16) {
        uint16_t b;
        memcpy(&b, (const char *)base + 2 * i, 2);
        return orc_bf16_to_double(b);
    }
    if (dt == ORC_I8)
        return (double)((const int8_t *)base)[i] * fp8_scale;
    return orc_e4m3_to_double(((const uint8_t *)base)[i]) * fp8_scale;
}

/* ------------------------------------------------------------------ */
/* Block-table indexing ([BMM] "PagedAttention：块表", equation)         */
/* ------------------------------------------------------------------ */

/* Token at logical position p of a sequence lives in physical block
 * table[p / S] at offset p % S.  Returns the physical block id. */
int orc_lookup(const int32_t *table, int64_t p, int S, int *offset)
{
    *offset = (int)(p % S);
    return table[p / S];
}

/* ------------------------------------------------------------------ */
/* Cache write (reshape_and_cache)                                      */
/* ------------------------------------------------------------------ */

/* Each new token i is appended at slot[i] ([KVO] §1.1: the new k_t, v_t are
 * appended to the cache; [BMM] listing, append_token).  The slot encodes
 * (block, offset) as block * S + offset.  k_new/v_new: [T][Hkv][D] of
 * src_dt; caches: [NB][S][Hkv][D] of cache_dt.  Same dtype: bit copy.
 * bf16 -> f32 widens; f32 -> bf16 rounds to nearest even; -> E4M3 stores
 * sat(RNE(x / scale)) with the division in fp32, scale being the per-head
 * scale of the element's KV head when k_head_scales / v_head_scales are
 * given (NULL: the per-tensor scale).
 * Returns ORC_BAD_SLOT (after writing every valid token) if any slot is
 * beyond the pool. */
int orc_reshape_and_cache(const void *k_new, const void *v_new, int src_dt,
                          const int64_t *slot, int T, void *k_cache,
                          void *v_cache, int cache_dt, int NB, int S, int Hkv,
                          int D, float k_scale, float v_scale,
                          const float *k_head_scales, const float *v_head_scales)
{
    if (T < 0 || NB <= 0 || S <= 0 || Hkv <= 0 || D <= 0)
        return ORC_BAD_ARG;
    if (narrow_dt(src_dt))
        return ORC_BAD_ARG;
    int status = ORC_OK;
    const size_t row = (size_t)Hkv * D;
    for (int i = 0; i < T; ++i) {
        int64_t sl = slot[i];
        if (sl < 0)
            continue;
        if (sl >= (int64_t)NB * S) {
            status = ORC_BAD_SLOT;
            continue;
        }
        int64_t blk = sl / S, off = sl % S;
        size_t dst0 = ((size_t)blk * S + (size_t)off) * row;
        for (int kv = 0; kv < 2; ++kv) {
            const void *src = kv ? v_new : k_new;
            void *dst = kv ? v_cache : k_cache;
            const float *head_scales = kv ? v_head_scales : k_head_scales;
            for (size_t e = 0; e < row; ++e) {
                float scale = head_scales ? head_scales[e / (size_t)D] : (kv ? v_scale : k_scale);
                size_t si = (size_t)i * row + e, di = dst0 + e;
                if (src_dt == cache_dt) {
                    size_t es = elem_size(src_dt);
                    memcpy((char *)dst + es * di, (const char *)src + es * si, es);
                    continue;
                }
                float x = (float)load_elem(src, src_dt, si, 1.0);
                if (cache_dt == ORC_F32) {
                    memcpy((char *)dst + 4 * di, &x, 4);
                } else if (cache_dt == ORC_BF16) {
                    uint16_t b = orc_f32_to_bf16(x);
                    memcpy((char *)dst + 2 * di, &b, 2);
                } else if (cache_dt == ORC_I8) {
                    float y = x / scale;
                    ((int8_t *)dst)[di] = orc_f32_to_i8(y);
                } else {
                    float y = x / scale;
                    ((uint8_t *)dst)[di] = orc_f32_to_e4m3(y);
                }
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------ */
/* Block copy for copy-on-write ([BMM] "共享与写时复制")                 */
/* ------------------------------------------------------------------ */

/* For each (src, dst) pair, in order, the whole physical block dst of both
 * caches becomes a byte copy of block src.  block_bytes is S*Hkv*D*elem. */
int orc_copy_blocks(void *k_cache, void *v_cache, size_t block_bytes, int NB,
                    const int64_t *pairs, int n)
{
    int status = ORC_OK;
    for (int i = 0; i < n; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= NB || d < 0 || d >= NB) {
            status = ORC_BAD_BLOCK;
            continue;
        }
        memmove((char *)k_cache + (size_t)d * block_bytes,
                (const char *)k_cache + (size_t)s * block_bytes, block_bytes);
        memmove((char *)v_cache + (size_t)d * block_bytes,
                (const char *)v_cache + (size_t)s * block_bytes, block_bytes);
    }
    return status;
}

/* Swap blocks between two pools (preemption: a preempted sequence's KV is
 * swapped out to CPU memory and back in later -- "从 PagedAttention 到 Chunked
 * Prefill" §3.1; "3.3 批处理与内存管理", scheduling and preemption).  For each
 * (src, dst) pair, block dst of the destination pool becomes a byte copy of
 * block src of the source pool, for K and for V. */
int orc_swap_blocks(const void *src_k, const void *src_v, int src_nb, void *dst_k,
                    void *dst_v, int dst_nb, size_t block_bytes,
                    const int64_t *pairs, int n)
{
    int status = ORC_OK;
    for (int i = 0; i < n; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= src_nb || d < 0 || d >= dst_nb) {
            status = ORC_BAD_BLOCK;
            continue;
        }
        memcpy((char *)dst_k + (size_t)d * block_bytes,
               (const char *)src_k + (size_t)s * block_bytes, block_bytes);
        memcpy((char *)dst_v + (size_t)d * block_bytes,
               (const char *)src_v + (size_t)s * block_bytes, block_bytes);
    }
    return status;
}

/* ------------------------------------------------------------------ */
/* Content hashes of full blocks (prefix caching)                       */
/* ------------------------------------------------------------------ */

/* FNV-1a, 64-bit (Fowler-Noll-Vo): start from the offset basis
 * 14695981039346656037; for each byte, xor it in, then multiply by the
 * prime 1099511628211 modulo 2^64. */
uint64_t orc_fnv1a64(const uint8_t *bytes, size_t n, uint64_t h)
{
    for (size_t i = 0; i < n; ++i) {
        h ^= (uint64_t)bytes[i];
        h *= 1099511628211ull;
    }
    return h;
}

#define ORC_FNV_BASIS 14695981039346656037ull

static void put_le64(uint8_t *b, uint64_t v)
{
    for (int i = 0; i < 8; ++i)
        b[i] = (uint8_t)(v >> (8 * i));
}

/* Hash-based prefix caching ("3.3 批处理与内存管理", "前缀缓存与
 * RadixAttention"): every FULL block is identified by its own tokens together
 * with the hash of all blocks before it.  Definition used here:
 *   d_j = FNV-1a-64 over the block's S token ids, each as 4 little-endian bytes
 *   h_0 = FNV-1a-64 over (8 zero bytes) ++ (d_0 as 8 little-endian bytes)
 *   h_j = FNV-1a-64 over (h_{j-1} as 8 LE bytes) ++ (d_j as 8 LE bytes)
 * Sequence s has tokens [cu_tokens[s], cu_tokens[s+1]) and floor(L_s / S) full
 * blocks, whose hashes go to out[out_offsets[s] + j]. */
void orc_block_hashes(const int32_t *tokens, const int64_t *cu_tokens, int B, int S,
                      const int64_t *out_offsets, uint64_t *out)
{
    for (int s = 0; s < B; ++s) {
        int64_t L = cu_tokens[s + 1] - cu_tokens[s];
        int64_t nfull = L / S;
        uint64_t prev = 0;
        for (int64_t j = 0; j < nfull; ++j) {
            uint64_t d = ORC_FNV_BASIS;
            for (int t = 0; t < S; ++t) {
                uint8_t b[4];
                uint32_t v = (uint32_t)tokens[cu_tokens[s] + j * S + t];
                for (int i = 0; i < 4; ++i)
                    b[i] = (uint8_t)(v >> (8 * i));
                d = orc_fnv1a64(b, 4, d);
            }
            uint8_t buf[16];
            put_le64(buf, prev);
            put_le64(buf + 8, d);
            prev = orc_fnv1a64(buf, 16, ORC_FNV_BASIS);
            out[out_offsets[s] + j] = prev;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Gather and textbook attention                                        */
/* ------------------------------------------------------------------ */

typedef struct {
    const void *k_cache, *v_cache;
    int cache_dt;
    double k_scale, v_scale; /* 1 unless cache_dt is E4M3 or INT8 */
    int NB, S, Hkv, D;
    const double *k_head, *v_head; /* per-KV-head scales replacing k_scale / v_scale, or NULL */
} orc_cache;

/* Gather positions [0, L) of KV head h of one sequence into contiguous
 * K[L][D], V[L][D] through its block table. */
static int gather(const orc_cache *c, const int32_t *table, int L, int h,
                  double *K, double *V)
{
    for (int p = 0; p < L; ++p) {
        int off;
        int blk = orc_lookup(table, p, c->S, &off);
        if (blk < 0 || blk >= c->NB)
            return ORC_BAD_BLOCK;
        size_t base = (((size_t)blk * c->S + (size_t)off) * c->Hkv + (size_t)h) * c->D;
        double ks = c->k_head ? c->k_head[h] : c->k_scale;
        double vs = c->v_head ? c->v_head[h] : c->v_scale;
        for (int d = 0; d < c->D; ++d) {
            K[(size_t)p * c->D + d] = load_elem(c->k_cache, c->cache_dt, base + d, ks);
            V[(size_t)p * c->D + d] = load_elem(c->v_cache, c->cache_dt, base + d, vs);
        }
    }
    return ORC_OK;
}

/* softmax(scale * q . K[0:n]^T) V[0:n] for one query vector, in double:
 * first pass finds the maximum logit, second pass forms exp-weights and
 * their sum, the weighted sum of V rows is divided by that sum. */
static void attend(const double *qv, const double *K, const double *V, int n,
                   int D, double scale, double *w, double *out)
{
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (n <= 0)
        return;
    double mx = -INFINITY;
    for (int p = 0; p < n; ++p) {
        double s = 0.0;
        for (int d = 0; d < D; ++d)
            s += qv[d] * K[(size_t)p * D + d];
        w[p] = scale * s;
        if (w[p] > mx)
            mx = w[p];
    }
    double sum = 0.0;
    for (int p = 0; p < n; ++p) {
        w[p] = exp(w[p] - mx);
        sum += w[p];
    }
    for (int p = 0; p < n; ++p)
        for (int d = 0; d < D; ++d)
            out[d] += w[p] * V[(size_t)p * D + d];
    for (int d = 0; d < D; ++d)
        out[d] /= sum;
}

/* Paged decode attention, one query token per sequence.
 *   q:  [B][Hq][D] of q_dt (f32 or bf16)
 *   block_tables: [B][MB] int32; context_lens: [B] int32
 *   seqs/nseqs: which sequences to evaluate (NULL = all, in order)
 *   out: [nseqs][Hq][D] double
 * Returns ORC_BAD_BLOCK if a table entry inside a context is out of range
 * (that sequence's rows are left NaN). */
int orc_paged_attention_decode(double *out, const void *q, int q_dt,
                               const void *k_cache, const void *v_cache,
                               int cache_dt, double k_scale, double v_scale,
                               const double *k_head_scales,
                               const double *v_head_scales,
                               int NB, int S, int Hkv, int D,
                               const int32_t *block_tables, int MB,
                               const int32_t *context_lens, int B, int Hq,
                               double scale, const int32_t *seqs, int nseqs,
                               int nthreads)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || S <= 0 || B < 0)
        return ORC_BAD_ARG;
    if (seqs == NULL)
        nseqs = B;
    const int G = Hq / Hkv;
    orc_cache c = {k_cache, v_cache, cache_dt,
                   narrow_dt(cache_dt) ? k_scale : 1.0,
                   narrow_dt(cache_dt) ? v_scale : 1.0, NB, S, Hkv, D,
                   narrow_dt(cache_dt) ? k_head_scales : NULL,
                   narrow_dt(cache_dt) ? v_head_scales : NULL};
    int status = ORC_OK;
    const long nunits = (long)nseqs * Hkv;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(max : status)
#endif
    for (long u = 0; u < nunits; ++u) {
        int i = (int)(u / Hkv), h = (int)(u % Hkv);
        int s = seqs ? seqs[i] : i;
        int L = context_lens[s];
        if (L > MB * S) {
            status = status > ORC_BAD_ARG ? status : ORC_BAD_ARG;
            continue;
        }
        double *K = malloc(sizeof(double) * ((size_t)L * D + 1));
        double *V = malloc(sizeof(double) * ((size_t)L * D + 1));
        double *w = malloc(sizeof(double) * ((size_t)L + 1));
        double *qv = malloc(sizeof(double) * (size_t)D);
        if (!K || !V || !w || !qv) {
            free(K); free(V); free(w); free(qv);
            status = ORC_NO_MEMORY;
            continue;
        }
        int st = gather(&c, block_tables + (size_t)s * MB, L, h, K, V);
        for (int g = 0; g < G; ++g) {
            int hq = h * G + g;
            double *o = out + ((size_t)i * Hq + hq) * D;
            if (st != ORC_OK) {
                for (int d = 0; d < D; ++d)
                    o[d] = NAN;
                continue;
            }
            for (int d = 0; d < D; ++d)
                qv[d] = load_elem(q, q_dt, ((size_t)s * Hq + hq) * D + d, 1.0);
            attend(qv, K, V, L, D, scale, w, o);
        }
        if (st != ORC_OK && st > status)
            status = st;
        free(K); free(V); free(w); free(qv);
    }
    return status;
}

/* One chunk of a chunked prefill ([BMM] "分块预填充"): NQ query tokens of
 * one sequence, token i at position q_start + i, attend causally to the
 * sequence's paged keys; the cache already holds the earlier chunks and
 * this chunk's own K/V, so kv_len >= q_start + NQ.  Query i sees positions
 * p <= q_start + i.
 *   q: [NQ][Hq][D]; table: one sequence's block table
 *   rows/nrows: which query tokens to evaluate (NULL = all)
 *   out: [nrows][Hq][D] double */
int orc_paged_prefill_chunk(double *out, const void *q, int q_dt, int NQ,
                            int q_start, const void *k_cache,
                            const void *v_cache, int cache_dt, double k_scale,
                            double v_scale, const double *k_head_scales,
                            const double *v_head_scales, int NB, int S, int Hkv, int D,
                            const int32_t *table, int kv_len, int Hq,
                            double scale, const int32_t *rows, int nrows,
                            int nthreads)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || S <= 0 || NQ < 0 ||
        q_start < 0 || kv_len < q_start + NQ)
        return ORC_BAD_ARG;
    if (rows == NULL)
        nrows = NQ;
    const int G = Hq / Hkv;
    orc_cache c = {k_cache, v_cache, cache_dt,
                   narrow_dt(cache_dt) ? k_scale : 1.0,
                   narrow_dt(cache_dt) ? v_scale : 1.0, NB, S, Hkv, D,
                   narrow_dt(cache_dt) ? k_head_scales : NULL,
                   narrow_dt(cache_dt) ? v_head_scales : NULL};
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(max : status)
#endif
    for (int h = 0; h < Hkv; ++h) {
        double *K = malloc(sizeof(double) * ((size_t)kv_len * D + 1));
        double *V = malloc(sizeof(double) * ((size_t)kv_len * D + 1));
        double *w = malloc(sizeof(double) * ((size_t)kv_len + 1));
        double *qv = malloc(sizeof(double) * (size_t)D);
        if (!K || !V || !w || !qv) {
            free(K); free(V); free(w); free(qv);
            status = ORC_NO_MEMORY;
            continue;
        }
        int st = gather(&c, table, kv_len, h, K, V);
        for (int r = 0; r < nrows; ++r) {
            int i = rows ? rows[r] : r;
            int visible = q_start + i + 1;
            for (int g = 0; g < G; ++g) {
                int hq = h * G + g;
                double *o = out + ((size_t)r * Hq + hq) * D;
                if (st != ORC_OK) {
                    for (int d = 0; d < D; ++d)
                        o[d] = NAN;
                    continue;
                }
                for (int d = 0; d < D; ++d)
                    qv[d] = load_elem(q, q_dt, ((size_t)i * Hq + hq) * D + d, 1.0);
                attend(qv, K, V, visible, D, scale, w, o);
            }
        }
        if (st != ORC_OK && st > status)
            status = st;
        free(K); free(V); free(w); free(qv);
    }
    return status;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
