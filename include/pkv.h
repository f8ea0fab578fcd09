/*
 * pkv.h -- C ABI of the paged KV-cache library (GB300 / sm_103a).
 *
 * One shared library, libpkv.so, with hand-written CUDA kernels for the
 * decode step of a paged KV cache.  Every entry point:
 *   - takes plain pointers and sizes (no framework types);
 *   - expects DEVICE pointers for every tensor argument unless stated,
 *     owned by the caller; the library never allocates, frees or
 *     synchronises device memory;
 *   - enqueues its work on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns after enqueueing;
 *   - validates shapes, dtypes and alignment on the host before launching
 *     and returns a status code; a failed check launches nothing;
 *   - reports data-dependent range errors found on the device (bad block
 *     ids, slots beyond the pool, bad lengths, a timed-out wait) by OR-ing
 *     PKV_DEVERR_* bits into `*device_error` (device memory, nullable), and
 *     skips the offending item.  It never traps.
 *
 * Layouts (row-major, innermost last):
 *   K / V cache, per layer:  [num_blocks][block_size][num_kv_heads][head_dim]
 *     -- the per-block layout [block_size, n_kv_heads, head_dim] of the
 *        KVBlock definition in "大模型推理的KV Cache优化全解" (block structure
 *        section), one layer at a time, K and V in separate tensors.
 *   block_tables: int32 [num_seqs][max_blocks_per_seq]; entry j of row s is
 *     the physical block holding tokens [j*S, (j+1)*S) of sequence s
 *     ("3.3 批处理与内存管理", section "PagedAttention：块表", equation:
 *     physical block = table[p / S], offset = p % S).  Entries past a
 *     sequence's last block are never read.
 *   context_lens: int32 [num_seqs]; tokens in each sequence, INCLUDING the
 *     token written by this step's reshape_and_cache.
 *   slot_mapping: int64 [num_tokens]; slot = block * S + offset; a negative
 *     slot marks a padding token that is skipped.
 *   q / out (decode): [num_seqs][num_q_heads][head_dim].
 *   GQA: query head hq reads KV head hq / G, G = num_q_heads / num_kv_heads.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 2

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shapes */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not built: dtype combo, head_dim, block_size, G */
    PKV_ERR_OUT_OF_RANGE = 3,  /* a host-checkable index or size beyond its limit */
    PKV_ERR_WORKSPACE = 4,     /* workspace missing, too small or misaligned */
    PKV_ERR_CUDA = 5           /* a CUDA runtime call or launch failed */
} pkv_status;

typedef enum {
    PKV_F32 = 0,
    PKV_BF16 = 1,
    PKV_FP8_E4M3 = 2,  /* OCP E4M3 (bias 7, max 448, no inf), per-tensor scale */
    PKV_INT8 = 3       /* symmetric int8 in [-127, 127], per-tensor scale */
} pkv_dtype;

/* Bits OR-ed into *device_error by the kernels. */
#define PKV_DEVERR_BAD_SLOT 0x1     /* slot >= num_blocks * block_size */
#define PKV_DEVERR_BAD_BLOCK 0x2    /* block id < 0 or >= num_blocks where one must be read */
#define PKV_DEVERR_BAD_LENGTH 0x4   /* context_len < 0 or > max_blocks_per_seq * block_size */
#define PKV_DEVERR_TIMEOUT 0x8      /* a bounded wait on an async copy gave up */
#define PKV_DEVERR_Q_RANGE 0x10     /* a query value the tensor-core operands cannot carry: beyond the f16 range
                                       (|q| >= 65520) in a decode over an FP8 or INT8 cache or a prefill over an
                                       INT8 cache (f16 operands); non-finite in a prefill over an FP8 cache */

/* Description of one layer's K and V cache pools. */
typedef struct {
    int32_t num_blocks;    /* physical blocks in the pool (NB) */
    int32_t block_size;    /* tokens per block (S): 4, 8, 16 or 32 */
    int32_t num_kv_heads;  /* Hkv */
    int32_t head_dim;      /* D: 64 or 128 */
    int32_t dtype;         /* pkv_dtype of the cache elements */
    float k_scale;         /* FP8 / INT8: stored code * k_scale is the key value; 1 otherwise */
    float v_scale;         /* FP8 / INT8: same for values */
    /* FP8 / INT8, optional: device arrays of num_kv_heads fp32 scales, one per KV head (the
     * finer granularity of the KV-quantisation discussion in "从 PagedAttention 到 Chunked
     * Prefill" §5.4 and the KV-cache optimisation overview's technique table).  When set,
     * KV head h uses k_head_scales[h] / v_head_scales[h] in place of k_scale / v_scale, in
     * the cache write and in every read.  NULL: the per-tensor scale.  Values must be finite
     * and positive (device data, not checked: other values give non-finite outputs). */
    const float* k_head_scales;
    const float* v_head_scales;
} pkv_cache_desc;

/*
 * Cache write ("reshape_and_cache").
 * Each step computes the new token's k_t, v_t and appends them to the cache
 * ("大模型推理的KV Cache优化全解", §1.1; "3.3 批处理与内存管理", section
 * "代码", append_token).  For token i with slot_mapping[i] >= 0:
 *   k_cache[slot / S][slot % S][h][:] = convert(k_new[i][h][:])   (same for v)
 * convert: same dtype -> bit copy; bf16 -> f32 exact; f32 -> bf16 round to
 * nearest even; -> FP8 E4M3: sat(RNE(x / scale)) with an fp32 division;
 * -> INT8: clamp(RNE(x / scale), -127, 127) with an fp32 division (the INT8
 * KV quantisation of "从 PagedAttention 到 Chunked Prefill" §5.4 and the
 * "INT8量化" row of "大模型推理的KV Cache优化全解", per-tensor scale).
 *   k_new, v_new: [num_tokens][num_kv_heads][head_dim] of src_dtype (f32 or bf16).
 * Tokens whose slot is beyond the pool set PKV_DEVERR_BAD_SLOT and are skipped.
 * Two tokens with the same slot race (one of them wins).
 * Alignment: k_new, v_new, k_cache, v_cache 16-byte aligned.
 */
pkv_status pkv_reshape_and_cache(const void* k_new, const void* v_new, int32_t src_dtype,
                                 const int64_t* slot_mapping, int32_t num_tokens,
                                 void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                 int32_t* device_error, void* stream);

/*
 * Bytes of device workspace pkv_paged_attention_decode needs for these
 * sizes on the CURRENT device (0 when num_splits == 1).  The workspace holds
 * the split-KV partial results (m, l, O) and one completion counter per
 * (sequence, KV head); the decode call clears the counters itself.
 */
pkv_status pkv_paged_attention_workspace_size(const pkv_cache_desc* cache, int32_t num_seqs,
                                              int32_t num_q_heads, int32_t num_splits,
                                              size_t* bytes);

/*
 * Paged decode attention over a ragged batch (one query token per sequence).
 * For every sequence s and query head hq (KV head h = hq / G):
 *   out[s][hq] = softmax(scale * q[s][hq] . K_s^T) V_s
 * where K_s / V_s are positions [0, context_lens[s]) gathered through the
 * block table ("3.3 批处理与内存管理", "PagedAttention：块表"), evaluated
 * block by block with the online-softmax recurrence of "从 PagedAttention 到
 * Chunked Prefill" §2.2 (running max m, running sum l, unnormalised O,
 * rescaled by exp(m_old - m_new) when the max grows; out = O / l).
 * A sequence with context length 0 gets an all-zero row.
 *
 * Split-KV: the work of all (sequence, KV head) pairs is laid end to end
 * block by block and cut into equal shares, one per worker warp, so that
 * long and short sequences load the GPU evenly; a pair cut across workers
 * produces partial (m, l, O) triples that the last finishing worker merges
 * (M = max m_p, l = sum e^(m_p - M) l_p, O = sum e^(m_p - M) O_p / l).
 *   num_splits == 0 : cut anywhere on block boundaries (balanced; default)
 *   num_splits == 1 : never cut a pair (single pass; workspace unused)
 *   num_splits == P : cut only on boundaries of partitions of
 *                     ceil(ceil(max_context_len / S) / P) blocks
 * Any choice gives the same result up to fp32 rounding order.
 *
 * Arithmetic: fp32 accumulation throughout.  FP8 / INT8 caches with 128-dim
 * heads, and bf16 caches of 128-dim heads in groups of G = 8, run q.K and P.V
 * on the tensor cores: cached codes and bf16 values enter exactly, q is taken
 * to f16 for one-byte caches (|q| >= 65520 sets PKV_DEVERR_Q_RANGE) and the
 * probabilities are rounded to f16 (bf16 for a bf16 cache) before P.V.  The
 * other cases compute on fp32 values throughout.
 *
 *   q:   [num_seqs][num_q_heads][head_dim], q_dtype f32 (with an f32 cache)
 *        or bf16 (with a bf16, FP8 or INT8 cache); out has q's dtype and shape.
 *   max_context_len: an upper bound of context_lens (0 = use
 *        max_blocks_per_seq * block_size); only shapes the partitions.
 *   workspace: >= pkv_paged_attention_workspace_size bytes, 16-byte
 *        aligned (may be NULL when num_splits == 1).  Concurrent calls must
 *        not share a workspace.
 * Supported: head_dim 64/128, block_size 4/8/16/32, G in {1, 2, 4, 8},
 *   num_seqs <= 8192.  Pointers q, out and the caches 16-byte aligned.
 */
pkv_status pkv_paged_attention_decode(void* out, const void* q, int32_t q_dtype,
                                      const void* k_cache, const void* v_cache,
                                      const pkv_cache_desc* cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, float scale, int32_t num_splits,
                                      int32_t max_context_len, void* workspace,
                                      size_t workspace_bytes, int32_t* device_error,
                                      void* stream);

/*
 * Paged decode attention over a batch whose sequences share physical blocks:
 * forked samples or beams, or sequences with a common prompt prefix, whose
 * tables name the same blocks ("3.3 批处理与内存管理", section "共享与写时复制":
 * blocks with a reference count above one).  Same arguments, result,
 * workspace and errors as pkv_paged_attention_decode (the size returned by
 * pkv_paged_attention_workspace_size is enough for this call).  A caller whose
 * block manager knows that the batch shares blocks calls this form.
 *
 * Every sequence still reads each of its blocks through its own table.  A
 * shared block is fetched from DRAM once and re-read from L2 by the other
 * sequences that hold it, so the K/V arrive faster than HBM delivers them and
 * the instruction cost per byte becomes the bound.  For bf16 caches of 128-dim
 * heads this form therefore runs the tensor-core kernel (one KV head per work
 * unit) at every GQA group, where pkv_paged_attention_decode keeps groups
 * below 8 on the CUDA cores, which stream DRAM-resident blocks slightly
 * faster.  For every other cache it is identical to pkv_paged_attention_decode.
 */
pkv_status pkv_paged_attention_decode_shared(void* out, const void* q, int32_t q_dtype,
                                             const void* k_cache, const void* v_cache,
                                             const pkv_cache_desc* cache,
                                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                                             const int32_t* context_lens, int32_t num_seqs,
                                             int32_t num_q_heads, float scale, int32_t num_splits,
                                             int32_t max_context_len, void* workspace,
                                             size_t workspace_bytes, int32_t* device_error,
                                             void* stream);

/*
 * One chunk of a chunked prefill ("3.3 批处理与内存管理", section "分块预填充":
 * the chunk's queries attend to a KV cache that already holds the earlier
 * chunks).  The chunk's own K/V must already be written (pkv_reshape_and_cache),
 * so kv_len >= q_start_pos + num_q_tokens.  Query token i (position
 * q_start_pos + i) and query head hq (KV head hq / G) attend causally:
 *   out[i][hq] = softmax(scale * q[i][hq] . K[0 .. q_start_pos + i]^T) V[0 .. q_start_pos + i]
 * with K/V gathered through block_table (one sequence, ceil(kv_len / S)
 * entries).  Runs on the tensor cores with fp32 accumulation:
 *   - bf16 cache: bf16 inputs, the softmax weights rounded to bf16 for P.V.
 *   - FP8 cache: 8-bit (E4M3) products on the cached codes as they are.  Each
 *     query row is scaled by a power of two (its largest magnitude to
 *     [128, 256)) and split into two E4M3 parts, hi + lo, which carry it
 *     exactly for elements within 2^-10 of the row's largest and to 2^-18 of
 *     that largest below; the softmax weights are split the same way (about
 *     8 significant bits, like bf16).  A non-finite query value sets
 *     PKV_DEVERR_Q_RANGE.
 *   - INT8 cache: the codes are widened to f16 on chip (exactly), the queries
 *     are taken to f16 (exact for |q| in [2^-14, 65504]; a value of 65520 or
 *     more sets PKV_DEVERR_Q_RANGE), the softmax weights rounded to f16.
 *   The per-tensor or per-head scales are applied to the scores and the output.
 *   q, out: [num_q_tokens][num_q_heads][128] bf16.
 * scale must be positive.
 * Supported (narrower than the decode call): bf16 queries, bf16, FP8 or INT8
 *   cache, head_dim 128 only, block_size 8/16/32 only (a 64-key tile is copied
 *   as whole blocks), G = num_q_heads / num_kv_heads dividing 128; other shapes
 *   return PKV_ERR_UNSUPPORTED.  No workspace.
 */
pkv_status pkv_paged_prefill_chunk(void* out, const void* q, int32_t q_dtype, int32_t num_q_tokens,
                                   int32_t q_start_pos, const void* k_cache, const void* v_cache,
                                   const pkv_cache_desc* cache, const int32_t* block_table, int32_t kv_len,
                                   int32_t num_q_heads, float scale, int32_t* device_error, void* stream);

/*
 * Several prefill chunks of different sequences in one launch (varlen form of
 * the chunked prefill in "3.3 批处理与内存管理", section "分块预填充", and of the
 * mixed batches of "从 PagedAttention 到 Chunked Prefill" §3.2, where prefill
 * chunks and decode tokens of different sequences share one step).  Chunk s owns query tokens [cu_q[s], cu_q[s+1]) of q/out; its token
 * i sits at position q_starts[s] + i of sequence s, whose first kv_lens[s]
 * keys are cached (the chunk's own keys included, so
 * kv_lens[s] >= q_starts[s] + cu_q[s+1] - cu_q[s]).  Each chunk computes
 * exactly what pkv_paged_prefill_chunk computes for it, with block table row
 * s of block_tables ([num_seqs][max_blocks_per_seq]).  A decode token is a
 * chunk of one query token.
 *   q, out: [total_q_tokens][num_q_heads][128] bf16; rows not covered by any
 *        chunk are not written.
 *   cu_q: [num_seqs + 1] device int32, non-decreasing, cu_q[num_seqs] <= total_q_tokens.
 *   q_starts, kv_lens: [num_seqs] device int32.
 * These arrays are read on the device: a violation (cu_q not monotone or past
 * total_q_tokens, kv_len too short, more table entries than max_blocks_per_seq)
 * sets PKV_DEVERR_BAD_LENGTH and leaves that chunk's rows unwritten; a table
 * entry outside the pool sets PKV_DEVERR_BAD_BLOCK.
 * The arithmetic per cache type is that of pkv_paged_prefill_chunk.
 * scale must be positive.
 * Supported (narrower than the decode call): bf16 queries, bf16, FP8 or INT8
 *   cache, head_dim 128 only, block_size 8/16/32 only, G dividing 128,
 *   num_seqs <= 2048; other shapes return PKV_ERR_UNSUPPORTED.  No workspace.
 */
pkv_status pkv_paged_prefill_varlen(void* out, const void* q, int32_t q_dtype, int32_t total_q_tokens,
                                    const int32_t* cu_q, const int32_t* q_starts, const int32_t* kv_lens,
                                    const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    int32_t num_seqs, int32_t num_q_heads, float scale,
                                    int32_t* device_error, void* stream);

/*
 * One launch for a mixed serving step: the decode tokens and the prefill chunks
 * of a step, of different sequences ("从 PagedAttention 到 Chunked Prefill"
 * §3.2: chunked prefill and decode share one batch; "3.3 批处理与内存管理",
 * section "分块预填充").  The chunks are described as for
 * pkv_paged_prefill_varlen (cu_q, q_starts, kv_lens, block_tables rows); the
 * first num_decode chunks are decode tokens: one query each (cu_q[s] = s for
 * s <= num_decode) at position kv_lens[s] - 1, computing what
 * pkv_paged_attention_decode computes for it (a violation sets
 * PKV_DEVERR_BAD_LENGTH).  The remaining chunks compute what
 * pkv_paged_prefill_chunk computes for them.
 *
 * One CTA per SM: each first runs its share of the prefill tiles, then works
 * through the decode tokens' K/V with the tensor-core decode (split-KV with
 * merges, one KV head per work unit); the decode stream is cut so that CTAs
 * that spent time on prefill tiles take less of it.
 *   workspace: >= pkv_paged_attention_mixed_workspace_size bytes (0 without
 *   decode tokens), 16-byte aligned; concurrent calls must not share it.
 * Per-tensor or per-head scales apply as in the decode and prefill calls.
 * Supported: bf16 queries, bf16, FP8 or INT8 cache, head_dim 128,
 *   block_size 16, G in {1, 2, 4, 8}, num_seqs <= 2048, num_decode <= 8192,
 *   devices of at most 256 SMs; other cases return PKV_ERR_UNSUPPORTED.
 */
pkv_status pkv_paged_attention_mixed(void* out, const void* q, int32_t q_dtype, int32_t total_q_tokens,
                                     const int32_t* cu_q, const int32_t* q_starts, const int32_t* kv_lens,
                                     const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                                     int32_t num_decode, int32_t num_q_heads, float scale, void* workspace,
                                     size_t workspace_bytes, int32_t* device_error, void* stream);

/* Bytes of device workspace pkv_paged_attention_mixed needs (on the current device). */
pkv_status pkv_paged_attention_mixed_workspace_size(const pkv_cache_desc* cache, int32_t num_decode,
                                                    int32_t num_q_heads, size_t* bytes);

/*
 * Copy whole physical blocks, for copy-on-write of shared blocks
 * ("3.3 批处理与内存管理", section "共享与写时复制": before a sequence writes
 * into a block whose reference count is above one, the engine copies the
 * block and points the sequence's table at the copy).  For each pair i:
 *   k_cache[dst_i] = k_cache[src_i];  v_cache[dst_i] = v_cache[src_i]
 * (all block_size slots, bit-exact).
 *   block_mapping: int64 [num_pairs][2] = (src, dst), device memory.
 * A dst may not appear as a src in the same call (the copies run
 * concurrently); ids outside [0, num_blocks) set PKV_DEVERR_BAD_BLOCK and
 * that pair is skipped.  num_pairs < 2^30 (PKV_ERR_OUT_OF_RANGE otherwise).
 */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                           const int64_t* block_mapping, int32_t num_pairs,
                           int32_t* device_error, void* stream);

/*
 * Paged decode attention for callers that cannot allocate device memory.
 * The paper has no counterpart: this is an interface convenience.
 *
 * pkv_paged_attention_decode needs a caller-provided workspace whenever it
 * splits the work (num_splits != 1).  Some callers cannot provide one: code
 * that may not call cudaMalloc once its memory plan is fixed, hosts that
 * own every device allocation and expose no allocator to plugins, or
 * language runtimes that reach this library only through plain C.  This
 * entry point computes the same result as pkv_paged_attention_decode
 * (same arguments minus the workspace) but keeps the split-KV scratch in a
 * static device array of PKV_STATIC_SCRATCH_BYTES that the library owns.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *     library routine.  The array occupies PKV_STATIC_SCRATCH_BYTES on every
 *     GPU that loads the library, until the process exits.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first
 *     call before any stream capture.  The address is kept for the life of
 *     the process: after cudaDeviceReset (or any teardown of the device's
 *     primary context) it is stale, so this entry point must not be called
 *     again in that process.
 *   - A batch whose scratch need (pkv_paged_attention_workspace_size) is
 *     above PKV_STATIC_SCRATCH_BYTES is rejected with PKV_ERR_WORKSPACE
 *     before anything is launched; num_splits == 1 needs no scratch.
 *   - Every call shares the one array.  Each call clears the completion
 *     counters it needs; the partial records keep the last call's contents.
 *     Calls whose work overlaps on the GPU (different streams or host
 *     threads without ordering between them) race on the array and give
 *     wrong results: serialise them.
 */
#define PKV_STATIC_SCRATCH_BYTES (12u * 1024u * 1024u)
pkv_status pkv_paged_attention_decode_static_scratch(
    void* out, const void* q, int32_t q_dtype, const void* k_cache, const void* v_cache,
    const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, float scale,
    int32_t num_splits, int32_t max_context_len, int32_t* device_error, void* stream);

/*
 * Swap whole blocks between two pools, for preemption by swapping ("从
 * PagedAttention 到 Chunked Prefill" §3.1 and "3.3 批处理与内存管理",
 * scheduling section: a preempted sequence's KV blocks move to CPU memory
 * and come back when it is resumed).  For each pair i:
 *   dst_k[dst_i] = src_k[src_i];  dst_v[dst_i] = src_v[src_i]   (whole blocks, bit-exact)
 * Either pool may be device memory or host memory the device can reach
 * (cudaHostAlloc / cudaHostRegister memory; any host memory on devices with
 * pageable-memory access, such as Grace-attached GPUs); the copies run in one
 * kernel over NVLink-C2C / PCIe.  `cache` gives the block geometry and dtype
 * (its num_blocks is not used); src_num_blocks / dst_num_blocks bound the ids.
 *   block_mapping: int64 [num_pairs][2] = (src, dst), device-accessible memory.
 * Destination blocks must be distinct; out-of-range ids set
 * PKV_DEVERR_BAD_BLOCK and that pair is skipped.  Pointers that the device
 * cannot dereference are rejected with PKV_ERR_INVALID_ARG.  num_pairs < 2^30
 * (PKV_ERR_OUT_OF_RANGE otherwise).
 */
pkv_status pkv_swap_blocks(const void* src_k, const void* src_v, int32_t src_num_blocks, void* dst_k,
                           void* dst_v, int32_t dst_num_blocks, const pkv_cache_desc* cache,
                           const int64_t* block_mapping, int32_t num_pairs, int32_t* device_error,
                           void* stream);

/*
 * Content hashes of full blocks, for hash-based prefix caching ("3.3
 * 批处理与内存管理", section "前缀缓存与 RadixAttention": each full block is
 * identified by its tokens together with the hash of all blocks before it; a
 * new request reuses every leading block whose hash is cached).  The pages
 * name no hash function; this one is FNV-1a, 64-bit, over little-endian bytes:
 *   d_j = FNV-1a(token ids of block j, 4 bytes each)
 *   h_j = FNV-1a(h_{j-1} as 8 bytes (0 before the first block) ++ d_j as 8 bytes)
 * Sequence s has tokens token_ids[cu_tokens[s] .. cu_tokens[s+1]) and
 * floor(L_s / block_size) full blocks; a partial last block has no hash.
 * Hash j of sequence s goes to hashes[out_offsets[s] + j] (out_offsets is
 * normally the exclusive prefix sum of the full-block counts).  Sequences
 * whose hashes would fall outside [0, hashes_capacity) set
 * PKV_DEVERR_BAD_SLOT and are skipped; a negative length sets
 * PKV_DEVERR_BAD_LENGTH.  All pointers are device memory.
 */
pkv_status pkv_block_hashes(const int32_t* token_ids, const int64_t* cu_tokens, int32_t num_seqs,
                            int32_t block_size, const int64_t* out_offsets, uint64_t* hashes,
                            int64_t hashes_capacity, int32_t* device_error, void* stream);

/* Human-readable name of a status code (static storage). */
const char* pkv_status_string(pkv_status status);

/* Details of the last failed call on the calling host thread ("" if none). */
const char* pkv_last_error(void);

/* PKV_ABI_VERSION of the loaded library. */
int32_t pkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
