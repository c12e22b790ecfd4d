/*
 * attn.h -- C ABI of libattn.so: exact scaled-dot-product attention on B300
 * (sm_103a), computed tile by tile with an online softmax so that the T x S
 * score matrix never reaches device memory.
 *
 *   O = softmax(Q K^T * scale + mask) V
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - All tensor arguments are DEVICE pointers to contiguous row-major arrays
 *    that the caller allocates, owns and frees (attn_fwd_host alone takes
 *    host arrays).  The library keeps no per-call state and allocates no
 *    device memory on these paths.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  A non-zero return means nothing was launched, except
 *    ATTN_ERR_CUDA, which reports a launch error seen right after launching.
 *  - Element types: ATTN_BF16 or ATTN_F16 inputs/outputs (the output has
 *    the input type) with float32 softmax and accumulation, or ATTN_F32 end
 *    to end (no TF32).  LSE is always float32.
 *  - Layouts ("Implementing attention from scratch", Core ideas, Shapes first):
 *      q, o     [B, Hq, T, D]
 *      k, v     [B, Hkv, S, D]
 *      lse      [B, Hq, T]
 *    Grouped-query attention ("Self-Attention: Implementation, Complexity,
 *    and Efficient Variants", follow-up on MQA/GQA; "Implementing attention
 *    from scratch", KV caching): Hq must be a multiple of Hkv, and query head
 *    h reads KV head h / (Hq / Hkv) (contiguous groups).
 *  - Masks ("Implementing attention from scratch", Masks and KV caching;
 *    "Building a causal self-attention block from scratch in PyTorch",
 *    Step 2): query row i sits at key position p_i = i + S - T (bottom-right
 *    alignment).  With L = key_lens[b] (S when key_lens is NULL):
 *        row i is a padded row       iff p_i >= L
 *        key j is visible to row i   iff j < L and (!causal or j <= p_i)
 *    A padded row, or a row that sees no key, is defined as O = 0 and
 *    LSE = -inf (the pages note a fully masked softmax row is NaN and must
 *    be handled explicitly).
 *  - LSE[i] = ln(sum over visible j of exp(scale * q_i . k_j)).
 */
#ifndef ATTN_B300_ATTN_H_
#define ATTN_B300_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA
 * include. */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, ...     */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request the library does not implement */
  ATTN_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned  */
  ATTN_ERR_CUDA = 4         /* CUDA runtime/driver error at or before launch */
} attn_status;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1, ATTN_F16 = 2 } attn_dtype;

/*
 * attn_fwd -- prefill forward: O and (optionally) the per-row LSE.
 *
 * Computes the masked attention described above for every (b, h, i)
 * ("Implementing attention from scratch", Core ideas: Shapes first, Masks,
 * Stable softmax; "FlashAttention", Transformers in Action section 9.4.1,
 * Figure 9.8: Q and K/V tiles stream through on-chip memory, partial results
 * are rescaled as the running row maximum grows, and the n x m score matrix
 * is never materialised).
 *
 *   q        [B,Hq,T,D]  dtype          (read)
 *   k, v     [B,Hkv,S,D] dtype          (read)
 *   o        [B,Hq,T,D]  dtype          (written; padded rows written as 0)
 *   lse      [B,Hq,T]    float32        (written; NULL = do not emit)
 *   key_lens [B]         int32, device  (read; NULL = every key valid;
 *                                        each value must lie in [0, S] --
 *                                        values are read on the device and
 *                                        clamped to [0, S])
 *   causal   0 or 1
 *   scale    > 0, finite (typically 1/sqrt(D))
 *
 * Supported: B, Hq, Hkv, T, S >= 1, Hq % Hkv == 0.
 *   ATTN_BF16, ATTN_F16: D in {64, 128}; q, k, v, o 16-byte aligned.
 *              Tensor-core path (tcgen05 MMAs with TMEM accumulators, TMA
 *              tile loads); P is rounded to the input type for P V.
 *   ATTN_F32:  1 <= D <= 256; 4-byte aligned.  Exact float32 path on the
 *              CUDA cores (FFMA, accurate expf), no TF32.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or
 * ATTN_ERR_CUDA.
 */
ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int Hq, int Hkv, int T, int S, int D, int dtype,
             int causal, const int32_t* key_lens, float scale,
             attn_stream_t stream);

/*
 * attn_fwd_host_workspace_size -- bytes of device memory attn_fwd_host needs
 * for these sizes: device copies of q, k, v, o, lse and key_lens, each at a
 * 256-byte aligned offset.  Returns 0 for invalid or unsupported sizes.
 */
ATTN_API size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int T, int S, int D,
                                             int dtype);

/*
 * attn_fwd_host -- attn_fwd on HOST buffers: copies q, k, v (and key_lens)
 * to the device, computes exactly what attn_fwd computes (same kernels,
 * bit-identical results), and copies o (and lse) back.  The computation is
 * the one attn_fwd cites; the pages have no counterpart for the copies,
 * which exist because a caller's tensors may live in host memory.
 *
 * The work is cut into stages along (sequence, KV head group) -- whole
 * sequences, or KV heads of one sequence, about 32 MiB of inputs each --
 * and pipelined over three streams: stage c's inputs are copied in on
 * copy_in while stage c-1 computes on `stream` and stage c-2's results are
 * copied out on copy_out, so a large call costs about its host-to-device
 * copy time rather than the sum of copies and compute.  Every operation is
 * ordered after the work already enqueued on `stream`, and work enqueued on
 * `stream` after this call is ordered after the last copy out (events; the
 * call is capturable in a CUDA graph).
 *
 *   q                 [B,Hq,T,D]   dtype, HOST     (read)
 *   k, v              [B,Hkv,S,D]  dtype, HOST     (read)
 *   o                 [B,Hq,T,D]   dtype, HOST     (written)
 *   lse               [B,Hq,T]     float32, HOST   (written; NULL = do not emit)
 *   key_lens          [B]          int32, HOST     (NULL = every key valid;
 *                                                   clamped to [0, S] as in
 *                                                   attn_fwd)
 *   workspace         device, >= attn_fwd_host_workspace_size(...) bytes,
 *                     16-byte aligned; owned by the caller, its contents on
 *                     entry do not matter; the device copies of the inputs
 *                     and results stay in it after the call
 *   stream            runs the kernels (and every copy when copy_in /
 *                     copy_out are NULL)
 *   copy_in, copy_out streams for the host-to-device and device-to-host
 *                     copies (NULL = `stream`, no overlap for that role)
 *
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister):
 * copies from or to pageable memory are correct but staged by the driver
 * and do not overlap.  All host buffers must stay valid, and the inputs
 * unmodified, until `stream` has completed the call's work.  Sizes, types
 * and masks as for attn_fwd.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG,
 * ATTN_ERR_UNSUPPORTED or ATTN_ERR_WORKSPACE with nothing enqueued, or
 * ATTN_ERR_CUDA if a copy, event or launch failed (part of the work may then
 * have been enqueued).
 */
ATTN_API int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int T, int S, int D, int dtype, int causal,
                           const int32_t* key_lens, float scale, void* workspace,
                           size_t ws_bytes, attn_stream_t stream, attn_stream_t copy_in,
                           attn_stream_t copy_out);

/*
 * attn_fwd_fp8 -- attn_fwd on FP8 E4M3 inputs ("Self-Attention:
 * Implementation, Complexity, and Efficient Variants", FlashAttention-3: FP8
 * support).  The attention of the dequantised inputs
 *     q = q_descale * Q8,  k = k_descale * K8,  v = v_descale * V8
 * with the masks, scale, GQA mapping and outputs of attn_fwd.  Scores are
 * exact products of the E4M3 values accumulated in fp32 (tcgen05
 * kind::f8f6f4); the softmax weights are rounded to E4M3 for P V (formed
 * as 2^7 times the weights relative to a running reference, so every weight
 * down to 2^-13 of the row's largest keeps E4M3's 3-bit mantissa); the
 * row sums and the LSE use the unrounded fp32 weights.
 *
 *   q                 [B,Hq,T,128]   E4M3 bytes     (read)
 *   k, v              [B,Hkv,S,128]  E4M3 bytes     (read)
 *   o                 [B,Hq,T,128]   bf16           (written)
 *   lse               [B,Hq,T]       float32        (written; NULL = do not emit)
 *   key_lens          [B]            int32, device  (NULL = all S keys valid)
 *   q_descale, k_descale, v_descale: finite, > 0
 *
 * Supported: D = 128 (else ATTN_ERR_UNSUPPORTED); q, k, v, o 16-byte
 * aligned.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or
 * ATTN_ERR_CUDA.
 */
ATTN_API int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int T, int S, int D, int causal,
                          const int32_t* key_lens, float scale, float q_descale,
                          float k_descale, float v_descale, attn_stream_t stream);

/*
 * attn_fwd_chunked -- chunked prefill against a KV cache: a chunk of up to T
 * new queries per sequence attends over that sequence's cache, which already
 * holds the chunk's own K/V rows (append them first, e.g. with one copy per
 * chunk).  "Implementing attention from scratch", KV caching: a new query's
 * position is the cache length plus its position within the chunk, and the
 * causal mask is aligned to that position (bottom-right, per sequence).
 *
 * Query row i of sequence b sits at key position p = q_pos[b] + i.  With
 * L = kv_lens[b] (clamped to [0, S_max]):
 *     key j is visible to row i   iff  j < L and (!causal or j <= p)
 *     row i is a padded row       iff  p >= L
 * A chunk shorter than T for sequence b (ragged chunks) is expressed by
 * kv_lens[b] = q_pos[b] + (its chunk length): rows past it are padded rows.
 * Padded rows and rows that see no key are written as O = 0, LSE = -inf.
 * attn_fwd is the special case q_pos[b] = S - T.  Cache rows at or past L
 * are never used, whatever they hold.
 *
 *   q                 [B,Hq,T,D]      dtype          (read)
 *   kcache, vcache    [B,Hkv,S_max,D] dtype          (read)
 *   o                 [B,Hq,T,D]      dtype          (written)
 *   lse               [B,Hq,T]        float32        (written; NULL = do not emit)
 *   q_pos             [B]             int32, device  (read; any value)
 *   kv_lens           [B]             int32, device  (read; clamped to [0, S_max])
 *
 * Supported sizes, types and alignment as for attn_fwd (S_max in place of
 * S).  q_pos and kv_lens must not be NULL.  Returns ATTN_OK,
 * ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
ATTN_API int attn_fwd_chunked(const void* q, const void* kcache, const void* vcache, void* o,
                              float* lse, const int32_t* q_pos, const int32_t* kv_lens,
                              int B, int Hq, int Hkv, int T, int S_max, int D, int dtype,
                              int causal, float scale, attn_stream_t stream);

/*
 * attn_fwd_kv_shard -- the prefill over one shard of the keys: the part of
 * sequence parallelism that runs on one GPU ("Building a causal
 * self-attention block from scratch in PyTorch", Extending It: distributed
 * attention, sharding Q/K/V across devices and recombining).  The keys of
 * each sequence are split into shards; this call computes, for the given
 * queries, the attention over the keys of one shard only, normalised over
 * that shard, with the shard's LSE.  attn_lse_merge then combines the
 * partials of all shards into the attention over every key.
 *
 * Positions are the sequence's own (global) key positions.  The shard holds
 * keys k_off .. k_off + S - 1; query row i of sequence b sits at position
 * p = q_pos[b] + i; L = key_lens[b] is the sequence's valid length:
 *     key k_off + j is visible to row i  iff  k_off + j < L and
 *                                              (!causal or k_off + j <= p)
 *     row i is a padded row               iff  p >= L
 * (bottom-right alignment: q_pos[b] = L - T for a sequence whose last query
 * is its last key).  Padded rows, and rows that see no key of this shard,
 * are written as O = 0, LSE = -inf; attn_lse_merge gives such a partial no
 * weight.  Shard key rows at or past L - k_off are never used.
 *
 *   q                 [B,Hq,T,D]   dtype          (read)
 *   k, v              [B,Hkv,S,D]  dtype          (read: the shard's keys)
 *   o                 [B,Hq,T,D]   dtype          (written)
 *   lse               [B,Hq,T]     float32        (written; NULL = do not emit,
 *                                                  but the merge needs it)
 *   q_pos, key_lens   [B]          int32, device  (read; global positions, any
 *                                                  value; not NULL)
 *   k_off             >= 0: global position of the shard's key row 0
 *
 * Supported sizes, types and alignment as for attn_fwd.  With k_off = 0, a
 * single shard holding every key and key_lens in [0, S], this is
 * attn_fwd_chunked.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG,
 * ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
ATTN_API int attn_fwd_kv_shard(const void* q, const void* k, const void* v, void* o, float* lse,
                               const int32_t* q_pos, const int32_t* key_lens, int k_off, int B,
                               int Hq, int Hkv, int T, int S, int D, int dtype, int causal,
                               float scale, attn_stream_t stream);

/*
 * attn_lse_merge -- combines n_parts partial results of the same queries
 * over disjoint key sets (e.g. one per key shard, from attn_fwd_kv_shard)
 * into the attention over all those keys, by the rescaling of the online
 * softmax ("Implementing attention from scratch", Core ideas, Stable
 * softmax: sums kept against a running maximum are rescaled by
 * exp(m_old - m_new)):
 *     LSE = ln sum_n exp(LSE_n),   O = sum_n exp(LSE_n - LSE) O_n
 * Partials with LSE_n = -inf add nothing; a row with no partial is written as
 * O = 0, LSE = -inf.  Per row: the maximum M of the partials' LSE, then
 * the sum over n = 0 .. n_parts - 1 in order with weights exp(LSE_n - M)
 * (float32 arithmetic, output rounded once).
 *
 *   o_parts    [n_parts,B,Hq,T,D]  dtype    (read)
 *   lse_parts  [n_parts,B,Hq,T]    float32  (read)
 *   o          [B,Hq,T,D]          dtype    (written; may not alias o_parts)
 *   lse        [B,Hq,T]            float32  (written; NULL = do not emit)
 *
 * Supported: dtype ATTN_BF16, ATTN_F16 or ATTN_F32 with D * element size a
 * multiple of 16 bytes, D <= 1024; o_parts and o 16-byte aligned.  Returns
 * ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED or ATTN_ERR_CUDA.
 */
ATTN_API int attn_lse_merge(const void* o_parts, const float* lse_parts, int n_parts, void* o,
                            float* lse, int B, int Hq, int T, int D, int dtype,
                            attn_stream_t stream);

/*
 * attn_bwd_workspace_size -- bytes of device scratch attn_bwd needs: one
 * float per query row for delta = rowsum(dO * O), the row term of the
 * softmax's chain rule that the backward forms once and reads for every key
 * tile ("Hands-on build guide: FlashAttention-style tiled attention kernel
 * in pure NumPy", Roadmap: gradient through attention by the chain rule;
 * "Self-Attention: Implementation, Complexity, and Efficient Variants",
 * FlashAttention: O(n) memory, nothing of size T x S is stored).  Returns 0
 * for invalid sizes.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int T);

/*
 * attn_bwd -- backward pass: dQ, dK, dV of the attention computed by attn_fwd
 * (or attn_fwd_chunked with the same q_pos), given dO and the forward's O
 * and LSE.  "Hands-on build guide: FlashAttention-style tiled attention
 * kernel in pure NumPy", Roadmap (gradient through attention by the chain
 * rule through the softmax); "Self-Attention: Implementation, Complexity,
 * and Efficient Variants", FlashAttention (the backward recomputes the
 * attention weights on chip instead of storing them):
 *
 *   P = exp(scale * Q K^T - LSE) on visible entries (0 elsewhere)
 *   dV = P^T dO,  dP = dO V^T,  delta = rowsum(dO * O)
 *   dS = P (dP - delta),  dQ = scale dS K,  dK = scale dS^T Q
 *
 * with the query heads of a GQA group summed into their KV head.  Padded
 * rows and rows that see no key take no part (their output is the constant
 * 0): their dQ is 0 and they add nothing to dK, dV.  Keys no row sees get
 * dK = dV = 0.  K/V rows at or past the valid length are never used.
 *
 *   q, o, dout  [B,Hq,T,D]   dtype (read)        q, dout finite on every row
 *   k, v        [B,Hkv,S,D]  dtype (read)
 *   lse         [B,Hq,T]     float32 (read: attn_fwd's LSE for these inputs)
 *   dq          [B,Hq,T,D]   dtype (written)
 *   dk, dv      [B,Hkv,S,D]  dtype (written)
 *   key_lens, q_pos, causal, scale: as for attn_fwd / attn_fwd_chunked
 *                            (q_pos NULL = bottom-right, S - T)
 *   workspace   >= attn_bwd_workspace_size(B, Hq, T) bytes, 16-byte aligned
 *
 * Supported:
 *   ATTN_BF16, ATTN_F16: D in {64, 128} (tcgen05 tensor cores, fp32
 *              accumulation; P and dS are rounded to the input type for the
 *              products); all pointers 16-byte aligned (lse, key_lens,
 *              q_pos: 4); B * Hq < 2^31 and at most 65535 tiles of 128 rows
 *              in T and in S.
 *   ATTN_F32:  1 <= D <= 256, 4-byte aligned; exact float32 on the CUDA
 *              cores (FFMA, accurate expf, no TF32), the counterpart of the
 *              fp32 forward.
 * No atomics: results do not depend on scheduling.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
 * ATTN_ERR_WORKSPACE or ATTN_ERR_CUDA.
 */
ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                      const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                      int Hq, int Hkv, int T, int S, int D, int dtype, int causal,
                      const int32_t* key_lens, const int32_t* q_pos, float scale,
                      void* workspace, size_t ws_bytes, attn_stream_t stream);

/*
 * attn_decode_workspace_size -- bytes of device scratch attn_decode needs for
 * a batch of B sequences, Hq query heads, caches of S_max positions and head
 * size D: the partial results (unnormalised output, running maximum and
 * denominator) of the pieces of the cache that are reduced independently
 * before they are merged with the online softmax's rescaling ("Implementing
 * attention from scratch", Core ideas, Stable softmax: partial sums kept
 * against a running maximum and rescaled by exp(m_old - m_new); KV caching:
 * one decode step reads the whole cache).  The caller allocates it (any
 * alignment >= 16 bytes) and may reuse it across calls on the same stream.
 * Returns 0 for invalid sizes.
 */
ATTN_API size_t attn_decode_workspace_size(int B, int Hq, int S_max, int D);

/*
 * attn_decode -- one decode step: a single new query per (b, h) attends over
 * the first kv_lens[b] cache rows ("Implementing attention from scratch",
 * KV caching: a decode step attends one new query over the cached
 * positions; with the query at position kv_lens[b]-1 the bottom-right causal
 * mask admits exactly rows 0..kv_lens[b]-1).  Split-KV: chunks of the cache
 * are reduced independently to (partial O, running max, denominator) and a
 * second pass merges them with the same exp(m_old - m_new) rescaling the
 * online softmax uses ("Implementing attention from scratch", Stable
 * softmax).
 *
 *   q         [B,Hq,D]          dtype   (read)
 *   kcache    [B,Hkv,S_max,D]   dtype   (read; rows >= kv_lens[b] ignored)
 *   vcache    [B,Hkv,S_max,D]   dtype   (read)
 *   kv_lens   [B] int32, device         (read; keys per sequence, INCLUDING
 *                                        the token just appended; values are
 *                                        clamped to [0, S_max]; 0 gives O = 0,
 *                                        LSE = -inf)
 *   o         [B,Hq,D]          dtype   (written)
 *   lse       [B,Hq] float32            (written; NULL = do not emit)
 *   workspace device scratch of >= attn_decode_workspace_size(B,Hq,S_max,D)
 *             bytes, 16-byte aligned; contents need no initialisation.
 *
 * Supported: dtype ATTN_BF16, ATTN_F16 or ATTN_F32; D in {64, 128};
 * Hq % Hkv == 0 and Hq / Hkv <= 16; q, caches, o 16-byte aligned.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
 * ATTN_ERR_WORKSPACE or ATTN_ERR_CUDA.
 */
ATTN_API int attn_decode(const void* q, const void* kcache, const void* vcache,
                const int32_t* kv_lens, void* o, float* lse, int B, int Hq,
                int Hkv, int S_max, int D, int dtype, float scale,
                void* workspace, size_t ws_bytes, attn_stream_t stream);

/*
 * attn_decode_append -- one generation step in one call: the new token's
 * K and V rows are appended to the caches and the step's query attends over
 * the cache including them.  "Implementing attention from scratch", KV
 * caching (the new token's keys and values are written at the cache length,
 * then the query attends over every cached position); "Building a causal
 * self-attention block from scratch in PyTorch", Step 5 (KVCache.update
 * before attention).  The same result as kv_cache_append with
 * pos[b] = kv_lens[b] - 1 followed by attn_decode, bit for bit, with one
 * launch less: the decode's split kernel writes the rows while it streams
 * the cache, replacing the one row it would have read stale.
 *
 *   q                 [B,Hq,D]        dtype          (read)
 *   kcache, vcache    [B,Hkv,S_max,D] dtype          (read; row kv_lens[b] - 1
 *                                                     of each (b, KV head)
 *                                                     written)
 *   k_new, v_new      [B,Hkv,D]       dtype          (read: the new token)
 *   kv_lens           [B]             int32, device  (valid rows INCLUDING the
 *                                                     new token; clamped to
 *                                                     [0, S_max] as in
 *                                                     attn_decode: a sequence
 *                                                     with kv_lens[b] <= 0
 *                                                     appends nothing, one
 *                                                     with kv_lens[b] > S_max
 *                                                     writes row S_max - 1)
 *   o, lse, scale, workspace: as for attn_decode (same workspace size)
 *
 * Supported: the types, sizes and alignment of attn_decode; k_new and
 * v_new 16-byte aligned.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG,
 * ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE or ATTN_ERR_CUDA.
 */
ATTN_API int attn_decode_append(const void* q, void* kcache, void* vcache, const void* k_new,
                                const void* v_new, const int32_t* kv_lens, void* o, float* lse,
                                int B, int Hq, int Hkv, int S_max, int D, int dtype, float scale,
                                void* workspace, size_t ws_bytes, attn_stream_t stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate device
 * memory.  (The pages have no counterpart; this is a library convenience.)
 *
 * Some callers cannot call cudaMalloc or hand the library a buffer: plugins
 * whose host framework owns every byte of device memory through its own
 * allocator, or real-time loops where cudaMalloc's implicit device
 * synchronisation and unbounded latency are not acceptable.  This entry
 * point takes the same arguments as attn_decode minus the workspace, and
 * uses instead a scratch array of ATTN_NOALLOC_SCRATCH_BYTES that the
 * library defines at file scope in device memory.  Every GPU on which the
 * library is loaded holds that array until the process exits.
 *
 *  - It allocates nothing and calls no allocating routine.
 *  - Requests whose workspace would exceed ATTN_NOALLOC_SCRATCH_BYTES
 *    (see attn_decode_workspace_size) return ATTN_ERR_WORKSPACE without
 *    launching anything; use attn_decode with your own workspace then.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the one array, which keeps whatever the last call left
 *    there.  Nothing in it needs clearing: each call writes every scratch
 *    slot it reads.  Calls that can overlap on the GPU (different streams,
 *    or different host threads) race on the array and must be serialised by
 *    the caller.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
ATTN_API int attn_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                                 const int32_t* kv_lens, void* o, float* lse, int B,
                                 int Hq, int Hkv, int S_max, int D, int dtype,
                                 float scale, attn_stream_t stream);

/*
 * kv_cache_append -- write one new token's K and V rows per (b, kv head) at
 * cache position pos[b] ("Building a causal self-attention block from
 * scratch in PyTorch", Step 5, KVCache.update appends the new token along
 * the sequence axis; "Implementing attention from scratch", KV caching: the
 * new token's offset is the cache length).  The cache is preallocated to
 * S_max positions, so an append is an O(1) row copy, not a concatenation.
 *
 *   kcache, vcache  [B,Hkv,S_max,D] dtype  (row pos[b] written)
 *   k_new, v_new    [B,Hkv,D]       dtype  (read)
 *   pos             [B] int32, device      (read, not modified: pass the
 *                                           cache length before the append,
 *                                           then decode with kv_lens = pos+1)
 *   dev_status      int32, device, or NULL (for every (b, g) whose pos[b] is
 *                                           outside [0, S_max) the row is
 *                                           NOT written and bit 0 is OR-ed
 *                                           into *dev_status)
 *
 * Supported: dtype ATTN_BF16, ATTN_F16 or ATTN_F32; D >= 1 with D *
 * element size a multiple of 16 bytes; all tensor pointers 16-byte aligned.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG or ATTN_ERR_CUDA.
 */
ATTN_API int kv_cache_append(void* kcache, void* vcache, const void* k_new,
                    const void* v_new, const int32_t* pos, int B, int Hkv,
                    int S_max, int D, int dtype, int* dev_status,
                    attn_stream_t stream);

/* attn_status_string -- static, human-readable text for a status code. */
ATTN_API const char* attn_status_string(int status);

/*
 * Diagnostics (not part of the attention arithmetic).
 *
 * attn_kernel_launches -- number of kernels this library has launched in
 *   this process (all entry points, all devices).  Host-side counter.
 *
 * attn_device_error -- reads (and, if `clear`, resets) the current device's
 *   error word, which a kernel sets instead of trapping when an internal
 *   pipeline wait exceeds its time limit.  0 means no error.  Synchronises
 *   the device.  Returns ATTN_OK or ATTN_ERR_CUDA.
 *
 * attn_selftest_wait_timeout -- checks the failure path of those waits:
 *   launches one warp that waits on a shared-memory barrier nothing will
 *   complete.  The wait gives up after its time limit (about one second),
 *   records ATTN_SELFTEST_ERROR in the device error word (unless an earlier
 *   error is already there) and returns; the context stays usable.  Returns
 *   ATTN_OK or ATTN_ERR_CUDA (launch status only).
 */
#define ATTN_SELFTEST_ERROR 0x1EE /* 0x100 (wait timed out) | site 0xEE */
ATTN_API unsigned long long attn_kernel_launches(void);
ATTN_API int attn_device_error(int* code, int clear);
ATTN_API int attn_selftest_wait_timeout(attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_B300_ATTN_H_ */
