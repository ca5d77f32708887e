/*
 * mla.h -- C ABI of libmla: Multi-head Latent Attention (MLA) decode over a
 * compressed latent KV cache, with the up-projections absorbed.
 *
 * The method (pages this library restates):
 *   - "MLA multi-head latent attention: low-rank compression and matrix
 *     absorption" (0539edu.com): section 2.2 (c_KV = h W_DKV, k = c_KV W_UK,
 *     v = c_KV W_UV), section 3.1 (q k^T = (q W_UK^T) c_KV^T and
 *     attn v = (attn c_KV) W_UV), sections 3.2 / 5.1 (absorbed inference with the
 *     weights viewed as [h, d_k, d_c] and [h, d_v, d_c]), section 5.2 (a
 *     preallocated latent cache written by position).
 *   - icman.com.cn MLA article, section 2 "decoupled RoPE": each cached token is
 *     a 512-wide latent c_KV followed by a 64-wide key k_R with RoPE applied.
 *   - attention-variants interview guide (hotelren.com): section 6.2 (one RoPE
 *     key shared by every head), section 7.3 (max-subtracted softmax).
 *   - "Gated MLA" (tahou.com): sections 2.6 / 3.2 (full-rank sigmoid output gate
 *     over the concatenated v width), section 3.3 (no positional encoding).
 *
 * Conventions shared by every call:
 *   - Every tensor argument is a DEVICE pointer owned by the caller, unless the
 *     argument says "host".  The library never allocates device memory and never
 *     synchronises the host, except in mla_get_device_error().  All work is queued
 *     asynchronously on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream).
 *   - Tensors are dense, row-major, with the shapes given in brackets; the cache
 *     may have padded rows (row_stride).  Element type is given by an mla_dtype
 *     argument: MLA_BF16 (bfloat16 storage, fp32 arithmetic) or MLA_F32.
 *   - Pointers must be 16-byte aligned.  Bad arguments that the host can see
 *     (null pointers, non-positive or unsupported sizes, misalignment, a
 *     workspace that is too small) return MLA_ERR_INVALID_ARG / MLA_ERR_WORKSPACE
 *     and launch nothing.  Bad values that only the device can see (an index or a
 *     sequence length out of range) are skipped/clamped by the kernels and
 *     recorded in a device error word, which mla_get_device_error() returns.
 *   - No exception crosses this ABI; every entry point returns mla_status.
 *   - With MLA_NVTX=1 in the environment (read at the first call), every compute
 *     entry point runs inside an NVTX range named after it, so that a profiler can
 *     select one operation's kernels; off, each call costs one branch.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,    /* a host-visible argument is invalid            */
  MLA_ERR_UNSUPPORTED = 2,    /* valid shape that this build has no kernel for */
  MLA_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed             */
  MLA_ERR_DEVICE_TIMEOUT = 4, /* a kernel's bounded wait expired (device word) */
  MLA_ERR_WORKSPACE = 5,      /* workspace pointer null or too small           */
  MLA_ERR_DEVICE_INDEX = 6    /* a device-side index/length was out of range   */
} mla_status;

typedef enum { MLA_BF16 = 0, MLA_F32 = 1 } mla_dtype;

/*
 * One layer's latent cache: data[b][t][0 : d_c + d_r] for b < B, t < N_max.
 * Row t of sequence b holds [c_KV(t) || RoPE(k_R(t), t)] (icman.com.cn section 2
 * cache-row figure; the position-indexed preallocated buffer of 0539edu.com
 * section 5.2).  row_stride >= d_c + d_r elements, and row_stride * element size
 * must be a multiple of 16 bytes.  The caller owns the buffer and the per-sequence
 * lengths; rows at t >= length may hold anything (they are never read into a
 * result).
 */
typedef struct {
  void* data;         /* device pointer, [B][N_max][row_stride] of dtype          */
  int32_t dtype;      /* mla_dtype                                                */
  int32_t B;          /* sequences                                                */
  int32_t N_max;      /* rows per sequence                                        */
  int32_t d_c;        /* latent width                                             */
  int32_t d_r;        /* decoupled RoPE key width (0 = no positional key)         */
  int32_t _pad;
  int64_t row_stride; /* elements between consecutive rows                        */
} mla_cache;

/*
 * A paged latent cache: rows live in fixed pages of MLA_PAGE_ROWS rows taken from
 * one pool, so sequences can grow without a per-sequence preallocation (the
 * position-indexed buffer of 0539edu.com section 5.2, split into pages).  Row t of
 * sequence b is row t % MLA_PAGE_ROWS of page block_table[b][t / MLA_PAGE_ROWS],
 * and holds [c_KV(t) || RoPE(k_R(t), t)] like mla_cache.  The caller owns the pool,
 * the block table and the page assignment; a page may belong to one sequence only.
 */
#define MLA_PAGE_ROWS 64
typedef struct {
  void* data;                  /* device pointer, [num_pages][MLA_PAGE_ROWS][row_stride] */
  int32_t dtype;               /* mla_dtype                                               */
  int32_t num_pages;           /* pages in the pool                                       */
  int32_t d_c;                 /* latent width                                            */
  int32_t d_r;                 /* decoupled RoPE key width (0 = no positional key)        */
  int64_t row_stride;          /* elements between consecutive rows (same rules as above) */
  const int32_t* block_table;  /* device pointer, [B][max_blocks] int32 page indices      */
  int32_t B;                   /* sequences                                               */
  int32_t max_blocks;          /* block-table entries per sequence; lengths <= 64 x this  */
} mla_paged_cache;

/* Version of this ABI (bumped on any incompatible change). */
MLA_API int32_t mla_abi_version(void);

/*
 * mla_build_source_hash -- a short hash of the sources this library was built
 * from (set by the build; "unknown" when built without it).  The Python binding
 * compares it with the sources beside it and refuses a library built from others.
 * (No counterpart on the pages: a build check.)
 */
MLA_API const char* mla_build_source_hash(void);

/* Human-readable name of a status code (static string, never NULL). */
MLA_API const char* mla_status_string(mla_status status);

/*
 * mla_cache_append -- write T new tokens into the latent cache.
 *   For each i < T: cache[seq_idx[i]][pos[i]] = [c_kv[i] || RoPE(k_r[i], pos[i])].
 *   RoPE rotates pairs (2j, 2j+1) of k_r by angle pos * base^(-2j/d_r) (the
 *   frequencies are formed in double precision, the angle to about 1e-6 rad).
 *   (Decoupled RoPE key: icman.com.cn section 2; hotelren.com section 6.2;
 *   append-by-position: 0539edu.com section 5.2.)
 *   c_kv     [T, d_c]   dtype = cache->dtype
 *   k_r      [T, d_r]   dtype = cache->dtype; may be NULL iff d_r == 0
 *   seq_idx  [T] int32  sequence of each row, in [0, B)
 *   pos      [T] int32  position of each row, in [0, N_max)
 *   A row whose seq_idx/pos is out of range is skipped and recorded as
 *   MLA_ERR_DEVICE_INDEX in the device error word.  Rows must not alias.
 */
MLA_API mla_status mla_cache_append(const mla_cache* cache, const void* c_kv, const void* k_r,
                                    const int32_t* seq_idx, const int32_t* pos, int32_t T,
                                    float rope_base, void* stream);

/*
 * mla_absorb_q -- fold W_UK into the query and rotate the RoPE part.
 *   q_cat[b][h] = [ q_nope[b][h] . W_UK[h]  ||  RoPE(q_rope[b][h], q_pos[b]) ]
 *   i.e. q_lat[b][h][c] = sum_d q_nope[b][h][d] * W_UK[h][d][c]
 *   (0539edu.com sections 3.1, 3.2 and 5.1: q W_UK^T computed once per query, with
 *   W_UK viewed as [h, d_k, d_c]).  Arithmetic in fp32; q_cat stored in dtype.
 *   q_nope [B, H, d_k]; q_rope [B, H, d_r] (NULL iff d_r == 0);
 *   q_pos [B] int32 (query position, normally length-1); W_UK [H, d_k, d_c];
 *   q_cat [B, H, d_c + d_r] (output).
 *   bf16: tensor-core kernel only; needs d_k % 64 == 0, d_c % 128 == 0,
 *   d_r <= 128 and (d_c + d_r) % 8 == 0 (MLA_ERR_UNSUPPORTED otherwise), and
 *   16-byte aligned q_nope, W_UK, q_cat and 4-byte aligned q_rope
 *   (MLA_ERR_INVALID_ARG otherwise).  f32: CUDA-core kernel, d_k <= 1600.
 */
MLA_API mla_status mla_absorb_q(const void* q_nope, const void* q_rope, const int32_t* q_pos,
                                const void* w_uk, void* q_cat, int32_t B, int32_t H, int32_t d_k,
                                int32_t d_c, int32_t d_r, int32_t dtype, float rope_base,
                                void* stream);

/*
 * mla_absorb_q_append -- mla_cache_append of T new rows and mla_absorb_q of B
 *   queries in one call: q_cat = [q_nope . W_UK || RoPE(q_rope, q_pos)] and
 *   cache[seq_idx[i]][pos[i]] = [c_kv[i] || RoPE(k_r[i], pos[i])], both with the
 *   same rope_base (d_c and d_r are the cache's, the dtype the cache's).  The
 *   results are bit-identical to the two calls.
 *   bf16: one tensor-core launch (the rows are written by the absorb grid's idle
 *   warps), so a decode step has one kernel boundary fewer; the limits and
 *   alignments of mla_absorb_q, plus a 16-byte aligned c_kv and a 4-byte aligned
 *   k_r (MLA_ERR_INVALID_ARG otherwise).  f32: the two CUDA-core kernels, one after the other.
 *   T == 0 appends nothing.  Bad rows are skipped and recorded as
 *   mla_cache_append does.  The query rows and the appended rows must not
 *   overlap in memory.
 */
MLA_API mla_status mla_absorb_q_append(const mla_cache* cache, const void* c_kv, const void* k_r,
                                       const int32_t* seq_idx, const int32_t* pos, int32_t T,
                                       const void* q_nope, const void* q_rope, const int32_t* q_pos,
                                       const void* w_uk, void* q_cat, int32_t B, int32_t H, int32_t d_k,
                                       float rope_base, void* stream);

/*
 * mla_decode_workspace_size -- bytes of device workspace mla_decode_attn needs
 * for B sequences and H heads of width d_c (split-KV partials, the block prefix
 * table and the split plan).  The size depends on the current device's SM count.
 * Returns 0 if the shape is unsupported.
 */
MLA_API size_t mla_decode_workspace_size(int32_t B, int32_t H, int32_t d_c, int32_t dtype);

/*
 * mla_decode_attn -- absorbed decode attention over the latent cache.
 *   For each sequence b with n = seq_lens[b] cached tokens and each head h:
 *     s_t  = scale * ( q_cat[b][h] . cache[b][t] )     over the d_c + d_r row
 *     p    = softmax_t(s)                              (max-subtracted)
 *     o_lat[b][h] = sum_t p_t * cache[b][t][0 : d_c]
 *     lse[b][h]   = ln sum_t exp(s_t)
 *   (0539edu.com sections 3.1-3.2: scores against c_KV directly, o_lat = P c_KV;
 *   the 64-wide rotated key term is the decoupled RoPE of icman.com.cn section 2;
 *   hotelren.com section 7.3 for the max subtraction.)
 *   The tokens of all sequences are split into equal runs across the GPU; each
 *   run produces an unnormalised partial (m, l, O) and a log-sum-exp combine
 *   merges the runs of each sequence (in two steps, groups of pieces and then the
 *   groups, when a batch of a few long sequences is cut into many pieces each).
 *   q_cat     [B, H, d_c + d_r]  dtype = cache->dtype
 *   seq_lens  [B] int32 device; 0 <= seq_lens[b] <= N_max.  A sequence of length 0
 *             gives o_lat = 0 and lse = -inf.  Out-of-range lengths are clamped
 *             and recorded as MLA_ERR_DEVICE_INDEX.
 *   workspace device scratch of at least mla_decode_workspace_size() bytes,
 *             256-byte aligned; contents need no initialisation; calls that
 *             share one workspace must be ordered on one stream.
 *   o_lat     [B, H, d_c] dtype (output);  lse [B, H] float32 or NULL.
 *   bf16 path: d_c = 512, d_r in {0, 64}, 1 <= H <= 128 (tensor-core kernel,
 *   bf16 operands, fp32 accumulation).  f32 path: any d_c <= 1024, d_r <= 256,
 *   H <= 1024 (fp32 CUDA-core kernel).  Other shapes: MLA_ERR_UNSUPPORTED.
 */
MLA_API mla_status mla_decode_attn(const void* q_cat, const mla_cache* cache,
                                   const int32_t* seq_lens, int32_t H, float scale,
                                   void* workspace, size_t workspace_bytes, void* o_lat,
                                   float* lse, void* stream);

/*
 * mla_decode_attn_partial -- decode attention over a range of each sequence's
 * cached rows, returned as a partial for a later merge.  For sequence b the query
 * attends to rows [row_begin[b], row_end[b]) only:
 *     o_part[b][h]   = sum_t softmax_t(s)_t * cache[b][t][0 : d_c],  t in the range
 *     lse_part[b][h] = ln sum_t exp(s_t)
 *   with s_t as in mla_decode_attn.  This is the unnormalised partial (m, l, O) of
 *   the range in log-sum-exp form: with m the row maximum and l = sum exp(s - m),
 *   O = o_part * l and lse_part = m + ln l.  Partials of disjoint ranges merge
 *   exactly into the attention over their union (mla_decode_merge).  It is the
 *   per-shard step of decode sharded by sequence position (the sequence-parallel
 *   remark of 0539edu.com, section 8: every shard holds some of each sequence's
 *   rows, computes its partial, and the partials are gathered and merged).
 *   q_cat, cache, H, scale, workspace: as mla_decode_attn.
 *   row_begin, row_end [B] int32 device: 0 <= row_begin[b] <= row_end[b] <= N_max
 *             (else clamped and recorded as MLA_ERR_DEVICE_INDEX).  An empty range
 *             gives o_part = 0 and lse_part = -inf.
 *   o_part    [B, H, d_c] bf16 (output);  lse_part [B, H] float32 (output, required).
 *   Limits: contiguous bf16 cache, d_c = 512, d_r in {0, 64}, 1 <= H <= 128
 *   (MLA_ERR_UNSUPPORTED otherwise).
 */
MLA_API mla_status mla_decode_attn_partial(const void* q_cat, const mla_cache* cache, const int32_t* row_begin,
                                           const int32_t* row_end, int32_t H, float scale, void* workspace,
                                           size_t workspace_bytes, void* o_part, float* lse_part, void* stream);

/*
 * mla_decode_merge -- merge k partials of disjoint row ranges (mla_decode_attn_partial
 * or any attention output with its log-sum-exp) into the attention over the union:
 *     M = max_s lse_s,  w_s = exp(lse_s - M)
 *     o_lat = sum_s w_s o_s / sum_s w_s,   lse = M + ln sum_s w_s
 *   (the max-subtracted softmax of hotelren.com, section 7.3, across row subsets).
 *   Rows whose partials are all empty (lse = -inf) give o_lat = 0 and lse = -inf.
 *   o_parts   [k, B, H, d_c] dtype, contiguous, device (e.g. gathered from k shards)
 *   lse_parts [k, B, H] float32, device
 *   o_lat     [B, H, d_c] dtype (output);  lse [B, H] float32 or NULL.
 *   fp32 arithmetic.  d_c % 8 == 0 (MLA_ERR_UNSUPPORTED otherwise); o_parts and
 *   o_lat 16-byte aligned.
 */
MLA_API mla_status mla_decode_merge(const void* o_parts, const float* lse_parts, int32_t k, int32_t B, int32_t H,
                                    int32_t d_c, int32_t dtype, void* o_lat, float* lse, void* stream);

/*
 * mla_prefill_workspace_size -- bytes of device workspace mla_prefill_attn needs
 * for B sequences of S queries each (block table and the partials of queries
 * whose rows are split across the GPU).  Returns 0 if the shape is unsupported.
 */
MLA_API size_t mla_prefill_workspace_size(int32_t B, int32_t S, int32_t H, int32_t d_c, int32_t dtype);

/*
 * mla_prefill_attn -- absorbed attention of a whole prompt over the latent cache.
 *   Prefill processes every prompt token at once (hotelren.com guide, section 2.1)
 *   with the absorbed query of each token (0539edu.com sections 3.1-3.2: the
 *   absorbed query and c_KV keep their [batch, seq, ...] shape).  The prompt's own
 *   rows must already be in the cache (mla_cache_append).  For sequence b, query i
 *   (position start = q_start[b] + i) and head h, with
 *   n = start + 1 rows if causal (rows 0..start: the diagonal is included) and
 *   n = q_start[b] + S rows otherwise:
 *     s_t  = scale * ( q_cat[b][i][h] . cache[b][t] ),  t < n
 *     o_lat[b][i][h] = sum_t softmax_t(s)_t * cache[b][t][0 : d_c]
 *     lse[b][i][h]   = ln sum_t exp(s_t)
 *   Every (b, i) is one attention problem with all H heads as the MMA rows; the
 *   rows of all problems are cut into equal runs across the GPU, exactly as in
 *   mla_decode_attn.
 *   q_cat     [B, S, H, d_c + d_r]  dtype = cache->dtype
 *   q_start   [B] int32 device; 0 <= q_start[b] and q_start[b] + S <= N_max,
 *             else the lengths are clamped and MLA_ERR_DEVICE_INDEX is recorded.
 *   causal    1: query i sees rows up to its own position; 0: all q_start[b] + S rows.
 *   workspace device scratch of at least mla_prefill_workspace_size() bytes,
 *             256-byte aligned (bf16 path; the f32 path ignores it).
 *   o_lat     [B, S, H, d_c] dtype (output);  lse [B, S, H] float32 or NULL.
 *   Shapes as mla_decode_attn; B * S * ceil(N_max / 64) must stay below 2^31.
 */
MLA_API mla_status mla_prefill_attn(const void* q_cat, const mla_cache* cache, const int32_t* q_start,
                                    int32_t S, int32_t H, float scale, int32_t causal, void* workspace,
                                    size_t workspace_bytes, void* o_lat, float* lse, void* stream);

/*
 * mla_out_up -- apply W_UV after attention, per head:
 *   o[b][h][d] = sum_c o_lat[b][h][c] * W_UV[h][d][c]
 *   (0539edu.com section 3.1, attn v = (attn c_KV) W_UV; weight view [h, d_v, d_c]
 *   of section 3.2).  o_lat [B, H, d_c]; W_UV [H, d_v, d_c]; o [B, H, d_v].
 *   fp32 arithmetic, dtype storage.
 *   bf16: tensor-core kernel only; needs d_c % 64 == 0 and d_v % 128 == 0
 *   (MLA_ERR_UNSUPPORTED otherwise) and 16-byte aligned o_lat, W_UV and o
 *   (MLA_ERR_INVALID_ARG otherwise).  f32: CUDA-core kernel, d_c <= 1024.
 */
MLA_API mla_status mla_out_up(const void* o_lat, const void* w_uv, void* o, int32_t B, int32_t H,
                              int32_t d_c, int32_t d_v, int32_t dtype, void* stream);

/*
 * mla_gate -- full-rank output gate of the gated variant, in place:
 *   o[b][j] *= sigmoid( sum_i h[b][i] * W_g[i][j] ),  j < width (= H * d_v)
 *   (tahou.com sections 2.6 and 3.2: one gate value per channel of the
 *   concatenated v-width output, computed from the token's own input).
 *   h [B, d_model]; W_g [d_model, width]; o [B, width] (read and written).
 *   bf16: tensor-core kernel only; needs d_model % 64 == 0 and width % 128 == 0
 *   (MLA_ERR_UNSUPPORTED otherwise) and 16-byte aligned h, W_g and o
 *   (MLA_ERR_INVALID_ARG otherwise).  f32: CUDA-core kernel, any shape.
 */
MLA_API mla_status mla_gate(const void* h, const void* w_g, void* o, int32_t B, int32_t d_model,
                            int32_t width, int32_t dtype, void* stream);

/*
 * mla_cache_append_paged -- mla_cache_append into a paged cache: row
 *   (seq_idx[i], pos[i]) goes to row pos[i] % MLA_PAGE_ROWS of page
 *   block_table[seq_idx[i]][pos[i] / MLA_PAGE_ROWS].  Arguments and RoPE as
 *   mla_cache_append.  A row whose sequence, position (pos >= 64 x max_blocks) or
 *   page index (outside [0, num_pages)) is out of range is skipped and recorded as
 *   MLA_ERR_DEVICE_INDEX.
 */
MLA_API mla_status mla_cache_append_paged(const mla_paged_cache* cache, const void* c_kv, const void* k_r,
                                          const int32_t* seq_idx, const int32_t* pos, int32_t T,
                                          float rope_base, void* stream);

/* mla_absorb_q_append with the rows placed in a paged cache (as
 * mla_cache_append_paged). */
MLA_API mla_status mla_absorb_q_append_paged(const mla_paged_cache* cache, const void* c_kv, const void* k_r,
                                             const int32_t* seq_idx, const int32_t* pos, int32_t T,
                                             const void* q_nope, const void* q_rope, const int32_t* q_pos,
                                             const void* w_uk, void* q_cat, int32_t B, int32_t H, int32_t d_k,
                                             float rope_base, void* stream);

/*
 * mla_decode_attn_paged -- mla_decode_attn over a paged cache (same result, bit
 *   for bit, as mla_decode_attn over a contiguous cache holding the same rows).
 *   seq_lens [B] int32 device, 0 <= seq_lens[b] <= 64 x max_blocks (clamped and
 *   recorded as MLA_ERR_DEVICE_INDEX otherwise); the first ceil(seq_lens[b] / 64)
 *   block-table entries of sequence b must name pages of the pool (an index
 *   outside [0, num_pages) is recorded as MLA_ERR_DEVICE_INDEX and page 0 is read
 *   instead).  Rows of the last page past seq_lens[b] may hold anything.
 *   Workspace as mla_decode_attn (mla_decode_workspace_size(B, ...)).  bf16 pool,
 *   d_c = 512, d_r in {0, 64}, 1 <= H <= 128; other shapes: MLA_ERR_UNSUPPORTED.
 */
MLA_API mla_status mla_decode_attn_paged(const void* q_cat, const mla_paged_cache* cache,
                                         const int32_t* seq_lens, int32_t H, float scale, void* workspace,
                                         size_t workspace_bytes, void* o_lat, float* lse, void* stream);

/*
 * mla_prefill_explicit_workspace_size -- bytes of device workspace
 * mla_prefill_explicit needs: the rebuilt K_nope and V, 2 x B x (start + S) x H x
 * 128 bf16.  0 if a size is not positive (start may be 0).
 */
MLA_API size_t mla_prefill_explicit_workspace_size(int32_t B, int32_t start, int32_t S, int32_t H);

/*
 * mla_prefill_explicit -- prefill of a prompt chunk without absorption.  Every
 *   head's keys and values are rebuilt from the cached latent rows (0539edu.com
 *   section 2.2: k = c_KV W_UK, v = c_KV W_UV; the same page notes that absorption
 *   makes prefill more expensive and that the explicit form is the precision
 *   fallback), and the prompt runs standard attention per head:
 *     k_h,t = [c_KV,t W_UK,h^T || k_R,t (as cached, rotated)]
 *     q_h,i = [q_nope[b][i][h] || RoPE(q_rope[b][i][h], start + i)]
 *     o[b][i][h] = sum_t softmax_t(scale q_h,i . k_h,t) c_KV,t W_UV,h^T
 *     lse[b][i][h] = ln sum_t exp(scale q_h,i . k_h,t)
 *   over t <= start + i when causal, t < start + S otherwise.  The result equals
 *   mla_prefill_attn followed by mla_out_up (same rows, same queries), with fewer
 *   FLOPs per score.  All sequences share the chunk offset `start`; rows
 *   0 .. start + S - 1 of every sequence must be in the cache.
 *   q_nope [B, S, H, 128], q_rope [B, S, H, 64] bf16 (unrotated); W_UK, W_UV
 *   [H, 128, 512] bf16; o [B, S, H, 128] bf16 (output); lse [B, S, H] float32 or
 *   NULL.  Workspace: mla_prefill_explicit_workspace_size(B, start, S, H) bytes,
 *   16-byte aligned.  Limits: bf16 cache with d_c = 512 and d_r = 64, d_k = d_v =
 *   128, H even (MLA_ERR_UNSUPPORTED otherwise); start + S <= N_max.
 */
MLA_API mla_status mla_prefill_explicit(const void* q_nope, const void* q_rope, const mla_cache* cache,
                                        const void* w_uk, const void* w_uv, int32_t start, int32_t S,
                                        int32_t causal, int32_t H, float scale, float rope_base,
                                        void* workspace, size_t workspace_bytes, void* o, float* lse,
                                        void* stream);

/*
 * mla_kv_down_workspace_size -- bytes of device workspace mla_kv_down_append needs
 * for T tokens (fp32 partial sums of the projection).  0 if T <= 0 or the sizes
 * are not positive.
 */
MLA_API size_t mla_kv_down_workspace_size(int32_t T, int32_t d_model, int32_t d_c, int32_t d_r,
                                          int32_t dtype);

/*
 * mla_kv_down_append -- the new tokens' cache rows straight from their hidden
 *   states, in place of computing c_kv / k_r separately and calling
 *   mla_cache_append:
 *     x        = h[i] W_DKV                          (0539edu.com section 2.2)
 *     c_KV     = x / sqrt(mean_j x_j^2 + eps) * gamma (RMSNorm after the
 *                                                     compression: section 6.3)
 *     k_R      = RoPE(h[i] W_KR, pos[i])             (hotelren.com section 6.2)
 *     cache[seq_idx[i]][pos[i]] = [c_KV || k_R]      (as mla_cache_append)
 *   The projection accumulates in fp32 (bf16 operands on the tensor cores for bf16
 *   caches), the norm and the rotation are fp32, the row is stored in the cache
 *   dtype.  Deterministic: the same inputs give the same bits.
 *   h        [T, d_model]         cache dtype, device
 *   w_dkvr   [d_model, d_c + d_r] cache dtype, device: W_DKV in columns [0, d_c),
 *                                 W_KR in columns [d_c, d_c + d_r)
 *   gamma    [d_c]                cache dtype, device: the RMSNorm gain
 *   eps      >= 0, added to the mean square
 *   seq_idx, pos [T] int32 device: as mla_cache_append (bad rows skipped and
 *            recorded as MLA_ERR_DEVICE_INDEX)
 *   workspace device scratch of mla_kv_down_workspace_size(T, d_model, d_c, d_r,
 *            dtype) bytes, 16-byte aligned (MLA_ERR_WORKSPACE otherwise).
 *   Limits: d_c even, d_c + d_r <= 1024 (MLA_ERR_UNSUPPORTED otherwise).  bf16
 *   caches project on the tensor cores only: d_model % 64 == 0 and
 *   (d_c + d_r) % 8 == 0 (MLA_ERR_UNSUPPORTED otherwise), 16-byte aligned h and
 *   w_dkvr (MLA_ERR_INVALID_ARG otherwise).  fp32 caches take a CUDA-core
 *   projection.  gamma is always applied: pass ones for an RMSNorm without gain.
 */
MLA_API mla_status mla_kv_down_append(const mla_cache* cache, const void* h, const void* w_dkvr,
                                      const void* gamma, float eps, const int32_t* seq_idx,
                                      const int32_t* pos, int32_t T, int32_t d_model, float rope_base,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* mla_kv_down_append into a paged cache (rows placed as mla_cache_append_paged). */
MLA_API mla_status mla_kv_down_append_paged(const mla_paged_cache* cache, const void* h,
                                            const void* w_dkvr, const void* gamma, float eps,
                                            const int32_t* seq_idx, const int32_t* pos, int32_t T,
                                            int32_t d_model, float rope_base, void* workspace,
                                            size_t workspace_bytes, void* stream);

/*
 * mla_decode_attn_noalloc -- mla_decode_attn for callers that cannot allocate.
 *   (No counterpart on the pages this library restates: it is a deployment aid.)
 *   Some callers cannot hand the library a workspace: code running under an
 *   allocator that must not be re-entered from where attention is called, runtimes
 *   whose device memory is fixed when they start, or embedders that only own the
 *   input and output buffers a host framework gives them.  This entry point computes exactly what mla_decode_attn does,
 *   with the same kernels, but takes the split-KV scratch from a buffer built into
 *   the library (about 25 MB per GPU that loads the library, held until the
 *   process exits), so it allocates nothing.
 *   Arguments are those of mla_decode_attn minus the workspace.  Limits: bf16 cache
 *   only (MLA_ERR_UNSUPPORTED otherwise) and at most 32 sequences (cache->B > 32
 *   returns MLA_ERR_WORKSPACE).  The first call on a device looks up the buffer's
 *   device address; make that first call before any stream capture.  All calls on
 *   a device share the one buffer: calls whose work could overlap on the GPU
 *   (unordered streams) race on it and must be serialised by the caller.  Nothing
 *   in the buffer needs clearing between calls.
 */
MLA_API mla_status mla_decode_attn_noalloc(const void* q_cat, const mla_cache* cache, const int32_t* seq_lens,
                                           int32_t H, float scale, void* o_lat, float* lse, void* stream);

/*
 * mla_get_device_error -- wait for the device, then read and clear the device
 * error word written by the kernels of this library on the current device.
 * Returns MLA_OK if no kernel recorded an error since the last call, otherwise
 * the recorded status (MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_DEVICE_INDEX).  If
 * `detail` is not NULL it receives the raw word (status in the low byte, the
 * site that recorded it above).
 */
MLA_API mla_status mla_get_device_error(uint32_t* detail);

/*
 * mla_debug_inject_fault -- fault injection for tests of the failure detection.
 *   (No counterpart on the pages: it exercises this library's bounded waits.)
 *   kind = 1: every later mla_decode_attn / mla_prefill_attn launch on the bf16
 *   tensor-core path issues no cache or query loads in its score CTAs, so the
 *   waits on those loads run out after their bound (about one second): the call
 *   records MLA_ERR_DEVICE_TIMEOUT in the device error word, its outputs are
 *   undefined, and the CUDA context stays usable.  kind = 0 switches it off.
 *   Nothing faults, traps or hangs.  Process-wide setting (an atomic switch that
 *   every later launch on any host thread or device reads); for tests only.  Returns MLA_ERR_INVALID_ARG for any
 *   other kind.
 */
MLA_API mla_status mla_debug_inject_fault(int32_t kind);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
