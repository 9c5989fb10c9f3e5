/*
 * relattn.h -- C ABI of the GB300 relative-attention forward library
 *              (librelattn.so, built for sm_103a).
 *
 * The operation (page "SGLang and Miles Add Day-0 Support for Inkling",
 * section "Attention with Relative Positional Embedding"): every query row
 * carries a relative feature r_{t,h}; a learned projection P turns it into
 * relative logits indexed by causal distance d,
 *
 *     rel_logits(t,h,d) = sum_c r[t,h,c] * P[c,d],          0 <= d < rel_extent,
 *
 * and the attention logit of query i, key j, head h is
 *
 *     l(i,j,h) = alpha * q_i . k_j + [0 <= i-j < rel_extent] * rel_logits(i,h,i-j).
 *
 * Future keys are masked; distances at or past rel_extent add no bias.
 * Sliding-window layers (same section, paragraph "Attention layout") keep key
 * j only when i - j < window.  Full layers may scale q and the relative logits
 * by a length-dependent factor; the page gives no formula, and this library
 * uses s(i) = max(1, ln(i+1)/ln(log_scale_base)), which multiplies the whole
 * logit.  All layers are GQA with head size 128 (page "vLLM Day-0 support for
 * TML Inkling", attention paragraph): query head h reads kv head
 * h / (num_heads_q / num_heads_kv).
 *
 * Outputs: out = softmax-weighted sum of v (bf16) and the per-row natural-log
 * logsumexp of the logits (fp32).
 *
 * Positions are bottom-right aligned: query row t of sequence b sits at
 * position (Lk_b - Lq_b) + t, where Lq_b / Lk_b come from cu_seqlens_q / _k.
 * Prefill has Lq_b == Lk_b; decode (<= 16 query rows, e.g. an MTP verify of 9
 * positions) has Lq_b <= Lk_b and the rows are causal among themselves.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or synchronises; work is enqueued on `stream`
 *     (a cudaStream_t; NULL = legacy default stream) and returns immediately.
 *   - Every function returns a relattn_status; nothing aborts or throws.
 *     Argument errors are found on the host before any launch.  cu_seqlens
 *     contents live on the device and are checked by the kernels: a sequence
 *     with Lk < Lq or lengths above max_seqlen_* is skipped and recorded in a
 *     device error word that relattn_get_device_error() reads.
 *   - Layouts are row-major with the last dimension contiguous:
 *       q   [total_q, num_heads_q,  128]        bf16
 *       k,v [total_k, num_heads_kv, 128]        bf16
 *       r   [total_q, num_heads_q,  r_dim]      bf16
 *       P   [r_dim, rel_extent]                 bf16 (shared by all heads)
 *       out [total_q, num_heads_q,  128]        bf16
 *       lse [num_heads_q, total_q]              fp32
 *     q, k, v, out must be 16-byte aligned.
 */
#ifndef RELATTN_H
#define RELATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RELATTN_OK = 0,
  RELATTN_ERR_INVALID_ARG = 1,  /* a pointer, size or flag is out of range      */
  RELATTN_ERR_UNSUPPORTED = 2,  /* valid attention, but outside what is built   */
  RELATTN_ERR_CUDA = 3,         /* a CUDA call or kernel launch failed          */
  RELATTN_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up           */
  RELATTN_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required   */
  RELATTN_ERR_DEVICE_ARGS = 6   /* kernels found inconsistent cu_seqlens        */
} relattn_status;

typedef struct relattn_params {
  const void *q;               /* bf16 [total_q, num_heads_q, 128]                  */
  const void *k;               /* bf16 [total_k, num_heads_kv, 128]                 */
  const void *v;               /* bf16 [total_k, num_heads_kv, 128]                 */
  const void *r;               /* bf16 [total_q, num_heads_q, r_dim]                */
  const void *P;               /* bf16 [r_dim, rel_extent]                          */
  const int32_t *cu_seqlens_q; /* device int32 [batch+1], query rows per sequence    */
  const int32_t *cu_seqlens_k; /* device int32 [batch+1], keys per sequence          */
  int32_t batch;               /* number of sequences                                */
  int32_t total_q;             /* cu_seqlens_q[batch] (host copy; sizes lse)         */
  int32_t total_k;             /* cu_seqlens_k[batch] (host copy)                    */
  int32_t max_seqlen_q;        /* upper bound on any Lq_b                            */
  int32_t max_seqlen_k;        /* upper bound on any Lk_b                            */
  int32_t num_heads_q;
  int32_t num_heads_kv;        /* divides num_heads_q                                */
  int32_t head_dim;            /* must be 128                                        */
  int32_t r_dim;               /* 0..64 (0: no relative bias)                        */
  int32_t rel_extent;          /* E >= 0: distances 0..E-1 carry bias                */
  int32_t window;              /* <= 0: full attention; else keep 0 <= i-j < window  */
  float alpha;                 /* logit scale, e.g. 1/sqrt(128)                      */
  float log_scale_base;        /* <= 0: off; else > 1, s(i)=max(1,ln(i+1)/ln(base))  */
  void *out;                   /* bf16 [total_q, num_heads_q, 128]                   */
  float *lse;                  /* fp32 [num_heads_q, total_q], natural log           */
  void *workspace;             /* decode scratch (device), may be NULL when none     */
  size_t workspace_bytes;
  int32_t num_splits;          /* decode: 0 = choose automatically                   */
} relattn_params;

/*
 * Prefill / chunked prefill: any Lq_b <= Lk_b.  rows are grouped into 128-row
 * query tiles per head; key tiles outside the causal / window range are
 * skipped.  Needs no workspace.
 *
 * Speed depends on the shape.  The tensor-core (tcgen05) kernels take the
 * call when q, k, v, out (and r, P with a bias) are 16-byte aligned, r_dim
 * and rel_extent are multiples of 8, rel_extent >= 64 (or no bias), r_dim
 * <= 64, and total_k >= 128.  Any other valid shape runs on a warp-level MMA
 * kernel with the same results, about 2-3x slower (277 vs 662 TFLOP/s on a
 * 4 x 8192 sliding-window prefill).
 */
relattn_status relattn_prefill(const relattn_params *params, void *stream);

/*
 * Decode: max_seqlen_q <= 16 query rows per sequence against a long KV
 * (page "vLLM Day-0 support for TML Inkling", FA4-with-sheared-bias paragraph:
 * the KV range is cut into num_splits pieces chosen from batch and KV length).
 * Each split writes a partial (out, lse) to the workspace and a combine kernel
 * merges them by their logsumexp.  num_splits = 0 picks the split count; the
 * chosen count is the one relattn_decode_workspace_size() sizes for.
 *
 * Speed depends on the shape.  Calls of at most 16 rows per kv head
 * (max_seqlen_q x num_heads_q / num_heads_kv <= 16) take the few-row
 * tensor-core kernel when q, k, v, out are 16-byte aligned and total_k >= 128:
 * any r_dim <= 64 and any rel_extent.  Wider calls (e.g. a 9-token verify of
 * a GQA-8 group) take the 128-row tensor-core kernel under the prefill's
 * conditions above.  Any other valid shape runs on a warp-level MMA kernel
 * with the same results, about 2x slower (2.7 vs 5.6 TB/s on a 9-row, 1M-key
 * decode).
 */
relattn_status relattn_decode(const relattn_params *params, void *stream);

/*
 * Workspace bytes relattn_decode needs for these params: the split partials
 * (fp32 out and lse of every split) when the keys are cut into several
 * splits, and, when max_seqlen_q x (num_heads_q / num_heads_kv) <= 16 and a
 * relative bias is on, room for the bias r . P: the larger of the bias of
 * every decode row at every distance below rel_extent (fp32, total_q x
 * num_heads_q x rel_extent; computed by a kernel before the decode) and, when
 * r is 16-byte aligned with r_dim a multiple of 8 and rel_extent <= 1152,
 * two slots per SM of one item's bias (fp32, rel_extent rounded up to 128 x
 * the item's rows rounded up to 4; computed inside the decode kernel on the
 * tensor cores).  0 when neither applies.  The workspace must be 16-byte
 * aligned; its contents are scratch.
 */
relattn_status relattn_decode_workspace_size(const relattn_params *params, size_t *bytes);

/* The split count relattn_decode will use for these params. */
relattn_status relattn_decode_num_splits(const relattn_params *params, int32_t *num_splits);

/*
 * Decode against a paged KV cache.  The keys of each sequence live in
 * fixed-size pages of a pool: key p of sequence b sits at pool row
 * block_table[b * max_pages_per_seq + p / page_size] * page_size + p % page_size
 * of params->k / params->v (bf16 [num_pages * page_size, num_heads_kv, 128]).
 * cu_seqlens_k keeps its meaning as cumulative key counts (Lk_b =
 * cu_seqlens_k[b+1] - cu_seqlens_k[b]); total_k is their sum (used for
 * planning only).  Everything else, including the split plan, the workspace
 * (relattn_decode_workspace_size) and the results, is relattn_decode's:
 * same arithmetic, bit-identical out / lse.  The pages give no paging
 * scheme; this is the block-table layout of paged serving caches.
 * Requirements: page_size a multiple of 128 (a 128-key tile stays inside a
 * page), max_pages_per_seq * page_size >= max_seqlen_k, num_pages *
 * page_size < 2^31, and the shapes the tcgen05 kernel takes (16-byte aligned
 * pointers; with a bias r_dim and E multiples of 8, r_dim <= 64, E >= 64);
 * else RELATTN_ERR_UNSUPPORTED.  A block-table entry outside [0, num_pages)
 * makes its keys read as zero and records RELATTN_ERR_DEVICE_ARGS.
 */
typedef struct relattn_paged_kv {
  const int32_t *block_table;  /* device int32 [batch, max_pages_per_seq]: pool page per block */
  int32_t max_pages_per_seq;
  int32_t page_size;           /* keys per page, a multiple of 128 */
  int32_t num_pages;           /* pages in the k / v pools */
} relattn_paged_kv;

relattn_status relattn_decode_paged(const relattn_params *params, const relattn_paged_kv *kv,
                                   void *stream);

/*
 * MXFP8 K / V cache (page "SGLang and Miles Add Day-0 Support for Inkling",
 * section "Relative Logits Optimization", paragraph "MXFP8 Support": K and V
 * stored in MXFP8, Q K^T as an MXFP8 product, P V in bf16 with V dequantised
 * on the fly).  The format is OCP Microscaling MXFP8: FP8 E4M3 codes (bias 7,
 * largest finite 448, S.1111.111 NaN) and one E8M0 scale byte b = 2^(b - 127)
 * per 32 consecutive elements of the last dimension.
 *
 * relattn_quantize_mxfp8: n_blocks blocks of 32 bf16 values (x, device,
 * 16-byte aligned, contiguous) -> codes (uint8 [n_blocks * 32], 16-byte
 * aligned) and scales (uint8 [n_blocks]).  Per block, e = floor(log2 amax) - 8
 * clamped to [-127, 127] (-127 for an all-zero block); each code is
 * x * 2^-e rounded to the nearest E4M3 value, ties to even, the sign kept
 * (-0 for a negative value that rounds to zero), saturating at 448.  For a
 * K / V cache [rows, heads, 128] the blocks are the 4 runs of 32 dims of every
 * (row, head): scales [rows, heads, 4].  x must not overlap codes or scales.
 * Finite inputs only.  Asynchronous on `stream`.
 */
relattn_status relattn_quantize_mxfp8(const void *x, int64_t n_blocks, void *codes, void *scales,
                                      void *stream);

typedef struct relattn_kv_mxfp8 {
  const void *k;               /* uint8 E4M3 [total_k, num_heads_kv, 128], 16-byte aligned */
  const void *v;               /* uint8 E4M3 [total_k, num_heads_kv, 128], 16-byte aligned */
  const void *k_scale;         /* uint8 E8M0 [total_k, num_heads_kv, 4], 4-byte aligned    */
  const void *v_scale;         /* uint8 E8M0 [total_k, num_heads_kv, 4], 4-byte aligned    */
} relattn_kv_mxfp8;

/*
 * Decode against an MXFP8 K / V cache.  Same arguments and results as
 * relattn_decode (params->k / params->v are ignored; kv gives the codes and
 * scales, contiguous rows cu_seqlens_k[b] + p like relattn_decode's K / V),
 * same split plan and workspace (relattn_decode_workspace_size of the same
 * params).  What it computes: the relative-attention forward with q rounded
 * through MXFP8 per 32 head dims of each row (Q K^T runs as an E4M3 x E4M3
 * product per 32-dim block, fp32 accumulate, block scales applied in fp32),
 * K = dequantised k codes, V = dequantised v codes (exact in bf16; P V in
 * bf16, fp32 accumulate).  Requires max_seqlen_q x (num_heads_q /
 * num_heads_kv) <= 16 (batched decode: one token of a GQA group up to 16, or a
 * few tokens of a smaller one), r_dim <= 64 and total_k >= 128; else
 * RELATTN_ERR_UNSUPPORTED.
 */
relattn_status relattn_decode_mxfp8(const relattn_params *params, const relattn_kv_mxfp8 *kv,
                                    void *stream);

/*
 * Log-sum-exp combine of split partials (the decode combine step, exposed so
 * partials from several KV shards can be merged):
 *   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s.
 * o_part  fp32 [num_splits, rows, 128]   (normalised partial outputs)
 * lse_part fp32 [num_splits, rows]        (-inf marks an empty partial)
 * out bf16 [rows, 128]; lse fp32 with element (row) at lse[row_to_lse(row)]
 * where rows are ordered (t, h) and lse is [num_heads, total_q]:
 * row = t * num_heads + h  ->  lse[h * total_q + t].
 */
relattn_status relattn_combine(const float *o_part, const float *lse_part, int32_t num_splits,
                               int32_t total_q, int32_t num_heads, void *out, float *lse,
                               void *stream);

/*
 * Decode without a caller workspace and without allocating.  (The Inkling
 * pages have no counterpart to this; it is an integration convenience.)
 *
 * Same computation, arguments and results as relattn_decode, except that the
 * split partials go to a fixed scratch array inside this library instead of
 * params->workspace (which is ignored).  It is meant for callers that cannot
 * call cudaMalloc where they run attention: engines that reserve all free
 * device memory for their own pools up front, plugin hosts that offer no
 * workspace hook, and latency-critical paths that cannot afford cudaMalloc's
 * implicit device synchronisation.  Nothing is allocated or freed by the call.
 *
 * Limits and sharing:
 *   - The scratch holds RELATTN_NOALLOC_SCRATCH_BYTES per device, for as long
 *     as the library is loaded.  When relattn_decode_workspace_size() reports
 *     more than that for these params, the call returns RELATTN_ERR_WORKSPACE
 *     and launches nothing (pass a smaller num_splits, or use relattn_decode).
 *   - The first call on a device looks up the array's device address (with
 *     that device current), and so does the first call after the device's
 *     context changes (a cudaDeviceReset loads the library's module again).
 *     Make those calls before any stream capture.
 *   - Every call on a device shares the one array.  No contents need to carry
 *     over between calls, but two calls whose kernels can overlap on the GPU
 *     (unordered streams) race on it: order them, or use relattn_decode.
 */
#define RELATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
relattn_status relattn_decode_noalloc(const relattn_params *params, void *stream);

/* Reads and clears the device error word (RELATTN_OK when clean).  Synchronises
 * `stream` to read it. */
relattn_status relattn_get_device_error(void *stream);

/* Raw device error word seen by the last relattn_get_device_error() call:
 * bit 0 = inconsistent cu_seqlens, bit 1 = a bounded wait gave up, bits 8+ =
 * the id of the wait that gave up first (diagnostics only). */
int32_t relattn_last_device_error_word(void);

/*
 * Backward pass (page "SGLang and Miles Add Day-0 Support for Inkling",
 * section "Customized Efficient Kernels for Train-Inference Consistency",
 * paragraph "Relative attention": the training side differentiates through
 * the attention scores and r while P stays frozen).  Given the forward's
 * inputs, its saved out / lse and the upstream gradient dout, it writes the
 * gradients of sum(dout * out):
 *   dq [total_q, Hq, 128], dk / dv [total_k, Hkv, 128], dr [total_q, Hq, r_dim]
 * (bf16; dk / dv summed over the query heads of each GQA group; no gradient
 * for P).  With D_i = dout_i . out_i and dl = p (dout_i . v_j - D_i):
 * dq_i = s_i alpha sum_j dl k_j, dk_j = sum_i s_i alpha dl q_i,
 * dv_j = sum_i p dout_i, dr_i = s_i sum_j dl P[:, i-j] over 0 <= i-j < E.
 * The softmax weights are recomputed from lse (fp32 arithmetic, bf16 MMA
 * operands).  Every key row of dk / dv is written (zero when no query sees
 * it); dq / dr rows of every query row are written.
 *
 * Layouts and conventions are the forward's (fwd.*); fwd.out and fwd.lse are
 * read, fwd.workspace / fwd.num_splits are ignored.  The workspace (device,
 * 16-byte aligned, at least relattn_backward_workspace_size() bytes) holds
 * D (4 * Hq * total_q bytes) and, with a bias, R = r . P for every row, head
 * and distance below E in fp32 (4 * total_q * Hq * E, E rounded up to 4) and
 * the part of dq from keys outside the bias band in fp32 (4 * total_q * Hq * 128);
 * and, when Hq / Hkv is even and at least 4, two fp32 halves of dk and of dv
 * (16 * total_k * Hkv * 128 bytes).  The contents are scratch: nothing is
 * read from it before this call writes it.
 * Requirements: every pointer 16-byte aligned, r_dim a multiple of 8 (0..64).
 * Errors: RELATTN_ERR_INVALID_ARG (NULL or unaligned pointers, bad sizes),
 * RELATTN_ERR_UNSUPPORTED (head_dim != 128, r_dim not a multiple of 8 or
 * above 64), RELATTN_ERR_WORKSPACE (workspace missing or too small);
 * inconsistent cu_seqlens contents skip the sequence and record
 * RELATTN_ERR_DEVICE_ARGS for relattn_get_device_error().
 */
typedef struct relattn_bwd_params {
  relattn_params fwd;          /* the forward call; fwd.out / fwd.lse are inputs here */
  const void *dout;            /* bf16 [total_q, num_heads_q, 128]                  */
  void *dq;                    /* bf16 [total_q, num_heads_q, 128]                  */
  void *dk;                    /* bf16 [total_k, num_heads_kv, 128]                 */
  void *dv;                    /* bf16 [total_k, num_heads_kv, 128]                 */
  void *dr;                    /* bf16 [total_q, num_heads_q, r_dim]; NULL if r_dim == 0 */
  void *workspace;             /* device, >= relattn_backward_workspace_size bytes  */
  size_t workspace_bytes;
} relattn_bwd_params;

relattn_status relattn_backward_workspace_size(const relattn_bwd_params *params, size_t *bytes);
relattn_status relattn_backward(const relattn_bwd_params *params, void *stream);

/*
 * Attention prologue: the step right before the attention forward (page
 * "SGLang and Miles Add Day-0 Support for Inkling", section "ShortConv
 * Optimization", paragraph "KV ShortConv + QK-norm + KV store"), for one
 * chunk of new rows of packed sequences:
 *   - K and V each go through ShortConv (section "Short Convolution"), a
 *     per-channel causal filter with W = 4 taps and the input added back:
 *         y[t,c] = x[t,c] + sum_{d=0}^{3} w[c,d] * x[t-d,c],
 *     channel c = kv_head * 128 + dim, taps over the sequence's rows;
 *   - Q and the convolved K are RMS-normalised per token and head over the
 *     128 dims: x * rsqrt(mean(x^2) + eps) * gamma (one gamma of 128 values
 *     for q, one for k, shared by the heads -- the pages give no detail);
 *   - the normalised K and the convolved V are written to the KV cache rows
 *     the attention reads: chunk row t of sequence b goes to cache row
 *     cu_seqlens_k[b] + (Lk_b - Lq_b) + t (the chunk is the sequence's tail).
 * Inputs before the chunk's first row come from conv_state_in[b] (the 3
 * pre-convolution inputs that precede it, oldest first), or are zero when
 * conv_state_in is NULL (the sequence starts with the chunk).  When
 * conv_state_out is not NULL it receives the last 3 pre-convolution inputs
 * of each sequence up to the chunk's end (earlier ones from the state in, or
 * zero); it must not overlap conv_state_in.  q_out may be q itself (in
 * place) but must not partly overlap it; the caches must not overlap k or v.
 * Cache rows outside the chunk's rows are left untouched.  Arithmetic in
 * fp32, every output rounded once to bf16.
 *
 * Errors: RELATTN_ERR_UNSUPPORTED for head_dim != 128;
 * RELATTN_ERR_INVALID_ARG for a NULL required pointer (all but the four
 * states, when batch > 0), negative sizes, num_heads_kv not dividing
 * num_heads_q, q / k / v / q_out / caches / states / conv and norm weights
 * not 16-byte aligned, eps not a finite number > 0.
 * cu_seqlens contents are checked on the device: a row outside its
 * sequence, Lq_b > Lk_b, or cache rows outside [0, total_k) skip the row and
 * record RELATTN_ERR_DEVICE_ARGS for relattn_get_device_error().  Nothing is
 * allocated; the call only enqueues work on `stream`.
 */
typedef struct relattn_prologue_params {
  const void *q;               /* bf16 [total_q, num_heads_q, 128] (pre-norm)          */
  const void *k;               /* bf16 [total_q, num_heads_kv, 128] (pre-conv)         */
  const void *v;               /* bf16 [total_q, num_heads_kv, 128] (pre-conv)         */
  const float *conv_k;         /* fp32 [num_heads_kv * 128, 4]: w[c, d], d = lag       */
  const float *conv_v;         /* fp32 [num_heads_kv * 128, 4]                         */
  const float *norm_q;         /* fp32 [128]                                           */
  const float *norm_k;         /* fp32 [128]                                           */
  float eps;                   /* > 0, e.g. 1e-6                                       */
  const int32_t *cu_seqlens_q; /* device int32 [batch+1]: the chunk's rows             */
  const int32_t *cu_seqlens_k; /* device int32 [batch+1]: cache rows per sequence      */
  int32_t batch;
  int32_t total_q;             /* cu_seqlens_q[batch] (host copy)                      */
  int32_t total_k;             /* cu_seqlens_k[batch] (host copy)                      */
  int32_t num_heads_q;
  int32_t num_heads_kv;
  int32_t head_dim;            /* must be 128                                          */
  void *q_out;                 /* bf16 [total_q, num_heads_q, 128]; may equal q        */
  void *k_cache;               /* bf16 [total_k, num_heads_kv, 128]                    */
  void *v_cache;               /* bf16 [total_k, num_heads_kv, 128]                    */
  const void *conv_state_in_k; /* bf16 [batch, 3, num_heads_kv * 128] or NULL          */
  const void *conv_state_in_v;
  void *conv_state_out_k;      /* bf16 [batch, 3, num_heads_kv * 128] or NULL          */
  void *conv_state_out_v;
} relattn_prologue_params;

relattn_status relattn_prologue(const relattn_prologue_params *params, void *stream);

/*
 * The prologue with the MXFP8 quantise fused in (page "SGLang and Miles Add
 * Day-0 Support for Inkling", section "Relative Logits Optimization",
 * paragraph "MXFP8 Support": the quantisation folded into the attention
 * prologue instead of a separate quantise-and-store step).  Same computation
 * and arguments as relattn_prologue; each k / v cache row it writes is also
 * stored as MXFP8 (the format of relattn_quantize_mxfp8: E4M3 codes and one
 * E8M0 scale per 32 dims) of its bf16-rounded values, so the codes equal
 * relattn_quantize_mxfp8 of the bf16 cache rows.  params->k_cache / v_cache
 * may be NULL (MXFP8 cache only).  cache->k / v: uint8 [total_k,
 * num_heads_kv, 128], 8-byte aligned; cache->k_scale / v_scale: uint8
 * [total_k, num_heads_kv, 4]; none may overlap the k / v inputs.
 */
typedef struct relattn_kv_mxfp8_out {
  void *k;
  void *v;
  void *k_scale;
  void *v_scale;
} relattn_kv_mxfp8_out;

relattn_status relattn_prologue_mxfp8(const relattn_prologue_params *params,
                                      const relattn_kv_mxfp8_out *cache, void *stream);

/* ------------------------------------------------------------------ test hooks
 *
 * Declared only with RELATTN_TEST_HOOKS defined, and exported only by the
 * test build of the library (librelattn_test.so, compiled with that macro).
 * The product library librelattn.so has none of them: its launches run with
 * every hook off.  None has a counterpart on the pages.  Each setting is
 * process-wide (an atomic read by the next launches of the same library);
 * tests set a hook, run one call, and clear it.
 */
#ifdef RELATTN_TEST_HOOKS

/* With tile >= 0, every later launch of the forward tensor-core kernels
 * leaves key tile `tile` (the tile-th 128-key tile a CTA of that kernel
 * visits) unloaded, so the wait of the MMA issuer on it runs out after its
 * bounded limit (about a second): the CTA gives up, drains its own copies and
 * MMAs, frees its tensor memory and exits, and relattn_get_device_error()
 * then returns RELATTN_ERR_TIMEOUT (outputs of affected rows are undefined).
 * tile = -1 restores normal operation; tile < -1 -> RELATTN_ERR_INVALID_ARG. */
relattn_status relattn_test_skip_k_tile(int32_t tile);

/* The bias-band launch of the two-launch prefill, and the walking decode
 * launch, run one CTA per SM, each walking several work items; with n > 0
 * they run at most n CTAs instead, so that small problems also take the
 * paths where a CTA moves from item to item.  Results are unchanged (only
 * the speed).  n = 0 restores the default; n < 0 -> RELATTN_ERR_INVALID_ARG. */
relattn_status relattn_test_band_ctas(int32_t n);

/* Failure path of relattn_prologue.  With tile >= 0 the staged prologue
 * kernel's producer never issues the copies of token tile `tile` (tiles of
 * consecutive chunk tokens, numbered from 0), so the waits of the CTA's
 * consumer warps on that stage run out after their bounded limit (about a
 * second): the CTA drains the copies it did issue and exits, and
 * relattn_get_device_error() then returns RELATTN_ERR_TIMEOUT (outputs of
 * that CTA's later tiles are undefined).  tile = -1 restores normal
 * operation; tile < -1 -> RELATTN_ERR_INVALID_ARG. */
relattn_status relattn_test_prologue_skip_tile(int32_t tile);

/* Failure path of relattn_backward, one tcgen05 kernel at a time.  kernel 0
 * is the dk / dv kernel (its step = one q / dout stage), kernel 1 the dq
 * kernel outside the bias band (its step = one K / V stage).  With step >= 0
 * that kernel's producer never issues the copies of its step `step`, so the
 * waits behind it run out after their bounded limit (about a second per wave
 * of CTAs): each such CTA drains what it issued, frees its tensor memory and
 * exits, and relattn_get_device_error() then returns RELATTN_ERR_TIMEOUT
 * with the first wait site that gave up in bits 8+ of
 * relattn_last_device_error_word() (sites 1-10: dk / dv kernel; 11-16: dq
 * kernel).  The gradients are then undefined.  step = -1 restores normal
 * operation; step < -1 or another kernel -> RELATTN_ERR_INVALID_ARG. */
relattn_status relattn_test_backward_skip_step(int32_t kernel, int32_t step);

#endif /* RELATTN_TEST_HOOKS */

/* Human-readable name of a status code (static string). */
const char *relattn_status_string(relattn_status status);

/* Library version, e.g. "relattn 0.1 sm_103a". */
const char *relattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RELATTN_H */
