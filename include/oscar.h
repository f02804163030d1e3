/*
 * oscar.h -- C ABI of the OSCAR mixed-precision INT2 KV-cache decode library
 * (CUDA, sm_103a).
 *
 * What it implements. OSCAR keeps each request's KV cache as one token pool
 * in three regions, "BF16 sink (64 tokens) | INT2 history | BF16 recent (256
 * tokens)" (news article "超越 TurboQuant，显存压力终于得到缓解！Together AI
 * 最新论文 OSCAR…", section "OSCAR 的设计思路"; MarkTechPost article "Together AI
 * 开源 OSCAR：一种用于长上下文 LLM 服务的注意力感知 2 位 KV 缓存量化系统",
 * section "服务系统：混合精度缓存布局"). History tokens are rotated by
 * R = U H_Had P_br (U from the attention-aware covariances C_Q and C_S,
 * H_Had the Walsh-Hadamard matrix, P_br bit reversal; MarkTechPost article,
 * "OSCAR 有何不同做法"), clipped to per-channel thresholds, quantised to
 * per-token asymmetric INT2 over 64-channel groups and packed 4 codes per
 * byte. Decode attention runs separately over the BF16 and INT2 segments and
 * merges them with an online-softmax (log-sum-exp) merge.
 *
 * Conventions for every call:
 *  - Return value: OSCAR_OK (0) or a negative OSCAR_ERR_* code. Nothing traps
 *    or aborts. Argument errors are detected on the host before any launch.
 *  - Memory: every device buffer is allocated and owned by the caller and
 *    must stay alive until the work enqueued on `stream` has finished. The
 *    library never allocates device memory; it carves the pool and workspace
 *    buffers handed to oscar_cache_create. Host pointers are read before the
 *    call returns.
 *  - Streams: `stream` is a cudaStream_t passed as void*; NULL is the legacy
 *    default stream. All device work of a call is enqueued on that stream, in
 *    order; calls never synchronise except oscar_get_status and
 *    oscar_profile_read.
 *  - Device-side errors (a page id outside the pool, a sequence longer than its
 *    page table allows) set bits in a device status word and the affected
 *    work is skipped; oscar_get_status reports them.
 *  - Threading: a cache handle may be used from one host thread at a time.
 *  - Fixed shape support: head_dim 128, group 64, page_size 64; sink and
 *    recent multiples of page_size; num_q_heads / num_kv_heads in {1,2,4,8}.
 *    Other values return OSCAR_ERR_UNSUPPORTED.
 *
 * Data layouts (all little-endian, row-major, no padding unless stated):
 *  - Per-request page tables are int32 device arrays owned by the caller:
 *      hist_pt [B][max_hist_pages]  INT2 page id of history page i
 *      bf16_pt [B][(sink+recent)/page_size]  BF16 page ids: the sink pages,
 *              then the recent ring pages
 *    Placement of position pos of a request with length L:
 *      pos < sink                        -> bf16_pt[pos / P], row pos % P
 *      pos >= max(sink, L - recent)      -> slot = (pos - sink) % recent,
 *                                           bf16_pt[sink/P + slot/P], row slot % P
 *      otherwise (history)               -> h = pos - sink,
 *                                           hist_pt[h / P], row h % P
 *    Requests may share sink and history pages (prefix caching); recent pages
 *    must be private to one request.
 *  - INT2 page block, one per (page, kv head), 5120 bytes in the default
 *    OSCAR_META_F16 format (the compact OSCAR_META_U8 format is described with
 *    its define below):
 *      [0, 2048)    K codes, row t at 32 t: channel j in byte j/4, bits 2(j%4)
 *      [2048, 4096) V codes, rows (2p, 2p+1) at 2048 + 64 p; channel octet o
 *                   (channels 8o..8o+7) is the 32-bit word at +4 o whose low
 *                   half is row 2p's two packed bytes (2o, 2o+1) and high half
 *                   row 2p+1's
 *      [4096, 4608) K metadata, row t at 4096 + 8 t: fp16 scale0, zero0,
 *                   scale1, zero1 (group g = channels 64g..64g+63)
 *      [4608, 5120) V metadata, same layout
 *    Dequantised value of channel j: zero_g + scale_g * code_j, in the rotated
 *    basis x R.
 *  - BF16 page block, one per (page, kv head), 32768 bytes: K [64][128] bf16
 *    then V [64][128] bf16.
 *  - Per layer, the pool holds the INT2 blocks [num_int2_pages][Hkv], the
 *    BF16 blocks [num_bf16_pages][Hkv] and the rotation parameters; offsets
 *    come from oscar_layer_offsets.
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define OSCAR_OK                 0
#define OSCAR_ERR_INVALID_ARG   (-1)  /* bad pointer, size, index or layout   */
#define OSCAR_ERR_UNSUPPORTED   (-2)  /* valid but not implemented shape      */
#define OSCAR_ERR_CUDA          (-3)  /* a CUDA runtime call failed           */
#define OSCAR_ERR_DEVICE_STATUS (-4)  /* device status word has error bits    */
#define OSCAR_ERR_TIMEOUT       (-5)  /* a bounded device wait gave up        */
#define OSCAR_ERR_NOT_ORTHOGONAL (-6) /* rotation rejected: max|U^T U - I| > 1e-3 */

/* bits of the device status word (oscar_get_status) */
#define OSCAR_STATUS_BAD_PAGE    1    /* a page id outside [0, pages)         */
#define OSCAR_STATUS_BAD_SEQLEN  2    /* seq_len < 1 or beyond its page table */
#define OSCAR_STATUS_TIMEOUT     4    /* a bounded wait expired               */
#define OSCAR_STATUS_NONFINITE   8    /* a NaN or infinity in an input q, k or v row (or in a
                                         rotated row the writers quantise); the row is still
                                         written: NaN and infinities are clipped like any value */
#define OSCAR_STATUS_SATURATED  16    /* an fp16 scale, range or zero of a history group fell
                                         outside +-65504 and was stored saturated (fp16 and
                                         codebook metadata formats; clip thresholds that keep
                                         every group inside +-65504 rule it out) */

/* V handling (MarkTechPost article, "服务系统：混合精度缓存布局": R_V may be
 * absorbed offline into the value/output projections). */
#define OSCAR_V_ABSORBED 0   /* caller's V is already v R_V; output is o R_V  */
#define OSCAR_V_EXPLICIT 1   /* V is raw; write path rotates history V and the
                                merge applies R_V^T to the INT2 partial       */

#define OSCAR_OUT_BF16 0
#define OSCAR_OUT_FP32 1

#define OSCAR_KIND_K 0
#define OSCAR_KIND_V 1

/* decode kernel choice (oscar_set_decode_algo) */
#define OSCAR_DECODE_SIMT 0  /* CUDA-core INT2 decode                          */
#define OSCAR_DECODE_MMA  1  /* tensor-core (mma.sync) INT2 decode             */
#define OSCAR_DECODE_TC   2  /* 5th-generation tensor-core (tcgen05, TMEM) INT2
                                decode: fp16 metadata and up to 4 query heads
                                per kv head; other layouts run OSCAR_DECODE_MMA */

/* INT2 group metadata format (oscar_layout.meta_format). The pages budget the
 * history at 2.25 bits per element (news article "超越 TurboQuant…", section
 * "精度表现": rotation baselines at about 2.25 BPE; 2 bits per code plus 16
 * bits per group of 64) without fixing how the 16 bits are split.
 *  OSCAR_META_F16: per (row, group) an fp16 scale and an fp16 zero (32 bits:
 *    2.5 bits per element, 5120-byte page blocks). The default.
 *  OSCAR_META_U8: per (row, group) two bytes mn8, mx8 (16 bits: 2.25 bits per
 *    element, 4608-byte page blocks): the clipped group's minimum and maximum
 *    rounded down / up to a grid of 255 steps over [-T, T], T the group's
 *    largest clip threshold. With D = fl32(2T / 255) and E = fl32(D / 3),
 *    zero' = fma(mn8, D, -T) and scale' = (mx8 - mn8) * E (float32); codes are
 *    round-to-nearest-even((y - zero') / scale') clamped to [0, 3], 0 where
 *    scale' = 0. Block layout: K codes [0, 2048), V codes [2048, 4096), K
 *    metadata [4096, 4352) at 4 bytes per row (mn8, mx8 of group 0, then of
 *    group 1), V metadata [4352, 4608). */
#define OSCAR_META_F16 0
#define OSCAR_META_U8  1
/* OSCAR_META_CB: the Lloyd-Max codebook variant (news article "超越 TurboQuant…",
 * section "总结与展望": the latest code adds a Lloyd-Max codebook to the
 * attention-aware rotation). The 2-bit code indexes a codebook of 4 levels
 * c_i = k_i / 255 (bytes 0 <= k_0 <= k_1 <= k_2 <= k_3 <= 255, one codebook
 * per (layer, kv head, K / V), set by oscar_set_codebook) on each group's
 * normalised range. Per (row, group) the metadata are fp16 range' =
 * fp16(max - min) and zero' = fp16(min) (RNE, saturating), in the bytes and
 * the 5120-byte block layout of OSCAR_META_F16 (range' in the scale slot).
 * Encoding in float32: t = (y - zero') / range', theta_i = (k_i + k_{i+1}) /
 * 510, code = number of i with t > theta_i (0 where range' = 0). Dequantised
 * value: zero' + range' * k_code / 255. (0, 85, 170, 255) gives the uniform
 * levels. */
#define OSCAR_META_CB  2

typedef struct oscar_layout {
  int num_layers;      /* >= 1                                                */
  int num_kv_heads;    /* Hkv >= 1                                            */
  int num_q_heads;     /* Hq, a multiple of Hkv, Hq/Hkv in {1,2,4,8}          */
  int head_dim;        /* 128                                                 */
  int group;           /* channels per quantisation group, 64                 */
  int page_size;       /* tokens per page, 64                                 */
  int sink;            /* S0, BF16 sink tokens, multiple of page_size (64)    */
  int recent;          /* W, BF16 recent ring, multiple of page_size (256)    */
  int num_int2_pages;  /* INT2 page capacity per layer                        */
  int num_bf16_pages;  /* BF16 page capacity per layer                        */
  int v_mode;          /* OSCAR_V_ABSORBED or OSCAR_V_EXPLICIT                */
  int max_batch;       /* largest B any call will pass                        */
  int max_splits;      /* largest number of history splits per (request, kv head) */
  int meta_format;     /* OSCAR_META_F16 (0) or OSCAR_META_U8 (1), see below   */
} oscar_layout;

typedef struct oscar_cache oscar_cache;

/* Bytes the caller must allocate (device memory, 256-byte aligned) for the
 * pool and the workspace of a layout. Either output pointer may be NULL. */
int oscar_cache_bytes(const oscar_layout* layout, size_t* pool_bytes, size_t* workspace_bytes);

/* Validate `layout` and bind the caller's pool and workspace (device
 * pointers, 256-byte aligned, sizes from oscar_cache_bytes). Allocates only the
 * host-side handle. The pool is not cleared. Errors: INVALID_ARG,
 * UNSUPPORTED, CUDA (device query failed). */
int oscar_cache_create(const oscar_layout* layout, void* pool, void* workspace, oscar_cache** out);

/* Free the host-side handle (not the caller's device buffers). NULL is a no-op. */
int oscar_cache_destroy(oscar_cache* cache);

/* Byte offsets, inside the pool buffer, of a layer's INT2 blocks, BF16 blocks
 * and rotation parameters. */
int oscar_layer_offsets(const oscar_cache* cache, int layer, size_t* int2_off, size_t* bf16_off,
                        size_t* params_off);

/* Load a layer's rotation and clip parameters (MarkTechPost article, "OSCAR
 * 有何不同做法": R_K = U_Q H_Had P_br, R_V = U_S H_Had P_br; "服务系统：混合精度
 * 缓存布局": clipping to calibration-derived percentile thresholds).
 *  U_K, U_V : host float32 [Hkv][128][128], row-major; column c is the c-th
 *             eigenvector (descending eigenvalue). R = U H P_br is applied as
 *             x -> x R to row vectors; H and P_br are never stored.
 *  tau_K, tau_V : host float32 [Hkv][128], clip thresholds in the rotated basis.
 *  U_V may be NULL in V-absorbed mode (then it is not used).
 * Each U is checked on the host: max|U^T U - I| > 1e-3 returns
 * OSCAR_ERR_NOT_ORTHOGONAL and nothing is copied. The copy is enqueued on
 * `stream`. */
int oscar_set_rotation(oscar_cache* cache, int layer, const float* U_K, const float* U_V,
                       const float* tau_K, const float* tau_V, void* stream);

/* Load a layer's codebooks (OSCAR_META_CB layouts; see OSCAR_META_CB).
 *  cb_K, cb_V : host uint8 [Hkv][4], each codebook non-decreasing.
 * oscar_set_rotation resets both to the uniform (0, 85, 170, 255), so call this
 * after it. Errors: INVALID_ARG (null pointer, bad layer, a decreasing
 * codebook), UNSUPPORTED (the layout is not OSCAR_META_CB), CUDA. The copy is
 * enqueued on `stream`. */
int oscar_set_codebook(oscar_cache* cache, int layer, const uint8_t* cb_K, const uint8_t* cb_V, void* stream);

/* Lloyd-Max calibration of one codebook on the host (news article "超越
 * TurboQuant…", section "总结与展望"): from rotated float32 calibration rows
 * x_rot [N][128] (host), clipped to tau [128], every 64-channel group with
 * max > min contributes its values normalised to u = (y - min) / (max - min).
 * Lloyd's iteration from the levels (0, 1/3, 2/3, 1): thresholds at the
 * midpoints, each level the mean of its cell (u <= t_0, t_0 < u <= t_1, ...;
 * an empty cell keeps its level), until no level moves by more than 1e-12 or
 * 1000 iterations; then cb[i] = rint(255 level_i) clamped and sorted.
 * Errors: INVALID_ARG (null pointer, N < 1). */
int oscar_calibrate_codebook(const float* x_rot, int N, const float* tau, uint8_t* cb);

/* Bulk write of B requests' prompt tokens (MarkTechPost article, "服务系统：
 * 混合精度缓存布局", write path: rotate, clip, quantise, pack).
 *  k, v        : device bf16 [total_tokens][Hkv][128], requests concatenated
 *  cu_seqlens  : device int32 [B+1], cu_seqlens[0] = 0, cu_seqlens[B] = total_tokens
 *  total_tokens: host copy of cu_seqlens[B]
 * Request r's token i sits at position i; its final length is
 * L_r = cu_seqlens[r+1] - cu_seqlens[r], which decides sink / history / recent
 * placement as above. In V-absorbed mode V is quantised without rotation. */
int oscar_quantize_prefill(oscar_cache* cache, int layer, int B, const void* k, const void* v,
                           const int32_t* cu_seqlens, int total_tokens, const int32_t* hist_pt,
                           int max_hist_pages, const int32_t* bf16_pt, void* stream);

/* The same bulk write from the prompt's hidden states, fused with the K and V
 * projections (MarkTechPost article, "服务系统：混合精度缓存布局": the write path
 * runs fused, so K and V are never written out and read back):
 *   K = bf16(x W_k^T), V = bf16(x W_v^T), rounded to nearest even,
 * then placed and quantised exactly as oscar_quantize_prefill does with those K
 * and V.
 *  x        : device bf16 [total_tokens][d_model], requests concatenated as in
 *             cu_seqlens (row-major, 16-byte aligned)
 *  w_k, w_v : device bf16 [Hkv * 128][d_model] (a linear layer's weight: output
 *             row j is kv head j / 128, channel j % 128), 16-byte aligned
 *  d_model  : a multiple of 64
 * The products accumulate in float32 on the tensor cores, then round to bf16.
 * Errors: INVALID_ARG (as oscar_quantize_prefill, d_model <= 0, a pointer not
 * 16-byte aligned), UNSUPPORTED (d_model not a multiple of 64, an odd Hkv,
 * B > 4096), CUDA. */
int oscar_project_quantize_prefill(oscar_cache* cache, int layer, int B, const void* x, int d_model,
                                   const void* w_k, const void* w_v, const int32_t* cu_seqlens,
                                   int total_tokens, const int32_t* hist_pt, int max_hist_pages,
                                   const int32_t* bf16_pt, void* stream);

/* Append one token per request at position seq_lens_before[r] (news article,
 * "OSCAR 的设计思路": a new token enters the recent window; the oldest recent
 * token is rotated / clipped / quantised / packed into the INT2 history).
 *  k, v            : device bf16 [B][Hkv][128]
 *  seq_lens_before : device int32 [B], lengths before this token
 * If seq_lens_before[r] >= sink + recent, the token at position
 * seq_lens_before[r] - recent is demoted to history slot
 * seq_lens_before[r] - recent - sink before its ring slot is overwritten.
 * As in oscar_decode_step, seq_lens_before, the page tables and the pool's
 * rows are read before the wait for the kernel launched just before; only
 * k and v may come from that kernel. */
int oscar_append_kv(oscar_cache* cache, int layer, int B, const void* k, const void* v,
                    const int32_t* seq_lens_before, const int32_t* hist_pt, int max_hist_pages,
                    const int32_t* bf16_pt, void* stream);

/* Decode attention for one query token per request (news article, "OSCAR 的设计
 * 思路": BF16 segment and INT2 segment computed separately, combined by an
 * online-softmax merge).
 *  q        : device bf16 [B][Hq][128], 16-byte aligned; query head i reads kv head i/(Hq/Hkv)
 *  seq_lens : device int32 [B], lengths including the current token (>= 1)
 *  sm_scale : softmax scale (1/sqrt(128) for standard attention)
 *  out      : device [B][Hq][128], bf16 or fp32 per out_dtype. In V-absorbed
 *             mode the output is in the rotated value basis (o R_V).
 *  lse      : device float32 [B][Hq] natural-log sum of exp(sm_scale q.k), or NULL
 * History logits use the rotated query q R_K against the dequantised keys,
 * equal to attending with inverse-rotated keys because R_K is orthogonal. */
int oscar_decode_attention(oscar_cache* cache, int layer, int B, const void* q, const int32_t* seq_lens,
                           const int32_t* hist_pt, int max_hist_pages, const int32_t* bf16_pt,
                           float sm_scale, void* out, int out_dtype, float* lse, void* stream);

/* One decode step of a layer: oscar_append_kv(k, v at position
 * seq_lens_before[r]) followed by oscar_decode_attention(q) over
 * seq_lens_before[r] + 1 tokens, with the same arguments, layouts and
 * results as those two calls, issued as one chain of three launches, each a
 * programmatic dependent of the one before it: one step prologue (per
 * request, kv head and K / V: the demoted row, and for K the query rows, are
 * rotated together on the tensor cores; the demoted row is quantised into
 * the history, the queries become the decode's fragments, the new token goes
 * to its ring slot), the decode kernel and the merge. The decode kernel
 * prefetches history pages the append cannot touch before it waits.
 * Ordering: only q, k and v may be produced by the kernel launched just
 * before this call. The prologue is a programmatic dependent of that kernel:
 * it reads seq_lens_before, the page tables and the pool's BF16 rows before
 * it waits for it. These inputs must be complete when that kernel starts
 * (host copies, or any earlier kernel). No kernel of this library writes
 * them early. */
int oscar_decode_step(oscar_cache* cache, int layer, int B, const void* q, const void* k, const void* v,
                      const int32_t* seq_lens_before, const int32_t* hist_pt, int max_hist_pages,
                      const int32_t* bf16_pt, float sm_scale, void* out, int out_dtype, float* lse, void* stream);

/* Shared-prefix variants (MarkTechPost article "Together AI 开源 OSCAR…",
 * section "服务系统：混合精度缓存布局": the pool stays compatible with paged
 * KV and prefix caching). The caller states that history pages
 * [0, shared_hist_pages) of every request are the same pages: the entries
 * hist_pt[r][0 .. shared_hist_pages) are equal for all r, and every request
 * holds at least that many history pages. The result is the same as the
 * call without the suffix.
 *
 * On the tensor-core path one extra kernel then reads each shared page once
 * per step for all B x Hq / Hkv queries of its kv head, in CTAs of 128 query
 * rows. Each page is expanded once into shared memory and both products run
 * as 128-row tensor-core tiles. The per-request kernel covers only each
 * request's own pages. The CUDA-core path ignores shared_hist_pages.
 *
 * With oscar_decode_step_shared, the token each step demotes must land in
 * the request's own pages, so every request's history must already extend
 * past the shared pages. Error behaviour is as in the plain calls, and
 * 0 <= shared_hist_pages <= max_hist_pages is checked on the host. */
int oscar_decode_attention_shared(oscar_cache* cache, int layer, int B, const void* q, const int32_t* seq_lens,
                                  const int32_t* hist_pt, int max_hist_pages, int shared_hist_pages,
                                  const int32_t* bf16_pt, float sm_scale, void* out, int out_dtype, float* lse,
                                  void* stream);
int oscar_decode_step_shared(oscar_cache* cache, int layer, int B, const void* q, const void* k, const void* v,
                             const int32_t* seq_lens_before, const int32_t* hist_pt, int max_hist_pages,
                             int shared_hist_pages, const int32_t* bf16_pt, float sm_scale, void* out, int out_dtype,
                             float* lse, void* stream);

/* Choose the INT2 decode kernel (OSCAR_DECODE_MMA by default). */
int oscar_set_decode_algo(oscar_cache* cache, int algo);

/* Synchronise the device, return the device status word in *code and clear
 * it. Returns OSCAR_ERR_DEVICE_STATUS when *code != 0. */
int oscar_get_status(oscar_cache* cache, int* code);

/* ---- test and debug entry points ----------------------------------------- */

/* Clip, quantise and pack pre-rotated float32 values into history rows,
 * skipping the rotation (for bit-exact checks of the quantiser and packing).
 *  kind   : OSCAR_KIND_K or OSCAR_KIND_V (writes that half of the row)
 *  xrot   : device float32 [N][Hkv][128], already in the rotated basis
 *  page_ids, rows : device int32 [N], INT2 page id and row (0..63) per token */
int oscar_pack_rotated(oscar_cache* cache, int layer, int kind, const float* xrot, const int32_t* page_ids,
                       const int32_t* rows, int N, void* stream);

/* y = x R (kind K: R_K, kind V: R_V) as the write path computes it.
 *  x : device bf16 [N][Hkv][128];  y : device float32 [N][Hkv][128] */
int oscar_rotate(oscar_cache* cache, int layer, int kind, const void* x, float* y, int N, void* stream);

/* ---- BF16 comparison kernel ---------------------------------------------- */

/* Workspace bytes of oscar_bf16_decode. */
int oscar_bf16_decode_workspace_bytes(int max_batch, int num_q_heads, int max_splits, size_t* bytes);

/* Decode attention over a plain all-BF16 paged cache, the baseline OSCAR's
 * speedups are measured against.
 *  kv_pages   : device bf16 [num_pages][Hkv][2][64][128] (K block then V block)
 *  page_table : device int32 [B][max_pages]; position pos -> page_table[pos/64], row pos%64
 *  workspace  : device, oscar_bf16_decode_workspace_bytes(B or more, Hq, max_splits) */
int oscar_bf16_decode(int B, int num_q_heads, int num_kv_heads, const void* kv_pages, int num_pages,
                      const void* q, const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                      float sm_scale, void* out, int out_dtype, float* lse, void* workspace,
                      size_t workspace_bytes, int max_splits, void* stream);

/* ---- offline calibration (host) ------------------------------------------ */

/* Offline calibration of one (layer, kv head) on the host (MarkTechPost
 * article, "OSCAR 有何不同做法"; visual guide step 2):
 *   C_Q = (1/N) sum_n q_n^T q_n over the N calibration queries,
 *   C_S = (1/N) V^T S^T S V with S = row-softmax(sm_scale Q K^T) (no mask),
 *   U_K, U_V = eigenvectors of C_Q, C_S (columns, descending eigenvalue,
 *   each column's largest-magnitude entry positive),
 *   tau_K[j] = c_K-quantile of |K R_K|[:, j], tau_V[j] = c_V-quantile of
 *   |V R_V|[:, j] (linear interpolation between order statistics).
 *  Q, K, V : host float32 [N][128]; outputs host float32 U [128][128], tau [128].
 *  eig_K, eig_V : optional host float64 [128] eigenvalue outputs (may be NULL). */
int oscar_calibrate(const float* Q, const float* K, const float* V, int N, float sm_scale, float c_K,
                    float c_V, float* U_K, float* U_V, float* tau_K, float* tau_V, double* eig_K,
                    double* eig_V);

/* ---- tracing ------------------------------------------------------------- */

/* Start tracing decode calls: while enabled, every oscar_decode_attention and
 * oscar_decode_step records a CUDA event pair on its stream around its
 * history kernel (the fused tensor-core decode kernel, or the CUDA-core
 * history kernel), the dominant launch of the call; at most `capacity` calls
 * are kept. The events separate that kernel from the programmatic overlap
 * with its neighbours, so it is timed alone. Event records can be captured
 * into a CUDA graph; the graph then re-records the same events on every
 * replay. */
int oscar_profile_begin(oscar_cache* cache, int capacity);

/* Stop, synchronise and report the summed device time (ms) of the traced
 * calls and their count. */
int oscar_profile_read(oscar_cache* cache, double* total_ms, int* launches);

/* ---- allocation-free decode ---------------------------------------------- */

#define OSCAR_ERR_TOO_LARGE (-7)  /* the call needs more than the fixed device scratch */

/* Decode attention that allocates nothing. The paper has no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc, such as serving
 * engines whose allocator already owns all device memory and forbids side
 * allocations, and hosts that may not allocate on a latency-critical path
 * (cudaMalloc can synchronise the device and take milliseconds).
 *
 * It computes exactly what oscar_decode_attention computes, with the same
 * arguments, except:
 *  - the cache is given by its layout and pool instead of a handle: `pool` is
 *    the device buffer a cache with this `layout` was created on (rotation and
 *    tokens already written through the other entry points);
 *  - no workspace is used: the scratch (status word, rotated queries, split
 *    partials) lives in a 4 MiB static device array inside the library, which
 *    every GPU that loads the library holds until the process exits;
 *  - this call's device status bits are copied to `status` (device int32,
 *    may be NULL) at the end of the call.
 * The call performs no cudaMalloc, cudaFree or other allocating call.
 * Set-up: the first call on a device resolves the array's address for that
 * device (cudaGetSymbolAddress) and configures the kernels. Every call shares the array and it keeps the
 * last call's contents (the status word is cleared at the start of each
 * call): calls that may overlap on the GPU (different streams, or threads
 * without ordering) race and give wrong results; calls ordered on one stream
 * are safe. The history is split into fewer pieces when needed to fit. A call
 * whose per-query state does not fit even with one history split, i.e. when
 * B * Hq * (560 + 528 * (1 + (sink + recent) / 64)) + B * Hkv * 4096 bytes plus
 * about 1.3 KB of rounding exceed 4 MiB (B * Hq above about 880 with the
 * default windows and Hq / Hkv = 4), returns OSCAR_ERR_TOO_LARGE before any
 * device work. */
int oscar_decode_attention_noalloc(const oscar_layout* layout, void* pool, int layer, int B, const void* q,
                                   const int32_t* seq_lens, const int32_t* hist_pt, int max_hist_pages,
                                   const int32_t* bf16_pt, float sm_scale, void* out, int out_dtype, float* lse,
                                   int* status, void* stream);

/* Record a timeline of the CTAs of every following tensor-core decode launch
 * (each launch overwrites it): for CTA i (linear block index) the eight
 * uint64 values at buf[8 i] are its id, SM id, start time, time its first
 * history page landed, time its last warp finished the main loop, time its
 * partials were written, 0, and the time its wait for the kernel before it
 * returned (history CTAs); times are %globaltimer nanoseconds.
 * buf: device memory for `capacity` records (64 bytes each); NULL stops
 * recording. CTAs beyond `capacity` are not recorded. */
int oscar_trace_ctas(oscar_cache* cache, void* buf, int capacity);

/* Record a timeline of every CTA of the following launches of this cache's
 * kernels (append, prefill, query prologue, decode, merge), accumulating
 * across launches until the buffer is full. buf: device uint64
 * [4 + 4 * capacity]; the caller zeroes buf[0], which counts the records
 * claimed (it may exceed `capacity`; the excess is not written). Record i is
 * buf[4 + 4 i .. 4 + 4 i + 3] = {kind | layer << 8 | SM << 24 | linear CTA
 * index << 32, start, end, mark}, times in %globaltimer nanoseconds, taken by
 * thread 0 on entry and when it leaves the kernel; mark is, for the merge, the
 * time its wait for the decode kernel returned and, for the step prologue,
 * the time its rotation was done, else 0. Kinds: 1 step prologue
 * with an append (oscar_append_kv, or append + query prologue in
 * oscar_decode_step), 2 query prologue alone (oscar_decode_attention),
 * 3 tensor-core decode, 4 merge, 5 CUDA-core history decode, 6 BF16 segment,
 * 7 prefill. Launches issued while a buffer is set keep
 * writing to it, also from CUDA graphs captured meanwhile; NULL stops
 * recording for later launches. */
int oscar_trace_timeline(oscar_cache* cache, void* buf, int capacity);

/* Failure-detection self-check: launches one warp that waits on a device
 * barrier nothing completes. Like every wait in the library it gives up after
 * 2 seconds of %globaltimer time and sets OSCAR_STATUS_TIMEOUT in the status
 * word (read with oscar_get_status). Nothing faults and nothing stays pending;
 * the cache remains usable. */
int oscar_check_wait_timeout(oscar_cache* cache, void* stream);

/* Human-readable name of a status code. */
const char* oscar_error_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* OSCAR_H */
