/*
 * gqaq.h -- C ABI of the GB300 (sm_103a) decode-attention library:
 * GQA attention with the query heads folded onto their KV heads, and Quest
 * query-aware page sparsity on top of it.
 *
 * Sources (page title + section):
 *  [OPT]   "Core ML Decode Optimization: Removing the 1.9 GiB Per-Token Copy
 *          Caused by GQA repeat_kv" (OptAI engineering blog). Section 3, "Fold
 *          Q Instead of Expanding KV" (the [B,Hq,1,D] -> [B,Hkv,G,D] reshape,
 *          h = G*kv + g, the decode code with scale, additive mask, softmax over
 *          the context axis and prob @ V). Section 5, "Query Heads Must Be
 *          Ordered by KV Group" (the contiguous-group precondition).
 *  [QUEST] "Quest: Query-Aware Sparsity for Efficient Long-Context LLM
 *          Inference" (reviewer's summary). The flowchart (score pages from
 *          min/max metadata, pick the top pages, read only their K and V,
 *          attend). The page-score section: m_{p,i} and M_{p,i} are kept per
 *          page and channel and updated when a key arrives, and
 *          U(p,q) = sum_i max(q_i m_{p,i}, q_i M_{p,i}). The token-budget section
 *          (B = K*S). The note that the first two layers stay dense.
 *
 * Conventions for every entry point
 *  - Tensors are dense row-major fp16 (IEEE binary16, passed as gqaq_half
 *    bits), int32 or fp32. Every pointer is a DEVICE pointer on the current
 *    CUDA device, 16-byte aligned, except `dims` (host).
 *  - The caller owns every buffer: caches, metadata, outputs and workspace.
 *    The library never allocates device memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream). They can be captured in a CUDA graph after one eager
 *    call on the device, because that first call loads the kernels. The
 *    return value reports host-side validation and launch errors only.
 *  - Layouts (B = batch, Hq/Hkv query/KV heads, G = Hq/Hkv, D = head_dim,
 *    Lmax = max_len, S = page_size, Pmax = ceil(Lmax/S)):
 *      q, out           [B][Hq][D]     fp16 (query heads grouped: h = G*kv + g)
 *      k_cache, v_cache [B][Hkv][Lmax][D] fp16 (one page = S consecutive rows)
 *      meta             [B][Hkv][Pmax][2][D] fp16 (page minimum row, then maximum)
 *      scores           [B][Hkv][Pmax] fp32
 *      page_idx         [B][Hkv][k] int32 (ascending, -1 padded)
 *      valid_len, pos   [B] int32
 *  - Supported: D in {64, 128}; G in {1, 2, 4, 8}; S in {8, 16, 32, 64} for the
 *    Quest calls (the Quest review's page-size trade-off);
 *    B*Hkv*Lmax < 2^31. Other shapes return GQAQ_ERR_UNSUPPORTED.
 *  - Values that live on the device are checked there. This covers valid_len
 *    outside [1, Lmax], page indices outside [0, ceil(valid_len/S)) and pos
 *    outside [0, Lmax). The kernels clamp or skip such values and raise a flag
 *    in the device status word (gqaq_device_status). They never read or write
 *    outside the buffers described here.
 *  - Every wait inside a kernel is bounded (GQAQ_OPT_WAIT_TIMEOUT_NS). On
 *    timeout the kernel sets GQAQ_DEV_TIMEOUT, lets its own copies in flight
 *    land and returns. It never traps.
 */
#ifndef GQAQ_H
#define GQAQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GQAQ_API __attribute__((visibility("default")))
#else
#define GQAQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gqaq_half; /* IEEE-754 binary16 bit pattern */

typedef enum {
    GQAQ_OK = 0,
    GQAQ_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad dims, k < 1, ... */
    GQAQ_ERR_UNSUPPORTED = 2, /* valid but not implemented (D, G, S, size limits) */
    GQAQ_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    GQAQ_ERR_CUDA = 4,        /* a CUDA runtime call or a launch failed */
    GQAQ_ERR_TIMEOUT = 5      /* reported by gqaq_device_status only */
} gqaq_status;

/* Device status word flags (bitwise OR), read with gqaq_device_status. */
enum {
    GQAQ_DEV_TIMEOUT = 1,  /* a bounded wait gave up */
    GQAQ_DEV_BAD_LEN = 2,  /* a valid_len outside [1, Lmax] was clamped */
    GQAQ_DEV_BAD_PAGE = 4, /* a page index outside [0, P) was skipped */
    GQAQ_DEV_BAD_POS = 8   /* an append position outside [0, Lmax) was skipped */
};

typedef struct {
    int batch;        /* B >= 1 */
    int num_q_heads;  /* Hq >= 1, a multiple of Hkv */
    int num_kv_heads; /* Hkv >= 1 */
    int head_dim;     /* D: 64 or 128 */
    int max_len;      /* Lmax >= 1: allocated rows per (sequence, KV head) */
    int page_size;    /* S: 8, 16, 32 or 64 (Quest calls); ignored by gqa_decode_attn */
} gqaq_dims;

/* Bytes of workspace that gqa_decode_attn and quest_sparse_attn need on the
 * current device for these dims (enough for both). The library sizes its
 * grid from the SM count, so the figure depends on the device.
 * With max_selected_pages = k > 0 (and a supported S) the figure also covers
 * quest_decode_attn's work-queue kernel for that k.
 * Returns 0 when the dims are invalid or unsupported.
 * The workspace starts with counters and flags (a ticket word, three words
 * per (sequence, KV head)) followed by scratch (fp32 partials, page keys and
 * lists). The counters must be zero when the workspace is first used:
 * zero-fill it once (cudaMemsetAsync) after allocating it. Every call leaves
 * them at zero again, so the workspace can be reused by any later call (of
 * any dims that fit) without clearing; gqa_decode_attn and quest_sparse_attn
 * do so even when their waits time out. */
GQAQ_API size_t gqaq_workspace_bytes(const gqaq_dims *dims, int max_selected_pages);

/* [OPT] section 3: dense decode attention with the query heads folded.
 * For every sequence b, KV head kv and group member g (h = G*kv + g):
 *   out[b][h] = sum_{t < valid_len[b]} softmax_t(scale * q[b][h] . k[b][kv][t]) v[b][kv][t].
 * Each KV head's K and V rows are read from HBM once for its G query rows.
 * No repeat_kv copy is ever made. The valid-length prefix stands in for the
 * additive context mask. fp32 accumulation; out is rounded to fp16 once
 * (round to nearest even). The context is split across the GPU's SMs, and
 * the split partials are combined by log-sum-exp.
 * The CTA that finishes a split (sequence, KV head) last merges its partials,
 * so one kernel launch does the whole call.
 * workspace: >= gqaq_workspace_bytes(dims, 0) bytes of device memory, zero
 * filled before its first use (see gqaq_workspace_bytes). Two calls that
 * overlap on the GPU must not share it. */
GQAQ_API int gqa_decode_attn(const gqaq_dims *dims, const gqaq_half *q, const gqaq_half *k_cache,
                    const gqaq_half *v_cache, const int32_t *valid_len, float scale,
                    gqaq_half *out, void *workspace, size_t workspace_bytes, void *stream);

/* [QUEST] page-score section: append one token per (sequence, KV head) and
 * update its page's metadata. Writes k_new[b][kv] / v_new[b][kv] ([B][Hkv][D])
 * to row pos[b] of the caches. For page p = pos[b] / S: if pos[b] % S == 0 the
 * page's min and max rows become k_new, otherwise they become the elementwise
 * min / max of their old value and k_new. Appending rows in order keeps the
 * exact page bounds. */
GQAQ_API int quest_append_kv(const gqaq_dims *dims, gqaq_half *k_cache, gqaq_half *v_cache,
                    gqaq_half *meta, const gqaq_half *k_new, const gqaq_half *v_new,
                    const int32_t *pos, void *stream);

/* [QUEST] page-score section: build the metadata from the cache. For each page
 * p in [page_begin, page_end) that holds a valid token, meta[b][kv][p] =
 * elementwise (min, max) over rows [p*S, min(p*S+S, valid_len[b])) of
 * k_cache[b][kv]. Pages with no valid token are left untouched.
 * Requires 0 <= page_begin <= page_end <= Pmax. */
GQAQ_API int quest_update_meta(const gqaq_dims *dims, const gqaq_half *k_cache, const int32_t *valid_len,
                      gqaq_half *meta, int page_begin, int page_end, void *stream);

/* [QUEST] page-score section: for every valid page p < ceil(valid_len[b]/S),
 *   scores[b][kv][p] = max_g sum_i max(q[b][G*kv+g][i] * m_{p,i}, q[b][G*kv+g][i] * M_{p,i}),
 * i.e. U(p,q), maximised over the KV head's G folded query rows. q is unscaled.
 * The page ranking is the same under any positive scale. Entries for pages
 * at or beyond P are not written. fp32 (every product of two fp16 values is
 * exact in fp32; the sums are rounded). */
GQAQ_API int quest_score_pages(const gqaq_dims *dims, const gqaq_half *q, const gqaq_half *meta,
                      const int32_t *valid_len, float *scores, void *stream);

/* [QUEST] token-budget section: per (b, kv), select the k pages with the
 * largest score among the P = ceil(valid_len[b]/S) valid pages. Equal scores go
 * to the lower page index. If P <= k, every page is selected. The selection
 * is written to page_idx[b][kv][0..k) in ascending page order, padded with -1.
 * Requires 1 <= k <= 65536 and Pmax <= 32768. workspace / workspace_bytes are
 * reserved (may be NULL / 0). */
GQAQ_API int quest_topk_pages(const gqaq_dims *dims, const float *scores, const int32_t *valid_len,
                     int k, int32_t *page_idx, void *workspace, size_t workspace_bytes,
                     void *stream);

/* [QUEST] flowchart, last two steps: attention over only the selected pages.
 * It is the same as gqa_decode_attn, except that sequence b / KV head kv
 * attends only to the tokens of pages page_idx[b][kv][j], for
 * j < min(k, ceil(valid_len[b]/S)). Page p contributes its rows
 * [p*S, min(p*S+S, valid_len[b])). Negative or out-of-range entries are
 * skipped. Indices must be distinct. workspace: as for gqa_decode_attn. */
GQAQ_API int quest_sparse_attn(const gqaq_dims *dims, const gqaq_half *q, const gqaq_half *k_cache,
                      const gqaq_half *v_cache, const int32_t *valid_len, const int32_t *page_idx,
                      int k, float scale, gqaq_half *out, void *workspace, size_t workspace_bytes,
                      void *stream);

/* Fused Quest decode step, one launch per layer. It does, in order, what
 * quest_append_kv, quest_score_pages, quest_topk_pages and quest_sparse_attn
 * do: when pos is not NULL, append k_new/v_new at row pos[b] and update that
 * page's min/max; score every valid page; select the k best pages (ties to
 * the lower index); attend over only their tokens ([QUEST] flowchart).
 * scores ([B][Hkv][Pmax] fp32) and page_idx ([B][Hkv][k] int32, ascending,
 * -1 padded) are optional outputs (NULL to skip). 1 <= k <= 65536.
 * With a workspace (>= gqaq_workspace_bytes(dims, k) bytes, zero-filled
 * before its first use, see gqaq_workspace_bytes) the step can run as one
 * work queue over the whole GPU: page-scoring and attention pieces of every
 * (sequence, KV head) are taken from a ticket counter; the last scorer of a
 * (sequence, KV head) selects its pages, the last attention piece merges its
 * softmax states. That covers Pmax <= 8192 pages. The other kernel hands one
 * (sequence, KV head) at a time to one thread-block cluster, whose CTAs meet
 * in distributed shared memory; it needs no workspace and requires k <= 1024.
 * By default (GQAQ_OPT_QUEST_KERNEL) the cluster kernel runs whenever
 * k <= 1024, and the work queue above that (GQAQ_ERR_WORKSPACE without a
 * workspace). Two calls that overlap on the GPU must not share a workspace.
 * After a call whose waits timed out (GQAQ_DEV_TIMEOUT), zero the workspace
 * again before reusing it. */
GQAQ_API int quest_decode_attn(const gqaq_dims *dims, const gqaq_half *q, gqaq_half *k_cache,
                               gqaq_half *v_cache, gqaq_half *meta, const gqaq_half *k_new,
                               const gqaq_half *v_new, const int32_t *pos, const int32_t *valid_len,
                               int k, float scale, gqaq_half *out, float *scores, int32_t *page_idx,
                               void *workspace, size_t workspace_bytes, void *stream);

/* gqa_decode_attn for callers that cannot allocate device memory. The source
 * pages have no counterpart to this call. A plugin or custom operator inside a
 * host framework is often handed only its input and output pointers: the
 * framework owns all device memory and forbids allocation while it runs. A
 * latency-critical decode loop may also refuse cudaMalloc/cudaFree, which can
 * synchronise the device. Such callers cannot supply gqa_decode_attn's
 * workspace, so this variant keeps its split-context scratch in a fixed 1 MiB
 * array inside the library's device memory. Every GPU that loads the library
 * holds that array until the process exits.
 * Arguments, layouts and results are those of gqa_decode_attn, without the
 * workspace. Returns GQAQ_ERR_WORKSPACE, launching nothing, when the shape needs
 * more scratch than 1 MiB: the split partials of gqa_decode_attn's grid for
 * this shape (at most one CTA per four 128-token tiles) plus its counters. At
 * G = 8 and D = 128 (8,320 bytes per CTA) that happens from about 500 tiles
 * of (sequence, KV head, 128 tokens) on a 152-SM GB300.
 * The first call on each device looks up the array's device address with that
 * device current and keeps it for the life of the process. Make that first
 * call before any stream capture, and do not use the library on a device
 * after cudaDeviceReset.
 * All calls share the one array. It is zero-filled when the library loads,
 * as the workspace contract asks, and every call leaves it so. Calls that
 * overlap on the GPU race on it. It allocates nothing. */
GQAQ_API int gqa_decode_attn_noalloc(const gqaq_dims *dims, const gqaq_half *q, const gqaq_half *k_cache,
                                     const gqaq_half *v_cache, const int32_t *valid_len, float scale,
                                     gqaq_half *out, void *stream);

/* Low-bit KV caches. The pages define no low-bit KV format: [OPT] section 5
 * ("KV Cache Update Operations Remain") names the cache-write path as the next
 * target, and [QUEST]'s section on its 7.03x kernel and 2.23x decode figures
 * states that its 4-bit condition is weight quantization, not a 4-bit KV
 * store. The two formats below are this library's own plainest choices.
 *
 * The 8-bit KV-cache variant. k_cache / v_cache are [B][Hkv][Lmax][D] bytes of
 * E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, largest finite 448) with one fp32 scale per tensor: a key
 * channel's value is k_scale * value(code), likewise for values.
 *
 * gqa_decode_attn over such a cache: [OPT] section 3's folded dense attention
 * with the keys and values dequantized on load (exactly, to fp16, then fp32
 * accumulation). Same arguments, layouts, workspace (and its zero-fill rule)
 * and results as gqa_decode_attn otherwise. D in {64, 128}. */
GQAQ_API int gqa_decode_attn_e4m3(const gqaq_dims *dims, const gqaq_half *q, const uint8_t *k_cache,
                                  const uint8_t *v_cache, float k_scale, float v_scale,
                                  const int32_t *valid_len, float scale, gqaq_half *out, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Append one token per (sequence, KV head) to an E4M3 cache: row pos[b] of
 * k_cache[b][kv] becomes the codes of k_new[b][kv] ([B][Hkv][D] fp16), each
 * RNE-satfinite(fp32(k) * k_inv_scale): the nearest E4M3 value, ties to the
 * even code, magnitudes beyond 448 saturated; likewise v with v_inv_scale.
 * pos[b] outside [0, Lmax) is skipped and raises GQAQ_DEV_BAD_POS. */
GQAQ_API int kv_append_e4m3(const gqaq_dims *dims, uint8_t *k_cache, uint8_t *v_cache, const gqaq_half *k_new,
                            const gqaq_half *v_new, const int32_t *pos, float k_inv_scale, float v_inv_scale,
                            void *stream);

/* Quest over an E4M3 cache: the page-score section's metadata and score, and
 * the flowchart's attention over the selected pages, with the 8-bit format
 * above. meta is [B][Hkv][Pmax][2][D] bytes: per page the E4M3 codes of each
 * channel's smallest, then largest key value (compared after decoding; a
 * zero bound is stored as the code 0x00, so each bound has one code; the
 * dequantized bounds are k_scale * value(code)). The cache holds no NaN
 * codes. 2*D bytes per page, half the fp16 metadata.
 *
 * quest_append_kv_e4m3: kv_append_e4m3's codes for row pos[b], then the
 * page's bounds as quest_append_kv keeps them (a token starting a page
 * replaces them). pos[b] outside [0, Lmax) is skipped and raises
 * GQAQ_DEV_BAD_POS. */
GQAQ_API int quest_append_kv_e4m3(const gqaq_dims *dims, uint8_t *k_cache, uint8_t *v_cache, uint8_t *meta,
                                  const gqaq_half *k_new, const gqaq_half *v_new, const int32_t *pos,
                                  float k_inv_scale, float v_inv_scale, void *stream);

/* Rebuild the bounds of pages [page_begin, page_end) from the codes of rows
 * below valid_len[b] (pages with no valid row are left untouched). Errors as
 * quest_update_meta. */
GQAQ_API int quest_update_meta_e4m3(const gqaq_dims *dims, const uint8_t *k_cache, const int32_t *valid_len,
                                    uint8_t *meta, int page_begin, int page_end, void *stream);

/* scores[b][kv][p] = k_scale * max_g sum_i max(q_i value(m_i), q_i value(M_i))
 * for pages p < ceil(valid_len[b] / S), q the unscaled fp16 query rows of KV
 * head kv (fp32 arithmetic; the products are exact). Later pages are not
 * written. k_scale must be finite and > 0, else GQAQ_ERR_INVALID_ARG. The
 * scores feed quest_topk_pages unchanged. */
GQAQ_API int quest_score_pages_e4m3(const gqaq_dims *dims, const gqaq_half *q, const uint8_t *meta, float k_scale,
                                    const int32_t *valid_len, float *scores, void *stream);

/* quest_sparse_attn over an E4M3 cache: attention over the tokens of the
 * listed pages with the keys and values dequantized on load (code value *
 * scale), fp32 accumulation, one rounding to fp16. Arguments, workspace and
 * errors as quest_sparse_attn and gqa_decode_attn_e4m3. */
GQAQ_API int quest_sparse_attn_e4m3(const gqaq_dims *dims, const gqaq_half *q, const uint8_t *k_cache,
                                    const uint8_t *v_cache, float k_scale, float v_scale, const int32_t *valid_len,
                                    const int32_t *page_idx, int k, float scale, gqaq_half *out, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* quest_decode_attn over an E4M3 cache, in one launch: the optional append
 * (quest_append_kv_e4m3's codes and bounds, with k_inv_scale / v_inv_scale),
 * quest_score_pages_e4m3's scores, quest_topk_pages' selection and
 * quest_sparse_attn_e4m3's attention over the selected pages. scores (times
 * k_scale) and page_idx are optional outputs as in quest_decode_attn. The
 * cluster kernel only: k <= 1024 (else GQAQ_ERR_UNSUPPORTED) and no
 * workspace; GQAQ_OPT_QUEST_EARLY_META applies as for quest_decode_attn.
 * k_scale must be finite and > 0. */
GQAQ_API int quest_decode_attn_e4m3(const gqaq_dims *dims, const gqaq_half *q, uint8_t *k_cache, uint8_t *v_cache,
                                    uint8_t *meta, const gqaq_half *k_new, const gqaq_half *v_new,
                                    const int32_t *pos, float k_inv_scale, float v_inv_scale, float k_scale,
                                    float v_scale, const int32_t *valid_len, int k, float scale, gqaq_half *out,
                                    float *scores, int32_t *page_idx, void *stream);

/* The 4-bit KV-cache variant (a format chosen here, see above: the plainest
 * one that keeps both contractions exact on integer levels): symmetric
 * INT4 with one fp32 scale per (token, KV head) row.
 *   k_codes, v_codes   [B][Hkv][Lmax][D/2] bytes: channel 2i of a row in the
 *                      low nibble of byte i, high nibble channel 2i+1; a
 *                      nibble holds level + 8, level in [-7, 7]
 *   k_scales, v_scales [B][Hkv][Lmax] fp32; value = level * scale
 * gqa_decode_attn_int4: [OPT] section 3's folded dense attention over such a
 * cache (levels exact in fp16; the K scale multiplies each fp32 score, the V
 * scale each token's probability). Same arguments, workspace and results as
 * gqa_decode_attn otherwise. Needs max_len % 4 == 0 (scale rows are loaded
 * as 16-byte multiples), else GQAQ_ERR_UNSUPPORTED. D in {64, 128}. */
GQAQ_API int gqa_decode_attn_int4(const gqaq_dims *dims, const gqaq_half *q, const uint8_t *k_codes,
                                  const float *k_scales, const uint8_t *v_codes, const float *v_scales,
                                  const int32_t *valid_len, float scale, gqaq_half *out, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Append one token per (sequence, KV head) to an INT4 cache: for the fp16 row
 * x = k_new[b][kv] ([B][Hkv][D]), scale = amax|x| / 7 and level =
 * clamp(rne(x / scale), -7, 7) in fp32 (a zero row: scale 0, levels 0),
 * written at row pos[b]; likewise v. pos[b] outside [0, Lmax) is skipped and
 * raises GQAQ_DEV_BAD_POS. */
GQAQ_API int kv_append_int4(const gqaq_dims *dims, uint8_t *k_codes, float *k_scales, uint8_t *v_codes,
                            float *v_scales, const gqaq_half *k_new, const gqaq_half *v_new, const int32_t *pos,
                            void *stream);

/* Prefill: causal attention of a chunk of q_len new tokens per sequence
 * ([OPT] "Prefill Needs Separate Design": for q_len > 1 the group axis is
 * merged into the sequence axis, so the G query heads of KV head kv and the
 * q_len tokens form one [G * q_len][D] row block, g outer, and every row
 * keeps its own causal mask).
 *   q, out     [B][Hq][q_len][D] fp16 (q_len rows per query head)
 *   k_cache, v_cache [B][Hkv][Lmax][D] fp16, already holding the chunk's keys
 *              and values at rows start[b] .. start[b]+q_len-1
 *   start      [B] int32, device: 0 <= start[b] <= Lmax - q_len
 * Token t of query head h of sequence b attends to rows 0 .. start[b]+t of
 * KV head h / G: out = softmax(scale q k^T) v over them, fp32 accumulation,
 * one rounding to fp16. With q_len = 1 and start = valid_len - 1 this is
 * gqa_decode_attn. A start outside its range raises GQAQ_DEV_BAD_POS and
 * gives that sequence a zero output. 1 <= q_len <= Lmax; D in {64, 128};
 * G in {1, 2, 4, 8}; page_size is ignored.
 * workspace: at least gqaq_prefill_workspace_bytes(dims, q_len) bytes, zero
 * filled once before first use; every call leaves its counters at zero. The
 * size depends on the SM count and GQAQ_OPT_PREFILL_SPLITS, so query it
 * again after changing that option. */
GQAQ_API size_t gqaq_prefill_workspace_bytes(const gqaq_dims *dims, int q_len);
GQAQ_API int gqa_prefill_attn(const gqaq_dims *dims, int q_len, const gqaq_half *q, const gqaq_half *k_cache,
                              const gqaq_half *v_cache, const int32_t *start, float scale, gqaq_half *out,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Human-readable name of a gqaq_status value (static string). */
GQAQ_API const char *gqaq_status_string(int status);

/* Library options (process-wide, read at launch time). */
enum {
    GQAQ_OPT_MAX_CTAS = 1,        /* cap on the persistent grid of the attention and
                                     score kernels; 0 = one wave of resident CTAs */
    GQAQ_OPT_WAIT_TIMEOUT_NS = 2, /* bound on every in-kernel wait; default 2e9 */
    GQAQ_OPT_TEST_STALL = 3,      /* nonzero: the attention kernels' producer issues
                                     no copy, so every consumer wait runs out
                                     (exercises the timeout path; outputs undefined) */
    GQAQ_OPT_CLUSTER_SIZE = 4,    /* CTAs per cluster of the fused Quest kernel (1, 2,
                                     4 or 8); 0 = chosen from the SM count and shape */
    GQAQ_OPT_PDL = 5,             /* nonzero (default): launch with programmatic stream
                                     serialization, so a kernel's launch overlaps the
                                     end of the previous one in the stream */
    GQAQ_OPT_QUEST_KERNEL = 6,    /* quest_decode_attn's kernel: 0 (default) = the
                                     cluster kernel when k <= 1024, else the work-queue
                                     kernel; 1 = cluster kernel; 2 = work-queue kernel
                                     (needs the workspace) */
    GQAQ_OPT_PREFILL_SPLITS = 7,  /* context splits per gqa_prefill_attn work item:
                                     0 (default) = enough CTAs for one wave; 1..32
                                     forced (larger splits may be empty) */
    GQAQ_OPT_PREFILL_KERNEL = 8,  /* gqa_prefill_attn's kernel: 0 (default) or 1 = the
                                     tensor-memory (tcgen05) kernel; 2 = the warp-level
                                     MMA kernel */
    GQAQ_OPT_QUEST_EARLY_META = 9, /* nonzero: quest_decode_attn's cluster kernel reads
                                     valid_len, pos and the first metadata tiles of its
                                     first (sequence, KV head) before it waits for the
                                     previous kernel in the stream (with GQAQ_OPT_PDL,
                                     while that kernel is still finishing). Tiles that
                                     hold rows pos-1 or pos are read after the wait.
                                     The caller guarantees that the previous kernel
                                     writes neither valid_len nor pos, nor any other
                                     page of meta. A decode loop whose previous kernel
                                     is another layer's attention, or this layer's
                                     previous step, satisfies it; quest_update_meta or
                                     a position update right before does not.
                                     Default 0. */
    GQAQ_OPT_DENSE_EARLY_KV = 10  /* nonzero: the dense attention calls (fp16, E4M3 and
                                     INT4 caches) read valid_len and start the first
                                     K/V tiles of their first context slice before
                                     they wait for the previous kernel in the stream.
                                     The tile holding each sequence's last valid row
                                     (the appended one) is read after the wait. The
                                     caller guarantees that the previous kernel writes
                                     neither valid_len nor any other row of the
                                     caches, as an append of that token or another
                                     layer's attention do. Default 0. */
};
GQAQ_API int gqaq_set_option(int option, int64_t value);

/* Copy the current device's status word (GQAQ_DEV_* flags) to *flags and
 * optionally reset it to 0. Synchronises the device. Returns GQAQ_OK, or
 * GQAQ_ERR_TIMEOUT if the word holds GQAQ_DEV_TIMEOUT. */
GQAQ_API int gqaq_device_status(int *flags, int reset);

/* Library version: major*10000 + minor*100 + patch. */
GQAQ_API int gqaq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQAQ_H */
