/*
 * aircache.h -- C ABI of the GB300 (sm_103a) AirCache compressor.
 *
 * AirCache compresses the visual part of a vision-language decoder's KV cache
 * once, right after prefill (paper notes "AirCache: Activating Inter-Modal
 * Relevancy KV Cache Compression for Efficient Large Vision-Language Model
 * Inference", ICCV 2025; section "Method details").  For every layer:
 *   1. elite observation window ("Key design 1", equations Att and k): the
 *      softmax row of the last text query over the text keys, averaged over
 *      the query heads, keeps the text positions j with P[j] >= alpha * max P;
 *   2. cross-modal scoring ("Key design 1", equations A_vtk and I_v): the elite
 *      text queries attend over [visual keys; elite text keys]; the visual
 *      columns are averaged over the elite rows and the query heads into I_v;
 *   3. layer budget ("Key design 2"): strength s_t = sum I_v and sample
 *      skewness s_k of I_v, normalised across the request's layers, give
 *      r_l = 1/2 (s'_t + s'_k) r and keep_l = clamp(floor(r_l N_v + 1/2), 1, N_v);
 *   4. selection and compaction ("Loss / training strategy", one-shot steps):
 *      the keep_l visual positions with the largest I_v (ties to the lower
 *      position), then every text position, gathered into a dense cache.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every data pointer is caller-owned DEVICE memory unless stated otherwise;
 *   the library allocates nothing, frees nothing and never synchronises, except
 *   aircache_get_error.  `stream` is a cudaStream_t (NULL = legacy default).
 * - Argument errors are detected on the host and returned before anything is
 *   enqueued.  Launch failures return AIRCACHE_ERR_CUDA.  Errors that only the
 *   GPU can see (inconsistent cu_seqlens/cu_visual contents, an elite set larger
 *   than max_elite, an output arena that is too small, a bounded wait that
 *   expired) are written to an error word in the workspace; read it with
 *   aircache_get_error.  Each entry point clears that word when it starts, so
 *   it reports the most recent call on that workspace.
 * - Calls are stateless.  Two calls may run concurrently only with distinct
 *   workspaces and outputs.
 * - Layout (varlen, token-major, like FlashAttention's varlen convention):
 *   request b owns prompt positions cu_seqlens[b] .. cu_seqlens[b+1]-1 of every
 *   layer's K and V; its first N_v[b] = cu_visual[b+1]-cu_visual[b] positions
 *   are visual, the remaining N_t[b] are text (visual first, X = Concat(X_v, X_t)),
 *   unless n_prefix puts some text before the visual span.
 *   Its text queries are rows cu_seqlens[b]-cu_visual[b] .. +N_t[b]-1 of the
 *   layer's Q_text.  K/V rows are [h_kv][head_dim], Q rows [h_q][head_dim], with
 *   element strides per token and per head; head_dim is contiguous.
 * - Inputs are post-RoPE.  Compaction keeps the values bit-exact; a decoder
 *   continuing from the compressed cache keeps the original positions
 *   (N_v + N_t onwards), not the compacted length.
 * - The per-layer visual index set is shared by all KV heads of the layer.
 */
#ifndef AIRCACHE_H
#define AIRCACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define AIRCACHE_API __attribute__((visibility("default")))
#else
#define AIRCACHE_API
#endif

#define AIRCACHE_MAX_LAYERS 256
#define AIRCACHE_VARIANT_WAIT_TEST (1 << 24)
#define AIRCACHE_MAX_TEXT 8192
#define AIRCACHE_NOALLOC_MAX_UNITS 2048  /* L * B limit of aircache_budget_noalloc */

typedef enum {
    AIRCACHE_OK = 0,
    AIRCACHE_ERR_INVALID_ARG = -1,   /* host: a bad pointer, size, stride or parameter */
    AIRCACHE_ERR_UNSUPPORTED = -2,   /* host: a valid problem this build does not handle */
    AIRCACHE_ERR_WORKSPACE = -3,     /* host: ws_bytes < aircache_workspace_size() */
    AIRCACHE_ERR_CUDA = -4,          /* a CUDA launch or memset failed */
    AIRCACHE_ERR_DEVICE_TIMEOUT = -5,  /* device: a bounded wait gave up */
    AIRCACHE_ERR_DEVICE_BOUNDS = -6,   /* device: cu_seqlens / cu_visual contents inconsistent */
    AIRCACHE_ERR_ELITE_OVERFLOW = -7,  /* device: an elite set larger than max_elite */
    AIRCACHE_ERR_CAPACITY = -8         /* device: output arena smaller than the compacted rows */
} aircache_status;

typedef enum { AIRCACHE_F32 = 0, AIRCACHE_BF16 = 1, AIRCACHE_INT8 = 2 } aircache_dtype;

/*
 * One compression problem: B requests, L layers.  All fields are read on the
 * host; the pointer fields marked "device" are read only by the GPU.
 */
typedef struct aircache_problem {
    int32_t num_layers;    /* L, 1..AIRCACHE_MAX_LAYERS */
    int32_t num_requests;  /* B >= 1 */
    int32_t h_q;           /* query heads; h_q % h_kv == 0 (query head h reads KV head h / (h_q/h_kv)) */
    int32_t h_kv;          /* key/value heads */
    int32_t head_dim;      /* D: 64 or 128 */
    int32_t dtype;         /* aircache_dtype of q_text, k and v */
    int32_t max_visual;    /* >= every N_v[b]; every N_v[b] must be >= 3 (skewness) */
    int32_t max_text;      /* >= every N_t[b], 1..AIRCACHE_MAX_TEXT; every N_t[b] >= 1 */
    int32_t max_elite;     /* cap on N_tk that the workspace is sized for; 0 means max_text */
    int32_t variant;       /* 0: the method.  Ablation variants (AirCache notes, "Ablation
                            * studies"): bits 0-7 the observation window -- 0 the elite
                            * window, 1 the last 16 text tokens, 2 the last 32, 3 every
                            * text token (a fixed window takes the elite set's place),
                            * 4 the last 32 visual tokens (their queries, from q_visual,
                            * over the visual keys only; aircache_compress on the
                            * streaming path only);
                            * bits 8-15 the layer budget -- 0 strength + skewness, 1
                            * uniform (r_l = r), 2 PyramidKV-style (linear in depth from
                            * (2 - 1/20) r to r/20), 3 strength only (s'_t r), 4
                            * skewness only (s'_k r); bits 16-23 the index sets -- 0
                            * one per layer, shared by the KV heads, 1 one per KV head
                            * (the edge-device compression page's group-wise top-k:
                            * KV head h keeps the keep_l visual positions with the
                            * largest I_v of its own g query heads; the budget stays
                            * the layer's; aircache_compress on the streaming path only
                            * -- else AIRCACHE_ERR_UNSUPPORTED, as from the staged
                            * calls -- and idx is then [L][h_kv][total_visual]);
                            * bit 24 (AIRCACHE_VARIANT_WAIT_TEST) a test hook for the
                            * device's bounded waits, not a variant of the method:
                            * the call's first kernel waits on a workspace flag that
                            * nothing sets, gives up after about 2^20 SM cycles, and
                            * records AIRCACHE_ERR_DEVICE_TIMEOUT; every later kernel
                            * of the call then returns without work.  The workspace
                            * stays usable (the next call clears the error word);
                            * other bits 0. */
    int64_t total_tokens;  /* == cu_seqlens[B] */
    int64_t total_visual;  /* == cu_visual[B] */
    const int32_t* cu_seqlens;  /* device [B+1], non-decreasing, cu_seqlens[0] == 0 */
    const int32_t* cu_visual;   /* device [B+1], non-decreasing, cu_visual[0] == 0 */
    const void* const* q_text;  /* HOST array [L] of device pointers: [total_tokens - total_visual] text rows */
    const void* const* k;       /* HOST array [L] of device pointers: [total_tokens] rows */
    const void* const* v;       /* HOST array [L] of device pointers: [total_tokens] rows.
                                   In aircache_compress and aircache_compact the values are
                                   read only by the compaction (the kept visual rows and
                                   every text row), so there v may also point to page-locked
                                   host memory that the device can address (cudaHostAlloc /
                                   cudaHostRegister, unified addressing): the compaction
                                   then reads those rows in place over the host link and
                                   the other rows never move.  The prefill entry points
                                   read every value and need them in device memory. */
    int64_t q_stride_tok;   /* elements between consecutive Q_text rows */
    int64_t q_stride_head;  /* elements between consecutive query heads */
    int64_t kv_stride_tok;  /* elements between consecutive K/V rows (same for K and V) */
    int64_t kv_stride_head; /* elements between consecutive KV heads */
    double alpha;           /* elite threshold, [0, 1] (the notes use 0.9) */
    double r;               /* mean visual retention ratio, (0, 1] */
    const int32_t* n_prefix;  /* optional device [B] (NULL: all 0): text tokens of request b
                                 BEFORE its visual span (a system prompt; the multimodal-
                                 layout page puts it there).  Request b's prompt is then
                                 [n_prefix[b] text][N_v[b] visual][the other text]; its
                                 text rows in q_text are all of its text tokens in prompt
                                 order; 0 <= n_prefix[b] <= N_t[b], else a device error
                                 AIRCACHE_ERR_DEVICE_BOUNDS.  Text is every non-visual
                                 token: the elite window and the scoring run over text
                                 indices as before, and compaction writes the kept visual
                                 rows, then every text row in text order. */
    const void* const* q_visual;  /* window 4 only (else NULL): HOST array [L] of device
                                     pointers to the visual tokens' post-RoPE queries,
                                     [total_visual] rows (request b's at cu_visual[b]..),
                                     with q_stride_tok / q_stride_head */
} aircache_problem;

/*
 * Bytes of device workspace a call on `p` needs (every entry point takes the
 * same workspace).  Returns 0 if `p` is invalid.  Host only; no CUDA call.
 * The workspace must be 256-byte aligned.
 */
AIRCACHE_API size_t aircache_workspace_size(const aircache_problem* p);

/*
 * Upper bound on the rows the compacted cache of `p` can hold, summed over all
 * layers and requests:  L * total_text + ceil(r * L * total_visual) + B * (2L + 1),
 * capped at L * total_tokens.  It holds because the budgets of a request
 * average to r over its layers and rounding/clamping add at most 3/2 per layer.
 * Returns -1 if `p` is invalid.  Host only; no CUDA call.
 */
AIRCACHE_API int64_t aircache_compress_bound(const aircache_problem* p);

/*
 * Steps 1-2: elite window and cross-modal scores of every (request, layer).
 *   iv    [L][total_visual] fp32: I_v of request b, layer l at
 *         iv[l * total_visual + cu_visual[b] + i], i < N_v[b].
 *   elite [L][B][max_text] int32: the first n_tk[l*B+b] entries of row (l, b)
 *         are that request's elite text positions (text-relative, ascending).
 *   n_tk  [L][B] int32: elite-set sizes N_tk (>= 1).
 */
AIRCACHE_API int aircache_score(const aircache_problem* p, void* ws, size_t ws_bytes,
                   float* iv, int32_t* elite, int32_t* n_tk, void* stream);

/*
 * Step 3: strength, skewness and keep counts from I_v (as written by
 * aircache_score).
 *   stats [L][B][2] fp64: (s_t, s_k) per (layer, request); may be NULL.
 *   keep  [L][B] int32: kept visual positions per (layer, request).
 */
AIRCACHE_API int aircache_budget(const aircache_problem* p, const float* iv, void* ws, size_t ws_bytes,
                    double* stats, int32_t* keep, void* stream);

/*
 * Step 3 without a workspace: the same strength, skewness and keep counts as
 * aircache_budget, for callers that cannot hand the library device memory --
 * for instance a serving engine that has given its whole memory pool to the
 * KV cache and must not call the allocator between requests, so it has no
 * aircache_workspace_size() bytes to pass.  The AirCache notes have no
 * counterpart of this call; it only changes where the scratch lives.
 *
 * Scratch: a fixed 41,216-byte array in the library's own device memory (one
 * per device, part of the loaded module): the error word, one arrival counter
 * per request and the (s_t, s_k) of each (layer, request).  Nothing is
 * allocated or freed.  The error word and the B counters must be zero when the
 * kernel starts; the call zeroes them itself with an asynchronous memset on
 * `stream` before its kernel.
 * Limit: num_layers * num_requests <= AIRCACHE_NOALLOC_MAX_UNITS (2048); a
 * larger problem returns AIRCACHE_ERR_UNSUPPORTED before anything is enqueued
 * (use aircache_budget with a workspace instead).
 * First call in a context: looks up the scratch address (cudaGetSymbolAddress,
 * which may load the module) with that context current and caches it under
 * the context's unique id; make that first call before capturing any stream.
 * Later calls in the same context reuse the address; a call made in another
 * context (a new one after cudaDeviceReset, or a second context of a
 * driver-API caller) looks it up again, since the address is only valid in
 * the context that was current when it was looked up.
 * Concurrency: the scratch is shared by every call on the device in the
 * process, so calls whose executions overlap (other streams, other host
 * threads) race on it and give wrong results; order them on one stream or
 * synchronise between them.
 *   iv, stats, keep: as in aircache_budget (stats may be NULL).
 *   device_status: NULL, or a device int32 that receives the device-side
 *     status (AIRCACHE_OK or an AIRCACHE_ERR_DEVICE_* code) by a 4-byte
 *     device-to-device copy enqueued after the kernel.  keep and stats are
 *     only meaningful when that status is AIRCACHE_OK; after an inconsistent
 *     request layout the keep counts of the affected request are written as 0.
 * Host-detected errors are returned as by aircache_budget.
 */
AIRCACHE_API int aircache_budget_noalloc(const aircache_problem* p, const float* iv, double* stats,
                                         int32_t* keep, int32_t* device_status, void* stream);

/*
 * Step 4a: top-keep selection.  For each (l, b) writes the keep[l*B+b] visual
 * positions (request-relative, ascending) with the largest I_v, ties to the
 * lower position, to idx[l * total_visual + cu_visual[b] + j].  Entries past
 * the keep count are left untouched.
 *   idx [L][total_visual] int32.
 */
AIRCACHE_API int aircache_select(const aircache_problem* p, const float* iv, const int32_t* keep,
                    void* ws, size_t ws_bytes, int32_t* idx, void* stream);

/*
 * Step 4b: compaction.  Writes, for each layer l and request b in that order,
 * the rows [K_v[idx]; K_t] (keep + N_t rows) of that (l, b), and the same for V,
 * into the dense arenas out_k / out_v ([rows][h_kv][head_dim], same dtype as
 * the input), bit-exact.  out_offsets [L*B + 1] int64 receives the first row of
 * each (l, b): rows of (l, b) are out_offsets[l*B+b] .. out_offsets[l*B+b+1]-1.
 * out_rows_capacity is the number of rows out_k and out_v can hold
 * (aircache_compress_bound rows always suffice).
 */
AIRCACHE_API int aircache_compact(const aircache_problem* p, const int32_t* idx, const int32_t* keep,
                     void* ws, size_t ws_bytes, void* out_k, void* out_v,
                     int64_t* out_offsets, int64_t out_rows_capacity, void* stream);

/*
 * Steps 1-4 in one call on one stream (the one-shot schedule: every layer is
 * scored, then every budget is set, then every layer is compacted).
 * keep [L][B] is required; iv [L][total_visual] and idx [L][total_visual] ([L][h_kv][total_visual] with one index set per KV head) are
 * optional (NULL keeps them inside the workspace).  Outputs as above.
 */
AIRCACHE_API int aircache_compress(const aircache_problem* p, void* ws, size_t ws_bytes,
                      void* out_k, void* out_v, int64_t* out_offsets, int64_t out_rows_capacity,
                      int32_t* keep, int32_t* idx, float* iv, void* stream);

/*
 * Waits for `stream`, then reads the device error word of `ws` into *status
 * (AIRCACHE_OK or a device error code).  The only entry point that blocks.
 */
AIRCACHE_API int aircache_get_error(const void* ws, void* stream, int32_t* status);

/* Static description of a status code. */
AIRCACHE_API const char* aircache_status_string(int status);

/*
 * Number of kernels one aircache_compress call on `p` launches (for launch
 * accounting), or -1 if `p` is invalid.  It depends on the scoring path, which
 * the problem alone decides: bf16 inputs whose per-layer key pointers are
 * evenly strided take the streaming path (7 kernels), others the wide path (5).
 * The first kernel clears the call's block of counters and its error word.
 */
AIRCACHE_API int aircache_compress_launches(const aircache_problem* p);

/* Scoring fused into prefill (AirCache notes, "Limitations and outlook": the
 * method's scoring costs the prefill 5-12 %; here it reads the prefill's own
 * logits instead of streaming the keys again).
 *
 * aircache_prefill: causal prefill attention of every layer of `p`,
 *   O_h = softmax_j(q_h . k_j / sqrt(D), j <= i within the request) V, for every
 *   prompt row i of every request and query head h (KV head h / (h_q / h_kv)).
 * aircache_prefill_compress: the same attention, and from it the whole one-shot
 *   compression of aircache_compress: the elite window on the prompt's own text
 *   queries, then each elite row's logits against every visual key and their
 *   log-sum-exp taken inside the prefill (no second pass over the keys), then
 *   I_v, the layer budgets, the selection and the compacted cache as
 *   aircache_compress produces them (the same arguments and outputs; I_v agrees
 *   with aircache_compress's within fp32 summation order).
 *
 * q_all: HOST array [L] of device pointers, evenly strided across layers, to the
 *   queries of EVERY prompt row, [total_tokens] rows in the order of k and v,
 *   element strides qa_stride_tok / qa_stride_head (D contiguous, 16-byte
 *   aligned); p->q_text and its strides are not read.
 * attn_out: HOST array [L] of device pointers, 16-byte aligned, the bf16 output
 *   [total_tokens] rows of h_q heads x D with element strides o_stride_tok /
 *   o_stride_head, written by both calls.
 * Supported: bf16, head_dim 128, visual-first prompts (n_prefix NULL), variant 0,
 *   k, v and q_all evenly strided across layers; else AIRCACHE_ERR_UNSUPPORTED
 *   (before any launch).  ws as for aircache_compress (aircache_workspace_size of
 *   p).  Errors as for aircache_compress; enqueued on `stream`, no allocation,
 *   no synchronisation.
 */
AIRCACHE_API int aircache_prefill(const aircache_problem* p, const void* const* q_all, int64_t qa_stride_tok,
                                  int64_t qa_stride_head, void* const* attn_out, int64_t o_stride_tok,
                                  int64_t o_stride_head, void* ws, size_t ws_bytes, void* stream);
AIRCACHE_API int aircache_prefill_compress(const aircache_problem* p, const void* const* q_all,
                                           int64_t qa_stride_tok, int64_t qa_stride_head, void* const* attn_out,
                                           int64_t o_stride_tok, int64_t o_stride_head, void* ws, size_t ws_bytes,
                                           void* out_k, void* out_v, int64_t* out_offsets,
                                           int64_t out_rows_capacity, int32_t* keep, int32_t* idx, float* iv,
                                           void* stream);

/*
 * aircache_compress with timing marks, for measurement: `events` is a host
 * array of n_events == aircache_compress_launches(p) + 1 cudaEvent_t handles
 * created by the caller; events[0] is recorded on `stream` before the first
 * kernel and events[i] right after kernel i, so the elapsed time between
 * consecutive events is that kernel's duration on the launching stream.
 * Results are identical to aircache_compress.
 */
AIRCACHE_API int aircache_compress_profile(const aircache_problem* p, void* ws, size_t ws_bytes,
                                           void* out_k, void* out_v, int64_t* out_offsets,
                                           int64_t out_rows_capacity, int32_t* keep, int32_t* idx,
                                           float* iv, void* const* events, int n_events, void* stream);

/* Name of kernel i (0-based, launch order) of aircache_compress on `p`, or NULL. */
AIRCACHE_API const char* aircache_kernel_name(const aircache_problem* p, int i);

/* ------------------------------------------------------------------ decode */

/*
 * One decode step of attention over cached K/V rows: the consumer of the
 * compressed cache.  A decode step brings one new query per sequence, which
 * reads every cached key and value (KV-cache tutorial page, section "Prefill
 * and Decode"; the append K_{1:t} = [K_{1:t-1}; k_t]); once the cache is
 * compacted, decoding is plain dense attention over the compacted rows (the
 * edge-device compression page, head-wise top-k scheme).  For sequence s and
 * query head h (KV head h / (h_q / h_kv)):
 *   out[s][h] = sum_j softmax_j(q[s][h] . k_j / sqrt(head_dim)) v_j
 * over the rows j = row_begin[s] .. row_end[s]-1 of the k / v arenas, plus the
 * row (k_new[s], v_new[s]) when k_new is given.  No mask: every cached row
 * precedes the query.  An empty sequence (no rows, no new row) gets out = 0.
 *
 * The arenas of aircache_compress plug in directly: for layer l of a batch of
 * B requests, row_begin = out_offsets + l*B and row_end = out_offsets + l*B + 1
 * (num_seqs = B); all layers at once use out_offsets and out_offsets + 1 with
 * num_seqs = L*B.  A full cache [rows][h_kv][head_dim] uses its own ranges.
 * Positions are the caller's: q and k_new are post-RoPE at the original
 * position (N_v + N_t + step), not the compacted length.
 *
 * Layout (element strides; head_dim contiguous):
 *   q      [num_seqs][h_q][head_dim]    q_stride_seq, q_stride_head
 *   k, v   [kv_rows][h_kv][head_dim]    kv_stride_row, kv_stride_head
 *   k_new, v_new [num_seqs][h_kv][head_dim]  new_stride_seq, new_stride_head
 *   out    [num_seqs][h_q][head_dim]    fp32, dense
 *   row_begin, row_end: device int64 [num_seqs].
 * With kv_dtype AIRCACHE_INT8 the cached rows are int8 codes c with
 * k_j = k_scale[s][h] * c_j (and likewise v); the kernel computes with the codes
 * exactly and applies the scales to the logits and to the weighted sum, so the
 * result is the attention over the dequantised rows (the new row stays bf16).
 * Requirements (else AIRCACHE_ERR_INVALID_ARG, or AIRCACHE_ERR_UNSUPPORTED
 * for the dtype / group limits): dtype AIRCACHE_BF16; kv_dtype AIRCACHE_BF16
 * or AIRCACHE_INT8 (then k_scale and v_scale given); head_dim 64 or 128;
 * h_q % h_kv == 0 and h_q / h_kv <= 16; k and v 16-byte aligned with
 * kv_stride_row and kv_stride_head multiples of 16 bytes (tensor-map rules);
 * 1 <= kv_rows <= 2^31 - 2^16; num_seqs <= 65535; q 16-byte aligned with
 * q_stride_seq and q_stride_head multiples of 8; max_rows >= 0.
 * max_rows is a hint, not a limit: the expected longest range, which sizes the
 * split of each sequence across CTAs (and the workspace).  Device-side, a
 * range with row_begin < 0, row_end < row_begin or row_end > kv_rows sets
 * AIRCACHE_ERR_DEVICE_BOUNDS in the workspace error word and that sequence's
 * output is left as zeros.
 */
typedef struct aircache_decode_problem {
    int32_t num_seqs;
    int32_t h_q;
    int32_t h_kv;
    int32_t head_dim;
    int32_t dtype;     /* of q (and of k_new, v_new): AIRCACHE_BF16 */
    int32_t kv_dtype;  /* of the cached rows k, v: AIRCACHE_BF16, or AIRCACHE_INT8 (codes of
                          aircache_quantize_int8, with k_scale / v_scale) */
    int64_t kv_rows;
    int64_t max_rows;
    const void* q;
    const void* k;
    const void* v;
    const int64_t* row_begin;
    const int64_t* row_end;
    const void* k_new;  /* optional (NULL: no new row); v_new must then be NULL too */
    const void* v_new;
    int64_t q_stride_seq;
    int64_t q_stride_head;
    int64_t kv_stride_row;
    int64_t kv_stride_head;
    int64_t new_stride_seq;
    int64_t new_stride_head;
    float* out;
    const float* k_scale;  /* AIRCACHE_INT8 only: [num_seqs][h_kv] fp32 scales of the codes of */
    const float* v_scale;  /* sequence s, KV head h (for the compacted arena of layer l: the
                              aircache_quantize_int8 scales + l*B*h_kv) */
    int32_t flags;         /* 0, or AIRCACHE_DECODE_EARLY_CACHE */
    int32_t reserved1;     /* 0 */
    const int32_t* row_index;  /* optional (NULL: ranges are arena rows): device [index_len]
                                  arena rows; row_begin[s] .. row_end[s]-1 then index this
                                  array, and sequence s attends over the rows it lists
                                  (gather-fused decode: the full cache with the row list of
                                  aircache_row_index, no compaction).  bf16 rows only.  A
                                  listed row outside [0, kv_rows) sets
                                  AIRCACHE_ERR_DEVICE_BOUNDS and reads row 0 instead. */
    int64_t index_len;         /* entries of row_index (the ranges' bound), >= 1 when given */
} aircache_decode_problem;

/*
 * AIRCACHE_DECODE_EARLY_CACHE: launch with programmatic dependent launch.  The
 * kernel may start while the kernel before it on the stream is finishing, and
 * reads row_begin, row_end and the cached rows right away; it waits for that
 * kernel (griddepcontrol.wait) before it reads q, k_new, v_new or the scales and
 * before it writes anything else than the error word.  Valid only when the
 * kernel launched just before on the stream writes neither the row ranges nor
 * the cached rows (in a decoder: the cache append of this step goes to k_new /
 * v_new, or happened earlier).  Consecutive layers of a decode step (one call
 * per layer) then overlap each kernel's start with the previous one's end.
 */
#define AIRCACHE_DECODE_EARLY_CACHE 1

/*
 * The row list of a compression without the copy: for every (l, b) of `p`, in
 * aircache_compact's row order (rows out_offsets[l*B+b] .. out_offsets[l*B+b+1]-1),
 * row_index[row] = the prompt position in layer l's K / V of that compacted
 * row (the kept visual positions, then every text position; n_prefix
 * respected).  keep, idx and out_offsets are aircache_compress's outputs
 * (one index set per layer: with one per KV head, AIRCACHE_ERR_UNSUPPORTED);
 * capacity is the length of row_index (too small: AIRCACHE_ERR_CAPACITY in
 * the workspace error word).  Decoding layer l over wl.k[l] with these rows
 * (aircache_decode with row_index) attends over the same rows as decoding the
 * compacted arena.  Two kernels: one clears the workspace's counters, one
 * writes the rows.
 */
AIRCACHE_API int aircache_row_index(const aircache_problem* p, const int32_t* keep, const int32_t* idx,
                                    const int64_t* out_offsets, void* ws, size_t ws_bytes, int32_t* row_index,
                                    int64_t capacity, void* stream);

/* Workspace bytes aircache_decode needs for `p` on the current device, or 0 if
 * `p` is invalid.  Depends on num_seqs, h_q, h_kv, head_dim, max_rows and the
 * device's SM count. */
AIRCACHE_API size_t aircache_decode_workspace_size(const aircache_decode_problem* p);

/* Enqueue the decode step on `stream` (one kernel, nothing else).  ws is
 * caller-owned device memory of at least aircache_decode_workspace_size(p)
 * bytes (256-byte aligned), ZEROED ONCE by the caller before its first use;
 * every call leaves it in that state again, so it can be reused call after
 * call with no memset between them (a memset node between consecutive decode
 * kernels costs several microseconds per layer).  Unlike the compression entry
 * points, aircache_decode does not clear the error word: a device error stays
 * recorded (aircache_get_error reports it) until the caller zeroes the
 * workspace again. */
AIRCACHE_API int aircache_decode(const aircache_decode_problem* p, void* ws, size_t ws_bytes, void* stream);

/* Number of CTAs the decode kernel splits each (sequence, KV head) into for `p`
 * on the current device, or -1 if `p` is invalid (for measurement). */
AIRCACHE_API int aircache_decode_splits(const aircache_decode_problem* p);

/* ------------------------------------------------------------- int8 storage */

/*
 * int8 storage of a compacted cache, applied after the token compression (LLM
 * KV-compression notes, section "Quantization stacked on compression":
 * quantise after compressing, with one scale per head taken from the head's
 * largest |value| over the quantisation range; KV-cache tutorial page, section
 * "Quantization": symmetric q = clip(round(x / s), q_min, q_max), x_hat = s q).
 * For every unit u (rows offsets[u] .. offsets[u+1]-1) and KV head h,
 * separately for K and V:
 *   s = max |x| / 127 in fp32 over the unit's rows and the head's head_dim values;
 *   q = clip(round(x / s), -127, 127), x / s in fp32 (correctly rounded),
 *       round half away from zero; a head whose values are all 0 has s = 0, q = 0.
 * The units of aircache_compress's arena are its (layer, request) pairs:
 * offsets = out_offsets, num_units = L*B.
 *
 * Layout: k, v bf16 [rows][h_kv][head_dim] (kv_stride_row, kv_stride_head
 * element strides); k8, v8 int8 dense [rows][h_kv][head_dim] (same row
 * numbering); k_scale, v_scale fp32 [num_units][h_kv]; offsets device int64
 * [num_units + 1].  Requirements (else AIRCACHE_ERR_INVALID_ARG): head_dim 64
 * or 128, dtype AIRCACHE_BF16, k and v 16-byte aligned with strides multiples
 * of 8 elements, k8 and v8 16-byte aligned, 1 <= rows, 0 <= num_units <= 2^27,
 * reserved0 == 0.  `status` (optional device int32) is cleared first, then
 * receives AIRCACHE_ERR_DEVICE_BOUNDS if a unit's range lies outside [0, rows)
 * (that unit's codes are not written).  One memset (when status is given)
 * and one kernel (a cluster of 8 CTAs per unit, KV head and K or V).
 */
typedef struct aircache_quant_problem {
    int32_t num_units;
    int32_t h_kv;
    int32_t head_dim;
    int32_t dtype;
    int32_t reserved0;
    int32_t reserved1;
    int64_t rows;
    const void* k;
    const void* v;
    int64_t kv_stride_row;
    int64_t kv_stride_head;
    const int64_t* offsets;
    int8_t* k8;
    int8_t* v8;
    float* k_scale;
    float* v_scale;
} aircache_quant_problem;

AIRCACHE_API int aircache_quantize_int8(const aircache_quant_problem* p, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* AIRCACHE_H */
