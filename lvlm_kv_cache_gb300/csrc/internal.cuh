// Internal interfaces of the AirCache CUDA library: the device-side problem
// description, the workspace carve-up and the kernel launchers.  Not installed;
// the public ABI is include/aircache.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/aircache.h"

namespace aircache {

// Device-visible description of one problem (host checks done).
struct Dev {
  int L, B, h_q, h_kv, d, g, dtype;
  int max_visual, max_text, max_elite;
  int elite_stride;      // entries per (layer, request) of the elite list: max(max_text, max_elite)
  int rows_max;          // h_q * max_elite: query rows per (layer, request)
  int rc_max;            // ceil(g * max_elite / 32): 32-row chunks per KV head
  int lse_stride;        // h_kv * rc_max * 32: floats of row LSEs per (layer, request)
  int64_t total_tokens, total_visual, total_text;
  const int32_t* cu_seqlens;
  const int32_t* cu_visual;
  const int32_t* n_prefix;  // optional [B]: text tokens before the visual span
  int64_t q_stride_tok, q_stride_head, kv_stride_tok, kv_stride_head;
  double alpha, r;
  float scale_log2;      // log2(e) / sqrt(D): logits are kept in base 2
  int stream_ok;         // 1: every unit takes the streaming scoring path (stream.cu)
  int mom_slots;         // ceil(max_visual / 128): moment records per unit
  int window_mode;       // 0 elite window; 1 / 2 / 3: last 16 / last 32 / every text token
  int budget_mode;       // 0 strength + skewness; 1 uniform; 2 PyramidKV-style; 3 strength; 4 skewness
  int head_sets;         // 1: one visual index set per KV head (I_v of each KV group)
  int chn;               // streaming pass-1 chunks per (unit, KV head): visual chunks + 1 text chunk
  int wait_test;         // 1: the first kernel's bounded wait on a flag nothing sets (a test hook)
  int q_all;             // 1: the query pointers cover every prompt row (fused prefill), so text
                         //    query j of a request is row text_tok(R, j), not R.txt0 + j
};

// Streaming scoring path: query rows are taken in chunks of this many (a unit
// with at most one chunk per KV head stores its logits), and a pass-1 work item
// covers this many 128-key visual tiles.
constexpr int kRowChunk = 32;
constexpr int kStreamTiles = 4;
// Rows per (layer, KV head) of the stored-logit buffer: units with at most
// this many query rows per KV head (two row chunks) keep their pass-1 logits
// and take pass 2; the others recompute them from the keys in pass 2k.
constexpr int kLgRows = 2 * kRowChunk;

struct LayerPtrs {
  const void* q[AIRCACHE_MAX_LAYERS];
  const void* qv[AIRCACHE_MAX_LAYERS];  // visual-token queries (window 4 only)
  const void* k[AIRCACHE_MAX_LAYERS];
  const void* v[AIRCACHE_MAX_LAYERS];
};

// Workspace carve-up.  The first block (error word and counters) is zeroed by
// every entry point.
struct Ws {
  int32_t* error;        // [1]
  uint32_t* cnt_all;     // [1]   requests whose budget is done
  unsigned long long* ticket;  // [1] next pass-1 work item of the wide scoring kernel
  unsigned long long* ticket_n;  // [1] next pass-1 work item of the streaming path
  int32_t* list_n;       // [4]   units on the streaming path, on the wide path, streaming units
                         //       without stored logits (pass 2k), the other streaming units
  unsigned long long* p2pack;  // [1] routing of the pass-2 units: (count << 32) + their total weight
  uint32_t* cnt_cmp;     // [1]   compaction chunks claimed after each CTA's first two
  uint32_t* cnt_req;     // [B]   layers of a request whose stats are done
  uint32_t* p2claim;     // [L*B] claimed pass-2 work items per (layer, request)
  uint32_t* cnt_p1;      // [L*B] finished pass-1 items per (layer, request)
  uint32_t* cnt_p2;      // [L*B] finished pass-2 items per (layer, request) (wide path); moment
                         //       records stored per unit (streaming path)
  uint32_t* lse_ready;   // [L*B] row log-sum-exps published
  int32_t* elite;        // [L*B*max_text]
  int32_t* n_tk;         // [L*B]
  int32_t* stream_list;  // [L*B] streaming units: those with more than kLgRows rows per KV head
                         //       (pass 2k) in slots [0, list_n[2]), the others (pass 2) in
                         //       [L*B - list_n[3], L*B) (any order within each)
  int4* stream_info;     // [L*B][2] the layout record of stream_list[i] (as uinfo, with .w of the second = u)
  uint32_t* p2wpre;      // [L*B] pass-2 units: the weight of the pass-2 units routed before the one in
                         //       this slot (weight = 256-key blocks x 32-row chunks per KV head)
  int32_t* wide_list;    // [L*B] units on the wide path (list_n[1] of them, any order)
  float* lg;             // [L][h_kv][kLgRows][lg stride] streaming path: logits of row r of KV head h
  float4* mom;           // [L*B][mom_slots][3] streaming path: moments of each key block / tile of I_v
  float4* lstat;         // [L*B] streaming path: the unit's (s_t, s_k) as float-float pairs
  float2* part_s;        // [L*B][h_kv][rc_max*32][chn] streaming pass 1: (max, sum of exp2) per (row, chunk)
  int4* uinfo;           // [L*B][2] {seq0, vis0, txt0, N_v}, {N_t, N_tk, 1, 0} per (layer, request)
  void* qel;             // [L*B][rows_max][D] elite query rows, row kvh*g*N_tk + hh*N_tk + e
  void* kel;             // [L*B][h_kv][max_elite][D] elite text keys
  float2* part;          // [L*B][TV+TT][rows_max] pass-1 (max, sum of exp2) per (tile, row)
  float* lse;            // [L*B][h_kv][rc_max][32] row log-sum-exp, base 2
  float* ivp;            // [G][L*total_visual] per-KV-group I_v partials (G > 1 only)
  float* iv;             // [L*total_visual]
  float* ivh;            // [L][h_kv][total_visual] I_v of each KV group (head_sets only)
  double* stats;         // [L*B*2]
  int32_t* keep;         // [L*B]
  int32_t* idx;          // [L*total_visual]; head_sets: [L][h_kv][total_visual]
  int64_t* out_offsets;  // [L*B+1]
  size_t zero_bytes;     // bytes of the zeroed block
};

// One request's slice of the packed layout, validated on the device.
struct Req {
  int64_t seq0;   // first prompt position in K/V
  int64_t vis0;   // first I_v slot
  int64_t txt0;   // first Q_text row
  int n_v, n_t;
  int n_p;        // text tokens before the visual span
};

__device__ __forceinline__ void set_error(int32_t* err, int code) {
  atomicCAS(err, 0, code);
}

__device__ __forceinline__ bool load_req(const Dev& p, int b, Req& r) {
  const int64_t s0 = p.cu_seqlens[b], s1 = p.cu_seqlens[b + 1];
  const int64_t v0 = p.cu_visual[b], v1 = p.cu_visual[b + 1];
  const int64_t n_v = v1 - v0, n_t = (s1 - s0) - n_v;
  bool ok = s0 >= 0 && s1 <= p.total_tokens && v0 >= 0 && v1 <= p.total_visual &&
            n_v >= 3 && n_v <= p.max_visual && n_t >= 1 && n_t <= p.max_text &&
            (s0 - v0) >= 0 && (s0 - v0) + n_t <= p.total_text;
  if (b == 0) ok = ok && s0 == 0 && v0 == 0;
  if (b == p.B - 1) ok = ok && s1 == p.total_tokens && v1 == p.total_visual;
  const int64_t n_p = p.n_prefix ? p.n_prefix[b] : 0;
  ok = ok && n_p >= 0 && n_p <= n_t;
  r.seq0 = s0;
  r.vis0 = v0;
  r.txt0 = s0 - v0;
  r.n_v = (int)n_v;
  r.n_t = (int)n_t;
  r.n_p = ok ? (int)n_p : 0;
  return ok;
}

// Prompt positions (rows of K and V) of visual index i and text index j: the
// prompt is [n_p text][n_v visual][n_t - n_p text].
__device__ __forceinline__ int64_t vis_tok(const Req& r, int64_t i) { return r.seq0 + r.n_p + i; }
__device__ __forceinline__ int64_t text_tok(const Req& r, int64_t j) {
  return r.seq0 + j + (j >= r.n_p ? r.n_v : 0);
}

// Row of text query j of request R in the query tensor: packed text rows, or
// (fused prefill) the prompt row of that text token.
__device__ __forceinline__ int64_t text_q_row(const Dev& p, const Req& r, int64_t j) {
  return p.q_all ? text_tok(r, j) : r.txt0 + j;
}

// Launch plan of the persistent scoring kernel.
struct ScoreLaunch {
  int TV, TT;      // visual / elite-text tile slots per unit
  int G;           // KV-head groups per tile
  int lag;         // units between a unit's two passes in the ticket order
  int tail;        // 1: also stats, budgets and offsets
  int grid;        // CTAs
  int allow_tma;   // 1: use TMA tensor copies when the layout allows
  long long tickets;
  int64_t out_capacity;
};
ScoreLaunch plan_score(const Dev& p, int sms, bool tail, int64_t out_capacity);

// Launchers (each returns cudaGetLastError() of its launches).
cudaError_t launch_elite(const Dev& p, const LayerPtrs& lp, const Ws& w, cudaStream_t s);
// compact_kernel in row-list mode: row_index[row] = the prompt position of each compacted row.
cudaError_t launch_row_index(const Dev& p, const LayerPtrs& lp, const Ws& w, int32_t* row_index, int64_t capacity,
                             cudaStream_t s);
cudaError_t launch_score(const Dev& p, const LayerPtrs& lp, const Ws& w, const ScoreLaunch& L,
                         cudaStream_t s);
// Stats and keep counts from I_v, one CTA per (layer, request); with
// `offsets` also the compacted-cache row offsets (checked against out_capacity).
cudaError_t launch_stats_budget(const Dev& p, const Ws& w, double* stats_out,
                                int64_t out_capacity, bool offsets, cudaStream_t s);
// budget (streaming path): the select kernel first derives the keep counts of
// its request from passes 2 / 2k's moment records and writes the statistics
// and keep counts; the row offsets (checked against out_capacity) come from the
// compaction, or from the selection's last CTA when !compact_makes_offsets(p).
cudaError_t launch_select(const Dev& p, const Ws& w, cudaStream_t s, bool budget = false,
                          int64_t out_capacity = 0);
// Streaming scoring path (stream.cu).  stream_eligible: the problem's dtype,
// sizes and key layout allow it (bf16, per-layer key pointers evenly strided);
// it depends on the problem alone, so the kernel sequence of a call is known on
// the host.  Pass 1 streams the keys and produces row partials (and, for units
// with one row chunk per KV head, their logits); pass 2 turns stored logits
// into I_v and merges the other units' row LSEs; pass 2k recomputes those
// units' logits from the keys.
struct StreamMaps {
  CUtensorMap kmap, kmap2, qmap, kelmap;  // keys (boxes of 128 / 256 rows), elite queries, elite keys
  CUtensorMap lgmap;                      // stored logits of the streaming path
};
bool stream_eligible(const Dev& p, const LayerPtrs& lp);
bool encode_stream_maps(const Dev& p, const LayerPtrs& lp, const Ws& w, StreamMaps* m);
cudaError_t launch_stream_p1(const Dev& p, const StreamMaps& m, const Ws& w, int sms, cudaStream_t s);
cudaError_t launch_stream_p2(const Dev& p, const StreamMaps& m, const Ws& w, int sms, cudaStream_t s);
cudaError_t launch_stream_p2k(const Dev& p, const StreamMaps& m, const Ws& w, int sms, cudaStream_t s);

// Fused prefill (prefill.cu): causal attention of every layer (bf16, D = 128,
// visual-first prompts); with `score`, also each elite row's visual logits
// (stored-logit buffer) and row partials, and the elite rows' text-key partials.
bool prefill_eligible(const Dev& p, const LayerPtrs& lp, int64_t qa_stride_tok, int64_t qa_stride_head,
                      int64_t o_stride_tok, int64_t o_stride_head);
cudaError_t launch_prefill(const Dev& p, const LayerPtrs& lp, const Ws& w, int64_t qa_stride_tok,
                           int64_t qa_stride_head, void* const* out, int64_t o_stride_tok, int64_t o_stride_head,
                           int max_tokens, bool score, int sms, cudaStream_t s);

// Launch `kernel` on `s` with programmatic stream serialization, so that its
// CTAs may start (and run up to pdl_wait()) while the previous kernel on the
// stream finishes.
template <typename Arg>
cudaError_t launch_pdl(void (*kernel)(Arg), dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Arg& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `func` on the current
// device, skipped when an earlier call already allowed at least `bytes`.
cudaError_t allow_smem(const void* func, int bytes);
cudaError_t launch_offsets(const Dev& p, const Ws& w, int64_t out_capacity, cudaStream_t s);
// aircache_budget_noalloc after host validation: stats, budgets and the
// optional device status copy, with the module's fixed scratch.
int budget_noalloc(const Dev& p, const float* iv, double* stats_out, int32_t* keep, int32_t* device_status,
                   cudaStream_t s);
// make_offsets (after the budget-mode selection): the compaction forms the row
// offsets from the keep counts itself when compact_makes_offsets(p); otherwise
// the selection's last CTA writes them.
bool compact_makes_offsets(const Dev& p);
cudaError_t launch_compact(const Dev& p, const LayerPtrs& lp, const Ws& w, void* out_k,
                           void* out_v, int64_t capacity, cudaStream_t s, bool make_offsets = false);

}  // namespace aircache
