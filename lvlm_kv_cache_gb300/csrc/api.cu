// Host runtime of the AirCache library: argument validation, workspace
// carve-up, and the C ABI entry points declared in include/aircache.h.  Every
// entry point validates on the host, then enqueues its kernels on the caller's
// stream; nothing here allocates, frees or synchronises except
// aircache_get_error.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.cuh"
#include "ptx.cuh"

namespace aircache {

cudaError_t allow_smem(const void* func, int bytes) {
  struct Entry {
    const void* func;
    int dev, bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& x : done) {
    if (x.func == func && x.dev == dev && x.bytes >= bytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.push_back(Entry{func, dev, bytes});
  return e;
}

}  // namespace aircache

using namespace aircache;

namespace {

constexpr size_t kAlign = 256;
// Kernels of one aircache_compress call, by scoring path (the first clears the
// call's zeroed block).
const char* const kStreamKernels[] = {"zero_block",   "elite_window",  "score_pass1",   "score_pass2",
                                      "score_pass2k", "budget_select", "gather_compact"};
const char* const kWideKernels[] = {"zero_block", "elite_window", "score_wide", "select_topk", "gather_compact"};
constexpr int kStreamCount = 7, kWideCount = 5;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int esize_of(int dtype) { return dtype == AIRCACHE_BF16 ? 2 : 4; }

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int validate(const aircache_problem* p) {
  if (!p) return AIRCACHE_ERR_INVALID_ARG;
  if (p->num_layers < 1 || p->num_layers > AIRCACHE_MAX_LAYERS) return AIRCACHE_ERR_INVALID_ARG;
  if (p->num_requests < 1) return AIRCACHE_ERR_INVALID_ARG;
  if (p->num_requests > 65535) return AIRCACHE_ERR_UNSUPPORTED;  // grid dimension
  if (p->h_q < 1 || p->h_kv < 1 || p->h_q % p->h_kv != 0) return AIRCACHE_ERR_INVALID_ARG;
  if (p->head_dim < 1) return AIRCACHE_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return AIRCACHE_ERR_UNSUPPORTED;
  if (p->dtype != AIRCACHE_F32 && p->dtype != AIRCACHE_BF16) return AIRCACHE_ERR_UNSUPPORTED;
  if (p->max_visual < 3 || p->max_text < 1) return AIRCACHE_ERR_INVALID_ARG;
  if (p->max_text > AIRCACHE_MAX_TEXT) return AIRCACHE_ERR_UNSUPPORTED;
  if (p->max_elite < 0 || p->max_elite > p->max_text) return AIRCACHE_ERR_INVALID_ARG;
  if ((p->variant & ~(0xffffff | AIRCACHE_VARIANT_WAIT_TEST)) != 0 || (p->variant & 0xff) > 4 ||
      ((p->variant >> 8) & 0xff) > 4 ||
      ((p->variant >> 16) & 0xff) > 1) {
    return AIRCACHE_ERR_INVALID_ARG;
  }
  const int64_t B = p->num_requests;
  const int64_t total_text = p->total_tokens - p->total_visual;
  if (p->total_visual < 3 * B || total_text < B) return AIRCACHE_ERR_INVALID_ARG;
  if (p->total_visual > B * p->max_visual || total_text > B * p->max_text) return AIRCACHE_ERR_INVALID_ARG;
  if (p->total_tokens > INT32_MAX) return AIRCACHE_ERR_UNSUPPORTED;
  if (!p->cu_seqlens || !p->cu_visual || !p->q_text || !p->k || !p->v) return AIRCACHE_ERR_INVALID_ARG;
  const int es = esize_of(p->dtype);
  for (int l = 0; l < p->num_layers; ++l) {
    if (!p->q_text[l] || !p->k[l] || !p->v[l]) return AIRCACHE_ERR_INVALID_ARG;
    if (!aligned16(p->q_text[l]) || !aligned16(p->k[l]) || !aligned16(p->v[l])) return AIRCACHE_ERR_INVALID_ARG;
  }
  if ((p->variant & 0xff) == 4) {  // the visual window reads the visual tokens' queries
    if (!p->q_visual) return AIRCACHE_ERR_INVALID_ARG;
    for (int l = 0; l < p->num_layers; ++l)
      if (!p->q_visual[l] || !aligned16(p->q_visual[l])) return AIRCACHE_ERR_INVALID_ARG;
  }
  const int64_t strides[4] = {p->q_stride_tok, p->q_stride_head, p->kv_stride_tok, p->kv_stride_head};
  for (int64_t st : strides) {
    if (st <= 0 || (st * es) % 16 != 0) return AIRCACHE_ERR_INVALID_ARG;
  }
  if (p->q_stride_head < p->head_dim && p->h_q > 1) return AIRCACHE_ERR_INVALID_ARG;
  if (p->kv_stride_head < p->head_dim && p->h_kv > 1) return AIRCACHE_ERR_INVALID_ARG;
  if (!(p->alpha >= 0.0 && p->alpha <= 1.0)) return AIRCACHE_ERR_INVALID_ARG;
  if (!(p->r > 0.0 && p->r <= 1.0)) return AIRCACHE_ERR_INVALID_ARG;
  // elite-window kernel holds one query row and P in shared memory
  const size_t elite_fixed = sizeof(float) * ((size_t)p->h_q * p->head_dim + 3 * (size_t)p->max_text + 2);
  if (elite_fixed > 200 * 1024) return AIRCACHE_ERR_UNSUPPORTED;
  const int64_t max_elite = p->max_elite ? p->max_elite : p->max_text;
  if ((int64_t)p->h_q * max_elite > (1 << 30)) return AIRCACHE_ERR_UNSUPPORTED;
  return AIRCACHE_OK;
}

// Device description of a validated problem.
Dev make_dev(const aircache_problem* p) {
  Dev d;
  std::memset(&d, 0, sizeof d);
  d.L = p->num_layers;
  d.B = p->num_requests;
  d.h_q = p->h_q;
  d.h_kv = p->h_kv;
  d.d = p->head_dim;
  d.g = p->h_q / p->h_kv;
  d.dtype = p->dtype;
  d.max_visual = p->max_visual;
  d.max_text = p->max_text;
  d.max_elite = p->max_elite ? p->max_elite : p->max_text;
  if ((p->variant & 0xff) == 4) d.max_elite = p->max_visual < 32 ? p->max_visual : 32;  // the visual window's rows
  d.elite_stride = d.max_text > d.max_elite ? d.max_text : d.max_elite;
  d.rows_max = d.h_q * d.max_elite;
  d.rc_max = (d.g * d.max_elite + 31) / 32;
  d.lse_stride = d.h_kv * d.rc_max * 32;
  d.total_tokens = p->total_tokens;
  d.total_visual = p->total_visual;
  d.total_text = p->total_tokens - p->total_visual;
  d.cu_seqlens = p->cu_seqlens;
  d.cu_visual = p->cu_visual;
  d.n_prefix = p->n_prefix;
  d.q_stride_tok = p->q_stride_tok;
  d.q_stride_head = p->q_stride_head;
  d.kv_stride_tok = p->kv_stride_tok;
  d.kv_stride_head = p->kv_stride_head;
  d.alpha = p->alpha;
  d.r = p->r;
  d.window_mode = p->variant & 0xff;
  d.budget_mode = (p->variant >> 8) & 0xff;
  d.head_sets = (p->variant >> 16) & 0xff;
  d.wait_test = (p->variant & AIRCACHE_VARIANT_WAIT_TEST) ? 1 : 0;
  d.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p->head_dim));
  const int tv = (d.max_visual + 127) / 128;
  d.chn = (tv + kStreamTiles - 1) / kStreamTiles + 1;
  d.stream_ok = 0;  // set per call from stream_eligible()
  d.mom_slots = (d.max_visual + 127) / 128;
  return d;
}

LayerPtrs make_ptrs(const aircache_problem* p) {
  LayerPtrs lp;
  std::memset(&lp, 0, sizeof lp);
  for (int l = 0; l < p->num_layers; ++l) {
    lp.q[l] = p->q_text[l];
    lp.qv[l] = p->q_visual ? p->q_visual[l] : nullptr;
    lp.k[l] = p->k[l];
    lp.v[l] = p->v[l];
  }
  return lp;
}

// Carve the workspace; with base == nullptr only the size is computed.
size_t carve(const Dev& d, char* base, Ws* w) {
  const size_t LB = (size_t)d.L * d.B;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* ptr = base ? base + off : nullptr;
    off = align_up(off + bytes);
    return ptr;
  };
  Ws t;
  std::memset(&t, 0, sizeof t);
  // zeroed block: error, cnt_all, ticket, ticket_n, list_n[4], p2pack, cnt_cmp,
  // cnt_req[B], cnt_p1/cnt_p2/lse_ready/p2claim[L*B]
  const size_t zbytes = 52 + sizeof(uint32_t) * (d.B + 4 * LB);
  char* zero = take(zbytes);
  t.error = reinterpret_cast<int32_t*>(zero);
  t.cnt_all = reinterpret_cast<uint32_t*>(zero ? zero + 4 : nullptr);
  t.ticket = reinterpret_cast<unsigned long long*>(zero ? zero + 8 : nullptr);
  t.ticket_n = reinterpret_cast<unsigned long long*>(zero ? zero + 16 : nullptr);
  t.list_n = reinterpret_cast<int32_t*>(zero ? zero + 24 : nullptr);
  t.p2pack = reinterpret_cast<unsigned long long*>(zero ? zero + 40 : nullptr);
  t.cnt_cmp = reinterpret_cast<uint32_t*>(zero ? zero + 48 : nullptr);
  t.cnt_req = reinterpret_cast<uint32_t*>(zero ? zero + 52 : nullptr);
  t.cnt_p1 = t.cnt_req ? t.cnt_req + d.B : nullptr;
  t.cnt_p2 = t.cnt_p1 ? t.cnt_p1 + LB : nullptr;
  t.lse_ready = t.cnt_p2 ? t.cnt_p2 + LB : nullptr;
  t.p2claim = t.lse_ready ? t.lse_ready + LB : nullptr;
  t.zero_bytes = zbytes;
  const size_t T1 = (size_t)(d.max_visual + 127) / 128 + (size_t)(d.max_elite + 127) / 128;  // score tile slots
  const size_t G = (size_t)(d.h_kv + 3) / 4;
  t.elite = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * LB * d.elite_stride));
  t.n_tk = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * LB));
  t.stream_list = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * LB));
  t.stream_info = reinterpret_cast<int4*>(take(sizeof(int4) * 2 * LB));
  t.p2wpre = reinterpret_cast<uint32_t*>(take(sizeof(uint32_t) * LB));
  t.wide_list = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * LB));
  if (d.dtype == AIRCACHE_BF16) {  // the streaming path exists for bf16 only
    const size_t kvrows = (size_t)d.L * d.h_kv;
    // rows of the streaming path's logit buffer: every request's keys, each
    // request starting at a multiple of 4 columns (4 columns of padding per request)
    const size_t stride = (size_t)(d.total_visual + 4 * (int64_t)d.B + 7) / 4 * 4;
    t.lg = reinterpret_cast<float*>(take(sizeof(float) * kvrows * kLgRows * stride));
    t.mom = reinterpret_cast<float4*>(take(sizeof(float4) * 3 * LB * (size_t)d.mom_slots));
    t.lstat = reinterpret_cast<float4*>(take(sizeof(float4) * LB));
    t.part_s = reinterpret_cast<float2*>(take(sizeof(float2) * LB * d.h_kv * d.rc_max * kRowChunk * d.chn));
  }
  t.uinfo = reinterpret_cast<int4*>(take(sizeof(int4) * 2 * LB));
  const size_t esz = d.dtype == AIRCACHE_BF16 ? 2 : 4;
  t.qel = take(esz * LB * d.rows_max * d.d);
  t.kel = take(esz * LB * d.h_kv * d.max_elite * d.d);
  t.part = reinterpret_cast<float2*>(take(sizeof(float2) * LB * T1 * d.rows_max));
  t.lse = reinterpret_cast<float*>(take(sizeof(float) * LB * d.lse_stride));
  t.ivp = G > 1 ? reinterpret_cast<float*>(take(sizeof(float) * G * (size_t)d.L * d.total_visual)) : nullptr;
  t.iv = reinterpret_cast<float*>(take(sizeof(float) * (size_t)d.L * d.total_visual));
  t.stats = reinterpret_cast<double*>(take(sizeof(double) * 2 * LB));
  t.keep = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * LB));
  // one index set per (layer, request), or per (layer, KV head, request)
  const size_t sets = d.head_sets ? (size_t)d.h_kv : 1;
  t.idx = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * sets * (size_t)d.L * d.total_visual));
  t.ivh = d.head_sets ? reinterpret_cast<float*>(take(sizeof(float) * sets * (size_t)d.L * d.total_visual)) : nullptr;
  t.out_offsets = reinterpret_cast<int64_t*>(take(sizeof(int64_t) * (LB + 1)));
  if (w) *w = t;
  return off;
}

int check_ws(const aircache_problem* p, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return AIRCACHE_ERR_INVALID_ARG;
  if (ws_bytes < aircache_workspace_size(p)) return AIRCACHE_ERR_WORKSPACE;
  return AIRCACHE_OK;
}

#define AC_TRY(expr)                                 \
  do {                                               \
    if ((expr) != cudaSuccess) return AIRCACHE_ERR_CUDA; \
  } while (0)

// SMs of the current device (the persistent scoring grid is one CTA per SM).
int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 148;
  return sms;
}

// The scoring path of a validated problem (known on the host: see stream_eligible).
bool stream_path(const aircache_problem* p) { return stream_eligible(make_dev(p), make_ptrs(p)); }

// Clears the call's zeroed block (error word, counters, flags).  A kernel, not a
// memset: the call's next kernel is launched with programmatic serialization and
// sets up while this one runs; every kernel so launched waits for its
// predecessor (griddepcontrol.wait) before it touches the block.  Launched
// without that attribute itself, so it starts after everything queued before it.
__global__ void __launch_bounds__(256) zero_kernel(uint32_t* z, int n) {
  pdl_trigger();
  for (int i = blockIdx.x * 256 + threadIdx.x; i < n; i += gridDim.x * 256) z[i] = 0u;
}

int begin(const Ws& w, cudaStream_t s) {
  const int n = (int)(w.zero_bytes / sizeof(uint32_t));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(64, (n + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, zero_kernel, reinterpret_cast<uint32_t*>(w.error), n) == cudaSuccess
             ? AIRCACHE_OK
             : AIRCACHE_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t aircache_workspace_size(const aircache_problem* p) {
  if (validate(p) != AIRCACHE_OK) return 0;
  return carve(make_dev(p), nullptr, nullptr);
}

int64_t aircache_compress_bound(const aircache_problem* p) {
  if (validate(p) != AIRCACHE_OK) return -1;
  const int64_t L = p->num_layers, B = p->num_requests;
  const int64_t text = p->total_tokens - p->total_visual;
  const double vis = std::ceil(p->r * (double)L * (double)p->total_visual);
  int64_t bound = L * text + (int64_t)vis + B * (2 * L + 1);
  const int64_t cap = L * p->total_tokens;
  return bound < cap ? bound : cap;
}

int aircache_score(const aircache_problem* p, void* ws, size_t ws_bytes, float* iv, int32_t* elite,
                   int32_t* n_tk, void* stream) {
  int rc = validate(p);
  if (rc != AIRCACHE_OK) return rc;
  if ((rc = check_ws(p, ws, ws_bytes)) != AIRCACHE_OK) return rc;
  if (!iv || !elite || !n_tk) return AIRCACHE_ERR_INVALID_ARG;
  if (((p->variant >> 16) & 0xff) != 0) return AIRCACHE_ERR_UNSUPPORTED;  // per-head sets: aircache_compress only
  if ((p->variant & 0xff) == 4) return AIRCACHE_ERR_UNSUPPORTED;          // the visual window: aircache_compress only
  const Dev d = make_dev(p);
  const LayerPtrs lp = make_ptrs(p);
  Ws w;
  carve(d, static_cast<char*>(ws), &w);
  w.iv = iv;
  w.elite = elite;
  w.n_tk = n_tk;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  Dev dn = d;
  StreamMaps maps;
  dn.stream_ok = stream_eligible(d, lp) ? 1 : 0;
  if (dn.stream_ok && !encode_stream_maps(dn, lp, w, &maps)) return AIRCACHE_ERR_CUDA;
  if ((rc = begin(w, s)) != AIRCACHE_OK) return rc;
  AC_TRY(launch_elite(dn, lp, w, s));
  if (dn.stream_ok) {
    AC_TRY(launch_stream_p1(dn, maps, w, sms, s));
    AC_TRY(launch_stream_p2(dn, maps, w, sms, s));
    AC_TRY(launch_stream_p2k(dn, maps, w, sms, s));
  } else {
    AC_TRY(launch_score(dn, lp, w, plan_score(dn, sms, false, 0), s));
  }
  return AIRCACHE_OK;
}

int aircache_budget(const aircache_problem* p, const float* iv, void* ws, size_t ws_bytes, double* stats,
                    int32_t* keep, void* stream) {
  int rc = validate(p);
  if (rc != AIRCACHE_OK) return rc;
  if ((rc = check_ws(p, ws, ws_bytes)) != AIRCACHE_OK) return rc;
  if (!iv || !keep) return AIRCACHE_ERR_INVALID_ARG;
  const Dev d = make_dev(p);
  Ws w;
  carve(d, static_cast<char*>(ws), &w);
  w.iv = const_cast<float*>(iv);
  w.keep = keep;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = begin(w, s)) != AIRCACHE_OK) return rc;
  AC_TRY(launch_stats_budget(d, w, stats, 0, false, s));
  return AIRCACHE_OK;
}

int aircache_budget_noalloc(const aircache_problem* p, const float* iv, double* stats, int32_t* keep,
                            int32_t* device_status, void* stream) {
  int rc = validate(p);
  if (rc != AIRCACHE_OK) return rc;
  if (!iv || !keep) return AIRCACHE_ERR_INVALID_ARG;
  if ((int64_t)p->num_layers * p->num_requests > AIRCACHE_NOALLOC_MAX_UNITS) return AIRCACHE_ERR_UNSUPPORTED;
  return budget_noalloc(make_dev(p), iv, stats, keep, device_status, static_cast<cudaStream_t>(stream));
}

int aircache_select(const aircache_problem* p, const float* iv, const int32_t* keep, void* ws,
                    size_t ws_bytes, int32_t* idx, void* stream) {
  int rc = validate(p);
  if (rc != AIRCACHE_OK) return rc;
  if ((rc = check_ws(p, ws, ws_bytes)) != AIRCACHE_OK) return rc;
  if (!iv || !keep || !idx) return AIRCACHE_ERR_INVALID_ARG;
  if (((p->variant >> 16) & 0xff) != 0) return AIRCACHE_ERR_UNSUPPORTED;
  const Dev d = make_dev(p);
  Ws w;
  carve(d, static_cast<char*>(ws), &w);
  w.iv = const_cast<float*>(iv);
  w.keep = const_cast<int32_t*>(keep);
  w.idx = idx;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = begin(w, s)) != AIRCACHE_OK) return rc;
  AC_TRY(launch_select(d, w, s));
  return AIRCACHE_OK;
}

int aircache_compact(const aircache_problem* p, const int32_t* idx, const int32_t* keep, void* ws,
                     size_t ws_bytes, void* out_k, void* out_v, int64_t* out_offsets,
                     int64_t out_rows_capacity, void* stream) {
  int rc = validate(p);
  if (rc != AIRCACHE_OK) return rc;
  if ((rc = check_ws(p, ws, ws_bytes)) != AIRCACHE_OK) return rc;
  if (!idx || !keep || !out_k || !out_v || !out_offsets || out_rows_capacity < 0) return AIRCACHE_ERR_INVALID_ARG;
  if (!aligned16(out_k) || !aligned16(out_v)) return AIRCACHE_ERR_INVALID_ARG;
  if (((p->variant >> 16) & 0xff) != 0) return AIRCACHE_ERR_UNSUPPORTED;
  const Dev d = make_dev(p);
  const LayerPtrs lp = make_ptrs(p);
  Ws w;
  carve(d, static_cast<char*>(ws), &w);
  w.idx = const_cast<int32_t*>(idx);
  w.keep = const_cast<int32_t*>(keep);
  w.out_offsets = out_offsets;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = begin(w, s)) != AIRCACHE_OK) return rc;
  AC_TRY(launch_offsets(d, w, out_rows_capacity, s));
  AC_TRY(launch_compact(d, lp, w, out_k, out_v, out_rows_capacity, s));
  return AIRCACHE_OK;
}

int aircache_row_index(const aircache_problem* p, const int32_t* keep, const int32_t* idx,
                       const int64_t* out_offsets, void* ws, size_t ws_bytes, int32_t* row_index, int64_t capacity,
                       void* stream) {
  int rc = validate(p);
  if (rc != AIRCACHE_OK) return rc;
  if ((rc = check_ws(p, ws, ws_bytes)) != AIRCACHE_OK) return rc;
  if (!keep || !idx || !out_offsets || !row_index || capacity < 0) return AIRCACHE_ERR_INVALID_ARG;
  if (((p->variant >> 16) & 0xff) != 0) return AIRCACHE_ERR_UNSUPPORTED;  // one row list: one set per layer
  const Dev d = make_dev(p);
  const LayerPtrs lp = make_ptrs(p);
  Ws w;
  carve(d, static_cast<char*>(ws), &w);
  w.keep = const_cast<int32_t*>(keep);
  w.idx = const_cast<int32_t*>(idx);
  w.out_offsets = const_cast<int64_t*>(out_offsets);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = begin(w, s)) != AIRCACHE_OK) return rc;
  AC_TRY(launch_row_index(d, lp, w, row_index, capacity, s));
  return AIRCACHE_OK;
}

static int compress_impl(const aircache_problem* p, void* ws, size_t ws_bytes, void* out_k, void* out_v,
                         int64_t* out_offsets, int64_t out_rows_capacity, int32_t* keep, int32_t* idx,
                         float* iv, void* const* events, int n_events, void* stream) {
  int rc = validate(p);
  if (rc != AIRCACHE_OK) return rc;
  if ((rc = check_ws(p, ws, ws_bytes)) != AIRCACHE_OK) return rc;
  if (!out_k || !out_v || !out_offsets || !keep || out_rows_capacity < 0) return AIRCACHE_ERR_INVALID_ARG;
  if (!aligned16(out_k) || !aligned16(out_v)) return AIRCACHE_ERR_INVALID_ARG;
  const Dev d = make_dev(p);
  const LayerPtrs lp = make_ptrs(p);
  Dev dn = d;
  dn.stream_ok = stream_eligible(d, lp) ? 1 : 0;
  if (d.head_sets && !dn.stream_ok) return AIRCACHE_ERR_UNSUPPORTED;  // per-head sets: the streaming path only
  if (d.window_mode == 4 && !dn.stream_ok) return AIRCACHE_ERR_UNSUPPORTED;  // the visual window: likewise
  if (events && n_events != (dn.stream_ok ? kStreamCount : kWideCount) + 1) return AIRCACHE_ERR_INVALID_ARG;
  Ws w;
  carve(d, static_cast<char*>(ws), &w);
  w.keep = keep;
  w.out_offsets = out_offsets;
  if (idx) w.idx = idx;
  if (iv) w.iv = iv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto mark = [&](int i) {
    return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
  };
  const int sms = sm_count();
  StreamMaps maps;
  if (dn.stream_ok && !encode_stream_maps(dn, lp, w, &maps)) return AIRCACHE_ERR_CUDA;
  int k = 0;
  AC_TRY(mark(k++));
  if ((rc = begin(w, s)) != AIRCACHE_OK) return rc;
  AC_TRY(mark(k++));
  AC_TRY(launch_elite(dn, lp, w, s));
  AC_TRY(mark(k++));
  if (dn.stream_ok) {
    AC_TRY(launch_stream_p1(dn, maps, w, sms, s));
    AC_TRY(mark(k++));
    AC_TRY(launch_stream_p2(dn, maps, w, sms, s));
    AC_TRY(mark(k++));
    AC_TRY(launch_stream_p2k(dn, maps, w, sms, s));
    AC_TRY(mark(k++));
  } else {
    AC_TRY(launch_score(dn, lp, w, plan_score(dn, sms, true, out_rows_capacity), s));
    AC_TRY(mark(k++));
  }
  AC_TRY(launch_select(dn, w, s, dn.stream_ok != 0, out_rows_capacity));
  AC_TRY(mark(k++));
  AC_TRY(launch_compact(dn, lp, w, out_k, out_v, out_rows_capacity, s, dn.stream_ok != 0));
  AC_TRY(mark(k++));
  return AIRCACHE_OK;
}

int aircache_compress(const aircache_problem* p, void* ws, size_t ws_bytes, void* out_k, void* out_v,
                      int64_t* out_offsets, int64_t out_rows_capacity, int32_t* keep, int32_t* idx,
                      float* iv, void* stream) {
  return compress_impl(p, ws, ws_bytes, out_k, out_v, out_offsets, out_rows_capacity, keep, idx, iv,
                       nullptr, 0, stream);
}

int aircache_compress_profile(const aircache_problem* p, void* ws, size_t ws_bytes, void* out_k,
                              void* out_v, int64_t* out_offsets, int64_t out_rows_capacity,
                              int32_t* keep, int32_t* idx, float* iv, void* const* events,
                              int n_events, void* stream) {
  if (!events) return AIRCACHE_ERR_INVALID_ARG;
  return compress_impl(p, ws, ws_bytes, out_k, out_v, out_offsets, out_rows_capacity, keep, idx, iv,
                       events, n_events, stream);
}

// The problem with its query pointers and strides replaced by the full-prompt
// queries of the fused prefill.
static aircache_problem with_q_all(const aircache_problem* p, const void* const* q_all, int64_t qa_stride_tok,
                                   int64_t qa_stride_head) {
  aircache_problem pp = *p;
  pp.q_text = q_all;
  pp.q_stride_tok = qa_stride_tok;
  pp.q_stride_head = qa_stride_head;
  return pp;
}

static int prefill_checks(const aircache_problem* pp, const void* const* attn_out, int64_t o_stride_tok,
                          int64_t o_stride_head, void* ws, size_t ws_bytes) {
  int rc = validate(pp);
  if (rc != AIRCACHE_OK) return rc;
  if ((rc = check_ws(pp, ws, ws_bytes)) != AIRCACHE_OK) return rc;
  if (!attn_out) return AIRCACHE_ERR_INVALID_ARG;
  for (int l = 0; l < pp->num_layers; ++l)
    if (!attn_out[l] || !aligned16(attn_out[l])) return AIRCACHE_ERR_INVALID_ARG;
  if (o_stride_tok <= 0 || o_stride_head <= 0 || (o_stride_head < pp->head_dim && pp->h_q > 1))
    return AIRCACHE_ERR_INVALID_ARG;
  if (pp->variant != 0 || pp->n_prefix) return AIRCACHE_ERR_UNSUPPORTED;  // the method's own path only
  const Dev d = make_dev(pp);
  if (!prefill_eligible(d, make_ptrs(pp), pp->q_stride_tok, pp->q_stride_head, o_stride_tok, o_stride_head))
    return AIRCACHE_ERR_UNSUPPORTED;
  for (int l = 0; l < pp->num_layers; ++l) {  // the attention reads every value: device memory only
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, pp->v[l]) != cudaSuccess) {
      cudaGetLastError();
      return AIRCACHE_ERR_UNSUPPORTED;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return AIRCACHE_ERR_UNSUPPORTED;
  }
  return AIRCACHE_OK;
}

int aircache_prefill(const aircache_problem* p, const void* const* q_all, int64_t qa_stride_tok,
                     int64_t qa_stride_head, void* const* attn_out, int64_t o_stride_tok, int64_t o_stride_head,
                     void* ws, size_t ws_bytes, void* stream) {
  if (!p || !q_all) return AIRCACHE_ERR_INVALID_ARG;
  const aircache_problem pp = with_q_all(p, q_all, qa_stride_tok, qa_stride_head);
  int rc = prefill_checks(&pp, attn_out, o_stride_tok, o_stride_head, ws, ws_bytes);
  if (rc != AIRCACHE_OK) return rc;
  Dev d = make_dev(&pp);
  d.q_all = 1;
  const LayerPtrs lp = make_ptrs(&pp);
  Ws w;
  carve(d, static_cast<char*>(ws), &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = begin(w, s)) != AIRCACHE_OK) return rc;
  AC_TRY(launch_prefill(d, lp, w, qa_stride_tok, qa_stride_head, attn_out, o_stride_tok, o_stride_head,
                        pp.max_visual + pp.max_text, false, sm_count(), s));
  return AIRCACHE_OK;
}

int aircache_prefill_compress(const aircache_problem* p, const void* const* q_all, int64_t qa_stride_tok,
                              int64_t qa_stride_head, void* const* attn_out, int64_t o_stride_tok,
                              int64_t o_stride_head, void* ws, size_t ws_bytes, void* out_k, void* out_v,
                              int64_t* out_offsets, int64_t out_rows_capacity, int32_t* keep, int32_t* idx,
                              float* iv, void* stream) {
  if (!p || !q_all) return AIRCACHE_ERR_INVALID_ARG;
  const aircache_problem pp = with_q_all(p, q_all, qa_stride_tok, qa_stride_head);
  int rc = prefill_checks(&pp, attn_out, o_stride_tok, o_stride_head, ws, ws_bytes);
  if (rc != AIRCACHE_OK) return rc;
  if (!out_k || !out_v || !out_offsets || !keep || out_rows_capacity < 0) return AIRCACHE_ERR_INVALID_ARG;
  if (!aligned16(out_k) || !aligned16(out_v)) return AIRCACHE_ERR_INVALID_ARG;
  Dev dn = make_dev(&pp);
  dn.q_all = 1;
  const LayerPtrs lp = make_ptrs(&pp);
  if (!stream_eligible(dn, lp)) return AIRCACHE_ERR_UNSUPPORTED;
  dn.stream_ok = 1;
  Ws w;
  carve(dn, static_cast<char*>(ws), &w);
  w.keep = keep;
  w.out_offsets = out_offsets;
  if (idx) w.idx = idx;
  if (iv) w.iv = iv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  StreamMaps maps;
  if (!encode_stream_maps(dn, lp, w, &maps)) return AIRCACHE_ERR_CUDA;
  if ((rc = begin(w, s)) != AIRCACHE_OK) return rc;
  AC_TRY(launch_elite(dn, lp, w, s));
  AC_TRY(launch_prefill(dn, lp, w, qa_stride_tok, qa_stride_head, attn_out, o_stride_tok, o_stride_head,
                        pp.max_visual + pp.max_text, true, sms, s));
  AC_TRY(launch_stream_p2(dn, maps, w, sms, s));
  AC_TRY(launch_stream_p2k(dn, maps, w, sms, s));
  AC_TRY(launch_select(dn, w, s, true, out_rows_capacity));
  AC_TRY(launch_compact(dn, lp, w, out_k, out_v, out_rows_capacity, s, true));
  return AIRCACHE_OK;
}

const char* aircache_kernel_name(const aircache_problem* p, int i) {
  if (validate(p) != AIRCACHE_OK) return nullptr;
  if (stream_path(p)) return (i >= 0 && i < kStreamCount) ? kStreamKernels[i] : nullptr;
  return (i >= 0 && i < kWideCount) ? kWideKernels[i] : nullptr;
}

int aircache_compress_launches(const aircache_problem* p) {
  if (validate(p) != AIRCACHE_OK) return -1;
  return stream_path(p) ? kStreamCount : kWideCount;
}

int aircache_get_error(const void* ws, void* stream, int32_t* status) {
  if (!ws || !status) return AIRCACHE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return AIRCACHE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return AIRCACHE_ERR_CUDA;
  *status = v;
  return AIRCACHE_OK;
}

const char* aircache_status_string(int status) {
  switch (status) {
    case AIRCACHE_OK: return "ok";
    case AIRCACHE_ERR_INVALID_ARG: return "invalid argument";
    case AIRCACHE_ERR_UNSUPPORTED: return "unsupported problem";
    case AIRCACHE_ERR_WORKSPACE: return "workspace too small";
    case AIRCACHE_ERR_CUDA: return "CUDA launch or memset failed";
    case AIRCACHE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case AIRCACHE_ERR_DEVICE_BOUNDS: return "inconsistent request layout seen on the device";
    case AIRCACHE_ERR_ELITE_OVERFLOW: return "elite set larger than max_elite";
    case AIRCACHE_ERR_CAPACITY: return "output arena too small";
    default: return "unknown status";
  }
}

}  // extern "C"
