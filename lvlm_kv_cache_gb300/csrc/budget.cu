// Layer budget (AirCache notes, "Key design 2": strength s_t, skewness s_k and
// r_hat = 1/2 (s'_t + s'_k) r) as a stand-alone stage over a given I_v.
//
// One CTA per (request, layer) computes that layer's (s_t, s_k) (float-float
// moments, see reduce.cuh); the CTA finishing a request's last layer (atomic
// arrival count) computes the request's keep counts, and in the fused
// compression the CTA finishing the last request writes the compacted-cache
// row offsets.  The wide scoring kernel computes the same quantities at its
// tail with the same device functions.  A separate one-CTA kernel writes the
// offsets for the staged compaction.  (On the streaming scoring path of the
// fused call passes 2 and 2k merge each unit's key-block moment records into
// its statistics, and the selection kernel derives the budgets from them:
// stream.cu, select.cu.)
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.cuh"
#include "ptx.cuh"
#include "reduce.cuh"

namespace aircache {
namespace {

constexpr int kStatsThreads = 256;   // stand-alone offsets kernel
constexpr int kTailThreads = 1024;   // one (layer, request) per CTA: one load round per moment pass
constexpr int kBarAll = 1;

struct StatsArgs {
  Dev p;
  Ws w;
  double* stats_out;      // optional caller copy of (s_t, s_k)
  int64_t out_capacity;   // rows of the output arena (offsets kernel only)
};

// (s_t, s_k) of one (layer, request) per CTA; the CTA finishing a request's
// last layer computes its keep counts; with OFFSETS, the CTA finishing the
// last request writes the compacted-cache row offsets.
template <int NT, bool OFFSETS>
__global__ void __launch_bounds__(NT) stats_budget_kernel(const __grid_constant__ StatsArgs a) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int b = blockIdx.x, l = blockIdx.y, u = l * p.B + b;
  const int tid = threadIdx.x;
  __shared__ ff redff[2 * (NT / 32) + 1];
  __shared__ long long seg[NT / 32 + 1];
  __shared__ int flag;
  pdl_trigger();
  pdl_wait();  // I_v
  if (*(volatile int32_t*)w.error != 0) return;
  Req R;
  const bool ok = load_req(p, b, R);
  if (ok) {
    const float* x = w.iv + (size_t)l * p.total_visual + R.vis0;
    const double2 m = unit_moments<NT>(x, R.n_v, tid, redff, kBarAll);
    if (tid == 0) {
      w.stats[2 * u] = m.x;
      w.stats[2 * u + 1] = m.y;
      if (a.stats_out) {
        a.stats_out[2 * u] = m.x;
        a.stats_out[2 * u + 1] = m.y;
      }
    }
  } else if (tid == 0) {
    set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
  }
  // every CTA arrives, also after an error, so that the request's last CTA
  // always runs and its keep counts are always written
  if (tid == 0) {
    __threadfence();
    flag = (atomicAdd(&w.cnt_req[b], 1u) == (unsigned)(p.L - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!flag) return;
  __threadfence();
  if (!ok || *(volatile int32_t*)w.error != 0) {
    // an inconsistent layout: the request's keep counts are 0 (the error word says why)
    for (int ll = tid; ll < p.L; ll += NT) w.keep[ll * p.B + b] = 0;
    return;
  }
  if (tid < 32) request_budget(p, b, R.n_v, w.stats, w.keep, tid);
  if constexpr (OFFSETS) {
    __threadfence();
    __syncthreads();
    if (tid == 0) flag = (atomicAdd(w.cnt_all, 1u) == (unsigned)(p.B - 1)) ? 1 : 0;
    __syncthreads();
    if (!flag) return;
    __threadfence();
    write_offsets<NT>(p, w.keep, w.out_offsets, w.error, a.out_capacity, seg, tid, kBarAll);
  }
}

// Stand-alone offsets (staged compaction): one CTA.
__global__ void __launch_bounds__(kStatsThreads) offsets_kernel(const __grid_constant__ StatsArgs a) {
  __shared__ long long seg[kStatsThreads];
  pdl_trigger();
  pdl_wait();
  if (*(volatile int32_t*)a.w.error != 0) return;
  const Dev& p = a.p;
  // every request's lengths and keep counts must be consistent before they size the arena
  for (int b = threadIdx.x; b < p.B; b += kStatsThreads) {
    Req R;
    if (!load_req(p, b, R)) set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
  }
  for (int u = threadIdx.x; u < p.L * p.B; u += kStatsThreads) {
    const int b = u % p.B;
    const int nv = p.cu_visual[b + 1] - p.cu_visual[b];
    const int k = a.w.keep[u];
    if (k < 0 || k > nv) set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  if (*(volatile int32_t*)a.w.error != 0) return;
  write_offsets<kStatsThreads>(p, a.w.keep, a.w.out_offsets, a.w.error, a.out_capacity, seg, threadIdx.x,
                               kBarAll);
}

// ---------------------------------------------------------------- fixed scratch
// Scratch of aircache_budget_noalloc, part of the module's device memory: the
// error word, one arrival counter per request and the (s_t, s_k) of every
// (layer, request), for at most AIRCACHE_NOALLOC_MAX_UNITS layer-request pairs.
// The error word and the counters must be 0 when the kernel starts; every call
// clears them on its stream first.  One copy per device, shared by every call
// in the process.
constexpr size_t kNaCntOff = 256;
constexpr size_t kNaStatsOff = kNaCntOff + sizeof(uint32_t) * AIRCACHE_NOALLOC_MAX_UNITS;
constexpr size_t kNaBytes = kNaStatsOff + 2 * sizeof(double) * AIRCACHE_NOALLOC_MAX_UNITS;
static_assert(kNaStatsOff % 256 == 0, "stats block alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaBytes];

// The scratch address belongs to the context in which the module was loaded:
// the cache is keyed on the driver's unique id of the current context, so a new
// context (after cudaDeviceReset, or a second context that a driver-API caller
// made current) looks the address up again instead of using a stale one.
struct NaEntry {
  unsigned long long ctx_id;
  char* addr;
};
std::mutex g_na_mutex;
std::vector<NaEntry> g_na_cache;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the current context (0 with none current, or where the driver lacks the call).
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch in the current context; looked up once per
// context (the lookup may load the module and make the device's primary
// context current), then cached under that context's id.
int noalloc_scratch(char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return AIRCACHE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  unsigned long long id = current_ctx_id();
  if (id != 0) {
    for (const NaEntry& e : g_na_cache) {
      if (e.ctx_id == id) {
        *out = e.addr;
        return AIRCACHE_OK;
      }
    }
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return AIRCACHE_ERR_CUDA;
  if (id == 0) id = current_ctx_id();  // the lookup made a context current
  if (id != 0) g_na_cache.push_back(NaEntry{id, static_cast<char*>(ptr)});
  *out = static_cast<char*>(ptr);
  return AIRCACHE_OK;
}

}  // namespace

int budget_noalloc(const Dev& p, const float* iv, double* stats_out, int32_t* keep, int32_t* device_status,
                   cudaStream_t s) {
  if ((long long)p.L * p.B > AIRCACHE_NOALLOC_MAX_UNITS) return AIRCACHE_ERR_UNSUPPORTED;
  char* base = nullptr;
  int rc = noalloc_scratch(&base);
  if (rc != AIRCACHE_OK) return rc;
  if (cudaMemsetAsync(base, 0, kNaCntOff + sizeof(uint32_t) * p.B, s) != cudaSuccess) return AIRCACHE_ERR_CUDA;
  StatsArgs a;
  std::memset(&a, 0, sizeof a);
  a.p = p;
  a.w.error = reinterpret_cast<int32_t*>(base);
  a.w.cnt_req = reinterpret_cast<uint32_t*>(base + kNaCntOff);
  a.w.stats = reinterpret_cast<double*>(base + kNaStatsOff);
  a.w.iv = const_cast<float*>(iv);
  a.w.keep = keep;
  a.stats_out = stats_out;
  a.out_capacity = 0;
  // the same kernel and block size as aircache_budget: the same reduction order
  stats_budget_kernel<kTailThreads, false><<<dim3(p.B, p.L), kTailThreads, 0, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return AIRCACHE_ERR_CUDA;
  if (device_status &&
      cudaMemcpyAsync(device_status, base, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess) {
    return AIRCACHE_ERR_CUDA;
  }
  return AIRCACHE_OK;
}

cudaError_t launch_stats_budget(const Dev& p, const Ws& w, double* stats_out, int64_t out_capacity,
                                bool offsets, cudaStream_t s) {
  StatsArgs a;
  a.p = p;
  a.w = w;
  a.stats_out = stats_out;
  a.out_capacity = out_capacity;
  return offsets ? launch_pdl(stats_budget_kernel<kTailThreads, true>, dim3(p.B, p.L), dim3(kTailThreads), 0, s, a)
                 : launch_pdl(stats_budget_kernel<kTailThreads, false>, dim3(p.B, p.L), dim3(kTailThreads), 0, s, a);
}

cudaError_t launch_offsets(const Dev& p, const Ws& w, int64_t out_capacity, cudaStream_t s) {
  StatsArgs a;
  a.p = p;
  a.w = w;
  a.stats_out = nullptr;
  a.out_capacity = out_capacity;
  return launch_pdl(offsets_kernel, dim3(1), dim3(kStatsThreads), 0, s, a);
}

}  // namespace aircache
