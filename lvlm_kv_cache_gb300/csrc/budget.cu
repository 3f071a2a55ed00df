// Layer budget (AirCache notes, "Key design 2": strength s_t, skewness s_k and
// r_hat = 1/2 (s'_t + s'_k) r).
//
// One CTA per (request, layer) reduces that layer's I_v in fp64 with a fixed
// reduction tree (deterministic): s_t = sum I_v, mu = s_t / N_v, the sample
// standard deviation sigma (n - 1) and
// s_k = N_v / ((N_v-1)(N_v-2)) * sum (I_v - mu)^3 / sigma^3  (0 when sigma = 0).
// The last layer of a request to finish (atomic arrival count) turns the
// request's L (s_t, s_k) pairs into keep counts:
//   s'_t = s_t / mean_l s_t            (1 if the mean is 0),
//   s'_k = (s_k - min_l s_k + 1e-6) / mean_l (s_k - min_l s_k + 1e-6),
//   r_l  = 1/2 (s'_t + s'_k) r,  keep_l = clamp(floor(r_l N_v + 1/2), 1, N_v),
// with the same operation order as a plain sequential evaluation and no fused
// multiply-adds, so the counts are reproducible bit for bit.  When asked, the
// last request to finish also writes the compacted-cache row offsets.
#include "internal.cuh"

namespace aircache {
namespace {

constexpr int kStatsThreads = 256;

struct StatsArgs {
  Dev p;
  Ws w;
  double* stats_out;      // optional caller copy of (s_t, s_k)
  int64_t out_capacity;   // rows of the output arena (offsets pass only)
  int offsets;            // 1: also write out_offsets
};

__device__ __forceinline__ double block_sum(double v, double* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int i = 0; i < kStatsThreads / 32; ++i) t += red[i];
  return t;
}

// out_offsets[u] for u = l*B + b: exclusive prefix of keep[u] + N_t[b]
// (one CTA; each thread scans a contiguous segment).
__device__ void write_offsets(const Dev& p, const Ws& w, int64_t capacity, long long* seg) {
  const int units = p.L * p.B;
  const int per = (units + kStatsThreads - 1) / kStatsThreads;
  const int u0 = threadIdx.x * per, u1 = min(units, u0 + per);
  long long local = 0;
  for (int u = u0; u < u1; ++u) {
    const int b = u % p.B;
    local += (long long)__ldcg(&w.keep[u]) + (p.cu_seqlens[b + 1] - p.cu_seqlens[b]) -
             (p.cu_visual[b + 1] - p.cu_visual[b]);
  }
  seg[threadIdx.x] = local;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long run = 0;
    for (int i = 0; i < kStatsThreads; ++i) {
      const long long v = seg[i];
      seg[i] = run;
      run += v;
    }
    w.out_offsets[units] = run;
    if (run > capacity) set_error(w.error, AIRCACHE_ERR_CAPACITY);
  }
  __syncthreads();
  long long run = seg[threadIdx.x];
  for (int u = u0; u < u1; ++u) {
    const int b = u % p.B;
    w.out_offsets[u] = run;
    run += (long long)__ldcg(&w.keep[u]) + (p.cu_seqlens[b + 1] - p.cu_seqlens[b]) -
           (p.cu_visual[b + 1] - p.cu_visual[b]);
  }
}

__global__ void __launch_bounds__(kStatsThreads) stats_budget_kernel(const __grid_constant__ StatsArgs a) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int b = blockIdx.x, l = blockIdx.y, u = l * p.B + b;
  const int tid = threadIdx.x;
  __shared__ double red[kStatsThreads / 32];
  __shared__ long long seg[kStatsThreads];
  __shared__ int flag, flag_all;
  if (*(volatile int32_t*)w.error != 0) return;
  Req R;
  if (!load_req(p, b, R)) {
    if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  const float* x = w.iv + (size_t)l * p.total_visual + R.vis0;
  const int n = R.n_v;

  double s = 0.0;
  for (int i = tid; i < n; i += kStatsThreads) s += (double)__ldcg(x + i);
  const double s_t = block_sum(s, red);
  const double mu = s_t / n;
  double m2 = 0.0;
  for (int i = tid; i < n; i += kStatsThreads) {
    const double dv = (double)__ldcg(x + i) - mu;
    m2 += dv * dv;
  }
  m2 = block_sum(m2, red);
  double m3 = 0.0;
  for (int i = tid; i < n; i += kStatsThreads) {
    const double dv = (double)__ldcg(x + i) - mu;
    m3 += dv * dv * dv;
  }
  m3 = block_sum(m3, red);
  const double sigma = sqrt(m2 / (n - 1));
  double s_k = 0.0;
  if (sigma > 0.0) s_k = (double)n / ((double)(n - 1) * (double)(n - 2)) * (m3 / (sigma * sigma * sigma));

  if (tid == 0) {
    w.stats[2 * u] = s_t;
    w.stats[2 * u + 1] = s_k;
    if (a.stats_out) {
      a.stats_out[2 * u] = s_t;
      a.stats_out[2 * u + 1] = s_k;
    }
    __threadfence();
    flag = (atomicAdd(&w.cnt_req[b], 1u) == (unsigned)(p.L - 1));
  }
  __syncthreads();
  if (!flag) return;

  // Last layer of request b: budgets of all its layers.
  if (tid == 0) {
    __threadfence();
    double mean_st = 0.0, min_sk = INFINITY;
    for (int ll = 0; ll < p.L; ++ll) {
      const int uu = ll * p.B + b;
      mean_st = __dadd_rn(mean_st, __ldcg(&w.stats[2 * uu]));
      min_sk = fmin(min_sk, __ldcg(&w.stats[2 * uu + 1]));
    }
    mean_st = __ddiv_rn(mean_st, (double)p.L);
    double mean_u = 0.0;
    for (int ll = 0; ll < p.L; ++ll) {
      const double sk = __ldcg(&w.stats[2 * (ll * p.B + b) + 1]);
      mean_u = __dadd_rn(mean_u, __dadd_rn(__dsub_rn(sk, min_sk), 1e-6));
    }
    mean_u = __ddiv_rn(mean_u, (double)p.L);
    for (int ll = 0; ll < p.L; ++ll) {
      const int uu = ll * p.B + b;
      const double st = __ldcg(&w.stats[2 * uu]);
      const double sk = __ldcg(&w.stats[2 * uu + 1]);
      const double st_n = (mean_st != 0.0) ? __ddiv_rn(st, mean_st) : 1.0;
      const double sk_n = __ddiv_rn(__dadd_rn(__dsub_rn(sk, min_sk), 1e-6), mean_u);
      const double rl = __dmul_rn(__dmul_rn(0.5, __dadd_rn(st_n, sk_n)), p.r);
      double kf = floor(__dadd_rn(__dmul_rn(rl, (double)n), 0.5));
      kf = fmin(fmax(kf, 1.0), (double)n);
      w.keep[uu] = (int32_t)kf;
    }
    __threadfence();
    flag_all = a.offsets ? (atomicAdd(w.cnt_all, 1u) == (unsigned)(p.B - 1)) : 0;
  }
  __syncthreads();
  if (!flag_all) return;
  __threadfence();
  write_offsets(p, w, a.out_capacity, seg);
}

// Stand-alone offsets (staged compaction): one CTA.
__global__ void __launch_bounds__(kStatsThreads) offsets_kernel(const __grid_constant__ StatsArgs a) {
  __shared__ long long seg[kStatsThreads];
  if (*(volatile int32_t*)a.w.error != 0) return;
  const Dev& p = a.p;
  // every request's lengths must be consistent before they size the arena
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
  write_offsets(p, a.w, a.out_capacity, seg);
}

}  // namespace

cudaError_t launch_stats_budget(const Dev& p, const Ws& w, double* stats_out, int64_t out_capacity,
                                bool offsets, cudaStream_t s) {
  StatsArgs a;
  a.p = p;
  a.w = w;
  a.stats_out = stats_out;
  a.out_capacity = out_capacity;
  a.offsets = offsets ? 1 : 0;
  stats_budget_kernel<<<dim3(p.B, p.L), kStatsThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_offsets(const Dev& p, const Ws& w, int64_t out_capacity, cudaStream_t s) {
  StatsArgs a;
  a.p = p;
  a.w = w;
  a.stats_out = nullptr;
  a.out_capacity = out_capacity;
  a.offsets = 1;
  offsets_kernel<<<1, kStatsThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace aircache
