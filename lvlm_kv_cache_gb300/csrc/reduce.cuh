// Block-level reductions shared by the scoring kernel's tail and the stand-alone
// budget kernel: the moments of one layer's I_v (strength s_t and sample
// skewness s_k, AirCache notes "Key design 2"), the per-request layer budget,
// and the compacted-cache row offsets.
//
// The moments use float-float ("double-single") arithmetic: each value is an
// unevaluated sum hi + lo of two floats, added with Knuth's two-sum and
// multiplied with an FMA-based exact product (Dekker), which carries ~48
// significant bits on the fp32 pipes.  GB300's fp64 pipe is far narrower than
// its fp32 pipes, so fp64 is used only for the handful of scalar operations at
// the end.  Every reduction runs in a fixed order, so results are identical run
// to run.
#pragma once

#include "internal.cuh"
#include "ptx.cuh"

namespace aircache {

struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff ff_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

__device__ __forceinline__ ff ff_fast_two_sum(float a, float b) {  // requires |a| >= |b| or a == 0
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = ff_two_sum(a.hi, b.hi);
  const ff t = ff_two_sum(a.lo, b.lo);
  s.lo = __fadd_rn(s.lo, t.hi);
  s = ff_fast_two_sum(s.hi, s.lo);
  s.lo = __fadd_rn(s.lo, t.lo);
  return ff_fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.hi, -p);
  e = __fmaf_rn(a.hi, b.lo, e);
  e = __fmaf_rn(a.lo, b.hi, e);
  return ff_fast_two_sum(p, e);
}

__device__ __forceinline__ double ff_to_double(ff a) { return (double)a.hi + (double)a.lo; }

__device__ __forceinline__ ff ff_from_double(double x) {
  const float hi = (float)x;
  return {hi, (float)(x - (double)hi)};
}

__device__ __forceinline__ ff ff_shfl_xor(ff a, int o) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}

// Sum over NT threads (all of them call it, tix = index within the group);
// every thread gets the result.  Each warp reduces with shuffles, then warp 0
// reduces the warp totals the same way: a fixed order, so the result is the
// same run to run.  `red` is shared scratch of NT/32 entries (2 * NT/32 for the
// pair version).
template <int NT>
__device__ __forceinline__ ff block_sum_ff(ff v, ff* red, int tix, int bar_id) {
  constexpr int NW = NT / 32;
  const int lane = tix & 31, warp = tix >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
  named_bar_sync(bar_id, NT);  // earlier readers of red are done
  if (lane == 0) red[warp] = v;
  named_bar_sync(bar_id, NT);
  if (warp == 0) {
    ff t = lane < NW ? red[lane] : ff{0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = ff_add(t, ff_shfl_xor(t, o));
    if (lane == 0) red[0] = t;
  }
  named_bar_sync(bar_id, NT);
  return red[0];
}

template <int NT>
__device__ __forceinline__ void block_sum_ff2(ff& a, ff& b, ff* red, int tix, int bar_id) {
  constexpr int NW = NT / 32;
  const int lane = tix & 31, warp = tix >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = ff_add(a, ff_shfl_xor(a, o));
    b = ff_add(b, ff_shfl_xor(b, o));
  }
  named_bar_sync(bar_id, NT);
  if (lane == 0) {
    red[warp] = a;
    red[NW + warp] = b;
  }
  named_bar_sync(bar_id, NT);
  if (warp == 0) {
    ff ta = lane < NW ? red[lane] : ff{0.f, 0.f};
    ff tb = lane < NW ? red[NW + lane] : ff{0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ta = ff_add(ta, ff_shfl_xor(ta, o));
      tb = ff_add(tb, ff_shfl_xor(tb, o));
    }
    if (lane == 0) {
      red[0] = ta;
      red[1] = tb;
    }
  }
  named_bar_sync(bar_id, NT);
  a = red[0];
  b = red[1];
}

// (s_t, s_k) of x[0..n) (n >= 3), computed by NT threads whose index within the
// group is tix; the result is valid in thread tix == 0 only.  `red` is shared
// scratch of 2 * NT/32 + 1 entries.  Each thread loads eight values before it adds
// any, so a pass costs n / (8 NT) memory round trips; the few fp64 scalar steps
// run in one thread (GB300's fp64 rate is a small fraction of its fp32 rate).
template <int NT>
__device__ __forceinline__ double2 unit_moments(const float* x, int n, int tix, ff* red, int bar_id) {
  constexpr int V = 8;
  ff s4[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  float v0[V];  // the first V values of this thread, kept for the second pass
#pragma unroll
  for (int q = 0; q < V; ++q) v0[q] = (tix + q * NT < n) ? __ldcg(x + tix + q * NT) : 0.f;
#pragma unroll
  for (int q = 0; q < V; ++q) s4[q & 3] = ff_add(s4[q & 3], ff{v0[q], 0.f});
  for (int i0 = tix + V * NT; i0 < n; i0 += V * NT) {
    float v[V];
#pragma unroll
    for (int q = 0; q < V; ++q) v[q] = (i0 + q * NT < n) ? __ldcg(x + i0 + q * NT) : 0.f;
#pragma unroll
    for (int q = 0; q < V; ++q) s4[q & 3] = ff_add(s4[q & 3], ff{v[q], 0.f});
  }
  ff s = ff_add(ff_add(s4[0], s4[1]), ff_add(s4[2], s4[3]));
  s = block_sum_ff<NT>(s, red, tix, bar_id);
  double s_t = 0.0;
  if (tix == 0) {
    s_t = ff_to_double(s);
    red[2 * (NT / 32)] = ff_from_double(s_t / n);  // the mean, for every thread
  }
  named_bar_sync(bar_id, NT);
  const ff mu = red[2 * (NT / 32)];
  ff m2q[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  ff m3q[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  for (int i0 = tix; i0 < n; i0 += V * NT) {
    float v[V];
#pragma unroll
    for (int q = 0; q < V; ++q) {
      v[q] = (i0 == tix) ? v0[q] : ((i0 + q * NT < n) ? __ldcg(x + i0 + q * NT) : 0.f);
    }
#pragma unroll
    for (int q = 0; q < V; ++q) {
      if (i0 + q * NT < n) {
        ff d = ff_two_sum(v[q], -mu.hi);
        d = ff_two_sum(d.hi, __fsub_rn(d.lo, mu.lo));
        const ff d2 = ff_mul(d, d);
        m2q[q & 3] = ff_add(m2q[q & 3], d2);
        m3q[q & 3] = ff_add(m3q[q & 3], ff_mul(d2, d));
      }
    }
  }
  ff m2 = ff_add(ff_add(m2q[0], m2q[1]), ff_add(m2q[2], m2q[3]));
  ff m3 = ff_add(ff_add(m3q[0], m3q[1]), ff_add(m3q[2], m3q[3]));
  block_sum_ff2<NT>(m2, m3, red, tix, bar_id);
  double s_k = 0.0;
  if (tix == 0) {
    const double M2 = ff_to_double(m2), M3 = ff_to_double(m3);
    const double sigma = sqrt(M2 / (n - 1));
    if (sigma > 0.0) s_k = (double)n / ((double)(n - 1) * (double)(n - 2)) * (M3 / (sigma * sigma * sigma));
  }
  return make_double2(s_t, s_k);
}

// Keep counts of request b from the (s_t, s_k) of its L layers (stats[2u],
// stats[2u+1], u = l*B + b):  s'_t = s_t/mean s_t (1 if the mean is 0),
// s'_k = (s_k - min s_k + 1e-6)/mean(.), r_l = 1/2 (s'_t + s'_k) r,
// keep = clamp(floor(r_l N_v + 1/2), 1, N_v).  NT threads; thread tix owns
// layers tix, tix+NT, ...  The two sums over layers run as fixed-order
// float-float reductions (about 48 significant bits: a different summation
// order than a sequential fp64 loop changes r_l N_v by ~1e-13 at most, which
// matters only within that distance of a half-integer); the per-layer steps
// run in fp64, one layer per thread.  `sh` is shared scratch of
// 2 * NT/32 + 4 doubles.
template <int NT>
__device__ __forceinline__ void request_budget(const Dev& p, int b, int n_v, const double* stats,
                                               int32_t* keep, double* sh, int tix, int bar_id) {
  constexpr int NW = NT / 32;
  constexpr int kMaxOwn = (AIRCACHE_MAX_LAYERS + NT - 1) / NT;
  static_assert(sizeof(ff) <= sizeof(double), "ff scratch overlays the double scratch");
  const int lane = tix & 31, warp = tix >> 5;
  ff* red = reinterpret_cast<ff*>(sh);
  double st[kMaxOwn], sk[kMaxOwn];
  ff st_sum{0.f, 0.f};
  double sk_min = INFINITY;
#pragma unroll
  for (int j = 0; j < kMaxOwn; ++j) {
    const int l = tix + j * NT;
    st[j] = l < p.L ? __ldcg(&stats[2 * (l * p.B + b)]) : 0.0;
    sk[j] = l < p.L ? __ldcg(&stats[2 * (l * p.B + b) + 1]) : INFINITY;
  }
#pragma unroll
  for (int j = 0; j < kMaxOwn; ++j) {
    st_sum = ff_add(st_sum, ff_from_double(st[j]));
    sk_min = fmin(sk_min, sk[j]);
  }
  // minimum of s_k: exact (a min is order-free); shuffled as two 32-bit halves
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sk_min = fmin(sk_min, __shfl_xor_sync(0xffffffffu, sk_min, o));
  st_sum = block_sum_ff<NT>(st_sum, red, tix, bar_id);
  named_bar_sync(bar_id, NT);  // everyone has read red[0]
  if (lane == 0) sh[NW + warp] = sk_min;
  named_bar_sync(bar_id, NT);
  if (warp == 0) {
    double m = lane < NW ? sh[NW + lane] : INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmin(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) sh[2 * NW + 1] = m;
  }
  named_bar_sync(bar_id, NT);
  const double min_sk = sh[2 * NW + 1];
  ff u_sum{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kMaxOwn; ++j) {
    if (tix + j * NT < p.L) u_sum = ff_add(u_sum, ff_from_double(__dadd_rn(__dsub_rn(sk[j], min_sk), 1e-6)));
  }
  u_sum = block_sum_ff<NT>(u_sum, red, tix, bar_id);
  if (tix == 0) {
    sh[2 * NW + 2] = __ddiv_rn(ff_to_double(st_sum), (double)p.L);
    sh[2 * NW + 3] = __ddiv_rn(ff_to_double(u_sum), (double)p.L);
  }
  named_bar_sync(bar_id, NT);
  const double mean_st = sh[2 * NW + 2], mean_u = sh[2 * NW + 3];
#pragma unroll
  for (int j = 0; j < kMaxOwn; ++j) {
    const int l = tix + j * NT;
    if (l < p.L) {
      const double st_n = (mean_st != 0.0) ? __ddiv_rn(st[j], mean_st) : 1.0;
      const double sk_n = __ddiv_rn(__dadd_rn(__dsub_rn(sk[j], min_sk), 1e-6), mean_u);
      const double rl = __dmul_rn(__dmul_rn(0.5, __dadd_rn(st_n, sk_n)), p.r);
      double kf = floor(__dadd_rn(__dmul_rn(rl, (double)n_v), 0.5));
      kf = fmin(fmax(kf, 1.0), (double)n_v);
      keep[l * p.B + b] = (int32_t)kf;
    }
  }
}

// out_offsets[u] (u = l*B + b): exclusive prefix over u of keep[u] + N_t[b];
// out_offsets[L*B] is the total.  Sets AIRCACHE_ERR_CAPACITY if the total
// exceeds `capacity`.  NT threads (a multiple of 32, at most 1024); thread tix
// owns a contiguous run of units; the per-thread totals are scanned with warp
// shuffles.  `seg` is shared scratch of NT/32 + 1 entries.
template <int NT>
__device__ __forceinline__ void write_offsets(const Dev& p, const int32_t* keep, int64_t* out_offsets,
                                              int32_t* err, int64_t capacity, long long* seg, int tix,
                                              int bar_id) {
  constexpr int NW = NT / 32;
  const int lane = tix & 31, warp = tix >> 5;
  const int units = p.L * p.B;
  const int per = (units + NT - 1) / NT;
  const int u0 = tix * per, u1 = min(units, u0 + per);
  long long local = 0;
  for (int u = u0; u < u1; ++u) {
    const int b = u % p.B;
    local += (long long)__ldcg(&keep[u]) + (p.cu_seqlens[b + 1] - p.cu_seqlens[b]) -
             (p.cu_visual[b + 1] - p.cu_visual[b]);
  }
  long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) seg[warp] = incl;
  named_bar_sync(bar_id, NT);
  if (warp == 0) {
    long long t = lane < NW ? seg[lane] : 0;
    long long ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += v;
    }
    if (lane < NW) seg[lane] = ti - t;  // exclusive prefix of the warp totals
    if (lane == 31) seg[NW] = ti;       // grand total
  }
  named_bar_sync(bar_id, NT);
  long long run = seg[warp] + incl - local;
  for (int u = u0; u < u1; ++u) {
    const int b = u % p.B;
    out_offsets[u] = run;
    run += (long long)__ldcg(&keep[u]) + (p.cu_seqlens[b + 1] - p.cu_seqlens[b]) -
           (p.cu_visual[b + 1] - p.cu_visual[b]);
  }
  if (tix == 0) {
    const long long total = seg[NW];
    out_offsets[units] = total;
    if (total > capacity) set_error(err, AIRCACHE_ERR_CAPACITY);
  }
}

}  // namespace aircache
