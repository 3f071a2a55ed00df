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
// every thread gets the result.  `red` is shared scratch of NT/32 entries.
template <int NT>
__device__ __forceinline__ ff block_sum_ff(ff v, ff* red, int tix, int bar_id) {
  const int lane = tix & 31, warp = tix >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
  named_bar_sync(bar_id, NT);
  if (lane == 0) red[warp] = v;
  named_bar_sync(bar_id, NT);
  ff t = red[0];
#pragma unroll
  for (int i = 1; i < NT / 32; ++i) t = ff_add(t, red[i]);
  return t;
}

// (s_t, s_k) of x[0..n) (n >= 3), computed by NT threads whose index within the
// group is tix.  Returns the pair in every thread.  Each thread loads eight
// values before it adds any, so a pass costs n / (8 NT) memory round trips.
template <int NT>
__device__ __forceinline__ double2 unit_moments(const float* x, int n, int tix, ff* red, int bar_id) {
  constexpr int V = 8;
  ff s4[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  for (int i0 = tix; i0 < n; i0 += V * NT) {
    float v[V];
#pragma unroll
    for (int q = 0; q < V; ++q) v[q] = (i0 + q * NT < n) ? __ldcg(x + i0 + q * NT) : 0.f;
#pragma unroll
    for (int q = 0; q < V; ++q) s4[q & 3] = ff_add(s4[q & 3], ff{v[q], 0.f});
  }
  ff s = ff_add(ff_add(s4[0], s4[1]), ff_add(s4[2], s4[3]));
  s = block_sum_ff<NT>(s, red, tix, bar_id);
  const double s_t = ff_to_double(s);
  const ff mu = ff_from_double(s_t / n);
  ff m2q[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  ff m3q[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  for (int i0 = tix; i0 < n; i0 += V * NT) {
    float v[V];
#pragma unroll
    for (int q = 0; q < V; ++q) v[q] = (i0 + q * NT < n) ? __ldcg(x + i0 + q * NT) : 0.f;
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
  m2 = block_sum_ff<NT>(m2, red, tix, bar_id);
  m3 = block_sum_ff<NT>(m3, red, tix, bar_id);
  const double M2 = ff_to_double(m2), M3 = ff_to_double(m3);
  const double sigma = sqrt(M2 / (n - 1));
  double s_k = 0.0;
  if (sigma > 0.0) s_k = (double)n / ((double)(n - 1) * (double)(n - 2)) * (M3 / (sigma * sigma * sigma));
  return make_double2(s_t, s_k);
}

// Keep counts of request b from the (s_t, s_k) of its L layers (stats[2u],
// stats[2u+1], u = l*B + b):  s'_t = s_t/mean s_t (1 if the mean is 0),
// s'_k = (s_k - min s_k + 1e-6)/mean(.), r_l = 1/2 (s'_t + s'_k) r,
// keep = clamp(floor(r_l N_v + 1/2), 1, N_v).  The sums over layers run in
// layer order and no multiply-add is fused, as in a plain sequential
// evaluation.  NT threads; thread tix handles layers tix, tix+NT, ...
template <int NT>
__device__ __forceinline__ void request_budget(const Dev& p, int b, int n_v, const double* stats,
                                               int32_t* keep, double* sh, int tix, int bar_id) {
  if (tix == 0) {
    // loads are issued eight layers at a time; the sums still run in layer order
    double mean_st = 0.0, min_sk = INFINITY, mean_u = 0.0;
    for (int l0 = 0; l0 < p.L; l0 += 8) {
      double st[8], sk[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int u = (l0 + q) * p.B + b;
        st[q] = (l0 + q < p.L) ? __ldcg(&stats[2 * u]) : 0.0;
        sk[q] = (l0 + q < p.L) ? __ldcg(&stats[2 * u + 1]) : INFINITY;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (l0 + q < p.L) {
          mean_st = __dadd_rn(mean_st, st[q]);
          min_sk = fmin(min_sk, sk[q]);
        }
      }
    }
    mean_st = __ddiv_rn(mean_st, (double)p.L);
    for (int l0 = 0; l0 < p.L; l0 += 8) {
      double sk[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) sk[q] = (l0 + q < p.L) ? __ldcg(&stats[2 * ((l0 + q) * p.B + b) + 1]) : 0.0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (l0 + q < p.L) mean_u = __dadd_rn(mean_u, __dadd_rn(__dsub_rn(sk[q], min_sk), 1e-6));
      }
    }
    sh[0] = mean_st;
    sh[1] = min_sk;
    sh[2] = __ddiv_rn(mean_u, (double)p.L);
  }
  named_bar_sync(bar_id, NT);
  const double mean_st = sh[0], min_sk = sh[1], mean_u = sh[2];
  for (int l = tix; l < p.L; l += NT) {
    const int u = l * p.B + b;
    const double st = __ldcg(&stats[2 * u]);
    const double sk = __ldcg(&stats[2 * u + 1]);
    const double st_n = (mean_st != 0.0) ? __ddiv_rn(st, mean_st) : 1.0;
    const double sk_n = __ddiv_rn(__dadd_rn(__dsub_rn(sk, min_sk), 1e-6), mean_u);
    const double rl = __dmul_rn(__dmul_rn(0.5, __dadd_rn(st_n, sk_n)), p.r);
    double kf = floor(__dadd_rn(__dmul_rn(rl, (double)n_v), 0.5));
    kf = fmin(fmax(kf, 1.0), (double)n_v);
    keep[u] = (int32_t)kf;
  }
}

// out_offsets[u] (u = l*B + b): exclusive prefix over u of keep[u] + N_t[b];
// out_offsets[L*B] is the total.  Sets AIRCACHE_ERR_CAPACITY if the total
// exceeds `capacity`.  NT threads; `seg` is shared scratch of NT entries.
template <int NT>
__device__ __forceinline__ void write_offsets(const Dev& p, const int32_t* keep, int64_t* out_offsets,
                                              int32_t* err, int64_t capacity, long long* seg, int tix,
                                              int bar_id) {
  const int units = p.L * p.B;
  const int per = (units + NT - 1) / NT;
  const int u0 = tix * per, u1 = min(units, u0 + per);
  long long local = 0;
  for (int u = u0; u < u1; ++u) {
    const int b = u % p.B;
    local += (long long)__ldcg(&keep[u]) + (p.cu_seqlens[b + 1] - p.cu_seqlens[b]) -
             (p.cu_visual[b + 1] - p.cu_visual[b]);
  }
  seg[tix] = local;
  named_bar_sync(bar_id, NT);
  if (tix == 0) {
    long long run = 0;
    for (int i = 0; i < NT; ++i) {
      const long long v = seg[i];
      seg[i] = run;
      run += v;
    }
    out_offsets[units] = run;
    if (run > capacity) set_error(err, AIRCACHE_ERR_CAPACITY);
  }
  named_bar_sync(bar_id, NT);
  long long run = seg[tix];
  for (int u = u0; u < u1; ++u) {
    const int b = u % p.B;
    out_offsets[u] = run;
    run += (long long)__ldcg(&keep[u]) + (p.cu_seqlens[b + 1] - p.cu_seqlens[b]) -
           (p.cu_visual[b + 1] - p.cu_visual[b]);
  }
}

}  // namespace aircache
