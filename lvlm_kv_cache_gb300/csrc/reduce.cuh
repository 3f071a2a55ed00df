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

__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }

// a / b for a float b: the rounded quotient of the leading part plus one
// correction from the exact remainder.
__device__ __forceinline__ ff ff_div_f(ff a, float b) {
  const float q1 = __fdiv_rn(a.hi, b);
  const ff r = ff_add(a, ff_neg(ff_mul(ff{q1, 0.f}, ff{b, 0.f})));
  return ff_fast_two_sum(q1, __fdiv_rn(r.hi, b));
}

// a / b: the quotient of the leading parts, then one correction from the
// remainder a - q b (formed exactly) — about 44 significant bits.
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  const float q1 = __fdividef(a.hi, b.hi);
  const ff r = ff_add(a, ff_neg(ff_mul(b, ff{q1, 0.f})));
  return ff_two_sum(q1, __fdividef(r.hi, b.hi));
}

// sqrt(a) for a >= 0: the float root s, then one Newton step s + (a - s^2) / 2s
// with the residual formed exactly.
__device__ __forceinline__ ff ff_sqrt(ff a) {
  if (!(a.hi > 0.f)) return {0.f, 0.f};
  const float s = sqrtf(a.hi);
  const ff r = ff_add(a, ff_neg(ff_mul(ff{s, 0.f}, ff{s, 0.f})));
  return ff_fast_two_sum(s, __fdividef(r.hi, 2.f * s));
}

// a < b for normalised values (|lo| at most half an ulp of hi).
__device__ __forceinline__ bool ff_lt(ff a, ff b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }

// floor(a) as a float (exact for |a| < 2^24): the floor of hi, one less when hi
// is an integer and lo is negative.
__device__ __forceinline__ float ff_floor(ff a) {
  const float f = floorf(a.hi);
  return (f == a.hi && a.lo < 0.f) ? f - 1.f : f;
}

// Sum over the 32 lanes of a warp (butterfly: every lane gets the same value,
// since ff_add is symmetric in its operands).
__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
  return v;
}

// The moments of a block of values, as one record: count n, the float-float
// sum and mean, the sums of squared and cubed deviations from the block mean
// (float-float), and the smallest and largest value (so that an all-equal set
// is recognised exactly).
struct Mom {
  float n;
  ff s, mean, m2, m3;
  float mn, mx;
};

// A record in global memory: three 16-byte words.
__device__ __forceinline__ void mom_store(float4* dst, const Mom& m) {
  dst[0] = make_float4(m.n, m.s.hi, m.s.lo, m.mn);
  dst[1] = make_float4(m.m2.hi, m.m2.lo, m.m3.hi, m.m3.lo);
  dst[2] = make_float4(m.mx, m.mean.hi, m.mean.lo, 0.f);
}
constexpr int kMomWords = 3;  // float4 words per record

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

// Sums of three float-float values over NT threads, fixed order (each warp by
// shuffles, then warp 0 over the warp totals); every thread gets the result.
// `red` is shared scratch of 3 * NT/32 entries.
template <int NT>
__device__ __forceinline__ void block_sum_ff3(ff& a, ff& b, ff& c, ff* red, int tix, int bar_id) {
  constexpr int NW = NT / 32;
  const int lane = tix & 31, warp = tix >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = ff_add(a, ff_shfl_xor(a, o));
    b = ff_add(b, ff_shfl_xor(b, o));
    c = ff_add(c, ff_shfl_xor(c, o));
  }
  named_bar_sync(bar_id, NT);  // earlier readers of red are done
  if (lane == 0) {
    red[warp] = a;
    red[NW + warp] = b;
    red[2 * NW + warp] = c;
  }
  named_bar_sync(bar_id, NT);
  if (warp == 0) {
    ff ta = lane < NW ? red[lane] : ff{0.f, 0.f};
    ff tb = lane < NW ? red[NW + lane] : ff{0.f, 0.f};
    ff tc = lane < NW ? red[2 * NW + lane] : ff{0.f, 0.f};
    // lanes >= NW hold zeros, and adding a zero float-float leaves a value
    // unchanged, so the butterfly starts at the highest level that pairs two
    // of the first NW lanes (lane 0 ends with the same sum)
#pragma unroll
    for (int o = NW / 2; o > 0; o >>= 1) {
      ta = ff_add(ta, ff_shfl_xor(ta, o));
      tb = ff_add(tb, ff_shfl_xor(tb, o));
      tc = ff_add(tc, ff_shfl_xor(tc, o));
    }
    if (lane == 0) {
      red[0] = ta;
      red[1] = tb;
      red[2] = tc;
    }
  }
  named_bar_sync(bar_id, NT);
  a = red[0];
  b = red[1];
  c = red[2];
}

// Moments of the values held by NT threads (each thread up to V values, valid
// where ok[i]; n = the number of valid values, n >= 1) in one pass: with a
// shift c near the values (any float; the same in every thread) the sums
// T_k = sum (x - c)^k, k = 1..3, are formed in float-float (x - c exactly),
// reduced once over the group, and turned into the central moments about the
// mean (q = T_1 / n):  M2 = T_2 - q T_1,  M3 = T_3 - 3 q T_2 + 2 q^2 T_1.
// The result is valid in thread tix == 0.  `red` is shared scratch of
// 3 * NT/32 ff, `redf` of 2 * NT/32 floats.
template <int NT, int V>
__device__ __forceinline__ Mom block_moments(const float (&x)[V], const bool (&ok)[V], float n, float c, ff* red,
                                             float* redf, int tix, int bar_id) {
  constexpr int NW = NT / 32;
  const int lane = tix & 31, warp = tix >> 5;
  ff t1{0.f, 0.f}, t2{0.f, 0.f}, t3{0.f, 0.f};
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    if (ok[i]) {
      const ff d = ff_two_sum(x[i], -c);  // exact
      const ff d2 = ff_mul(d, d);
      t1 = ff_add(t1, d);
      t2 = ff_add(t2, d2);
      t3 = ff_add(t3, ff_mul(d2, d));
      mn = fminf(mn, x[i]);
      mx = fmaxf(mx, x[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    redf[warp] = mn;
    redf[NW + warp] = mx;
  }
  block_sum_ff3<NT>(t1, t2, t3, red, tix, bar_id);  // its barriers also publish redf
  Mom r;
  r.n = n;
  if (tix == 0) {
    const ff q = ff_div_f(t1, n);
    r.s = ff_add(ff_mul(ff{n, 0.f}, ff{c, 0.f}), t1);
    r.mean = ff_add(ff{c, 0.f}, q);
    r.m2 = ff_add(t2, ff_neg(ff_mul(q, t1)));
    r.m3 = ff_add(ff_add(t3, ff_neg(ff_mul(ff_mul(ff{3.f, 0.f}, q), t2))), ff_mul(ff_mul(ff{2.f, 0.f}, ff_mul(q, q)), t1));
    r.mn = redf[0];
    r.mx = redf[NW];
    for (int i = 1; i < NW; ++i) {
      r.mn = fminf(r.mn, redf[i]);
      r.mx = fmaxf(r.mx, redf[NW + i]);
    }
  }
  return r;
}

// Sample skewness n / ((n-1)(n-2)) M3 / sigma^3, sigma^2 = M2 / (n-1), in
// float-float (n < 2^24, so n-1, n-2 and their product are exact); 0 for an
// all-equal set or sigma = 0.
__device__ __forceinline__ ff skew_ff(float n, ff m2, ff m3, bool all_equal) {
  if (all_equal) return {0.f, 0.f};
  const ff var = ff_div_f(m2, n - 1.f);
  if (!(var.hi > 0.f)) return {0.f, 0.f};
  const ff s3 = ff_mul(var, ff_sqrt(var));
  const ff den = ff_mul(s3, ff_mul(ff{n - 1.f, 0.f}, ff{n - 2.f, 0.f}));
  return ff_div(ff_mul(m3, ff{n, 0.f}), den);
}

// (s_t, s_k) of one (layer, request) from its block records rec[0..nslots),
// by one warp (every lane gets the result).  The union's moments about the
// overall mean mu: with delta_j = mean_j - mu,
//   M2 = sum_j M2_j + n_j delta_j^2,
//   M3 = sum_j M3_j + 3 delta_j M2_j + n_j delta_j^3
// (the block's own deviations sum to zero).  Lane j takes records j, j+32, ...;
// the lane totals are summed in a fixed butterfly order.
__device__ __forceinline__ void layer_stats_warp(const float4* rec, int nslots, int lane, ff& s_t, ff& s_k) {
  // records lane and lane + 32 are loaded once (all three words, up front) and
  // kept in registers for the second pass; any further ones are read twice
  float4 h0[2], h1[2], h2[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int j = lane + 32 * q;
    const bool ok = j < nslots;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    h0[q] = ok ? __ldcg(rec + (size_t)j * kMomWords) : z;
    h1[q] = ok ? __ldcg(rec + (size_t)j * kMomWords + 1) : z;
    h2[q] = ok ? __ldcg(rec + (size_t)j * kMomWords + 2) : z;
  }
  float n = 0.f, mn = INFINITY, mx = -INFINITY;
  ff s{0.f, 0.f};
  auto first = [&](const float4& w0, const float4& w2) {
    n += w0.x;  // integers below 2^24: exact
    s = ff_add(s, ff{w0.y, w0.z});
    mn = fminf(mn, w0.w);
    mx = fmaxf(mx, w2.x);
  };
#pragma unroll
  for (int q = 0; q < 2; ++q)
    if (lane + 32 * q < nslots) first(h0[q], h2[q]);
  for (int j = lane + 64; j < nslots; j += 32)
    first(__ldcg(rec + (size_t)j * kMomWords), __ldcg(rec + (size_t)j * kMomWords + 2));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n += __shfl_xor_sync(0xffffffffu, n, o);
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  s = warp_sum_ff(s);
  const ff mu = ff_div_f(s, n);
  ff m2{0.f, 0.f}, m3{0.f, 0.f};
  auto second = [&](const float4& w0, const float4& w1, const float4& w2) {
    const ff nj{w0.x, 0.f}, m2j{w1.x, w1.y}, m3j{w1.z, w1.w};
    const ff d = ff_add(ff{w2.y, w2.z}, ff_neg(mu));
    const ff nd2 = ff_mul(nj, ff_mul(d, d));
    m2 = ff_add(m2, ff_add(m2j, nd2));
    m3 = ff_add(m3, ff_add(m3j, ff_add(ff_mul(ff_mul(ff{3.f, 0.f}, d), m2j), ff_mul(nd2, d))));
  };
#pragma unroll
  for (int q = 0; q < 2; ++q)
    if (lane + 32 * q < nslots) second(h0[q], h1[q], h2[q]);
  for (int j = lane + 64; j < nslots; j += 32)
    second(__ldcg(rec + (size_t)j * kMomWords), __ldcg(rec + (size_t)j * kMomWords + 1),
           __ldcg(rec + (size_t)j * kMomWords + 2));
  m2 = warp_sum_ff(m2);
  m3 = warp_sum_ff(m3);
  s_t = s;
  s_k = skew_ff(n, m2, m3, !(mx > mn));
}

// Keep counts of request b from the (s_t, s_k) of its L layers, by one warp
// (lane j owns layers j, j+32, ...):  s'_t = s_t/mean s_t (1 if the mean is 0),
// s'_k = (s_k - min s_k + 1e-6)/mean(.), r_l = 1/2 (s'_t + s'_k) r,
// keep = clamp(floor(r_l N_v + 1/2), 1, N_v).  `get(l, st, sk)` yields layer
// l's pair.  Float-float throughout (about 44 significant bits per division:
// against an fp64 evaluation r_l N_v moves by ~1e-10 at most, which matters only
// within that distance of a half-integer); the layer sums are fixed-order
// butterflies, so the result is the same run to run.
template <typename Get, typename Put>
__device__ __forceinline__ void request_budget_warp_put(const Dev& p, int n_v, Get get, Put put, int lane) {
  // The loops over a lane's layers stay rolled (re-reading the pairs through
  // `get`): this runs once per request, so its code is usually cold in the
  // instruction cache and its size, not its arithmetic, sets the time.
  ff st_sum{0.f, 0.f}, sk_min{INFINITY, 0.f};
#pragma unroll 1
  for (int l = lane; l < p.L; l += 32) {
    ff st, sk;
    get(l, st, sk);
    st_sum = ff_add(st_sum, st);
    if (ff_lt(sk, sk_min)) sk_min = sk;
  }
  st_sum = warp_sum_ff(st_sum);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const ff t{__shfl_xor_sync(0xffffffffu, sk_min.hi, o), __shfl_xor_sync(0xffffffffu, sk_min.lo, o)};
    if (ff_lt(t, sk_min)) sk_min = t;
  }
  constexpr float kEpsHi = (float)1e-6;
  constexpr float kEpsLo = (float)(1e-6 - (double)kEpsHi);
  const ff eps{kEpsHi, kEpsLo};
  ff u_sum{0.f, 0.f};
#pragma unroll 1
  for (int l = lane; l < p.L; l += 32) {
    ff st, sk;
    get(l, st, sk);
    u_sum = ff_add(u_sum, ff_add(ff_add(sk, ff_neg(sk_min)), eps));  // u_l
  }
  u_sum = warp_sum_ff(u_sum);
  const ff mean_st = ff_div_f(st_sum, (float)p.L), mean_u = ff_div_f(u_sum, (float)p.L);
  const float r_hi = (float)p.r;
  const ff r{r_hi, (float)(p.r - (double)r_hi)};
#pragma unroll 1
  for (int l = lane; l < p.L; l += 32) {
    ff st, sk;
    get(l, st, sk);
    const ff u_l = ff_add(ff_add(sk, ff_neg(sk_min)), eps);
    float kf;
    if (p.budget_mode == 1 || p.budget_mode == 2) {
      // ablation budgets that do not look at the statistics (uniform; PyramidKV-
      // style, linear in depth from (2 - 1/20) r to r/20): fp64, in the oracle's
      // order of operations, so that structured values such as r N_v = x.5 round
      // the same way
      double rl = p.r;
      if (p.budget_mode == 2) {
        const double r_top = __ddiv_rn(p.r, 20.0);
        const double r_bottom = __dsub_rn(__dmul_rn(2.0, p.r), r_top);
        const double t = p.L > 1 ? __ddiv_rn((double)l, (double)(p.L - 1)) : 0.5;
        rl = __dadd_rn(r_bottom, __dmul_rn(__dsub_rn(r_top, r_bottom), t));
      }
      kf = (float)floor(__dadd_rn(__dmul_rn(rl, (double)n_v), 0.5));
    } else {
      const ff st_n = (mean_st.hi != 0.f) ? ff_div(st, mean_st) : ff{1.f, 0.f};
      const ff sk_n = ff_div(u_l, mean_u);
      // the method: 1/2 (s'_t + s'_k) r; ablations: s'_t r (3), s'_k r (4)
      const ff mix = p.budget_mode == 3 ? st_n
                     : p.budget_mode == 4 ? sk_n
                                          : ff_mul(ff{0.5f, 0.f}, ff_add(st_n, sk_n));
      const ff rl = ff_mul(mix, r);
      kf = ff_floor(ff_add(ff_mul(rl, ff{(float)n_v, 0.f}), ff{0.5f, 0.f}));
    }
    kf = fminf(fmaxf(kf, 1.f), (float)n_v);
    put(l, (int32_t)kf);
  }
}

// The same, writing keep[l * B + b].
template <typename Get>
__device__ __forceinline__ void request_budget_warp(const Dev& p, int b, int n_v, Get get, int32_t* keep,
                                                    int lane) {
  request_budget_warp_put(
      p, n_v, get, [&](int l, int32_t k) { keep[l * p.B + b] = k; }, lane);
}

// request_budget_warp over (s_t, s_k) pairs stored as doubles (stats[2u],
// stats[2u+1], u = l*B + b).
__device__ __forceinline__ void request_budget(const Dev& p, int b, int n_v, const double* stats,
                                               int32_t* keep, int lane) {
  request_budget_warp(
      p, b, n_v,
      [&](int l, ff& st, ff& sk) {
        st = ff_from_double(__ldcg(&stats[2 * (l * p.B + b)]));
        sk = ff_from_double(__ldcg(&stats[2 * (l * p.B + b) + 1]));
      },
      keep, lane);
}

// out_offsets[u] (u = l*B + b): exclusive prefix over u of keep[u] + N_t[b];
// out_offsets[L*B] is the total.  Sets AIRCACHE_ERR_CAPACITY if the total
// exceeds `capacity` (unless err is null).  NT threads (a multiple of 32, at most 1024); thread tix
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
    if (total > capacity && err) set_error(err, AIRCACHE_ERR_CAPACITY);
  }
}

}  // namespace aircache
