// Elite observation window (AirCache notes, "Key design 1": equations Att and k).
//
// One CTA per (request, layer).  For every query head h the last text query is
// dotted with the N_t text keys of KV head h/g; each head's row is softmaxed in
// fp32 (base-2 logits, max-subtracted) and the rows are summed over heads into
// P (the head mean up to the common factor 1/H_q, which the threshold test does
// not see).  The elite set is {j : P[j] >= alpha * max P}, written in ascending
// order.  Heads are processed in chunks whose logits fit in shared memory.
#include "internal.cuh"

namespace aircache {
namespace {

constexpr int kEliteThreads = 256;

struct EliteArgs {
  Dev p;
  LayerPtrs lp;
  Ws w;
  int head_chunk;  // heads whose logits are held at once
};

template <typename T>
__device__ __forceinline__ float dot_row(const float* __restrict__ qs, const T* __restrict__ krow,
                                         int d);

template <>
__device__ __forceinline__ float dot_row<float>(const float* __restrict__ qs,
                                                const float* __restrict__ krow, int d) {
  float acc = 0.f;
  const float4* k4 = reinterpret_cast<const float4*>(krow);
  for (int i = 0; i < d / 4; ++i) {
    const float4 kv = __ldg(k4 + i);
    acc = fmaf(qs[4 * i + 0], kv.x, acc);
    acc = fmaf(qs[4 * i + 1], kv.y, acc);
    acc = fmaf(qs[4 * i + 2], kv.z, acc);
    acc = fmaf(qs[4 * i + 3], kv.w, acc);
  }
  return acc;
}

template <>
__device__ __forceinline__ float dot_row<__nv_bfloat16>(const float* __restrict__ qs,
                                                        const __nv_bfloat16* __restrict__ krow,
                                                        int d) {
  float acc = 0.f;
  const uint4* k4 = reinterpret_cast<const uint4*>(krow);
  for (int i = 0; i < d / 8; ++i) {
    const uint4 raw = __ldg(k4 + i);
    const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 kv = __bfloat1622float2(pr[j]);
      acc = fmaf(qs[8 * i + 2 * j], kv.x, acc);
      acc = fmaf(qs[8 * i + 2 * j + 1], kv.y, acc);
    }
  }
  return acc;
}

template <typename T>
__device__ __forceinline__ float to_float(T x);
template <>
__device__ __forceinline__ float to_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__global__ void __launch_bounds__(kEliteThreads) elite_kernel(const __grid_constant__ EliteArgs a) {
  const Dev& p = a.p;
  const int b = blockIdx.x, l = blockIdx.y;
  const int u = l * p.B + b;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kEliteThreads / 32;

  Req R;
  if (!load_req(p, b, R)) {
    if (tid == 0) set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  const int n_t = R.n_t, d = p.d, HC = a.head_chunk;

  extern __shared__ float smem[];
  float* qs = smem;                              // [h_q][d] last text query, fp32
  float* P = qs + p.h_q * d;                     // [max_text] sum over heads of softmax rows
  float* lg = P + p.max_text;                    // [HC][max_text] base-2 logits
  float* hmax = lg + (size_t)HC * p.max_text;    // [HC]
  float* hinv = hmax + HC;                       // [HC]
  __shared__ float red[kWarps];
  __shared__ int wcount[kWarps];

  const T* qbase = reinterpret_cast<const T*>(a.lp.q[l]);
  const T* qlast = qbase + (R.txt0 + n_t - 1) * p.q_stride_tok;
  for (int i = tid; i < p.h_q * d; i += kEliteThreads) {
    const int h = i / d, c = i % d;
    qs[i] = to_float<T>(qlast[h * p.q_stride_head + c]);
  }
  for (int j = tid; j < n_t; j += kEliteThreads) P[j] = 0.f;
  __syncthreads();

  const T* kbase = reinterpret_cast<const T*>(a.lp.k[l]);
  for (int h0 = 0; h0 < p.h_q; h0 += HC) {
    const int hc = min(HC, p.h_q - h0);
    for (int i = tid; i < hc * n_t; i += kEliteThreads) {
      const int hh = i / n_t, j = i % n_t;
      const int h = h0 + hh;
      const T* krow = kbase + (R.seq0 + R.n_v + j) * p.kv_stride_tok + (h / p.g) * p.kv_stride_head;
      lg[(size_t)hh * p.max_text + j] = dot_row<T>(qs + h * d, krow, d) * p.scale_log2;
    }
    __syncthreads();
    for (int hh = warp; hh < hc; hh += kWarps) {
      const float* row = lg + (size_t)hh * p.max_text;
      float m = -INFINITY;
      for (int j = lane; j < n_t; j += 32) m = fmaxf(m, row[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float s = 0.f;
      for (int j = lane; j < n_t; j += 32) s += exp2f(row[j] - m);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) {
        hmax[hh] = m;
        hinv[hh] = 1.f / s;
      }
    }
    __syncthreads();
    for (int j = tid; j < n_t; j += kEliteThreads) {
      float acc = P[j];
      for (int hh = 0; hh < hc; ++hh) acc += exp2f(lg[(size_t)hh * p.max_text + j] - hmax[hh]) * hinv[hh];
      P[j] = acc;
    }
    __syncthreads();
  }

  // max P
  float m = -INFINITY;
  for (int j = tid; j < n_t; j += kEliteThreads) m = fmaxf(m, P[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) m = fmaxf(m, red[i]);
  const float thr = (float)p.alpha * m;

  // ordered compaction of {j : P[j] >= thr}
  int32_t* out = a.w.elite + (size_t)u * p.max_text;
  int base = 0;
  for (int j0 = 0; j0 < n_t; j0 += kEliteThreads) {
    const int j = j0 + tid;
    const bool take = j < n_t && P[j] >= thr;
    const unsigned bal = __ballot_sync(0xffffffffu, take);
    const int before = __popc(bal & ((1u << lane) - 1u));
    __syncthreads();
    if (lane == 0) wcount[warp] = __popc(bal);
    __syncthreads();
    int wbase = 0, total = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      wbase += (i < warp) ? wcount[i] : 0;
      total += wcount[i];
    }
    const int pos = base + wbase + before;
    if (take && pos < p.max_elite) out[pos] = j;
    base += total;
  }
  if (tid == 0) {
    a.w.n_tk[u] = base;
    if (base > p.max_elite) set_error(a.w.error, AIRCACHE_ERR_ELITE_OVERFLOW);
  }
}

}  // namespace

cudaError_t launch_elite(const Dev& p, const LayerPtrs& lp, const Ws& w, cudaStream_t s) {
  EliteArgs a;
  a.p = p;
  a.lp = lp;
  a.w = w;
  const size_t budget = 96 * 1024;
  const size_t fixed = sizeof(float) * ((size_t)p.h_q * p.d + p.max_text);
  long long hc = (long long)((budget > fixed ? budget - fixed : 0) / sizeof(float)) / (p.max_text + 2);
  if (hc < 1) hc = 1;
  if (hc > p.h_q) hc = p.h_q;
  a.head_chunk = (int)hc;
  const size_t smem = fixed + sizeof(float) * (size_t)hc * (p.max_text + 2);
  dim3 grid(p.B, p.L);
  if (p.dtype == AIRCACHE_BF16) {
    cudaFuncSetAttribute(elite_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    elite_kernel<__nv_bfloat16><<<grid, kEliteThreads, smem, s>>>(a);
  } else {
    cudaFuncSetAttribute(elite_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    elite_kernel<float><<<grid, kEliteThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace aircache
