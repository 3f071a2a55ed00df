// int8 storage of a compacted cache (LLM KV-compression notes, "Quantization
// stacked on compression": quantise after the token compression, one scale per
// head from its largest |value|; KV-cache tutorial page, "Quantization":
// symmetric q = clip(round(x / s), q_min, q_max), x_hat = s q).
//
// One CTA per (unit, KV head, K or V).  Pass 1 streams the unit's rows of that
// head (16-byte loads, 8 bf16 each) and reduces max |x|; pass 2 reads them again
// (from L2: a unit-head of the 7B arena is ~0.2 MB) and writes the codes, 8
// bytes per 16-byte chunk.  s and x / s are IEEE fp32 (correctly rounded
// division, roundf half away from zero), so the codes are exact functions of
// the inputs.
#include <cuda_bf16.h>

#include "internal.cuh"

namespace aircache {
namespace {

constexpr int kQuantThreads = 256;

struct QuantArgs {
  const __nv_bfloat16* src[2];  // k, v
  int8_t* dst[2];               // k8, v8
  float* scale[2];              // k_scale, v_scale
  const int64_t* offsets;
  int32_t* status;
  int64_t rows, stride_row, stride_head;
  int h_kv;
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ int code(float x, float s) {
  if (s == 0.f) return 0;
  const float r = roundf(__fdiv_rn(x, s));
  return (int)fminf(fmaxf(r, -127.f), 127.f);
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads) quant_kernel(const __grid_constant__ QuantArgs a) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per row of one head
  const int u = blockIdx.x, h = blockIdx.y, which = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float red[kQuantThreads / 32];
  const int64_t b = a.offsets[u], e = a.offsets[u + 1];
  if (b < 0 || e < b || e > a.rows) {
    if (tid == 0 && h == 0 && which == 0 && a.status) atomicCAS(a.status, 0, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t n = (e - b) * kChunks;
  const __nv_bfloat16* src = a.src[which] + b * a.stride_row + (int64_t)h * a.stride_head;
  auto chunk = [&](int64_t c) {
    const int64_t row = c / kChunks;
    return *reinterpret_cast<const uint4*>(src + row * a.stride_row + (c % kChunks) * 8);
  };
  float big = 0.f;
  for (int64_t c = tid; c < n; c += kQuantThreads) {
    const uint4 w = chunk(c);
    big = fmaxf(big, fmaxf(fmaxf(fabsf(bf_lo(w.x)), fabsf(bf_hi(w.x))), fmaxf(fabsf(bf_lo(w.y)), fabsf(bf_hi(w.y)))));
    big = fmaxf(big, fmaxf(fmaxf(fabsf(bf_lo(w.z)), fabsf(bf_hi(w.z))), fmaxf(fabsf(bf_lo(w.w)), fabsf(bf_hi(w.w)))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) big = fmaxf(big, __shfl_xor_sync(0xffffffffu, big, off));
  if (lane == 0) red[warp] = big;
  __syncthreads();
  big = red[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) big = fmaxf(big, red[w]);
  const float s = __fdiv_rn(big, 127.f);
  if (tid == 0) a.scale[which][(int64_t)u * a.h_kv + h] = s;
  int8_t* dst = a.dst[which] + (b * a.h_kv + h) * D;
  for (int64_t c = tid; c < n; c += kQuantThreads) {
    const uint4 w = chunk(c);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    uint32_t packed[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int c0 = code(bf_lo(words[2 * k]), s), c1 = code(bf_hi(words[2 * k]), s);
      const int c2 = code(bf_lo(words[2 * k + 1]), s), c3 = code(bf_hi(words[2 * k + 1]), s);
      packed[k] = (uint32_t)(c0 & 0xff) | ((uint32_t)(c1 & 0xff) << 8) | ((uint32_t)(c2 & 0xff) << 16) |
                  ((uint32_t)(c3 & 0xff) << 24);
    }
    const int64_t row = c / kChunks;
    *reinterpret_cast<uint2*>(dst + row * a.h_kv * D + (c % kChunks) * 8) = make_uint2(packed[0], packed[1]);
  }
}

}  // namespace
}  // namespace aircache

using namespace aircache;

extern "C" int aircache_quantize_int8(const aircache_quant_problem* p, int32_t* status, void* stream) {
  if (!p) return AIRCACHE_ERR_INVALID_ARG;
  auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  if (p->num_units < 0 || p->num_units > (1 << 29) || p->h_kv <= 0 || p->h_kv > 65535 ||
      (p->head_dim != 64 && p->head_dim != 128) || p->dtype != AIRCACHE_BF16 || p->reserved0 != 0 ||
      p->reserved1 != 0 || p->rows < 1 || !p->k || !p->v || !p->k8 || !p->v8 || !p->k_scale || !p->v_scale ||
      !p->offsets || !al16(p->k) || !al16(p->v) || !al16(p->k8) || !al16(p->v8) || p->kv_stride_row <= 0 ||
      p->kv_stride_head <= 0 || p->kv_stride_row % 8 != 0 || p->kv_stride_head % 8 != 0)
    return AIRCACHE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return AIRCACHE_ERR_CUDA;
  if (p->num_units == 0) return AIRCACHE_OK;
  QuantArgs a;
  a.src[0] = static_cast<const __nv_bfloat16*>(p->k);
  a.src[1] = static_cast<const __nv_bfloat16*>(p->v);
  a.dst[0] = p->k8;
  a.dst[1] = p->v8;
  a.scale[0] = p->k_scale;
  a.scale[1] = p->v_scale;
  a.offsets = p->offsets;
  a.status = status;
  a.rows = p->rows;
  a.stride_row = p->kv_stride_row;
  a.stride_head = p->kv_stride_head;
  a.h_kv = p->h_kv;
  const dim3 grid(p->num_units, p->h_kv, 2);
  if (p->head_dim == 128)
    quant_kernel<128><<<grid, kQuantThreads, 0, s>>>(a);
  else
    quant_kernel<64><<<grid, kQuantThreads, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? AIRCACHE_OK : AIRCACHE_ERR_CUDA;
}
