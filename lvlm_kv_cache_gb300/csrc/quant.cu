// int8 storage of a compacted cache (LLM KV-compression notes, "Quantization
// stacked on compression": quantise after the token compression, one scale per
// head from its largest |value|; KV-cache tutorial page, "Quantization":
// symmetric q = clip(round(x / s), q_min, q_max), x_hat = s q).
//
// One thread-block cluster of kQuantCluster CTAs per (unit, KV head, K or V),
// each CTA a slice of the unit's rows.  Pass 1 streams the slice of that head
// (16-byte loads, 8 bf16 each, kBatch in flight per thread) and reduces max |x|;
// the cluster combines the slices' maxima through distributed shared memory;
// pass 2 reads the slice again (from L2) and writes the codes, 8 bytes per
// 16-byte chunk.  s and x / s are IEEE fp32 (correctly rounded
// division, roundf half away from zero), so the codes are exact functions of
// the inputs (a reciprocal fast path falls back to the division wherever the
// two could round differently).
#include <cuda_bf16.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace aircache {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantCluster = 8;

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

// clip(round(x / s)) with x / s correctly rounded, s > 0, |x| <= 127 s.
// The quotient is first taken as t = x * (1/s) (both correctly rounded:
// within 1.6e-5 of the exact quotient, and the correctly rounded quotient is
// within 3.9e-6 of that).  Away from half-integers both round to the same
// integer, and round-to-nearest-even (rint) equals round-half-away there; within
// 4e-5 of a half-integer the correctly rounded division and roundf decide.
// |t| < 127.5 always, so no clip is needed.
__device__ __forceinline__ int code(float x, float s, float rs) {
  const float t = x * rs;
  const float rt = rintf(t);
  if (fabsf(t - rt) > 0.5f - 4e-5f) return (int)roundf(__fdiv_rn(x, s));
  return (int)rt;
}

// four codes -> one word, byte i = code i
__device__ __forceinline__ uint32_t pack4(int c0, int c1, int c2, int c3) {
  return __byte_perm(__byte_perm(c0, c1, 0x0040), __byte_perm(c2, c3, 0x0040), 0x5410);
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads) quant_kernel(const __grid_constant__ QuantArgs a) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per row of one head
  const int u = blockIdx.x / kQuantCluster, rank = blockIdx.x % kQuantCluster;
  const int h = blockIdx.y, which = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float red[kQuantThreads / 32];
  __shared__ float slice_max;
  int64_t b = a.offsets[u], e = a.offsets[u + 1];
  if (b < 0 || e < b || e > a.rows) {  // the unit is skipped, but every CTA still meets the cluster barriers
    if (tid == 0 && rank == 0 && h == 0 && which == 0 && a.status)
      atomicCAS(a.status, 0, AIRCACHE_ERR_DEVICE_BOUNDS);
    b = e = 0;
  }
  const int64_t per = (e - b + kQuantCluster - 1) / kQuantCluster;
  const int64_t r0 = b + rank * per, r1 = r0 + per < e ? r0 + per : e;
  const int64_t n = r1 > r0 ? (r1 - r0) * kChunks : 0;
  const __nv_bfloat16* src = a.src[which] + r0 * a.stride_row + (int64_t)h * a.stride_head;
  auto chunk = [&](int64_t c) {
    const int64_t row = c / kChunks;
    return *reinterpret_cast<const uint4*>(src + row * a.stride_row + (c % kChunks) * 8);
  };
  // kBatch independent 16-byte loads per thread in flight: one CTA streams a
  // whole unit-head, so its memory parallelism sets the pace
  constexpr int kBatch = 8;
  // max |x| on the bf16 bit patterns: for finite values, |x| orders as the
  // integer (bits & 0x7fff); two 16-bit lanes per word
  uint32_t mx2 = 0;
  for (int64_t c0 = tid; c0 < n; c0 += (int64_t)kQuantThreads * kBatch) {
    uint4 w[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t c = c0 + (int64_t)j * kQuantThreads;
      w[j] = c < n ? chunk(c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      mx2 = __vmaxu2(mx2, __vmaxu2(w[j].x & 0x7fff7fffu, w[j].y & 0x7fff7fffu));
      mx2 = __vmaxu2(mx2, __vmaxu2(w[j].z & 0x7fff7fffu, w[j].w & 0x7fff7fffu));
    }
  }
  const uint32_t mbits = __reduce_max_sync(0xffffffffu, max(mx2 & 0xffffu, mx2 >> 16));
  float big = __uint_as_float(mbits << 16);
  if (lane == 0) red[warp] = big;
  __syncthreads();
  if (tid == 0) {
    float m = red[0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) m = fmaxf(m, red[w]);
    slice_max = m;
  }
  cluster_sync_all();
  big = 0.f;
#pragma unroll
  for (int x = 0; x < kQuantCluster; ++x) big = fmaxf(big, ld_cluster_f32(cluster_map(smem_u32(&slice_max), x)));
  cluster_sync_all();  // every rank has read the others' maxima
  const float s = __fdiv_rn(big, 127.f);
  const float rs = s == 0.f ? 0.f : __frcp_rn(s);
  if (tid == 0 && rank == 0) a.scale[which][(int64_t)u * a.h_kv + h] = s;  // 0 for an empty unit
  int8_t* dst = a.dst[which] + (r0 * a.h_kv + h) * D;
  for (int64_t c0 = tid; c0 < n; c0 += (int64_t)kQuantThreads * kBatch) {
    uint4 wb[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t c = c0 + (int64_t)j * kQuantThreads;
      wb[j] = c < n ? chunk(c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
    const int64_t c = c0 + (int64_t)j * kQuantThreads;
    if (c >= n) break;
    const uint4 w = wb[j];
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    uint32_t packed[2] = {0u, 0u};
    if (s != 0.f) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        packed[k] = pack4(code(bf_lo(words[2 * k]), s, rs), code(bf_hi(words[2 * k]), s, rs),
                          code(bf_lo(words[2 * k + 1]), s, rs), code(bf_hi(words[2 * k + 1]), s, rs));
      }
    }
    const int64_t row = c / kChunks;
    *reinterpret_cast<uint2*>(dst + row * a.h_kv * D + (c % kChunks) * 8) = make_uint2(packed[0], packed[1]);
    }
  }
}

}  // namespace
}  // namespace aircache

using namespace aircache;

extern "C" int aircache_quantize_int8(const aircache_quant_problem* p, int32_t* status, void* stream) {
  if (!p) return AIRCACHE_ERR_INVALID_ARG;
  auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  if (p->num_units < 0 || p->num_units > (1 << 27) || p->h_kv <= 0 || p->h_kv > 65535 ||
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p->num_units * kQuantCluster, p->h_kv, 2);
  cfg.blockDim = dim3(kQuantThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kQuantCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = p->head_dim == 128 ? cudaLaunchKernelEx(&cfg, quant_kernel<128>, a)
                                             : cudaLaunchKernelEx(&cfg, quant_kernel<64>, a);
  return err == cudaSuccess ? AIRCACHE_OK : AIRCACHE_ERR_CUDA;
}
