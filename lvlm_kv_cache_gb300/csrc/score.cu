// Cross-modal scoring (AirCache notes, "Key design 1": equations A_vtk and I_v).
//
// For one (layer l, request b) the query rows are every (query head h, elite
// text position e): H_q * N_tk rows, grouped by KV head (g * N_tk rows read the
// same keys).  Each row is a softmax over the N_v visual keys followed by the
// N_tk elite text keys (the "virtual key" range [0, N_v + N_tk)); I_v[i] is the
// mean over all rows of the probability of visual key i.
//
// The softmax needs each row's log-sum-exp over every key before any
// probability can be pooled, so the work is two passes over the keys, each a
// grid of C CTAs per (l, b) that take key tiles t = c, c+C, ...:
//   pass 1: logits -> per-row running (max, sum of exp) over the CTA's tiles ->
//           partials; the last CTA of (l, b) to finish combines the C partials
//           of every row, in a fixed order, into the row's log-sum-exp;
//   pass 2: logits again -> per visual key, sum over rows of exp(logit - lse),
//           scaled by 1/(H_q N_tk) -> I_v.
// Logits are base 2 (scaled by log2(e)/sqrt(D)) so that every exponential is
// an exp2f.  Pass 2 walks the layers in reverse so that its re-reads of K find
// the most recently streamed layers still in L2.
//
// bf16 inputs: logits come from mma.sync m16n8k16 (bf16 x bf16 -> fp32; every
// product is exact in fp32), keys as the M dimension (16 per warp, 64 per
// tile), query rows as N (32 per chunk).  fp32 inputs: CUDA-core FMAs.
#include "internal.cuh"

namespace aircache {
namespace {

struct ScoreArgs {
  Dev p;
  LayerPtrs lp;
  Ws w;
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

// 16-byte async copy global -> shared; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t r[4], const void* ptr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(ptr)));
}

__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ tile shapes

template <typename T, int D>
struct Shape {
  static constexpr int kElem = sizeof(T);
  static constexpr int kVecPerRow = D * kElem / 16;           // 16-byte chunks per row
  static constexpr int kPad = 16 / kElem;                     // one 16-byte pad per row
  static constexpr int kStride = D + kPad;                    // smem row stride (elements)
  static constexpr int kKBytes = kTileKeys * kStride * kElem;
  static constexpr int kQBytes = kRowChunk * kStride * kElem;
  static constexpr int kLStride = kTileKeys + 4;              // logits row stride (floats)
  static constexpr int kLBytes = kRowChunk * kLStride * 4;
  static constexpr int kFixedBytes = 2 * kKBytes + kQBytes + kLBytes + kRowChunk * 4;
};

// Per-(l, b) context shared by both passes.
struct Unit {
  Req R;
  int l, b, u, n_tk, n_keys;
  const int32_t* elite;
};

__device__ __forceinline__ bool load_unit(const Dev& p, const Ws& w, int l, int b, Unit& U) {
  if (!load_req(p, b, U.R)) return false;
  U.l = l;
  U.b = b;
  U.u = l * p.B + b;
  U.n_tk = w.n_tk[U.u];
  if (U.n_tk < 1 || U.n_tk > p.max_elite || U.n_tk > U.R.n_t) return false;
  U.n_keys = U.R.n_v + U.n_tk;
  U.elite = w.elite + (size_t)U.u * p.max_text;
  return true;
}

// Elite position e of the unit, clamped into [0, N_t) so that a corrupt list can
// never address outside the request.
__device__ __forceinline__ int elite_at(const Unit& U, int e) {
  return min(max(__ldg(U.elite + e), 0), U.R.n_t - 1);
}

// Issue the async copy of key tile t of KV head kvh (keys >= limit are zero).
template <typename T, int D>
__device__ __forceinline__ void load_k_tile(const Dev& p, const Unit& U, const T* kbase, int t,
                                            int kvh, int limit, T* Ks) {
  using S = Shape<T, D>;
  for (int i = threadIdx.x; i < kTileKeys * S::kVecPerRow; i += kScoreThreads) {
    const int row = i / S::kVecPerRow, vec = i % S::kVecPerRow;
    const int c = t * kTileKeys + row;
    const T* src = kbase;
    int bytes = 0;
    if (c < limit) {
      const int64_t pos = (c < U.R.n_v) ? (int64_t)c : (int64_t)U.R.n_v + elite_at(U, c - U.R.n_v);
      src = kbase + (U.R.seq0 + pos) * p.kv_stride_tok + (int64_t)kvh * p.kv_stride_head + vec * (16 / sizeof(T));
      bytes = 16;
    }
    cp_async16(Ks + row * S::kStride + vec * (16 / sizeof(T)), src, bytes);
  }
}

// Issue the async copy of query rows [r0, r0 + kRowChunk) of KV head kvh.
template <typename T, int D>
__device__ __forceinline__ void load_q_chunk(const Dev& p, const Unit& U, const T* qbase, int kvh,
                                             int r0, int rows_g, T* Qs) {
  using S = Shape<T, D>;
  for (int i = threadIdx.x; i < kRowChunk * S::kVecPerRow; i += kScoreThreads) {
    const int n = i / S::kVecPerRow, vec = i % S::kVecPerRow;
    const int r = r0 + n;
    const T* src = qbase;
    int bytes = 0;
    if (r < rows_g) {
      const int hh = r / U.n_tk, e = r % U.n_tk;
      const int h = kvh * p.g + hh;
      const int64_t trow = U.R.txt0 + elite_at(U, e);
      src = qbase + trow * p.q_stride_tok + (int64_t)h * p.q_stride_head + vec * (16 / sizeof(T));
      bytes = 16;
    }
    cp_async16(Qs + n * S::kStride + vec * (16 / sizeof(T)), src, bytes);
  }
}

// Logits of the tile against the row chunk: Ls[n][m] = log2(e)/sqrt(D) * q_n . k_m.
template <typename T, int D>
struct TileLogits;

template <int D>
struct TileLogits<__nv_bfloat16, D> {
  using S = Shape<__nv_bfloat16, D>;
  static __device__ __forceinline__ void run(const __nv_bfloat16* Ks, const __nv_bfloat16* Qs,
                                             float* Ls, int rows, float scale) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
    const int ntiles = (rows + 7) >> 3;  // n8 tiles with at least one live row
    const __nv_bfloat16* a_base = Ks + (warp * 16 + (lane & 15)) * S::kStride + 8 * (lane >> 4);
    const __nv_bfloat16* b_base = Qs + ((lane & 7) + 8 * (lane >> 4)) * S::kStride + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4];
      ldmatrix_x4(a, a_base + kk * 16);
      uint32_t bq[4];
      ldmatrix_x4(bq, b_base + kk * 16);
      mma_bf16(acc[0], a, bq[0], bq[1]);
      if (ntiles > 1) mma_bf16(acc[1], a, bq[2], bq[3]);
      if (ntiles > 2) {
        ldmatrix_x4(bq, b_base + 16 * S::kStride + kk * 16);
        mma_bf16(acc[2], a, bq[0], bq[1]);
        if (ntiles > 3) mma_bf16(acc[3], a, bq[2], bq[3]);
      }
    }
    const int m0 = warp * 16 + (lane >> 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < ntiles) {
        const int n0 = j * 8 + 2 * (lane & 3);
        Ls[n0 * S::kLStride + m0] = acc[j][0] * scale;
        Ls[(n0 + 1) * S::kLStride + m0] = acc[j][1] * scale;
        Ls[n0 * S::kLStride + m0 + 8] = acc[j][2] * scale;
        Ls[(n0 + 1) * S::kLStride + m0 + 8] = acc[j][3] * scale;
      }
    }
  }
};

template <int D>
struct TileLogits<float, D> {
  using S = Shape<float, D>;
  static __device__ __forceinline__ void run(const float* Ks, const float* Qs, float* Ls, int rows,
                                             float scale) {
    // thread -> key m = tid % 64, rows [16 * (tid / 64), +16)
    const int m = threadIdx.x % kTileKeys, rg = threadIdx.x / kTileKeys;
    for (int n = rg * 16; n < rg * 16 + 16; ++n) {
      if (n >= rows) break;
      float acc = 0.f;
      const float* kr = Ks + m * S::kStride;
      const float* qr = Qs + n * S::kStride;
#pragma unroll 8
      for (int i = 0; i < D; ++i) acc = fmaf(qr[i], kr[i], acc);
      Ls[n * S::kLStride + m] = acc * scale;
    }
  }
};

// ------------------------------------------------------------ pass 1

template <typename T, int D>
__global__ void __launch_bounds__(kScoreThreads)
score_pass1_kernel(const __grid_constant__ ScoreArgs a) {
  using S = Shape<T, D>;
  const Dev& p = a.p;
  const int c = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31;
  if (*(volatile int32_t*)a.w.error != 0) return;
  Unit U;
  if (!load_unit(p, a.w, l, b, U)) {
    if (tid == 0) set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  extern __shared__ __align__(16) unsigned char smem[];
  T* Kb[2] = {reinterpret_cast<T*>(smem), reinterpret_cast<T*>(smem + S::kKBytes)};
  T* Qs = reinterpret_cast<T*>(smem + 2 * S::kKBytes);
  float* Ls = reinterpret_cast<float*>(smem + 2 * S::kKBytes + S::kQBytes);

  const T* kbase = reinterpret_cast<const T*>(a.lp.k[l]);
  const T* qbase = reinterpret_cast<const T*>(a.lp.q[l]);
  const int ntiles = (U.n_keys + kTileKeys - 1) / kTileKeys;
  const int rows_g = p.g * U.n_tk;
  const int C = gridDim.x;
  float2* part = a.w.part + ((size_t)U.u * C + c) * p.rows_max;

  // thread -> row n = tid / 4, key quarter q4 = tid % 4 (16 keys)
  const int n = tid >> 2, q4 = tid & 3;
  if (c >= ntiles) {
    for (int r = tid; r < p.h_kv * rows_g; r += kScoreThreads) part[r] = make_float2(-INFINITY, 0.f);
  }
  for (int kvh = 0; kvh < p.h_kv && c < ntiles; ++kvh) {
    for (int r0 = 0; r0 < rows_g; r0 += kRowChunk) {
      const int rows = min(kRowChunk, rows_g - r0);
      float m_run = -INFINITY, s_run = 0.f;
      __syncthreads();
      load_q_chunk<T, D>(p, U, qbase, kvh, r0, rows_g, Qs);
      load_k_tile<T, D>(p, U, kbase, c, kvh, U.n_keys, Kb[0]);
      cp_async_commit();
      int it = 0;
      for (int t = c; t < ntiles; t += C, ++it) {
        if (t + C < ntiles) {
          load_k_tile<T, D>(p, U, kbase, t + C, kvh, U.n_keys, Kb[(it + 1) & 1]);
          cp_async_commit();
          cp_async_wait<1>();
        } else {
          cp_async_wait<0>();
        }
        __syncthreads();
        TileLogits<T, D>::run(Kb[it & 1], Qs, Ls, rows, p.scale_log2);
        __syncthreads();
        // running (max, sum exp2) of row n over this tile's live keys
        const int kmax = min(kTileKeys, U.n_keys - t * kTileKeys);
        float tm = -INFINITY;
        const float* lr = Ls + n * S::kLStride + q4 * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (q4 * 16 + i < kmax) tm = fmaxf(tm, lr[i]);
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
        const float m_new = fmaxf(m_run, tm);
        float ts = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (q4 * 16 + i < kmax) ts += exp2f(lr[i] - m_new);
        ts += __shfl_xor_sync(0xffffffffu, ts, 1);
        ts += __shfl_xor_sync(0xffffffffu, ts, 2);
        s_run = s_run * exp2f(m_run - m_new) + ts;  // m_run = -inf: factor 0
        m_run = m_new;
        __syncthreads();
      }
      cp_async_wait<0>();
      if (q4 == 0 && n < rows) part[kvh * rows_g + r0 + n] = make_float2(m_run, s_run);
    }
  }

  // The last CTA of this (l, b) combines the partials of every row.
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (tid == 0) is_last = (atomicAdd(&a.w.cnt_unit[U.u], 1u) == (unsigned)(C - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int rows_total = p.h_q * U.n_tk;
  const float2* pu = a.w.part + (size_t)U.u * C * p.rows_max;
  float* lse = a.w.lse + (size_t)U.u * p.rows_max;
  for (int r = tid; r < rows_total; r += kScoreThreads) {
    float M = -INFINITY;
    for (int cc = 0; cc < C; ++cc) M = fmaxf(M, __ldcg(&pu[(size_t)cc * p.rows_max + r].x));
    float Ssum = 0.f;
    for (int cc = 0; cc < C; ++cc) {
      const float2 v = __ldcg(&pu[(size_t)cc * p.rows_max + r]);
      if (v.y > 0.f) Ssum += v.y * exp2f(v.x - M);
    }
    lse[r] = M + log2f(Ssum);
  }
  (void)lane;
}

// ------------------------------------------------------------ pass 2

template <typename T, int D>
__global__ void __launch_bounds__(kScoreThreads)
score_pass2_kernel(const __grid_constant__ ScoreArgs a) {
  using S = Shape<T, D>;
  const Dev& p = a.p;
  const int c = blockIdx.x, b = blockIdx.y, l = p.L - 1 - (int)blockIdx.z;
  const int tid = threadIdx.x;
  if (*(volatile int32_t*)a.w.error != 0) return;
  Unit U;
  if (!load_unit(p, a.w, l, b, U)) {
    if (tid == 0) set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  extern __shared__ __align__(16) unsigned char smem[];
  T* Kb[2] = {reinterpret_cast<T*>(smem), reinterpret_cast<T*>(smem + S::kKBytes)};
  T* Qs = reinterpret_cast<T*>(smem + 2 * S::kKBytes);
  float* Ls = reinterpret_cast<float*>(smem + 2 * S::kKBytes + S::kQBytes);
  float* lse_s = reinterpret_cast<float*>(smem + 2 * S::kKBytes + S::kQBytes + S::kLBytes);
  float* acc = reinterpret_cast<float*>(smem + S::kFixedBytes);  // [tiles_per_cta][64]

  const T* kbase = reinterpret_cast<const T*>(a.lp.k[l]);
  const T* qbase = reinterpret_cast<const T*>(a.lp.q[l]);
  const int ntiles = (U.R.n_v + kTileKeys - 1) / kTileKeys;  // visual keys only
  const int rows_g = p.g * U.n_tk;
  const int C = gridDim.x;
  const float* lse = a.w.lse + (size_t)U.u * p.rows_max;
  const int my_tiles = (c < ntiles) ? (ntiles - c + C - 1) / C : 0;
  if (my_tiles == 0) return;
  for (int i = tid; i < my_tiles * kTileKeys; i += kScoreThreads) acc[i] = 0.f;

  // thread -> key m = tid / 2, row half = tid % 2 (rows [16 * half, +16))
  const int m = tid >> 1, half = tid & 1;
  for (int kvh = 0; kvh < p.h_kv; ++kvh) {
    for (int r0 = 0; r0 < rows_g; r0 += kRowChunk) {
      const int rows = min(kRowChunk, rows_g - r0);
      __syncthreads();
      load_q_chunk<T, D>(p, U, qbase, kvh, r0, rows_g, Qs);
      if (tid < kRowChunk) lse_s[tid] = (tid < rows) ? __ldcg(lse + kvh * rows_g + r0 + tid) : 0.f;
      load_k_tile<T, D>(p, U, kbase, c, kvh, U.R.n_v, Kb[0]);
      cp_async_commit();
      int it = 0;
      for (int t = c; t < ntiles; t += C, ++it) {
        if (t + C < ntiles) {
          load_k_tile<T, D>(p, U, kbase, t + C, kvh, U.R.n_v, Kb[(it + 1) & 1]);
          cp_async_commit();
          cp_async_wait<1>();
        } else {
          cp_async_wait<0>();
        }
        __syncthreads();
        TileLogits<T, D>::run(Kb[it & 1], Qs, Ls, rows, p.scale_log2);
        __syncthreads();
        float s = 0.f;
        const int rb = half * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (rb + i < rows) s += exp2f(Ls[(rb + i) * S::kLStride + m] - lse_s[rb + i]);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        if (half == 0) acc[it * kTileKeys + m] += s;
        __syncthreads();
      }
      cp_async_wait<0>();
    }
  }
  __syncthreads();
  const float inv = 1.f / (float)(p.h_q * U.n_tk);
  float* iv = a.w.iv + (size_t)l * p.total_visual + U.R.vis0;
  for (int i = tid; i < my_tiles * kTileKeys; i += kScoreThreads) {
    const int key = (c + (i / kTileKeys) * C) * kTileKeys + (i % kTileKeys);
    if (key < U.R.n_v) iv[key] = acc[i] * inv;
  }
}

template <typename T, int D>
cudaError_t launch_pass(const Dev& p, const LayerPtrs& lp, const Ws& w, cudaStream_t s, int pass) {
  using S = Shape<T, D>;
  ScoreArgs a;
  a.p = p;
  a.lp = lp;
  a.w = w;
  dim3 grid(p.chunks, p.B, p.L);
  if (pass == 1) {
    const size_t smem = S::kFixedBytes;
    cudaFuncSetAttribute(score_pass1_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    score_pass1_kernel<T, D><<<grid, kScoreThreads, smem, s>>>(a);
  } else {
    const size_t smem = S::kFixedBytes + (size_t)p.tiles_per_cta * kTileKeys * sizeof(float);
    cudaFuncSetAttribute(score_pass2_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    score_pass2_kernel<T, D><<<grid, kScoreThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t dispatch(const Dev& p, const LayerPtrs& lp, const Ws& w, cudaStream_t s, int pass) {
  if (p.dtype == AIRCACHE_BF16) {
    return p.d == 128 ? launch_pass<__nv_bfloat16, 128>(p, lp, w, s, pass)
                      : launch_pass<__nv_bfloat16, 64>(p, lp, w, s, pass);
  }
  return p.d == 128 ? launch_pass<float, 128>(p, lp, w, s, pass)
                    : launch_pass<float, 64>(p, lp, w, s, pass);
}

}  // namespace

cudaError_t launch_score_pass1(const Dev& p, const LayerPtrs& lp, const Ws& w, cudaStream_t s) {
  return dispatch(p, lp, w, s, 1);
}
cudaError_t launch_score_pass2(const Dev& p, const LayerPtrs& lp, const Ws& w, cudaStream_t s) {
  return dispatch(p, lp, w, s, 2);
}

}  // namespace aircache
