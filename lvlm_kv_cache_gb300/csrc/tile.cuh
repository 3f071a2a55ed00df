// The logit tile shared by the elite-window and scoring kernels: 128 keys
// (rows of a K tile in shared memory) against up to 32 query rows (a Q chunk in
// shared memory), scaled to base-2 logits, left in registers in the mma.sync
// accumulator layout.
#pragma once

#include "internal.cuh"
#include "ptx.cuh"

namespace aircache {

constexpr int kTK = 128;  // keys per tile (8 warps x 16)
constexpr int kRC = 32;   // query rows per chunk (4 n8 MMA tiles)

// Shared-memory geometry of one (K tile, Q chunk) stage: rows padded by 16 bytes
// so that ldmatrix row addresses fall in distinct banks.
template <typename T, int D>
struct TileGeom {
  static constexpr int kRowBytes = D * (int)sizeof(T);
  static constexpr int kStride = D + 16 / (int)sizeof(T);  // elements
  static constexpr int kRowPitch = kStride * (int)sizeof(T);
  static constexpr int kKBytes = kTK * kRowPitch;
  static constexpr int kQBytes = kRC * kRowPitch;
  static constexpr int kStageBytes = kKBytes + kQBytes;
};

// acc[j][0..1]: key kA = 16*warp + lane/4, rows 8j + 2(lane%4) + {0,1};
// acc[j][2..3]: key kA + 8, same rows.  Values are log2(e)/sqrt(D) * q . k.
// Rows >= `rows` hold unspecified values.
template <typename T, int D>
struct TileLogits;

template <int D>
struct TileLogits<__nv_bfloat16, D> {
  using C = TileGeom<__nv_bfloat16, D>;
  static __device__ __forceinline__ void run(const __nv_bfloat16* Ks, const __nv_bfloat16* Qs, int rows,
                                             float scale, int warp, int lane, float acc[4][4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
    const __nv_bfloat16* a_base = Ks + (warp * 16 + (lane & 15)) * C::kStride + 8 * (lane >> 4);
    const __nv_bfloat16* b_base = Qs + ((lane & 7) + 8 * (lane >> 4)) * C::kStride + 8 * ((lane >> 3) & 1);
    if (rows > 16) {
      __syncwarp();  // ldmatrix / mma are warp-collective: the whole warp, converged
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4], b0[4], b1[4];
        ldmatrix_x4(a, a_base + kk * 16);
        ldmatrix_x4(b0, b_base + kk * 16);
        ldmatrix_x4(b1, b_base + 16 * C::kStride + kk * 16);
        mma_bf16_16816(acc[0], a, b0[0], b0[1]);
        mma_bf16_16816(acc[1], a, b0[2], b0[3]);
        mma_bf16_16816(acc[2], a, b1[0], b1[1]);
        mma_bf16_16816(acc[3], a, b1[2], b1[3]);
      }
    } else {
      __syncwarp();  // ldmatrix / mma are warp-collective: the whole warp, converged
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4], b0[4];
        ldmatrix_x4(a, a_base + kk * 16);
        ldmatrix_x4(b0, b_base + kk * 16);
        mma_bf16_16816(acc[0], a, b0[0], b0[1]);
        mma_bf16_16816(acc[1], a, b0[2], b0[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] *= scale;
  }
};

template <int D>
struct TileLogits<float, D> {
  using C = TileGeom<float, D>;
  static __device__ __forceinline__ void run(const float* Ks, const float* Qs, int rows, float scale,
                                             int warp, int lane, float acc[4][4]) {
    const float* ka = Ks + (warp * 16 + (lane >> 2)) * C::kStride;
    const float* kb = ka + 8 * C::kStride;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = 8 * j + 2 * (lane & 3) + e;
        float sa = 0.f, sb = 0.f;
        if (8 * j < rows) {
          const float* q = Qs + row * C::kStride;
#pragma unroll 8
          for (int i = 0; i < D; ++i) {
            sa = fmaf(q[i], ka[i], sa);
            sb = fmaf(q[i], kb[i], sb);
          }
        }
        acc[j][e] = sa * scale;
        acc[j][2 + e] = sb * scale;
      }
    }
  }
};

}  // namespace aircache
