// TMA tensor maps (host) and tiled tensor copies global -> shared (device),
// shared by the scoring kernels.  Maps use the 128-byte swizzle with a box
// that is 128 bytes wide, so a copied tile lands as 128-byte column slabs:
// slab j of a tile holds bytes 128j..128j+127 of every row, rows 128 bytes
// apart, 16-byte chunks XOR-swizzled by (row & 7).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace aircache {

// Shared-memory address of 16-byte chunk `chunk` of row `row` in a swizzled slab.
__device__ __forceinline__ uint32_t swz(uint32_t slab, int row, int chunk) {
  return slab + (uint32_t)(row * 128) + (uint32_t)((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read exactly once: evict it before anything else.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}

// tma_load_4d with an L2 cache policy.
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3, %4, %5}], [%6], %7;\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// The "memory" clobber keeps the compiler from moving the shared-memory read
// above the barrier wait that guards the data (the operand is only an address).
__device__ __forceinline__ void ldsm_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// ------------------------------------------------------------------ host

inline PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
  }
  return fn;
}

template <typename T>
CUtensorMapDataType tma_type() {
  return sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

// A 2-D map over dense rows of D elements, box = (128 bytes, rows_box).
template <typename T>
bool encode_rows(CUtensorMap* m, const void* base, int d, long long rows, int rows_box) {
  auto enc = tma_encoder();
  if (!enc || rows < 1 || !base) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * sizeof(T)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / sizeof(T)), (cuuint32_t)rows_box};
  cuuint32_t es[2] = {1, 1};
  return enc(m, tma_type<T>(), 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The 4-D map (D, H_kv, tokens, layers) over every layer's keys, box
// (128 bytes, 1 head, rows_box tokens, 1 layer), if the per-layer pointers are
// evenly strided.
template <typename T>
bool encode_keys(CUtensorMap* m, const Dev& p, const LayerPtrs& lp, int rows_box) {
  auto enc = tma_encoder();
  if (!enc) return false;
  const char* k0 = reinterpret_cast<const char*>(lp.k[0]);
  const long long lstride = (p.L > 1) ? (reinterpret_cast<const char*>(lp.k[1]) - k0) : 16;
  if (lstride <= 0 || lstride % 16 != 0) return false;
  for (int l = 2; l < p.L; ++l) {
    if (reinterpret_cast<const char*>(lp.k[l]) - k0 != (long long)l * lstride) return false;
  }
  cuuint64_t dims[4] = {(cuuint64_t)p.d, (cuuint64_t)p.h_kv, (cuuint64_t)p.total_tokens, (cuuint64_t)p.L};
  cuuint64_t strides[3] = {(cuuint64_t)p.kv_stride_head * sizeof(T), (cuuint64_t)p.kv_stride_tok * sizeof(T),
                           (cuuint64_t)lstride};
  cuuint32_t box[4] = {(cuuint32_t)(128 / sizeof(T)), 1, (cuuint32_t)rows_box, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, tma_type<T>(), 4, const_cast<char*>(k0), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 2-D map over an fp32 matrix of `rows` rows of `cols` elements (cols a
// multiple of 4, so rows are 16-byte aligned), box (box_cols, box_rows), no
// swizzle: a copied box lands row-major, box_cols floats per row.
inline bool encode_logits(CUtensorMap* m, const float* base, long long cols, long long rows, int box_cols,
                          int box_rows) {
  auto enc = tma_encoder();
  if (!enc || rows < 1 || cols < 1 || cols % 4 != 0 || !base) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * sizeof(float)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace aircache
