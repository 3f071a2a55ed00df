// One decode step of attention over cached K/V rows: the consumer of the
// compacted cache (KV-cache tutorial page, section "Prefill and Decode": each
// step's single query reads every cached key and value; edge-device
// compression page, head-wise top-k scheme: after compaction, decoding is
// dense attention over the kept rows).
//
// Split-K over the rows.  CTA (x, h, s) takes the x-th slice of sequence s's
// row range for KV head h and every query head of h's group (g <= 16, padded
// to the 16 rows of an mma.sync A operand).  A producer warp reads the range
// and streams 64-row K and V tiles of that head with TMA through a ring of
// stages (bf16: 128-byte swizzle; int8 codes: the swizzle of the row's width,
// widened to f16 on their way into the fragments); four consumer warps each
// take 16 rows of a tile:
//   S = Q K^T      A = Q (16 heads x 16 d, in registers), B = K (ldmatrix;
//                  int8: the lane's codes read as words),
//   online softmax in base 2 per head, P rounded to bf16 (int8 cache: to f16,
//                  scaled by 2^14; the normaliser sums the rounded weights, so
//                  the output is an exact convex combination with relatively
//                  perturbed weights),
//   O += P V       A = P (the S accumulators repacked), B = V (ldmatrix.trans;
//                  int8: byte pairs of two rows from one 16- or 8-byte read
//                  per row, with permuted value columns).
// The warps' (max, sum, O) merge in shared memory.  The slices of one
// (sequence, KV head) then merge in one of three ways: a single slice writes
// the output; up to 8 slices form a thread-block cluster and every rank merges
// its share of the output columns from all ranks' shared memory; more slices
// write partials and the last CTA to finish (an atomic count, no waiting)
// merges them.  The step's own (k_new, v_new) row joins the final merge.  An
// int8 cache's scales fold into the logit multiplier and the weighted sum.
// With AIRCACHE_DECODE_EARLY_CACHE the kernel is launched with programmatic
// dependent launch and reads the ranges and rows before waiting for the kernel
// before it.
//
// Traffic per launch: every cached row's K and V of each KV head once
// (2 * head_dim * element bytes per row and head), the queries, and the fp32
// output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace aircache {
namespace {

constexpr int kDecRows = 64;          // rows per K/V tile
constexpr int kDecWarps = 4;          // consumer warps, 16 rows each
constexpr int kDecThreads = (kDecWarps + 1) * 32;
constexpr int kDecMaxGroup = 16;      // query heads per KV head
constexpr int kDecMaxSplit = 64;
constexpr int kDecMaxCluster = 8;     // slices per (sequence, KV head) merged through a cluster
constexpr int kDecZeroBlock = 256;    // error word, then the per-(s, h) counters

constexpr int cmax(int a, int b) { return a > b ? a : b; }

// Q8: the cached rows are int8 codes (one row-major tile per stage, in the
// 128-byte swizzle, 64-byte for D = 64), widened to f16 (exact integers) on
// their way into the MMA fragments, which then run with f16 operands (Q
// converted once, P packed to f16).  Keys: the head dimension is permuted
// alike for Q and K so that a lane's key codes are contiguous.  Values: n-tile
// t's column n is the value column n*(D/8) + t, so a lane's codes of a row are
// one contiguous piece; the output columns are put back in order when the
// warps merge.
template <int D, bool Q8>
struct DecCfg {
  static constexpr int kSlabs = D / 64;                       // 128-byte bf16 column slabs per row
  static constexpr int kTileBytes = kDecRows * D * (Q8 ? 1 : 2);  // one K (or V) tile
  static constexpr int kStages = Q8 ? (D == 128 ? 4 : 6) : (D == 128 ? 3 : 5);
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQPitch = D + 8;                       // bf16 elements per staged query row
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kMerge = kDecWarps * (kDecMaxGroup * D + 2 * kDecMaxGroup) * 4;
  static constexpr int kPartEnd = 45056 + kDecMaxGroup * D * 4 + kDecMaxGroup * 8;  // the cluster partial's end
  static constexpr int kMain = (cmax(cmax(kRing, kMerge), kPartEnd) + 1023) / 1024 * 1024;
  static constexpr int kQBytes = kDecMaxGroup * kQPitch * 2;
  // 1024-byte alignment slack for the swizzled ring
  static constexpr int kSmem = 1024 + kMain + kQBytes + 2 * kStages * 8 + 64 + 3 * kDecMaxGroup * 4;
  static_assert(32768 + kDecMaxGroup * kDecMaxSplit * 12 <= 45056, "merge scratch below the cluster partial");
  static_assert(kSmem <= 113 * 1024, "two CTAs per SM");
};

struct DecArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int64_t* row_begin;
  const int64_t* row_end;
  float* out;
  int32_t* error;
  uint32_t* count;   // [S * h_kv]
  float2* part_ml;   // [S * h_q * n_split] (max, sum) of each slice, base 2
  float* part_o;     // [S * h_q * n_split * D]
  int64_t kv_rows;
  int64_t q_stride_seq, q_stride_head, new_stride_seq, new_stride_head;
  int h_q, h_kv, group, n_split;
  const float* k_scale;  // int8 caches: [S * h_kv]
  const float* v_scale;
  float scale_log2;  // log2(e) / sqrt(D)
  int early;         // AIRCACHE_DECODE_EARLY_CACHE: ranges and rows read before the dependency wait
  const int32_t* row_index;  // gather mode: arena rows listed per range position
  int64_t range_len;         // bound of the ranges: kv_rows, or the row list's length
  int64_t col_stride_head;   // gather mode: elements between KV heads in a row
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi, float& lo_r, float& hi_r) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  lo_r = __low2float(t);
  hi_r = __high2float(t);
  return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi, float& lo_r, float& hi_r) {
  __half2 t = __floats2half2_rn(lo, hi);
  lo_r = __low2float(t);
  hi_r = __high2float(t);
  return *reinterpret_cast<uint32_t*>(&t);
}
// D(16x8, fp32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The int8 path multiplies in f16 (codes are exact there), the bf16 path in bf16.
template <bool F16>
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    mma_f16_16816(c, a, b0, b1);
  } else {
    mma_bf16_16816(c, a, b0, b1);
  }
}
// P leaves the int8 path's softmax scaled by 2^14 (its largest weight, 1,
// becomes 16384 < 65504): weights down to 2^-28 stay normal f16 numbers.
constexpr float kP16 = 16384.f;

__device__ __forceinline__ void ldsm_x4_trans(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// Two int8 codes (the bytes `sel` picks of u4, whose top bits the caller has
// flipped) -> two f16, exactly, without a conversion instruction: code c
// becomes the unsigned byte u = c + 128 (flip
// the top bit), the byte permute places u in the low mantissa bits of the f16
// 0x6400 (= 1024), so the half is 1024 + u, and one packed subtraction of 1152
// leaves c (every integer below 2048 is an f16).
__device__ __forceinline__ uint32_t widen2_f16(uint32_t u4, uint32_t sel) {
  uint32_t t = __byte_perm(u4, 0x64646464u, sel);
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&t), __float2half2_rn(1152.f));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte offset within an int8 tile of the 128-byte swizzle (D = 128: rows of
// 128 bytes, 16-byte pieces XORed with the row mod 8) or the 64-byte swizzle
// (D = 64: pieces XORed with bits 7-8 of the offset), as the TMA copy places
// them (each tile starts on a 1024-byte boundary).
template <int D>
__device__ __forceinline__ int swz8(int off) {
  return off ^ (((off >> 7) & (D == 128 ? 7 : 3)) << 4);
}

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Four rows (r0..r3) of a 2-D tensor map whose box is one row high, landing as
// four consecutive box rows at dst (the Blackwell tile::gather4 form).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int col, int r0, int r1, int r2,
                                            int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5, %6}], [%7];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

template <int D, bool CL, bool Q8, bool GA>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap vmap,
                                                             const __grid_constant__ DecArgs a) {
  using C = DecCfg<D, Q8>;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = dsm;                                                   // [stages][K tile, V tile]
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(dsm + C::kMain);  // [16][kQPitch]
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + C::kMain + C::kQBytes);
  uint64_t* empty = full + C::kStages;
  int* ctl = reinterpret_cast<int*>(empty + C::kStages);                 // [16]
  // the slices' (max, sum) and merge weights live in the ring once it is idle,
  // above the 32 KB the per-warp merge and the final reduction use
  float2* mlbuf = reinterpret_cast<float2*>(ring + 32768);               // [16][kDecMaxSplit]
  float* coef = reinterpret_cast<float*>(mlbuf + kDecMaxGroup * kDecMaxSplit);  // [16][kDecMaxSplit]
  float* pbuf = reinterpret_cast<float*>(ring + 45056);                  // [16][D] this slice's O (clusters)
  float2* pml = reinterpret_cast<float2*>(ring + 45056 + kDecMaxGroup * D * 4);  // [16] its (max, sum)
  float* xnew = reinterpret_cast<float*>(ctl + 16);                      // [16] new row's base-2 logit
  float* rnorm = xnew + kDecMaxGroup;                                    // [16]
  float* cnew = rnorm + kDecMaxGroup;                                    // [16] new row's weight

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int g = a.group;

  pdl_trigger();  // the next kernel on the stream may launch; it waits for this one before using its output
  if (warp == kDecWarps && lane == 0) {
    // ---- producer lane: this CTA's slice of the sequence's rows, then the
    // first tiles right away (the queries load meanwhile)
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
    if (!a.early) pdl_wait();  // the ranges and rows may come from the previous kernel
    const int64_t b = a.row_begin[s], e = a.row_end[s];
    const bool ok = b >= 0 && e >= b && e <= a.range_len;
    if (!ok && split == 0 && h == 0) set_error(a.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    const int64_t n = ok ? e - b : 0;
    int64_t per = (n + a.n_split - 1) / a.n_split;
    per = (n >= (int64_t)kDecRows * a.n_split) ? (per + kDecRows - 1) / kDecRows * kDecRows : (per + 15) / 16 * 16;
    const int64_t lo = b + (int64_t)split * per;
    const int64_t hi = lo + per < e ? lo + per : e;
    const int row0 = (int)(lo & 0x7fffffff);
    const int nrows = ok && hi > lo ? (int)(hi - lo) : 0;
    ctl[0] = row0;
    ctl[1] = nrows;
    ctl[2] = ok ? 1 : 0;
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDecWarps);
    }
    fence_mbar_init();
    const int ntiles = GA ? 0 : (nrows + kDecRows - 1) / kDecRows;  // gather mode: the warp issues every tile
    for (int i = 0; i < ntiles && i < C::kStages; ++i) {
      const uint32_t kb = smem_u32(ring + i * C::kStageBytes);
      mbar_arrive_expect_tx(&full[i], C::kStageBytes);
      if (Q8) {
        tma_load_3d(kb, &kmap, 0, h, row0 + i * kDecRows, &full[i]);
        tma_load_3d(kb + C::kTileBytes, &vmap, 0, h, row0 + i * kDecRows, &full[i]);
      } else {
#pragma unroll
        for (int sl = 0; sl < C::kSlabs; ++sl) {
          tma_load_3d(kb + sl * kDecRows * 128, &kmap, sl * 64, h, row0 + i * kDecRows, &full[i]);
          tma_load_3d(kb + C::kTileBytes + sl * kDecRows * 128, &vmap, sl * 64, h, row0 + i * kDecRows, &full[i]);
        }
      }
    }
  }
  // ---- query rows of the group, zero-padded to 16 heads (after the previous
  // kernel on the stream is done: it may have written q; everything below
  // comes after this wait in every thread but the producer's early reads)
  pdl_wait();
  for (int c = tid; c < kDecMaxGroup * (D / 8); c += kDecThreads) {
    const int hh = c / (D / 8), ch = c % (D / 8);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (hh < g) {
      val = *reinterpret_cast<const uint4*>(a.q + (int64_t)s * a.q_stride_seq +
                                            (int64_t)(h * g + hh) * a.q_stride_head + ch * 8);
    }
    *reinterpret_cast<uint4*>(qs + hh * C::kQPitch + ch * 8) = val;
  }
  __syncthreads();
  const int row0 = ctl[0], nrows = ctl[1];
  const bool ok = ctl[2] != 0;
  const bool has_new = a.k_new != nullptr && ok;
  const int ntiles = (nrows + kDecRows - 1) / kDecRows;

  if (warp == kDecWarps && GA) {
    // ---- gather producer: the warp reads each tile's 64 listed rows (rows past
    // the slice end repeat its first row; they are masked) and issues the
    // four-row gathers, one group of K or V per lane
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % C::kStages;
      if (i >= C::kStages) {  // one lane waits for the stage, the warp follows its verdict
        bool freed = true;
        if (lane == 0) freed = mbar_wait(&empty[st], ((i / C::kStages) - 1) & 1);
        if (!__shfl_sync(0xffffffffu, freed ? 1 : 0, 0)) {
          if (lane == 0) set_error(a.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
          break;
        }
      }
      int rr[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = i * kDecRows + lane + 32 * q;
        int v = __ldg(a.row_index + row0 + (j < nrows ? j : 0));
        if (v < 0 || v >= a.kv_rows) {
          set_error(a.error, AIRCACHE_ERR_DEVICE_BOUNDS);
          v = 0;
        }
        rr[q] = v;
      }
      const uint32_t kb = smem_u32(ring + st * C::kStageBytes);
      // lane L issues four-row group L % 16 of K (L < 16) or of V (L >= 16),
      // every column slab: the rows of its group come by shuffles
      const int gg = lane & 15;
      int rv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int pos = 4 * gg + t;
        const int a0 = __shfl_sync(0xffffffffu, rr[0], pos & 31), a1 = __shfl_sync(0xffffffffu, rr[1], pos & 31);
        rv[t] = pos < 32 ? a0 : a1;
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[st], C::kStageBytes);
      __syncwarp();
      fence_proxy_async_smem();  // the consumers' generic reads of this stage come first
      const uint32_t base = kb + (lane >= 16 ? C::kTileBytes : 0) + gg * 512;
#pragma unroll
      for (int sl = 0; sl < C::kSlabs; ++sl) {
        const int col = (int)(h * a.col_stride_head) + sl * 64;
        tma_gather4(base + sl * kDecRows * 128, lane >= 16 ? &vmap : &kmap, col, rv[0], rv[1], rv[2], rv[3],
                    &full[st]);
      }
      __syncwarp();
    }
    __syncwarp();
    if (CL) {  // the two cluster barriers of the slice merge below
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }
  if (warp == kDecWarps) {
    // ---- producer: the remaining tiles, each into the stage its predecessor freed
    if (lane == 0) {
      for (int i = C::kStages; i < ntiles; ++i) {
        const int st = i % C::kStages;
        if (!mbar_wait(&empty[st], ((i / C::kStages) - 1) & 1)) {
          set_error(a.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
          break;
        }
        fence_proxy_async_smem();  // the consumers' generic reads of this stage come first
        const uint32_t kb = smem_u32(ring + st * C::kStageBytes);
        mbar_arrive_expect_tx(&full[st], C::kStageBytes);
        const int r = row0 + i * kDecRows;
        if (Q8) {
          tma_load_3d(kb, &kmap, 0, h, r, &full[st]);
          tma_load_3d(kb + C::kTileBytes, &vmap, 0, h, r, &full[st]);
        } else {
#pragma unroll
          for (int sl = 0; sl < C::kSlabs; ++sl) {
            tma_load_3d(kb + sl * kDecRows * 128, &kmap, sl * 64, h, r, &full[st]);
            tma_load_3d(kb + C::kTileBytes + sl * kDecRows * 128, &vmap, sl * 64, h, r, &full[st]);
          }
        }
      }
    }
    __syncwarp();
    if (CL) {  // the two cluster barriers of the slice merge below
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }
  // ---- consumers
  const int hA = lane >> 2;  // heads of this thread's accumulator rows: hA and hA + 8
  const int cq = lane & 3;
  uint32_t qa[D / 16][4];
  if constexpr (Q8) {
    // int8 cache: the head dimension is permuted so that each thread takes its
    // key codes as whole words (k-step kk of quad lane cq covers
    // d = cq*D/4 + 4kk + 0..3: k = 2cq, 2cq+1 -> +0, +1; k = 2cq+8, 2cq+9 ->
    // +2, +3); Q's A fragments are read from the staged rows the same way
    const __nv_bfloat16* q0 = qs + hA * C::kQPitch + cq * (D / 4);
    const __nv_bfloat16* q1 = q0 + 8 * C::kQPitch;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint2 x = *reinterpret_cast<const uint2*>(q0 + 4 * kk);
      const uint2 y = *reinterpret_cast<const uint2*>(q1 + 4 * kk);
      qa[kk][0] = x.x;
      qa[kk][1] = y.x;
      qa[kk][2] = x.y;
      qa[kk][3] = y.y;
    }
  } else {
    const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      ldmatrix_x4(qa[kk], qs + (ri + 8 * (mi & 1)) * C::kQPitch + 16 * kk + 8 * (mi >> 1));
    }
  }
  // int8 cache: Q enters the f16 MMA as Q * 2^e, with e chosen so that the
  // group's largest |q| lands in [2^14, 2^15) (no f16 overflow; scaling by a
  // power of two is exact, and a bf16 value fits an f16 mantissa)
  float qscale = 1.f;
  if constexpr (Q8) {
    float mx = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qa[kk][j]));
        mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (mx > 0.f && mx < INFINITY) {
      int ex;
      (void)frexpf(mx, &ex);  // mx = f * 2^ex, f in [0.5, 1)
      qscale = ldexpf(1.f, min(15 - ex, 120));  // (a subnormal maximum: no overflow)
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qa[kk][j]));
        const __half2 hq = __floats2half2_rn(f.x * qscale, f.y * qscale);
        qa[kk][j] = *reinterpret_cast<const uint32_t*>(&hq);
      }
  }
  float o[D / 8][4];
#pragma unroll
  for (int t = 0; t < D / 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  const int r0 = 16 * warp;
  // logits in base 2; an int8 cache folds its key scale in here (q . (s c) = s (q . c))
  const float kmult = Q8 ? a.scale_log2 * a.k_scale[(int64_t)s * a.h_kv + h] / qscale : a.scale_log2;
  bool alive = true;

  for (int i = 0; i < ntiles && alive; ++i) {
    const int st = i % C::kStages;
    if (!mbar_wait(&full[st], (i / C::kStages) & 1)) {
      if (lane == 0) set_error(a.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      alive = false;
      break;
    }
    const int valid = nrows - i * kDecRows - r0;  // rows of this warp's 16 that belong to the slice
    if (valid > 0) {
      uint32_t kb, vb;
      int rb;                          // this warp's first row in the tile it reads
      constexpr int kSlabStride = (Q8 ? 16 : kDecRows) * 128;
      uint32_t kq[2][Q8 ? D / 16 : 1];  // int8: this thread's key codes of rows hA and hA + 8
      if constexpr (Q8) {
        // keys: the thread's D/4 codes of each of its two rows, as words (rows
        // past the slice end read as 0); the tile is in the int8 swizzle
        const uint8_t* kt = ring + st * C::kStageBytes;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int rr = 8 * t + hA;
#pragma unroll
          for (int v = 0; v < D / 64; ++v) {
            const uint4 x = rr < valid ? *reinterpret_cast<const uint4*>(
                                             kt + swz8<D>((r0 + rr) * D + cq * (D / 4) + 16 * v))
                                       : make_uint4(0, 0, 0, 0);
            kq[t][4 * v] = x.x;
            kq[t][4 * v + 1] = x.y;
            kq[t][4 * v + 2] = x.z;
            kq[t][4 * v + 3] = x.w;
          }
        }
        kb = vb = 0;
        rb = 0;
      } else {
      kb = smem_u32(ring + st * C::kStageBytes);
      vb = kb + C::kTileBytes;
      rb = r0;
      if (valid < 16) {
        // rows past the slice end may hold anything (another sequence, unused
        // arena rows): zero their V so that 0-weight rows add exactly 0
        uint8_t* vrow = ring + st * C::kStageBytes + C::kTileBytes;
        for (int c = lane; c < 16 * C::kSlabs * 8; c += 32) {
          const int rr = c / (C::kSlabs * 8), rest = c % (C::kSlabs * 8);
          if (rr >= valid) {
            *reinterpret_cast<uint4*>(vrow + (rest >> 3) * kDecRows * 128 + (r0 + rr) * 128 + (rest & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
      }
      __syncwarp();
      }
      // S = Q K^T for 16 rows: two n-tiles of 8 rows
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if constexpr (Q8) {
        // B fragments from the codes: bytes 0, 1 of a word -> b0, bytes 2, 3 -> b1
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint32_t x = kq[t][kk] ^ 0x80808080u;
            mma16816<true>(sc[t], qa[kk], widen2_f16(x, 0x4140u), widen2_f16(x, 0x4342u));
          }
        }
      } else {
        const int mi = lane >> 3, ri = lane & 7;
        const int row = rb + ri + 8 * (mi >> 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t kf[4];
          ldsm_x4(kf, swz(kb + (kk >> 2) * kSlabStride, row, 2 * (kk & 3) + (mi & 1)));
          mma16816<Q8>(sc[0], qa[kk], kf[0], kf[1]);
          mma16816<Q8>(sc[1], qa[kk], kf[2], kf[3]);
        }
      }
      // online softmax, base 2; rows at or past `valid` get weight 0
      float tA = -INFINITY, tB = -INFINITY;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool in = 8 * t + 2 * cq + e < valid;
          sc[t][e] = in ? sc[t][e] * kmult : -INFINITY;
          sc[t][2 + e] = in ? sc[t][2 + e] * kmult : -INFINITY;
          tA = fmaxf(tA, sc[t][e]);
          tB = fmaxf(tB, sc[t][2 + e]);
        }
      }
      tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 1));
      tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 2));
      tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 1));
      tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 2));
      const float nA = fmaxf(mA, tA), nB = fmaxf(mB, tB);  // finite: row 0 of the slab is valid
      const float fA = fast_exp2(mA - nA), fB = fast_exp2(mB - nB);
      mA = nA;
      mB = nB;
      uint32_t pa[4];
      float sA = 0.f, sB = 0.f;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float x0, x1;
        if constexpr (Q8) {
          pa[2 * t] = pack_f16(kP16 * fast_exp2(sc[t][0] - nA), kP16 * fast_exp2(sc[t][1] - nA), x0, x1);
          sA += (x0 + x1) * (1.f / kP16);
          pa[2 * t + 1] = pack_f16(kP16 * fast_exp2(sc[t][2] - nB), kP16 * fast_exp2(sc[t][3] - nB), x0, x1);
          sB += (x0 + x1) * (1.f / kP16);
        } else {
          pa[2 * t] = pack_bf16(fast_exp2(sc[t][0] - nA), fast_exp2(sc[t][1] - nA), x0, x1);
          sA += x0 + x1;
          pa[2 * t + 1] = pack_bf16(fast_exp2(sc[t][2] - nB), fast_exp2(sc[t][3] - nB), x0, x1);
          sB += x0 + x1;
        }
      }
      lA = lA * fA + sA;
      lB = lB * fB + sB;
#pragma unroll
      for (int t = 0; t < D / 8; ++t) {
        o[t][0] *= fA;
        o[t][1] *= fA;
        o[t][2] *= fB;
        o[t][3] *= fB;
      }
      // O += P V
      if constexpr (Q8) {
        // B fragments straight from the value tile: lane (n, c) takes rows 2c,
        // 2c+1, 2c+8, 2c+9 of the warp's 16, value columns n*(D/8) .. +D/8-1
        // (one piece per row); n-tile t pairs byte t of two rows (rows past
        // the slice end hold finite codes and get weight 0)
        const uint8_t* vt = ring + st * C::kStageBytes + C::kTileBytes;
        uint32_t vw[4][D / 32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int rr = r0 + 2 * cq + (j & 1) + 8 * (j >> 1);
          const int off = swz8<D>(rr * D + hA * (D / 8));
          if constexpr (D == 128) {
            const uint4 x = *reinterpret_cast<const uint4*>(vt + off);
            vw[j][0] = x.x ^ 0x80808080u;
            vw[j][1] = x.y ^ 0x80808080u;
            vw[j][2] = x.z ^ 0x80808080u;
            vw[j][3] = x.w ^ 0x80808080u;
          } else {
            const uint2 x = *reinterpret_cast<const uint2*>(vt + off);
            vw[j][0] = x.x ^ 0x80808080u;
            vw[j][1] = x.y ^ 0x80808080u;
          }
        }
#pragma unroll
        for (int t = 0; t < D / 8; ++t) {
          const uint32_t sel = (uint32_t)(t & 3) | ((uint32_t)((t & 3) + 4) << 4);
          const uint32_t b0 = widen2_f16(__byte_perm(vw[0][t >> 2], vw[1][t >> 2], sel), 0x4140u);
          const uint32_t b1 = widen2_f16(__byte_perm(vw[2][t >> 2], vw[3][t >> 2], sel), 0x4140u);
          mma16816<true>(o[t], pa, b0, b1);
        }
      } else {
        // B = V rows via the transposing ldmatrix, two n-tiles of 8 d per load
        const int mi = lane >> 3, ri = lane & 7;
        const int row = rb + ri + 8 * (mi & 1);
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          uint32_t vf[4];
          ldsm_x4_trans(vf, swz(vb + (np >> 2) * kSlabStride, row, 2 * (np & 3) + (mi >> 1)));
          mma16816<Q8>(o[2 * np], pa, vf[0], vf[1]);
          mma16816<Q8>(o[2 * np + 1], pa, vf[2], vf[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---- merge the four warps' (max, sum, O)
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  named_bar_sync(1, kDecWarps * 32);  // every warp is done with the ring
  float* ow = reinterpret_cast<float*>(ring);           // [warp][16][D]
  float* mw = ow + kDecWarps * kDecMaxGroup * D;         // [warp][16]
  float* lw = mw + kDecWarps * kDecMaxGroup;             // [warp][16]
#pragma unroll
  for (int t = 0; t < D / 8; ++t) {
    const int d = 8 * t + 2 * cq;
    *reinterpret_cast<float2*>(ow + (warp * kDecMaxGroup + hA) * D + d) = make_float2(o[t][0], o[t][1]);
    *reinterpret_cast<float2*>(ow + (warp * kDecMaxGroup + hA + 8) * D + d) = make_float2(o[t][2], o[t][3]);
  }
  if (cq == 0) {
    mw[warp * kDecMaxGroup + hA] = mA;
    mw[warp * kDecMaxGroup + hA + 8] = mB;
    lw[warp * kDecMaxGroup + hA] = lA;
    lw[warp * kDecMaxGroup + hA + 8] = lB;
  }
  const bool single = !CL && a.n_split == 1;
  const int rank = blockIdx.x;  // rank in the cluster (CL): the cluster spans the slices
  if (has_new && (single || CL)) {
    // the new row's base-2 logit per query head (one warp per head)
    for (int hh = warp; hh < g; hh += kDecWarps) {
      float dot = 0.f;
      const __nv_bfloat16* qh = qs + hh * C::kQPitch;
      const __nv_bfloat16* kn = a.k_new + (int64_t)s * a.new_stride_seq + (int64_t)h * a.new_stride_head;
      for (int d = lane; d < D; d += 32) dot += __bfloat162float(qh[d]) * __bfloat162float(kn[d]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (lane == 0) xnew[hh] = dot * a.scale_log2;
    }
  }
  named_bar_sync(1, kDecWarps * 32);
  const int64_t head0 = (int64_t)s * a.h_q + (int64_t)h * g;  // first query head of the group
  // an int8 cache's value scale multiplies the cached rows' weighted sum (and
  // undoes the 2^14 its f16 weights carry; the sums of weights do not carry it)
  const float vmult = Q8 ? a.v_scale[(int64_t)s * a.h_kv + h] * (1.f / kP16) : 1.f;
  for (int idx = tid; idx < g * D; idx += kDecWarps * 32) {
    const int hh = idx / D, d = idx % D;
    // int8 values: column d sits where n-tile d % (D/8) keeps its column d / (D/8)
    const int dsrc = Q8 ? 8 * (d % (D / 8)) + d / (D / 8) : d;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, mw[w * kDecMaxGroup + hh]);
    float osum = 0.f, lsum = 0.f;
    if (m != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mx = mw[w * kDecMaxGroup + hh];
        if (mx != -INFINITY) {
          const float c = fast_exp2(mx - m);
          osum += c * ow[(w * kDecMaxGroup + hh) * D + dsrc];
          lsum += c * lw[w * kDecMaxGroup + hh];
        }
      }
    }
    if (single) {
      // the whole sequence is this slice: finish here
      float onum = osum * vmult, den = lsum;
      if (has_new) {
        const float xn = xnew[hh];
        const float top = fmaxf(m, xn);
        const float c = m == -INFINITY ? 0.f : fast_exp2(m - top);
        const float cn = fast_exp2(xn - top);
        const __nv_bfloat16* vn = a.v_new + (int64_t)s * a.new_stride_seq + (int64_t)h * a.new_stride_head;
        onum = c * osum * vmult + cn * __bfloat162float(vn[d]);
        den = c * lsum + cn;
      }
      a.out[(head0 + hh) * D + d] = (ok && den > 0.f) ? onum / den : 0.f;
    } else if (CL) {
      pbuf[hh * D + d] = osum;
      if (d == 0) pml[hh] = make_float2(m, lsum);
    } else {
      const int64_t slot = (head0 + hh) * a.n_split + split;
      a.part_o[slot * D + d] = osum;
      if (d == 0) a.part_ml[slot] = make_float2(m, lsum);
    }
  }
  if (single) return;
  if (CL) {
    // ---- slices of one cluster: every rank reads all ranks' (max, sum),
    // then merges its share of the output columns straight from the ranks'
    // shared memory
    cluster_sync_all();
    const int nsp = a.n_split;
    for (int i = tid; i < g * nsp; i += kDecWarps * 32) {
      const int hh = i / nsp, x = i % nsp;
      const uint32_t ad = cluster_map(smem_u32(pml + hh), (uint32_t)x);
      mlbuf[hh * kDecMaxSplit + x] = make_float2(ld_cluster_f32(ad), ld_cluster_f32(ad + 4));
    }
    named_bar_sync(1, kDecWarps * 32);
    for (int hh = warp; hh < g; hh += kDecWarps) {
      const float xn = has_new ? xnew[hh] : -INFINITY;
      float m = xn;
      for (int x = lane; x < nsp; x += 32) m = fmaxf(m, mlbuf[hh * kDecMaxSplit + x].x);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float lsum = 0.f;
      for (int x = lane; x < nsp; x += 32) {
        const float2 ml = mlbuf[hh * kDecMaxSplit + x];
        const float c = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - m);
        coef[hh * kDecMaxSplit + x] = c;
        lsum += c * ml.y;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      if (lane == 0) {
        const float cn = has_new ? fast_exp2(xn - m) : 0.f;
        cnew[hh] = cn;
        lsum += cn;
        rnorm[hh] = (ok && lsum > 0.f) ? 1.f / lsum : 0.f;
      }
    }
    named_bar_sync(1, kDecWarps * 32);
    constexpr int kC4 = D / 4;
    for (int j = rank + nsp * tid; j < g * kC4; j += nsp * kDecWarps * 32) {
      const int hh = j / kC4, c4 = j % kC4;
      const uint32_t base = smem_u32(pbuf + hh * D + 4 * c4);
      float4 v[kDecMaxCluster];
#pragma unroll
      for (int x = 0; x < kDecMaxCluster; ++x) {
        v[x] = x < nsp ? ld_cluster_f32x4(cluster_map(base, (uint32_t)x)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int x = 0; x < kDecMaxCluster; ++x) {
        const float c = x < nsp ? coef[hh * kDecMaxSplit + x] : 0.f;
        acc.x += c * v[x].x;
        acc.y += c * v[x].y;
        acc.z += c * v[x].z;
        acc.w += c * v[x].w;
      }
      acc.x *= vmult;
      acc.y *= vmult;
      acc.z *= vmult;
      acc.w *= vmult;
      if (has_new) {
        const __nv_bfloat16* vn =
            a.v_new + (int64_t)s * a.new_stride_seq + (int64_t)h * a.new_stride_head + 4 * c4;
        const float cn = cnew[hh];
        acc.x += cn * __bfloat162float(vn[0]);
        acc.y += cn * __bfloat162float(vn[1]);
        acc.z += cn * __bfloat162float(vn[2]);
        acc.w += cn * __bfloat162float(vn[3]);
      }
      const float rn = rnorm[hh];
      float* o4 = a.out + (head0 + hh) * D + 4 * c4;
      o4[0] = acc.x * rn;
      o4[1] = acc.y * rn;
      o4[2] = acc.z * rn;
      o4[3] = acc.w * rn;
    }
    cluster_sync_all();  // the partials stay readable until every rank is done
    return;
  }
  __threadfence();
  named_bar_sync(1, kDecWarps * 32);
  if (tid == 0) {
    const uint32_t before = atomicAdd(&a.count[(int64_t)s * a.h_kv + h], 1u);
    ctl[3] = before == (uint32_t)(a.n_split - 1);
  }
  named_bar_sync(1, kDecWarps * 32);
  if (!ctl[3]) return;

  // ---- last slice of this (sequence, KV head): merge the slices and the new row
  if (tid == 0) a.count[(int64_t)s * a.h_kv + h] = 0;  // every call leaves the counters at zero
  __threadfence();
  for (int i = tid; i < g * a.n_split; i += kDecWarps * 32) {
    const int hh = i / a.n_split, x = i % a.n_split;
    mlbuf[hh * kDecMaxSplit + x] = __ldcg(&a.part_ml[(head0 + hh) * a.n_split + x]);
  }
  for (int hh = warp; hh < g && has_new; hh += kDecWarps) {
    float dot = 0.f;
    const __nv_bfloat16* qh = qs + hh * C::kQPitch;
    const __nv_bfloat16* kn = a.k_new + (int64_t)s * a.new_stride_seq + (int64_t)h * a.new_stride_head;
    for (int d = lane; d < D; d += 32) dot += __bfloat162float(qh[d]) * __bfloat162float(kn[d]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (lane == 0) xnew[hh] = dot * a.scale_log2;
  }
  named_bar_sync(1, kDecWarps * 32);
  for (int hh = warp; hh < g; hh += kDecWarps) {
    const float xn = has_new ? xnew[hh] : -INFINITY;
    float m = xn;
    for (int x = lane; x < a.n_split; x += 32) m = fmaxf(m, mlbuf[hh * kDecMaxSplit + x].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float lsum = 0.f;
    for (int x = lane; x < a.n_split; x += 32) {
      const float2 ml = mlbuf[hh * kDecMaxSplit + x];
      const float c = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - m);
      coef[hh * kDecMaxSplit + x] = c;
      lsum += c * ml.y;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if (lane == 0) {
      const float cn = has_new ? fast_exp2(xn - m) : 0.f;
      cnew[hh] = cn;
      lsum += cn;
      rnorm[hh] = (ok && lsum > 0.f) ? 1.f / lsum : 0.f;
    }
  }
  named_bar_sync(1, kDecWarps * 32);
  // slices split across thread groups (float4 columns x slice groups): every
  // slice's partial is finite (empty slices wrote zeros), so the loads need no
  // condition and issue back to back
  constexpr int kD4 = D / 4;
  constexpr int kXG = kDecWarps * 32 / kD4;
  const int d4 = tid % kD4, xg = tid / kD4;
  float4* red = reinterpret_cast<float4*>(ring);  // [kXG][16][kD4]
  for (int hh = 0; hh < g; ++hh) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* src = reinterpret_cast<const float4*>(a.part_o + (head0 + hh) * a.n_split * D) + d4;
#pragma unroll 4
    for (int x = xg; x < a.n_split; x += kXG) {
      const float c = coef[hh * kDecMaxSplit + x];
      const float4 pv = __ldcg(src + (int64_t)x * kD4);
      acc.x += c * pv.x;
      acc.y += c * pv.y;
      acc.z += c * pv.z;
      acc.w += c * pv.w;
    }
    red[(xg * kDecMaxGroup + hh) * kD4 + d4] = acc;
  }
  named_bar_sync(1, kDecWarps * 32);
  for (int idx = tid; idx < g * D; idx += kDecWarps * 32) {
    const int hh = idx / D, d = idx % D;
    const float* rf = reinterpret_cast<const float*>(red);
    float acc = 0.f;
#pragma unroll
    for (int x = 0; x < kXG; ++x) acc += rf[(x * kDecMaxGroup + hh) * D + d];
    acc *= vmult;
    if (has_new) {
      const __nv_bfloat16* vn = a.v_new + (int64_t)s * a.new_stride_seq + (int64_t)h * a.new_stride_head;
      acc += cnew[hh] * __bfloat162float(vn[d]);
    }
    a.out[(head0 + hh) * D + d] = acc * rnorm[hh];
  }
}

// ------------------------------------------------------------------ host

struct DecPlan {
  bool cluster;  // slices merge inside a thread-block cluster
  bool q8;       // the cached rows are int8 codes
  int d, g, n_split;
  size_t zero_bytes, ml_off, o_off, total;
};

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Validates `p` and sizes the launch; returns AIRCACHE_OK or an error code.
int decode_plan(const aircache_decode_problem* p, DecPlan& pl) {
  if (!p) return AIRCACHE_ERR_INVALID_ARG;
  if (p->num_seqs < 0 || p->num_seqs > 65535 || p->h_q <= 0 || p->h_kv <= 0 || p->h_q % p->h_kv != 0 ||
      (p->head_dim != 64 && p->head_dim != 128) || p->kv_rows < 1 || (p->flags & ~AIRCACHE_DECODE_EARLY_CACHE) != 0 ||
      p->reserved1 != 0 ||
      p->kv_rows > 0x7fff0000LL || p->max_rows < 0)
    return AIRCACHE_ERR_INVALID_ARG;
  if (p->kv_dtype != AIRCACHE_BF16 && p->kv_dtype != AIRCACHE_INT8) return AIRCACHE_ERR_INVALID_ARG;
  if (p->dtype != AIRCACHE_BF16 || p->h_q / p->h_kv > kDecMaxGroup) return AIRCACHE_ERR_UNSUPPORTED;
  pl.q8 = p->kv_dtype == AIRCACHE_INT8;
  // tensor-map strides are multiples of 16 bytes: 8 bf16 or 16 int8 elements
  const int64_t sm = pl.q8 ? 16 : 8;
  if (pl.q8 && (!p->k_scale || !p->v_scale || p->kv_stride_row % sm != 0 || p->kv_stride_head % sm != 0))
    return AIRCACHE_ERR_INVALID_ARG;
  if (!p->q || !p->k || !p->v || !p->row_begin || !p->row_end || !p->out || (!p->k_new) != (!p->v_new))
    return AIRCACHE_ERR_INVALID_ARG;
  auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  if (!al16(p->k) || !al16(p->v) || !al16(p->q) || p->kv_stride_row <= 0 || p->kv_stride_head <= 0 ||
      p->kv_stride_row % 8 != 0 || p->kv_stride_head % 8 != 0 || p->q_stride_seq % 8 != 0 ||
      p->q_stride_head % 8 != 0 || p->q_stride_seq < 0 || p->q_stride_head < 0)
    return AIRCACHE_ERR_INVALID_ARG;
  if (p->k_new && (p->new_stride_seq < 0 || p->new_stride_head < 0)) return AIRCACHE_ERR_INVALID_ARG;
  if (p->row_index && (p->index_len < 1 || p->index_len > 0x7fff0000LL)) return AIRCACHE_ERR_INVALID_ARG;
  if (p->row_index && pl.q8) return AIRCACHE_ERR_UNSUPPORTED;  // gathered rows: bf16 only
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  pl.d = p->head_dim;
  pl.g = p->h_q / p->h_kv;
  const long long pairs = (long long)p->num_seqs * p->h_kv;
  // At most one wave of two resident CTAs per SM.  Slices of one (sequence,
  // KV head) form a thread-block cluster (up to 8) and merge through
  // distributed shared memory, which costs about a microsecond, so slices may
  // be as short as 128 rows.  Only long ranges over few (sequence, head) pairs
  // go wider than 8 slices; those merge through global memory (a fence, an
  // atomic, a reload: a few microseconds), with slices of at least 512 rows.
  const long long per_pair = pairs > 0 ? 2LL * sms / pairs : 1;
  auto clampll = [](long long x, long long lo, long long hi) { return x < lo ? lo : (x > hi ? hi : x); };
  long long want = clampll(std::min<long long>(per_pair, (p->max_rows + 127) / 128), 1, kDecMaxCluster);
  pl.cluster = want > 1;
  const long long wide = std::min<long long>(per_pair, (p->max_rows + 511) / 512);
  if (wide > kDecMaxCluster) {
    want = std::min<long long>(wide, kDecMaxSplit);
    pl.cluster = false;
  }
  pl.n_split = (int)want;
  const size_t slots = (size_t)p->num_seqs * p->h_q * pl.n_split;
  pl.zero_bytes = kDecZeroBlock + round256(sizeof(uint32_t) * (size_t)pairs);
  pl.ml_off = pl.zero_bytes;
  pl.o_off = pl.ml_off + round256(sizeof(float2) * slots);
  pl.total = pl.o_off + round256(sizeof(float) * slots * pl.d);
  return AIRCACHE_OK;
}

bool encode_arena(CUtensorMap* m, const void* base, const aircache_decode_problem* p) {
  auto enc = tma_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)p->head_dim, (cuuint64_t)p->h_kv, (cuuint64_t)p->kv_rows};
  if (p->kv_dtype == AIRCACHE_INT8) {
    // int8 codes: whole rows of one head per box (128 or 64 bytes), in the
    // swizzle of that width (the consumers undo it with swz8)
    cuuint64_t strides8[2] = {(cuuint64_t)p->kv_stride_head, (cuuint64_t)p->kv_stride_row};
    cuuint32_t box8[3] = {(cuuint32_t)p->head_dim, 1, (cuuint32_t)kDecRows};
    cuuint32_t es8[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides8, box8, es8,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               p->head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t strides[2] = {(cuuint64_t)p->kv_stride_head * 2, (cuuint64_t)p->kv_stride_row * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kDecRows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The arena as a 2-D tensor [kv_rows][heads' columns] whose box is one row of
// 64 elements: the form of the four-row gathers.
bool encode_gather(CUtensorMap* m, const void* base, const aircache_decode_problem* p) {
  auto enc = tma_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)((p->h_kv - 1) * p->kv_stride_head + p->head_dim), (cuuint64_t)p->kv_rows};
  cuuint64_t strides[1] = {(cuuint64_t)p->kv_stride_row * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool Q8, bool GA>
int launch_decode(const aircache_decode_problem* p, const DecPlan& pl, uint8_t* ws, cudaStream_t s) {
  auto launch_pdl3 = [](void (*k)(CUtensorMap, CUtensorMap, DecArgs), dim3 grid, dim3 block, size_t smem,
                        cudaStream_t st, const CUtensorMap& km, const CUtensorMap& vm, const DecArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, km, vm, a);
  };
  CUtensorMap km, vm;
  if (GA) {
    if (!encode_gather(&km, p->k, p) || !encode_gather(&vm, p->v, p)) return AIRCACHE_ERR_UNSUPPORTED;
  } else if (!encode_arena(&km, p->k, p) || !encode_arena(&vm, p->v, p)) {
    return AIRCACHE_ERR_UNSUPPORTED;
  }
  DecArgs a;
  a.q = static_cast<const __nv_bfloat16*>(p->q);
  a.k_new = static_cast<const __nv_bfloat16*>(p->k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(p->v_new);
  a.row_begin = p->row_begin;
  a.row_end = p->row_end;
  a.out = p->out;
  a.error = reinterpret_cast<int32_t*>(ws);
  a.count = reinterpret_cast<uint32_t*>(ws + kDecZeroBlock);
  a.part_ml = reinterpret_cast<float2*>(ws + pl.ml_off);
  a.part_o = reinterpret_cast<float*>(ws + pl.o_off);
  a.kv_rows = p->kv_rows;
  a.q_stride_seq = p->q_stride_seq;
  a.q_stride_head = p->q_stride_head;
  a.new_stride_seq = p->new_stride_seq;
  a.new_stride_head = p->new_stride_head;
  a.h_q = p->h_q;
  a.h_kv = p->h_kv;
  a.group = pl.g;
  a.n_split = pl.n_split;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  a.k_scale = p->k_scale;
  a.v_scale = p->v_scale;
  a.early = (p->flags & AIRCACHE_DECODE_EARLY_CACHE) != 0;
  a.row_index = p->row_index;
  a.range_len = GA ? p->index_len : p->kv_rows;
  a.col_stride_head = p->kv_stride_head;
  const int smem = DecCfg<D, Q8>::kSmem;
  const dim3 grid(pl.n_split, p->h_kv, p->num_seqs);
  if (pl.cluster) {
    if (allow_smem(reinterpret_cast<const void*>(&decode_kernel<D, true, Q8, GA>), smem) != cudaSuccess)
      return AIRCACHE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pl.n_split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.early ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, decode_kernel<D, true, Q8, GA>, km, vm, a) != cudaSuccess) return AIRCACHE_ERR_CUDA;
  } else {
    if (allow_smem(reinterpret_cast<const void*>(&decode_kernel<D, false, Q8, GA>), smem) != cudaSuccess)
      return AIRCACHE_ERR_CUDA;
    if (a.early) {
      if (launch_pdl3(decode_kernel<D, false, Q8, GA>, grid, dim3(kDecThreads), smem, s, km, vm, a) != cudaSuccess)
        return AIRCACHE_ERR_CUDA;
    } else {
      decode_kernel<D, false, Q8, GA><<<grid, kDecThreads, smem, s>>>(km, vm, a);
    }
  }
  return cudaGetLastError() == cudaSuccess ? AIRCACHE_OK : AIRCACHE_ERR_CUDA;
}

}  // namespace
}  // namespace aircache

using namespace aircache;

extern "C" {

size_t aircache_decode_workspace_size(const aircache_decode_problem* p) {
  DecPlan pl;
  return decode_plan(p, pl) == AIRCACHE_OK ? pl.total : 0;
}

int aircache_decode_splits(const aircache_decode_problem* p) {
  DecPlan pl;
  return decode_plan(p, pl) == AIRCACHE_OK ? pl.n_split : -1;
}

int aircache_decode(const aircache_decode_problem* p, void* ws, size_t ws_bytes, void* stream) {
  DecPlan pl;
  const int rc = decode_plan(p, pl);
  if (rc != AIRCACHE_OK) return rc;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0) return AIRCACHE_ERR_INVALID_ARG;
  if (ws_bytes < pl.total) return AIRCACHE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (p->num_seqs == 0) return AIRCACHE_OK;
  if (pl.q8) return pl.d == 128 ? launch_decode<128, true, false>(p, pl, w, s) : launch_decode<64, true, false>(p, pl, w, s);
  if (p->row_index)
    return pl.d == 128 ? launch_decode<128, false, true>(p, pl, w, s) : launch_decode<64, false, true>(p, pl, w, s);
  return pl.d == 128 ? launch_decode<128, false, false>(p, pl, w, s) : launch_decode<64, false, false>(p, pl, w, s);
}

}  // extern "C"
