// Compaction of the kept rows into the decode cache (AirCache notes, "Loss /
// training strategy": the compressed cache is what decoding reads; every text
// position is kept after the selected visual positions).
//
// The output arena holds, for each layer l and request b in that order, the
// rows [K_v[idx]; K_t] (and the same rows of V) as dense [h_kv][head_dim] rows.
// A persistent grid of warps walks the output rows; each warp finds its row's
// (l, b) by binary search over the row offsets (staged in shared memory; after
// the budget-mode selection every CTA forms them itself from the keep counts,
// and CTA 0 writes them out),
// resolves the source position and copies the K and V rows with 16-byte loads
// and stores.  Bit-exact: no arithmetic touches the data.
#include "internal.cuh"
#include "ptx.cuh"
#include "reduce.cuh"

namespace aircache {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyWarps = kCopyThreads / 32;
constexpr int kMaxSmemOffsets = 4096;

struct CompactArgs {
  Dev p;
  LayerPtrs lp;
  Ws w;
  void* out_k;
  void* out_v;
  int64_t capacity;  // rows out_k / out_v hold (or entries of row_index)
  int32_t* row_index;  // non-null: write each row's prompt position instead of copying it
  int make_offsets;    // 1: form the row offsets from the keep counts (at most kMaxSmemOffsets units)
};

__global__ void __launch_bounds__(kCopyThreads) compact_kernel(const __grid_constant__ CompactArgs a) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ long long offs[kMaxSmemOffsets + 1];
  __shared__ long long seg[kCopyWarps + 1];
  pdl_trigger();
  pdl_wait();  // selections, keep counts and row offsets
  if (*(volatile int32_t*)w.error != 0) return;
  const int units = p.L * p.B;
  const bool in_smem = units <= kMaxSmemOffsets;
  if (a.make_offsets && in_smem) {
    // exclusive prefix of keep + N_t over the units, in shared memory; CTA 0
    // also writes it to the caller's offsets (and flags a capacity overflow)
    write_offsets<kCopyThreads>(p, w.keep, reinterpret_cast<int64_t*>(offs), blockIdx.x == 0 ? w.error : nullptr,
                                a.capacity, seg, tid, 1);
    __syncthreads();
    if (blockIdx.x == 0)
      for (int i = tid; i <= units; i += kCopyThreads) w.out_offsets[i] = offs[i];
  } else if (in_smem) {
    for (int i = tid; i <= units; i += kCopyThreads) offs[i] = w.out_offsets[i];
  }
  __syncthreads();
  const long long* off = in_smem ? offs : reinterpret_cast<const long long*>(w.out_offsets);
  const long long total = off[units];
  if (total > a.capacity || total < 0) {
    if (tid == 0) set_error(w.error, AIRCACHE_ERR_CAPACITY);
    return;
  }

  const int esize = (p.dtype == AIRCACHE_BF16) ? 2 : 4;
  const int vec_per_head = p.d * esize / 16;
  const int vec_per_row = p.h_kv * vec_per_head;
  const int64_t elems_per_vec = 16 / esize;
  uint4* outk = reinterpret_cast<uint4*>(a.out_k);
  uint4* outv = reinterpret_cast<uint4*>(a.out_v);

  const long long warps = (long long)gridDim.x * kCopyWarps;
  for (long long row = (long long)blockIdx.x * kCopyWarps + warp; row < total; row += warps) {
    // unit u with off[u] <= row < off[u+1]
    int lo = 0, hi = units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int u = lo, l = u / p.B, b = u % p.B;
    const long long j = row - off[u];
    Req R;
    const bool ok = load_req(p, b, R);
    const int kp = w.keep[u];
    // kept visual rows first, then every text row in text order; with one set
    // per KV head the visual row differs per head (resolved per vector below)
    const size_t set0 = p.head_sets ? (size_t)l * p.h_kv : (size_t)l;
    int64_t tok = -1;
    if (j < kp) {
      const int64_t pos = w.idx[set0 * p.total_visual + R.vis0 + j];
      if (pos >= 0 && pos < R.n_v) tok = vis_tok(R, pos);
    } else if (j - kp < R.n_t) {
      tok = text_tok(R, j - kp);
    }
    if (!ok || tok < 0) {
      if (lane == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
      continue;
    }
    if (a.row_index) {  // the row list of a gather-fused decode: no copy
      if (lane == 0) a.row_index[row] = (int32_t)tok;
      continue;
    }
    const char* kb = reinterpret_cast<const char*>(a.lp.k[l]);
    const char* vb = reinterpret_cast<const char*>(a.lp.v[l]);
    uint4 kbuf[4], vbuf[4];
    for (int v0 = 0; v0 < vec_per_row; v0 += 4 * 32) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int vec = v0 + i * 32 + lane;
        if (vec < vec_per_row) {
          const int head = vec / vec_per_head, part = vec % vec_per_head;
          int64_t t = tok;
          if (p.head_sets && j < kp && head > 0) {
            const int64_t pos = w.idx[(set0 + head) * p.total_visual + R.vis0 + j];
            t = (pos >= 0 && pos < R.n_v) ? vis_tok(R, pos) : tok;
            if (pos < 0 || pos >= R.n_v) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
          }
          const int64_t eo = t * p.kv_stride_tok + head * p.kv_stride_head + part * elems_per_vec;
          kbuf[i] = __ldg(reinterpret_cast<const uint4*>(kb + eo * esize));
          vbuf[i] = __ldg(reinterpret_cast<const uint4*>(vb + eo * esize));
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int vec = v0 + i * 32 + lane;
        if (vec < vec_per_row) {
          outk[row * vec_per_row + vec] = kbuf[i];
          outv[row * vec_per_row + vec] = vbuf[i];
        }
      }
    }
  }
}

}  // namespace

bool compact_makes_offsets(const Dev& p) { return (long long)p.L * p.B <= kMaxSmemOffsets; }

cudaError_t launch_compact(const Dev& p, const LayerPtrs& lp, const Ws& w, void* out_k, void* out_v,
                           int64_t capacity, cudaStream_t s, bool make_offsets) {
  CompactArgs a;
  a.make_offsets = make_offsets && compact_makes_offsets(p) ? 1 : 0;
  a.p = p;
  a.lp = lp;
  a.w = w;
  a.out_k = out_k;
  a.out_v = out_v;
  a.capacity = capacity;
  a.row_index = nullptr;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_pdl(compact_kernel, dim3(sms * 4), dim3(kCopyThreads), 0, s, a);
}

}  // namespace aircache

namespace aircache {

cudaError_t launch_row_index(const Dev& p, const LayerPtrs& lp, const Ws& w, int32_t* row_index, int64_t capacity,
                             cudaStream_t s) {
  CompactArgs a;
  a.p = p;
  a.lp = lp;
  a.w = w;
  a.out_k = nullptr;
  a.out_v = nullptr;
  a.capacity = capacity;
  a.row_index = row_index;
  a.make_offsets = 0;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_pdl(compact_kernel, dim3(sms), dim3(kCopyThreads), 0, s, a);
}

}  // namespace aircache
