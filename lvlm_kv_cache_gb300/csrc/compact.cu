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
//
// Bulk form (compact_bulk_kernel; every KV head of a token in one contiguous
// row, one index set per layer): each CTA takes chunks of R consecutive output
// rows (its first two by index, the rest claimed from a counter).  R threads
// resolve the chunk's source tokens; each thread then moves its row's K and V
// rows into shared memory with bulk copies (a run of consecutive tokens as one
// copy; one mbarrier per buffer counts the bytes), and one thread writes the
// chunk back with two bulk stores (the chunk's output rows are contiguous).
// A chunk is resolved two iterations before it is stored and loaded one
// before, so the index lookups and the loads overlap the stores.
#include "internal.cuh"
#include "ptx.cuh"
#include "reduce.cuh"
#include "timeline.cuh"

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
  AIRCACHE_KT(6);
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

constexpr int kBulkThreads = 128;
constexpr int kBulkBuf = 48 * 1024;  // one buffer: R rows of K, then R rows of V
constexpr int kBulkMaxRows = 64;

__global__ void __launch_bounds__(kBulkThreads) compact_bulk_kernel(const __grid_constant__ CompactArgs a) {
  AIRCACHE_KT(6);
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int tid = threadIdx.x;
  extern __shared__ __align__(128) unsigned char bsm[];  // [2][kBulkBuf], then the row offsets [L*B + 1]
  long long* offs = reinterpret_cast<long long*>(bsm + 2 * kBulkBuf);
  __shared__ long long seg[kBulkThreads / 32 + 1];
  __shared__ long long tok_s[3][kBulkMaxRows];  // three resolved chunks: stored, loading, next
  __shared__ long long claim_s[4];              // claimed chunk ids, by iteration
  __shared__ __align__(8) uint64_t full[2];
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
  }
  pdl_trigger();
  pdl_wait();  // selections, keep counts (and row offsets)
  if (*(volatile int32_t*)w.error != 0) return;
  const int units = p.L * p.B;  // at most kMaxSmemOffsets on this path
  if (a.make_offsets) {
    write_offsets<kBulkThreads>(p, w.keep, reinterpret_cast<int64_t*>(offs), blockIdx.x == 0 ? w.error : nullptr,
                                a.capacity, seg, tid, 1);
    __syncthreads();
    if (blockIdx.x == 0)
      for (int i = tid; i <= units; i += kBulkThreads) w.out_offsets[i] = offs[i];
  } else {
    for (int i = tid; i <= units; i += kBulkThreads) offs[i] = w.out_offsets[i];
  }
  __syncthreads();
  const long long total = offs[units];
  if (total > a.capacity || total < 0) {
    if (tid == 0) set_error(w.error, AIRCACHE_ERR_CAPACITY);
    return;
  }
  const int esize = (p.dtype == AIRCACHE_BF16) ? 2 : 4;
  const uint32_t row_bytes = (uint32_t)(p.h_kv * p.d * esize);
  // rows per chunk: at most what a buffer holds, evened out so that the rows
  // split into a whole number of equal rounds of chunks over the grid (the
  // last chunks are then as long as the others)
  const int Rmax = min(kBulkMaxRows, (int)(kBulkBuf / 2 / row_bytes));
  const long long per_cta = (total + (long long)gridDim.x * Rmax - 1) / ((long long)gridDim.x * Rmax);
  const int R = per_cta > 0 ? (int)((total + gridDim.x * per_cta - 1) / (gridDim.x * per_cta)) : Rmax;
  const long long chunks = (total + R - 1) / R;
  // thread r < R: the source token of row r of chunk c into slot sl (-1: past the end or invalid)
  auto resolve = [&](long long c, int sl) {
    if (tid >= R) return;
    const long long row = c * R + tid;
    long long tok = -1;
    if (c < chunks && row < total) {
      int lo = 0, hi = units - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= row) lo = mid; else hi = mid - 1;
      }
      const int u = lo, l = u / p.B, b = u % p.B;
      const long long j = row - offs[u];
      Req Rq;
      const bool ok = load_req(p, b, Rq);
      const int kp = w.keep[u];
      if (j < kp) {
        const int64_t pos = w.idx[(size_t)l * p.total_visual + Rq.vis0 + j];
        if (pos >= 0 && pos < Rq.n_v) tok = vis_tok(Rq, pos);
      } else if (j - kp < Rq.n_t) {
        tok = text_tok(Rq, j - kp);
      }
      if (!ok || tok < 0) {
        set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
        tok = -1;
      }
      tok = tok >= 0 ? ((long long)l << 40) | tok : -1;  // the layer rides in the high bits
    }
    tok_s[sl][tid] = tok;
  };
  // bytes of the rows of slot sl (thread 0, for the buffer's expected-transaction count)
  auto chunk_bytes = [&](int sl) {
    uint32_t bytes = 0;
    for (int r = 0; r < R; ++r)
      if (tok_s[sl][r] >= 0) bytes += 2 * row_bytes;
    return bytes;
  };
  // rows of consecutive tokens are adjacent in K and V (dense token stride)
  const bool dense = (size_t)p.kv_stride_tok * esize == row_bytes;
  // thread r < R: the bulk loads of slot sl's rows into buffer buf, issued in
  // parallel by the threads (one thread issuing a chunk's 2R copies back to back
  // set the pace of a chunk); a run of consecutive tokens (the text rows, and
  // neighbouring kept visual rows) is one copy, issued by the run's first row
  auto load_row = [&](int sl, int buf) {
    if (tid >= R) return;
    const long long t = tok_s[sl][tid];
    if (t < 0) return;
    if (dense && tid > 0 && tok_s[sl][tid - 1] >= 0 && tok_s[sl][tid - 1] == t - 1) return;  // inside a run
    int n = 1;
    if (dense)
      while (tid + n < R && tok_s[sl][tid + n] == t + n) ++n;
    unsigned char* kd = bsm + buf * kBulkBuf;
    unsigned char* vd = kd + R * row_bytes;
    const int l = (int)(t >> 40);
    const long long tok = t & ((1LL << 40) - 1);
    const size_t off = (size_t)tok * p.kv_stride_tok * esize;
    bulk_g2s(kd + tid * row_bytes, reinterpret_cast<const char*>(a.lp.k[l]) + off, n * row_bytes, &full[buf]);
    bulk_g2s(vd + tid * row_bytes, reinterpret_cast<const char*>(a.lp.v[l]) + off, n * row_bytes, &full[buf]);
  };
  // Chunks are claimed: the first two of a CTA are blockIdx.x and
  // blockIdx.x + grid, the later ones come from a counter (from 2 * grid on),
  // so that CTAs on SMs that copy faster take more of them.  Chunk k of the CTA
  // is claimed three iterations ahead (by the last thread, which resolves no
  // row) into claim_s[k % 4], resolved two ahead into slot k % 3, loaded one
  // ahead into buffer k % 2 and stored in iteration k.
  const long long G = gridDim.x;
  auto claim = [&]() { return 2 * G + (long long)atomicAdd(w.cnt_cmp, 1u); };
  if (tid == kBulkThreads - 1) claim_s[2] = claim();
  if (tid == 0) {
    claim_s[0] = blockIdx.x;
    claim_s[1] = blockIdx.x + G;
  }
  long long c = blockIdx.x;
  resolve(c, 0);
  resolve(c + G, 1);
  __syncthreads();
  if (tid == 0 && c < chunks) mbar_arrive_expect_tx(&full[0], chunk_bytes(0));
  __syncthreads();
  if (c < chunks) load_row(0, 0);
  for (int k = 0; c < chunks; ++k) {
    const int buf = k & 1;
    const long long cn = claim_s[(k + 1) & 3];
    if (tid == kBulkThreads - 1) claim_s[(k + 3) & 3] = cn < chunks ? claim() : chunks;
    resolve(claim_s[(k + 2) & 3], (k + 2) % 3);  // overlaps the loads and stores in flight
    __syncthreads();
    if (tid == 0 && cn < chunks) {
      bulk_wait_read_all();  // the stores of chunk k - 1 have read buffer buf ^ 1
      mbar_arrive_expect_tx(&full[buf ^ 1], chunk_bytes((k + 1) % 3));
    }
    __syncthreads();
    if (cn < chunks) load_row((k + 1) % 3, buf ^ 1);
    if (tid == 0) {
      if (!mbar_wait(&full[buf], (uint32_t)((k >> 1) & 1))) {
        set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      } else {
        const int nr = (int)min((long long)R, total - c * R);
        const unsigned char* kd = bsm + buf * kBulkBuf;
        bulk_s2g(reinterpret_cast<char*>(a.out_k) + (size_t)c * R * row_bytes, kd, nr * row_bytes);
        bulk_s2g(reinterpret_cast<char*>(a.out_v) + (size_t)c * R * row_bytes, kd + R * row_bytes, nr * row_bytes);
        bulk_commit();
      }
    }
    __syncthreads();  // slot k % 3 and claim k are rewritten by the next iterations
    c = cn;
  }
  if (tid == 0) bulk_wait_all();  // the stores are complete before the buffers go away
}

}  // namespace

bool compact_bulk_ok(const Dev& p, const LayerPtrs& lp) {
  const int esize = (p.dtype == AIRCACHE_BF16) ? 2 : 4;
  const long long row_bytes = (long long)p.h_kv * p.d * esize;
  if (p.head_sets || (p.h_kv > 1 && p.kv_stride_head != p.d) || row_bytes > kBulkBuf / 2 ||
      (long long)p.L * p.B > kMaxSmemOffsets)
    return false;
  // values in page-locked host memory (read in place): the warp copies
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, lp.v[0]) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

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
  if (compact_bulk_ok(p, lp)) {
    const int smem = 2 * kBulkBuf + (int)sizeof(long long) * (p.L * p.B + 1);
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(compact_bulk_kernel), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(compact_bulk_kernel, dim3(sms * 2), dim3(kBulkThreads), smem, s, a);
  }
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

AIRCACHE_TIMELINE_EXPORT(compact)
