// Per-layer top-k selection of visual positions by I_v (the retention step that
// the AirCache budget feeds: the keep_l highest-scoring visual tokens of layer l
// stay in the cache, ties to the lower position, emitted in ascending order).
//
// One CTA of 1024 threads per (request, layer).  I_v is mapped to
// order-preserving 32-bit keys, held in shared memory when the unit fits
// (otherwise re-read from global memory each pass).  A 4-digit (8-bit)
// MSB-first radix select finds the exact keep-th largest key T and how many
// keys equal to T are still wanted; histogram increments are aggregated over
// the lanes of a warp that share a digit, and after the first digit the keys
// that can still be T are compacted so the later passes touch only them.  A
// final sweep in which each thread owns a contiguous run of positions emits
// every key > T plus the lowest-position keys == T, in ascending position,
// with block-wide exclusive scans (one when every key == T is taken).
// Integer work only: the result is exact and deterministic.
#include "internal.cuh"
#include "ptx.cuh"

namespace aircache {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSmemKeys = 24 * 1024;  // units up to this many keys are staged in shared memory

struct SelectArgs {
  Dev p;
  Ws w;
  int smem_keys;  // capacity of the dynamic shared-memory key buffer
};

// Larger float <=> larger key (handles -0.0 and negatives, which I_v never has).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix over the CTA of one int per thread; *total receives the sum.
// `wsum` is shared scratch of kSelWarps + 1 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();  // earlier readers of wsum are done
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int t = wsum[lane];  // kSelWarps == 32
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += x;
    }
    wsum[lane] = ti - t;
    if (lane == 31) wsum[kSelWarps] = ti;
  }
  __syncthreads();
  *total = wsum[kSelWarps];
  return wsum[warp] + incl - v;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const __grid_constant__ SelectArgs a) {
  static_assert(kSelWarps == 32, "the warp-total scan assumes 32 warps");
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int b = blockIdx.x, l = blockIdx.y, u = l * p.B + b;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  extern __shared__ uint32_t keys_s[];  // [smem_keys] keys, then [smem_keys] candidates
  __shared__ unsigned hist[256];
  __shared__ int wsum[kSelWarps + 1];
  __shared__ unsigned sel_digit, sel_above, sel_count;
  pdl_trigger();
  pdl_wait();  // I_v and the keep counts
  if (*(volatile int32_t*)w.error != 0) return;
  Req R;
  if (!load_req(p, b, R)) {
    if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  const int n = R.n_v;
  const int k = w.keep[u];
  if (k < 0 || k > n) {
    if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  const float* x = w.iv + (size_t)l * p.total_visual + R.vis0;
  int32_t* out = w.idx + (size_t)l * p.total_visual + R.vis0;
  if (k == n) {
    for (int i = tid; i < n; i += kSelThreads) out[i] = i;
    return;
  }
  if (k == 0) return;
  const bool staged = n <= a.smem_keys;
  if (staged) {
    for (int i0 = tid; i0 < n; i0 += 8 * kSelThreads) {
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = (i0 + q * kSelThreads < n) ? __ldcg(x + i0 + q * kSelThreads) : 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (i0 + q * kSelThreads < n) keys_s[i0 + q * kSelThreads] = order_key(v[q]);
      }
    }
  }
  auto key_at = [&](int i) -> uint32_t { return staged ? keys_s[i] : order_key(__ldcg(x + i)); };

  uint32_t* cand = keys_s + a.smem_keys;  // keys still able to be the answer (staged units)
  int n_cand = n;                         // after the first digit: their number
  uint32_t prefix = 0, mask = 0;
  unsigned want = (unsigned)k;  // keys >= the answer still to account for
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    const bool from_cand = staged && shift < 24;
    const int m = from_cand ? n_cand : n;
    for (int i0 = 0; i0 < m; i0 += kSelThreads) {
      const int i = i0 + tid;
      const uint32_t key = i < m ? (from_cand ? cand[i] : key_at(i)) : 0u;
      const bool in = i < m && (key & mask) == prefix;
      const unsigned digit = in ? ((key >> shift) & 255u) : 256u;
      // one increment per distinct digit of the warp
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], (unsigned)__popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane owns digits [8*(31-lane), 8*(31-lane)+8): lane 0 the highest
      unsigned cnt[8];
      unsigned lsum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = hist[8 * (31 - lane) + (7 - i)];  // descending digits
        lsum += cnt[i];
      }
      unsigned incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const unsigned excl = incl - lsum;  // count of digits above this lane's range
      if (excl < want && want <= incl) {
        unsigned run = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (run < want && want <= run + cnt[i]) {
            sel_digit = 8 * (31 - lane) + (7 - i);
            sel_above = run;
            sel_count = cnt[i];
          }
          run += cnt[i];
        }
      }
    }
    __syncthreads();
    want -= sel_above;
    prefix |= sel_digit << shift;
    mask |= 255u << shift;
    if (staged && shift == 24) {
      // compact the keys whose top digit is the selected one (order is irrelevant
      // here: one shared counter, one atomic per warp and pass over the keys)
      if (tid == 0) sel_above = 0;
      __syncthreads();
      for (int i0 = 0; i0 < n; i0 += kSelThreads) {
        const int i = i0 + tid;
        const bool c = i < n && (keys_s[i] & mask) == prefix;
        const unsigned bal = __ballot_sync(0xffffffffu, c);
        int base = 0;
        if (lane == 0 && bal) base = (int)atomicAdd(&sel_above, (unsigned)__popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (c) cand[base + __popc(bal & ((1u << lane) - 1u))] = keys_s[i];
      }
      __syncthreads();
      n_cand = (int)sel_above;
      __syncthreads();
    }
  }
  const unsigned eq_all = sel_count;  // keys equal to the answer
  // prefix = exact key of the keep-th largest: take every key > prefix and the
  // first `want` keys == prefix in position order.  Thread tid owns positions
  // [tid * per, tid * per + per).
  const int per = (n + kSelThreads - 1) / kSelThreads;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  if (want == eq_all) {
    // every key equal to the answer is taken: keys >= prefix, one scan
    int n_take = 0;
    for (int i = i0; i < i1; ++i) n_take += key_at(i) >= prefix ? 1 : 0;
    int take_total;
    int pos = block_excl_scan(n_take, wsum, &take_total);
    for (int i = i0; i < i1; ++i) {
      if (key_at(i) >= prefix) out[pos++] = i;
    }
    return;
  }
  int n_eq = 0;
  for (int i = i0; i < i1; ++i) n_eq += key_at(i) == prefix ? 1 : 0;
  int eq_total;
  int eq_rank = block_excl_scan(n_eq, wsum, &eq_total);
  int n_take = 0;
  {
    int r = eq_rank;
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = key_at(i);
      if (key > prefix) {
        ++n_take;
      } else if (key == prefix) {
        if (r < (int)want) ++n_take;
        ++r;
      }
    }
  }
  int take_total;
  int pos = block_excl_scan(n_take, wsum, &take_total);
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = key_at(i);
    if (key > prefix) {
      out[pos++] = i;
    } else if (key == prefix) {
      if (eq_rank < (int)want) out[pos++] = i;
      ++eq_rank;
    }
  }
  (void)lane;
}

}  // namespace

cudaError_t launch_select(const Dev& p, const Ws& w, cudaStream_t s) {
  SelectArgs a;
  a.p = p;
  a.w = w;
  a.smem_keys = p.max_visual < kSmemKeys ? p.max_visual : kSmemKeys;
  const int smem = 2 * (int)sizeof(uint32_t) * a.smem_keys;  // keys + candidates
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(select_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_kernel, dim3(p.B, p.L), dim3(kSelThreads), smem, s, a);
}

}  // namespace aircache
