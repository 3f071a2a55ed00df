// Per-layer top-k selection of visual positions by I_v (the retention step that
// the AirCache budget feeds: the keep_l highest-scoring visual tokens of layer l
// stay in the cache, ties to the lower position, emitted in ascending order).
//
// One CTA per (request, layer).  I_v is mapped to order-preserving 32-bit keys;
// a 4-digit (8-bit) MSB-first radix select finds the exact keep-th largest key
// T and how many keys equal to T are still wanted; a final ordered sweep emits
// every key > T plus the lowest-position keys == T, in ascending position, via
// block-wide ballot scans.  Integer work only: the result is exact and
// deterministic.
#include "internal.cuh"

namespace aircache {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

struct SelectArgs {
  Dev p;
  Ws w;
};

// Larger float <=> larger key (handles -0.0 and negatives, which I_v never has).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block prefix of a per-thread flag; returns this thread's prefix,
// *total receives the block total.
__device__ __forceinline__ int block_scan_flag(bool f, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, f);
  const int before = __popc(bal & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < kSelWarps; ++i) {
    base += (i < warp) ? wsum[i] : 0;
    tot += wsum[i];
  }
  *total = tot;
  return base + before;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const __grid_constant__ SelectArgs a) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int b = blockIdx.x, l = blockIdx.y, u = l * p.B + b;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ unsigned hist[256];
  __shared__ int wsum[kSelWarps];
  __shared__ unsigned sel_digit, sel_above;
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

  uint32_t prefix = 0, mask = 0;
  unsigned want = (unsigned)k;  // keys >= the answer still to account for
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kSelThreads) {
      const uint32_t key = order_key(__ldcg(x + i));
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
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
          }
          run += cnt[i];
        }
      }
    }
    __syncthreads();
    want -= sel_above;
    prefix |= sel_digit << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix = exact key of the keep-th largest; take all keys > prefix and the
  // first `want` keys == prefix in position order.
  int base = 0, eq_base = 0;
  for (int i0 = 0; i0 < n; i0 += kSelThreads) {
    const int i = i0 + tid;
    const uint32_t key = (i < n) ? order_key(__ldcg(x + i)) : 0u;
    const bool eq = i < n && key == prefix;
    const bool gt = i < n && key > prefix;
    int eq_total;
    const int eq_rank = eq_base + block_scan_flag(eq, wsum, &eq_total);
    const bool take = gt || (eq && eq_rank < (int)want);
    int tk_total;
    const int pos = base + block_scan_flag(take, wsum, &tk_total);
    if (take) out[pos] = i;
    base += tk_total;
    eq_base += eq_total;
  }
  (void)lane;
}

}  // namespace

cudaError_t launch_select(const Dev& p, const Ws& w, cudaStream_t s) {
  SelectArgs a;
  a.p = p;
  a.w = w;
  select_kernel<<<dim3(p.B, p.L), kSelThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace aircache
