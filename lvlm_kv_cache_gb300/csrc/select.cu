// Per-layer top-k selection of visual positions by I_v (the retention step that
// the AirCache budget feeds: the keep_l highest-scoring visual tokens of layer l
// stay in the cache, ties to the lower position, emitted in ascending order).
//
// One CTA of 1024 threads per (request, layer).  I_v is mapped to
// order-preserving 32-bit keys, held in shared memory when the unit fits
// (otherwise re-read from global memory each pass).  An MSB-first radix select
// finds the exact keep-th largest key T and how many keys equal to T are still
// wanted (it stops early once every key of the selected bucket is taken).  The
// digits are 11 bits wide and start below the highest bit in which the unit's
// smallest and largest keys differ: the I_v of a layer spans a few octaves, so
// digits taken from the top of the word would put nearly every key in one
// bucket (and its shared-memory counter).  After the first digit the keys that
// can still be T are compacted, so the later passes touch only them.  The emission splits the positions into 32
// contiguous segments, one per warp, and takes every key > T plus the
// lowest-position keys == T with ballots and one scan of the warp totals, so
// the output is in ascending position order.
// Integer work only: the result is exact and deterministic.
//
// On the streaming path of the fused call the kernel also takes the layer
// budget ("Key design 2") off the critical path of a kernel of its own.
// Passes 2 and 2k have already merged each unit's key-block moment records
// into its layer statistics (s_t, s_k) (float-float).  While its keys are
// staged, the CTA reads the statistics of every layer of its request, warp 0
// turns them into the request's keep counts (the same arithmetic in every CTA
// of the request), and the CTA keeps its own layer's count.  The
// compacted-cache row offsets then come from the compaction kernel (or, for
// more units than it stages, from the last CTA of this one to arrive).
#include "internal.cuh"
#include "ptx.cuh"
#include "reduce.cuh"
#include "timeline.cuh"

namespace aircache {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSmemKeys = 24 * 1024;  // units up to this many keys are staged in shared memory
constexpr int kMaxBins = 2048;        // widest digit: 11 bits
constexpr int kEmitStep = 2;          // 32-key groups per step of the emission sweeps (short code: it runs once)

struct SelectArgs {
  Dev p;
  Ws w;
  int smem_keys;          // capacity of the dynamic shared-memory key buffer
  int budget;             // 1 (streaming path): the CTA first computes its request's layer budgets
                          // from the layer statistics that passes 2 / 2k merged, and writes its own
                          // layer's keep count and statistics
  int64_t out_capacity;   // rows of the output arena (budget mode)
  int offsets;            // budget mode: the last CTA writes the row offsets (else the compaction does)
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
  AIRCACHE_KT(5);
  static_assert(kSelWarps == 32, "the warp-total scans assume 32 warps");
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int b = blockIdx.x, l = blockIdx.y, u = l * p.B + b;
  const int hs = blockIdx.z;  // KV head of the set (one set per layer unless head_sets)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  extern __shared__ uint32_t keys_s[];  // [smem_keys] keys, then [smem_keys] candidates
  __shared__ unsigned hist[kMaxBins];
  __shared__ int wsum[kSelWarps + 1];
  __shared__ int wgt[kSelWarps + 1], weq[kSelWarps + 1];
  __shared__ unsigned sel_digit, sel_above, sel_count, n_cand_s;
  __shared__ uint32_t wmin[kSelWarps], wmax[kSelWarps];
  __shared__ ff st_s[AIRCACHE_MAX_LAYERS], sk_s[AIRCACHE_MAX_LAYERS];
  __shared__ int32_t keep_s[AIRCACHE_MAX_LAYERS];
  __shared__ long long off_seg[kSelWarps + 1];
  __shared__ int last_s;
  pdl_trigger();
  pdl_wait();  // I_v, and the keep counts or (budget mode) the moment records
  if (*(volatile int32_t*)w.error != 0) return;  // an earlier kernel reported an error
  Req R{};
  const bool ok_req = load_req(p, b, R);
  if (!ok_req) R.vis0 = 0;
  const int n = ok_req ? R.n_v : 0;
  // one set per layer from I_v, or one per KV head from that KV group's I_v
  const size_t set = p.head_sets ? (size_t)l * p.h_kv + hs : (size_t)l;
  const float* x = (p.head_sets ? w.ivh : w.iv) + set * p.total_visual + R.vis0;
  int32_t* out = w.idx + set * p.total_visual + R.vis0;
  const bool staged = n <= a.smem_keys;
  if (a.budget && ok_req && warp == 0) {
    // warp 0: the request's keep counts, while the other warps stage the keys.
    // (s_t, s_k) of every layer of the request were merged from the unit's
    // moment records by the pass-2 (or pass-2k) CTA that wrote its last one.
    for (int ll = lane; ll < p.L; ll += 32) {
      const float4 v = __ldcg(&w.lstat[ll * p.B + b]);
      st_s[ll] = ff{v.x, v.y};
      sk_s[ll] = ff{v.z, v.w};
    }
    __syncwarp();
    request_budget_warp_put(
        p, R.n_v,
        [&](int ll, ff& st, ff& sk) {
          st = st_s[ll];
          sk = sk_s[ll];
        },
        [&](int ll, int32_t kk) { keep_s[ll] = kk; }, lane);
  }
  // stage the keys (when they fit) and find the smallest and largest (in
  // budget mode warp 0 takes no part)
  const int sw = a.budget ? 1 : 0;                  // warps left out of the staging
  const int st0 = tid - 32 * sw, nst = kSelThreads - 32 * sw;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int i0 = st0; st0 >= 0 && i0 < n; i0 += 8 * nst) {
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = (i0 + q * nst < n) ? __ldcg(x + i0 + q * nst) : 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (i0 + q * nst < n) {
        const uint32_t key = order_key(v[q]);
        if (staged) keys_s[i0 + q * nst] = key;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    wmin[warp] = kmin;
    wmax[warp] = kmax;
  }
  __syncthreads();
  kmin = __reduce_min_sync(0xffffffffu, wmin[lane]);
  kmax = __reduce_max_sync(0xffffffffu, wmax[lane]);
  auto key_at = [&](int i) -> uint32_t { return staged ? keys_s[i] : order_key(__ldcg(x + i)); };

  uint32_t* cand = keys_s + a.smem_keys;  // keys still able to be T (staged units, after the first digit)
  int n_cand = n;
  // every key shares the bits above the highest bit in which kmin and kmax differ
  int top = kmin == kmax ? -1 : 31 - __clz((int)(kmin ^ kmax));
  uint32_t mask = top >= 31 ? 0u : ~((2u << top) - 1u);
  if (top < 0) mask = 0xffffffffu;
  uint32_t prefix = kmin & mask;
  // the first digit's histogram needs the keys only
  if (top >= 0) {
    const int bits = min(11, top + 1), shift = top - bits + 1;
    const uint32_t dmask = (1u << bits) - 1u;
    for (int i = tid; i < (1 << bits); i += kSelThreads) hist[i] = 0;
    __syncthreads();  // also: the staged keys are in shared memory
    for (int i = tid; i < n; i += kSelThreads) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
    }
  }
  if (*(volatile int32_t*)w.error != 0) return;
  if (!ok_req) {
    if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  int k;
  if (a.budget) {
    // warp 0's keep counts: published by the barriers of the key staging above
    k = keep_s[l];
    if (hs == 0) {
      // this layer's keep count and statistics; unless the compaction forms
      // the row offsets, the last CTA to get here writes them from every keep count
      if (tid == 0) {
        w.keep[u] = k;
        w.stats[2 * u] = ff_to_double(st_s[l]);
        w.stats[2 * u + 1] = ff_to_double(sk_s[l]);
      }
      if (a.offsets) {
        if (tid == 0) {
          __threadfence();
          last_s = atomicAdd(w.cnt_all, 1u) == (unsigned)(p.L * p.B - 1) ? 1 : 0;
        }
        __syncthreads();
        if (last_s) {
          __threadfence();
          write_offsets<kSelThreads>(p, w.keep, w.out_offsets, w.error, a.out_capacity, off_seg, tid, 1);
        }
      }
    }
  } else {
    k = __ldcg(&w.keep[u]);
  }
  if (k < 0 || k > n) {
    if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  if (k == n) {
    for (int i = tid; i < n; i += kSelThreads) out[i] = i;
    return;
  }
  if (k == 0) return;
  unsigned want = (unsigned)k;  // keys >= T still to account for
  bool all_taken = false;       // every key of the selected bucket is taken: T = prefix, no ties to break
  if (tid == 0) sel_count = (unsigned)n;  // all keys equal: every one is == T
  for (int pass = 0; top >= 0; ++pass) {
    const int bits = min(11, top + 1);
    const int shift = top - bits + 1;
    top = shift - 1;
    const int nb = 1 << bits;
    const uint32_t dmask = (uint32_t)nb - 1u;
    if (pass > 0) {  // pass 0's histogram was counted above
      for (int i = tid; i < nb; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      const bool from_cand = staged;
      const int m = from_cand ? n_cand : n;
      for (int i = tid; i < m; i += kSelThreads) {
        const uint32_t key = from_cand ? cand[i] : key_at(i);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
      }
    }
    __syncthreads();
    // bins in descending digit order: thread t owns positions t*bpt .. t*bpt+bpt-1
    const int bpt = nb > kSelThreads ? nb / kSelThreads : 1;  // 2 or 1
    const unsigned c0 = tid * bpt < nb ? hist[nb - 1 - tid * bpt] : 0u;
    const unsigned c1 = bpt > 1 ? hist[nb - 2 - tid * bpt] : 0u;
    int total;
    const unsigned excl = (unsigned)block_excl_scan((int)(c0 + c1), wsum, &total);
    if (tid * bpt < nb && excl < want && want <= excl + c0) {
      sel_digit = (unsigned)(nb - 1 - tid * bpt);
      sel_above = excl;
      sel_count = c0;
    } else if (bpt > 1 && excl + c0 < want && want <= excl + c0 + c1) {
      sel_digit = (unsigned)(nb - 2 - tid * bpt);
      sel_above = excl + c0;
      sel_count = c1;
    }
    __syncthreads();
    want -= sel_above;
    prefix |= sel_digit << shift;
    mask |= dmask << shift;
    if (want == sel_count) {
      all_taken = true;  // keys >= prefix are exactly the keep largest
      break;
    }
    if (staged && pass == 0) {
      // compact the keys of the selected bucket (order is irrelevant here: one
      // shared counter, one atomic per warp and pass over the keys)
      if (tid == 0) n_cand_s = 0;
      __syncthreads();
      for (int i0 = 0; i0 < n; i0 += kSelThreads) {
        const int i = i0 + tid;
        const bool c = i < n && (keys_s[i] & mask) == prefix;
        const unsigned bal = __ballot_sync(0xffffffffu, c);
        int base = 0;
        if (lane == 0 && bal) base = (int)atomicAdd(&n_cand_s, (unsigned)__popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (c) cand[base + __popc(bal & ((1u << lane) - 1u))] = keys_s[i];
      }
      __syncthreads();
      n_cand = (int)n_cand_s;
    }
  }
  // prefix = T (exact unless all_taken, when every key >= prefix is taken).
  // Take every key > T and the first `want` keys == T in position order.
  // Warp w scans the positions [w*seg, (w+1)*seg) in steps of 32.
  const unsigned keep_eq = all_taken ? 0u : want;
  const uint32_t thr = prefix;
  const int seg = ((n + kSelWarps - 1) / kSelWarps + 31) / 32 * 32;
  const int s0 = warp * seg, s1 = min(n, s0 + seg);
  const unsigned lt = (1u << lane) - 1u;
  __syncthreads();  // sel_count of the last pass is read above by every thread
  int gt = 0, eq = 0;
  for (int i0 = s0; i0 < s1; i0 += kEmitStep * 32) {
    uint32_t kk[kEmitStep];
#pragma unroll
    for (int q = 0; q < kEmitStep; ++q) {
      const int i = i0 + 32 * q + lane;
      kk[q] = i < s1 ? key_at(i) : 0u;
    }
#pragma unroll
    for (int q = 0; q < kEmitStep; ++q) {
      const int i = i0 + 32 * q + lane;
      const bool g = i < s1 && (all_taken ? kk[q] >= thr : kk[q] > thr);
      const bool e = i < s1 && !all_taken && kk[q] == thr;
      gt += __popc(__ballot_sync(0xffffffffu, g));
      eq += __popc(__ballot_sync(0xffffffffu, e));
    }
  }
  if (lane == 0) {
    wgt[warp] = gt;
    weq[warp] = eq;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefixes of the warp totals
    int tg = wgt[lane], te = weq[lane];
    int ig = tg, ie = te;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yg = __shfl_up_sync(0xffffffffu, ig, o), ye = __shfl_up_sync(0xffffffffu, ie, o);
      if (lane >= o) {
        ig += yg;
        ie += ye;
      }
    }
    wgt[lane] = ig - tg;
    weq[lane] = ie - te;
  }
  __syncthreads();
  int gt_run = wgt[warp], eq_run = weq[warp];
  for (int i0 = s0; i0 < s1; i0 += kEmitStep * 32) {
    uint32_t kk[kEmitStep];
#pragma unroll
    for (int q = 0; q < kEmitStep; ++q) {
      const int i = i0 + 32 * q + lane;
      kk[q] = i < s1 ? key_at(i) : 0u;
    }
#pragma unroll
    for (int q = 0; q < kEmitStep; ++q) {
      const int i = i0 + 32 * q + lane;
      const bool g = i < s1 && (all_taken ? kk[q] >= thr : kk[q] > thr);
      const bool e = i < s1 && !all_taken && kk[q] == thr;
      const unsigned bg = __ballot_sync(0xffffffffu, g), be = __ballot_sync(0xffffffffu, e);
      const int eq_before = eq_run + __popc(be & lt);
      // output slot = keys taken before position i = (keys > T before i) + min(keys == T before i, keep_eq)
      const int pos = gt_run + __popc(bg & lt) + min(eq_before, (int)keep_eq);
      if (g || (e && eq_before < (int)keep_eq)) out[pos] = i;
      gt_run += __popc(bg);
      eq_run += __popc(be);
    }
  }
}

}  // namespace

cudaError_t launch_select(const Dev& p, const Ws& w, cudaStream_t s, bool budget, int64_t out_capacity) {
  SelectArgs a;
  a.p = p;
  a.w = w;
  a.budget = budget ? 1 : 0;
  a.out_capacity = out_capacity;
  a.offsets = budget && !compact_makes_offsets(p) ? 1 : 0;
  a.smem_keys = p.max_visual < kSmemKeys ? p.max_visual : kSmemKeys;
  const int smem = 2 * (int)sizeof(uint32_t) * a.smem_keys;  // keys + candidates
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(select_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_kernel, dim3(p.B, p.L, p.head_sets ? p.h_kv : 1), dim3(kSelThreads), smem, s, a);
}

}  // namespace aircache

AIRCACHE_TIMELINE_EXPORT(select)
