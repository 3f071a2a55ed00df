// Elite observation window (AirCache notes, "Key design 1": equations Att and k).
//
// One thread-block cluster per (request, layer), one CTA per group of KV heads
// (a single KV head when H_kv <= 8).  The last text query of every head is
// dotted with the N_t text keys of its KV head: the text keys stream through a
// ring of shared-memory stages (128 keys of one KV head per stage, cp.async),
// and the logit tile is the same MMA tile as the scoring kernel's (query rows =
// the g heads of that KV head).  Base-2 logits are kept in shared memory, each
// head's row is softmaxed in fp32 (max-subtracted), and the CTA sums its heads'
// rows into a partial P.  The partials are added across the cluster through
// distributed shared memory in CTA order, so every CTA holds the same P (the
// head mean up to the common factor 1/H_q, which the threshold test does not
// see).  The elite set is {j : P[j] >= alpha * max P}, in ascending order;
// each CTA then gathers the elite query rows and text keys of its own KV heads.
// When the logits of a CTA's heads do not fit in shared memory, its KV heads
// are processed in chunks and the partial P accumulates across chunks.
#include "internal.cuh"
#include "ptx.cuh"
#include "tile.cuh"
#include "timeline.cuh"

namespace aircache {
namespace {

constexpr int kEliteThreads = 256;
constexpr int kEliteWarps = kEliteThreads / 32;
constexpr int kSmemBudget = 220 * 1024;
constexpr int kSmemBudget2 = 110 * 1024;  // two CTAs per SM
constexpr int kMaxCluster = 8;  // portable cluster size
constexpr int kGatherBatch = 8; // 16-byte loads in flight per thread in the gathers

struct EliteArgs {
  Dev p;
  LayerPtrs lp;
  Ws w;
  int kv_chunk;    // KV heads whose logits are held at once
  int kv_per_cta;  // KV heads of one CTA of the cluster
};

// Issue the cp.async copies of item i of a KV-head chunk: items run over
// (kv head, query-row chunk, key tile).  Keys >= N_t and rows >= g are zero.
template <typename T, int D>
__device__ __forceinline__ void load_item(const Dev& p, const Req& R, const char* kbase, const char* qbase,
                                          int kv0, int n_rc, int n_kt, int i, unsigned char* stage) {
  using G = TileGeom<T, D>;
  const int per_kv = n_rc * n_kt;
  const int kvh = kv0 + i / per_kv, rc = (i % per_kv) / n_kt, t = i % n_kt;
  constexpr int kVec = G::kRowBytes / 16;
  for (int c = threadIdx.x; c < kTK * kVec; c += kEliteThreads) {
    const int row = c / kVec, v = c % kVec;
    const int key = t * kTK + row;
    const char* src = kbase;
    int bytes = 0;
    if (key < R.n_t) {
      src = kbase + (text_tok(R, key) * p.kv_stride_tok + (int64_t)kvh * p.kv_stride_head) * sizeof(T) + 16 * v;
      bytes = 16;
    }
    cp_async16(stage + row * G::kRowPitch + 16 * v, src, bytes);
  }
  for (int c = threadIdx.x; c < kRC * kVec; c += kEliteThreads) {
    const int n = c / kVec, v = c % kVec;
    const int hh = rc * kRC + n;
    const char* src = qbase;
    int bytes = 0;
    if (hh < p.g) {
      const int h = kvh * p.g + hh;
      src = qbase + (text_q_row(p, R, R.n_t - 1) * p.q_stride_tok + (int64_t)h * p.q_stride_head) * sizeof(T) +
            16 * v;
      bytes = 16;
    }
    cp_async16(stage + G::kKBytes + n * G::kRowPitch + 16 * v, src, bytes);
  }
}

template <typename T, int D, int NS>
__global__ void __launch_bounds__(kEliteThreads, 2) elite_kernel(const __grid_constant__ EliteArgs a) {
  AIRCACHE_KT(0);
  pdl_trigger();  // the next kernel may set up while this one runs
  using G = TileGeom<T, D>;
  constexpr int kVec = G::kRowBytes / 16;
  const Dev& p = a.p;
  // grid (C, B, L), cluster (C, 1, 1): blockIdx.x is the rank within the cluster
  const int rank = blockIdx.x, C = gridDim.x;
  const int b = blockIdx.y, l = blockIdx.z, u = l * p.B + b;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g4 = lane >> 2, c4 = lane & 3;

  if (p.wait_test) {
    // test hook: a bounded wait on a flag of the zeroed workspace block that no
    // kernel of this call sets (the wide path's LSE-ready flag of unit 0; this
    // call does no scoring), so it runs out and reports a timeout; the kernels
    // after this one see the error and return
    pdl_wait();  // the zeroed block
    if (rank == 0 && b == 0 && l == 0 && threadIdx.x == 0 && !wait_flag(a.w.lse_ready, 1LL << 20))
      set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
    return;
  }
  Req R;
  if (!load_req(p, b, R)) {  // the same verdict in every CTA of the cluster
    pdl_wait();
    if (rank == 0 && tid == 0) set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  const int n_t = R.n_t;
  const int hc = a.kv_chunk * p.g;  // heads per chunk
  const int kvb = min(p.h_kv, rank * a.kv_per_cta), kve = min(p.h_kv, kvb + a.kv_per_cta);

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stages = smem;
  float* lg = reinterpret_cast<float*>(smem + NS * G::kStageBytes);  // [hc][max_text]
  float* P = lg + (size_t)hc * p.max_text;                          // [max_text] this CTA's heads
  float* Pt = P + p.max_text;                                        // [max_text] every head
  float* hmax = Pt + p.max_text;                                     // [hc]
  float* hinv = hmax + hc;                                           // [hc]
  int32_t* pos_s = reinterpret_cast<int32_t*>(hinv + hc);            // [max_elite]
  __shared__ float red[kEliteWarps];
  __shared__ int wcount[kEliteWarps];

  const char* kbase = reinterpret_cast<const char*>(a.lp.k[l]);
  const char* qbase = reinterpret_cast<const char*>(a.lp.q[l]);
  const char* qvbase = reinterpret_cast<const char*>(a.lp.qv[l]);
  int base = 0;
  int32_t* out = a.w.elite + (size_t)u * p.elite_stride;
  if (p.window_mode == 4) {
    // the visual window: the last min(32, N_v) visual tokens (their queries
    // score; they add no keys: theirs are visual keys already)
    base = min(32, R.n_v);
    for (int e = tid; e < base; e += kEliteThreads) {
      pos_s[e] = R.n_v - base + e;
      if (rank == 0) out[e] = R.n_v - base + e;
    }
  } else if (p.window_mode != 0) {
    // an ablation window takes the elite set's place: the last 16 / 32 text
    // tokens or every one (the same in every CTA of the cluster)
    const int wsz = p.window_mode == 1 ? 16 : (p.window_mode == 2 ? 32 : n_t);
    base = min(wsz, n_t);
    for (int e = tid; e < base; e += kEliteThreads) {
      if (e < p.max_elite) {
        pos_s[e] = n_t - base + e;
        if (rank == 0) out[e] = n_t - base + e;
      }
    }
  } else {
    for (int j = tid; j < n_t; j += kEliteThreads) P[j] = 0.f;

    const int n_kt = (n_t + kTK - 1) / kTK;
    const int n_rc = (p.g + kRC - 1) / kRC;
    for (int kv0 = kvb; kv0 < kve; kv0 += a.kv_chunk) {
      const int kv1 = min(kve, kv0 + a.kv_chunk);
      const int items = (kv1 - kv0) * n_rc * n_kt;
      __syncthreads();
  #pragma unroll
      for (int i = 0; i < NS - 1; ++i) {
        if (i < items) load_item<T, D>(p, R, kbase, qbase, kv0, n_rc, n_kt, i, stages + i * G::kStageBytes);
        cp_async_commit();
      }
      for (int i = 0; i < items; ++i) {
        const int pre = i + NS - 1;
        if (pre < items) load_item<T, D>(p, R, kbase, qbase, kv0, n_rc, n_kt, pre, stages + (pre % NS) * G::kStageBytes);
        cp_async_commit();
        cp_async_wait<NS - 1>();
        __syncthreads();
        const int per_kv = n_rc * n_kt;
        const int kvh = kv0 + i / per_kv, rc = (i % per_kv) / n_kt, t = i % n_kt;
        const int rows = min(kRC, p.g - rc * kRC);
        const unsigned char* st = stages + (i % NS) * G::kStageBytes;
        float acc[4][4];
        TileLogits<T, D>::run(reinterpret_cast<const T*>(st), reinterpret_cast<const T*>(st + G::kKBytes), rows,
                              p.scale_log2, warp, lane, acc);
        const int kA = t * kTK + warp * 16 + g4;
  #pragma unroll
        for (int j = 0; j < 4; ++j)
  #pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int row = 8 * j + 2 * c4 + e;
            if (row < rows) {
              const int hrow = (kvh - kv0) * p.g + rc * kRC + row;  // head within the chunk
              float* lr = lg + (size_t)hrow * p.max_text;
              if (kA < n_t) lr[kA] = acc[j][e];
              if (kA + 8 < n_t) lr[kA + 8] = acc[j][2 + e];
            }
          }
        __syncthreads();
      }
      cp_async_wait<0>();
      // per-head softmax statistics
      const int hcur = (kv1 - kv0) * p.g;
      for (int hh = warp; hh < hcur; hh += kEliteWarps) {
        const float* row = lg + (size_t)hh * p.max_text;
        float m = -INFINITY;
        for (int j = lane; j < n_t; j += 32) m = fmaxf(m, row[j]);
  #pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float s = 0.f;
        for (int j = lane; j < n_t; j += 32) s += exp2f(row[j] - m);
  #pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) {
          hmax[hh] = m;
          hinv[hh] = 1.f / s;
        }
      }
      __syncthreads();
      for (int j = tid; j < n_t; j += kEliteThreads) {
        float accp = P[j];
        for (int hh = 0; hh < hcur; ++hh) accp += exp2f(lg[(size_t)hh * p.max_text + j] - hmax[hh]) * hinv[hh];
        P[j] = accp;
      }
    }
    // P over every head: the CTAs' partials added in rank order (the same sum,
    // bit for bit, in every CTA of the cluster)
    __syncthreads();
    cluster_sync_all();  // every CTA's partial P is complete
    for (int j = tid; j < n_t; j += kEliteThreads) {
      const uint32_t pj = smem_u32(P + j);
      float s = 0.f;
      for (int c = 0; c < C; ++c) s += ld_cluster_f32(cluster_map(pj, (uint32_t)c));
      Pt[j] = s;
    }
    cluster_sync_all();  // no CTA reads another's partial after this point

    // max P
    float m = -INFINITY;
    for (int j = tid; j < n_t; j += kEliteThreads) m = fmaxf(m, Pt[j]);
  #pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
  #pragma unroll
    for (int i = 1; i < kEliteWarps; ++i) m = fmaxf(m, red[i]);
    const float thr = (float)p.alpha * m;

    // ordered compaction of {j : P[j] >= thr}
    for (int j0 = 0; j0 < n_t; j0 += kEliteThreads) {
      const int j = j0 + tid;
      const bool take = j < n_t && Pt[j] >= thr;
      const unsigned bal = __ballot_sync(0xffffffffu, take);
      const int before = __popc(bal & ((1u << lane) - 1u));
      __syncthreads();
      if (lane == 0) wcount[warp] = __popc(bal);
      __syncthreads();
      int wbase = 0, total = 0;
  #pragma unroll
      for (int i = 0; i < kEliteWarps; ++i) {
        wbase += (i < warp) ? wcount[i] : 0;
        total += wcount[i];
      }
      const int pos = base + wbase + before;
      if (take && pos < p.max_elite) {
        pos_s[pos] = j;
        if (rank == 0) out[pos] = j;
      }
      base += total;
    }
  }
  // Gather this CTA's elite query rows (row kvh*g*N_tk + hh*N_tk + e) and elite
  // text keys into dense buffers: the scoring kernel then addresses them by
  // arithmetic alone.  Each row's source and destination are worked out once,
  // by one thread, into a table in the (now free) stage buffers; the copy loop
  // then moves 16-byte pieces with kGatherBatch loads in flight per thread.
  if (base <= p.max_elite) {
    __syncthreads();  // the elite positions are in shared memory; the stages are free
    const int n_tk = base;
    const int rows_g = p.g * n_tk;
    const bool vq = p.window_mode == 4;  // window 4: visual tokens' query rows; no keys added
    const int nq = (kve - kvb) * rows_g, nk = vq ? 0 : (kve - kvb) * n_tk;
    const int tab = NS * G::kStageBytes / (2 * (int)sizeof(void*));  // rows per table
    const uint4** srcp = reinterpret_cast<const uint4**>(stages);
    uint4** dstp = reinterpret_cast<uint4**>(stages) + tab;
    uint4* qdst = reinterpret_cast<uint4*>(a.w.qel) + ((size_t)u * p.rows_max + (size_t)kvb * rows_g) * kVec;
    uint4* kdst = reinterpret_cast<uint4*>(a.w.kel) + (size_t)u * p.h_kv * p.max_elite * kVec;
    for (int r0 = 0; r0 < nq + nk; r0 += tab) {
      const int n = min(tab, nq + nk - r0);
      for (int r = r0 + tid; r < r0 + n; r += kEliteThreads) {
        const char* src;
        uint4* dst;
        if (r < nq) {
          const int kvh = kvb + r / rows_g, rr = r % rows_g, hh = rr / n_tk, e = rr % n_tk;
          const int pos = min(max(pos_s[e], 0), (vq ? R.n_v : n_t) - 1);
          src = (vq ? qvbase : qbase) + ((vq ? R.vis0 + pos : text_q_row(p, R, pos)) * p.q_stride_tok +
                                         (int64_t)(kvh * p.g + hh) * p.q_stride_head) *
                                            sizeof(T);
          dst = qdst + (size_t)r * kVec;
        } else {
          const int j = r - nq, kvh = kvb + j / n_tk, e = j % n_tk;
          const int pos = min(max(pos_s[e], 0), n_t - 1);
          src = kbase + (text_tok(R, pos) * p.kv_stride_tok + (int64_t)kvh * p.kv_stride_head) * sizeof(T);
          dst = kdst + ((size_t)kvh * p.max_elite + e) * kVec;
        }
        srcp[r - r0] = reinterpret_cast<const uint4*>(src);
        dstp[r - r0] = dst;
      }
      __syncthreads();
      const int nel = n * kVec;
      for (int i0 = tid; i0 < nel; i0 += kGatherBatch * kEliteThreads) {
        uint4 v[kGatherBatch];
#pragma unroll
        for (int q = 0; q < kGatherBatch; ++q) {
          const int i = i0 + q * kEliteThreads;
          if (i < nel) v[q] = __ldg(srcp[i / kVec] + i % kVec);
        }
#pragma unroll
        for (int q = 0; q < kGatherBatch; ++q) {
          const int i = i0 + q * kEliteThreads;
          if (i < nel) dstp[i / kVec][i % kVec] = v[q];
        }
      }
      __syncthreads();  // the table is reused by the next chunk
    }
  }
  // the call's zeroed block (error word, routing counters) is cleared by the
  // kernel before this one: every thread waits for it here, so that this grid
  // completes after it
  pdl_wait();
  if (rank == 0 && tid == 0) {
    a.w.n_tk[u] = base;
    // the unit's layout, so that the scoring kernel resolves a work item with one
    // load; .x is the first VISUAL prompt position (the scoring kernels read
    // visual keys only: the elite text keys are gathered here)
    a.w.uinfo[2 * u] = make_int4((int)vis_tok(R, 0), (int)R.vis0, (int)R.txt0, R.n_v);
    a.w.uinfo[2 * u + 1] = make_int4(R.n_t, base, 1, 0);
    if (base > p.max_elite) {
      set_error(a.w.error, AIRCACHE_ERR_ELITE_OVERFLOW);
    } else {
      // route the unit to its scoring path
      if (p.stream_ok) {
        // units whose logits are recomputed in pass 2k (more than kLgRows query
        // rows per KV head: the heavier work) fill the list from the front, the
        // others from the back: the streaming pass claims the heavy ones first
        atomicAdd(&a.w.list_n[0], 1);
        int slot;
        if (p.g * base > kLgRows) {
          slot = atomicAdd(&a.w.list_n[2], 1);
        } else {
          // the pass-2 units also carry their weight (256-key blocks x 32-row
          // chunks per KV head) and the weight routed before them, for pass 2's
          // balanced partition: one 64-bit atomic assigns both
          const unsigned wgt = (unsigned)(((R.n_v + 255) / 256) * ((p.g * base + kRowChunk - 1) / kRowChunk));
          const unsigned long long old = atomicAdd(a.w.p2pack, (1ULL << 32) | wgt);
          slot = p.L * p.B - 1 - (int)(old >> 32);
          a.w.p2wpre[slot] = (uint32_t)old;
        }
        a.w.stream_list[slot] = u;
        a.w.stream_info[2 * slot] = make_int4((int)vis_tok(R, 0), (int)R.vis0, (int)R.txt0, R.n_v);
        a.w.stream_info[2 * slot + 1] = make_int4(R.n_t, base, 1, u);
      } else {
        a.w.wide_list[atomicAdd(&a.w.list_n[1], 1)] = u;
      }
    }
  }
}

template <typename T, int D, int NS>
cudaError_t launch_ns(const EliteArgs& a, int C, size_t smem, cudaStream_t s) {
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(elite_kernel<T, D, NS>), (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.p.B, a.p.L);
  cfg.blockDim = dim3(kEliteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, elite_kernel<T, D, NS>, a);
}

template <typename T, int D>
cudaError_t launch_t(const Dev& p, const LayerPtrs& lp, const Ws& w, cudaStream_t s) {
  using G = TileGeom<T, D>;
  EliteArgs a;
  a.p = p;
  a.lp = lp;
  a.w = w;
  // KV heads split over a cluster of at most kMaxCluster CTAs
  a.kv_per_cta = (p.h_kv + kMaxCluster - 1) / kMaxCluster;
  const int C = (p.h_kv + a.kv_per_cta - 1) / a.kv_per_cta;
  // NS stages, logits of kv_chunk KV heads, two P rows, per-head stats, elite positions
  auto bytes = [&](int ns, int kvc) {
    const size_t hc = (size_t)kvc * p.g;
    return (size_t)ns * G::kStageBytes + sizeof(float) * (hc * p.max_text + 2 * (size_t)p.max_text + 2 * hc) +
           sizeof(int32_t) * (size_t)p.max_elite;
  };
  int ns = 4;
  if (bytes(4, a.kv_per_cta) > (size_t)kSmemBudget) ns = 2;
  int kvc = a.kv_per_cta;
  while (kvc > 1 && bytes(ns, kvc) > (size_t)kSmemBudget) --kvc;
  // more CTAs than SMs: the CTAs are short and latency-bound, so two per SM
  // (two stages, fewer heads' logits at once) beat one with a deeper ring
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if ((long long)C * p.B * p.L > sms) {
    for (int ns2 = 2; ns2 >= 1; --ns2) {  // one stage: the two CTAs of an SM overlap each other's loads
      int kvc2 = a.kv_per_cta;
      while (kvc2 > 1 && bytes(ns2, kvc2) > (size_t)kSmemBudget2) --kvc2;
      if (bytes(ns2, kvc2) <= (size_t)kSmemBudget2) {
        ns = ns2;
        kvc = kvc2;
        break;
      }
    }
  }
  a.kv_chunk = kvc;
  const size_t smem = bytes(ns, kvc);
  if (ns == 4) return launch_ns<T, D, 4>(a, C, smem, s);
  return ns == 2 ? launch_ns<T, D, 2>(a, C, smem, s) : launch_ns<T, D, 1>(a, C, smem, s);
}

}  // namespace

cudaError_t launch_elite(const Dev& p, const LayerPtrs& lp, const Ws& w, cudaStream_t s) {
  if (p.dtype == AIRCACHE_BF16) {
    return p.d == 128 ? launch_t<__nv_bfloat16, 128>(p, lp, w, s) : launch_t<__nv_bfloat16, 64>(p, lp, w, s);
  }
  return p.d == 128 ? launch_t<float, 128>(p, lp, w, s) : launch_t<float, 64>(p, lp, w, s);
}

}  // namespace aircache

AIRCACHE_TIMELINE_EXPORT(elite)
