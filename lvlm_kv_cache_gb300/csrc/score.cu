// Cross-modal scoring (AirCache notes, "Key design 1": equations A_vtk and I_v),
// then the per-layer strength / skewness and the per-request budget ("Key
// design 2"), in one persistent kernel.
//
// Problem.  For one (layer l, request b) -- a "unit" -- the query rows are all
// pairs (query head h, elite text position e): H_q * N_tk rows, grouped by KV
// head (g = H_q/H_kv heads x N_tk rows read the same keys).  Each row is a
// softmax over the N_v visual keys and the N_tk elite text keys; I_v[i] is the
// mean over all rows of the probability of visual key i.  A row's
// probabilities need its log-sum-exp over every key, so each key tile is
// visited twice:
//   pass 1: logits -> per (tile, row) max and sum of exp2 -> partials; the CTA
//           that completes a unit's last pass-1 item merges the partials of
//           every row (fixed order) into the row's log-sum-exp and publishes
//           it with a release flag;
//   pass 2: logits again -> per visual key, sum over rows of exp2(logit - lse),
//           scaled by 1/(H_q N_tk) -> I_v.  The CTA completing a unit's last
//           pass-2 item computes the unit's (s_t, s_k); the one completing a
//           request's last unit computes its keep counts; the last request
//           writes the compacted-cache row offsets.
// Key tiles are 128 keys of one KV head: the visual tiles of the unit, then
// the elite text keys (gathered densely by the elite-window kernel) in tiles
// of their own.
//
// Schedule.  A persistent grid (one CTA per SM).  A work item is (unit, tile,
// group of up to 4 KV heads) of one pass.  Pass-1 items are claimed from one
// atomic counter in unit order; pass-2 items of a unit are claimed from a
// per-unit counter, but only once that unit's LSEs are published, and each
// CTA prefers them to pass-1 work.  So pass 2 of a unit follows its pass 1
// closely (the re-read of its keys hits L2), no CTA idles while pass-1 work
// remains, and a CTA waits for a flag only when every pass-1 item has been
// claimed -- by running CTAs that finish them without waiting -- so the grid
// always makes progress (every wait is bounded anyway).
//
// CTA (12 warps).  A scheduler warp claims items and queues them in shared
// memory; an issuer warp turns queued items into ring stages; eight consumer
// warps compute; two service warps finish units (LSE merge; I_v moments,
// budgets, offsets) from a shared-memory mailbox, off the consumers' path.  A
// stage is a K tile (128 keys x D) and a Q chunk (32 query rows x D), as
// 128-byte column slabs in the 128-byte-swizzled layout, plus 32 row LSEs.
// With a tensor map over the keys (per-layer K pointers evenly strided, as in a
// stacked cache) the issuer moves a stage with a handful of TMA tensor copies;
// otherwise its 32 lanes copy it with 16-byte cp.async into the same layout.
// Consumers compute the 32 x 128 logit tile with mma.sync (bf16 x bf16 -> fp32,
// exact products; query rows are the M dimension, each warp owns 16 keys of the
// N dimension) or with fp32 FMAs for fp32 inputs, release the stage, and run
// the pass's epilogue from registers.  Logits are base 2 (log2(e)/sqrt(D)).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "internal.cuh"
#include "ptx.cuh"
#include "reduce.cuh"
#include "tmap.cuh"

namespace aircache {
namespace {

constexpr int kTK = 128;            // keys per tile
constexpr int kRC = 32;             // query rows per chunk
constexpr int kCW = 8;              // consumer warps (16 keys each)
constexpr int kCT = kCW * 32;       // consumer threads
constexpr int kIssuerWarp = kCW;    // warp 8
constexpr int kSchedWarp = kCW + 1; // warp 9
constexpr int kSvcWarp0 = kCW + 2;  // warps 10, 11
constexpr int kSvcT = 64;           // service threads
constexpr int kThreads = (kCW + 4) * 32;
constexpr int kBar = 1;             // named barrier of the consumer threads
constexpr int kBarSvc = 3;          // named barrier of the service threads
constexpr int kHG = 4;              // KV heads per work item
constexpr int kQN = 4;              // scheduler -> issuer queue depth
constexpr int kMN = 64;             // consumer -> service mailbox depth

enum : int { kEnd = 0, kP1 = 1, kP2 = 2 };
enum : int { kSvcEnd = 0, kSvcDone1 = 1, kSvcDone2 = 2 };  // end; a pass-1 / pass-2 item finished

// Stage geometry: rows of D elements split into 128-byte slabs; slab j of all
// rows of a tile is contiguous, 16-byte chunks XOR-swizzled by (row & 7).
template <typename T, int D>
struct Geo {
  static constexpr int kEs = (int)sizeof(T);
  static constexpr int kRowBytes = D * kEs;
  static constexpr int kNH = kRowBytes / 128;  // slabs per row
  static constexpr int kSlabElems = 128 / kEs;
  static constexpr int kKSlab = kTK * 128;
  static constexpr int kQSlab = kRC * 128;
  static constexpr int kKBytes = kNH * kKSlab;
  static constexpr int kQBytes = kNH * kQSlab;
  static constexpr int kLseOff = kKBytes + kQBytes;
  static constexpr int kRing = (kLseOff + kRC * 4 + 1023) / 1024 * 1024;
  static constexpr int kStages = (4 * kRing <= 200 * 1024) ? 4 : (3 * kRing <= 200 * 1024 ? 3 : 2);
};

struct StageHdr {
  int kind, u, b, l, tile, kvh, grp, r0, rows, rows_g, n_v, n_tk, klim, key0, first, last;
  long long vis0;
};

// A work item, scheduler -> issuer.
struct Item {
  int kind, u, b, l, tile, grp, klim, text, n_v, n_t, n_tk, pad;
  long long seq0, vis0;
};

// A unit to finish, consumers -> service.
struct SvcJob {
  int kind, u, b, l, n_v, n_tk;
  long long vis0;
};

// Shared-memory control block (after the stages).
struct Ctl {
  StageHdr hdr[4];
  uint64_t full[4], empty[4];
  Item iq[kQN];
  int iq_state[kQN];  // 0 free, 1 full
  SvcJob mb[kMN];
  int mb_seq[kMN];    // the mailbox ticket a free slot expects
  int mb_ready[kMN];  // ticket + 1 once filled
  int mb_tail;
  int p2done[8];      // pass-2 items: consumer warps finished, by item sequence
  int svc_flag[4];
  SvcJob svc_job;
  float2 red[2 * kCW * kRC];
  ff svc_red[2 * (kSvcT / 32) + 1];
  long long svc_seg[kSvcT];
};

struct PArgs {
  CUtensorMap kmap;    // K of every layer: (D, H_kv, tokens, layers)
  CUtensorMap qmap;    // gathered elite query rows: (D, rows)
  CUtensorMap kelmap;  // gathered elite text keys: (D, rows)
  Dev p;
  LayerPtrs lp;
  Ws w;
  int TV, TT;      // visual / text tile slots per unit (pass 1 has TV + TT, pass 2 has TV)
  int G;           // KV-head groups per tile
  int tail;        // 1: stats, budgets and offsets after pass 2
  int tma;         // 1: stages move by TMA tensor copies
  int pad;
  long long n_p1;  // pass-1 tickets: units x (TV + TT) x G
  int64_t out_capacity;
};

constexpr int kCtlBytes = ((int)sizeof(Ctl) + 127) / 128 * 128;

// volatile shared-memory flag helpers (with CTA-scope fences around them)
__device__ __forceinline__ int ld_vol(const int* p) { return *(const volatile int*)p; }
__device__ __forceinline__ void st_vol(int* p, int v) { *(volatile int*)p = v; }

// Wait until *p == v; false after `limit` cycles.
__device__ __forceinline__ bool wait_eq(const int* p, int v, long long limit) {
  if (ld_vol(p) == v) return true;
  const long long t0 = clock64();
  while (ld_vol(p) != v) {
    if (clock64() - t0 > limit) return false;
    __nanosleep(32);
  }
  return true;
}

// ------------------------------------------------------------------ logits

// acc[mt][nt][0..1]: query row 16mt + lane/4, keys 16*warp + 8nt + 2(lane%4) + {0,1};
// acc[mt][nt][2..3]: query row 16mt + lane/4 + 8, same keys.  Values are
// log2(e)/sqrt(D) * q . k; rows >= `rows` hold unspecified values.
template <typename T, int D>
struct Logits;

template <int D>
struct Logits<__nv_bfloat16, D> {
  using Gm = Geo<__nv_bfloat16, D>;
  static __device__ __forceinline__ void run(uint32_t ks, uint32_t qs, int rows, float scale, int warp, int lane,
                                             float acc[2][2][4]) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
    const int kr = 16 * warp + (lane & 7) + 8 * (lane >> 4);
    const int kc = (lane >> 3) & 1;
    const int qr = lane & 15;
    const int qc = lane >> 4;
    if (rows > 16) {
      __syncwarp();  // ldmatrix / mma are warp-collective: the whole warp, converged
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int slab = kk >> 2, c0 = (kk & 3) * 2;
        uint32_t b[4], a0[4], a1[4];
        ldsm_x4(b, swz(ks + slab * Gm::kKSlab, kr, c0 + kc));
        ldsm_x4(a0, swz(qs + slab * Gm::kQSlab, qr, c0 + qc));
        ldsm_x4(a1, swz(qs + slab * Gm::kQSlab, 16 + qr, c0 + qc));
        mma_bf16_16816(acc[0][0], a0, b[0], b[1]);
        mma_bf16_16816(acc[0][1], a0, b[2], b[3]);
        mma_bf16_16816(acc[1][0], a1, b[0], b[1]);
        mma_bf16_16816(acc[1][1], a1, b[2], b[3]);
      }
    } else {
      __syncwarp();  // ldmatrix / mma are warp-collective: the whole warp, converged
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int slab = kk >> 2, c0 = (kk & 3) * 2;
        uint32_t b[4], a0[4];
        ldsm_x4(b, swz(ks + slab * Gm::kKSlab, kr, c0 + kc));
        ldsm_x4(a0, swz(qs + slab * Gm::kQSlab, qr, c0 + qc));
        mma_bf16_16816(acc[0][0], a0, b[0], b[1]);
        mma_bf16_16816(acc[0][1], a0, b[2], b[3]);
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][nt][i] *= scale;
  }
};

template <int D>
struct Logits<float, D> {
  using Gm = Geo<float, D>;
  // element i of a row in the swizzled slab layout
  static __device__ __forceinline__ float at(const unsigned char* tile, int slab_bytes, int row, int i) {
    const int slab = i / Gm::kSlabElems, w = i % Gm::kSlabElems;
    const int off = slab * slab_bytes + row * 128 + ((((w >> 2) ^ (row & 7)) << 4)) + (w & 3) * 4;
    return *reinterpret_cast<const float*>(tile + off);
  }
  static __device__ __forceinline__ void run(const unsigned char* ks, const unsigned char* qs, int rows, float scale,
                                             int warp, int lane, float acc[2][2][4]) {
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = 16 * mt + g + 8 * (i >> 1);
          const int key = 16 * warp + 8 * nt + 2 * c + (i & 1);
          float s = 0.f;
          if (row < rows) {
            for (int d = 0; d < D; ++d) s = fmaf(at(qs, Gm::kQSlab, row, d), at(ks, Gm::kKSlab, key, d), s);
          }
          acc[mt][nt][i] = s * scale;
        }
  }
};

// ------------------------------------------------------------------ scheduler

// Unit of position k of the wide-path list.
__device__ __forceinline__ int unit_of(const Ws& w, int k) { return __ldcg(&w.wide_list[k]); }

__device__ __forceinline__ bool unit_valid(const Dev& p, const int4& i0, const int4& i1) {
  const long long seq0 = i0.x, vis0 = i0.y, txt0 = i0.z;
  const int n_v = i0.w, n_t = i1.x, n_tk = i1.y;
  return i1.z == 1 && n_tk >= 1 && n_tk <= p.max_elite && n_tk <= n_t && n_v >= 3 && n_v <= p.max_visual &&
         seq0 >= 0 && seq0 + n_v <= p.total_tokens && txt0 >= 0 && txt0 + n_t <= p.total_text &&
         vis0 >= 0 && vis0 + n_v <= p.total_visual;
}

// Pass-1 item from ticket t1 (false: an empty slot of a shorter unit).
__device__ __forceinline__ bool p1_item(const PArgs& a, long long t1, Item& it, bool& bad) {
  const Dev& p = a.p;
  const long long S1 = (long long)(a.TV + a.TT) * a.G;
  const int k = (int)(t1 / S1), slot = (int)(t1 % S1);
  const int u = unit_of(a.w, k);
  if (u < 0 || u >= p.L * p.B) {
    bad = true;
    return false;
  }
  const int4 i0 = __ldcg(&a.w.uinfo[2 * u]);
  const int4 i1 = __ldcg(&a.w.uinfo[2 * u + 1]);
  if (!unit_valid(p, i0, i1)) {
    bad = true;
    return false;
  }
  const int tile = slot / a.G;
  const int n_v = i0.w, n_tk = i1.y;
  const bool text = tile >= a.TV;
  const int klim = text ? min(kTK, n_tk - (tile - a.TV) * kTK) : min(kTK, n_v - tile * kTK);
  if (klim <= 0) return false;
  it.kind = kP1;
  it.u = u;
  it.b = u % p.B;
  it.l = u / p.B;
  it.tile = tile;
  it.grp = slot % a.G;
  it.text = text ? 1 : 0;
  it.n_v = n_v;
  it.n_t = i1.x;
  it.n_tk = n_tk;
  it.klim = klim;
  it.seq0 = i0.x;
  it.vis0 = i0.y;
  return true;
}

// One thread (lane 0 of the scheduler warp).  Each round it looks at the first
// unit (in order) that may still have pass-2 items; if that unit's LSEs are
// published it claims one of them, and otherwise (or as well) it claims the
// next pair of pass-1 tickets.  The flag check and the pass-1 claim are issued
// together so that their latencies overlap.
__device__ void scheduler(const PArgs& a, Ctl* c) {
  const Dev& p = a.p;
  const int U = __ldcg(&a.w.list_n[1]);  // units on this path
  const long long n_p1 = (long long)U * (a.TV + a.TT) * a.G;
  bool p1_done = false, stop = false;
  int scan_k = 0, scan_u = 0, scan_items = -1;
  int4 s0 = make_int4(0, 0, 0, 0), s1 = make_int4(0, 0, 0, 0);
  int qi = 0;
  long long wait0 = 0;
  bool waiting = false;
  auto push = [&](const Item& it) -> bool {
    const int slot = qi % kQN;
    if (!wait_eq(&c->iq_state[slot], 0, 2 * kWaitCycles)) {
      set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      return false;  // the issuer has stopped
    }
    c->iq[slot] = it;
    __threadfence_block();
    st_vol(&c->iq_state[slot], 1);
    ++qi;
    return true;
  };
  while (!stop) {
    if (*(volatile int32_t*)a.w.error != 0) break;
    if (scan_k < U && scan_items < 0) {
      scan_u = unit_of(a.w, scan_k);
      if (scan_u < 0 || scan_u >= p.L * p.B) {
        set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
        break;
      }
      s0 = __ldcg(&a.w.uinfo[2 * scan_u]);
      s1 = __ldcg(&a.w.uinfo[2 * scan_u + 1]);
      if (!unit_valid(p, s0, s1)) {
        set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
        break;
      }
      scan_items = ((s0.w + kTK - 1) / kTK) * a.G;
    }
    // issue both requests before using either
    const uint32_t ready = (scan_k < U) ? ld_relaxed(&a.w.lse_ready[scan_u]) : 0u;
    const long long t1 = p1_done ? -1 : (long long)atomicAdd(a.w.ticket, 2ULL);
    bool progressed = false;
    if (ready) {
      fence_acquire_gpu();
      const int ci = (int)atomicAdd(&a.w.p2claim[scan_u], 1u);
      if (ci < scan_items) {
        Item it{};
        it.kind = kP2;
        it.u = scan_u;
        it.b = scan_u % p.B;
        it.l = scan_u / p.B;
        it.tile = ci / a.G;
        it.grp = ci % a.G;
        it.text = 0;
        it.n_v = s0.w;
        it.n_t = s1.x;
        it.n_tk = s1.y;
        it.klim = min(kTK, it.n_v - it.tile * kTK);
        it.seq0 = s0.x;
        it.vis0 = s0.y;
        if (!push(it)) return;
      } else {
        ++scan_k;  // this unit's pass-2 items are all taken
        scan_items = -1;
      }
      progressed = true;
    }
    if (!p1_done) {
      for (int q = 0; q < 2; ++q) {
        if (t1 + q >= n_p1) {
          p1_done = true;
          break;
        }
        Item it{};
        bool bad = false;
        if (p1_item(a, t1 + q, it, bad)) {
          if (!push(it)) return;
        } else if (bad) {
          set_error(a.w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
          stop = true;
          break;
        }
      }
      progressed = true;
    }
    if (scan_k >= U) break;  // all work claimed
    if (!progressed) {
      // only pass-2 work of units still being finished remains
      if (!waiting) {
        waiting = true;
        wait0 = clock64();
      } else if (clock64() - wait0 > kWaitCycles) {
        set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
        break;
      }
      __nanosleep(128);
    } else {
      waiting = false;
    }
  }
  Item end{};
  end.kind = kEnd;
  push(end);
}

// ------------------------------------------------------------------ issuer

template <typename T, int D>
__device__ void issuer(const PArgs& a, Ctl* c, unsigned char* stages) {
  using Gm = Geo<T, D>;
  constexpr int NS = Gm::kStages;
  const Dev& p = a.p;
  const int lane = threadIdx.x & 31;
  const size_t row_bytes = Gm::kRowBytes;
  long long st = 0;  // stage counter
  for (int qi = 0;; ++qi) {
    const int slot = qi % kQN;
    int okq = 1;
    if (lane == 0) okq = wait_eq(&c->iq_state[slot], 1, 4 * kWaitCycles) ? 1 : 0;
    okq = __shfl_sync(0xffffffffu, okq, 0);
    __threadfence_block();
    Item it = c->iq[slot];
    __syncwarp();
    if (lane == 0 && okq) st_vol(&c->iq_state[slot], 0);
    if (!okq) {
      if (lane == 0) set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      it.kind = kEnd;
    }
    if (it.kind == kP2 && lane == 0) fence_proxy_async_global();  // LSEs written by another CTA, read by copies
    const int rows_g = p.g * it.n_tk;
    const int n_rc = (rows_g + kRC - 1) / kRC;
    const int kv0 = it.grp * kHG, kv1 = min(p.h_kv, kv0 + kHG);
    const int n_st = (it.kind == kEnd) ? 1 : (kv1 - kv0) * n_rc;
    for (int si = 0; si < n_st; ++si, ++st) {
      const int s = (int)(st % NS);
      int oke = 1;
      if (lane == 0) oke = mbar_wait(&c->empty[s], (uint32_t)(((st / NS) & 1) ^ 1)) ? 1 : 0;
      oke = __shfl_sync(0xffffffffu, oke, 0);
      if (!oke) {
        if (lane == 0) set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
        cp_async_wait<0>();
        return;  // consumers give up on their own (longer) wait
      }
      if (it.kind == kEnd) {
        if (lane == 0) c->hdr[s].kind = kEnd;
        __syncwarp();
        if (a.tma) {
          if (lane == 0) mbar_arrive(&c->full[s]);
        } else {
          mbar_arrive(&c->full[s]);
          if (lane == 0) mbar_arrive(&c->full[s]);
        }
        cp_async_wait<0>();
        return;
      }
      const int kvh = kv0 + si / n_rc, rc = si % n_rc;
      const int r0 = rc * kRC;
      const int qvalid = min(kRC, rows_g - r0);
      const long long qrow_idx = (long long)it.u * p.rows_max + kvh * rows_g + r0;
      const float* lse = a.w.lse + (size_t)it.u * p.lse_stride + (kvh * p.rc_max + rc) * kRC;
      unsigned char* base = stages + (size_t)s * Gm::kRing;
      if (lane == 0) {
        StageHdr& h = c->hdr[s];
        h.kind = it.kind;
        h.u = it.u;
        h.b = it.b;
        h.l = it.l;
        h.tile = it.tile;
        h.kvh = kvh;
        h.grp = it.grp;
        h.r0 = r0;
        h.rows = qvalid;
        h.rows_g = rows_g;
        h.n_v = it.n_v;
        h.n_tk = it.n_tk;
        h.klim = it.klim;
        h.key0 = it.text ? -1 : it.tile * kTK;
        h.first = (si == 0);
        h.last = (si == n_st - 1);
        h.vis0 = it.vis0;
      }
      const long long krow_idx = ((long long)it.u * p.h_kv + kvh) * p.max_elite + (long long)(it.tile - a.TV) * kTK;
      if (a.tma) {
        if (lane == 0) {
          const uint32_t kb = smem_u32(base), qb = kb + Gm::kKBytes;
          fence_proxy_async_smem();  // the stage was last read by generic loads
          mbar_arrive_expect_tx(&c->full[s], (uint32_t)(Gm::kKBytes + Gm::kQBytes + (it.kind == kP2 ? kRC * 4 : 0)));
#pragma unroll
          for (int sl = 0; sl < Gm::kNH; ++sl) {
            if (it.text) {
              tma_load_2d(kb + sl * Gm::kKSlab, &a.kelmap, sl * Gm::kSlabElems, (int)krow_idx, &c->full[s]);
            } else {
              tma_load_4d(kb + sl * Gm::kKSlab, &a.kmap, sl * Gm::kSlabElems, kvh, (int)(it.seq0 + it.tile * kTK),
                          it.l, &c->full[s]);
            }
            tma_load_2d(qb + sl * Gm::kQSlab, &a.qmap, sl * Gm::kSlabElems, (int)qrow_idx, &c->full[s]);
          }
          if (it.kind == kP2) bulk_g2s(base + Gm::kLseOff, lse, kRC * 4, &c->full[s]);
        }
      } else {
        const char* krow;
        long long kstride;
        if (it.text) {
          krow = reinterpret_cast<const char*>(a.w.kel) + krow_idx * row_bytes;
          kstride = (long long)row_bytes;
        } else {
          krow = reinterpret_cast<const char*>(a.lp.k[it.l]) +
                 ((it.seq0 + (long long)it.tile * kTK) * p.kv_stride_tok + (long long)kvh * p.kv_stride_head) *
                     Gm::kEs;
          kstride = p.kv_stride_tok * Gm::kEs;
        }
        const char* qrow = reinterpret_cast<const char*>(a.w.qel) + qrow_idx * row_bytes;
        const uint32_t kb = smem_u32(base), qb = kb + Gm::kKBytes;
        constexpr int kCh = Gm::kRowBytes / 16;  // 16-byte chunks per row
        for (int i = lane; i < kTK * kCh; i += 32) {
          const int row = i / kCh, ch = i % kCh;
          const bool live = row < it.klim;
          const char* src = live ? krow + row * kstride + 16 * ch : krow;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(
                           swz(kb + (ch >> 3) * Gm::kKSlab, row, ch & 7)),
                       "l"(src), "r"(live ? 16 : 0)
                       : "memory");
        }
        for (int i = lane; i < kRC * kCh; i += 32) {
          const int row = i / kCh, ch = i % kCh;
          const bool live = row < qvalid;
          const char* src = live ? qrow + row * row_bytes + 16 * ch : qrow;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(
                           swz(qb + (ch >> 3) * Gm::kQSlab, row, ch & 7)),
                       "l"(src), "r"(live ? 16 : 0)
                       : "memory");
        }
        if (it.kind == kP2 && lane < kRC * 4 / 16) {
          cp_async16(base + Gm::kLseOff + 16 * lane, reinterpret_cast<const char*>(lse) + 16 * lane, 16);
        }
        __syncwarp();
        cp_async_mbar_arrive(&c->full[s]);
        if (lane == 0) mbar_arrive(&c->full[s]);  // releases the stage header
      }
    }
  }
}

// ------------------------------------------------------------------ mailbox

// Post a job to the service warps (one thread).
__device__ __forceinline__ void post_job(const PArgs& a, Ctl* c, const SvcJob& job) {
  const int m = atomicAdd(&c->mb_tail, 1);
  const int slot = m % kMN;
  if (!wait_eq(&c->mb_seq[slot], m, kWaitCycles)) {
    set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
    return;
  }
  c->mb[slot] = job;
  __threadfence_block();
  st_vol(&c->mb_ready[slot], m + 1);
}

// ------------------------------------------------------------------ service

// The two service warps: finish units posted by the consumers.
__device__ void service(const PArgs& a, Ctl* c) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int tix = threadIdx.x - kSvcWarp0 * 32;
  for (int m = 0;; ++m) {
    const int slot = m % kMN;
    if (tix == 0) {
      if (wait_eq(&c->mb_ready[slot], m + 1, 8 * kWaitCycles)) {
        __threadfence_block();
        c->svc_job = c->mb[slot];
        st_vol(&c->mb_seq[slot], m + kMN);
      } else {
        set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
        c->svc_job.kind = kSvcEnd;
      }
    }
    named_bar_sync(kBarSvc, kSvcT);
    const SvcJob job = c->svc_job;
    named_bar_sync(kBarSvc, kSvcT);
    if (job.kind == kSvcEnd) return;
    // count the item; only the unit's last item goes on
    if (tix == 0) {
      __threadfence();
      const int ntv = (job.n_v + kTK - 1) / kTK;
      const int ntt = (job.n_tk + kTK - 1) / kTK;
      const unsigned items = (unsigned)((job.kind == kSvcDone1 ? ntv + ntt : ntv) * a.G);
      uint32_t* cnt = (job.kind == kSvcDone1) ? w.cnt_p1 : w.cnt_p2;
      c->svc_flag[2] = (atomicAdd(&cnt[job.u], 1u) == items - 1u) ? 1 : 0;
    }
    named_bar_sync(kBarSvc, kSvcT);
    const bool last = c->svc_flag[2] != 0;
    named_bar_sync(kBarSvc, kSvcT);
    if (!last) continue;
    __threadfence();
    if (job.kind == kSvcDone1) {
      // row r of the unit: one thread merges the row's tile partials (stored
      // contiguously) in tile order -> LSE (deterministic)
      const int rows_g = p.g * job.n_tk;
      const int rows_total = p.h_q * job.n_tk;
      const int TS = a.TV + a.TT;
      const int ntv = (job.n_v + kTK - 1) / kTK;
      const int ntiles = ntv + (job.n_tk + kTK - 1) / kTK;
      float* lse_u = w.lse + (size_t)job.u * p.lse_stride;
      for (int r = tix; r < rows_total; r += kSvcT) {
        const float2* pr = w.part + ((size_t)job.u * p.rows_max + r) * TS;
        float mx = -INFINITY, sm = 0.f;
        for (int t0 = 0; t0 < ntiles; t0 += 8) {
          float2 v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int t = t0 + q;
            const int ts = t < ntv ? t : a.TV + (t - ntv);
            v[q] = (t < ntiles) ? __ldcg(pr + ts) : make_float2(-INFINITY, 0.f);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (v[q].y > 0.f) {
              if (v[q].x > mx) {
                sm = sm * exp2f(mx - v[q].x) + v[q].y;
                mx = v[q].x;
              } else {
                sm += v[q].y * exp2f(v[q].x - mx);
              }
            }
          }
        }
        const int kvh = r / rows_g, rr = r % rows_g;
        lse_u[(kvh * p.rc_max + rr / kRC) * kRC + rr % kRC] = mx + log2f(sm);
      }
      __threadfence();
      named_bar_sync(kBarSvc, kSvcT);
      if (tix == 0) st_release(&w.lse_ready[job.u], 1u);
      continue;
    }
    // a unit's I_v is complete
    float* iv = w.iv + (size_t)job.l * p.total_visual + job.vis0;
    if (a.G > 1) {
      const float inv = 1.f / (float)(p.h_q * job.n_tk);
      for (int i = tix; i < job.n_v; i += kSvcT) {
        float s2 = 0.f;
        for (int gg = 0; gg < a.G; ++gg) s2 += __ldcg(&w.ivp[((size_t)gg * p.L + job.l) * p.total_visual + job.vis0 + i]);
        iv[i] = s2 * inv;
      }
      __threadfence();
      named_bar_sync(kBarSvc, kSvcT);
    }
    if (!a.tail) continue;
    const double2 mo = unit_moments<kSvcT>(iv, job.n_v, tix, c->svc_red, kBarSvc);
    if (tix == 0) {
      w.stats[2 * job.u] = mo.x;
      w.stats[2 * job.u + 1] = mo.y;
      __threadfence();
      c->svc_flag[0] = (atomicAdd(&w.cnt_req[job.b], 1u) == (unsigned)(p.L - 1)) ? 1 : 0;
    }
    named_bar_sync(kBarSvc, kSvcT);
    if (!c->svc_flag[0]) continue;
    __threadfence();
    if (tix < 32) request_budget(p, job.b, job.n_v, w.stats, w.keep, tix);
    __threadfence();
    named_bar_sync(kBarSvc, kSvcT);
    if (tix == 0) c->svc_flag[1] = (atomicAdd(w.cnt_all, 1u) == (unsigned)(p.B - 1)) ? 1 : 0;
    named_bar_sync(kBarSvc, kSvcT);
    if (!c->svc_flag[1]) continue;
    __threadfence();
    write_offsets<kSvcT>(p, w.keep, w.out_offsets, w.error, a.out_capacity, c->svc_seg, tix, kBarSvc);
  }
}

// ------------------------------------------------------------------ consumers

template <typename T, int D>
__device__ void consumers(const PArgs& a, Ctl* c, unsigned char* stages) {
  using Gm = Geo<T, D>;
  constexpr int NS = Gm::kStages;
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, c4 = lane & 3;
  long long it = 0, p1_it = 0, p2_items = 0;
  float accK[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // pass-2 sums of this thread's 4 keys over the item
  while (true) {
    const int s = (int)(it % NS);
    const uint32_t ph = (uint32_t)((it / NS) & 1);
    // Longer than the issuer's and scheduler's waits combined: a stage can be
    // late only by those bounded waits, so every consumer warp reaches the same
    // verdict here and none is left alone at a named barrier.
    if (!mbar_wait(&c->full[s], ph, 8 * kWaitCycles)) {
      if (lane == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      break;
    }
    const StageHdr h = c->hdr[s];
    if (h.kind == kEnd) break;
    unsigned char* base = stages + (size_t)s * Gm::kRing;
    const int mts = h.rows > 16 ? 2 : 1;

    float lse[2][2];
    if (h.kind == kP2) {
      const float* ls = reinterpret_cast<const float*>(base + Gm::kLseOff);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) lse[mt][hh] = ls[16 * mt + g4 + 8 * hh];
    }

    float acc[2][2][4];
    if constexpr (sizeof(T) == 2) {
      Logits<T, D>::run(smem_u32(base), smem_u32(base + Gm::kKBytes), h.rows, p.scale_log2, warp, lane, acc);
    } else {
      Logits<T, D>::run(base, base + Gm::kKBytes, h.rows, p.scale_log2, warp, lane, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c->empty[s]);  // stage fully read: the issuer may refill it

    if (h.kind == kP1) {
      float2* rb = c->red + (p1_it & 1) * kCW * kRC;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        if (mt < mts) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float v[4];
            float m = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int key = 16 * warp + 8 * nt + 2 * c4 + e;
                v[2 * nt + e] = key < h.klim ? acc[mt][nt][2 * hh + e] : -INFINITY;
                m = fmaxf(m, v[2 * nt + e]);
              }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            float sum = 0.f;
            if (m != -INFINITY) {
#pragma unroll
              for (int q = 0; q < 4; ++q) sum += exp2f(v[q] - m);
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (c4 == 0) rb[warp * kRC + 16 * mt + g4 + 8 * hh] = make_float2(m, sum);
          }
        }
      }
      named_bar_sync(kBar, kCT);
      if (warp == 0) {
        if (lane < h.rows) {
          float M = -INFINITY;
#pragma unroll
          for (int ww = 0; ww < kCW; ++ww) M = fmaxf(M, rb[ww * kRC + lane].x);
          float S = 0.f;
#pragma unroll
          for (int ww = 0; ww < kCW; ++ww) {
            const float2 v = rb[ww * kRC + lane];
            if (v.y > 0.f) S += v.y * exp2f(v.x - M);
          }
          w.part[((size_t)h.u * p.rows_max + h.kvh * h.rows_g + h.r0 + lane) * (a.TV + a.TT) + h.tile] =
              make_float2(M, S);
        }
        if (h.last) {
          // the item's partials are all written (by this warp): hand the
          // item's completion to the service warps, which count it
          __threadfence();
          __syncwarp();
          if (lane == 0) post_job(a, c, SvcJob{kSvcDone1, h.u, h.b, h.l, h.n_v, h.n_tk, h.vis0});
        }
      }
      ++p1_it;
    } else {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (16 * mt + g4 + 8 * hh < h.rows) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) accK[nt][e] += exp2f(acc[mt][nt][2 * hh + e] - lse[mt][hh]);
          }
        }
      if (h.last) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float v = accK[nt][e];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            accK[nt][e] = v;
          }
        if (g4 == 0) {
          const float inv = 1.f / (float)(p.h_q * h.n_tk);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int key = h.key0 + 16 * warp + 8 * nt + 2 * c4 + e;
              if (key < h.n_v) {
                if (a.G == 1) {
                  w.iv[(size_t)h.l * p.total_visual + h.vis0 + key] = accK[nt][e] * inv;
                } else {
                  w.ivp[((size_t)h.grp * p.L + h.l) * p.total_visual + h.vis0 + key] = accK[nt][e];
                }
              }
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) accK[nt][e] = 0.f;
        if (a.tail || a.G > 1) {
          // the last consumer warp to finish the item hands it to the service
          __threadfence();
          __syncwarp();
          if (lane == 0) {
            int* done = &c->p2done[p2_items & 7];
            if (atomicAdd(done, 1) == kCW - 1) {
              *done = 0;
              post_job(a, c, SvcJob{kSvcDone2, h.u, h.b, h.l, h.n_v, h.n_tk, h.vis0});
            }
          }
        }
        ++p2_items;
      }
    }
    ++it;
  }
  // every consumer warp is past its last post: end the service
  named_bar_sync(kBar, kCT);
  if (tid == 0) post_job(a, c, SvcJob{kSvcEnd, 0, 0, 0, 0, 0, 0});
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const __grid_constant__ PArgs a) {
  using Gm = Geo<T, D>;
  constexpr int NS = Gm::kStages;
  extern __shared__ unsigned char smem_raw[];
  // stages need 1024-byte alignment (the 128-byte swizzle repeats every 8 rows)
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char* stages = smem;
  Ctl* c = reinterpret_cast<Ctl*>(smem + NS * Gm::kRing);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      // TMA: one arrival (with the byte count); cp.async: one per issuer lane + the header release
      mbar_init(&c->full[s], a.tma ? 1 : 33);
      mbar_init(&c->empty[s], kCW);
    }
    for (int i = 0; i < kQN; ++i) c->iq_state[i] = 0;
    for (int i = 0; i < kMN; ++i) {
      c->mb_seq[i] = i;
      c->mb_ready[i] = 0;
    }
    c->mb_tail = 0;
    for (int i = 0; i < 8; ++i) c->p2done[i] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if (warp < kCW) {
    consumers<T, D>(a, c, stages);
  } else if (warp == kIssuerWarp) {
    issuer<T, D>(a, c, stages);
  } else if (warp == kSchedWarp) {
    if ((threadIdx.x & 31) == 0) scheduler(a, c);
  } else {
    service(a, c);
  }
}

// ------------------------------------------------------------------ host

template <typename T, int D>
cudaError_t launch_t(const Dev& p, const LayerPtrs& lp, const Ws& w, const ScoreLaunch& L, cudaStream_t s) {
  using Gm = Geo<T, D>;
  PArgs a;
  std::memset(&a, 0, sizeof a);
  a.p = p;
  a.lp = lp;
  a.w = w;
  a.TV = L.TV;
  a.TT = L.TT;
  a.G = L.G;
  a.tail = L.tail;
  a.n_p1 = L.tickets;
  a.out_capacity = L.out_capacity;
  const long long U = (long long)p.L * p.B;
  a.tma = (L.allow_tma && encode_keys<T>(&a.kmap, p, lp, kTK) &&
           encode_rows<T>(&a.qmap, w.qel, p.d, U * p.rows_max, kRC) &&
           encode_rows<T>(&a.kelmap, w.kel, p.d, U * p.h_kv * p.max_elite, kTK))
              ? 1
              : 0;
  const int smem = Gm::kStages * Gm::kRing + kCtlBytes + 1024;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(score_kernel<T, D>), smem);
  if (e != cudaSuccess) return e;
  score_kernel<T, D><<<L.grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

ScoreLaunch plan_score(const Dev& p, int sms, bool tail, int64_t out_capacity) {
  ScoreLaunch L;
  const int esize = p.dtype == AIRCACHE_BF16 ? 2 : 4;
  L.TV = (p.max_visual + kTK - 1) / kTK;
  L.TT = (p.max_elite + kTK - 1) / kTK;
  L.G = (p.h_kv + kHG - 1) / kHG;
  (void)esize;
  const int U = p.L * p.B;
  L.lag = 0;
  L.tail = tail ? 1 : 0;
  L.tickets = (long long)U * (long long)(L.TV + L.TT) * L.G;  // pass-1 items
  long long grid = sms;
  if (grid > L.tickets) grid = L.tickets;
  L.grid = (int)(grid < 1 ? 1 : grid);
  L.out_capacity = out_capacity;
  L.allow_tma = 1;
  return L;
}

cudaError_t launch_score(const Dev& p, const LayerPtrs& lp, const Ws& w, const ScoreLaunch& L, cudaStream_t s) {
  if (p.dtype == AIRCACHE_BF16) {
    return p.d == 128 ? launch_t<__nv_bfloat16, 128>(p, lp, w, L, s) : launch_t<__nv_bfloat16, 64>(p, lp, w, L, s);
  }
  return p.d == 128 ? launch_t<float, 128>(p, lp, w, L, s) : launch_t<float, 64>(p, lp, w, L, s);
}

}  // namespace aircache
