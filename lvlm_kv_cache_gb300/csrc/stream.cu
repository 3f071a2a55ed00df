// Cross-modal scores (AirCache notes, "Key design 1": equations A_vtk and I_v)
// on the streaming path: bf16 inputs whose keys a TMA tensor map can address.
//
// Problem.  For one (layer l, request b) -- a "unit" -- the query rows are the
// pairs (query head, elite text position): g * N_tk rows read each KV head
// (g = H_q/H_kv).  Each row is a softmax over the N_v visual keys and the N_tk
// elite text keys; I_v[i] is the mean over all H_q N_tk rows of the
// probability of visual key i.  With an elite threshold near the notes'
// alpha = 0.9 the window holds a few text tokens, so a unit has few rows and
// many keys, and scoring is a stream over the keys.  Rows are taken in chunks
// of 32 (the N extent of one tensor-core logit tile).
//
// Pass 1 (score_pass1, persistent, one CTA per SM).  A work item is (unit, KV
// head, chunk of four 128-key visual tiles) or (unit, KV head, the elite text
// keys); it runs once per row chunk of the unit.  A producer thread takes the
// CTA's index as its first item, claims the rest from an atomic counter, and
// moves each key tile into a shared-memory
// ring with one TMA tensor copy per 128-byte column slab; the row chunk's
// queries come with its first tile.  One thread issues the logit tiles on the
// tensor cores (tcgen05: D[key][row] = K[key] . Q[row], M = 128 keys, N = 32
// rows, fp32 accumulators in tensor memory, four accumulator buffers), and eight
// epilogue warps read them back one key per thread (32 rows in registers),
// store them (below) and keep per-row sums of exp2 of the base-2 logits against
// a per-warp reference; at the item's end the sums are reduce-scattered over
// the lanes and the warps' pairs merged in a fixed order into one partial
// (max, sum of exp2) per (row, item).  A unit with at most two row chunks per
// KV head (64 rows) also writes its visual logits to a row-major buffer (4
// bytes per row and key: cheaper than reading a 256-byte key row again; the
// logits of the units in flight stay in L2).  The keys of a unit with a single
// row chunk are read once, with an L2 evict-first policy.
//
// Pass 2 (score_pass2, persistent, two CTAs per SM).  Units with stored logits: each CTA takes a
// contiguous range of (unit, 256 keys) items, merges a unit's row partials
// (chunk order) into row log-sum-exps when it enters the unit, then sums
// exp2(logit - lse) over every row of every KV head for each key.  Units
// without stored logits (more than 64 rows per KV head): the CTAs first merge
// their row LSEs into the workspace for pass 2k.
//
// Pass 2k (score_pass2k, persistent).  Units without stored logits: a work item is (unit,
// key tile); for each KV head the tile is loaded once and its B fragments stay
// in registers while that head's row chunks (queries + LSEs) stream through a
// small TMA ring; per-key sums of exp2(logit - lse) over every row give the
// tile's I_v directly.
//
// Passes 2 and 2k also reduce each key block's I_v to a moment record (256
// keys in pass 2, a 128-key tile in pass 2k) and count the records per unit.
// The CTA whose record completes a unit merges the unit's records into its
// layer statistics (s_t, s_k).  The budgets and the selection follow in the
// selection kernel (select.cu), the row offsets in the compaction.
#include <cstring>

#include "internal.cuh"
#include "ptx.cuh"
#include "reduce.cuh"
#include "tmap.cuh"
#include "umma.cuh"
#include "timeline.cuh"

namespace aircache {
namespace {

constexpr int kTK = 128;                  // keys per tile
constexpr int kRC = kRowChunk;            // query rows per chunk
constexpr int kCK = kStreamTiles;         // visual tiles per pass-1 item
constexpr int kCW = 8;                    // consumer warps
constexpr int kCT = kCW * 32;             // consumer threads
constexpr int kThreads1 = kCT + 64;       // + the producer warp and the MMA warp
constexpr int kMmaWarp = kCW + 1;         // issues the pass-1 MMAs; allocates the TMEM
constexpr int kNB = 4;                    // pass-1 TMEM accumulator buffers
constexpr int kTmemStage = 2 * kRowChunk; // TMEM columns of one buffer: two 128-key tiles x 32 rows
constexpr int kTmemCols = kNB * kTmemStage;
constexpr int kBarC = 1;                  // named barrier of the consumer threads
constexpr int kT2 = 256;                  // pass-2 / pass-2k threads
constexpr int kBarT2 = 1;                 // named barrier over all kT2 threads
constexpr int kMaxStages = 12;
constexpr int kNQ = 4;                    // pass-2k query-chunk ring

enum : int { kEnd = 0, kVis = 1, kTxt = 2 };

template <int D>
struct SGeo {
  static constexpr int kKS = D / 16;       // mma k-steps
  static constexpr int kNH = D * 2 / 128;  // 128-byte slabs per bf16 row
  static constexpr int kKSlab = kTK * 128;
  static constexpr int kKBytes = kNH * kKSlab;
  static constexpr int kQSlab = kRC * 128;
  static constexpr int kQBytes = kNH * kQSlab;
  // pass 1: ring of 256-key stages, two query buffers, control
  static constexpr int kSK = 2 * kTK;       // keys per pass-1 stage
  static constexpr int kSSlab = kSK * 128;  // one 128-byte column slab of a stage
  static constexpr int kSBytes = kNH * kSSlab;
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kQOff = kStages * kSBytes;
  static constexpr int kCtlOff = kQOff + 2 * kQBytes;
  static_assert(kStages <= kMaxStages, "ring depth");
  // pass 2k: one key tile, kNQ query chunks (+ their LSEs), control
  static constexpr int kQ2 = (kQBytes + kRC * 4 + 1023) / 1024 * 1024;
  static constexpr int kCtl2Off = kKBytes + kNQ * kQ2;
};

struct SArgs {
  CUtensorMap kmap;    // keys of every layer: (D, H_kv, tokens, layers), box 128 tokens (pass 2k)
  CUtensorMap kmap2;   // the same keys, box 256 tokens (pass 1)
  CUtensorMap qmap;    // gathered elite query rows (D, rows), box 32 rows
  CUtensorMap kelmap;  // gathered elite text keys (D, rows), box 128 rows
  CUtensorMap lgmap;   // stored logits (columns, rows), box 256 columns x 8 rows
  Dev p;
  Ws w;
};

// Logit buffer: row r of KV head h of layer l holds the logits of every
// request's visual keys; request b's keys start at column lg_col0(vis0, b),
// a multiple of 4 (so that pairs of keys are 8-byte aligned), and rows are
// lg_stride(p) floats apart.
__device__ __forceinline__ long long lg_col0(long long vis0, int b) { return (vis0 + 3) / 4 * 4 + 4LL * b; }
__device__ __forceinline__ long long lg_stride(const Dev& p) { return (p.total_visual + 4LL * p.B + 7) / 4 * 4; }

__device__ __forceinline__ float2 merge_ms(float2 a, float2 b) {
  const float m = fmaxf(a.x, b.x);
  if (m == -INFINITY) return make_float2(-INFINITY, 0.f);
  return make_float2(m, a.y * fast_exp2(a.x - m) + b.y * fast_exp2(b.x - m));
}

__device__ __forceinline__ bool stream_unit(const Dev& p, int u, const int4& i0, const int4& i1) {
  const int n_v = i0.w, n_t = i1.x, n_tk = i1.y;
  return u >= 0 && u < p.L * p.B && i1.z == 1 && n_tk >= 1 && (n_tk <= n_t || p.window_mode == 4) &&
         n_tk <= p.max_elite &&
         n_v >= 3 && n_v <= p.max_visual && i0.x >= 0 && (long long)i0.x + n_v <= p.total_tokens &&
         i0.y >= 0 && (long long)i0.y + n_v <= p.total_visual;
}

__device__ __forceinline__ int rows_per_kv(const Dev& p) { return p.rc_max * kRC; }

// Slot in stream_list / stream_info of position li of the streaming units in
// claim order (units without stored logits first; n_multi of n_total).
__device__ __forceinline__ int stream_slot(const Dev& p, int li, int n_multi, int n_total) {
  return li < n_multi ? li : p.L * p.B - (n_total - li);
}

// Row partial (row, chunk) of KV head kvh of unit u.
__device__ __forceinline__ size_t part_index(const Dev& p, int u, int kvh, int row, int chunk) {
  return (((size_t)u * p.h_kv + kvh) * rows_per_kv(p) + row) * p.chn + chunk;
}

// Merge row `row`'s partials in chunk order (visual chunks, then the text chunk)
// into its base-2 log-sum-exp (one thread).  Loads are issued sixteen chunks
// (and the text chunk) at a time; a padding partial (-inf, 0) leaves the merge
// unchanged, so the batch size does not change the result.
__device__ __forceinline__ float row_lse(const Dev& p, const Ws& w, int u, int kvh, int row, int chv) {
  const float2* pr = w.part_s + part_index(p, u, kvh, row, 0);
  const float2 txt = __ldcg(pr + p.chn - 1);
  float2 ms = make_float2(-INFINITY, 0.f);
  for (int c0 = 0; c0 < chv; c0 += 16) {
    float2 v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = (c0 + q < chv) ? __ldcg(pr + c0 + q) : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int q = 0; q < 16; ++q) ms = merge_ms(ms, v[q]);
  }
  ms = merge_ms(ms, txt);
  return ms.x + log2f(ms.y);
}

// ------------------------------------------------------------------ pass 1

struct Hdr {
  int kind, u, l, kvh, key0, klim, rows, r0, first, last, chunk, qbuf, store, b;
  long long vis0;
};

struct Ctl1 {
  uint64_t full[kMaxStages], empty[kMaxStages], qempty[2];
  uint64_t tfull[kNB], tempty[kNB];  // TMEM accumulator buffers: MMA done / read by every epilogue warp
  Hdr hdr[kMaxStages];
  Hdr thdr[kNB];                     // the stage header of what TMEM buffer b holds
  float2 red[2][2][4][kRC];          // [warpgroup][parity][warp][row] per-warp stage partials
  uint32_t tmem;                     // TMEM base address
};

// One thread.  Items (unit, KV head, chunk of four visual tiles or the elite
// text keys) are claimed from an atomic counter; the claim after the current
// one and its unit's layout record (stored beside the list slot by the elite
// kernel) are fetched while the current item's stages are issued, so no
// dependent load stalls the ring between items.  A visual stage is 256 keys
// (one TMA box of 256 rows per column slab), a text stage up to 128 elite keys.
template <int D>
__device__ void p1_producer(const SArgs& a, Ctl1* c, unsigned char* sm) {
  using Gm = SGeo<D>;
  constexpr int NS = Gm::kStages;
  const Dev& p = a.p;
  const Ws& w = a.w;
  const uint32_t sbase = smem_u32(sm);
  const long long per_unit = (long long)p.h_kv * p.chn;
  const int n_total = __ldcg(&w.list_n[0]), n_multi = __ldcg(&w.list_n[2]);
  const long long total = (long long)n_total * per_unit;
  const uint64_t evict_first = l2_evict_first_policy();
  auto record = [&](long long claim, int4& r0, int4& r1) {
    if (claim < total) {
      const int slot = stream_slot(p, (int)(claim / per_unit), n_multi, n_total);
      r0 = __ldcg(&w.stream_info[2 * slot]);
      r1 = __ldcg(&w.stream_info[2 * slot + 1]);
    }
  };
  long long st = 0;  // stages issued
  int sub = 0;       // row-chunk passes issued (selects the query buffer)
  bool ok = true;
  // the CTA's first item is its index, the later ones come from the counter
  // (after the first grid-size items): no atomic round trip before the first stage
  const long long G = gridDim.x;
  long long claim = blockIdx.x;
  long long next = G + (long long)atomicAdd(w.ticket_n, 1ULL);
  int4 i0 = make_int4(0, 0, 0, 0), i1 = make_int4(0, 0, 0, 0);
  record(claim, i0, i1);
  while (ok && claim < total) {
    int4 n0 = make_int4(0, 0, 0, 0), n1 = make_int4(0, 0, 0, 0);
    record(next, n0, n1);                                                   // used by the next item
    const long long next2 = G + (long long)atomicAdd(w.ticket_n, 1ULL);  // the claim after that
    const int rem = (int)(claim % per_unit);
    const int kvh = rem / p.chn, ch = rem % p.chn;
    const int u = i1.w;
    if (!stream_unit(p, u, i0, i1)) {
      set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
      break;
    }
    const int n_v = i0.w, n_tk = i1.y, rows = p.g * n_tk;
    const int n_rc = (rows + kRC - 1) / kRC;
    const int tv = (n_v + kTK - 1) / kTK;
    const int chv = (tv + kCK - 1) / kCK;
    const bool skip = ch < p.chn - 1 && ch >= chv;  // a chunk past this unit's keys
    if (!skip) {
      int kind, key0, nkeys, stage_keys;
      if (ch < p.chn - 1) {
        kind = kVis;
        key0 = ch * kCK * kTK;
        nkeys = min(kCK * kTK, n_v - key0);
        stage_keys = Gm::kSK;
      } else {
        kind = kTxt;  // elite text keys: at most max_elite <= 8192, 128 per stage
        key0 = 0;
        nkeys = p.window_mode == 4 ? 0 : n_tk;  // the visual window adds no keys: one empty stage
        stage_keys = kTK;
      }
      const int nst = max(1, (nkeys + stage_keys - 1) / stage_keys);
      const uint32_t kbytes = kind == kVis ? (uint32_t)Gm::kSBytes : (uint32_t)(Gm::kNH * kTK * 128);
      const int l = u / p.B;
      for (int rc = 0; ok && rc < n_rc; ++rc, ++sub) {
        const int qb = sub & 1;
        // the query buffer is free once the MMAs of the pass that used it before have completed
        if (!mbar_wait(&c->qempty[qb], (uint32_t)(((sub >> 1) & 1) ^ 1))) {
          ok = false;
          break;
        }
        for (int j = 0; j < nst; ++j, ++st) {
          const int s = (int)(st % NS);
          if (!mbar_wait(&c->empty[s], (uint32_t)(((st / NS) & 1) ^ 1))) {
            ok = false;
            break;
          }
          const int k0 = key0 + j * stage_keys;
          Hdr& h = c->hdr[s];
          h.kind = kind;
          h.u = u;
          h.l = l;
          h.kvh = kvh;
          h.key0 = k0;
          h.klim = min(stage_keys, (kind == kVis ? n_v : nkeys) - k0);
          h.rows = min(kRC, rows - rc * kRC);
          h.r0 = rc * kRC;
          h.first = (j == 0);
          h.last = (j == nst - 1);
          h.chunk = ch;
          h.qbuf = qb;
          h.store = (kind == kVis && n_rc * kRC <= kLgRows) ? 1 : 0;
          h.b = u % p.B;
          h.vis0 = i0.y;
          fence_proxy_async_smem();  // the stage (and query buffer) were last read by generic loads
          mbar_arrive_expect_tx(&c->full[s], kbytes + (j == 0 ? (uint32_t)Gm::kQBytes : 0u));
          const uint32_t kdst = sbase + (uint32_t)(s * Gm::kSBytes);
#pragma unroll
          for (int sl = 0; sl < Gm::kNH; ++sl) {
            if (kind == kVis) {
              if (n_rc == 1) {  // read once
                tma_load_4d_hint(kdst + sl * Gm::kSSlab, &a.kmap2, sl * 64, kvh, i0.x + k0, l, &c->full[s],
                                 evict_first);
              } else {  // read again by the next row chunk
                tma_load_4d(kdst + sl * Gm::kSSlab, &a.kmap2, sl * 64, kvh, i0.x + k0, l, &c->full[s]);
              }
            } else {
              tma_load_2d(kdst + sl * Gm::kSSlab, &a.kelmap, sl * 64, (u * p.h_kv + kvh) * p.max_elite + k0,
                          &c->full[s]);
            }
          }
          if (j == 0) {
            const uint32_t qdst = sbase + (uint32_t)(Gm::kQOff + qb * Gm::kQBytes);
#pragma unroll
            for (int sl = 0; sl < Gm::kNH; ++sl) {
              tma_load_2d(qdst + sl * Gm::kQSlab, &a.qmap, sl * 64, u * p.rows_max + kvh * rows + rc * kRC,
                          &c->full[s]);
            }
          }
        }
      }
    }
    claim = next;
    next = next2;
    i0 = n0;
    i1 = n1;
  }
  if (!ok) {
    set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
    return;  // consumers give up on their own (longer) wait
  }
  const int s = (int)(st % NS);
  if (!mbar_wait(&c->empty[s], (uint32_t)(((st / NS) & 1) ^ 1))) {
    set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
    return;
  }
  c->hdr[s].kind = kEnd;
  mbar_arrive(&c->full[s]);
}

// One thread.  For every stage the producer filled: wait for the TMA bytes and
// for a free TMEM buffer of the warpgroup that owns the stage's row-chunk pass
// (passes alternate between the two epilogue warpgroups, like the query
// buffers: warpgroup g takes the passes with query buffer g and owns TMEM
// buffers 2g and 2g + 1), hand the stage header to that buffer, and issue the
// logit tile(s) D[key][row] = K[key] . Q[row] (M = 128 keys per tile, N = 32
// query rows, K = D in steps of 16) on the tensor cores.  The stage is released
// to the producer, the query buffer after the last stage of a pass, and the
// accumulators to the warpgroup, each when those MMAs complete.
template <int D>
__device__ void p1_mma(const SArgs& a, Ctl1* c, unsigned char* sm, uint32_t tmem) {
  using Gm = SGeo<D>;
  constexpr int NS = Gm::kStages;
  constexpr int KS = Gm::kKS;
  const uint32_t sbase = smem_u32(sm);
  constexpr uint32_t idesc = umma_idesc_bf16(kTK, kRC);
  long long ng[2] = {0, 0};  // stages handed to each warpgroup
  // the next TMEM buffer of warpgroup g, once its previous use is read
  auto take = [&](int g, int& b) -> bool {
    b = 2 * g + (int)(ng[g] & 1);
    const bool ok = mbar_wait(&c->tempty[b], (uint32_t)(((ng[g] >> 1) & 1) ^ 1), 8 * kWaitCycles);
    ++ng[g];
    return ok;
  };
  for (long long it = 0;; ++it) {
    const int s = (int)(it % NS);
    if (!mbar_wait(&c->full[s], (uint32_t)((it / NS) & 1), 8 * kWaitCycles)) {
      set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      return;
    }
    const Hdr h = c->hdr[s];
    if (h.kind == kEnd) {
      for (int g = 0; g < 2; ++g) {  // both warpgroups learn of the end
        int b;
        if (!take(g, b)) {
          set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
          return;
        }
        c->thdr[b] = h;
        mbar_arrive(&c->tfull[b]);
        mbar_arrive(&c->tfull[b]);
      }
      return;
    }
    int b;
    if (!take(h.qbuf, b)) {
      set_error(a.w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      return;
    }
    c->thdr[b] = h;
    tc_fence_after();
    const int ntiles = h.klim > kTK ? 2 : (h.klim > 0 ? 1 : 0);
    const uint32_t kst = sbase + (uint32_t)(s * Gm::kSBytes);
    const uint32_t qst = sbase + (uint32_t)(Gm::kQOff + h.qbuf * Gm::kQBytes);
    for (int t = 0; t < ntiles; ++t) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const uint32_t ka = kst + (uint32_t)((kk >> 2) * Gm::kSSlab + t * kTK * 128 + (kk & 3) * 32);
        const uint32_t qb = qst + (uint32_t)((kk >> 2) * Gm::kQSlab + (kk & 3) * 32);
        umma_bf16(tmem + (uint32_t)(b * kTmemStage + t * kRC), umma_desc_sw128(ka), umma_desc_sw128(qb), idesc,
                  kk > 0 ? 1u : 0u);
      }
    }
    umma_commit(&c->empty[s]);                   // the stage may be refilled once these MMAs have read it
    if (h.last) umma_commit(&c->qempty[h.qbuf]);  // and the query buffer after the pass's last stage
    umma_commit(&c->tfull[b]);                   // the accumulators are written
    mbar_arrive(&c->tfull[b]);                   // the header copy is visible
  }
}

// Reduce-scatter of 32 per-row values over the lanes of a warp (31 shuffles):
// afterwards lane t returns the sum over all lanes of row t.  `v` is consumed.
__device__ __forceinline__ float warp_rows_sum(float (&v)[kRC], int lane) {
#pragma unroll
  for (int o = kRC / 2; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < o; ++j) {
      const float send = up ? v[j] : v[j + o];
      const float keep = up ? v[j + o] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// The same for (max, sum of exp2) pairs with different maxima; the lower
// lanes' partial is always the first operand, so every lane merges in one order.
__device__ __forceinline__ float2 warp_rows_merge(float (&m)[kRC], float (&s)[kRC], int lane) {
#pragma unroll
  for (int o = kRC / 2; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < o; ++j) {
      const float2 send = up ? make_float2(m[j], s[j]) : make_float2(m[j + o], s[j + o]);
      const float2 keep = up ? make_float2(m[j + o], s[j + o]) : make_float2(m[j], s[j]);
      const float2 other =
          make_float2(__shfl_xor_sync(0xffffffffu, send.x, o), __shfl_xor_sync(0xffffffffu, send.y, o));
      const float2 r = up ? merge_ms(other, keep) : merge_ms(keep, other);
      m[j] = r.x;
      s[j] = r.y;
    }
  }
  return make_float2(m[0], s[0]);
}

// v[lane] without dynamic register indexing: the reduce-scatter's selection
// pattern without the exchange (31 selects, depth 5).  `v` is consumed.
__device__ __forceinline__ float pick_lane(float (&v)[kRC], int lane) {
#pragma unroll
  for (int o = kRC / 2; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < o; ++j) v[j] = up ? v[j + o] : v[j];
  }
  return v[0];
}

// Two warpgroups of four warps; warpgroup g takes the row-chunk passes of query
// buffer g (every other pass), so the two work on consecutive items at once.
// Warp w reads TMEM lane quarter w % 4 of both key tiles of a stage: thread
// (w, lane) holds the 32 row logits of keys 32(w%4) + lane and 128 + 32(w%4) +
// lane.  It stores them (units with stored logits: row-major logit buffer, coalesced
// across the warp) and keeps, per row, a sum of exp2(scaled logit - m) against
// a reference m shared by the warp: the scaled logit of the warp's first key in
// the item.  A logit more than 2^6 above the reference (never seen on the
// workloads here) moves that thread's reference up and rescales its sum.  At
// the item's end the warp's sums are reduce-scattered (lane t: row t) and the
// warpgroup's four pairs are merged in order into the item's row partial.
template <int D>
__device__ void p1_epilogue(const SArgs& a, Ctl1* c, uint32_t tmem) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = warp >> 2, q = warp & 3;
  const float scale = p.scale_log2;
  const long long LS = lg_stride(p);
  const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
  const int k0 = 32 * q, k1 = kTK + 32 * q;  // this warp's first key in each tile of a stage
  float m[kRC], s[kRC];
#pragma unroll
  for (int r = 0; r < kRC; ++r) {
    m[r] = 0.f;
    s[r] = 0.f;
  }
  bool has_ref = false, resc = false;
  int par = 0;
  for (long long k = 0;; ++k) {
    const int b = 2 * g + (int)(k & 1);
    if (!mbar_wait(&c->tfull[b], (uint32_t)((k >> 1) & 1), 16 * kWaitCycles)) {
      if (lane == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      return;
    }
    __syncwarp();  // tcgen05.ld is warp-collective: the whole warp, converged
    tc_fence_after();
    const Hdr h = c->thdr[b];
    if (h.kind == kEnd) return;
    if (h.first) {
      has_ref = false;
      resc = false;
#pragma unroll
      for (int r = 0; r < kRC; ++r) s[r] = 0.f;
    }
    const bool busy0 = k0 < h.klim, busy1 = k1 < h.klim;  // warp-uniform
    // tile 0 first; the buffer is released after the last TMEM load of the stage
    float v[kRC];
    if (busy0) {
      tmem_ld32(tl + (uint32_t)(b * kTmemStage), v);
      tmem_wait_ld();
    }
    auto release = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->tempty[b]);  // this warp is done with the buffer
    };
    if (!busy1) release();
    if (busy0) {
      if (!has_ref) {
        // lane 0's key exists whenever the warp is busy
#pragma unroll
        for (int r = 0; r < kRC; ++r) m[r] = __shfl_sync(0xffffffffu, v[r], 0) * scale;
        has_ref = true;
      }
      float* dst = nullptr;
      if (h.store)
        dst = w.lg + (((size_t)h.l * p.h_kv + h.kvh) * kLgRows + h.r0) * LS + lg_col0(h.vis0, h.b) + h.key0;
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        if (t == 1) {
          if (!busy1) break;
          __syncwarp();
          tmem_ld32(tl + (uint32_t)(b * kTmemStage + kRC), v);
          tmem_wait_ld();
          release();
        }
        const int key = (t ? k1 : k0) + lane;
        if (key < h.klim) {
          // blocks of 8 rows: the block's exponents are computed first and
          // checked against the reference once, so the block's exponentials
          // and sums carry no branch between them
#pragma unroll
          for (int g8 = 0; g8 < kRC / 8; ++g8) {
            if (8 * g8 < h.rows) {
              float d[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) d[j] = fmaf(v[8 * g8 + j], scale, -m[8 * g8 + j]);
              const float dmax = fmaxf(fmaxf(fmaxf(d[0], d[1]), fmaxf(d[2], d[3])),
                                       fmaxf(fmaxf(d[4], d[5]), fmaxf(d[6], d[7])));
              if (dst) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (8 * g8 + j < h.rows) dst[(size_t)(8 * g8 + j) * LS + key] = v[8 * g8 + j];
              }
              if (dmax > 64.f) {  // a logit far above the reference: move it (rare)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  if (d[j] > 64.f) {
                    s[8 * g8 + j] *= fast_exp2(-d[j]);
                    m[8 * g8 + j] = v[8 * g8 + j] * scale;
                    d[j] = 0.f;
                  }
                }
                resc = true;
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) s[8 * g8 + j] += fast_exp2(d[j]);
            }
          }
        }
      }
    }
    if (h.last) {
      float2 pr;
      if (!has_ref) {
        pr = make_float2(-INFINITY, 0.f);
      } else if (!__any_sync(0xffffffffu, resc)) {
        const float S = warp_rows_sum(s, lane);
        pr = make_float2(pick_lane(m, lane), S);
      } else {
        pr = warp_rows_merge(m, s, lane);
      }
      c->red[g][par][q][lane] = pr;
      named_bar_sync(kBarC + g, 4 * 32);
      if (q == 0 && lane < h.rows) {
        float2 ms = c->red[g][par][0][lane];
#pragma unroll
        for (int ww = 1; ww < 4; ++ww) ms = merge_ms(ms, c->red[g][par][ww][lane]);
        w.part_s[part_index(p, h.u, h.kvh, h.r0 + lane, h.chunk)] = ms;
      }
      par ^= 1;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads1, 1) stream_p1_kernel(const __grid_constant__ SArgs a) {
  AIRCACHE_KT(1);
  using Gm = SGeo<D>;
  extern __shared__ unsigned char smem_raw[];
  // tiles need 1024-byte alignment (the 128-byte swizzle repeats every 8 rows)
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Ctl1* c = reinterpret_cast<Ctl1*>(sm + Gm::kCtlOff);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Gm::kStages; ++s) {
      mbar_init(&c->full[s], 1);
      mbar_init(&c->empty[s], 1);
    }
    for (int b = 0; b < kNB; ++b) {
      mbar_init(&c->tfull[b], 2);  // the MMA completion and the header hand-off
      mbar_init(&c->tempty[b], 4);  // the four warps of the warpgroup that reads it
    }
    mbar_init(&c->qempty[0], 1);
    mbar_init(&c->qempty[1], 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_alloc(&c->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem;
  pdl_trigger();
  if (threadIdx.x == kCT) {  // the producer's tensor maps, fetched while the elite kernel runs
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&a.kmap2)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&a.qmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&a.kelmap)) : "memory");
  }
  pdl_wait();  // the elite kernel's lists, query rows and elite keys
  if (*(volatile int32_t*)a.w.error == 0) {  // else an earlier kernel reported an error
    if (threadIdx.x < kCT) {
      p1_epilogue<D>(a, c, tmem);
    } else if (threadIdx.x == kCT) {
      p1_producer<D>(a, c, sm);
    } else if (threadIdx.x == kCT + 32) {
      p1_mma<D>(a, c, sm, tmem);
    }
  }
  __syncwarp();  // the role threads rejoin their warps
  tc_fence_before();
  __syncthreads();  // every TMEM read and every MMA of this CTA is done
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ pass 2

constexpr int kKeysP2 = kT2;                  // keys per pass-2 item (one per thread)
constexpr int kP2Box = 8;                     // logit rows per TMA box
constexpr int kP2Slice = kRC * kKeysP2 * 4;   // one KV head's logits of an item (32 KB)
constexpr int kP2Stages = 3;                  // slices in flight (two CTAs per SM)
constexpr int kMomT = 128;                    // pass-2 moment threads (two values each)
constexpr int kT2p = kT2 + 32 + kMomT;        // pass-2 threads: streamers, the producer warp, moment warps
constexpr int kP2Prod = kT2 / 32;             // the producer warp
constexpr int kBarP2S = 1;                    // named barrier of the streamers
constexpr int kBarP2M = 2;                    // named barrier of the moment warps
constexpr int kP2CtlOff = kP2Stages * kP2Slice;

// What a pass-2 stage holds: the logits of KV head kvh for item (unit u, key
// block kb), or the end of the CTA's walk (state 1), or a unit record that
// failed validation (state 2).
struct P2Rec {
  int state, u, l, b, kb, n_v, n_tk, rows, kvh, rc;
  long long vis0;
};

// Hand-off of one item's I_v from the streaming warps to the moment warps.
struct P2Hand {
  int u, kb, n, end;
  int nb;  // the unit's 256-key blocks (its moment records)
};

struct Ctl2p {
  uint64_t full[kP2Stages], empty[kP2Stages];
  uint64_t hfull[2], hempty[2];  // hand-off buffers: filled by the streamers, released by the moment warps
  P2Rec rec[kP2Stages];
  P2Hand hand[2];
  float hx[2][kKeysP2];
};

// The walk of a CTA's items over the pass-2 units (unit si in slot L*B - 1 - si,
// in routing order) and their 256-key blocks kb.  Item (si, kb) starts at
// weight wpre(si) + kb * nrc (nrc = 32-row chunks per KV head); the CTA takes
// the items that start in its share [lo, hi) of the total weight.  The unit's
// layout record (seq0, vis0, txt0, n_v), (n_t, n_tk, 1, u) and weight prefix
// are loaded once per unit.
struct P2Cursor {
  int si, kb, n;
  unsigned long long hi;
  int loaded = -1;
  int4 r0, r1;
  unsigned long long wpre;
  int nrc, nkb;
};

// Move the cursor to the first item at or after it (the cursor stays on it).
// Returns 0 past the CTA's share, 1 with the item in `r`, 2 for a unit record
// that fails validation.
__device__ __forceinline__ int p2_item(const Dev& p, const Ws& w, P2Cursor& cu, P2Rec& r) {
  while (cu.si < cu.n) {
    if (cu.si != cu.loaded) {
      cu.loaded = cu.si;
      const int slot = p.L * p.B - 1 - cu.si;
      cu.r0 = __ldcg(&w.stream_info[2 * slot]);
      cu.r1 = __ldcg(&w.stream_info[2 * slot + 1]);
      cu.wpre = __ldcg(&w.p2wpre[slot]);
      if (!stream_unit(p, cu.r1.w, cu.r0, cu.r1) || p.g * cu.r1.y > kLgRows) return 2;
      cu.nrc = (p.g * cu.r1.y + kRC - 1) / kRC;
      cu.nkb = (cu.r0.w + kKeysP2 - 1) / kKeysP2;
    }
    if (cu.wpre + (unsigned long long)cu.kb * cu.nrc >= cu.hi) return 0;
    if (cu.kb < cu.nkb) {
      const int4 r0 = cu.r0, r1 = cu.r1;
      r.state = 0;
      r.u = r1.w;
      r.l = r1.w / p.B;
      r.b = r1.w % p.B;
      r.kb = cu.kb;
      r.n_v = r0.w;
      r.n_tk = r1.y;
      r.rows = p.g * r1.y;
      r.kvh = 0;
      r.rc = 0;
      r.vis0 = r0.y;
      return 1;
    }
    ++cu.si;
    cu.kb = 0;
  }
  return 0;
}

// Step past the current item.
__device__ __forceinline__ void p2_next(P2Cursor& cu) { ++cu.kb; }

// The pass-2 unit that holds weight position `lo` (the largest si with
// wpre(si) <= lo), by the 32 lanes of a warp: each round probes 32 evenly
// spaced units and keeps the span after the last one at or below `lo`.
__device__ __forceinline__ int p2_find(const Dev& p, const Ws& w, int n, unsigned long long lo, int lane) {
  int a = 0, b = n;  // answer in [a, b); wpre(a) <= lo
  while (b - a > 1) {
    const int step = (b - a + 31) / 32;
    const int k = a + lane * step;
    const bool le = k < b && (unsigned long long)__ldcg(&w.p2wpre[p.L * p.B - 1 - k]) <= lo;
    const unsigned bal = __ballot_sync(0xffffffffu, le);
    const int last = 31 - __clz((int)bal);  // lane 0 always qualifies
    a += last * step;
    b = min(b, a + step);
  }
  return a;
}

// Pass 2 for units with stored logits (g * N_tk <= 64), persistent: CTA c takes
// a contiguous range of the (unit, 256-key block) items.  A producer warp walks
// the range and loads, for each item, KV head and 32-row chunk, those logits
// (256 keys) by TMA into a ring of 32 KB shared-memory stages, with a record of
// what the stage holds.  Streaming thread t owns key k0 + t and sums
// exp2(logit - lse) over the rows of every KV head, writes I_v and hands the
// item's values to the moment warps (double-buffered), which reduce them to the
// item's moment record while the streamers go on.  The row LSEs of a unit are
// merged from pass 1's partials (one row per thread) when the walk enters the unit.
// Units without stored logits: every thread first helps publish their row LSEs
// for pass 2k.

// Shared state of a pass-2 CTA.
// After a moment record of unit u is stored by lane 0 of the calling warp: count
// it in cnt_p2 and, if it completes the unit (nb records), merge the unit's
// records into its layer statistics (s_t, s_k).  The selection kernel then
// reads one record per layer instead of merging them in every CTA of the
// request.  The merge is the function the selection used, on the same records
// in the same order: the keep counts do not change.  One warp.
__device__ __forceinline__ void unit_record_done(const Dev& p, const Ws& w, int u, int nb, int lane) {
  int last = 0;
  if (lane == 0) {
    unsigned old;  // release: the record before its count
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;\n" : "=r"(old) : "l"(w.cnt_p2 + u) : "memory");
    last = old == (unsigned)(nb - 1) ? 1 : 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();  // (acquire) the unit's other records, counted by other CTAs
  ff s_t, s_k;
  layer_stats_warp(w.mom + (size_t)u * p.mom_slots * kMomWords, nb, lane, s_t, s_k);
  if (lane == 0) w.lstat[u] = make_float4(s_t.hi, s_t.lo, s_k.hi, s_k.lo);
}

struct P2Smem {
  unsigned char* sm;  // stage area
  Ctl2p* c;           // ring and the moment hand-off
  float* lse_s;       // [h_kv][kLgRows] row LSEs of the current unit
  ff* red;
  float* redf;
};

// Hand an item (or the end) from the 256 streamers to the moment warps.  The
// caller's values go to hx[hb][key] where `ok`; every streamer arrives.
__device__ __forceinline__ bool p2_hand_off(Ctl2p* c, int& n_hand, const P2Hand& h, int nval, const float* x,
                                            const int* key, const bool* ok) {
  const int hb = n_hand & 1;
  if (!mbar_wait(&c->hempty[hb], (uint32_t)(((n_hand >> 1) & 1) ^ 1), 4 * kWaitCycles)) return false;
  for (int i = 0; i < nval; ++i) {
    if (ok[i]) c->hx[hb][key[i]] = x[i];
  }
  if (threadIdx.x == 0) c->hand[hb] = h;
  mbar_arrive(&c->hfull[hb]);
  ++n_hand;
  return true;
}

// Moment warps: one record per handed-off item, until the end record.  They
// are idle until the first item arrives, and the first pass through the
// float-float code costs several microseconds of instruction fetches; so the
// loop starts with one pass over zeros (n = -1) whose record is discarded,
// through the same code, while the streamers are still on the first item.
__device__ __forceinline__ void p2_moments(const Dev& p, const Ws& w, const P2Smem& S, int mt) {
  Ctl2p* c = S.c;
  for (int n = -1;; ++n) {
    const int hb = n & 1;
    const bool warm = n < 0;
    if (!warm && !mbar_wait(&c->hfull[hb], (uint32_t)((n >> 1) & 1), 4 * kWaitCycles)) {
      if (mt == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      return;
    }
    P2Hand h;
    float xv[2] = {0.f, 0.f};
    float sh = 0.f;
    if (warm) {
      h.u = h.kb = h.end = 0;
      h.n = 2 * kMomT;
    } else {
      h = c->hand[hb];
      const float* hx = c->hx[hb];
      xv[0] = (!h.end && mt < h.n) ? hx[mt] : 0.f;
      xv[1] = (!h.end && mt + kMomT < h.n) ? hx[mt + kMomT] : 0.f;
      // shift: the mean of four of the item's values (the same in every thread)
      sh = h.end ? 0.f
                 : 0.25f * ((hx[0] + hx[min(64, h.n - 1)]) + (hx[min(128, h.n - 1)] + hx[min(192, h.n - 1)]));
      mbar_arrive(&c->hempty[hb]);
    }
    if (h.end) return;
    bool okv[2] = {mt < h.n, mt + kMomT < h.n};
    const Mom mb = block_moments<kMomT, 2>(xv, okv, (float)h.n, sh, S.red, S.redf, mt, kBarP2M);
    if (warm || mt >= 32) continue;
    if (mt == 0) mom_store(w.mom + ((size_t)h.u * p.mom_slots + h.kb) * kMomWords, mb);
    unit_record_done(p, w, h.u, h.nb, mt);
  }
}

// Stored-logit role: the producer warp (warp kP2Prod) and the 256 streamers
// over the items of the units with stored logits that start in weight [lo, hi).
__device__ __forceinline__ void p2_single(const SArgs& a, const P2Smem& S, unsigned long long lo,
                                          unsigned long long hi, int n) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  Ctl2p* c = S.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* slices = reinterpret_cast<const float*>(S.sm);  // [kP2Stages][32][256]
  if (warp == kP2Prod) {
    // producer: the warp finds the first unit of the share, then one thread
    // fills the ring and sends the end record
    const int si0 = lo < hi ? p2_find(p, w, n, lo, lane) : n;
    if (lane != 0) return;
    fence_proxy_async_global();  // the logits were written by the previous kernel's generic stores
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&a.lgmap)) : "memory");
    P2Cursor cu;
    cu.si = si0;
    cu.n = n;
    cu.hi = hi;
    cu.kb = 0;
    if (si0 < n) {
      // the first block of unit si0 that starts at or after lo
      const int slot = p.L * p.B - 1 - si0;
      const unsigned long long wp = __ldcg(&w.p2wpre[slot]);
      const int nrc = (p.g * __ldcg(&w.stream_info[2 * slot + 1]).y + kRC - 1) / kRC;
      if (nrc > 0 && lo > wp) cu.kb = (int)((lo - wp + nrc - 1) / nrc);
    }
    P2Rec pr = {};
    int pstate = p2_item(p, w, cu, pr);
    for (long long st = 0;; ++st) {
      const int slot = (int)(st % kP2Stages);
      if (!mbar_wait(&c->empty[slot], (uint32_t)(((st / kP2Stages) & 1) ^ 1), 4 * kWaitCycles)) {
        set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
        return;
      }
      if (pstate != 1) {
        c->rec[slot].state = pstate == 0 ? 1 : 2;
        mbar_arrive(&c->full[slot]);
        return;
      }
      c->rec[slot] = pr;
      const int rows_c = min(kRC, pr.rows - pr.rc * kRC);
      const int nb = (rows_c + kP2Box - 1) / kP2Box;
      fence_proxy_async_smem();  // the slot was last read by generic loads
      mbar_arrive_expect_tx(&c->full[slot], (uint32_t)(nb * kP2Box * kKeysP2 * 4));
      const int x = (int)(lg_col0(pr.vis0, pr.b) + (long long)pr.kb * kKeysP2);
      const int y = (pr.l * p.h_kv + pr.kvh) * kLgRows + pr.rc * kRC;
      for (int j = 0; j < nb; ++j) {
        tma_load_2d(smem_u32(S.sm + slot * kP2Slice + j * kP2Box * kKeysP2 * 4), &a.lgmap, x, y + j * kP2Box,
                    &c->full[slot]);
      }
      // stages run over (KV head, row chunk), head-major
      if (++pr.rc * kRC >= pr.rows) {
        pr.rc = 0;
        if (++pr.kvh == p.h_kv) {
          p2_next(cu);
          pstate = p2_item(p, w, cu, pr);
        }
      }
    }
  }
  if (warp > kP2Prod) return;
  // streamers
  const float scale = p.scale_log2;  // stored logits are raw q.k
  int cur_u = -1, n_hand = 0;
  float acc = 0.f, acc_h = 0.f;
  for (long long stage = 0;; ++stage) {
    const int slot = (int)(stage % kP2Stages);
    if (!mbar_wait(&c->full[slot], (uint32_t)((stage / kP2Stages) & 1), 4 * kWaitCycles)) {
      if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
      break;
    }
    const P2Rec it = c->rec[slot];
    if (it.state != 0) {
      if (it.state == 2 && tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
      break;
    }
    if (it.kvh == 0 && it.rc == 0) {
      if (it.u != cur_u) {
        // the unit's row LSEs, one row per thread (each row's partials loaded at once)
        named_bar_sync(kBarP2S, kT2);  // every streamer is done with the previous unit's LSEs
        const int chv = ((it.n_v + kTK - 1) / kTK + kCK - 1) / kCK;
        const int nr = p.h_kv * it.rows;
        for (int q = tid; q < nr; q += kT2) {
          const int kvh = q / it.rows, r = q % it.rows;
          S.lse_s[kvh * kLgRows + r] = row_lse(p, w, it.u, kvh, r, chv);
        }
        named_bar_sync(kBarP2S, kT2);
        cur_u = it.u;
      }
      acc = 0.f;
    }
    const float* x = slices + (size_t)slot * (kRC * kKeysP2) + tid;
    const float* ls = S.lse_s + it.kvh * kLgRows + it.rc * kRC;
    const int rows_c = min(kRC, it.rows - it.rc * kRC);
    if (it.rc == 0) acc_h = 0.f;  // this KV head's rows
    int r = 0;
    for (; r + 8 <= rows_c; r += 8) {
#pragma unroll
      for (int q = 0; q < 8; ++q) acc_h += fast_exp2(fmaf(x[(r + q) * kKeysP2], scale, -ls[r + q]));
    }
    for (; r < rows_c; ++r) acc_h += fast_exp2(fmaf(x[r * kKeysP2], scale, -ls[r]));
    __syncwarp();
    if (lane == 0) mbar_arrive(&c->empty[slot]);  // this warp is done with the slot and its record
    if ((it.rc + 1) * kRC < it.rows) continue;  // the head's next row chunk follows
    acc += acc_h;
    if (p.head_sets) {
      // the KV group's own I_v: its g query heads and the elite rows
      const int key = it.kb * kKeysP2 + tid;
      if (key < it.n_v)
        w.ivh[((size_t)it.l * p.h_kv + it.kvh) * p.total_visual + it.vis0 + key] = acc_h / (float)(p.g * it.n_tk);
    }
    if (it.kvh == p.h_kv - 1) {
      const int key = it.kb * kKeysP2 + tid;
      const float v = acc / (float)(p.h_q * it.n_tk);
      const bool ok = key < it.n_v;
      if (ok) w.iv[(size_t)it.l * p.total_visual + it.vis0 + key] = v;
      P2Hand h;
      h.u = it.u;
      h.kb = it.kb;
      h.n = min(kKeysP2, it.n_v - it.kb * kKeysP2);
      h.end = 0;
      h.nb = (it.n_v + kKeysP2 - 1) / kKeysP2;
      if (!p2_hand_off(c, n_hand, h, 1, &v, &tid, &ok)) {
        if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
        return;
      }
    }
  }
  P2Hand h;
  h.u = h.kb = h.n = h.nb = 0;
  h.end = 1;
  const bool no = false;
  const float zero = 0.f;
  if (!p2_hand_off(c, n_hand, h, 1, &zero, &tid, &no) && tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
}

__global__ void __launch_bounds__(kT2p, 2) stream_p2_kernel(const __grid_constant__ SArgs a) {
  AIRCACHE_KT(2);
  const Dev& p = a.p;
  const Ws& w = a.w;
  extern __shared__ unsigned char smem_raw[];
  __shared__ ff red[3 * (kMomT / 32)];
  __shared__ float redf[2 * (kMomT / 32)];
  P2Smem S;
  S.sm = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
  S.c = reinterpret_cast<Ctl2p*>(S.sm + kP2CtlOff);
  S.lse_s = reinterpret_cast<float*>(S.sm + kP2CtlOff + sizeof(Ctl2p));
  S.red = red;
  S.redf = redf;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < kP2Stages; ++i) {
      mbar_init(&S.c->full[i], 1);
      mbar_init(&S.c->empty[i], kT2 / 32);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.c->hfull[i], kT2);
      mbar_init(&S.c->hempty[i], kMomT);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // pass 1's partials and logits
  if (*(volatile int32_t*)w.error != 0) return;
  const int n_total = __ldcg(&w.list_n[0]), n_multi = __ldcg(&w.list_n[2]);
  const int LB = p.L * p.B;
  // units with stored logits, partitioned by weight (blocks x row chunks)
  const unsigned long long pack = __ldcg(w.p2pack);
  const int n_single = (int)(pack >> 32);
  const unsigned long long W = pack & 0xffffffffULL;
  if (n_total < 0 || n_total > LB || n_multi < 0 || n_multi > n_total || n_single != n_total - n_multi) {
    if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
    return;
  }
  // units without stored logits: row LSEs for pass 2k
  for (int m = blockIdx.x; m < n_multi; m += gridDim.x) {
    const int u = __ldcg(&w.stream_list[m]);
    const int4 i0 = (u >= 0 && u < LB) ? __ldcg(&w.uinfo[2 * u]) : make_int4(0, 0, 0, 0);
    const int4 i1 = (u >= 0 && u < LB) ? __ldcg(&w.uinfo[2 * u + 1]) : make_int4(0, 0, 0, 0);
    if (!stream_unit(p, u, i0, i1)) {
      if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
      return;
    }
    const int rows = p.g * i1.y;
    const int chv = ((i0.w + kTK - 1) / kTK + kCK - 1) / kCK;
    float* lse_u = w.lse + (size_t)u * p.lse_stride;
    for (int q = tid; q < p.h_kv * rows; q += kT2p) {
      const int kvh = q / rows, r = q % rows;
      lse_u[kvh * rows_per_kv(p) + r] = row_lse(p, w, u, kvh, r, chv);
    }
  }
  if (warp > kP2Prod) {
    p2_moments(p, w, S, tid - kT2 - 32);
    return;
  }
  const unsigned long long lo = W * blockIdx.x / gridDim.x, hi = W * (blockIdx.x + 1) / gridDim.x;
  p2_single(a, S, lo, hi, n_single);
}

// ------------------------------------------------------------------ pass 2k

struct Ctl2 {
  uint64_t kfull, qfull[kNQ];
};

// Units without stored logits.  Item = (unit, key tile): for each KV head in turn the
// key tile's B fragments are loaded into registers (the buffer is refilled
// with the next head's tile at once), and the head's row chunks stream through
// a ring of query chunks with their LSEs.  Each thread sums exp2(logit - lse)
// for its four keys over every row it sees; a reduction over the lanes that
// share those keys gives the tile's final I_v.
template <int D>
__global__ void __launch_bounds__(kT2, 1) stream_p2k_kernel(const __grid_constant__ SArgs a) {
  AIRCACHE_KT(3);
  using Gm = SGeo<D>;
  constexpr int KS = Gm::kKS;
  const Dev& p = a.p;
  const Ws& w = a.w;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Ctl2* c = reinterpret_cast<Ctl2*>(sm + Gm::kCtl2Off);
  __shared__ ff red[3 * (kT2 / 32)];
  __shared__ float redf[2 * (kT2 / 32)];
  __shared__ float shs[4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, c4 = lane & 3;
  const uint32_t sbase = smem_u32(sm);
  if (tid == 0) {
    mbar_init(&c->kfull, 1);
    for (int i = 0; i < kNQ; ++i) mbar_init(&c->qfull[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // pass 2's row LSEs
  if (*(volatile int32_t*)w.error != 0) return;
  const int TVmax = (p.max_visual + kTK - 1) / kTK;
  const long long total = (long long)__ldcg(&w.list_n[2]) * TVmax;
  const int kr = 16 * warp + (lane & 7) + 8 * (lane >> 4);
  const int kc = (lane >> 3) & 1;
  const int qr = lane & 15, qc = lane >> 4;
  const float scale = p.scale_log2;
  const long long TV = p.total_visual;
  uint32_t kph = 0;  // key-tile barrier phase
  long long qn = 0;  // query chunks consumed (ring position)
  if (tid == 0) fence_proxy_async_global();  // LSEs were written by the previous kernel's generic stores
  for (long long item = blockIdx.x; item < total; item += gridDim.x) {
    const int li = (int)(item / TVmax), tile = (int)(item % TVmax);
    const int u = __ldcg(&w.stream_list[li]);  // slots [0, list_n[2]): the units without stored logits
    const int4 i0 = (u >= 0 && u < p.L * p.B) ? __ldcg(&w.uinfo[2 * u]) : make_int4(0, 0, 0, 0);
    const int4 i1 = (u >= 0 && u < p.L * p.B) ? __ldcg(&w.uinfo[2 * u + 1]) : make_int4(0, 0, 0, 0);
    if (!stream_unit(p, u, i0, i1)) {
      if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_BOUNDS);
      return;
    }
    const int n_v = i0.w, n_tk = i1.y, rows = p.g * n_tk;
    const int tv = (n_v + kTK - 1) / kTK;
    if (tile >= tv) continue;  // a tile past this unit's keys (same verdict in every thread)
    const int n_rc = (rows + kRC - 1) / kRC;
    const int steps = p.h_kv * n_rc;  // (KV head, row chunk) pairs, head-major
    const int l = u / p.B;
    const int klim = min(kTK, n_v - tile * kTK);
    auto issue_k = [&](int kvh) {
      fence_proxy_async_smem();  // the buffer's previous contents were read by ldmatrix
      mbar_arrive_expect_tx(&c->kfull, (uint32_t)Gm::kKBytes);
#pragma unroll
      for (int sl = 0; sl < Gm::kNH; ++sl) {
        tma_load_4d(sbase + sl * Gm::kKSlab, &a.kmap, sl * 64, kvh, i0.x + tile * kTK, l, &c->kfull);
      }
    };
    auto issue_q = [&](int step, long long pos) {
      const int kvh = step / n_rc, rc = step % n_rc;
      const int slot = (int)(pos % kNQ);
      const uint32_t qdst = sbase + (uint32_t)(Gm::kKBytes + slot * Gm::kQ2);
      fence_proxy_async_smem();  // the slot's previous contents were read by ldmatrix and loads
      mbar_arrive_expect_tx(&c->qfull[slot], (uint32_t)(Gm::kQBytes + kRC * 4));
#pragma unroll
      for (int sl = 0; sl < Gm::kNH; ++sl) {
        tma_load_2d(qdst + sl * Gm::kQSlab, &a.qmap, sl * 64, u * p.rows_max + kvh * rows + rc * kRC,
                    &c->qfull[slot]);
      }
      const float* lse = w.lse + (size_t)u * p.lse_stride + (size_t)kvh * rows_per_kv(p) + rc * kRC;
      bulk_g2s(sm + Gm::kKBytes + slot * Gm::kQ2 + Gm::kQBytes, lse, kRC * 4, &c->qfull[slot]);
    };
    if (tid == 0) {
      issue_k(0);
      for (int st = 0; st < min(steps, kNQ); ++st) issue_q(st, qn + st);
    }
    float accK[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    int step = 0;
    for (int kvh = 0; kvh < p.h_kv; ++kvh) {
      float accH[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // this KV head's rows
      if (!mbar_wait(&c->kfull, kph, 4 * kWaitCycles)) {
        if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
        return;
      }
      kph ^= 1;
      uint32_t kf[KS][4];
      __syncwarp();  // ldmatrix / mma are warp-collective: the whole warp, converged
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const int slab = kk >> 2, c0 = (kk & 3) * 2;
        ldsm_x4(kf[kk], swz(sbase + slab * Gm::kKSlab, kr, c0 + kc));
      }
      __syncthreads();  // the key buffer is free again
      if (tid == 0 && kvh + 1 < p.h_kv) issue_k(kvh + 1);
      for (int rc = 0; rc < n_rc; ++rc, ++qn, ++step) {
        const int slot = (int)(qn % kNQ);
        if (!mbar_wait(&c->qfull[slot], (uint32_t)((qn / kNQ) & 1), 4 * kWaitCycles)) {
          if (tid == 0) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
          return;
        }
        const int rows_c = min(kRC, rows - rc * kRC);
        const uint32_t qs = sbase + (uint32_t)(Gm::kKBytes + slot * Gm::kQ2);
        const float* ls = reinterpret_cast<const float*>(sm + Gm::kKBytes + slot * Gm::kQ2 + Gm::kQBytes);
        float acc[2][2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
        const int mts = rows_c > 16 ? 2 : 1;
        __syncwarp();  // ldmatrix / mma are warp-collective: the whole warp, converged
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int slab = kk >> 2, c0 = (kk & 3) * 2;
          uint32_t qa[4];
          ldsm_x4(qa, swz(qs + slab * Gm::kQSlab, qr, c0 + qc));
          mma_bf16_16816(acc[0][0], qa, kf[kk][0], kf[kk][1]);
          mma_bf16_16816(acc[0][1], qa, kf[kk][2], kf[kk][3]);
          if (mts > 1) {
            ldsm_x4(qa, swz(qs + slab * Gm::kQSlab, 16 + qr, c0 + qc));
            mma_bf16_16816(acc[1][0], qa, kf[kk][0], kf[kk][1]);
            mma_bf16_16816(acc[1][1], qa, kf[kk][2], kf[kk][3]);
          }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int row = 16 * mt + g4 + 8 * hh;
            if (mt < mts && row < rows_c) {
              const float lse = ls[row];
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) accH[nt][e] += fast_exp2(fmaf(acc[mt][nt][2 * hh + e], scale, -lse));
            }
          }
        __syncthreads();  // every thread is done with the slot
        if (tid == 0 && step + kNQ < steps) issue_q(step + kNQ, qn + kNQ);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          accK[nt][e] += accH[nt][e];
          if (p.head_sets) {
            // the KV group's own I_v (lanes with the same c4 hold the same keys)
            float v = accH[nt][e];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            const int key = 16 * warp + 8 * nt + 2 * c4 + e;
            if (g4 == 0 && key < klim)
              w.ivh[((size_t)l * p.h_kv + kvh) * TV + i0.y + (long long)tile * kTK + key] = v / (float)(p.g * n_tk);
          }
        }
    }
    // per key: the sum over every row (lanes with the same c4 hold the same keys)
    float* iv = w.iv + (size_t)l * TV + i0.y;
    const float denom = (float)(p.h_q * n_tk);
    float xv[4];
    bool okv[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = accK[nt][e];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        const int key = 16 * warp + 8 * nt + 2 * c4 + e;
        xv[2 * nt + e] = v / denom;
        okv[2 * nt + e] = g4 == 0 && key < klim;
        if (okv[2 * nt + e]) iv[(long long)tile * kTK + key] = xv[2 * nt + e];
      }
    // this tile's moments, for the unit's layer statistics; shift: the mean of the
    // tile's values at keys 0, 32, 64, 96 that exist (warps 0, 2, 4, 6, lane 0)
    if ((warp & 1) == 0 && lane == 0) shs[warp >> 1] = okv[0] ? xv[0] : 0.f;
    named_bar_sync(kBarT2, kT2);
    const int nsh = min(4, (klim + 31) / 32);
    float sh = shs[0];
    for (int i = 1; i < nsh; ++i) sh += shs[i];
    sh /= (float)nsh;
    const Mom mb = block_moments<kT2, 4>(xv, okv, (float)klim, sh, red, redf, tid, kBarT2);
    if (warp == 0) {
      if (tid == 0) mom_store(w.mom + ((size_t)u * p.mom_slots + tile) * kMomWords, mb);
      unit_record_done(p, w, u, tv, lane);
    }
  }
}

template <int D>
cudaError_t launch_p1_t(const Dev& p, const StreamMaps& m, const Ws& w, int sms, cudaStream_t s) {
  using Gm = SGeo<D>;
  SArgs a;
  std::memset(&a, 0, sizeof a);
  a.kmap2 = m.kmap2;
  a.qmap = m.qmap;
  a.kelmap = m.kelmap;
  a.p = p;
  a.w = w;
  const int smem = Gm::kCtlOff + (int)sizeof(Ctl1) + 1024;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(stream_p1_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(stream_p1_kernel<D>, dim3(sms), dim3(kThreads1), smem, s, a);
}

template <int D>
cudaError_t launch_p2k_t(const Dev& p, const StreamMaps& m, const Ws& w, int sms, cudaStream_t s) {
  using Gm = SGeo<D>;
  SArgs a;
  std::memset(&a, 0, sizeof a);
  a.kmap = m.kmap;
  a.qmap = m.qmap;
  a.p = p;
  a.w = w;
  const int smem = Gm::kCtl2Off + (int)sizeof(Ctl2) + 1024;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(stream_p2k_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(stream_p2k_kernel<D>, dim3(2 * sms), dim3(kT2), smem, s, a);
}

}  // namespace

bool stream_eligible(const Dev& p, const LayerPtrs& lp) {
  if (p.dtype != AIRCACHE_BF16 || (p.d != 64 && p.d != 128)) return false;
  if ((p.max_visual + kKeysP2 - 1) / kKeysP2 > 65535 || p.h_kv * kLgRows * (int)sizeof(float) > 16 * 1024) return false;
  const long long U = (long long)p.L * p.B;
  if (U * p.rows_max + kRC > INT32_MAX || U * p.h_kv * p.max_elite + kTK > INT32_MAX) {
    return false;  // TMA row coordinates are 32-bit
  }
  CUtensorMap m;
  return encode_keys<__nv_bfloat16>(&m, p, lp, kTK);
}

bool encode_stream_maps(const Dev& p, const LayerPtrs& lp, const Ws& w, StreamMaps* m) {
  const long long U = (long long)p.L * p.B;
  return w.lg && w.part_s && encode_keys<__nv_bfloat16>(&m->kmap, p, lp, kTK) &&
         encode_keys<__nv_bfloat16>(&m->kmap2, p, lp, 2 * kTK) &&
         encode_rows<__nv_bfloat16>(&m->qmap, w.qel, p.d, U * p.rows_max, kRC) &&
         encode_rows<__nv_bfloat16>(&m->kelmap, w.kel, p.d, U * p.h_kv * p.max_elite, kTK) &&
         encode_logits(&m->lgmap, w.lg, (p.total_visual + 4LL * p.B + 7) / 4 * 4, (long long)p.L * p.h_kv * kLgRows,
                       kKeysP2, kP2Box);
}

cudaError_t launch_stream_p1(const Dev& p, const StreamMaps& m, const Ws& w, int sms, cudaStream_t s) {
  return p.d == 128 ? launch_p1_t<128>(p, m, w, sms, s) : launch_p1_t<64>(p, m, w, sms, s);
}

cudaError_t launch_stream_p2(const Dev& p, const StreamMaps& m, const Ws& w, int sms, cudaStream_t s) {
  SArgs a;
  std::memset(&a, 0, sizeof a);
  a.lgmap = m.lgmap;
  a.p = p;
  a.w = w;
  const int smem = kP2CtlOff + (int)sizeof(Ctl2p) + (int)sizeof(float) * p.h_kv * kLgRows + 128;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(stream_p2_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(stream_p2_kernel, dim3(2 * sms), dim3(kT2p), smem, s, a);
}

cudaError_t launch_stream_p2k(const Dev& p, const StreamMaps& m, const Ws& w, int sms, cudaStream_t s) {
  return p.d == 128 ? launch_p2k_t<128>(p, m, w, sms, s) : launch_p2k_t<64>(p, m, w, sms, s);
}

}  // namespace aircache

AIRCACHE_TIMELINE_EXPORT(stream)
