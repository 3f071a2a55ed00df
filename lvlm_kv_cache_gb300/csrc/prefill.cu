// Causal prefill attention with the AirCache scoring inputs fused in (AirCache
// notes, "Limitations and outlook": the method adds its scoring to the prefill;
// here the prefill's own logits feed it, so the scoring needs no second pass
// over the keys).
//
// Attention.  One CTA per (layer, request, query head, 128-row query tile), the
// heaviest tiles first; D = 128, bf16, causal within each packed request.  A
// producer warp brings the query tile once and the key and value tiles of the
// request's key tiles 0..t through two-stage TMA rings (128-byte swizzle).  One
// thread issues the tensor-core MMAs: S_j = Q K_j^T into one of two TMEM
// buffers, and O += P_j V_j into a TMEM accumulator (V read MN-major, so no
// transposed copy is made); S_{j+1} is issued before P_j V_j so that the
// softmax of one tile overlaps the MMAs of the next.  Four softmax warps own
// one query row per thread (the TMEM lane of the row): a row maximum, then
// P = exp2(S log2(e)/sqrt(D) - m) rounded to bf16 into a swizzled shared
// tile for the next MMA, with m a reference that moves only when the row's
// maximum grows by more than 2^8 (then O and the row sum are rescaled in TMEM
// first).  The epilogue divides O by the row sum and writes bf16 rows.
//
// Scoring (AirCache notes, "Key design 1").  A query row that is one of its
// request's elite text positions (the elite kernel ran first) owns, in its
// thread, its logits against every visual key: while the visual key tiles
// pass, it stores the raw logits to the stored-logit buffer of the streaming
// path (when its unit has at most 64 query rows per KV head), and it sums the
// probabilities its softmax forms for the visual keys, against the row's
// reference and rescaled with the row sum: (reference, that sum) is the row's
// visual partial, a (max, sum of exp2) pair like the scoring kernels' own.  A small kernel adds each elite row's partial over the elite
// text keys (the scoring softmax has no causal mask, so these are not the
// prefill's own), and the streaming pass 2 / 2k, budget, selection and
// compaction follow unchanged.
#include <cstring>

#include "internal.cuh"
#include "ptx.cuh"
#include "tmap.cuh"
#include "umma.cuh"

namespace aircache {
namespace {

constexpr int kQT = 128;           // query rows per CTA (= TMEM lanes)
constexpr int kKT = 128;           // keys per tile
constexpr int kSlabB = 128 * 128;  // one [128 rows][64 bf16] slab: 16 KB
constexpr int kTileB = 2 * kSlabB; // a [128][128] bf16 tile: 32 KB
constexpr int kPThreads = 192;     // producer warp, MMA warp, four softmax warps
constexpr float kRescaleLog2 = 8.f;
constexpr int kOffQ = 0;
constexpr int kOffK = kTileB;            // two stages
constexpr int kOffV = kOffK + 2 * kTileB;  // two stages
constexpr int kOffP = kOffV + 2 * kTileB;
constexpr int kOffCtl = kOffP + kTileB;
constexpr uint32_t kTmemCols = 512;      // S buffers at 0 and 128, O at 256
constexpr uint32_t kTmemO = 256;

struct PCtl {
  uint64_t qfull, kfull[2], kempty[2], vfull[2], vempty[2], sfull[2], sempty[2], pfull, pfree, ofull;
  uint32_t tmem;
};

struct OutPtrs {
  void* o[AIRCACHE_MAX_LAYERS];
};

struct PArgs {
  CUtensorMap qmap;  // every layer's queries (D, H_q, tokens, layers), box (64, 1, 128, 1)
  CUtensorMap kmap;  // keys (D, H_kv, tokens, layers), box (64, 1, 128, 1)
  CUtensorMap vmap;  // values, the same
  Dev p;
  Ws w;
  int score;         // 1: the scoring inputs of the elite rows as well
  int n_qt;          // query tiles of the longest request
  int64_t o_stride_tok, o_stride_head;  // output strides (elements)
  OutPtrs out;
};

static_assert(sizeof(PArgs) <= 4096, "kernel parameter space");

// Row partial index of the streaming path (as the scoring kernels lay it out).
__device__ __forceinline__ size_t part_idx(const Dev& p, int u, int kvh, int row, int chunk) {
  return (((size_t)u * p.h_kv + kvh) * (p.rc_max * kRowChunk) + row) * p.chn + chunk;
}

__device__ __forceinline__ long long lg_col(long long vis0, int b) { return (vis0 + 3) / 4 * 4 + 4LL * b; }
__device__ __forceinline__ long long lg_width(const Dev& p) { return (p.total_visual + 4LL * p.B + 7) / 4 * 4; }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(const __grid_constant__ PArgs a) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  PCtl* c = reinterpret_cast<PCtl*>(sm + kOffCtl);
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the tile of this CTA: heaviest (largest t) first
  const long long per = (long long)p.L * p.B * p.h_q;
  const int t = a.n_qt - 1 - (int)(blockIdx.x / per);
  const long long rest = blockIdx.x % per;
  const int h = (int)(rest % p.h_q), b = (int)((rest / p.h_q) % p.B), l = (int)(rest / ((long long)p.h_q * p.B));
  const int kvh = h / p.g, hh = h % p.g;
  pdl_trigger();
  pdl_wait();  // the elite lists (scoring) and nothing else: the inputs are the caller's
  if (*(volatile int32_t*)w.error != 0) return;
  const int64_t s0 = p.cu_seqlens[b], s1 = p.cu_seqlens[b + 1];
  const int64_t q0 = s0 + (int64_t)t * kQT;
  if (q0 >= s1) return;  // the request has fewer tiles
  const int nkt = t + 1;
  if (threadIdx.x == 0) {
    mbar_init(&c->qfull, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->kfull[i], 1);
      mbar_init(&c->kempty[i], 1);
      mbar_init(&c->vfull[i], 1);
      mbar_init(&c->vempty[i], 1);
      mbar_init(&c->sfull[i], 1);
      mbar_init(&c->sempty[i], 4);
    }
    mbar_init(&c->pfull, 4);
    mbar_init(&c->pfree, 1);
    mbar_init(&c->ofull, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(&c->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem;

  if (warp == 0) {
    if (lane == 0) {
      // producer
      mbar_arrive_expect_tx(&c->qfull, (uint32_t)kTileB);
      for (int sl = 0; sl < 2; ++sl)
        tma_load_4d(sbase + kOffQ + sl * kSlabB, &a.qmap, sl * 64, h, (int)q0, l, &c->qfull);
      bool ok = true;
      for (int j = 0; j < nkt && ok; ++j) {
        const int st = j & 1;
        const uint32_t par = (uint32_t)(((j >> 1) & 1) ^ 1);
        const int key0 = (int)(s0 + (int64_t)j * kKT);
        if (!mbar_wait(&c->kempty[st], par)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&c->kfull[st], (uint32_t)kTileB);
        for (int sl = 0; sl < 2; ++sl)
          tma_load_4d(sbase + kOffK + st * kTileB + sl * kSlabB, &a.kmap, sl * 64, kvh, key0, l, &c->kfull[st]);
        if (!mbar_wait(&c->vempty[st], par)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&c->vfull[st], (uint32_t)kTileB);
        for (int sl = 0; sl < 2; ++sl)
          tma_load_4d(sbase + kOffV + st * kTileB + sl * kSlabB, &a.vmap, sl * 64, kvh, key0, l, &c->vfull[st]);
      }
      if (!ok) set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issue: S_j = Q K_j^T (M = 128 queries, N = 128 keys), then
      // O += P_{j-1} V_{j-1} (M = 128 queries, N = 128 = D, K = 128 keys)
      constexpr uint32_t idS = umma_idesc_bf16(kQT, kKT);
      constexpr uint32_t idO = umma_idesc_bf16_bmn(kQT, 128);
      bool ok = mbar_wait(&c->qfull, 0);
      auto pv = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&c->pfull, (uint32_t)(j & 1), 4 * kWaitCycles)) return false;
        if (!mbar_wait(&c->vfull[st], (uint32_t)((j >> 1) & 1))) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t pa = sbase + kOffP + (kk >> 2) * kSlabB + (kk & 3) * 32;
          const uint32_t vb = sbase + kOffV + st * kTileB + kk * 16 * 128;
          umma_bf16(tmem + kTmemO, umma_desc_sw128(pa), umma_desc_sw128_mn(vb, kSlabB, 1024), idO,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&c->vempty[st]);
        umma_commit(&c->pfree);
        return true;
      };
      for (int j = 0; ok && j < nkt; ++j) {
        const int st = j & 1;
        ok = mbar_wait(&c->kfull[st], (uint32_t)((j >> 1) & 1)) &&
             mbar_wait(&c->sempty[st], (uint32_t)(((j >> 1) & 1) ^ 1), 4 * kWaitCycles);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t qa = sbase + kOffQ + (kk >> 2) * kSlabB + (kk & 3) * 32;
          const uint32_t kb = sbase + kOffK + st * kTileB + (kk >> 2) * kSlabB + (kk & 3) * 32;
          umma_bf16(tmem + (uint32_t)(st * kKT), umma_desc_sw128(qa), umma_desc_sw128(kb), idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&c->kempty[st]);
        umma_commit(&c->sfull[st]);
        if (j > 0) ok = pv(j - 1);
      }
      if (ok) ok = pv(nkt - 1);
      if (ok) umma_commit(&c->ofull);
      else set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
    }
  } else {
    // softmax warps: thread = query row r (its TMEM lane)
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const int64_t qrow = q0 + r;
    const bool valid = qrow < s1;
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    const float scale = p.scale_log2;
    const uint32_t prow = sbase + kOffP + (uint32_t)r * 128;
    // scoring role of this row: its elite index, if it is an elite text position
    const int u = l * p.B + b;
    int e_idx = -1, n_tk = 0, n_v = 0;
    float* lgdst = nullptr;
    if (a.score && valid) {
      n_v = (int)(p.cu_visual[b + 1] - p.cu_visual[b]);
      const int64_t j_text = qrow - s0 - n_v;  // visual-first prompts
      n_tk = __ldcg(&w.n_tk[u]);
      if (j_text >= 0 && n_tk >= 1 && n_tk <= p.max_elite) {
        const int32_t* el = w.elite + (size_t)u * p.elite_stride;
        for (int e = 0; e < n_tk; ++e)
          if (__ldcg(el + e) == (int32_t)j_text) e_idx = e;
      }
      if (e_idx >= 0 && p.g * n_tk <= kLgRows) {
        const long long LS = lg_width(p);
        lgdst = w.lg + (((size_t)l * p.h_kv + kvh) * kLgRows + (size_t)hh * n_tk + e_idx) * LS +
                lg_col(p.cu_visual[b], b);
      }
    }
    float s_vis = 0.f;  // a scoring row's sum over the visual keys, against m_ref (base 2)
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int st = j & 1;
      if (!mbar_wait(&c->sfull[st], (uint32_t)((j >> 1) & 1), 4 * kWaitCycles)) {
        ok = false;
        break;
      }
      __syncwarp();
      tc_fence_after();
      const int64_t k0 = s0 + (int64_t)j * kKT;
      const uint32_t tS = tl + (uint32_t)(st * kKT);
      // pass A: the row's maximum over its causal keys; the scoring rows also
      // store their visual logits and keep their visual partial
      float mx = -INFINITY;
      for (int c4 = 0; c4 < 4; ++c4) {
        float v[32];
        tmem_ld32(tS + 32 * c4, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (k0 + 32 * c4 + i <= qrow) mx = fmaxf(mx, v[i]);
        if (lgdst && k0 + 32 * c4 < s0 + n_v) {
          // a scoring row stores its raw visual logits (16-byte stores; the
          // row's columns start 16-byte aligned)
          const int kv0 = (int)(k0 - s0) + 32 * c4;  // visual index of v[0]
          if (kv0 + 32 <= n_v) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<float4*>(lgdst + kv0 + 4 * i) =
                  make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < n_v - kv0) lgdst[kv0 + i] = v[i];
          }
        }
      }
      const float mxs = mx * scale;
      // P_j goes where P_{j-1} was: wait for that MMA (which also leaves O stable)
      if (j > 0 && !mbar_wait(&c->pfree, (uint32_t)((j - 1) & 1), 4 * kWaitCycles)) {
        ok = false;
        break;
      }
      if (mxs > m_ref + kRescaleLog2 || m_ref == -INFINITY) {
        const float m_new = fmaxf(mxs, m_ref);
        if (j > 0 && m_ref != -INFINITY) {
          const float f = fast_exp2(m_ref - m_new);
          l_sum *= f;
          s_vis *= f;
          tc_fence_after();
          for (int c4 = 0; c4 < 4; ++c4) {
            float o[32];
            tmem_ld32(tl + kTmemO + 32 * c4, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tmem_st32(tl + kTmemO + 32 * c4, o);
          }
          tmem_wait_st();
        }
        m_ref = m_new;
      }
      // pass B: probabilities, the row sum, and the bf16 P row (swizzled); a
      // scoring row also sums its visual keys' probabilities (the same values,
      // against the same reference, rescaled with the row sum)
      const float neg = m_ref == -INFINITY ? 0.f : -m_ref;
      for (int c4 = 0; c4 < 4; ++c4) {
        float v[32];
        tmem_ld32(tS + 32 * c4, v);
        tmem_wait_ld();
        float vis = 0.f;
        const int64_t kvis = s0 + n_v - (k0 + 32 * c4);  // keys of this chunk below it are visual
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const bool in = k0 + 32 * c4 + i <= qrow && m_ref != -INFINITY;
          v[i] = in ? fast_exp2(fmaf(v[i], scale, neg)) : 0.f;
          l_sum += v[i];
          if (i < kvis) vis += v[i];
        }
        if (e_idx >= 0) s_vis += vis;
        // keys 32 c4 .. 32 c4 + 31: slab c4 / 2, 16-byte chunks 4 (c4 % 2) .. + 3
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = 4 * (c4 & 1) + q;
          const uint32_t addr = prow + (uint32_t)((c4 >> 1) * kSlabB) + (uint32_t)((chunk ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr),
                       "r"(pack_bf16(v[8 * q], v[8 * q + 1])), "r"(pack_bf16(v[8 * q + 2], v[8 * q + 3])),
                       "r"(pack_bf16(v[8 * q + 4], v[8 * q + 5])), "r"(pack_bf16(v[8 * q + 6], v[8 * q + 7]))
                       : "memory");
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();  // the P tile is read by the tensor cores next
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&c->sempty[st]);
        mbar_arrive(&c->pfull);
      }
    }
    if (ok && mbar_wait(&c->ofull, 0, 4 * kWaitCycles)) {
      __syncwarp();
      tc_fence_after();
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out.o[l]) + qrow * a.o_stride_tok +
                            (int64_t)h * a.o_stride_head;
      for (int c4 = 0; c4 < 4; ++c4) {
        float o[32];
        tmem_ld32(tl + kTmemO + 32 * c4, o);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 pk;
            pk.x = pack_bf16(o[8 * q] * inv, o[8 * q + 1] * inv);
            pk.y = pack_bf16(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
            pk.z = pack_bf16(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
            pk.w = pack_bf16(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
            *reinterpret_cast<uint4*>(orow + 32 * c4 + 8 * q) = pk;
          }
        }
      }
      if (e_idx >= 0) {
        // the row's visual partial in chunk 0, the other visual chunks empty
        const int chv = ((n_v + 127) / 128 + kStreamTiles - 1) / kStreamTiles;
        const int row = hh * n_tk + e_idx;
        w.part_s[part_idx(p, u, kvh, row, 0)] = make_float2(m_ref, s_vis);
        for (int ch = 1; ch < chv; ++ch) w.part_s[part_idx(p, u, kvh, row, ch)] = make_float2(-INFINITY, 0.f);
      }
    } else if (lane == 0) {
      set_error(w.error, AIRCACHE_ERR_DEVICE_TIMEOUT);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();  // every MMA and TMEM access of the CTA is done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Each elite row's partial over the elite text keys (the scoring softmax sees
// every elite text key: no causal mask), written as the streaming path's text
// chunk.  One warp per (unit, KV head, row); lanes split the head dimension.
__global__ void __launch_bounds__(256) elite_text_kernel(const __grid_constant__ PArgs a) {
  const Dev& p = a.p;
  const Ws& w = a.w;
  pdl_trigger();
  pdl_wait();  // the elite lists, query rows and keys
  if (*(volatile int32_t*)w.error != 0) return;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  const int rmax = p.g * p.max_elite;  // rows per (unit, KV head)
  const long long total = (long long)p.L * p.B * p.h_kv * rmax;
  for (long long i = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); i < total; i += warps) {
    const int row = (int)(i % rmax);
    const int kvh = (int)((i / rmax) % p.h_kv);
    const int u = (int)(i / ((long long)rmax * p.h_kv));
    const int n_tk = __ldcg(&w.n_tk[u]);
    if (n_tk < 1 || n_tk > p.max_elite || row >= p.g * n_tk) continue;
    const __nv_bfloat16* qr = reinterpret_cast<const __nv_bfloat16*>(w.qel) +
                              ((size_t)u * p.rows_max + (size_t)kvh * p.g * n_tk + row) * p.d;
    float qv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) qv[k] = __bfloat162float(qr[lane * 4 + k]);
    float m = -INFINITY, s = 0.f;
    for (int e = 0; e < n_tk; ++e) {
      const __nv_bfloat16* kr = reinterpret_cast<const __nv_bfloat16*>(w.kel) +
                                (((size_t)u * p.h_kv + kvh) * p.max_elite + e) * p.d;
      float d = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) d = fmaf(qv[k], __bfloat162float(kr[lane * 4 + k]), d);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      const float x = d * p.scale_log2;
      if (x > m) {
        s *= fast_exp2(m - x);
        m = x;
      }
      s += fast_exp2(x - m);
    }
    if (lane == 0) w.part_s[part_idx(p, u, kvh, row, p.chn - 1)] = make_float2(m, s);
  }
}

// 4-D TMA map (D, H, tokens, layers) over per-layer pointers that are evenly
// strided, box (64 elements, 1 head, 128 tokens, 1 layer), 128-byte swizzle.
bool encode_4d(CUtensorMap* m, const void* const* ptrs, int L, int d, int heads, long long tokens,
               long long stride_head, long long stride_tok) {
  auto enc = tma_encoder();
  if (!enc) return false;
  const char* b0 = reinterpret_cast<const char*>(ptrs[0]);
  const long long lstride = L > 1 ? reinterpret_cast<const char*>(ptrs[1]) - b0 : 16;
  if (lstride <= 0 || lstride % 16 != 0) return false;
  for (int l = 2; l < L; ++l)
    if (reinterpret_cast<const char*>(ptrs[l]) - b0 != (long long)l * lstride) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)tokens, (cuuint64_t)L};
  cuuint64_t strides[3] = {(cuuint64_t)stride_head * 2, (cuuint64_t)stride_tok * 2, (cuuint64_t)lstride};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)kQT, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<char*>(b0), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_eligible(const Dev& p, const LayerPtrs& lp, int64_t qa_stride_tok, int64_t qa_stride_head,
                      int64_t o_stride_tok, int64_t o_stride_head) {
  if (p.dtype != AIRCACHE_BF16 || p.d != 128 || p.n_prefix != nullptr || p.window_mode != 0 || p.head_sets)
    return false;
  if (qa_stride_head < 128 && p.h_q > 1) return false;
  if ((qa_stride_tok * 2) % 16 || (qa_stride_head * 2) % 16 || (o_stride_tok * 2) % 16 || (o_stride_head * 2) % 16)
    return false;
  CUtensorMap m;
  return encode_4d(&m, lp.q, p.L, p.d, p.h_q, p.total_tokens, qa_stride_head, qa_stride_tok) &&
         encode_4d(&m, lp.k, p.L, p.d, p.h_kv, p.total_tokens, p.kv_stride_head, p.kv_stride_tok) &&
         encode_4d(&m, lp.v, p.L, p.d, p.h_kv, p.total_tokens, p.kv_stride_head, p.kv_stride_tok);
}

cudaError_t launch_prefill(const Dev& p, const LayerPtrs& lp, const Ws& w, int64_t qa_stride_tok,
                           int64_t qa_stride_head, void* const* out, int64_t o_stride_tok, int64_t o_stride_head,
                           int max_tokens, bool score, int sms, cudaStream_t s) {
  PArgs a;
  std::memset(&a, 0, sizeof a);
  if (!encode_4d(&a.qmap, lp.q, p.L, p.d, p.h_q, p.total_tokens, qa_stride_head, qa_stride_tok) ||
      !encode_4d(&a.kmap, lp.k, p.L, p.d, p.h_kv, p.total_tokens, p.kv_stride_head, p.kv_stride_tok) ||
      !encode_4d(&a.vmap, lp.v, p.L, p.d, p.h_kv, p.total_tokens, p.kv_stride_head, p.kv_stride_tok))
    return cudaErrorInvalidValue;
  a.p = p;
  a.w = w;
  a.score = score ? 1 : 0;
  a.n_qt = (max_tokens + kQT - 1) / kQT;
  a.o_stride_tok = o_stride_tok;
  a.o_stride_head = o_stride_head;
  for (int l = 0; l < p.L; ++l) a.out.o[l] = out[l];
  const int smem = kOffCtl + (int)sizeof(PCtl) + 1024;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(prefill_kernel), smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)a.n_qt * p.L * p.B * p.h_q;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (score) {
    e = launch_pdl(elite_text_kernel, dim3(4 * sms), dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(prefill_kernel, dim3((unsigned)grid), dim3(kPThreads), smem, s, a);
}

}  // namespace aircache
