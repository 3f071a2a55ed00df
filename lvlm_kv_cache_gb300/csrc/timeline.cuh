// Device timeline of a call, compiled in only with -DAIRCACHE_TIMELINE: a
// separate build of the library (libaircache_timeline.so, `bench.py
// --timeline`); the product library has none of it.  Each instrumented
// kernel's CTAs record the entry time of their first thread and the latest
// exit time of their warps (globaltimer, ns) in a table of the translation
// unit; aircache_timeline_read_<unit> copies the table to the host and
// aircache_timeline_clear_<unit> zeroes it.
#pragma once

#ifdef AIRCACHE_TIMELINE
#include <cuda_runtime.h>

namespace aircache {
namespace tl {

constexpr int kKernels = 8;   // kernel slots (see AIRCACHE_KT's callers)
constexpr int kCtas = 4096;   // CTAs recorded per kernel (flat block index)
static __device__ unsigned long long g_kt[kKernels][kCtas][2];

__device__ __forceinline__ unsigned long long now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct Guard {
  int k, c;
  __device__ explicit Guard(int kid) : k(kid) {
    c = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    if (threadIdx.x == 0 && c < kCtas) g_kt[k][c][0] = now();
  }
  __device__ ~Guard() {
    if (c < kCtas && (threadIdx.x & 31) == 0) atomicMax(&g_kt[k][c][1], now());
  }
};

}  // namespace tl
}  // namespace aircache

#define AIRCACHE_KT(kid) ::aircache::tl::Guard aircache_kt_guard_(kid)
#define AIRCACHE_TIMELINE_EXPORT(unit)                                                                \
  extern "C" __attribute__((visibility("default"))) int aircache_timeline_read_##unit(void* host) {    \
    return (int)cudaMemcpyFromSymbol(host, ::aircache::tl::g_kt, sizeof(::aircache::tl::g_kt));       \
  }                                                                                                    \
  extern "C" __attribute__((visibility("default"))) int aircache_timeline_clear_##unit() {            \
    void* p = nullptr;                                                                                 \
    cudaError_t e = cudaGetSymbolAddress(&p, ::aircache::tl::g_kt);                                   \
    if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(::aircache::tl::g_kt));                          \
    return (int)e;                                                                                     \
  }
#else
#define AIRCACHE_KT(kid)
#define AIRCACHE_TIMELINE_EXPORT(unit)
#endif
