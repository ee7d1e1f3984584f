// Phase timeline of the step's kernels, compiled in only with -DQSA_TRACE
// (the separate tracing build of the library, libqsa_trace.so); in the
// product build every mark below expands to nothing.
//
// Each traced translation unit owns one table of kTraceSlots 64-bit words per
// CTA for its kernels' first kTraceCtas CTAs: %globaltimer stamps (ns) taken
// at fixed points of the CTA, and its SM id. Slots:
//   0 start (first instruction)
//   1 dependency wait released (griddepcontrol.wait returned)
//   2 main work done (the latest of the CTA's warps where they finish apart)
//   3 end (last instruction before exit)
//   4 SM id + 1 (0: no record)
//   5 attention: a piece of a split unit published (the last one)
//   6 attention: a merge of pieces done (the last one)
// Timestamps are read back by qsa_trace_read (include/qsa.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qsa {

constexpr int kTraceCtas = 4096;
constexpr int kTraceSlots = 8;

#ifdef QSA_TRACE
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned trace_smid() {
  unsigned s;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
  return s;
}
// the translation unit's table (internal linkage: one per unit, no device linking)
#define QSA_TRACE_TABLE static __device__ unsigned long long g_qsa_trace[kTraceCtas * kTraceSlots];
// thread 0 of the CTA stamps slot s (and the CTA's SM with the start)
#define QSA_MARK(s)                                                                           \
  do {                                                                                        \
    if (threadIdx.x == 0 && blockIdx.x < (unsigned)kTraceCtas) {                              \
      g_qsa_trace[blockIdx.x * kTraceSlots + (s)] = trace_now();                              \
      if ((s) == 0) g_qsa_trace[blockIdx.x * kTraceSlots + 4] = trace_smid() + 1ull;          \
    }                                                                                         \
  } while (0)
// lane 0 of every warp that gets here: the latest stamp wins
#define QSA_MARK_LAST(s)                                                                      \
  do {                                                                                        \
    if ((threadIdx.x & 31) == 0 && blockIdx.x < (unsigned)kTraceCtas)                         \
      atomicMax(&g_qsa_trace[blockIdx.x * kTraceSlots + (s)], trace_now());                   \
  } while (0)
// host side of the unit: copy its table out (n_ctas records) and/or zero it
#define QSA_TRACE_HOST(fn)                                                                    \
  cudaError_t fn(unsigned long long* host, int n_ctas, bool clear) {                          \
    if (n_ctas < 0 || n_ctas > kTraceCtas) return cudaErrorInvalidValue;                      \
    cudaError_t e = cudaSuccess;                                                              \
    if (host && n_ctas > 0)                                                                   \
      e = cudaMemcpyFromSymbol(host, g_qsa_trace, sizeof(unsigned long long) * kTraceSlots * n_ctas); \
    if (e == cudaSuccess && clear) {                                                          \
      void* p = nullptr;                                                                      \
      e = cudaGetSymbolAddress(&p, g_qsa_trace);                                              \
      if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(g_qsa_trace));                        \
      if (e == cudaSuccess) e = cudaDeviceSynchronize();                                      \
    }                                                                                         \
    return e;                                                                                 \
  }
#else
#define QSA_TRACE_TABLE
#define QSA_MARK(s) \
  do {              \
  } while (0)
#define QSA_MARK_LAST(s) \
  do {                   \
  } while (0)
#define QSA_TRACE_HOST(fn) \
  cudaError_t fn(unsigned long long*, int, bool) { return cudaErrorNotSupported; }
#endif

// per translation unit: score kernels, top-k kernels, attention kernel
cudaError_t trace_score(unsigned long long* host, int n_ctas, bool clear);
cudaError_t trace_topk(unsigned long long* host, int n_ctas, bool clear);
cudaError_t trace_attn(unsigned long long* host, int n_ctas, bool clear);

}  // namespace qsa
