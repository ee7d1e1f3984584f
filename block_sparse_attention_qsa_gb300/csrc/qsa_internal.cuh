// Internal declarations shared by the libqsa translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "qsa.h"

namespace qsa {

constexpr int kBlock = 4;        // tokens per micro-block
constexpr int kTopK = 512;       // selected full blocks per query
constexpr int kWidth = 2051;     // selection buffer width: 512 * 4 + 3
constexpr int kDim = 128;        // index and attention head dim
constexpr int kGroup = 8;        // query heads per KV head
constexpr int kMaxNq = 4;        // verify queries per request

// Device error kinds recorded in the workspace header.
enum DevErr : int32_t {
  kErrNone = 0, kErrQueryPos = 1, kErrPage = 2, kErrSelPos = 3, kErrDraft = 4, kErrTimeout = 5
};

// Draft-step reuse: a draft query attends over a reused selection row plus at
// most kMaxDraftGap positions after the row's own query.
constexpr int kMaxDraftGap = QSA_MAX_DRAFT_GAP;
constexpr int kDraftWidth = kWidth + kMaxDraftGap;

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets from the 256-aligned base).
//   [0, 256)           header: int32 err_kind, err_request, err_query, err_value
//   tickets            int32 [units]           arrival counters of split units
//   partials           float [grid][2][kPartFloats]  pieces of units split between CTAs
//   scores (decode)    float [B][n_q][max_blocks]
//   sel_row            int32 [B][n_q][2051 + kMaxDraftGap]  cache row (KV head 0) of each
//                      selected position (row stride 2051, or 2051 + kMaxDraftGap for draft steps)
// ---------------------------------------------------------------------------
constexpr int kPartFloats = 2 * kGroup + kGroup * kDim;  // m[8], l[8], acc[8][128]

struct WsLayout {
  size_t tickets, partials, scores, sel_row, total;
  int units, tiles, grid, cl;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Work plan of the attention kernel (shared by sizing and launch): the
// units * tiles tiles form one stream, cut into `grid` contiguous shares of
// equal length, one per CTA (stream-K); or, for few units, each unit is one
// cluster of `cl` CTAs.
struct AttnPlan {
  int units;   // batch * n_q * n_kv_heads
  int tiles;   // tiles of selected positions per unit
  int grid;    // CTAs of the stream-K form
  int cl = 0;  // > 1: the cluster form, cl CTAs (one cluster) per unit
};
AttnPlan attn_plan(const qsa_dims& d, int num_sms);
WsLayout ws_layout(const qsa_dims& d, int num_sms);

int device_sm_count();

// Host-side per-device state of a launcher (SM count, occupancy, the dynamic
// shared-memory limit set on a kernel), safe to use from several host threads.
class DeviceSlots {
 public:
  static constexpr int kMaxDevices = 64;
  // the current device's value, computed by init() on first use; a result
  // <= 0 is returned but not kept, so a failed query is retried next time
  template <typename F>
  int get(F&& init) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return init();
    std::lock_guard<std::mutex> lock(mu_);
    if (v_[dev] <= 0) v_[dev] = init();
    return v_[dev];
  }
  // raises kern's dynamic shared-memory limit on the current device to at
  // least `bytes` (never lowers it, so concurrent callers cannot undo each other)
  template <typename K>
  cudaError_t raise_smem(K kern, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices)
      return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    std::lock_guard<std::mutex> lock(mu_);
    if ((size_t)v_[dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) v_[dev] = (int)bytes;
    return e;
  }

 private:
  std::mutex mu_;
  int v_[kMaxDevices] = {};
};

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void record_error(int32_t* hdr, int32_t kind, int32_t r, int32_t j,
                                             int32_t value) {
  if (atomicCAS(hdr, 0, kind) == 0) {
    hdr[1] = r;
    hdr[2] = j;
    hdr[3] = value;
  }
}

__device__ __forceinline__ int n_full_of(int p) { return (p + 1) >> 2; }

// thread-block clusters: rank, size, the hardware barrier (release / acquire),
// and loads from / stores to another CTA's shared memory (distributed shared memory)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the two halves of a cluster barrier, for a wait placed long after the arrival
// (e.g. arrive at the start, wait before the first access to another CTA's
// shared memory, which must not come before every CTA of the cluster started)
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// address of `p` (this CTA's shared memory) in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ uint32_t ld_peer(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Order-preserving 32-bit key of a score: a larger score has a larger key;
// -0.0 maps like +0.0 and NaN below every number. The top 11 bits are the
// selector's first radix digit.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
constexpr int kHistBins = 2048;  // first radix digit: top 11 key bits

// ---------------------------------------------------------------------------
// host-side launch helper: cudaLaunchKernelEx with optional PDL attribute
// ---------------------------------------------------------------------------
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Where the compressed keys live: contiguous [B][max_blocks][H][128] (table
// null) or in the KV cache's pages, [num_pages][page_size / 4][H][128], found
// through the request's page table (block b of request r: page
// table[r][b >> bpp_shift], slot b & ((1 << bpp_shift) - 1)).
struct KcPages {
  const int32_t* table;  // [B][max_pages], or null: contiguous
  int max_pages, num_pages, bpp_shift;
};

// ---------------------------------------------------------------------------
// launchers implemented in the kernel translation units
// ---------------------------------------------------------------------------
cudaError_t launch_compress(const qsa_dims& d, const __nv_bfloat16* idx_keys, const int32_t* q_pos,
                            const int32_t* block_lo, __nv_bfloat16* kc, int32_t* err,
                            cudaStream_t s, const int32_t* page_table = nullptr);
cudaError_t launch_score(const qsa_dims& d, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                         const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s, bool pdl,
                         const int32_t* page_table = nullptr);
// page_table / sel_row (optional, inside qsa_decode): also write each selected
// position's cache row for KV head 0, so attention skips the page lookup
cudaError_t launch_topk(const qsa_dims& d, const float* scores, const int32_t* q_pos,
                        int32_t* sel_blk, int32_t* sel_pos, int32_t* err, const int32_t* page_table,
                        int32_t* sel_row, cudaStream_t s, bool pdl);
// many queries per request (a prefill chunk) against the request's blocks
// withhold_first_copy: the failure-detection test (qsa_test_chunk_timeout)
cudaError_t launch_score_chunk(const qsa_dims& d, int n_chunk, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                               const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s,
                               bool withhold_first_copy = false);
// draft step: reused selection rows plus the positions since -> cache rows
cudaError_t launch_draft_resolve(const qsa_dims& d, const int32_t* sel_pos, const int32_t* sel_q_pos, int n_sel,
                                 const int32_t* src, const int32_t* q_pos, const int32_t* page_table,
                                 int32_t* sel_row, int32_t* err, cudaStream_t s);
// selected positions -> cache rows (KV head 0) with all index checks
cudaError_t launch_resolve(const qsa_dims& d, const int32_t* sel_pos, const int32_t* q_pos,
                           const int32_t* page_table, int32_t* sel_row, int32_t* err, cudaStream_t s);
cudaError_t launch_attn(const qsa_dims& d, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* sel_row, void* out,
                        int32_t* tickets, float* partials, const AttnPlan& plan, cudaStream_t s, bool pdl);

}  // namespace qsa
