// Sparse attention for callers that cannot allocate device memory.
//
// qsa_sparse_attn keeps its split-KV scratch (arrival tickets and per-split
// softmax partials) in a caller-provided workspace. Some callers cannot make
// that allocation: code that runs where cudaMalloc is forbidden or unsafe
// (inside a custom allocator's own callbacks, in a process whose memory pool
// is fixed up front, in plugins that are handed tensors but no allocator).
// For them qsa_sparse_attn_noalloc uses a scratch array that lives in this
// library's own device image instead: a file-scope __device__ array of
// kScratchBytes that every GPU which loads the library holds until the
// process exits.
#include <mutex>

#include "qsa_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr size_t kHeaderBytes = 256;                // device error record

// [header][tickets, 256-aligned][split partials]
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

// Device addresses of g_attn_scratch, one per device, found once. In host
// code the name g_attn_scratch is only a host-side stand-in for the symbol,
// never a device address, so kernels receive the looked-up address instead.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

qsa_status scratch_on_current_device(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return QSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) return QSA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return QSA_OK;
}

}  // namespace

extern "C" qsa_status qsa_sparse_attn_noalloc(const qsa_dims* dims, const void* q, const void* k_cache,
                                              const void* v_cache, const float* k_scale,
                                              const float* v_scale, const int32_t* page_table,
                                              const int32_t* sel_pos, const int32_t* q_pos, void* out,
                                              void* stream) {
  size_t unused = 0;
  const qsa_status st = qsa_workspace_size(dims, &unused);  // validates the geometry
  if (st != QSA_OK) return st;
  if (!q || !k_cache || !v_cache || !page_table || !sel_pos || !q_pos || !out) return QSA_ERR_INVALID_ARG;
  if (dims->kv_dtype == QSA_KV_FP8_E4M3 && (!k_scale || !v_scale)) return QSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) & 15u) || (reinterpret_cast<uintptr_t>(v_cache) & 15u) ||
      (reinterpret_cast<uintptr_t>(q) & 3u))
    return QSA_ERR_INVALID_ARG;

  // The usual split plan, with fewer splits if its partials would not fit.
  qsa::AttnPlan plan = qsa::attn_plan(*dims, qsa::device_sm_count());
  const size_t ticket_bytes = qsa::align_up((size_t)plan.units * sizeof(int32_t), 256);
  const size_t part_bytes = (size_t)qsa::kPartFloats * sizeof(float);
  if (kHeaderBytes + ticket_bytes >= kScratchBytes) return QSA_ERR_WORKSPACE;
  const size_t room = kScratchBytes - kHeaderBytes - ticket_bytes;
  const size_t max_split = room / (part_bytes * (size_t)plan.units);
  if (max_split < 1) return QSA_ERR_WORKSPACE;  // even one split per unit is too large
  if ((size_t)plan.nsplit > max_split) {
    const int covered = plan.nsplit * plan.tiles_per_split;  // tiles the plan spans
    plan.nsplit = (int)max_split;
    plan.tiles_per_split = (covered + plan.nsplit - 1) / plan.nsplit;
  }

  void* scratch = nullptr;
  const qsa_status ss = scratch_on_current_device(&scratch);
  if (ss != QSA_OK) return ss;
  unsigned char* base = static_cast<unsigned char*>(scratch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error record and the arrival tickets must start at zero every call
  if (cudaMemsetAsync(base, 0, kHeaderBytes + ticket_bytes, s) != cudaSuccess) return QSA_ERR_CUDA;
  const cudaError_t e = qsa::launch_attn(
      *dims, q, k_cache, v_cache, k_scale, v_scale, page_table, sel_pos, q_pos, out,
      reinterpret_cast<int32_t*>(base), reinterpret_cast<int32_t*>(base + kHeaderBytes),
      reinterpret_cast<float*>(base + kHeaderBytes + ticket_bytes), plan, s, false);
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
