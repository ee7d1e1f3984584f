// Sparse attention for callers that cannot allocate device memory.
//
// qsa_sparse_attn keeps its scratch (the resolved cache rows, arrival tickets
// and the softmax partials of units split between CTAs) in a caller-provided
// workspace. Some callers cannot make
// that allocation: code that runs where cudaMalloc is forbidden or unsafe
// (inside a custom allocator's own callbacks, in a process whose memory pool
// is fixed up front, in plugins that are handed tensors but no allocator).
// For them qsa_sparse_attn_noalloc uses a scratch array that lives in this
// library's own device image instead: a file-scope __device__ array of
// kScratchBytes that every GPU which loads the library holds until the
// process exits.
#include <initializer_list>

#include "qsa_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr size_t kHeaderBytes = 256;                 // device error record

// [header][tickets][cache rows][partials], each part 256-aligned
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

// Device address of g_attn_scratch on the current device. In host code the
// name g_attn_scratch is only a host-side stand-in for the symbol, never a
// device address, so kernels receive the looked-up address instead. It is
// looked up on every call (a query of the runtime, no stream work): a device
// reset reloads the array, possibly at another address, and a cached pointer
// would then be stale. The first lookup on a device loads the array.
qsa_status scratch_on_current_device(void** addr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) return QSA_ERR_CUDA;
  *addr = p;
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
      (reinterpret_cast<uintptr_t>(q) & 15u))
    return QSA_ERR_INVALID_ARG;
  // 4-byte and 2-byte elements: their scalar loads and stores need that alignment
  for (const void* p4 : {static_cast<const void*>(k_scale), static_cast<const void*>(v_scale),
                         static_cast<const void*>(page_table), static_cast<const void*>(sel_pos),
                         static_cast<const void*>(q_pos)})
    if (reinterpret_cast<uintptr_t>(p4) & 3u) return QSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) & 1u) return QSA_ERR_INVALID_ARG;

  // The usual plan, with fewer CTAs (so fewer partials) if it would not fit.
  qsa::AttnPlan plan = qsa::attn_plan(*dims, qsa::device_sm_count());
  const size_t rows = (size_t)dims->batch * dims->n_q;
  const size_t ticket_bytes = qsa::align_up((size_t)plan.units * sizeof(int32_t), 256);
  const size_t row_bytes = qsa::align_up(rows * dims->width * sizeof(int32_t), 256);
  const size_t piece_bytes = 2 * (size_t)qsa::kPartFloats * sizeof(float);  // two per CTA
  const size_t fixed = kHeaderBytes + ticket_bytes + row_bytes;
  if (fixed + piece_bytes > kScratchBytes) return QSA_ERR_WORKSPACE;  // not even one CTA fits
  const size_t max_grid = (kScratchBytes - fixed) / piece_bytes;
  if ((size_t)plan.grid > max_grid) plan.grid = (int)max_grid;

  void* scratch = nullptr;
  const qsa_status ss = scratch_on_current_device(&scratch);
  if (ss != QSA_OK) return ss;
  unsigned char* base = static_cast<unsigned char*>(scratch);
  int32_t* err = reinterpret_cast<int32_t*>(base);
  int32_t* tickets = reinterpret_cast<int32_t*>(base + kHeaderBytes);
  int32_t* sel_row = reinterpret_cast<int32_t*>(base + kHeaderBytes + ticket_bytes);
  float* partials = reinterpret_cast<float*>(base + fixed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error record and the arrival tickets must start at zero every call
  if (cudaMemsetAsync(base, 0, kHeaderBytes + ticket_bytes, s) != cudaSuccess) return QSA_ERR_CUDA;
  if (qsa::launch_resolve(*dims, sel_pos, q_pos, page_table, sel_row, err, s) != cudaSuccess) return QSA_ERR_CUDA;
  const cudaError_t e = qsa::launch_attn(*dims, q, k_cache, v_cache, k_scale, v_scale, sel_row, out, tickets,
                                         partials, plan, s, true);
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
