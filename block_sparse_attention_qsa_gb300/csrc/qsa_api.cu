// C ABI of libqsa.so: argument checks, workspace planning and kernel chaining.
#include <math.h>
#include <string.h>

#include <algorithm>

#include "qsa_internal.cuh"
#include "qsa_trace.cuh"

namespace qsa {

int device_sm_count() {
  static DeviceSlots sms;
  const int n = sms.get([] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return v;
  });
  return n > 0 ? n : 1;
}

WsLayout ws_layout(const qsa_dims& d, int num_sms) {
  WsLayout w;
  const AttnPlan pl = attn_plan(d, num_sms);
  w.units = pl.units;
  w.tiles = pl.tiles;
  w.grid = pl.grid;
  w.cl = pl.cl;
  qsa_dims dd = d;  // a draft step's wider selection may take more CTAs
  dd.width = kDraftWidth;
  const int grid_max = std::max(pl.grid, attn_plan(dd, num_sms).grid);
  const size_t rows = (size_t)d.batch * d.n_q;
  size_t off = 256;  // header
  w.tickets = off;
  off = align_up(off + (size_t)pl.units * sizeof(int32_t), 256);
  w.partials = off;
  off = align_up(off + (size_t)grid_max * 2 * kPartFloats * sizeof(float), 256);
  w.scores = off;
  off = align_up(off + rows * d.max_blocks * sizeof(float), 256);
  w.sel_row = off;
  off = align_up(off + rows * kDraftWidth * sizeof(int32_t), 256);
  w.total = off;
  return w;
}

}  // namespace qsa

using namespace qsa;

namespace {

qsa_status check_dims(const qsa_dims* d) {
  if (!d) return QSA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->n_q < 1 || d->max_blocks < 1 || d->max_pages < 1 || d->num_pages < 1 ||
      d->n_kv_heads < 1 || d->n_idx_heads < 1 || d->page_size < 1)
    return QSA_ERR_INVALID_ARG;
  if (d->n_q > kMaxNq || d->n_idx_heads > 4 || d->idx_dim != kDim || d->head_dim != kDim ||
      d->n_q_heads != kGroup * d->n_kv_heads || d->block != kBlock || d->topk != kTopK ||
      d->width != kWidth)
    return QSA_ERR_UNSUPPORTED;
  if (d->page_size < 16 || d->page_size > 256 || (d->page_size & (d->page_size - 1)) != 0)
    return QSA_ERR_UNSUPPORTED;
  if (d->kv_dtype != QSA_KV_BF16 && d->kv_dtype != QSA_KV_FP8_E4M3) return QSA_ERR_UNSUPPORTED;
  if (!(d->sm_scale >= 0.f) || isinf(d->sm_scale)) return QSA_ERR_INVALID_ARG;
  // 32-bit index limits of the kernels
  if ((long long)d->num_pages * d->n_kv_heads * d->page_size >= (1LL << 31)) return QSA_ERR_UNSUPPORTED;
  if ((long long)d->max_blocks * kBlock >= (1LL << 31)) return QSA_ERR_UNSUPPORTED;
  if ((long long)d->max_pages * d->page_size >= (1LL << 31)) return QSA_ERR_UNSUPPORTED;
  if ((long long)d->batch * d->n_q * d->n_kv_heads * 128 >= (1LL << 31)) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

qsa_status check_ws(const qsa_dims* d, void* ws, size_t ws_bytes, WsLayout* out) {
  if (!ws) return QSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return QSA_ERR_WORKSPACE;
  const WsLayout w = ws_layout(*d, device_sm_count());
  if (ws_bytes < w.total) return QSA_ERR_WORKSPACE;
  if (out) *out = w;
  return QSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// every non-null pointer is a multiple of `a` bytes (a power of two); the
// kernels' scalar loads and stores of 4-byte and 2-byte elements need it
template <typename... P>
bool aligned_all(uintptr_t a, P... ps) {
  return ((ps == nullptr || (reinterpret_cast<uintptr_t>(ps) & (a - 1)) == 0) && ...);
}

qsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA; }

inline int32_t* err_word(void* ws) { return static_cast<int32_t*>(ws); }

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

}  // namespace

extern "C" {

int32_t qsa_abi_version(void) { return QSA_ABI_VERSION; }

const char* qsa_status_str(qsa_status s) {
  switch (s) {
    case QSA_OK: return "QSA_OK";
    case QSA_ERR_INVALID_ARG: return "QSA_ERR_INVALID_ARG";
    case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
    case QSA_ERR_WORKSPACE: return "QSA_ERR_WORKSPACE";
    case QSA_ERR_BAD_INDEX: return "QSA_ERR_BAD_INDEX";
    case QSA_ERR_TIMEOUT: return "QSA_ERR_TIMEOUT";
    case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
  }
  return "QSA_UNKNOWN_STATUS";
}

void qsa_dims_default(qsa_dims* d) {
  if (!d) return;
  memset(d, 0, sizeof(*d));
  d->batch = 1;
  d->n_q = 1;
  d->n_idx_heads = 1;
  d->idx_dim = kDim;
  d->n_q_heads = 16;
  d->n_kv_heads = 2;
  d->head_dim = kDim;
  d->page_size = 64;
  d->topk = kTopK;
  d->block = kBlock;
  d->width = kWidth;
  d->sm_scale = 0.f;
  d->kv_dtype = QSA_KV_BF16;
}

qsa_status qsa_workspace_size(const qsa_dims* dims, size_t* bytes) {
  const qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (!bytes) return QSA_ERR_INVALID_ARG;
  *bytes = ws_layout(*dims, device_sm_count()).total;
  return QSA_OK;
}

qsa_status qsa_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes == 0) return QSA_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_compress_keys(const qsa_dims* dims, const void* idx_keys, const int32_t* q_pos,
                             const int32_t* block_lo, void* kc, void* ws, size_t ws_bytes,
                             void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (dims->batch > 65535) return QSA_ERR_UNSUPPORTED;  // one grid row (y) per request
  if (!idx_keys || !q_pos || !kc) return QSA_ERR_INVALID_ARG;
  if (!aligned16(idx_keys) || !aligned16(kc) || !aligned_all(4, q_pos, block_lo)) return QSA_ERR_INVALID_ARG;
  if ((st = check_ws(dims, ws, ws_bytes, nullptr)) != QSA_OK) return st;
  cudaError_t e = launch_compress(*dims, static_cast<const __nv_bfloat16*>(idx_keys), q_pos, block_lo,
                                  static_cast<__nv_bfloat16*>(kc), err_word(ws),
                                  static_cast<cudaStream_t>(stream));
  return from_cuda(e);
}

qsa_status qsa_compress_keys_paged(const qsa_dims* dims, const void* idx_keys, const int32_t* q_pos,
                                   const int32_t* block_lo, const int32_t* page_table, void* kc_cache,
                                   void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (dims->batch > 65535) return QSA_ERR_UNSUPPORTED;  // one grid row (y) per request
  if (!idx_keys || !q_pos || !page_table || !kc_cache) return QSA_ERR_INVALID_ARG;
  if (!aligned16(idx_keys) || !aligned16(kc_cache) || !aligned_all(4, q_pos, page_table)) return QSA_ERR_INVALID_ARG;
  if ((st = check_ws(dims, ws, ws_bytes, nullptr)) != QSA_OK) return st;
  return from_cuda(launch_compress(*dims, static_cast<const __nv_bfloat16*>(idx_keys), q_pos, block_lo,
                                   static_cast<__nv_bfloat16*>(kc_cache), err_word(ws),
                                   static_cast<cudaStream_t>(stream), page_table));
}

qsa_status qsa_score_paged(const qsa_dims* dims, const void* q_idx, const void* kc_cache,
                           const int32_t* page_table, const int32_t* q_pos, float* scores, void* ws,
                           size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (dims->batch > QSA_MAX_SCORE_BATCH) return QSA_ERR_UNSUPPORTED;  // per-request tables in shared memory
  if (!q_idx || !kc_cache || !page_table || !q_pos || !scores) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(kc_cache) || !aligned_all(4, page_table, q_pos, scores))
    return QSA_ERR_INVALID_ARG;
  if ((st = check_ws(dims, ws, ws_bytes, nullptr)) != QSA_OK) return st;
  return from_cuda(launch_score(*dims, static_cast<const __nv_bfloat16*>(q_idx),
                                static_cast<const __nv_bfloat16*>(kc_cache), q_pos, scores, err_word(ws),
                                static_cast<cudaStream_t>(stream), false, page_table));
}

qsa_status qsa_score(const qsa_dims* dims, const void* q_idx, const void* kc, const int32_t* q_pos,
                     float* scores, void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (dims->batch > QSA_MAX_SCORE_BATCH) return QSA_ERR_UNSUPPORTED;  // per-request tables in shared memory
  if (!q_idx || !kc || !q_pos || !scores) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(kc) || !aligned_all(4, q_pos, scores)) return QSA_ERR_INVALID_ARG;
  if ((st = check_ws(dims, ws, ws_bytes, nullptr)) != QSA_OK) return st;
  return from_cuda(launch_score(*dims, static_cast<const __nv_bfloat16*>(q_idx),
                                static_cast<const __nv_bfloat16*>(kc), q_pos, scores, err_word(ws),
                                static_cast<cudaStream_t>(stream), false));
}

qsa_status qsa_score_chunk(const qsa_dims* dims, int32_t n_chunk, const void* q_idx, const void* kc,
                           const int32_t* q_pos, float* scores, void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (n_chunk < 1 || n_chunk > QSA_MAX_CHUNK) return QSA_ERR_INVALID_ARG;
  if (!q_idx || !kc || !q_pos || !scores) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(kc) || !aligned_all(4, q_pos, scores)) return QSA_ERR_INVALID_ARG;
  if ((long long)dims->batch * n_chunk * dims->max_blocks >= (1LL << 40)) return QSA_ERR_UNSUPPORTED;
  if (dims->batch > 65535) return QSA_ERR_UNSUPPORTED;  // one grid row (z) per request
  if ((st = check_ws(dims, ws, ws_bytes, nullptr)) != QSA_OK) return st;
  return from_cuda(launch_score_chunk(*dims, n_chunk, static_cast<const __nv_bfloat16*>(q_idx),
                                      static_cast<const __nv_bfloat16*>(kc), q_pos, scores, err_word(ws),
                                      static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_test_chunk_timeout(const qsa_dims* dims, int32_t n_chunk, const void* q_idx, const void* kc,
                                  const int32_t* q_pos, float* scores, void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (n_chunk < 1 || n_chunk > QSA_MAX_CHUNK) return QSA_ERR_INVALID_ARG;
  if (!q_idx || !kc || !q_pos || !scores) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(kc) || !aligned_all(4, q_pos, scores)) return QSA_ERR_INVALID_ARG;
  if ((long long)dims->batch * n_chunk * dims->max_blocks >= (1LL << 40)) return QSA_ERR_UNSUPPORTED;
  if (dims->batch > 65535) return QSA_ERR_UNSUPPORTED;
  if ((st = check_ws(dims, ws, ws_bytes, nullptr)) != QSA_OK) return st;
  return from_cuda(launch_score_chunk(*dims, n_chunk, static_cast<const __nv_bfloat16*>(q_idx),
                                      static_cast<const __nv_bfloat16*>(kc), q_pos, scores, err_word(ws),
                                      static_cast<cudaStream_t>(stream), true));
}

qsa_status qsa_trace_read(int32_t kernel, uint64_t* host, int32_t n_ctas, int32_t clear) {
  if (n_ctas < 0 || n_ctas > kTraceCtas || (n_ctas > 0 && !host)) return QSA_ERR_INVALID_ARG;
  static_assert(QSA_TRACE_SLOTS == kTraceSlots, "trace record size");
  unsigned long long* h = reinterpret_cast<unsigned long long*>(host);
  cudaError_t e;
  switch (kernel) {
    case QSA_TRACE_SCORE: e = trace_score(h, n_ctas, clear != 0); break;
    case QSA_TRACE_TOPK: e = trace_topk(h, n_ctas, clear != 0); break;
    case QSA_TRACE_ATTN: e = trace_attn(h, n_ctas, clear != 0); break;
    default: return QSA_ERR_INVALID_ARG;
  }
  if (e == cudaErrorNotSupported) return QSA_ERR_UNSUPPORTED;
  return from_cuda(e);
}

qsa_status qsa_topk(const qsa_dims* dims, const float* scores, const int32_t* q_pos,
                    int32_t* sel_blk, int32_t* sel_pos, void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (!scores || !q_pos || !sel_blk || !sel_pos) return QSA_ERR_INVALID_ARG;
  if (!aligned_all(4, scores, q_pos, sel_blk, sel_pos)) return QSA_ERR_INVALID_ARG;
  if ((st = check_ws(dims, ws, ws_bytes, nullptr)) != QSA_OK) return st;
  return from_cuda(launch_topk(*dims, scores, q_pos, sel_blk, sel_pos, err_word(ws), nullptr, nullptr,
                               static_cast<cudaStream_t>(stream), false));
}

qsa_status qsa_sparse_attn(const qsa_dims* dims, const void* q, const void* k_cache,
                           const void* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* page_table, const int32_t* sel_pos, const int32_t* q_pos,
                           void* out, void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (!q || !k_cache || !v_cache || !page_table || !sel_pos || !q_pos || !out)
    return QSA_ERR_INVALID_ARG;
  if (dims->kv_dtype == QSA_KV_FP8_E4M3 && (!k_scale || !v_scale)) return QSA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q))
    return QSA_ERR_INVALID_ARG;
  if (!aligned_all(4, k_scale, v_scale, page_table, sel_pos, q_pos) || !aligned_all(2, out))
    return QSA_ERR_INVALID_ARG;
  WsLayout w;
  if ((st = check_ws(dims, ws, ws_bytes, &w)) != QSA_OK) return st;
  const AttnPlan pl{w.units, w.tiles, w.grid, w.cl};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* srow = at<int32_t>(ws, w.sel_row);
  if (launch_resolve(*dims, sel_pos, q_pos, page_table, srow, err_word(ws), s) != cudaSuccess)
    return QSA_ERR_CUDA;
  return from_cuda(launch_attn(*dims, q, k_cache, v_cache, k_scale, v_scale, srow, out,
                               at<int32_t>(ws, w.tickets), at<float>(ws, w.partials), pl, s, true));
}

qsa_status qsa_resolve(const qsa_dims* dims, const int32_t* sel_pos, const int32_t* q_pos,
                       const int32_t* page_table, int32_t* sel_row, void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (!sel_pos || !q_pos || !page_table || !sel_row) return QSA_ERR_INVALID_ARG;
  if (!aligned_all(4, sel_pos, q_pos, page_table, sel_row)) return QSA_ERR_INVALID_ARG;
  if ((st = check_ws(dims, ws, ws_bytes, nullptr)) != QSA_OK) return st;
  return from_cuda(launch_resolve(*dims, sel_pos, q_pos, page_table, sel_row, err_word(ws),
                                  static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_sparse_attn_rows(const qsa_dims* dims, const void* q, const void* k_cache, const void* v_cache,
                                const float* k_scale, const float* v_scale, const int32_t* sel_row, void* out,
                                void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (!q || !k_cache || !v_cache || !sel_row || !out) return QSA_ERR_INVALID_ARG;
  if (dims->kv_dtype == QSA_KV_FP8_E4M3 && (!k_scale || !v_scale)) return QSA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q))
    return QSA_ERR_INVALID_ARG;
  if (!aligned_all(4, k_scale, v_scale, sel_row) || !aligned_all(2, out)) return QSA_ERR_INVALID_ARG;
  WsLayout w;
  if ((st = check_ws(dims, ws, ws_bytes, &w)) != QSA_OK) return st;
  const AttnPlan pl{w.units, w.tiles, w.grid, w.cl};
  return from_cuda(launch_attn(*dims, q, k_cache, v_cache, k_scale, v_scale, sel_row, out,
                               at<int32_t>(ws, w.tickets), at<float>(ws, w.partials), pl,
                               static_cast<cudaStream_t>(stream), true));
}

}  // extern "C"

namespace {

// The fused step; kc_paged: the compressed keys live in the KV cache's pages.
qsa_status decode_impl(const qsa_dims* dims, const void* q_idx, const void* kc, const void* q,
                       const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
                       const int32_t* page_table, const int32_t* q_pos, float* scores, int32_t* sel_blk,
                       int32_t* sel_pos, void* out, void* ws, size_t ws_bytes, void* stream, bool kc_paged) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (dims->batch > QSA_MAX_SCORE_BATCH) return QSA_ERR_UNSUPPORTED;  // per-request tables in shared memory
  if (!q_idx || !kc || !q || !k_cache || !v_cache || !page_table || !q_pos || !out)
    return QSA_ERR_INVALID_ARG;
  if (dims->kv_dtype == QSA_KV_FP8_E4M3 && (!k_scale || !v_scale)) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(kc) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(q))
    return QSA_ERR_INVALID_ARG;
  if (!aligned_all(4, k_scale, v_scale, page_table, q_pos, scores, sel_blk, sel_pos) || !aligned_all(2, out))
    return QSA_ERR_INVALID_ARG;
  WsLayout w;
  if ((st = check_ws(dims, ws, ws_bytes, &w)) != QSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* sc = scores ? scores : at<float>(ws, w.scores);
  cudaError_t e = launch_score(*dims, static_cast<const __nv_bfloat16*>(q_idx),
                               static_cast<const __nv_bfloat16*>(kc), q_pos, sc, err_word(ws), s, false,
                               kc_paged ? page_table : nullptr);
  if (e != cudaSuccess) return QSA_ERR_CUDA;
  int32_t* srow = at<int32_t>(ws, w.sel_row);
  // block ids and positions only when the caller asked for them; attention needs the cache rows
  e = launch_topk(*dims, sc, q_pos, sel_blk, sel_pos, err_word(ws), page_table, srow, s, true);
  if (e != cudaSuccess) return QSA_ERR_CUDA;
  const AttnPlan pl{w.units, w.tiles, w.grid, w.cl};
  e = launch_attn(*dims, q, k_cache, v_cache, k_scale, v_scale, srow, out, at<int32_t>(ws, w.tickets),
                  at<float>(ws, w.partials), pl, s, true);
  return from_cuda(e);
}

}  // namespace

extern "C" {

qsa_status qsa_decode(const qsa_dims* dims, const void* q_idx, const void* kc, const void* q,
                      const void* k_cache, const void* v_cache, const float* k_scale,
                      const float* v_scale, const int32_t* page_table, const int32_t* q_pos,
                      float* scores, int32_t* sel_blk, int32_t* sel_pos, void* out, void* ws,
                      size_t ws_bytes, void* stream) {
  return decode_impl(dims, q_idx, kc, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, scores, sel_blk,
                     sel_pos, out, ws, ws_bytes, stream, false);
}

qsa_status qsa_decode_paged(const qsa_dims* dims, const void* q_idx, const void* kc_cache, const void* q,
                            const void* k_cache, const void* v_cache, const float* k_scale,
                            const float* v_scale, const int32_t* page_table, const int32_t* q_pos,
                            float* scores, int32_t* sel_blk, int32_t* sel_pos, void* out, void* ws,
                            size_t ws_bytes, void* stream) {
  return decode_impl(dims, q_idx, kc_cache, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, scores,
                     sel_blk, sel_pos, out, ws, ws_bytes, stream, true);
}

qsa_status qsa_draft_attn(const qsa_dims* dims, const void* q, const void* k_cache, const void* v_cache,
                          const float* k_scale, const float* v_scale, const int32_t* page_table,
                          const int32_t* sel_pos, const int32_t* sel_q_pos, int32_t n_sel, const int32_t* src,
                          const int32_t* q_pos, void* out, void* ws, size_t ws_bytes, void* stream) {
  qsa_status st = check_dims(dims);
  if (st != QSA_OK) return st;
  if (!q || !k_cache || !v_cache || !page_table || !sel_pos || !sel_q_pos || !src || !q_pos || !out)
    return QSA_ERR_INVALID_ARG;
  if (n_sel < 1 || n_sel > kMaxNq) return QSA_ERR_INVALID_ARG;
  if (dims->kv_dtype == QSA_KV_FP8_E4M3 && (!k_scale || !v_scale)) return QSA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q))
    return QSA_ERR_INVALID_ARG;
  if (!aligned_all(4, k_scale, v_scale, page_table, sel_pos, sel_q_pos, src, q_pos) || !aligned_all(2, out))
    return QSA_ERR_INVALID_ARG;
  WsLayout w;
  if ((st = check_ws(dims, ws, ws_bytes, &w)) != QSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* srow = at<int32_t>(ws, w.sel_row);
  if (launch_draft_resolve(*dims, sel_pos, sel_q_pos, n_sel, src, q_pos, page_table, srow, err_word(ws), s) !=
      cudaSuccess)
    return QSA_ERR_CUDA;
  qsa_dims dd = *dims;  // attention over the widened selection
  dd.width = kDraftWidth;
  const AttnPlan pl = attn_plan(dd, device_sm_count());
  return from_cuda(launch_attn(dd, q, k_cache, v_cache, k_scale, v_scale, srow, out, at<int32_t>(ws, w.tickets),
                               at<float>(ws, w.partials), pl, s, true));
}

qsa_status qsa_check_errors(void* ws, void* stream, int32_t* info) {
  if (!ws) return QSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return QSA_ERR_CUDA;
  int32_t hdr[4] = {0, 0, 0, 0};
  if (cudaMemcpy(hdr, ws, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess) return QSA_ERR_CUDA;
  if (info) memcpy(info, hdr, sizeof(hdr));
  if (hdr[0] == 0) return QSA_OK;
  if (cudaMemsetAsync(ws, 0, sizeof(hdr), s) != cudaSuccess) return QSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QSA_ERR_CUDA;
  return hdr[0] == kErrTimeout ? QSA_ERR_TIMEOUT : QSA_ERR_BAD_INDEX;
}

}  // extern "C"
