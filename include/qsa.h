/*
 * qsa.h -- C ABI of libqsa.so: the decode / MTP-verify step of Qwen Sparse
 * Attention (QSA) on one GB300 (sm_103a).
 *
 * The step, as the pages state it (arex-research.com, "LightSeek 公告
 * TokenSpeed 服务 Qwen3.8-Flash-Next ...", section "稀疏选择、CuTe DSL 内核与
 * MTP 复用：四类优化", bullets 1-4; 10100.com, section "第一处"):
 *   1. tokens form micro-blocks of 4; each block has a compressed index key;
 *   2. every full block is scored against each query's index query and the
 *      scores go to an FP32 buffer; up to 4 verify queries of one request
 *      share each compressed-key tile load (bullet 2);
 *   3. a persistent radix selector keeps the top 512 blocks per query; the
 *      current unfilled block is kept without selection; the selection buffer
 *      is 2,051 positions wide (bullet 1);
 *   4. sparse attention over the selected positions with a BF16 query and a
 *      BF16 or FP8-E4M3 KV cache (bullet 3); the three kernels are chained
 *      with programmatic dependent launch (bullet 4).
 * Around the step: qsa_compress_keys (the compressed keys themselves),
 * qsa_draft_attn (MTP draft steps reusing a selection), the *_paged entry
 * points (compressed keys kept in the KV cache's pages), qsa_score_chunk
 * (scoring a chunk of many queries per request), qsa_sparse_attn_noalloc
 * (attention without a caller workspace), and qsa_resolve /
 * qsa_sparse_attn_rows (qsa_sparse_attn's two launches, separately).
 *
 * Readings where the pages are silent:
 *   - full blocks of a query at position p: b < (p + 1) / 4; the unfilled
 *     block holds positions 4 * ((p + 1) / 4) .. p, (p + 1) % 4 of them;
 *   - compressed key = FP32 mean of the block's 4 BF16 index keys, summed in
 *     token order, rounded to BF16 (qsa_compress_keys);
 *   - score = dot(index query, compressed key) summed over index heads, FP32;
 *   - top-k ties go to the lower block index; -0.0 == +0.0; NaN ranks last;
 *   - the selection buffer lists selected blocks ascending (4 positions
 *     each), then the unfilled block's positions, then -1;
 *   - query head h reads KV head h / (n_q_heads / n_kv_heads); softmax scale
 *     sm_scale (default 1/sqrt(head_dim)); FP8 values are code * scale with
 *     one FP32 scale per KV head, separate for K and V.
 *
 * Layouts (all row-major, all device memory owned by the caller):
 *   q_idx      bf16  [batch][n_q][n_idx_heads][idx_dim]
 *   idx_keys   bf16  [batch][4 * max_blocks][n_idx_heads][idx_dim]
 *   kc         bf16  [batch][max_blocks][n_idx_heads][idx_dim]
 *   kc_cache   bf16  [num_pages][page_size / 4][n_idx_heads][idx_dim]
 *                                        (the *_paged entry points)
 *   q_pos      int32 [batch][n_q]        position of each query token; the
 *                                        query's own K/V is already cached
 *   scores     fp32  [batch][n_q][max_blocks]   (entries past a query's
 *                                        full blocks are left untouched)
 *   sel_blk    int32 [batch][n_q][topk]  ascending, -1 padded
 *   sel_pos    int32 [batch][n_q][width] ascending, -1 padded
 *   q, out     bf16  [batch][n_q][n_q_heads][head_dim]
 *   k_cache, v_cache  bf16 or uint8 (E4M3 codes)
 *                     [num_pages][n_kv_heads][page_size][head_dim]
 *   k_scale, v_scale  fp32 [n_kv_heads]  (read only for FP8; may be NULL
 *                                         for BF16)
 *   page_table int32 [batch][max_pages]  token t of request r lives in page
 *                                        page_table[r][t / page_size], slot
 *                                        t % page_size
 *
 * Execution: every call is asynchronous on `stream` (a cudaStream_t passed as
 * void*; NULL = the legacy default stream) and allocates nothing. Argument
 * and shape errors return synchronously before anything is launched.
 * Data-dependent errors found on the device (a query position outside the
 * buffers, a page id outside the cache, a selected position after its query)
 * are recorded in the workspace header and the offending item is skipped (a
 * query with a bad position gets no scores, an all -1 selection and a zero
 * output; a bad selected position or page is left out of the softmax);
 * qsa_check_errors() reports them. No call aborts or throws.
 *
 * Alignment: idx_keys, q_idx, kc (or kc_cache), q, k_cache and v_cache are read with
 * 16-byte vector loads or copies and must be 16-byte aligned; the other
 * arrays need the alignment of their element type. A misaligned pointer
 * returns QSA_ERR_INVALID_ARG before anything is launched.
 *
 * Workspace: every entry point takes `ws`, a caller-owned device buffer of at
 * least qsa_workspace_size() bytes, 256-byte aligned, zero-filled once before
 * its first use (qsa_workspace_init). The kernels leave it in a state ready
 * for the next call. Calls that share a workspace must not overlap on the
 * GPU (issue them on one stream).
 *
 * Supported geometry: idx_dim == head_dim == 128, n_q in 1..4,
 * n_idx_heads in 1..4, n_q_heads == 8 * n_kv_heads, block == 4, topk == 512,
 * width == 2051, page_size a power of two in 16..256; anything else returns
 * QSA_ERR_UNSUPPORTED.
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_ABI_VERSION 1

/* Most positions a draft query may lie after the query whose selection it
 * reuses (qsa_draft_attn). */
#define QSA_MAX_DRAFT_GAP 64

/* Most requests in one qsa_score / qsa_score_paged / qsa_decode /
 * qsa_decode_paged call (the scoring kernel keeps two small per-request tables
 * in shared memory); larger batches return QSA_ERR_UNSUPPORTED. */
#define QSA_MAX_SCORE_BATCH 16384

/* Most queries per request in one qsa_score_chunk call. */
#define QSA_MAX_CHUNK 65536

typedef enum {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1, /* null pointer, bad size or stride */
  QSA_ERR_UNSUPPORTED = 2, /* geometry outside the supported set */
  QSA_ERR_WORKSPACE = 3,   /* ws too small or misaligned */
  QSA_ERR_BAD_INDEX = 4,   /* device found an out-of-range position/page */
  QSA_ERR_TIMEOUT = 5,     /* a bounded device wait gave up */
  QSA_ERR_CUDA = 6         /* a CUDA runtime call failed */
} qsa_status;

typedef enum { QSA_KV_BF16 = 0, QSA_KV_FP8_E4M3 = 1 } qsa_kv_dtype;

typedef struct {
  int32_t batch;       /* requests in the step, >= 1 */
  int32_t n_q;         /* query tokens per request (1 decode, 4 verify) */
  int32_t n_idx_heads; /* index heads whose scores are summed */
  int32_t idx_dim;     /* index head dim, 128 */
  int32_t n_q_heads;   /* attention query heads, 16 */
  int32_t n_kv_heads;  /* attention KV heads, 2 */
  int32_t head_dim;    /* 128 */
  int32_t page_size;   /* tokens per KV page, 64 */
  int32_t max_blocks;  /* row stride (in blocks) of kc and scores */
  int32_t max_pages;   /* row stride of page_table */
  int32_t num_pages;   /* pages in k_cache / v_cache */
  int32_t topk;        /* 512 */
  int32_t block;       /* 4 */
  int32_t width;       /* selection width, topk * block + block - 1 = 2051 */
  float sm_scale;      /* softmax scale; 0 selects 1/sqrt(head_dim) */
  int32_t kv_dtype;    /* qsa_kv_dtype */
} qsa_dims;

/* ABI version of the loaded library (QSA_ABI_VERSION it was built with). */
int32_t qsa_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* qsa_status_str(qsa_status s);

/* Fill `dims` with the defaults of the pages' geometry (16/2 heads of 128,
 * 1 index head of 128, pages of 64, top-512 of 4-token blocks, width 2,051,
 * BF16 KV); the caller then sets batch, n_q, max_blocks, max_pages,
 * num_pages and anything else it changes. */
void qsa_dims_default(qsa_dims* dims);

/* Bytes of workspace the entry points need for `dims` on the current device.
 * The size depends on the device's SM count (it sizes the attention partials). */
qsa_status qsa_workspace_size(const qsa_dims* dims, size_t* bytes);

/* Zero `ws` (ws_bytes bytes) on `stream`. Required once after allocating a
 * workspace; the kernels keep it clean afterwards. */
qsa_status qsa_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Compressed index key of each full block (the pages' bullet 1 "compute a
 * compressed index key per micro-block"; the formula is this library's
 * reading: FP32 mean of the 4 keys, summed in token order, rounded to BF16).
 * For request r, writes kc[r][b] for block_lo[r] <= b < (P_r + 1) / 4 where
 * P_r = max_j q_pos[r][j]; block_lo may be NULL (= 0 for every request), so
 * an engine can refresh only the blocks its newest tokens completed. At most
 * 65,535 requests per call (also for qsa_compress_keys_paged). */
qsa_status qsa_compress_keys(const qsa_dims* dims, const void* idx_keys, const int32_t* q_pos,
                             const int32_t* block_lo, void* kc, void* ws, size_t ws_bytes,
                             void* stream);

/* Step 1: FP32 block scores (bullet 1: "block scores are written to an FP32
 * buffer"; bullet 2: up to 4 queries of a request share one compressed-key
 * load). For each request r, query j at p = q_pos[r][j] and full block
 * b < (p + 1) / 4: scores[r][j][b] = sum_h sum_d q_idx[r][j][h][d] *
 * kc[r][b][h][d] in FP32. Each compressed key is read from HBM once per
 * request and used for all n_q queries. */
qsa_status qsa_score(const qsa_dims* dims, const void* q_idx, const void* kc, const int32_t* q_pos,
                     float* scores, void* ws, size_t ws_bytes, void* stream);

/* Steps 2-3: top-k block selection and the selection buffer (bullet 1:
 * persistent radix selector over the FP32 scores, at most 512 full blocks,
 * the unfilled block kept, width 2,051). For each (r, j): sel_blk = the
 * min(topk, n_full) highest-scoring full blocks, ties to the lower index,
 * ascending, -1 padded; sel_pos = their positions 4b..4b+3 ascending, then
 * 4 * n_full .. p, then -1 up to width. Bit-exact and deterministic. */
qsa_status qsa_topk(const qsa_dims* dims, const float* scores, const int32_t* q_pos,
                    int32_t* sel_blk, int32_t* sel_pos, void* ws, size_t ws_bytes, void* stream);

/* Step 4: sparse attention over the selected positions (bullet 3: BF16
 * query, BF16 or FP8-E4M3 KV cache, decode and MTP verify). For each (r, j)
 * and query head h with KV head g = h / (n_q_heads / n_kv_heads):
 * out = softmax(sm_scale * q K^T) V over the positions t >= 0 of
 * sel_pos[r][j], with K, V read through page_table (times k_scale[g] /
 * v_scale[g] for FP8). FP32 softmax statistics and accumulation, BF16 out.
 * A selected position after q_pos[r][j] (a causality violation) or one whose
 * page id is outside the cache is reported and skipped. */
qsa_status qsa_sparse_attn(const qsa_dims* dims, const void* q, const void* k_cache,
                           const void* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* page_table, const int32_t* sel_pos, const int32_t* q_pos,
                           void* out, void* ws, size_t ws_bytes, void* stream);

/* qsa_sparse_attn in its two launches. qsa_resolve turns the selected
 * positions into cache rows: sel_row[r][j][i] = the row of position
 * sel_pos[r][j][i] for KV head 0 in k_cache / v_cache viewed as
 * [num_pages * n_kv_heads * page_size][128], i.e.
 * (page_table[r][t / page_size] * n_kv_heads) * page_size + t % page_size
 * (KV head g adds g * page_size), and -1 where sel_pos is -1 or the position
 * is rejected (after q_pos[r][j], or its page id outside the cache: reported
 * as in qsa_sparse_attn). sel_row is [B][n_q][width] int32, caller-owned.
 * qsa_sparse_attn_rows is the attention of qsa_sparse_attn over such rows
 * (same output, bit for bit); a row below 0, or one whose last KV head would
 * lie outside the cache, is skipped without a report. Rows computed once can
 * serve several attention calls. */
qsa_status qsa_resolve(const qsa_dims* dims, const int32_t* sel_pos, const int32_t* q_pos,
                       const int32_t* page_table, int32_t* sel_row, void* ws, size_t ws_bytes, void* stream);
qsa_status qsa_sparse_attn_rows(const qsa_dims* dims, const void* q, const void* k_cache, const void* v_cache,
                                const float* k_scale, const float* v_scale, const int32_t* sel_row, void* out,
                                void* ws, size_t ws_bytes, void* stream);

/* The fused step (bullet 4: "QSA logits -> select -> attention" chained with
 * programmatic dependent launch): qsa_score, qsa_topk and qsa_sparse_attn
 * back to back on `stream`. scores, sel_blk and sel_pos are optional outputs:
 * with NULL the scores stay in the workspace and the block ids and positions
 * are not written (attention reads the cache rows the selector writes). */
qsa_status qsa_decode(const qsa_dims* dims, const void* q_idx, const void* kc, const void* q,
                      const void* k_cache, const void* v_cache, const float* k_scale,
                      const float* v_scale, const int32_t* page_table, const int32_t* q_pos,
                      float* scores, int32_t* sel_blk, int32_t* sel_pos, void* out, void* ws,
                      size_t ws_bytes, void* stream);

/* qsa_sparse_attn for callers that cannot allocate device memory (code run
 * where cudaMalloc is not allowed, a process whose memory pool is fixed up
 * front, a plugin handed tensors but no allocator). The pages have no
 * counterpart: it is a deployment convenience of this library. Same inputs,
 * output and arithmetic as qsa_sparse_attn, but no workspace argument: its
 * scratch (resolved cache rows, arrival tickets, softmax partials) lives in a
 * 16 MiB array in the library's own device image, which every GPU that loads
 * the library keeps until the process exits.
 * The call allocates nothing (no cudaMalloc, no cudaFree, no allocating
 * library routine). Every call looks up that array's device address
 * (cudaGetSymbolAddress) on the current device, so it stays valid after a
 * device reset, which reloads the array; the first call on a device also
 * loads the array there, so make it before any stream capture. Every call
 * shares the one array per device and clears
 * its counters at the start, so calls that overlap on the GPU (different
 * streams, or different host threads on one device) race: issue them in
 * order on one stream. The CTA count is lowered to fit the array; when even
 * one CTA does not fit, that is batch * n_q above about 2,040 at 2 KV heads,
 * the call returns QSA_ERR_WORKSPACE before launching anything. Device-side index errors are
 * skipped as in qsa_sparse_attn, but there is no workspace to read them back
 * from: use qsa_sparse_attn to diagnose them. */
qsa_status qsa_sparse_attn_noalloc(const qsa_dims* dims, const void* q, const void* k_cache,
                                   const void* v_cache, const float* k_scale, const float* v_scale,
                                   const int32_t* page_table, const int32_t* sel_pos,
                                   const int32_t* q_pos, void* out, void* stream);

/* Scoring a chunk of many queries per request (a prefill chunk) against the
 * request's blocks: the score of step 1 (arex-research.com, section
 * "四类优化", bullets 1-2) for n_chunk queries at once, which makes it a dense
 * BF16 product over (query, block) pairs. dims gives batch, n_idx_heads,
 * max_blocks (its n_q is not used). q_idx is [B][n_chunk][n_idx_heads][128]
 * BF16, q_pos [B][n_chunk], kc as for qsa_score, scores
 * [B][n_chunk][max_blocks] FP32: scores[r][i][b] = sum_h sum_d
 * q_idx[r][i][h][d] * kc[r][b][h][d] in FP32 for b < (q_pos[r][i] + 1) / 4;
 * other entries are not written. 1 <= n_chunk <= QSA_MAX_CHUNK and batch <=
 * 65,535, else QSA_ERR_INVALID_ARG / QSA_ERR_UNSUPPORTED before any launch.
 * Runs on the tensor cores through TMA tensor maps of q_idx and kc (built on
 * the host each call; both 16-byte aligned, as checked). A max_blocks that is
 * a multiple of 32 makes every score row start on a 128-byte boundary, which
 * the kernel's row stores are fastest with (max_blocks is the buffers' block
 * capacity, so padding it costs only memory). The kernel's waits between its
 * own warps are bounded: one that gives up is reported as QSA_ERR_TIMEOUT by
 * qsa_check_errors (kind 5), with that call's scores incomplete. */
qsa_status qsa_score_chunk(const qsa_dims* dims, int32_t n_chunk, const void* q_idx, const void* kc,
                           const int32_t* q_pos, float* scores, void* ws, size_t ws_bytes, void* stream);

/* Failure-detection test of the bounded waits (no counterpart on the pages):
 * qsa_score_chunk with the first TMA copy of the kernel's first CTA left out,
 * so that CTA's wait for it runs into its clock limit (about one second).
 * The CTA then records the timeout, stops issuing work, waits (bounded) for
 * its own copies in flight, frees its tensor memory and returns; the other
 * CTAs finish normally. qsa_check_errors afterwards returns QSA_ERR_TIMEOUT
 * (kind 5), and the context stays usable. The scores of the first CTA's tiles
 * are not written. Same arguments and checks as qsa_score_chunk. */
qsa_status qsa_test_chunk_timeout(const qsa_dims* dims, int32_t n_chunk, const void* q_idx, const void* kc,
                                  const int32_t* q_pos, float* scores, void* ws, size_t ws_bytes, void* stream);

/* Phase timeline of the fused step's kernels (tracing; no counterpart on the
 * pages). Only the tracing build of the library (libqsa_trace.so, compiled
 * with -DQSA_TRACE) records anything; the product build returns
 * QSA_ERR_UNSUPPORTED and has no marks in its kernels. kernel selects the
 * table: QSA_TRACE_SCORE (qsa_score's kernel), QSA_TRACE_TOPK (the
 * selector, either form) or QSA_TRACE_ATTN (the attention kernel). Each CTA
 * below 4,096 of the kernel's most recent launches owns QSA_TRACE_SLOTS
 * uint64 words: %globaltimer (ns) at its start [0], at the release of its
 * wait on the previous kernel [1], when its main work was done [2] (the
 * latest of its warps where they finish apart), at its end [3], its SM id
 * plus one [4], and for attention the time it published a piece of a split
 * unit [5] and finished a merge of pieces [6]; a slot not reached is 0 (the
 * caller zeroes the tables with clear). host: n_ctas * QSA_TRACE_SLOTS words,
 * or null (with n_ctas 0) to only clear. Synchronous: waits for the device.
 * 0 <= n_ctas <= 4,096, else QSA_ERR_INVALID_ARG. */
enum { QSA_TRACE_SCORE = 0, QSA_TRACE_TOPK = 1, QSA_TRACE_ATTN = 2, QSA_TRACE_SLOTS = 8 };
qsa_status qsa_trace_read(int32_t kernel, uint64_t* host, int32_t n_ctas, int32_t clear);

/* Paged compressed keys (the pages place the selected history "in the
 * cache", 10100.com "第一处"; here the compressed keys live in the KV
 * cache's pages too, found through the same page table). kc_cache is
 * [num_pages][page_size / 4][n_idx_heads][128] BF16: page p holds the
 * compressed keys of the page_size / 4 blocks whose tokens it holds; block b
 * of request r is slot b % (page_size / 4) of page
 * page_table[r][b / (page_size / 4)]. Same arithmetic and results, bit for
 * bit, as qsa_compress_keys / qsa_score / qsa_decode on the contiguous
 * layout. A page id outside the cache is reported (kind 2) and its blocks are
 * skipped (not written; scored as zero). */
qsa_status qsa_compress_keys_paged(const qsa_dims* dims, const void* idx_keys, const int32_t* q_pos,
                                   const int32_t* block_lo, const int32_t* page_table, void* kc_cache,
                                   void* ws, size_t ws_bytes, void* stream);
qsa_status qsa_score_paged(const qsa_dims* dims, const void* q_idx, const void* kc_cache,
                           const int32_t* page_table, const int32_t* q_pos, float* scores, void* ws,
                           size_t ws_bytes, void* stream);
qsa_status qsa_decode_paged(const qsa_dims* dims, const void* q_idx, const void* kc_cache, const void* q,
                            const void* k_cache, const void* v_cache, const float* k_scale,
                            const float* v_scale, const int32_t* page_table, const int32_t* q_pos,
                            float* scores, int32_t* sel_blk, int32_t* sel_pos, void* out, void* ws,
                            size_t ws_bytes, void* stream);

/* MTP draft steps reusing an earlier selection (arex-research.com, section
 * "四类优化" heading: "MTP 复用"; 10100.com, "第三处": later draft steps reuse
 * the attention positions selected before, instead of scoring and selecting
 * again). Scoring and top-k are skipped; only attention runs. dims describes
 * the draft step: batch, n_q = draft queries per request (1..4), heads and
 * cache as for qsa_sparse_attn, width 2,051. sel_pos [B][n_sel][2051] holds
 * selection rows made by qsa_topk / qsa_decode for queries at positions
 * sel_q_pos [B][n_sel] (n_sel 1..4). Draft query j of request r, at position
 * p = q_pos[r][j], reuses row src[r][j] (0 <= src < n_sel), made for
 * p_src = sel_q_pos[r][src[r][j]]: out[r][j] = softmax(sm_scale q K^T) V over
 * the valid positions of that row plus every position p_src + 1 .. p, which
 * the row cannot hold (p_src <= p <= p_src + QSA_MAX_DRAFT_GAP). A draft
 * query outside that range (or a bad src) is reported (kind 4) and gets a
 * zero output; bad pages and selected positions after p_src are reported and
 * skipped as in qsa_sparse_attn. The workspace is sized by
 * qsa_workspace_size for dims. */
qsa_status qsa_draft_attn(const qsa_dims* dims, const void* q, const void* k_cache, const void* v_cache,
                          const float* k_scale, const float* v_scale, const int32_t* page_table,
                          const int32_t* sel_pos, const int32_t* sel_q_pos, int32_t n_sel, const int32_t* src,
                          const int32_t* q_pos, void* out, void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, reads and clears the device error record in `ws`.
 * Returns QSA_OK if no device-side error was recorded since the last check,
 * else QSA_ERR_BAD_INDEX (or QSA_ERR_TIMEOUT). `info` (may be NULL) receives
 * 4 int32: error kind (1 query position, 2 page id, 3 selected position,
 * 4 draft query not after its reused selection, 5 a bounded wait inside the
 * chunked-scoring kernel gave up), request, query, offending value. */
qsa_status qsa_check_errors(void* ws, void* stream, int32_t* info);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
