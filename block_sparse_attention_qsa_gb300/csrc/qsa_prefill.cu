// Chunked (prefill) scoring: many queries of one request against its blocks.
//
// The pages score the full 4-token blocks of a request against its verify
// queries (arex-research.com, section "四类优化", bullets 1-2). When a request
// brings a chunk of many new tokens at once, each of them is a query of the
// same scoring step, and the step becomes a dense product
//   S[i][b] = sum_h sum_d q_idx[i][h][d] * kc[b][h][d]
// over the chunk's queries i and the request's blocks b: a BF16 GEMM with
// FP32 accumulation, each query keeping only its causal blocks
// b < floor((p_i + 1) / 4).
//
// Design. One CTA per tile of 128 blocks x 64 queries of one request, 8
// warps of 32 blocks x 32 queries on mma.sync m16n8k16. Each index head is
// one 128-wide k stage: the tile's key rows and query rows are copied into
// shared memory with cp.async (rows padded so ldmatrix is conflict-free),
// the first while the tile's query positions are read, the next head's while
// one head is multiplied. The FP32 tile goes back through shared memory so
// that each query's scores are written as consecutive blocks. For a chunk of
// 1,024 queries the scores written (4 bytes per query and block) are several
// times the bytes read and about four times the tensor work's time at the
// measured peaks: the kernel is bound by HBM writes, not by the tensor cores.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kBM = 128;            // blocks per tile (M)
constexpr int kBN = 64;             // queries per tile (N)
constexpr int kBK = 128;            // one index head's dims per k stage
constexpr int kLd = kBK + 8;        // padded row, in BF16 elements (272 bytes)
constexpr int kPThreads = 256;      // 8 warps: 4 along M x 2 along N
constexpr int kStageElems = (kBM + kBN) * kLd;
constexpr int kOutLd = kBM + 4;     // padded row of the FP32 output tile

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte async copy; src_bytes 0 fills zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kPThreads) score_chunk_kernel(const __nv_bfloat16* __restrict__ q_idx,
                                                              const __nv_bfloat16* __restrict__ kc,
                                                              const int32_t* __restrict__ q_pos,
                                                              float* __restrict__ scores, int32_t* err,
                                                              int n_chunk, int H, int max_blocks) {
  extern __shared__ __align__(16) __nv_bfloat16 psm[];
  __shared__ int s_nf[kBN];  // causal blocks of each query of the tile (0 for none)
  __shared__ int s_nf_max;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b0 = blockIdx.x * kBM, i0 = blockIdx.y * kBN, r = blockIdx.z;

  // stage h: the tile's 128 key rows and 64 query rows of index head h
  auto stage = [&](int h, int buf) {
    __nv_bfloat16* A = psm + buf * kStageElems;
    __nv_bfloat16* B = A + kBM * kLd;
    for (int c = tid; c < kBM * 16; c += kPThreads) {  // 16 chunks of 16 bytes per row
      const int row = c >> 4, ch = c & 15;
      const int b = b0 + row;
      const bool ok = b < max_blocks;
      const __nv_bfloat16* src = kc + (((size_t)r * max_blocks + (ok ? b : 0)) * H + h) * kBK + ch * 8;
      cp_async16(A + row * kLd + ch * 8, src, ok ? 16 : 0);
    }
    for (int c = tid; c < kBN * 16; c += kPThreads) {
      const int row = c >> 4, ch = c & 15;
      const int i = i0 + row;
      const bool ok = i < n_chunk;
      const __nv_bfloat16* src = q_idx + (((size_t)r * n_chunk + (ok ? i : 0)) * H + h) * kBK + ch * 8;
      cp_async16(B + row * kLd + ch * 8, src, ok ? 16 : 0);
    }
  };

  // the tile's first head is copied while the queries' positions are read
  stage(0, 0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  if (tid == 0) s_nf_max = 0;
  __syncthreads();
  if (tid < kBN) {
    const int i = i0 + tid;
    int nf = 0;
    if (i < n_chunk) {
      const int p = q_pos[(size_t)r * n_chunk + i];
      if (p < 0 || n_full_of(p) > max_blocks) {
        if (blockIdx.x == 0) record_error(err, kErrQueryPos, r, i, p);
      } else {
        nf = n_full_of(p);
      }
    }
    s_nf[tid] = nf;
    atomicMax(&s_nf_max, nf);
  }
  __syncthreads();
  if (b0 >= s_nf_max) {  // no query of the tile sees these blocks
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    return;
  }

  const int wm = warp & 3, wn = warp >> 2;  // this warp's 32 blocks x 32 queries
  float acc[2][4][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) acc[mi][ni][0] = acc[mi][ni][1] = acc[mi][ni][2] = acc[mi][ni][3] = 0.f;

  for (int h = 0; h < H; ++h) {
    const int buf = h & 1;  // one stage buffer when H == 1
    if (h + 1 < H) stage(h + 1, buf ^ 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // stage h has landed
    __syncthreads();
    const __nv_bfloat16* A = psm + buf * kStageElems;
    const __nv_bfloat16* B = A + kBM * kLd;
#pragma unroll
    for (int ks = 0; ks < kBK / 16; ++ks) {
      uint32_t a[2][4], b[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
        ldmatrix_x4(a[mi], A + (wm * 32 + mi * 16 + (lane & 15)) * kLd + ks * 16 + (lane >> 4) * 8);
      // two n8 tiles per ldmatrix.x4: (n rows, k 0-7), (n rows, k 8-15) of tiles 2j and 2j + 1
#pragma unroll
      for (int j = 0; j < 2; ++j)
        ldmatrix_x4(b[j], B + (wn * 32 + j * 16 + (lane >> 4) * 8 + (lane & 7)) * kLd + ks * 16 +
                              ((lane >> 3) & 1) * 8);
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          mma_bf16(acc[mi][2 * j], a[mi], b[j][0], b[j][1]);
          mma_bf16(acc[mi][2 * j + 1], a[mi], b[j][2], b[j][3]);
        }
    }
    __syncthreads();  // the stage is free for the copy two heads on
  }

  // the FP32 tile, queries x blocks, through shared memory
  float* T = reinterpret_cast<float*>(psm);
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) {
      const int m = wm * 32 + mi * 16 + g, n = wn * 32 + ni * 8 + 2 * c;
      T[n * kOutLd + m] = acc[mi][ni][0];
      T[(n + 1) * kOutLd + m] = acc[mi][ni][1];
      T[n * kOutLd + m + 8] = acc[mi][ni][2];
      T[(n + 1) * kOutLd + m + 8] = acc[mi][ni][3];
    }
  __syncthreads();
  // each warp writes whole query rows: 128 consecutive blocks, causal ones only
  for (int n = warp; n < kBN; n += kPThreads / 32) {
    const int i = i0 + n;
    if (i >= n_chunk) break;
    const int nf = s_nf[n];
    float* dst = scores + ((size_t)r * n_chunk + i) * max_blocks + b0;
#pragma unroll
    for (int k = 0; k < kBM / 32; ++k) {
      const int m = k * 32 + lane;
      if (b0 + m < nf) dst[m] = T[n * kOutLd + m];
    }
  }
}

}  // namespace

cudaError_t launch_score_chunk(const qsa_dims& d, int n_chunk, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                               const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s) {
  // two stage buffers only when there is a second index head to overlap with
  // (one head: 52 KB per CTA, four CTAs per SM)
  const size_t smem = (size_t)(d.n_idx_heads > 1 ? 2 : 1) * kStageElems * sizeof(__nv_bfloat16);
  static_assert((size_t)kBN * kOutLd * sizeof(float) <= (size_t)kStageElems * sizeof(__nv_bfloat16),
                "output tile larger than a stage buffer");
  static DeviceSlots smem_slots;
  if (const cudaError_t e = smem_slots.raise_smem(score_chunk_kernel, smem); e != cudaSuccess) return e;
  const dim3 grid((d.max_blocks + kBM - 1) / kBM, (n_chunk + kBN - 1) / kBN, d.batch);
  return launch_k(score_chunk_kernel, grid, dim3(kPThreads), smem, s, false, q_idx, kc, q_pos, scores, err, n_chunk,
                  d.n_idx_heads, d.max_blocks);
}

}  // namespace qsa
