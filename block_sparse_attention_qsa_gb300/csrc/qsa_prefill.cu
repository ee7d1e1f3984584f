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
// Design (Blackwell tensor cores). One CTA of 4 warps per tile of 128 blocks
// x 128 queries of one request. For each index head, TMA copies the tile's
// 128 compressed-key rows and 128 query rows (256 bytes each) into shared
// memory in the 128-byte swizzled layout the tensor core reads, completing an
// mbarrier; one thread issues tcgen05.mma (M = 128 blocks, N = 128 queries,
// K = 16 per instruction) into an FP32 accumulator in tensor memory (TMEM:
// lane = block, column = query), and tcgen05.commit signals the epilogue. Two
// heads' stages are in flight when there are several heads. The epilogue
// reads the accumulator back with tcgen05.ld: warp w owns TMEM lanes (blocks)
// 32w..32w+31, so for every query a warp stores 32 consecutive scores (128
// contiguous bytes) of that query's row, the causal ones only. Scores are
// 4 bytes per (query, block) against 0.5 read, so the kernel is bound by the
// score writes, not by the tensor cores.
//
// Every wait (mbarrier phases) is bounded by a clock limit; past it the kernel
// records a timeout in the workspace header, issues nothing more, waits
// (bounded again) for its own copies in flight, frees its TMEM and returns.
#include <cuda.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kTM = 128;        // blocks per tile (MMA M, TMEM lanes)
constexpr int kTN = 128;        // queries per tile (MMA N, TMEM columns)
constexpr int kPThreads = 128;  // 4 warps: each reads 32 TMEM lanes in the epilogue
constexpr int kHalfBytes = kTM * 128;      // one 64-dim half of a tile's rows: 128 rows x 128 B (16 KB)
constexpr int kStageBytes = 4 * kHalfBytes;  // keys (2 halves) + queries (2 halves) of one index head
constexpr uint32_t kTmemCols = kTN;        // FP32 accumulator columns
constexpr long long kWaitCycles = 1LL << 31;  // about one second at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// waits for the phase with the given parity to complete; false after the clock limit
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
}

// 3-D tiled TMA load of box (x, y, z) into shared memory, completing on bar
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout (rows of 128 bytes, 8-row groups 1,024 bytes apart, the
// layout TMA writes with 128-byte swizzling): start address >> 4 in bits
// 0-13, leading-dimension offset (unused by this layout) 1 in bits 16-29,
// stride between 8-row groups (1,024 >> 4) in bits 32-45, descriptor version
// 1 in bits 46-47, swizzle mode 2 (128 bytes) in bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: FP32 accumulator (bits
// 4-5 = 1), BF16 A and B (bits 7-9 and 10-12 = 1), both K-major (bits 15, 16
// = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTN >> 3) << 17) |
                            ((uint32_t)(kTM >> 4) << 24);

__device__ __forceinline__ void mma_bf16_tmem(uint32_t d_tmem, uint64_t a, uint64_t b, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"((uint32_t)acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive FP32 accumulator columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kPThreads) score_chunk_kernel(const __grid_constant__ CUtensorMap tm_kc,
                                                              const __grid_constant__ CUtensorMap tm_q,
                                                              const int32_t* __restrict__ q_pos,
                                                              float* __restrict__ scores, int32_t* err,
                                                              int n_chunk, int H, int max_blocks, int stages) {
  extern __shared__ uint8_t psm_raw[];
  // stage buffers at a 1,024-byte boundary (the swizzle pattern repeats every 1,024 bytes)
  uint8_t* psm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(psm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[2], empty_bar[2], done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_nf[kTN];  // causal blocks of each query of the tile (0 for none)
  __shared__ int s_nf_max;
  __shared__ int s_timeout;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b0 = blockIdx.x * kTM, i0 = blockIdx.y * kTN, r = blockIdx.z;

  if (tid == 0) {
    s_nf_max = 0;
    s_timeout = 0;
  }
  __syncthreads();
  {
    const int i = i0 + tid;  // kPThreads == kTN: one query per thread
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
  if (b0 >= s_nf_max) return;  // no query of the tile sees these blocks: nothing allocated or issued

  // TMEM accumulator (one warp allocates) and the barriers (one thread)
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&done_bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;

  if (tid == 0) {
    // producer and MMA issuer
    auto load_head = [&](int h, int s) {
      const uint32_t base = smem_u32(psm + s * kStageBytes);
      const uint32_t bar = smem_u32(&full_bar[s]);
      mbar_expect_tx(bar, kStageBytes);
      tma_load_3d(base, &tm_kc, h * 128, b0, r, bar);
      tma_load_3d(base + kHalfBytes, &tm_kc, h * 128 + 64, b0, r, bar);
      tma_load_3d(base + 2 * kHalfBytes, &tm_q, h * 128, i0, r, bar);
      tma_load_3d(base + 3 * kHalfBytes, &tm_q, h * 128 + 64, i0, r, bar);
    };
    bool pending[2] = {false, false};  // a stage's copy issued and not yet seen complete
    uint32_t pend_par[2] = {0u, 0u};    // the phase parity that copy completes
    for (int h = 0; h < stages && h < H; ++h) {
      load_head(h, h);
      pending[h] = true;
    }
    bool ok = true;
    for (int h = 0; h < H && ok; ++h) {
      const int s = h % stages;
      const uint32_t par = (uint32_t)(h / stages) & 1u;
      if (!mbar_wait(smem_u32(&full_bar[s]), par)) {
        ok = false;
        break;
      }
      pending[s] = false;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t a0 = smem_u32(psm + s * kStageBytes), bq = a0 + 2 * kHalfBytes;
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // 16 dims per instruction: 4 steps of 32 bytes in each 64-dim half
        const uint32_t off = (uint32_t)(k >> 2) * kHalfBytes + (uint32_t)(k & 3) * 32u;
        mma_bf16_tmem(tmem, sw128_desc(a0 + off), sw128_desc(bq + off), h > 0 || k > 0);
      }
      if (h + stages < H) {
        mma_commit(smem_u32(&empty_bar[s]));  // the stage is free once these MMAs have read it
        if (!mbar_wait(smem_u32(&empty_bar[s]), par)) {
          ok = false;
          break;
        }
        load_head(h + stages, s);
        pending[s] = true;
        pend_par[s] = par ^ 1u;
      }
    }
    if (!ok) {
      s_timeout = 1;
      record_error(err, kErrTimeout, r, i0, b0);
      for (int s = 0; s < 2; ++s)  // copies still in flight land before the CTA leaves (bounded)
        if (pending[s]) mbar_wait(smem_u32(&full_bar[s]), pend_par[s]);
    }
    mma_commit(smem_u32(&done_bar));  // arrives once every MMA issued above has completed
  }
  __syncwarp();

  // epilogue: warp w reads TMEM lanes 32w..32w+31 (blocks b0 + 32w + lane)
  const bool done = mbar_wait(smem_u32(&done_bar), 0);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (!done && lane == 0) {
    s_timeout = 1;
    record_error(err, kErrTimeout, r, i0, b0);
  }
  __syncthreads();
  if (!s_timeout) {
    const int b = b0 + warp * 32 + lane;
    float* dst = scores + (size_t)r * n_chunk * max_blocks + b;
#pragma unroll 1
    for (int c0 = 0; c0 < kTN; c0 += 32) {
      if (i0 + c0 >= n_chunk) break;  // warp-uniform
      float v[32];
      __syncwarp();
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        const int i = i0 + c0 + n;
        if (i < n_chunk && b < s_nf[c0 + n]) dst[(size_t)i * max_blocks] = v[n];
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library links no driver library directly)
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// [B][rows][H * 128] BF16 as a 3-D tensor map with boxes of 64 dims x 128
// rows x 1, swizzled by 128 bytes (rows past `rows` read as zeros)
bool make_map(CUtensorMap* m, const __nv_bfloat16* base, int H, int rows, int B) {
  const EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)H * 128, (cuuint64_t)rows, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)H * 256, (cuuint64_t)rows * H * 256};
  const cuuint32_t box[3] = {64, (cuuint32_t)kTM, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_score_chunk(const qsa_dims& d, int n_chunk, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                               const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s) {
  static_assert(kTM == kTN && kPThreads == kTN, "one query per thread when reading positions");
  alignas(64) CUtensorMap tm_kc, tm_q;
  if (!make_map(&tm_kc, kc, d.n_idx_heads, d.max_blocks, d.batch) ||
      !make_map(&tm_q, q_idx, d.n_idx_heads, n_chunk, d.batch))
    return cudaErrorInvalidValue;
  // one stage when there is one index head (three CTAs per SM), else two
  // (the next head's copy overlaps this head's MMAs)
  const int stages = d.n_idx_heads > 1 ? 2 : 1;
  const size_t smem = (size_t)stages * kStageBytes + 1024;
  static DeviceSlots smem_slots;
  if (const cudaError_t e = smem_slots.raise_smem(score_chunk_kernel, smem); e != cudaSuccess) return e;
  const dim3 grid((d.max_blocks + kTM - 1) / kTM, (n_chunk + kTN - 1) / kTN, d.batch);
  return launch_k(score_chunk_kernel, grid, dim3(kPThreads), smem, s, false, tm_kc, tm_q, q_pos, scores, err,
                  n_chunk, d.n_idx_heads, d.max_blocks, stages);
}

}  // namespace qsa
