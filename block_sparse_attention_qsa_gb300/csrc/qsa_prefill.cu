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
// Design (Blackwell tensor cores). Tiles of 128 blocks x 128 queries of one
// request. For each index head, TMA copies the tile's 128 compressed-key rows
// and 128 query rows (256 bytes each) into shared memory in the 128-byte
// swizzled layout the tensor core reads, completing an mbarrier; tcgen05.mma
// (M = 128 blocks, N = 128 queries, K = 16 per instruction) accumulates into
// FP32 tensor memory (TMEM: lane = block, column = query), and tcgen05.commit
// hands the accumulator to the epilogue, which reads it back with tcgen05.ld:
// each warp owns 32 TMEM lanes (blocks), so for every query a warp stores 32
// consecutive scores (128 contiguous bytes) of that query's row, the causal
// ones only. One persistent CTA per SM runs the three roles in separate warps
// (copies, MMAs, eight epilogue warps) over a ring of shared-memory stages and
// two TMEM accumulators, so one tile's stores overlap the next tile's copies
// and MMAs. Scores are 4 bytes per (query, block) against 0.5 read, so the
// kernel is bound by the score writes, not by the tensor cores.
//
// Every wait (mbarrier phases) is bounded by a clock limit; past it the kernel
// records a timeout in the workspace header, every role stops issuing work,
// the copy warp waits (bounded again) for its copies in flight, and the CTA
// frees its TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kTM = 128;        // blocks per tile (MMA M, TMEM lanes)
constexpr int kTN = 128;        // queries per tile (MMA N, TMEM columns)
constexpr int kAHalf = kTM * 128;          // one 64-dim half of the tile's key rows: 128 rows x 128 B (16 KB)
constexpr int kBHalf = kTN * 128;          // one 64-dim half of the tile's query rows (16 KB)
constexpr int kStageBytes = 2 * kAHalf + 2 * kBHalf;  // keys + queries of one index head (64 KB)
constexpr uint32_t kTmemCols = kTN;        // FP32 accumulator columns of one tile
constexpr int kAccs = 2;                   // accumulators in TMEM (2 x 128 columns)
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

// 32 consecutive FP32 accumulator columns of this thread's TMEM lane; the
// values are usable after tcgen05.wait::ld
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, float (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]),
        "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]),
        "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]),
        "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
      : "r"(taddr)
      : "memory");
}

// Causal extent of one tile's queries, computed by a whole warp (every lane
// gets the result): the largest and smallest number of full blocks any of the
// queries i0..i0+127 sees (absent or bad positions count as 0 blocks).
struct TileNf {
  int mx, mn;
};
__device__ __forceinline__ TileNf tile_nf(const int32_t* q_pos, int r, int i0, int n_chunk, int max_blocks) {
  const int lane = threadIdx.x & 31;
  int mx = 0, mn = 0x7fffffff;
#pragma unroll
  for (int k = 0; k < kTN / 32; ++k) {
    const int i = i0 + 32 * k + lane;
    int nf = 0;
    if (i < n_chunk) {
      const int p = q_pos[(size_t)r * n_chunk + i];
      if (p >= 0 && n_full_of(p) <= max_blocks) nf = n_full_of(p);
    }
    mx = max(mx, nf);
    mn = min(mn, nf);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  return {mx, mn};
}

// Persistent, warp-specialised: warp 0 issues the TMA copies into a ring of
// kStages shared-memory stages (one index head of one tile each), warp 1 the
// MMAs into kAccs TMEM accumulators in turn, warps 2-9 drain finished
// accumulators to the score rows (two warps per 32 TMEM lanes, each taking
// every other 32-query chunk of the 128 query columns), so a tile's stores
// overlap the next tile's copies and MMAs. Tiles are (request, 128 queries,
// 128 blocks), blocks fastest, taken round-robin by the CTAs (measured: tiles
// of 64 queries, with four accumulators, were slower). A tile whose blocks no query of it sees is
// skipped by every role alike, except a CTA's first tile, whose copies are
// issued before the causal extents are known (its stores are then masked
// off). The causal extent of each of the CTA's first kNfTable tiles is
// computed once, by all warps, while that first tile's copies are in flight.
constexpr int kStages = 3;
constexpr int kEpiWarps = 8;
constexpr int kRoleThreads = 32 * (2 + kEpiWarps);
constexpr int kNfTable = 128;

__global__ void __launch_bounds__(kRoleThreads, 1) score_chunk_kernel(const __grid_constant__ CUtensorMap tm_kc,
                                                                    const __grid_constant__ CUtensorMap tm_q,
                                                                    const int32_t* __restrict__ q_pos,
                                                                    float* __restrict__ scores, int32_t* err,
                                                                    int n_chunk, int H, int max_blocks, int B,
                                                                    int withhold) {
  extern __shared__ uint8_t psm_raw[];
  // stage buffers at a 1,024-byte boundary (the swizzle pattern repeats every 1,024 bytes)
  uint8_t* psm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(psm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], acc_full[kAccs], acc_empty[kAccs];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int2 s_nf[kNfTable];  // (largest, smallest) causal blocks of the queries of the CTA's k-th tile
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int BT = (max_blocks + kTM - 1) / kTM, QT = (n_chunk + kTN - 1) / kTN;
  const long long n_tiles = (long long)B * QT * BT;

  if (warp == 1) {  // the MMA warp owns the accumulators (kAccs x 64 columns)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kAccs * kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < kAccs; ++a) {
      mbar_init(smem_u32(&acc_full[a]), 1);
      mbar_init(smem_u32(&acc_empty[a]), kEpiWarps);  // one arrival per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // tile t = blockIdx.x + k gridDim.x -> (request, query tile, block tile)
  auto tile_of = [&](long long t, int& r, int& qt, int& bt) {
    bt = (int)(t % BT);
    qt = (int)((t / BT) % QT);
    r = (int)(t / ((long long)BT * QT));
  };
  // copies of index head h of tile (r, qt, bt) into ring stage `stage`
  auto issue = [&](int stage, int h, int r, int qt, int bt) {
    const uint32_t base = smem_u32(psm + stage * kStageBytes);
    const uint32_t bar = smem_u32(&full_bar[stage]);
    mbar_expect_tx(bar, kStageBytes);
    tma_load_3d(base, &tm_kc, h * 128, bt * kTM, r, bar);
    tma_load_3d(base + kAHalf, &tm_kc, h * 128 + 64, bt * kTM, r, bar);
    tma_load_3d(base + 2 * kAHalf, &tm_q, h * 128, qt * kTN, r, bar);
    tma_load_3d(base + 2 * kAHalf + kBHalf, &tm_q, h * 128 + 64, qt * kTN, r, bar);
  };
  // the first tile's first heads go out at once (its ring stages are fresh).
  // withhold (the failure-detection test only): CTA 0 leaves its first copy
  // out, so the MMA warp's wait for it runs into the clock limit
  const int pre = min(H, kStages);
  const bool held = withhold && blockIdx.x == 0;
  if (tid == 0 && (long long)blockIdx.x < n_tiles) {
    int r, qt, bt;
    tile_of(blockIdx.x, r, qt, bt);
    for (int h = held ? 1 : 0; h < pre; ++h) issue(h, h, r, qt, bt);
  }
  for (int k = warp; k < kNfTable; k += kRoleThreads / 32) {
    const long long t = blockIdx.x + (long long)k * gridDim.x;
    if (t >= n_tiles) break;
    int r, qt, bt;
    tile_of(t, r, qt, bt);
    const TileNf tn = tile_nf(q_pos, r, qt * kTN, n_chunk, max_blocks);
    if (lane == 0) s_nf[k] = make_int2(tn.mx, tn.mn);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  // causal extent of the CTA's k-th tile (a whole warp calls this)
  auto nf_of = [&](int k, int r, int qt) -> TileNf {
    if (k < kNfTable) {
      const int2 v = s_nf[k];
      return {v.x, v.y};
    }
    return tile_nf(q_pos, r, qt * kTN, n_chunk, max_blocks);
  };
  // whether the copy and MMA roles process the CTA's k-th tile (and the
  // epilogue drains it): some query sees its blocks, or it is the first tile
  auto live = [&](int k, int bt, const TileNf& tn) { return k == 0 || bt * kTM < tn.mx; };

  // bounded wait that also gives up once another role has
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    while (!mbar_try_wait(a, parity)) {
      if (s_abort) return false;
      if (clock64() - t0 > kWaitCycles) {
        s_abort = 1;
        record_error(err, kErrTimeout, 0, 0, warp);
        return false;
      }
    }
    return true;
  };

  if (warp == 0) {
    // ---- TMA producer ----
    // the stages the first tile's early copies took
    int stage = pre % kStages;
    uint32_t phase = pre == kStages ? 1u : 0u;
    bool issued[kStages] = {};
    uint32_t issued_par[kStages] = {};
    for (int s = 0; s < pre; ++s) issued[s] = (long long)blockIdx.x < n_tiles && !(held && s == 0);
    int k = 0;
    for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++k) {
      int r, qt, bt;
      tile_of(t, r, qt, bt);
      if (!live(k, bt, nf_of(k, r, qt))) continue;
      bool ok = true;
      for (int h = k == 0 ? pre : 0; h < H && ok; ++h) {
        if (lane == 0) {
          ok = wait(&empty_bar[stage], phase ^ 1u);
          if (ok) {
            issue(stage, h, r, qt, bt);
            issued[stage] = true;
            issued_par[stage] = phase;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    if (lane == 0 && s_abort) {
      // copies still in flight land before the CTA leaves (bounded)
      for (int s = 0; s < kStages; ++s) {
        if (!issued[s]) continue;
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(&full_bar[s]), issued_par[s]) && clock64() - t0 < kWaitCycles) {
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    int k = 0;
    for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++k) {
      int r, qt, bt;
      tile_of(t, r, qt, bt);
      if (!live(k, bt, nf_of(k, r, qt))) continue;
      bool ok = true;
      if (lane == 0) {
        ok = wait(&acc_empty[acc], acc_phase ^ 1u);  // the epilogue has drained this accumulator
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + (uint32_t)(acc * kTmemCols);
        for (int h = 0; h < H && ok; ++h) {
          ok = wait(&full_bar[stage], phase);
          if (!ok) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t a0 = smem_u32(psm + stage * kStageBytes), bq = a0 + 2 * kAHalf;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // 16 dims per instruction: 4 steps of 32 bytes in each 64-dim half
            const uint32_t step = (uint32_t)(kk & 3) * 32u;
            mma_bf16_tmem(d, sw128_desc(a0 + (uint32_t)(kk >> 2) * kAHalf + step),
                          sw128_desc(bq + (uint32_t)(kk >> 2) * kBHalf + step), h > 0 || kk > 0);
          }
          mma_commit(smem_u32(&empty_bar[stage]));  // the stage is free once these MMAs have read it
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(smem_u32(&acc_full[acc]));  // the accumulator is complete
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (++acc == kAccs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. blocks
    // b0 + 32 (w % 4) + lane, and the 32-query column chunks half, half + 2 ----
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    const size_t row = (size_t)max_blocks;
    int k = 0;
    for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++k) {
      int r, qt, bt;
      tile_of(t, r, qt, bt);
      const int b0 = bt * kTM, i0 = qt * kTN;
      if (bt == 0 && warp == 2) {  // report bad positions once per query
        for (int kk = 0; kk < kTN / 32; ++kk) {
          const int i = i0 + 32 * kk + lane;
          if (i < n_chunk) {
            const int p = q_pos[(size_t)r * n_chunk + i];
            if (p < 0 || n_full_of(p) > max_blocks) record_error(err, kErrQueryPos, r, i, p);
          }
        }
      }
      const TileNf tn = nf_of(k, r, qt);
      if (!live(k, bt, tn)) continue;
      if (!wait(&acc_full[acc], acc_phase)) break;
      __syncwarp();
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int b = b0 + quarter * 32 + lane;
      const bool whole = b0 + kTM <= tn.mn && i0 + kTN <= n_chunk;  // every score of the tile is causal
      for (int c0 = 32 * half; c0 < kTN; c0 += 64) {
        if (i0 + c0 >= n_chunk) break;  // warp-uniform
        float v[32];
        tmem_ld32_nowait(tmem + (uint32_t)(acc * kTmemCols) + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        float* d0 = scores + ((size_t)r * n_chunk + i0 + c0) * row + b;
        if (whole) {
#pragma unroll
          for (int n = 0; n < 32; ++n) d0[(size_t)n * row] = v[n];
        } else {
          // this lane's query c0 + lane: its causal blocks, shared by shuffles
          const int i = i0 + c0 + lane;
          int nf = 0;
          if (i < n_chunk) {
            const int p = q_pos[(size_t)r * n_chunk + i];
            if (p >= 0 && n_full_of(p) <= max_blocks) nf = n_full_of(p);
          }
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            const int nfn = __shfl_sync(0xffffffffu, nf, n);
            if (b < nfn) d0[(size_t)n * row] = v[n];  // nfn is 0 past the chunk's last query
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&acc_empty[acc])) : "memory");
      if (++acc == kAccs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kAccs * kTmemCols) : "memory");
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

// [B][rows][H * 128] BF16 as a 3-D tensor map with boxes of 64 dims x
// box_rows rows x 1, swizzled by 128 bytes (rows past `rows` read as zeros)
bool make_map(CUtensorMap* m, const __nv_bfloat16* base, int H, int rows, int B, int box_rows) {
  const EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)H * 128, (cuuint64_t)rows, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)H * 256, (cuuint64_t)rows * H * 256};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_score_chunk(const qsa_dims& d, int n_chunk, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                               const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s,
                               bool withhold_first_copy) {
  alignas(64) CUtensorMap tm_kc, tm_q;
  if (!make_map(&tm_kc, kc, d.n_idx_heads, d.max_blocks, d.batch, kTM) ||
      !make_map(&tm_q, q_idx, d.n_idx_heads, n_chunk, d.batch, kTN))
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)kStages * kStageBytes + 1024;
  static DeviceSlots smem_slots;
  if (const cudaError_t e = smem_slots.raise_smem(score_chunk_kernel, smem); e != cudaSuccess) return e;
  // one persistent CTA per SM (its shared-memory ring and 256 TMEM columns
  // leave room for no second one), never more CTAs than tiles
  const long long tiles = (long long)d.batch * ((n_chunk + kTN - 1) / kTN) * ((d.max_blocks + kTM - 1) / kTM);
  const int grid = (int)std::min<long long>(tiles, device_sm_count());
  return launch_k(score_chunk_kernel, dim3(grid), dim3(kRoleThreads), smem, s, false, tm_kc, tm_q, q_pos, scores,
                  err, n_chunk, d.n_idx_heads, d.max_blocks, d.batch, withhold_first_copy ? 1 : 0);
}

}  // namespace qsa
