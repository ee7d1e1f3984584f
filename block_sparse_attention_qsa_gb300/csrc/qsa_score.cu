// Compressed index keys and FP32 block scores.
//
// Scoring follows the pages' QSA selection pipeline (arex-research.com,
// section "四类优化", bullets 1-2): every full 4-token block of a request is
// scored against each of its (up to 4) verify queries, and the compressed
// keys are loaded once per request and shared by all queries.
//
// GB300 design: the path is a stream over the compressed keys (256 B per
// block per index head), so the kernel is written for HBM bandwidth, not for
// tensor cores. Each warp owns a contiguous range of (request, block-pair)
// units, balanced over the whole batch. A lane loads one 16-byte chunk (8 BF16
// dims) per block straight into registers with no-L1-allocate 128-bit loads,
// widens it with shifts (BF16 is the top half of an FP32) and multiplies it
// against the 4 queries' matching dims with packed FP32 FMAs (FFMA2). The key
// tile is thereby shared by the 4 queries in registers rather than shared
// memory. A reduce-scatter butterfly over the lanes of a block then leaves
// each query's total on its own lanes, so every query costs one shuffle chain.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// compressed keys: kc[r][b] = bf16( (((k0 + k1) + k2) + k3) * 0.25 ), FP32
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) compress_kernel(const uint4* __restrict__ idx_keys,
                                                       const int32_t* __restrict__ q_pos,
                                                       const int32_t* __restrict__ block_lo,
                                                       uint4* __restrict__ kc, int32_t* err,
                                                       int n_q, int H, int max_blocks) {
  const int r = blockIdx.y;
  __shared__ int s_lo, s_hi;
  if (threadIdx.x == 0) {
    int pmax = -1;
    for (int j = 0; j < n_q; ++j) {
      const int p = q_pos[r * n_q + j];
      if (p < 0 || n_full_of(p) > max_blocks) {
        if (blockIdx.x == 0) record_error(err, kErrQueryPos, r, j, p);
      } else {
        pmax = max(pmax, p);
      }
    }
    s_hi = pmax < 0 ? 0 : n_full_of(pmax);
    s_lo = block_lo ? max(0, block_lo[r]) : 0;
  }
  __syncthreads();
  const int cpb = H * 16;  // 16-byte chunks per token row
  const long long total = (long long)max(0, s_hi - s_lo) * cpb;
  const uint4* src_r = idx_keys + (size_t)r * max_blocks * kBlock * cpb;
  uint4* dst_r = kc + (size_t)r * max_blocks * cpb;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = s_lo + (int)(i / cpb);
    const int c = (int)(i % cpb);
    const uint4* src = src_r + (size_t)b * kBlock * cpb + c;
    const uint4 k0 = src[0], k1 = src[cpb], k2 = src[2 * cpb], k3 = src[3 * cpb];
    const uint32_t* w0 = &k0.x;
    const uint32_t* w1 = &k1.x;
    const uint32_t* w2 = &k2.x;
    const uint32_t* w3 = &k3.x;
    uint4 o;
    uint32_t* ow = &o.x;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 a = bf16x2_to_f2(w0[w]), b1 = bf16x2_to_f2(w1[w]);
      const float2 c2 = bf16x2_to_f2(w2[w]), d = bf16x2_to_f2(w3[w]);
      const float lo = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(a.x, b1.x), c2.x), d.x), 0.25f);
      const float hi = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(a.y, b1.y), c2.y), d.y), 0.25f);
      const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
      ow[w] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst_r[(size_t)b * cpb + c] = o;
  }
}

// ---------------------------------------------------------------------------
// scores
// ---------------------------------------------------------------------------
template <int H>
struct ScoreGeom {
  static constexpr int G = (H % 2 == 0) ? 32 : 16;  // lanes covering one block
  static constexpr int C = H * 16 / G;              // 16-B chunks per lane per block
  static constexpr int BPW = 32 / G;                // blocks per warp step (a "unit")
  static constexpr int UNR = 8 / C;                 // units in flight per lane
};

// Reduce a[0..NQ) over the G lanes of a block; returns the total of query
// `q` on every lane, and `q` depends on the lane (reduce-scatter).
template <int G, int NQ>
__device__ __forceinline__ float reduce_scatter(const float (&a)[NQ], int lane, int& q) {
  if constexpr (NQ == 4) {
    constexpr int B1 = G / 2, B2 = G / 4;
    const bool h1 = lane & B1;
    float k0 = h1 ? a[2] : a[0], k1 = h1 ? a[3] : a[1];
    const float s0 = h1 ? a[0] : a[2], s1 = h1 ? a[1] : a[3];
    k0 += __shfl_xor_sync(kFull, s0, B1);
    k1 += __shfl_xor_sync(kFull, s1, B1);
    const bool h2 = lane & B2;
    float k = h2 ? k1 : k0;
    const float s = h2 ? k0 : k1;
    k += __shfl_xor_sync(kFull, s, B2);
#pragma unroll
    for (int o = B2 / 2; o >= 1; o >>= 1) k += __shfl_xor_sync(kFull, k, o);
    q = (h1 ? 2 : 0) + (h2 ? 1 : 0);
    return k;
  } else if constexpr (NQ == 2) {
    constexpr int B1 = G / 2;
    const bool h1 = lane & B1;
    float k = h1 ? a[1] : a[0];
    const float s = h1 ? a[0] : a[1];
    k += __shfl_xor_sync(kFull, s, B1);
#pragma unroll
    for (int o = B1 / 2; o >= 1; o >>= 1) k += __shfl_xor_sync(kFull, k, o);
    q = h1 ? 1 : 0;
    return k;
  } else {
    float k = a[0];
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) k += __shfl_xor_sync(kFull, k, o);
    q = 0;
    return k;
  }
}

template <int H, int NQ>
__global__ void __launch_bounds__(256) score_kernel(const __nv_bfloat16* __restrict__ q_idx,
                                                    const uint4* __restrict__ kc,
                                                    const int32_t* __restrict__ q_pos,
                                                    float* __restrict__ scores, int32_t* err,
                                                    int B, int n_q, int max_blocks) {
  using Geo = ScoreGeom<H>;
  constexpr int G = Geo::G, C = Geo::C, BPW = Geo::BPW, UNR = Geo::UNR;
  constexpr int CPB = H * 16;  // 16-B chunks per block
  extern __shared__ int s_off[];  // [B + 1] first unit of each request

  pdl_wait();  // no-op unless launched as a dependent
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    int carry = 0;
    for (int base = 0; base < B; base += 32) {
      const int r = base + lane;
      int units = 0;
      if (r < B) {
        int nb = 0;
        for (int j = 0; j < n_q; ++j) {
          const int p = q_pos[r * n_q + j];
          if (p < 0 || n_full_of(p) > max_blocks) {
            if (blockIdx.x == 0) record_error(err, kErrQueryPos, r, j, p);
          } else {
            nb = max(nb, n_full_of(p));
          }
        }
        units = (nb + BPW - 1) / BPW;
      }
      int v = units;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
      }
      if (r < B) s_off[r] = carry + v - units;
      carry += __shfl_sync(kFull, v, 31);
    }
    if (lane == 0) s_off[B] = carry;
  }
  __syncthreads();

  const int U = s_off[B];
  const long long warps_total = (long long)gridDim.x * (blockDim.x / 32);
  const long long gw = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int u = (int)(U * gw / warps_total);
  const int u_end = (int)(U * (gw + 1) / warps_total);

  // request holding unit u: last r with s_off[r] <= u
  int lo = 0, hi = B;  // invariant s_off[lo] <= u < s_off[hi] (when u < U)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] <= u) lo = mid; else hi = mid;
  }
  int r = lo;

  const int slot = (G == 16) ? (lane >> 4) : 0;  // block within the unit
  int chunk[C];
#pragma unroll
  for (int i = 0; i < C; ++i) chunk[i] = (G == 16) ? i * 16 + (lane & 15) : i * 32 + lane;

  while (u < u_end) {
    while (s_off[r + 1] <= u) ++r;
    const int seg_end = min(u_end, s_off[r + 1]);
    const int u0 = s_off[r];

    // this request's queries, widened to FP32 pairs, in the lane's dims
    float2 qf[NQ][C][4];
    int nbq[NQ];
    int nb_r = 0;
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      int p = -1;
      if (j < n_q) p = q_pos[r * n_q + j];
      const bool ok = p >= 0 && n_full_of(p) <= max_blocks;
      nbq[j] = ok ? n_full_of(p) : 0;
      nb_r = max(nb_r, nbq[j]);
#pragma unroll
      for (int i = 0; i < C; ++i) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (j < n_q)
          v = *reinterpret_cast<const uint4*>(q_idx + ((size_t)(r * n_q + j) * CPB + chunk[i]) * 8);
        qf[j][i][0] = bf16x2_to_f2(v.x);
        qf[j][i][1] = bf16x2_to_f2(v.y);
        qf[j][i][2] = bf16x2_to_f2(v.z);
        qf[j][i][3] = bf16x2_to_f2(v.w);
      }
    }
    const uint4* kc_r = kc + (size_t)r * max_blocks * CPB;
    float* sc_r = scores + (size_t)r * n_q * max_blocks;

    for (; u < seg_end; u += UNR) {
      uint4 kv[UNR][C];
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const int b = (u + k - u0) * BPW + slot;
        const bool ok = (u + k < seg_end) && (b < nb_r);
#pragma unroll
        for (int i = 0; i < C; ++i)
          kv[k][i] = ok ? ld_stream(kc_r + (size_t)b * CPB + chunk[i]) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        float2 acc[NQ];
#pragma unroll
        for (int j = 0; j < NQ; ++j) acc[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < C; ++i) {
          const uint32_t* w = &kv[k][i].x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kf = bf16x2_to_f2(w[e]);
#pragma unroll
            for (int j = 0; j < NQ; ++j) acc[j] = __ffma2_rn(kf, qf[j][i][e], acc[j]);
          }
        }
        float a[NQ];
#pragma unroll
        for (int j = 0; j < NQ; ++j) a[j] = acc[j].x + acc[j].y;
        int qsel;
        const float tot = reduce_scatter<G, NQ>(a, lane, qsel);
        const int b = (u + k - u0) * BPW + slot;
        constexpr int kStoreMask = (NQ == 4) ? (G / 4 - 1) : (NQ == 2 ? (G / 2 - 1) : (G - 1));
        int nb_sel = 0;
#pragma unroll
        for (int j = 0; j < NQ; ++j) nb_sel = (j == qsel) ? nbq[j] : nb_sel;
        if ((lane & kStoreMask) == 0 && (u + k < seg_end) && b < nb_sel)
          sc_r[(size_t)qsel * max_blocks + b] = tot;
      }
    }
    u = seg_end;  // the unrolled loop may step past the end of this request's units
  }
  pdl_trigger();
}

template <int H, int NQ>
cudaError_t launch_score_t(const qsa_dims& d, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                           const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s,
                           bool pdl) {
  auto kern = score_kernel<H, NQ>;
  const size_t smem = (size_t)(d.batch + 1) * sizeof(int);
  static int occ_cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int occ = dev < 64 ? occ_cache[dev] : 0;
  if (occ == 0) {
    if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 256, smem);
    if (occ < 1) occ = 1;
    if (dev < 64 && smem <= 48 * 1024) occ_cache[dev] = occ;
  }
  // upper bound of the work, in units, to avoid launching idle warps
  using Geo = ScoreGeom<H>;
  const long long units_ub = (long long)d.batch * ((d.max_blocks + Geo::BPW - 1) / Geo::BPW);
  long long warps = (long long)device_sm_count() * occ * 8;
  const long long want = (units_ub + 3) / 4;  // at least ~4 units per warp
  if (want < warps) warps = want;
  const int grid = (int)((warps + 7) / 8 > 0 ? (warps + 7) / 8 : 1);
  return launch_k(kern, dim3(grid), dim3(256), smem, s, pdl, q_idx,
                  reinterpret_cast<const uint4*>(kc), q_pos, scores, err, d.batch, d.n_q,
                  d.max_blocks);
}

template <int H>
cudaError_t launch_score_h(const qsa_dims& d, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                           const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s,
                           bool pdl) {
  if (d.n_q == 1) return launch_score_t<H, 1>(d, q_idx, kc, q_pos, scores, err, s, pdl);
  if (d.n_q == 2) return launch_score_t<H, 2>(d, q_idx, kc, q_pos, scores, err, s, pdl);
  return launch_score_t<H, 4>(d, q_idx, kc, q_pos, scores, err, s, pdl);
}

}  // namespace

cudaError_t launch_compress(const qsa_dims& d, const __nv_bfloat16* idx_keys, const int32_t* q_pos,
                            const int32_t* block_lo, __nv_bfloat16* kc, int32_t* err,
                            cudaStream_t s) {
  const long long chunks = (long long)d.max_blocks * d.n_idx_heads * 16;
  long long gx = (chunks + 255) / 256;
  const long long cap = (long long)device_sm_count() * 8;
  if (gx > cap) gx = cap;
  if (gx < 1) gx = 1;
  return launch_k(compress_kernel, dim3((unsigned)gx, d.batch), dim3(256), 0, s, false,
                  reinterpret_cast<const uint4*>(idx_keys), q_pos, block_lo,
                  reinterpret_cast<uint4*>(kc), err, d.n_q, d.n_idx_heads, d.max_blocks);
}

cudaError_t launch_score(const qsa_dims& d, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                         const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s,
                         bool pdl) {
  switch (d.n_idx_heads) {
    case 1: return launch_score_h<1>(d, q_idx, kc, q_pos, scores, err, s, pdl);
    case 2: return launch_score_h<2>(d, q_idx, kc, q_pos, scores, err, s, pdl);
    case 3: return launch_score_h<3>(d, q_idx, kc, q_pos, scores, err, s, pdl);
    default: return launch_score_h<4>(d, q_idx, kc, q_pos, scores, err, s, pdl);
  }
}

}  // namespace qsa
