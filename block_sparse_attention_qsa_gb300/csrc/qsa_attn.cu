// Sparse attention over the selected positions (decode and MTP verify).
//
// The pages (arex-research.com, section "四类优化", bullet 3) describe a
// sparse-attention kernel for the model's own attention geometry that handles
// plain decode and MTP verification with a BF16 query and a BF16 or FP8-E4M3
// KV cache; 10100.com ("第一处") adds that the selected history must then be
// found in the cache. The geometry here is theirs as this library reads it:
// 16 query heads over 2 KV heads of dim 128, a paged cache of 64-token pages.
//
// Design. One CTA of 4 warps per (request, query, KV head, split of the
// selection buffer). The CTA resolves its positions to cache rows through the
// page table once; from then on every warp works alone on 8 positions of
// each 32-position tile. The selected K/V rows are random 256-byte (BF16) or
// 128-byte (FP8) rows, so the kernel is a gather: measured on GB300, 128-bit
// loads straight into registers, with each warp reading whole rows, sustain a
// much higher share of HBM bandwidth for such gathers than staging through
// shared memory. So K and V never touch shared memory:
//
//  * S^T = K Q^T on the tensor cores (mma.sync m16n8k16, FP32 accumulate):
//    the warp's 8 positions are the M rows, the KV group's 8 query heads the
//    N columns. A lane's 16-byte loads of K rows are its A fragments directly,
//    because the head dim is visited in a lane-dependent order that Q's B
//    fragments follow too (a dot product does not depend on the order of its
//    terms).
//  * softmax is online, in FP32, in the exp2 domain, per head;
//  * O^T = V^T P^T: V rows loaded the same way are turned into A fragments
//    with movmatrix (an in-register 8x8 transpose), P^T is the softmax tile
//    transposed the same way, and the output's dim order (permuted by the V
//    loads) is undone when it is written.
//
// FP8 rows are widened to FP16 in registers (exact for E4M3); K's scale
// folds into the softmax scale and V's into the output. The warps' softmax
// states merge through shared memory; splits write (max, sum, acc) partials
// to the workspace and the last CTA of a (request, query, KV head) to arrive,
// counted by an atomic ticket, merges them and resets the ticket, so there is
// no spin-wait anywhere.
#include <cuda_fp8.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kWarpPos = 8;     // positions per warp step
constexpr int kTile = 4 * kWarpPos;  // positions per CTA step: 4 warps
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 8x8 transpose of 16-bit elements held one pair per lane (lane 4g + c holds
// row g, columns 2c and 2c+1).
__device__ __forceinline__ uint32_t movt(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// two E4M3 codes (low byte first) -> FP16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// BF16 pair -> FP16 pair (Q of the FP8 path)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) {
  return pack2<true>(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Register layout of one lane's share of a 128-dim row, for lane = 4g + c.
//   BF16 rows (256 B): 4 loads of 16 B at chunks c, c+4, c+8, c+12 -> 16
//   pairs; pair (i, e) holds dims 8(c + 4i) + 2e + {0,1}.
//   FP8 rows (128 B): 2 loads of 16 B at chunks c, c+4 -> 16 pairs after
//   widening; pair (i, e) holds dims 16(c + 4i) + 2e + {0,1}.
// Pair p = 4i + e (BF16) or 8i + e (FP8) is the lane's p-th pair.
//   K: k-step ks (16 of the 128 dims) uses pairs 2ks and 2ks + 1 of a row.
//   V: the 8x8 block k (logical dims 8k..8k+7) holds pair k of each row.
template <bool FP8>
struct RowRegs {
  static constexpr int kLoads = FP8 ? 2 : 4;
  static constexpr int kRowBytes = FP8 ? 128 : 256;
  uint32_t pr[16];  // 16 pairs of 16-bit values

  __device__ __forceinline__ void load(const uint8_t* row, int c, bool ok) {
    uint4 raw[kLoads];
#pragma unroll
    for (int i = 0; i < kLoads; ++i) raw[i] = ok ? ldg16(row + (c + 4 * i) * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (FP8) {
          pr[8 * i + 2 * e] = e4m3x2_to_h2(w[e]);
          pr[8 * i + 2 * e + 1] = e4m3x2_to_h2(w[e] >> 16);
        } else {
          pr[4 * i + e] = w[e];
        }
      }
    }
  }
};

// physical head dim of logical output dim L (the V block k = L / 8 holds
// column j = L % 8 = 2c + f from lane column c)
template <bool FP8>
__device__ __forceinline__ int phys_dim(int L) {
  const int k = L >> 3, j = L & 7, c = j >> 1, f = j & 1;
  if constexpr (FP8) return 16 * (c + 4 * (k >> 3)) + 2 * (k & 7) + f;
  return 8 * (c + 4 * (k >> 2)) + 2 * (k & 3) + f;
}

struct AttnArgs {
  const __nv_bfloat16* q;
  const void* k_cache;
  const void* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* page_table;
  const int32_t* sel_pos;
  const int32_t* q_pos;
  __nv_bfloat16* out;
  int32_t* err;
  int32_t* tickets;
  float* partials;
  int n_q, n_kv, page_shift, max_pages, num_pages, width, nsplit, tiles_per_split;
  float sm_scale;
};

size_t attn_smem_bytes(int tiles_per_split) {
  // cache rows of the split's positions + warp merge buffer [4][8][128] + stats
  return (size_t)tiles_per_split * kTile * 4 + 4 * kGroup * kDim * 4 + 512;
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 4) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  int32_t* s_rows = reinterpret_cast<int32_t*>(smem);                         // [tps * 64]
  float* wacc = reinterpret_cast<float*>(s_rows + a.tiles_per_split * kTile);  // [4][8][128]
  float* s_ml = wacc + 4 * kGroup * kDim;                                      // [4][8] m, [4][8] l, M[8], L[8]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, c4 = lane & 3;
  const int unit = blockIdx.x / a.nsplit, split = blockIdx.x % a.nsplit;
  const int g = unit % a.n_kv, row = unit / a.n_kv;
  const int r = row / a.n_q;
  const int n_q_heads = a.n_kv * kGroup;

  // ---- prologue independent of the previous kernel: Q fragments, scales ----
  // B fragment of k-step ks for head gq: the lane's pairs 2ks, 2ks + 1 of Q's row
  uint32_t qb[16];
  {
    const __nv_bfloat16* qrow = a.q + ((size_t)row * n_q_heads + g * kGroup + gq) * kDim;
    if constexpr (FP8) {
      // dims 16(c + 4i) .. +15 for i = 0, 1 (32 bytes of BF16 each)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 lo = *reinterpret_cast<const uint4*>(qrow + 16 * (c4 + 4 * i));
        const uint4 hi = *reinterpret_cast<const uint4*>(qrow + 16 * (c4 + 4 * i) + 8);
        qb[8 * i + 0] = bf2_to_h2(lo.x);
        qb[8 * i + 1] = bf2_to_h2(lo.y);
        qb[8 * i + 2] = bf2_to_h2(lo.z);
        qb[8 * i + 3] = bf2_to_h2(lo.w);
        qb[8 * i + 4] = bf2_to_h2(hi.x);
        qb[8 * i + 5] = bf2_to_h2(hi.y);
        qb[8 * i + 6] = bf2_to_h2(hi.z);
        qb[8 * i + 7] = bf2_to_h2(hi.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + 8 * (c4 + 4 * i));
        qb[4 * i + 0] = v.x;
        qb[4 * i + 1] = v.y;
        qb[4 * i + 2] = v.z;
        qb[4 * i + 3] = v.w;
      }
    }
  }
  const float kscale = FP8 ? a.k_scale[g] : 1.f;
  const float vscale = FP8 ? a.v_scale[g] : 1.f;
  const float scale_log2 = a.sm_scale * kscale * kLog2e;
  const int p = a.q_pos[row];
  const bool p_ok = p >= 0 && (p >> a.page_shift) < a.max_pages;
  if (!p_ok && split == 0 && tid == 0 && g == 0) record_error(a.err, kErrQueryPos, r, row % a.n_q, p);

  pdl_wait();  // sel_pos comes from the selection kernel

  // ---- resolve this split's positions to cache rows ----
  const int pos0 = split * a.tiles_per_split * kTile;
  const int npos = min(a.tiles_per_split * kTile, a.width - pos0);
  __shared__ int s_last;
  if (tid == 0) s_last = -1;
  __syncthreads();
  int my_last = -1;
  const int32_t* sp = a.sel_pos + (size_t)row * a.width + pos0;
  const int32_t* pt = a.page_table + (size_t)r * a.max_pages;
  const int page_mask = (1 << a.page_shift) - 1;
  for (int i = tid; i < a.tiles_per_split * kTile; i += kThreads) {
    int ri = -1;
    if (i < npos && p_ok) {
      const int t = sp[i];
      if (t > p) {
        if (g == 0) record_error(a.err, kErrSelPos, r, row % a.n_q, t);
      } else if (t >= 0) {
        const int page = pt[t >> a.page_shift];
        if (page < 0 || page >= a.num_pages) {
          if (g == 0) record_error(a.err, kErrPage, r, row % a.n_q, page);
        } else {
          ri = (page * a.n_kv + g) * (page_mask + 1) + (t & page_mask);
          my_last = i;
        }
      }
    }
    s_rows[i] = ri;
  }
  if (my_last >= 0) atomicMax(&s_last, my_last);
  __syncthreads();
  const int ntiles = (s_last + kTile) / kTile;  // tiles holding a valid position

  // ---- per warp: 8 positions of every tile ----
  // S^T uses A rows 0..7 (rows 8..15 are zero) and O^T uses k = 0..7 of each
  // mma: half the tensor work is idle, which costs nothing here, and it halves
  // the K/V registers so that 16 warps per SM keep gathers in flight.
  using RR = RowRegs<FP8>;
  const uint8_t* kbase = static_cast<const uint8_t*>(a.k_cache);
  const uint8_t* vbase = static_cast<const uint8_t*>(a.v_cache);
  float m_run[2] = {kNegInf, kNegInf}, l_run[2] = {0.f, 0.f};  // heads 2c4, 2c4 + 1
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  RR kr, vr;  // row gq of the warp's 8 positions
  int ri = -1;
  if (ntiles > 0) {
    ri = s_rows[warp * kWarpPos + gq];
    kr.load(kbase + (size_t)max(ri, 0) * RR::kRowBytes, c4, ri >= 0);
    vr.load(vbase + (size_t)max(ri, 0) * RR::kRowBytes, c4, ri >= 0);
  }
  for (int t = 0; t < ntiles; ++t) {
    // S^T (8 positions x 8 heads)
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) mma16816<FP8>(s, kr.pr[2 * ks], 0u, kr.pr[2 * ks + 1], 0u, qb[2 * ks], qb[2 * ks + 1]);
    const bool ok = ri >= 0;
    // the next tile's row, and its K loads now that K is consumed
    int nri = -1;
    const bool more = t + 1 < ntiles;
    if (more) {
      nri = s_rows[(t + 1) * kTile + warp * kWarpPos + gq];
      kr.load(kbase + (size_t)max(nri, 0) * RR::kRowBytes, c4, nri >= 0);
    }
    // online softmax; s[0], s[1]: position gq, heads 2c4, 2c4 + 1
    const float x0 = ok ? s[0] * scale_log2 : kNegInf;
    const float x1 = ok ? s[1] * scale_log2 : kNegInf;
    float mA = x0, mB = x1;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mA = fmaxf(mA, __shfl_xor_sync(kFull, mA, o));
      mB = fmaxf(mB, __shfl_xor_sync(kFull, mB, o));
    }
    const float nA = fmaxf(m_run[0], mA), nB = fmaxf(m_run[1], mB);
    const float bA = nA == kNegInf ? 0.f : nA, bB = nB == kNegInf ? 0.f : nB;
    const float alA = exp2f(m_run[0] - bA), alB = exp2f(m_run[1] - bB);
    const float p0 = exp2f(x0 - bA), p1 = exp2f(x1 - bB);
    l_run[0] = l_run[0] * alA + p0;
    l_run[1] = l_run[1] * alB + p1;
    m_run[0] = nA;
    m_run[1] = nB;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      acc[i][0] *= alA;
      acc[i][1] *= alB;
      acc[i][2] *= alA;
      acc[i][3] *= alB;
    }
    // P^T as the B fragment (k = position 0..7, n = head)
    const uint32_t pb = movt(pack2<FP8>(p0, p1));
    // O^T (logical dims x heads) += V^T P^T; m-tile mt = logical dims 16mt .. 16mt + 15
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
      mma16816<FP8>(acc[mt], movt(vr.pr[2 * mt]), movt(vr.pr[2 * mt + 1]), 0u, 0u, pb, 0u);
    if (more) {
      vr.load(vbase + (size_t)max(nri, 0) * RR::kRowBytes, c4, nri >= 0);
      ri = nri;
    }
  }
  // ---- merge the 4 warps ----
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l_run[0] += __shfl_xor_sync(kFull, l_run[0], o);
    l_run[1] += __shfl_xor_sync(kFull, l_run[1], o);
  }
  float* cm = s_ml;       // [4][8]
  float* cl = s_ml + 32;  // [4][8]
  if (gq == 0) {
    cm[warp * 8 + 2 * c4] = m_run[0];
    cm[warp * 8 + 2 * c4 + 1] = m_run[1];
    cl[warp * 8 + 2 * c4] = l_run[0];
    cl[warp * 8 + 2 * c4 + 1] = l_run[1];
  }
  __syncthreads();
  float fac[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int h = 2 * c4 + e;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * 8 + h]);
    fac[e] = exp2f(m_run[e] - (M == kNegInf ? 0.f : M));
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int d0 = phys_dim<FP8>(16 * mt + gq), d1 = phys_dim<FP8>(16 * mt + gq + 8);
    float* w0 = wacc + (warp * 8 + 2 * c4) * kDim;
    float* w1 = w0 + kDim;
    w0[d0] = acc[mt][0] * fac[0];
    w1[d0] = acc[mt][1] * fac[1];
    w0[d1] = acc[mt][2] * fac[0];
    w1[d1] = acc[mt][3] * fac[1];
  }
  float* sM = s_ml + 64;  // [8]
  float* sL = s_ml + 72;  // [8]
  if (tid < 8) {
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * 8 + tid]);
    const float Mb = M == kNegInf ? 0.f : M;
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) L += cl[w * 8 + tid] * exp2f(cm[w * 8 + tid] - Mb);
    sM[tid] = M;
    sL[tid] = L;
  }
  __syncthreads();
  // thread tid owns dim d = tid of all 8 heads
  float o[8];
#pragma unroll
  for (int h = 0; h < 8; ++h)
    o[h] = wacc[(0 * 8 + h) * kDim + tid] + wacc[(1 * 8 + h) * kDim + tid] +
           wacc[(2 * 8 + h) * kDim + tid] + wacc[(3 * 8 + h) * kDim + tid];
  __nv_bfloat16* orow = a.out + ((size_t)row * n_q_heads + g * kGroup) * kDim;
  if (a.nsplit == 1) {
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float l = sL[h];
      orow[h * kDim + tid] = __float2bfloat16_rn(l > 0.f ? o[h] / l * vscale : 0.f);
    }
    pdl_trigger();
    return;
  }

  // ---- split-KV: publish the partial, the last arrival merges ----
  float* part = a.partials + ((size_t)unit * a.nsplit + split) * kPartFloats;
  if (tid < 8) {
    part[tid] = sM[tid];
    part[8 + tid] = sL[tid];
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) part[16 + h * kDim + tid] = o[h];
  __threadfence();
  __syncthreads();
  __shared__ int s_is_last;
  if (tid == 0) s_is_last = (atomicAdd(&a.tickets[unit], 1) == a.nsplit - 1);
  __syncthreads();
  if (!s_is_last) {
    pdl_trigger();
    return;
  }
  __threadfence();
  // every split's (max, sum) at once, then the accumulators 4 splits at a time
  const float* parts = a.partials + (size_t)unit * a.nsplit * kPartFloats;
  float* sm_m = wacc;                       // [nsplit][8] (the merge buffer is free now)
  float* sm_l = wacc + a.nsplit * kGroup;   // [nsplit][8]
  for (int i = tid; i < a.nsplit * kGroup; i += kThreads) {
    const int sidx = i >> 3, h = i & 7;
    sm_m[i] = __ldcg(parts + (size_t)sidx * kPartFloats + h);
    sm_l[i] = __ldcg(parts + (size_t)sidx * kPartFloats + kGroup + h);
  }
  __syncthreads();
  if (tid < kGroup) {
    float Ms = kNegInf;
    for (int sidx = 0; sidx < a.nsplit; ++sidx) Ms = fmaxf(Ms, sm_m[sidx * kGroup + tid]);
    const float Mbs = (Ms == kNegInf) ? 0.f : Ms;
    float Ls = 0.f;
    for (int sidx = 0; sidx < a.nsplit; ++sidx) Ls += sm_l[sidx * kGroup + tid] * exp2f(sm_m[sidx * kGroup + tid] - Mbs);
    sM[tid] = Mbs;
    sL[tid] = Ls;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 8; ++h) o[h] = 0.f;
  for (int s0 = 0; s0 < a.nsplit; s0 += 4) {
    float x[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float* ps = parts + (size_t)(s0 + k) * kPartFloats + 2 * kGroup + tid;
#pragma unroll
      for (int h = 0; h < 8; ++h) x[k][h] = (s0 + k < a.nsplit) ? __ldcg(ps + h * kDim) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (s0 + k >= a.nsplit) break;
#pragma unroll
      for (int h = 0; h < 8; ++h) o[h] += exp2f(sm_m[(s0 + k) * kGroup + h] - sM[h]) * x[k][h];
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const float l = sL[h];
    orow[h * kDim + tid] = __float2bfloat16_rn(l > 0.f ? o[h] / l * vscale : 0.f);
  }
  if (tid == 0) a.tickets[unit] = 0;
  pdl_trigger();
}

template <bool FP8>
cudaError_t launch_attn_t(const AttnArgs& args, int grid, int tiles_per_split, cudaStream_t s, bool pdl) {
  const size_t smem = attn_smem_bytes(tiles_per_split);
  static size_t set_bytes[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || set_bytes[dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) set_bytes[dev] = smem;
  }
  return launch_k(attn_kernel<FP8>, dim3(grid), dim3(kThreads), smem, s, pdl, args);
}

}  // namespace

AttnPlan attn_plan(const qsa_dims& d, int num_sms) {
  AttnPlan pl;
  pl.units = d.batch * d.n_q * d.n_kv_heads;
  const int tiles_total = (d.width + kTile - 1) / kTile;
  const long long target = 4LL * num_sms * 4;  // ~4 waves of 4 resident CTAs per SM
  long long ns = (target + pl.units - 1) / pl.units;
  if (ns < 1) ns = 1;
  if (ns > tiles_total) ns = tiles_total;
  pl.tiles_per_split = (tiles_total + (int)ns - 1) / (int)ns;
  pl.nsplit = (tiles_total + pl.tiles_per_split - 1) / pl.tiles_per_split;
  return pl;
}

cudaError_t launch_attn(const qsa_dims& d, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* page_table,
                        const int32_t* sel_pos, const int32_t* q_pos, void* out, int32_t* err,
                        int32_t* tickets, float* partials, const AttnPlan& plan, cudaStream_t s,
                        bool pdl) {
  AttnArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.page_table = page_table;
  a.sel_pos = sel_pos;
  a.q_pos = q_pos;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.err = err;
  a.tickets = tickets;
  a.partials = partials;
  a.n_q = d.n_q;
  a.n_kv = d.n_kv_heads;
  int shift = 0;
  while ((1 << shift) < d.page_size) ++shift;
  a.page_shift = shift;
  a.max_pages = d.max_pages;
  a.num_pages = d.num_pages;
  a.width = d.width;
  a.nsplit = plan.nsplit;
  a.tiles_per_split = plan.tiles_per_split;
  a.sm_scale = d.sm_scale > 0.f ? d.sm_scale : 1.0f / sqrtf((float)d.head_dim);
  const int grid = plan.units * plan.nsplit;
  if (d.kv_dtype == QSA_KV_FP8_E4M3) return launch_attn_t<true>(a, grid, plan.tiles_per_split, s, pdl);
  return launch_attn_t<false>(a, grid, plan.tiles_per_split, s, pdl);
}

}  // namespace qsa
