// Sparse attention over the selected positions (decode and MTP verify).
//
// The pages (arex-research.com, section "四类优化", bullet 3) describe a
// sparse-attention kernel for the model's own attention geometry that handles
// plain decode and MTP verification with a BF16 query and a BF16 or FP8-E4M3
// KV cache; 10100.com ("第一处") adds that the selected history must then be
// found in the cache. The geometry here is theirs as this library reads it:
// 16 query heads over 2 KV heads of dim 128, a paged cache of 64-token pages.
//
// Design: one CTA per (request, query, KV head, split of the selection
// buffer). The CTA resolves its positions through the page table once, then
// streams 64-position K/V tiles into shared memory with 16-byte cp.async
// gathers (3-stage pipeline, XOR-swizzled rows so ldmatrix is conflict-free).
// Each of the 4 warps owns 16 positions of a tile: S = Q K^T and O += P V run
// on tensor cores (m16n8k16, FP32 accumulate) with the 8 query heads of the
// KV group as the M rows, and the softmax is online in FP32 in the exp2
// domain. FP8 tiles are widened to FP16 in shared memory (exact) before the
// MMAs; K's scale folds into the softmax scale and V's into the output.
// Splits write (max, sum, acc) partials to the workspace; the last CTA of a
// (request, query, KV head) to arrive, counted by an atomic ticket, merges
// them and resets the ticket, so there is no spin-wait anywhere.
#include <cuda_fp8.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kTile = 64;       // positions per pipeline stage
constexpr int kStages = 3;
constexpr int kThreads = 128;   // 4 warps x 16 positions
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16) * B(16x8) + D; rows 8..15 of A are zero here (a1 = a3 = 0).
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
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

// byte offset of 16-B chunk c (0..15) of row `pos` in a [64][128] 16-bit tile
__device__ __forceinline__ uint32_t swz(int pos, int c) {
  return (uint32_t)(pos * 256 + ((c ^ (pos & 7)) << 4));
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

template <bool FP8>
struct AttnSmem {
  static constexpr int kRaw = FP8 ? 128 : 256;  // bytes per cached row
  static constexpr int kStageBytes = 2 * kTile * kRaw;  // K + V
  static constexpr int kConvBytes = FP8 ? 2 * kTile * 256 : 0;  // FP16 K + V
  static size_t bytes(int tiles_per_split) {
    return (size_t)kStages * kStageBytes + kConvBytes + (size_t)tiles_per_split * kTile * 4 + 512;
  }
};

template <bool FP8>
__global__ void __launch_bounds__(kThreads) attn_kernel(const AttnArgs a) {
  using SM = AttnSmem<FP8>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage = smem;                                          // [kStages][K|V][64][raw]
  uint8_t* conv = smem + kStages * SM::kStageBytes;               // FP8 only: [K|V][64][256]
  int32_t* s_rows = reinterpret_cast<int32_t*>(conv + SM::kConvBytes);  // cache row of each position
  float* s_ml = reinterpret_cast<float*>(s_rows + a.tiles_per_split * kTile);  // [2][4][8] + [2][8]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, c4 = lane & 3;  // mma fragment row / column pair
  const int unit = blockIdx.x / a.nsplit, split = blockIdx.x % a.nsplit;
  const int g = unit % a.n_kv, row = unit / a.n_kv;
  const int r = row / a.n_q;
  const int n_q_heads = a.n_kv * kGroup;

  // ---- prologue independent of the previous kernel: Q fragments, scales ----
  const __nv_bfloat16* qrow = a.q + ((size_t)row * n_q_heads + g * kGroup + gq) * kDim;
  uint32_t qa[8][2];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + hh * 8 + 2 * c4);
      if constexpr (FP8) {
        const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
        qa[kk][hh] = pack2<true>(lo, hi);
      } else {
        qa[kk][hh] = w;
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

  // ---- pipeline ----
  const uint8_t* kc8 = static_cast<const uint8_t*>(a.k_cache);
  const uint8_t* vc8 = static_cast<const uint8_t*>(a.v_cache);
  auto issue = [&](int buf, int tile) {
    uint8_t* kb = stage + buf * SM::kStageBytes;
    uint8_t* vb = kb + kTile * SM::kRaw;
    constexpr int CPR = SM::kRaw / 16;  // 16-B chunks per row
#pragma unroll
    for (int it = 0; it < kTile * CPR / kThreads; ++it) {
      const int idx = it * kThreads + tid;
      const int pos = idx / CPR, c = idx % CPR;
      const int ri = s_rows[tile * kTile + pos];
      const size_t off = (size_t)(ri < 0 ? 0 : ri) * SM::kRaw + c * 16;
      uint32_t dk, dv;
      if constexpr (FP8) {
        dk = smem_u32(kb + pos * 128 + c * 16);
        dv = smem_u32(vb + pos * 128 + c * 16);
      } else {
        dk = smem_u32(kb + swz(pos, c));
        dv = smem_u32(vb + swz(pos, c));
      }
      cp_async16(dk, kc8 + off, ri >= 0);
      cp_async16(dv, vc8 + off, ri >= 0);
    }
  };

  float m_run = kNegInf, l_run = 0.f;
  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) issue(s, s);
    cp_async_commit();
  }
  for (int t = 0; t < ntiles; ++t) {
    if (t + kStages - 1 < ntiles) issue((t + kStages - 1) % kStages, t + kStages - 1);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const uint8_t* kb = stage + (t % kStages) * SM::kStageBytes;
    const uint8_t* vb = kb + kTile * SM::kRaw;
    if constexpr (FP8) {
      // widen E4M3 -> FP16 (exact) into the swizzled 16-bit tile layout
      uint8_t* kh = conv;
      uint8_t* vh = conv + kTile * 256;
#pragma unroll
      for (int it = 0; it < 2 * kTile * 8 / kThreads; ++it) {
        const int idx = it * kThreads + tid;
        const int which = idx / (kTile * 8), rem = idx % (kTile * 8);
        const int pos = rem / 8, c = rem % 8;
        const uint4 raw = *reinterpret_cast<const uint4*>((which ? vb : kb) + pos * 128 + c * 16);
        const uint32_t* rw = &raw.x;
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(rw[e] & 0xffffu), __NV_E4M3);
          const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(rw[e] >> 16), __NV_E4M3);
          h[2 * e] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
          h[2 * e + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
        }
        uint8_t* dst = which ? vh : kh;
        *reinterpret_cast<uint4*>(dst + swz(pos, 2 * c)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst + swz(pos, 2 * c + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
      }
      __syncthreads();
      kb = kh;
      vb = vh;
    }

    // S = Q K^T for this warp's 16 positions (2 n-tiles of 8)
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int mi = lane >> 3, rr = lane & 7;
    const int prow = warp * 16 + (mi >> 1) * 8 + rr;  // K row this lane addresses
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(smem_u32(kb + swz(prow, 2 * kk + (mi & 1))), b0, b1, b2, b3);
      mma16816<FP8>(s[0], qa[kk][0], qa[kk][1], b0, b1);
      mma16816<FP8>(s[1], qa[kk][0], qa[kk][1], b2, b3);
    }
    // mask, online softmax (row gq; columns 8*nt + 2*c4 + e)
    const int32_t* rows_t = s_rows + t * kTile + warp * 16;
    float x[2][2];
    float mt = kNegInf;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool ok = rows_t[nt * 8 + 2 * c4 + e] >= 0;
        x[nt][e] = ok ? s[nt][e] * scale_log2 : kNegInf;
        mt = fmaxf(mt, x[nt][e]);
      }
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float m_new = fmaxf(m_run, mt);
    const float base = (m_new == kNegInf) ? 0.f : m_new;
    const float alpha = exp2f(m_run - base);
    float pr[2][2];
    float psum = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pr[nt][e] = exp2f(x[nt][e] - base);
        psum += pr[nt][e];
      }
    l_run = l_run * alpha + psum;
    m_run = m_new;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      acc[i][0] *= alpha;
      acc[i][1] *= alpha;
    }
    const uint32_t pa0 = pack2<FP8>(pr[0][0], pr[0][1]);
    const uint32_t pa2 = pack2<FP8>(pr[1][0], pr[1][1]);
    // O += P V: ldmatrix.trans of V rows (positions) x 8-dim column blocks
    const int vrow = warp * 16 + (mi & 1) * 8 + rr;
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(smem_u32(vb + swz(vrow, 2 * dp + (mi >> 1))), b0, b1, b2, b3);
      mma16816<FP8>(acc[2 * dp], pa0, pa2, b0, b1);
      mma16816<FP8>(acc[2 * dp + 1], pa0, pa2, b2, b3);
    }
    __syncthreads();  // this stage's buffers are refilled next iteration
  }
  cp_async_wait<0>();

  // ---- merge the 4 warps ----
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  float* cm = s_ml;       // [4][8]
  float* cl = s_ml + 32;  // [4][8]
  if (c4 == 0) {
    cm[warp * 8 + gq] = m_run;
    cl[warp * 8 + gq] = l_run;
  }
  __syncthreads();
  float M = kNegInf;
#pragma unroll
  for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * 8 + gq]);
  const float Mb = (M == kNegInf) ? 0.f : M;
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) L += cl[w * 8 + gq] * exp2f(cm[w * 8 + gq] - Mb);
  const float f = exp2f(m_run - Mb);
  float* wacc = reinterpret_cast<float*>(stage);  // [4][8][128], the stage buffers are idle now
#pragma unroll
  for (int dt = 0; dt < 16; ++dt) {
    *reinterpret_cast<float2*>(&wacc[(warp * 8 + gq) * kDim + dt * 8 + 2 * c4]) =
        make_float2(acc[dt][0] * f, acc[dt][1] * f);
  }
  __syncthreads();
  // thread tid owns dim d = tid of all 8 heads
  float o[8];
#pragma unroll
  for (int h = 0; h < 8; ++h)
    o[h] = wacc[(0 * 8 + h) * kDim + tid] + wacc[(1 * 8 + h) * kDim + tid] +
           wacc[(2 * 8 + h) * kDim + tid] + wacc[(3 * 8 + h) * kDim + tid];
  float* sM = s_ml + 64;  // [8]
  float* sL = s_ml + 72;  // [8]
  if (warp == 0 && c4 == 0) {
    sM[gq] = M;
    sL[gq] = L;
  }
  __syncthreads();
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
  const float* parts = a.partials + (size_t)unit * a.nsplit * kPartFloats;
  if (tid < 8) {
    float Ms = kNegInf;
    for (int sidx = 0; sidx < a.nsplit; ++sidx) Ms = fmaxf(Ms, __ldcg(parts + (size_t)sidx * kPartFloats + tid));
    const float Mbs = (Ms == kNegInf) ? 0.f : Ms;
    float Ls = 0.f;
    for (int sidx = 0; sidx < a.nsplit; ++sidx) {
      const float* ps = parts + (size_t)sidx * kPartFloats;
      Ls += __ldcg(ps + 8 + tid) * exp2f(__ldcg(ps + tid) - Mbs);
    }
    sM[tid] = Mbs;
    sL[tid] = Ls;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 8; ++h) o[h] = 0.f;
  for (int sidx = 0; sidx < a.nsplit; ++sidx) {
    const float* ps = parts + (size_t)sidx * kPartFloats;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float w = exp2f(__ldcg(ps + h) - sM[h]);
      o[h] += w * __ldcg(ps + 16 + h * kDim + tid);
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
  const size_t smem = AttnSmem<FP8>::bytes(tiles_per_split);
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
  const long long target = 4LL * num_sms * 2;  // ~4 waves of 2 resident CTAs per SM
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
