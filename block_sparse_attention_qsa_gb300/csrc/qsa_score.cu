// Compressed index keys and FP32 block scores.
//
// Scoring follows the pages' QSA selection pipeline (arex-research.com,
// section "四类优化", bullets 1-2): every full 4-token block of a request is
// scored against each of its (up to 4) verify queries, and the compressed
// keys are loaded once per request and shared by all queries.
//
// GB300 design: the step streams the compressed keys (256 B per block per
// index head) once, so the kernel is built for HBM bandwidth. Each warp owns
// a contiguous, balanced range of 16-block units across the whole batch and
// keeps several units of 128-bit no-L1-allocate loads in flight. The 4-query
// contraction runs on the tensor cores (mma.sync, FP32 accumulate) straight
// from the loaded registers, so the key tile is shared by the 4 queries in
// registers rather than in shared memory and the ALUs stay idle.
#include "qsa_internal.cuh"
#include "qsa_trace.cuh"

namespace qsa {
namespace {

QSA_TRACE_TABLE

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
// the 16-byte chunks of block b's compressed key row of request r, or null
// for a page outside the cache (recorded)
__device__ __forceinline__ uint4* kc_row(uint4* kc, const KcPages& kp, int r, int b, int max_blocks, int cpb,
                                         int32_t* err) {
  if (!kp.table) return kc + ((size_t)r * max_blocks + b) * cpb;
  const int pi = b >> kp.bpp_shift;
  const int page = pi < kp.max_pages ? kp.table[(size_t)r * kp.max_pages + pi] : -1;
  if (page < 0 || page >= kp.num_pages) {
    record_error(err, kErrPage, r, 0, page);
    return nullptr;
  }
  return kc + ((((size_t)page) << kp.bpp_shift) + (b & ((1 << kp.bpp_shift) - 1))) * cpb;
}

__global__ void __launch_bounds__(256) compress_kernel(const uint4* __restrict__ idx_keys,
                                                       const int32_t* __restrict__ q_pos,
                                                       const int32_t* __restrict__ block_lo,
                                                       uint4* __restrict__ kc, int32_t* err,
                                                       int n_q, int H, int max_blocks, const KcPages kp) {
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
    uint4* dst = kc_row(kc, kp, r, b, max_blocks, cpb, err);
    if (dst) dst[c] = o;
  }
}

// ---------------------------------------------------------------------------
// scores on tensor cores
//
// Per request the scores are the skinny product S[j][b] = sum_k q[j][k] *
// kc[b][k] over k = (head, dim), with n_q <= 4 queries and thousands of
// blocks. One warp computes 16 blocks x 8 query columns per mma.sync
// m16n8k16 (BF16 in, FP32 accumulate; BF16 x BF16 products are exact in
// FP32): the 16 blocks are the A rows and the queries the B columns (columns
// n_q..7 are zero). The tensor cores take over the multiply-adds and the
// cross-lane reduction, so a lane only loads and stores.
//
// Fragment layout (lane = 4 * g + c): the lane owns A rows g and g + 8 and,
// in each 16-wide k step, k columns {2c, 2c+1, 2c+8, 2c+9}; B column g with
// the same k rows. Since a dot product does not depend on the order of its
// terms, k is permuted inside each 32-dim chunk so that the lane's 8 dims
// 8c..8c+7 of the chunk are exactly its k columns of two k steps: one 16-byte
// load of block row g (and one of row g + 8) fills the A fragments of two
// mma, and the query chunk at the same dims fills the B fragments.
// ---------------------------------------------------------------------------
template <int H>
struct ScoreGeom {
  static constexpr int STEPS = 4 * H;             // 32-dim chunks per block row
  // 16-block units (4 KB per index head) in flight per warp. One 256-thread
  // CTA per SM with 4 units in flight streams as fast as 4 CTAs with one unit
  // each, and leaves room on every SM for the selector's CTAs, which then
  // launch early (programmatic dependent launch) and start the moment the
  // scores are complete.
  static constexpr int PD = H == 1 ? 4 : 1;
  static constexpr int MIN_CTAS = 1;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int H, bool PAGED>
__global__ void __launch_bounds__(256, ScoreGeom<H>::MIN_CTAS) score_kernel(const __nv_bfloat16* __restrict__ q_idx,
                                                    const uint4* __restrict__ kc,
                                                    const int32_t* __restrict__ q_pos,
                                                    float* __restrict__ scores, int32_t* err,
                                                    int B, int n_q, int max_blocks, const KcPages kp) {
  using Geo = ScoreGeom<H>;
  constexpr int STEPS = Geo::STEPS, PD = Geo::PD;
  constexpr int CPB = H * 16;  // 16-B chunks per block row
  extern __shared__ int s_off[];  // [B + 1] first unit (16 blocks) of each request
  int* s_nb = s_off + B + 1;      // [B] full blocks of each request (its longest query)

  QSA_MARK(0);
  pdl_wait();  // no-op unless launched as a dependent
  QSA_MARK(1);
  // Let the selector launch now: its CTAs take each SM as this kernel's CTA
  // there exits, and its own wait still covers all of this grid's scores.
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    int carry = 0;
    for (int base = 0; base < B; base += 32) {
      const int r = base + lane;
      int units = 0;
      if (r < B) {
        int pv[kMaxNq];  // all of the request's positions in flight at once
#pragma unroll
        for (int j = 0; j < kMaxNq; ++j) pv[j] = j < n_q ? q_pos[r * n_q + j] : 0;
        int nb = 0;
#pragma unroll
        for (int j = 0; j < kMaxNq; ++j) {
          if (j >= n_q) break;
          const int p = pv[j];
          if (p < 0 || n_full_of(p) > max_blocks) {
            if (blockIdx.x == 0) record_error(err, kErrQueryPos, r, j, p);
          } else {
            nb = max(nb, n_full_of(p));
          }
        }
        units = (nb + 15) / 16;
        s_nb[r] = nb;
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

  int lo = 0, hi = B;  // last r with s_off[r] <= u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] <= u) lo = mid; else hi = mid;
  }
  int r = lo;
  const int g = lane >> 2, c = lane & 3;

  while (u < u_end) {
    while (s_off[r + 1] <= u) ++r;
    const int seg_end = min(u_end, s_off[r + 1]);
    const int u0 = s_off[r];

    // B fragments: query g (zero past n_q), dims 8c..8c+7 of every 32-dim chunk
    uint4 qf[STEPS];
    const int nb_r = s_nb[r];  // bounds this request's key loads without waiting for q_pos
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(q_idx + (size_t)(r * n_q + (g < n_q ? g : 0)) * CPB * 8);
#pragma unroll
      for (int s = 0; s < STEPS; ++s) qf[s] = (g < n_q) ? qrow[s * 4 + c] : make_uint4(0, 0, 0, 0);
    }
    // this lane stores queries 2c, 2c+1 (lanes with c < 2): their positions are
    // loaded here and turned into block bounds only at the first store, so the
    // key loads below do not wait for them
    const int p0 = (c < 2 && 2 * c < n_q) ? q_pos[r * n_q + 2 * c] : -1;
    const int p1 = (c < 2 && 2 * c + 1 < n_q) ? q_pos[r * n_q + 2 * c + 1] : -1;
    auto bound = [&](int p) { return (p >= 0 && n_full_of(p) <= max_blocks) ? n_full_of(p) : 0; };
    const uint4* kc_r = kc + (size_t)r * max_blocks * CPB;
    float* sc_r = scores + (size_t)r * n_q * max_blocks;

    // paged keys: the page ids of a batch's rows g and g + 8 are loaded one
    // batch ahead, so the key loads do not wait for the page table
    const int32_t* pt_r = PAGED ? kp.table + (size_t)r * kp.max_pages : nullptr;
    int pg[PD][2];
    auto load_pages = [&](int ub) {
#pragma unroll
      for (int k = 0; k < PD; ++k) {
        const int b = (ub + k - u0) * 16 + g;
        const bool in = ub + k < seg_end;
        // a page index past the table reads as page -1 (reported as a bad page)
        const int i0 = b >> kp.bpp_shift, i1 = (b + 8) >> kp.bpp_shift;
        pg[k][0] = (in && b < nb_r) ? (i0 < kp.max_pages ? pt_r[i0] : -1) : -1;
        pg[k][1] = (in && b + 8 < nb_r) ? (i1 < kp.max_pages ? pt_r[i1] : -1) : -1;
      }
    };
    if constexpr (PAGED) load_pages(u);
    for (; u < seg_end; u += PD) {
      uint4 lo_v[PD][STEPS], hi_v[PD][STEPS];
      int pc[PD][2];
      if constexpr (PAGED) {
#pragma unroll
        for (int k = 0; k < PD; ++k) {
          pc[k][0] = pg[k][0];
          pc[k][1] = pg[k][1];
        }
        if (u + PD < seg_end) load_pages(u + PD);
      }
#pragma unroll
      for (int k = 0; k < PD; ++k) {
        const int b = (u + k - u0) * 16 + g;
        const bool in = u + k < seg_end;
        const bool ok0 = in && b < nb_r, ok1 = in && b + 8 < nb_r;
        const uint4* row0;
        const uint4* row1;
        bool okp0 = ok0, okp1 = ok1;
        if constexpr (PAGED) {
          const int bm = (1 << kp.bpp_shift) - 1;
          okp0 = ok0 && pc[k][0] >= 0 && pc[k][0] < kp.num_pages;
          okp1 = ok1 && pc[k][1] >= 0 && pc[k][1] < kp.num_pages;
          if (ok0 && !okp0) record_error(err, kErrPage, r, 0, pc[k][0]);
          if (ok1 && !okp1) record_error(err, kErrPage, r, 0, pc[k][1]);
          row0 = kc + (okp0 ? ((((size_t)pc[k][0]) << kp.bpp_shift) + (b & bm)) * CPB : 0) + c;
          row1 = kc + (okp1 ? ((((size_t)pc[k][1]) << kp.bpp_shift) + ((b + 8) & bm)) * CPB : 0) + c;
        } else {
          row0 = kc_r + (size_t)b * CPB + c;
          row1 = row0 + (size_t)8 * CPB;
        }
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
          lo_v[k][s] = okp0 ? ld_stream(row0 + 4 * s) : make_uint4(0, 0, 0, 0);
          hi_v[k][s] = okp1 ? ld_stream(row1 + 4 * s) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int k = 0; k < PD; ++k) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
          mma_bf16_16816(acc, lo_v[k][s].x, hi_v[k][s].x, lo_v[k][s].y, hi_v[k][s].y, qf[s].x, qf[s].y);
          mma_bf16_16816(acc, lo_v[k][s].z, hi_v[k][s].z, lo_v[k][s].w, hi_v[k][s].w, qf[s].z, qf[s].w);
        }
        const int b = (u + k - u0) * 16 + g;
        if (c < 2 && u + k < seg_end) {
          // read here, after the key loads (a volatile move is not hoisted out of the loop)
          int q0, q1;
          asm volatile("mov.b32 %0, %1;" : "=r"(q0) : "r"(p0));
          asm volatile("mov.b32 %0, %1;" : "=r"(q1) : "r"(p1));
          const int nb0 = bound(q0), nb1 = bound(q1);
          float* s0 = sc_r + (size_t)(2 * c) * max_blocks;
          float* s1 = s0 + max_blocks;
          if (b < nb0) s0[b] = acc[0];
          if (b < nb1) s1[b] = acc[1];
          if (b + 8 < nb0) s0[b + 8] = acc[2];
          if (b + 8 < nb1) s1[b + 8] = acc[3];
        }
      }
    }
    u = seg_end;  // the unrolled loop may step past the end of this request's units
  }
  QSA_MARK_LAST(2);
  QSA_MARK_LAST(3);
}

int shift_of(int x) {
  int sh = 0;
  while ((1 << sh) < x) ++sh;
  return sh;
}

KcPages kc_pages(const qsa_dims& d, const int32_t* page_table) {
  KcPages kp;
  kp.table = page_table;
  kp.max_pages = d.max_pages;
  kp.num_pages = d.num_pages;
  kp.bpp_shift = shift_of(d.page_size / kBlock);
  return kp;
}

template <int H, bool PAGED>
cudaError_t launch_score_h(const qsa_dims& d, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                           const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s,
                           bool pdl, const KcPages& kp) {
  auto kern = score_kernel<H, PAGED>;
  const size_t smem = (size_t)(2 * d.batch + 1) * sizeof(int);
  static DeviceSlots occ_slots, smem_slots;  // one pair per instantiation
  const cudaError_t e = smem_slots.raise_smem(kern, smem);
  if (e != cudaSuccess) return e;
  // resident CTAs per SM: bound by registers (the per-request tables are small)
  int occ = occ_slots.get([&] {
    int o = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, 256, 0) == cudaSuccess ? o : 0;
  });
  if (occ < 1) occ = 1;
  // upper bound of the work, in 16-block units, to avoid launching idle warps
  const long long units_ub = (long long)d.batch * ((d.max_blocks + 15) / 16);
  long long warps = (long long)device_sm_count() * occ * 8;
  const long long want = (units_ub + 1) / 2;  // at least ~2 units per warp
  if (want < warps) warps = want;
  const int grid = (int)((warps + 7) / 8 > 0 ? (warps + 7) / 8 : 1);
  return launch_k(kern, dim3(grid), dim3(256), smem, s, pdl, q_idx, reinterpret_cast<const uint4*>(kc), q_pos,
                  scores, err, d.batch, d.n_q, d.max_blocks, kp);
}

}  // namespace

QSA_TRACE_HOST(trace_score)

cudaError_t launch_compress(const qsa_dims& d, const __nv_bfloat16* idx_keys, const int32_t* q_pos,
                            const int32_t* block_lo, __nv_bfloat16* kc, int32_t* err,
                            cudaStream_t s, const int32_t* page_table) {
  const long long chunks = (long long)d.max_blocks * d.n_idx_heads * 16;
  long long gx = (chunks + 255) / 256;
  const long long cap = (long long)device_sm_count() * 8;
  if (gx > cap) gx = cap;
  if (gx < 1) gx = 1;
  return launch_k(compress_kernel, dim3((unsigned)gx, d.batch), dim3(256), 0, s, false,
                  reinterpret_cast<const uint4*>(idx_keys), q_pos, block_lo,
                  reinterpret_cast<uint4*>(kc), err, d.n_q, d.n_idx_heads, d.max_blocks, kc_pages(d, page_table));
}

cudaError_t launch_score(const qsa_dims& d, const __nv_bfloat16* q_idx, const __nv_bfloat16* kc,
                         const int32_t* q_pos, float* scores, int32_t* err, cudaStream_t s,
                         bool pdl, const int32_t* page_table) {
  const KcPages kp = kc_pages(d, page_table);
  if (page_table) {
    switch (d.n_idx_heads) {
      case 1: return launch_score_h<1, true>(d, q_idx, kc, q_pos, scores, err, s, pdl, kp);
      case 2: return launch_score_h<2, true>(d, q_idx, kc, q_pos, scores, err, s, pdl, kp);
      case 3: return launch_score_h<3, true>(d, q_idx, kc, q_pos, scores, err, s, pdl, kp);
      default: return launch_score_h<4, true>(d, q_idx, kc, q_pos, scores, err, s, pdl, kp);
    }
  }
  switch (d.n_idx_heads) {
    case 1: return launch_score_h<1, false>(d, q_idx, kc, q_pos, scores, err, s, pdl, kp);
    case 2: return launch_score_h<2, false>(d, q_idx, kc, q_pos, scores, err, s, pdl, kp);
    case 3: return launch_score_h<3, false>(d, q_idx, kc, q_pos, scores, err, s, pdl, kp);
    default: return launch_score_h<4, false>(d, q_idx, kc, q_pos, scores, err, s, pdl, kp);
  }
}

}  // namespace qsa
