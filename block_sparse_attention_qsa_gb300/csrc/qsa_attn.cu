// Sparse attention over the selected positions (decode and MTP verify).
//
// The pages (arex-research.com, section "四类优化", bullet 3) describe a
// sparse-attention kernel for the model's own attention geometry that handles
// plain decode and MTP verification with a BF16 query and a BF16 or FP8-E4M3
// KV cache; 10100.com ("第一处") adds that the selected history must then be
// found in the cache. The geometry here is theirs as this library reads it:
// 16 query heads over 2 KV heads of dim 128, a paged cache of 64-token pages.
//
// Design (stream-K). The (request, query, KV head) units times their tiles
// of selected positions form one stream of tiles, cut into equal contiguous
// shares, one per resident 4-warp CTA, so every CTA does the same work and
// the kernel has no wave tail. Within a tile every warp works alone on 16
// positions (BF16; lane 4g + c holds positions g and g + 8) or 32 (FP8; g,
// g + 8, g + 16, g + 24), so that a warp step moves 8 KB of K and V for either
// cache type. The selected K/V rows are random 256-byte (BF16) or 128-byte (FP8) rows, so the
// kernel is a gather: measured on GB300, 128-bit loads straight into
// registers, with each warp reading whole rows, sustain a much higher share
// of HBM bandwidth for such gathers than staging through shared memory. So K
// and V never touch shared memory:
//
//  * S^T = K Q^T on the tensor cores (mma.sync m16n8k16, FP32 accumulate):
//    each 16 of the warp's positions are the M rows of one mma, the KV
//    group's 8 query heads the N columns. A lane's 16-byte loads of K rows
//    are its A fragments directly, because the head dim is visited in a
//    lane-dependent order that Q's B fragments follow too (a dot product does
//    not depend on the order of its terms).
//  * softmax is online, in FP32, in the exp2 domain, per head;
//  * O^T = V^T P^T: V rows loaded the same way are turned into A fragments
//    with movmatrix (an in-register 8x8 transpose), P^T is the softmax tile
//    transposed the same way, and the output's dim order (permuted by the V
//    loads) is undone when it is written.
//
// Each lane looks two tiles ahead in the selection, so the K/V loads of the
// next tile are in flight across unit boundaries. FP8 codes stay packed in
// registers and are widened to FP16 (exact for E4M3) right before their mma;
// the BF16 query of that FP16 contraction is scaled per head by a power of
// two into FP16's range (exact: BF16's 8 significant bits fit FP16's 11), the
// factor folded back into the head's softmax scale like K's scale; V's scale
// folds into the output. The warps'
// softmax states merge through shared memory; a unit split between CTAs
// publishes (max, sum, acc) pieces to the workspace and the last piece to
// arrive, counted by an atomic ticket, merges them and resets the ticket, so
// there is no spin-wait anywhere.
//
// Cluster form (up to mid-size batches, chosen by attn_plan): each unit is
// one thread-block cluster whose CTAs split its tiles evenly and run the same
// warp loop; each CTA then stores its piece's values of every other CTA's
// share of the outputs into that CTA's shared memory (distributed shared
// memory), and after one hardware cluster barrier every CTA merges its share
// locally, with no workspace round trip. Measured on GB300 it beats stream-K's even shares
// wherever no CTA gets more than about twice stream-K's tiles and the
// clusters still place in one wave.
#include <algorithm>

#include "qsa_internal.cuh"
#include "qsa_trace.cuh"

namespace qsa {
namespace {

QSA_TRACE_TABLE

constexpr int kTile = 64;       // BF16 positions per CTA step: 4 warps of 16 (FP8: 4 of 32)
// resident CTAs per SM: BF16 rows take twice the registers of FP8 codes
// (two rows of K and V per lane: 64 registers against 32)
template <bool FP8>
constexpr int kCtasPerSm = 3;
template <bool FP8>
constexpr int kRowsPerLane = FP8 ? 4 : 2;
// Small batches: each CTA takes at least this many tiles (192 BF16 or 256 FP8
// positions), so a unit is cut into few pieces and the merge of the last one
// to arrive stays short. Measured at batch 1, BF16: 1 tile 35.1 us per step,
// 2 tiles 30.7, 3 tiles 28.9, 4 tiles 33.5 (the first and last with an older
// build); FP8 (tiles twice as long): 2 tiles 31.0, 3 tiles 32.1.
template <bool FP8>
constexpr int kMinTilesPerCta = FP8 ? 2 : 3;
constexpr int kMergeBatch = 4;  // pieces whose accumulators are read at once
constexpr int kMaxCluster = 16;  // CTAs per unit in the cluster form (non-portable above 8)
// inbox of the cluster form: C sources x (4 ceil(256 / C)) outputs; checked
// below to cover every C in 2..kMaxCluster (at most 15 x 72 = 1,080 floats),
// a multiple of 4 (float4 reads)
constexpr int kInboxAcc = 1088;
constexpr bool inbox_fits(int c) {
  return c > kMaxCluster || (c * 4 * ((256 + c - 1) / c) <= kInboxAcc && inbox_fits(c + 1));
}
static_assert(inbox_fits(2) && kInboxAcc % 4 == 0, "cluster-form inbox too small");
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

// atomic add of 1 with acquire-release semantics at GPU scope; returns the old value
__device__ __forceinline__ int ticket_acq_rel(int32_t* p) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

// a 32-bit load issued at this point of the program (its use may come much later)
__device__ __forceinline__ int ld_issue(const int32_t* p) {
  int v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// 2^x on the special-function unit (the PTX ex2.approx.ftz instruction:
// relative error about 2^-22, results below the normal range flushed to zero,
// 2^-inf = 0). Used for the per-step softmax terms, whose arguments are <= 0.
__device__ __forceinline__ float exp2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// four E4M3 codes (bytes 0-3 of w) -> FP16x2 of codes 0, 1 (lo) and of codes
// 2, 3 (hi), exact: the word's two halves go straight to the hardware
// conversion, with no masking, shifting or repacking around it
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// BF16 pair times f (a power of two) -> FP16 pair (Q of the FP8 path)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w, float f) {
  return pack2<true>(__uint_as_float(w << 16) * f, __uint_as_float(w & 0xffff0000u) * f);
}

// Exponent shift s of a query head whose largest magnitude is amax: amax *
// 2^-s lies in [2^14, 2^15), so the head's BF16 values times 2^-s are FP16
// values exactly (BF16 keeps 8 significant bits, FP16 11, and the range down
// to amax * 2^-29 stays normal); the score is multiplied back by 2^s in the
// softmax scale. Clamped so that 2^-s and 2^s are normal FP32 numbers.
__device__ __forceinline__ int q_shift(float amax) {
  if (!(amax > 0.f)) return 0;
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;
  return min(126, max(-126, e - 14));
}
__device__ __forceinline__ float pow2(int s) { return __uint_as_float((uint32_t)(127 + s) << 23); }

// Register layout of one lane's share of a 128-dim row, for lane = 4g + c.
//   BF16 rows (256 B): 4 loads of 16 B at chunks c, c+4, c+8, c+12 -> 16
//   pairs; pair (i, e) holds dims 8(c + 4i) + 2e + {0,1}.
//   FP8 rows (128 B): 2 loads of 16 B at chunks c, c+4, kept as 8 raw words
//   of 4 E4M3 codes; pair (i, e) holds dims 16(c + 4i) + 2e + {0,1} and is the
//   low (e even) or high half of raw word 4i + e/2, widened to FP16 (exact)
//   where it is used.
// Pair p = 4i + e (BF16) or 8i + e (FP8) is the lane's p-th pair.
//   K: k-step ks (16 of the 128 dims) uses pairs 2ks and 2ks + 1 of a row
//      (FP8: the two halves of raw word ks).
//   V: the 8x8 block k (logical dims 8k..8k+7) holds pair k of each row
//      (FP8: blocks 2m and 2m + 1 are the two halves of raw word m).
template <bool FP8>
struct RowRegs {
  static constexpr int kLoads = FP8 ? 2 : 4;
  static constexpr int kRowBytes = FP8 ? 128 : 256;
  uint32_t pr[FP8 ? 8 : 16];  // BF16: 16 pairs; FP8: 8 raw words (16 pairs of codes)

  __device__ __forceinline__ void load(const uint8_t* row, int c, bool ok) {
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const uint4 v = ok ? ldg16(row + (c + 4 * i) * 16) : make_uint4(0, 0, 0, 0);
      pr[4 * i + 0] = v.x;
      pr[4 * i + 1] = v.y;
      pr[4 * i + 2] = v.z;
      pr[4 * i + 3] = v.w;
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
  const int32_t* sel_row;  // cache row (KV head 0) of every selected position, -1 for none
  int row_lim;             // a KV-head-0 row r is used only if 0 <= r < row_lim (all heads in the cache)
  __nv_bfloat16* out;
  int32_t* tickets;
  float* partials;
  long long total;  // units * tiles: the tile stream the CTAs share
  int tiles, grid, n_kv, page_size, width;
  int cl;  // cluster form: CTAs per unit (its cluster), else 0
  float sm_scale;
};

// First tile of CTA c's share of the tile stream, and the CTA holding tile w.
__device__ __forceinline__ long long tile_begin(const AttnArgs& a, int c) {
  return (long long)c * a.total / a.grid;
}
__device__ __forceinline__ int cta_of_tile(const AttnArgs& a, long long w) {
  return (int)(((w + 1) * a.grid - 1) / a.total);
}

// Where the row look-ahead stands: tile t of KV head g of (request, query) row.
struct Cursor {
  int t, g, row;
};

// CL: the cluster form for few units. Each unit is one thread-block cluster
// of a.cl CTAs, CTA k taking the unit's tiles [k T / cl, (k+1) T / cl); the
// CTAs' pieces are pushed through distributed shared memory to the CTAs that
// own each 1 / cl of the unit's outputs and merged there after one cluster
// barrier, with no workspace, fence or ticket.
template <bool FP8, bool CL>
__global__ void __launch_bounds__(kThreads, kCtasPerSm<FP8>) attn_kernel(const AttnArgs a) {
  __shared__ __align__(16) __nv_bfloat16 sQ[2][kGroup * kDim];
  __shared__ __align__(16) float wacc[4 * kGroup * kDim];  // [warp][head][dim]
  __shared__ float s_ml[96];
  __shared__ int s_last;
  // cluster form: the other CTAs' values of this CTA's outputs (its inbox)
  __shared__ __align__(16) float inbox[CL ? kInboxAcc + 16 * kMaxCluster : 4];

  // positions per warp step: lane 4g + c holds rows g + 8k, k < R, so each
  // pair of rows fills the 16 M rows of a score mma and the k of a PV mma.
  // BF16: 2 rows (16 positions); FP8: 4 rows (32 positions), so that a step
  // moves as many bytes for either cache type
  constexpr int R = kRowsPerLane<FP8>;
  constexpr int POS = 8 * R;
  constexpr int TILE = 4 * POS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, c4 = lane & 3;
  const int ent = warp * POS + gq;  // this lane's first position within a tile (then ent + 8k)
  const int n_q_heads = a.n_kv * kGroup;
  const int P = a.page_size;
  using RR = RowRegs<FP8>;
  const uint8_t* kbase = static_cast<const uint8_t*>(a.k_cache);
  const uint8_t* vbase = static_cast<const uint8_t*>(a.v_cache);

  const int cta = blockIdx.x;
  QSA_MARK(0);
  long long w0, w1;
  if constexpr (CL) {
    // every CTA of the cluster must have started before another stores into
    // its shared memory: arrive now, wait before the pushes below
    cluster_arrive_relaxed();
    // one unit per cluster (the host keeps cl <= tiles, so no share is empty)
    const int uu = cta / a.cl, rk = cta - uu * a.cl;
    w0 = (long long)uu * a.tiles + (long long)rk * a.tiles / a.cl;
    w1 = (long long)uu * a.tiles + (long long)(rk + 1) * a.tiles / a.cl;
  } else {
    w0 = tile_begin(a, cta);
    w1 = tile_begin(a, cta + 1);
  }
  if (!CL && w0 >= w1) {
    QSA_MARK(3);
    pdl_trigger();
    return;
  }
  int u = (int)(w0 / a.tiles);
  int t = (int)(w0 - (long long)u * a.tiles);

  // the 8 query rows of unit uu (2 KB, contiguous) into sQ[buf]
  auto stage_q = [&](int uu, int buf) {
    const uint8_t* src = reinterpret_cast<const uint8_t*>(a.q + (size_t)uu * kGroup * kDim) + tid * 16;
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(reinterpret_cast<uint8_t*>(sQ[buf]) + tid * 16);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  };
  stage_q(u, 0);  // the query is not produced by the previous kernel
  asm volatile("cp.async.commit_group;" ::: "memory");

  pdl_wait();  // the selection is
  QSA_MARK(1);

  // Row look-ahead: the selection entries of tile w + 2 are loaded while tile w
  // is processed, and turn into cache rows for the K/V loads of tile w + 1.
  Cursor L{t, u % a.n_kv, u / a.n_kv};
  auto load_entry = [&](bool in_range, int off) {
    const int i = L.t * TILE + ent + off;
    return (in_range && i < a.width) ? ld_issue(a.sel_row + (size_t)L.row * a.width + i) : -1;
  };
  auto advance = [&]() {
    if (++L.t == a.tiles) {
      L.t = 0;
      if (++L.g == a.n_kv) {
        L.g = 0;
        ++L.row;
      }
    }
  };
  // this lane's rows of tile w: positions ent + 8k, k < R (R rows of 16-row mma tiles)
  int e1[R];
  int ri[R];
  {
    int e0[R];
#pragma unroll
    for (int k = 0; k < R; ++k) e0[k] = load_entry(true, 8 * k);
    const int g0 = L.g;
    advance();
#pragma unroll
    for (int k = 0; k < R; ++k) {
      e1[k] = load_entry(w0 + 1 < w1, 8 * k);
      ri[k] = (unsigned)e0[k] < (unsigned)a.row_lim ? e0[k] + g0 * P : -1;
    }
  }
  int g1 = L.g;
  advance();
  long long wl = w0 + 2;  // tile of the cursor

  RR kr[R], vr[R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    kr[k].load(kbase + (size_t)max(ri[k], 0) * RR::kRowBytes, c4, ri[k] >= 0);
    vr[k].load(vbase + (size_t)max(ri[k], 0) * RR::kRowBytes, c4, ri[k] >= 0);
  }

  long long w = w0;
  for (int buf = 0;; buf ^= 1) {
    // ---- one segment: tiles [t, t + seg) of unit u ----
    const int row = u / a.n_kv, g = u - row * a.n_kv;
    const long long seg_w0 = w;
    const int seg = (int)min((long long)(a.tiles - t), w1 - w);
    const bool more = !CL && w + seg < w1;  // the share continues with unit u + 1 (never in the cluster form)
    if (more) stage_q(u + 1, buf ^ 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // this unit's query has landed
    __syncthreads();

    uint32_t qb[16];  // B fragments of the KV group's 8 query heads (head gq)
    float qs[2] = {1.f, 1.f};  // FP8: 2^s of heads 2c4 and 2c4 + 1 (their FP16 query scaling undone)
    {
      const __nv_bfloat16* qh = sQ[buf] + gq * kDim;
      if constexpr (FP8) {
        // the query stays BF16 in meaning: each head is scaled by a power of
        // two into FP16's range (exact) before the FP16 contraction
        uint32_t wd[16];
        uint32_t amax = 0;  // largest |q| bits of this lane's 32 dims of head gq
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint4 lo = *reinterpret_cast<const uint4*>(qh + 16 * (c4 + 4 * i));
          const uint4 hi = *reinterpret_cast<const uint4*>(qh + 16 * (c4 + 4 * i) + 8);
          const uint32_t w8[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            wd[8 * i + e] = w8[e];
            // magnitudes of BF16 values order like their bit patterns
            amax = max(amax, max((w8[e] << 16) & 0x7fff0000u, w8[e] & 0x7fff0000u));
          }
        }
        amax = max(amax, __shfl_xor_sync(kFull, amax, 1));
        amax = max(amax, __shfl_xor_sync(kFull, amax, 2));
        const int sh = q_shift(__uint_as_float(amax));  // head gq
        const float down = pow2(-sh);
#pragma unroll
        for (int e = 0; e < 16; ++e) qb[e] = bf2_to_h2(wd[e], down);
        qs[0] = pow2(__shfl_sync(kFull, sh, 4 * (2 * c4)));
        qs[1] = pow2(__shfl_sync(kFull, sh, 4 * (2 * c4 + 1)));
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(qh + 8 * (c4 + 4 * i));
          qb[4 * i + 0] = v.x;
          qb[4 * i + 1] = v.y;
          qb[4 * i + 2] = v.z;
          qb[4 * i + 3] = v.w;
        }
      }
    }
    const float kscale = FP8 ? a.k_scale[g] : 1.f;
    const float vscale = FP8 ? a.v_scale[g] : 1.f;
    // per head of this lane's two score columns (FP8: times the query's 2^s)
    const float scale_log2A = a.sm_scale * kscale * kLog2e * qs[0];
    const float scale_log2B = a.sm_scale * kscale * kLog2e * qs[1];

    float m_run[2] = {kNegInf, kNegInf}, l_run[2] = {0.f, 0.f};  // heads 2c4, 2c4 + 1
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    for (int i = 0; i < seg; ++i, ++w) {
      // S^T (POS positions x 8 heads): R / 2 mma tiles of 16 positions (rows 2j, 2j + 1)
      float s[R / 2][4];
#pragma unroll
      for (int j = 0; j < R / 2; ++j) {
        s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          if constexpr (FP8) {
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_h2x2(kr[2 * j].pr[ks], a0, a2);
            e4m3x4_to_h2x2(kr[2 * j + 1].pr[ks], a1, a3);
            mma16816<true>(s[j], a0, a1, a2, a3, qb[2 * ks], qb[2 * ks + 1]);
          } else {
            mma16816<false>(s[j], kr[2 * j].pr[2 * ks], kr[2 * j + 1].pr[2 * ks], kr[2 * j].pr[2 * ks + 1],
                            kr[2 * j + 1].pr[2 * ks + 1], qb[2 * ks], qb[2 * ks + 1]);
          }
        }
      }
      bool ok[R];
#pragma unroll
      for (int k = 0; k < R; ++k) ok[k] = ri[k] >= 0;
      // the next tile of the share (this unit or the next): its K rows now
      const bool next = w + 1 < w1;
      int nri[R];
#pragma unroll
      for (int k = 0; k < R; ++k) {
        nri[k] = (unsigned)e1[k] < (unsigned)a.row_lim ? e1[k] + g1 * P : -1;
        e1[k] = load_entry(wl < w1, 8 * k);
      }
      g1 = L.g;
      advance();
      ++wl;
      if (next) {
#pragma unroll
        for (int k = 0; k < R; ++k) kr[k].load(kbase + (size_t)max(nri[k], 0) * RR::kRowBytes, c4, nri[k] >= 0);
      }
      // online softmax; s[j][0], s[j][1]: row 2j (position ent + 16j), heads 2c4,
      // 2c4 + 1; s[j][2], s[j][3]: row 2j + 1 (position ent + 16j + 8)
      float x[R / 2][4];
      float mA = kNegInf, mB = kNegInf;
#pragma unroll
      for (int j = 0; j < R / 2; ++j) {
        x[j][0] = ok[2 * j] ? s[j][0] * scale_log2A : kNegInf;
        x[j][1] = ok[2 * j] ? s[j][1] * scale_log2B : kNegInf;
        x[j][2] = ok[2 * j + 1] ? s[j][2] * scale_log2A : kNegInf;
        x[j][3] = ok[2 * j + 1] ? s[j][3] * scale_log2B : kNegInf;
        mA = fmaxf(mA, fmaxf(x[j][0], x[j][2]));
        mB = fmaxf(mB, fmaxf(x[j][1], x[j][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(kFull, mA, o));
        mB = fmaxf(mB, __shfl_xor_sync(kFull, mB, o));
      }
      const float nA = fmaxf(m_run[0], mA), nB = fmaxf(m_run[1], mB);
      const float bA = nA == kNegInf ? 0.f : nA, bB = nB == kNegInf ? 0.f : nB;
      const float alA = exp2_sfu(m_run[0] - bA), alB = exp2_sfu(m_run[1] - bB);
      // the accumulators need rescaling only when a running maximum moved (once
      // the first tiles are in, rarely); an unmoved -inf maximum means nothing
      // has been accumulated yet
      const bool moved = !__all_sync(kFull, nA == m_run[0] && nB == m_run[1]);
      float sumA = 0.f, sumB = 0.f;
      uint32_t pb[R];  // P^T fragments: row k's probabilities, transposed
#pragma unroll
      for (int j = 0; j < R / 2; ++j) {
        const float p0 = exp2_sfu(x[j][0] - bA), p1 = exp2_sfu(x[j][1] - bB);
        const float p2 = exp2_sfu(x[j][2] - bA), p3 = exp2_sfu(x[j][3] - bB);
        sumA += p0 + p2;
        sumB += p1 + p3;
        pb[2 * j] = movt(pack2<FP8>(p0, p1));
        pb[2 * j + 1] = movt(pack2<FP8>(p2, p3));
      }
      l_run[0] = l_run[0] * alA + sumA;
      l_run[1] = l_run[1] * alB + sumB;
      m_run[0] = nA;
      m_run[1] = nB;
      if (moved) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          acc[k][0] *= alA;
          acc[k][1] *= alB;
          acc[k][2] *= alA;
          acc[k][3] *= alB;
        }
      }
      // O^T += V^T P^T, one k step of 16 positions per pair of rows
#pragma unroll
      for (int j = 0; j < R / 2; ++j) {
        if constexpr (FP8) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t v0, v1, v2, v3;
            e4m3x4_to_h2x2(vr[2 * j].pr[mt], v0, v1);
            e4m3x4_to_h2x2(vr[2 * j + 1].pr[mt], v2, v3);
            mma16816<true>(acc[mt], movt(v0), movt(v1), movt(v2), movt(v3), pb[2 * j], pb[2 * j + 1]);
          }
        } else {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
            mma16816<false>(acc[mt], movt(vr[2 * j].pr[2 * mt]), movt(vr[2 * j].pr[2 * mt + 1]),
                            movt(vr[2 * j + 1].pr[2 * mt]), movt(vr[2 * j + 1].pr[2 * mt + 1]), pb[2 * j],
                            pb[2 * j + 1]);
        }
      }
      if (next) {
#pragma unroll
        for (int k = 0; k < R; ++k) vr[k].load(vbase + (size_t)max(nri[k], 0) * RR::kRowBytes, c4, nri[k] >= 0);
      }
#pragma unroll
      for (int k = 0; k < R; ++k) ri[k] = nri[k];
    }

    // ---- merge the 4 warps (the next unit's first K/V rows are in flight) ----
    QSA_MARK_LAST(2);
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
      for (int k = 0; k < 4; ++k) M = fmaxf(M, cm[k * 8 + h]);
      fac[e] = exp2f(m_run[e] - (M == kNegInf ? 0.f : M));
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = phys_dim<FP8>(16 * mt + gq), d1 = phys_dim<FP8>(16 * mt + gq + 8);
      float* r0 = wacc + (warp * 8 + 2 * c4) * kDim;
      float* r1 = r0 + kDim;
      r0[d0] = acc[mt][0] * fac[0];
      r1[d0] = acc[mt][1] * fac[1];
      r0[d1] = acc[mt][2] * fac[0];
      r1[d1] = acc[mt][3] * fac[1];
    }
    float* sM = s_ml + 64;  // [8]
    float* sL = s_ml + 72;  // [8]
    if (tid < 8) {
      float M = kNegInf;
#pragma unroll
      for (int k = 0; k < 4; ++k) M = fmaxf(M, cm[k * 8 + tid]);
      const float Mb = M == kNegInf ? 0.f : M;
      float Ls = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) Ls += cl[k * 8 + tid] * exp2f(cm[k * 8 + tid] - Mb);
      sM[tid] = M;
      sL[tid] = Ls;
    }
    __syncthreads();
    // thread tid owns dim tid of all 8 heads
    float o[8];
#pragma unroll
    for (int h = 0; h < 8; ++h)
      o[h] = wacc[(0 * 8 + h) * kDim + tid] + wacc[(1 * 8 + h) * kDim + tid] +
             wacc[(2 * 8 + h) * kDim + tid] + wacc[(3 * 8 + h) * kDim + tid];
    __nv_bfloat16* orow = a.out + ((size_t)row * n_q_heads + g * kGroup) * kDim;

    if (!CL && t == 0 && seg == a.tiles) {
      // the whole unit is in this share: write the output
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float l = sL[h];
        orow[h * kDim + tid] = __float2bfloat16_rn(l > 0.f ? o[h] / l * vscale : 0.f);
      }
    } else if constexpr (CL) {
      // ---- the cluster's pieces: CTA k owns quads [k per, (k+1) per) of the
      // unit's 256 four-dim output quads. Every CTA stores its piece's values
      // for each owner's outputs, and its (max, sum), straight into that
      // owner's inbox (distributed shared memory stores, in flight while the
      // CTAs wait at the barrier); after the one barrier each owner merges
      // from its own shared memory, and no CTA touches another's again ----
      const int C = a.cl, rk = (int)cluster_rank();
      constexpr int kQuads = kGroup * kDim / 4;
      const int per = (kQuads + C - 1) / C, span = 4 * per;  // outputs per owner
      float* in_acc = inbox;               // [C][span]: the sources' accumulators of this CTA's outputs
      float* in_ml = inbox + kInboxAcc;    // [C][16]: the sources' (max[8], sum[8])
      cluster_wait();  // every CTA of the cluster has started
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const int oi = h * kDim + tid, r = oi / span;
        st_peer_f32(peer_addr(in_acc + rk * span + (oi - r * span), r), o[h]);
      }
      for (int i = tid; i < 16 * C; i += kThreads) {
        const int r = i >> 4, e = i & 15;
        st_peer_f32(peer_addr(in_ml + rk * 16 + e, r), e < 8 ? sM[e] : sL[e - 8]);
      }
      cluster_sync();  // release / acquire: every store above is visible to its owner
      const int q_end = min(kQuads, (rk + 1) * per);
      for (int qd = rk * per + tid; qd < q_end; qd += kThreads) {
        const int oi = 4 * qd, h = oi / kDim, li = oi - rk * span;
        float M = kNegInf;
        for (int j = 0; j < C; ++j) M = fmaxf(M, in_ml[16 * j + h]);
        const float Mb = M == kNegInf ? 0.f : M;
        float L = 0.f, O0 = 0.f, O1 = 0.f, O2 = 0.f, O3 = 0.f;
        for (int j = 0; j < C; ++j) {
          const float4 x = *reinterpret_cast<const float4*>(in_acc + j * span + li);
          const float f = exp2f(in_ml[16 * j + h] - Mb);
          L += in_ml[16 * j + 8 + h] * f;
          O0 += x.x * f;
          O1 += x.y * f;
          O2 += x.z * f;
          O3 += x.w * f;
        }
        const float sc = L > 0.f ? vscale / L : 0.f;
        __nv_bfloat16* dst = orow + oi;  // dims oi .. oi + 3 of head h
        if ((reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(O0 * sc, O1 * sc), hi = __floats2bfloat162_rn(O2 * sc, O3 * sc);
          uint2 pk;
          memcpy(&pk.x, &lo, 4);
          memcpy(&pk.y, &hi, 4);
          *reinterpret_cast<uint2*>(dst) = pk;
        } else {  // an output buffer aligned to 2 bytes only
          dst[0] = __float2bfloat16_rn(O0 * sc);
          dst[1] = __float2bfloat16_rn(O1 * sc);
          dst[2] = __float2bfloat16_rn(O2 * sc);
          dst[3] = __float2bfloat16_rn(O3 * sc);
        }
      }
      QSA_MARK(6);
    } else {
      // ---- a piece of the unit: publish it, the last piece to arrive merges ----
      // slot 2c: the share's first segment, 2c + 1: its last (only these two can be pieces)
      const int slot = 2 * cta + (seg_w0 == w0 ? 0 : 1);
      float* part = a.partials + (size_t)slot * kPartFloats;
      if (tid < 8) {
        part[tid] = sM[tid];
        part[8 + tid] = sL[tid];
      }
#pragma unroll
      for (int h = 0; h < 8; ++h) part[16 + h * kDim + tid] = o[h];
      const long long uw0 = (long long)u * a.tiles;
      const int c_first = cta_of_tile(a, uw0), n_piece = cta_of_tile(a, uw0 + a.tiles - 1) - c_first + 1;
      // The barrier orders every thread's stores of the piece before thread 0's
      // ticket, an acquire-release add at GPU scope: its release makes them
      // (cumulatively) visible to whoever takes a later ticket, and for the
      // CTA that takes the last one its acquire, passed on by the barrier
      // after it, orders every thread's reads of the other pieces after all
      // of their releases.
      __syncthreads();
      if (tid == 0) s_last = (ticket_acq_rel(&a.tickets[u]) == n_piece - 1);
      QSA_MARK(5);
      __syncthreads();
      if (s_last) {
        // every piece's (max, sum) at once, with the first kMergeBatch pieces'
        // accumulators already on their way; then the rest kMergeBatch at a time
        float* pm = wacc;                        // [n_piece][8] (the merge buffer is free now)
        float* pl = wacc + n_piece * kGroup;     // [n_piece][8]
        int* ps = reinterpret_cast<int*>(wacc + 2 * n_piece * kGroup);  // [n_piece] slots
        for (int k = tid; k < n_piece; k += kThreads) {
          const int cc = c_first + k;
          ps[k] = 2 * cc + (tile_begin(a, cc) >= uw0 ? 0 : 1);
        }
        __syncthreads();
        float x[kMergeBatch][8];  // 32 loads in flight per thread
        auto load_batch = [&](int k0) {
#pragma unroll
          for (int kk = 0; kk < kMergeBatch; ++kk) {
            const bool in = k0 + kk < n_piece;
            const float* pp = a.partials + (size_t)(in ? ps[k0 + kk] : 0) * kPartFloats + 2 * kGroup + tid;
#pragma unroll
            for (int h = 0; h < 8; ++h) x[kk][h] = in ? __ldcg(pp + h * kDim) : 0.f;
          }
        };
        load_batch(0);
        for (int i = tid; i < n_piece * kGroup; i += kThreads) {
          const float* pp = a.partials + (size_t)ps[i >> 3] * kPartFloats;
          pm[i] = __ldcg(pp + (i & 7));
          pl[i] = __ldcg(pp + kGroup + (i & 7));
        }
        __syncthreads();
        if (tid < kGroup) {
          float Ms = kNegInf;
          for (int k = 0; k < n_piece; ++k) Ms = fmaxf(Ms, pm[k * kGroup + tid]);
          const float Mbs = (Ms == kNegInf) ? 0.f : Ms;
          float Ls = 0.f;
          for (int k = 0; k < n_piece; ++k) Ls += pl[k * kGroup + tid] * exp2f(pm[k * kGroup + tid] - Mbs);
          sM[tid] = Mbs;
          sL[tid] = Ls;
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 8; ++h) o[h] = 0.f;
        for (int k0 = 0; k0 < n_piece; k0 += kMergeBatch) {
          if (k0 > 0) load_batch(k0);
#pragma unroll
          for (int kk = 0; kk < kMergeBatch; ++kk) {
            if (k0 + kk >= n_piece) break;
#pragma unroll
            for (int h = 0; h < 8; ++h) o[h] += exp2f(pm[(k0 + kk) * kGroup + h] - sM[h]) * x[kk][h];
          }
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float l = sL[h];
          orow[h * kDim + tid] = __float2bfloat16_rn(l > 0.f ? o[h] / l * vscale : 0.f);
        }
        if (tid == 0) a.tickets[u] = 0;  // ready for the next launch
        QSA_MARK(6);
      }
    }
    if (!more) break;
    ++u;
    t = 0;
  }
  QSA_MARK(3);
  pdl_trigger();
}

// Selected positions -> cache rows of KV head 0 (-1 for none), with the
// checks of the query position, the selection and the page table.
__global__ void __launch_bounds__(256) resolve_kernel(const int32_t* __restrict__ sel_pos,
                                                      const int32_t* __restrict__ q_pos,
                                                      const int32_t* __restrict__ page_table,
                                                      int32_t* __restrict__ sel_row, int32_t* err, int n_q,
                                                      int n_kv, int page_shift, int max_pages, int num_pages,
                                                      int width) {
  pdl_trigger();  // the attention kernel waits for this whole grid anyway
  const int row = blockIdx.x, r = row / n_q, j = row - r * n_q;
  const int p = q_pos[row];
  const bool p_ok = p >= 0 && (p >> page_shift) < max_pages;
  if (!p_ok && threadIdx.x == 0) record_error(err, kErrQueryPos, r, j, p);
  const int page_mask = (1 << page_shift) - 1;
  for (int i = threadIdx.x; i < width; i += blockDim.x) {
    int ri = -1;
    const int pos = sel_pos[(size_t)row * width + i];
    if (p_ok && pos >= 0) {
      if (pos > p) {
        record_error(err, kErrSelPos, r, j, pos);
      } else {
        const int page = page_table[(size_t)r * max_pages + (pos >> page_shift)];
        if (page < 0 || page >= num_pages)
          record_error(err, kErrPage, r, j, page);
        else
          ri = ((page * n_kv) << page_shift) + (pos & page_mask);
      }
    }
    sel_row[(size_t)row * width + i] = ri;
  }
}

// Draft steps: row (r, j) of the widened selection = the reused row's
// positions (checked against the row's own query position p_src), then
// p_src + 1 .. p, as cache rows of KV head 0 (-1 for none).
__global__ void __launch_bounds__(256) draft_resolve_kernel(const int32_t* __restrict__ sel_pos,
                                                            const int32_t* __restrict__ sel_q_pos, int n_sel,
                                                            const int32_t* __restrict__ src,
                                                            const int32_t* __restrict__ q_pos,
                                                            const int32_t* __restrict__ page_table,
                                                            int32_t* __restrict__ sel_row, int32_t* err, int n_q,
                                                            int n_kv, int page_shift, int max_pages, int num_pages) {
  pdl_trigger();  // the attention kernel waits for this whole grid anyway
  const int row = blockIdx.x, r = row / n_q, j = row - r * n_q;
  const int sj = src[row];
  const bool s_ok = sj >= 0 && sj < n_sel;
  const int ps = s_ok ? sel_q_pos[r * n_sel + sj] : -1;
  const int p = q_pos[row];
  const bool ok = s_ok && ps >= 0 && p >= ps && p - ps <= kMaxDraftGap && (p >> page_shift) < max_pages;
  if (!ok && threadIdx.x == 0) record_error(err, kErrDraft, r, j, s_ok ? p : sj);
  const int page_mask = (1 << page_shift) - 1;
  const int32_t* reused = sel_pos + ((size_t)r * n_sel + (s_ok ? sj : 0)) * kWidth;
  for (int i = threadIdx.x; i < kDraftWidth; i += blockDim.x) {
    int pos = -1;
    if (ok) {
      if (i < kWidth) {
        pos = reused[i];
        if (pos > ps) {
          record_error(err, kErrSelPos, r, j, pos);
          pos = -1;
        }
      } else if (i - kWidth < p - ps) {
        pos = ps + 1 + (i - kWidth);
      }
    }
    int ri = -1;
    if (pos >= 0) {
      const int page = page_table[(size_t)r * max_pages + (pos >> page_shift)];
      if (page < 0 || page >= num_pages)
        record_error(err, kErrPage, r, j, page);
      else
        ri = ((page * n_kv) << page_shift) + (pos & page_mask);
    }
    sel_row[(size_t)row * kDraftWidth + i] = ri;
  }
}

int page_shift_of(int page_size) {
  int shift = 0;
  while ((1 << shift) < page_size) ++shift;
  return shift;
}

}  // namespace

QSA_TRACE_HOST(trace_attn)

// whether clusters of n attention CTAs can be placed on the current device,
// per cache type (1 yes, 2 no)
DeviceSlots cluster_ok[2][kMaxCluster + 1];

AttnPlan attn_plan(const qsa_dims& d, int num_sms) {
  AttnPlan pl;
  pl.units = d.batch * d.n_q * d.n_kv_heads;
  const int tile = d.kv_dtype == QSA_KV_FP8_E4M3 ? 2 * kTile : kTile;
  pl.tiles = (d.width + tile - 1) / tile;
  const long long total = (long long)pl.units * pl.tiles;
  const long long resident =
      (long long)(d.kv_dtype == QSA_KV_FP8_E4M3 ? kCtasPerSm<true> : kCtasPerSm<false>) * num_sms;
  const int min_tiles = d.kv_dtype == QSA_KV_FP8_E4M3 ? kMinTilesPerCta<true> : kMinTilesPerCta<false>;
  const long long most = (total + min_tiles - 1) / min_tiles;
  pl.grid = (int)(most < resident ? most : resident);
  // The cluster form, where its merge on chip outweighs stream-K's balance:
  // each unit split over c <= kMaxCluster CTAs, with no CTA more than twice
  // the tiles of stream-K's largest share, and the clusters taking at most
  // 4/5 of the resident CTA slots, or 17/20 when that leaves fewer than 4
  // CTAs per unit (clusters must fit inside one GPC: large clusters filling
  // most slots do not place in one wave). Its CTAs' pieces merge through
  // distributed shared memory instead of the workspace (pl.grid keeps the
  // stream-K count, which the workspace is sized for and which the launch
  // falls back to). Measured against stream-K (config 2): batch 1 29.8 ->
  // 27.3 us, 4 34.7 -> 31.2, 8 41.7 -> 39.4, 12 49.6 -> 47.1, 16 56.1 ->
  // 53.3, 24 70.6 -> 68.1; batch 32 (one CTA per unit at most) stays
  // stream-K. Clusters of 7 at batch 8 filling 448 of 456 slots took 49.7
  // us, of 8 at batch 6 filling 384 took 37.5 against 36.1 with 7. Clusters
  // of 16 at batch 1 (128 CTAs, one per SM): 26.5 -> 24.9 us against 11; at
  // batch 2 (256 CTAs) 26.6 -> 27.1, so only where each CTA has an SM; with
  // FP8 (tiles of 128 positions) 16 against 9 was slower (24.6 -> 25.1 us).
  pl.cl = 0;
  const long long share = (total + pl.grid - 1) / pl.grid;
  // BF16: as many CTAs per unit as keep each on an SM of its own (more CTAs,
  // shorter loops); otherwise no fewer than min_tiles tiles per CTA
  long long want = std::min<long long>(kMaxCluster, pl.tiles);
  if (d.kv_dtype == QSA_KV_FP8_E4M3 || (long long)pl.units * want > num_sms)
    want = std::min<long long>(want, (pl.tiles + min_tiles - 1) / min_tiles);
  const long long units = std::max(pl.units, 1);
  long long c = std::min<long long>(want, resident * 4 / 5 / units);
  if (c < 4) c = std::min<long long>(want, resident * 17 / 20 / units);
  if (c >= 2 && (pl.tiles + c - 1) / c <= 2 * share) pl.cl = (int)c;
  return pl;
}

cudaError_t launch_resolve(const qsa_dims& d, const int32_t* sel_pos, const int32_t* q_pos,
                           const int32_t* page_table, int32_t* sel_row, int32_t* err, cudaStream_t s) {
  return launch_k(resolve_kernel, dim3(d.batch * d.n_q), dim3(256), 0, s, false, sel_pos, q_pos, page_table,
                  sel_row, err, d.n_q, d.n_kv_heads, page_shift_of(d.page_size), d.max_pages, d.num_pages,
                  d.width);
}

cudaError_t launch_draft_resolve(const qsa_dims& d, const int32_t* sel_pos, const int32_t* sel_q_pos, int n_sel,
                                 const int32_t* src, const int32_t* q_pos, const int32_t* page_table,
                                 int32_t* sel_row, int32_t* err, cudaStream_t s) {
  return launch_k(draft_resolve_kernel, dim3(d.batch * d.n_q), dim3(256), 0, s, false, sel_pos, sel_q_pos, n_sel,
                  src, q_pos, page_table, sel_row, err, d.n_q, d.n_kv_heads, page_shift_of(d.page_size),
                  d.max_pages, d.num_pages);
}

cudaError_t launch_attn(const qsa_dims& d, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* sel_row, void* out,
                        int32_t* tickets, float* partials, const AttnPlan& plan, cudaStream_t s, bool pdl) {
  AttnArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.sel_row = sel_row;
  // rows of every KV head of a position stay inside the cache
  a.row_lim = (int)((long long)d.num_pages * d.n_kv_heads * d.page_size - (long long)(d.n_kv_heads - 1) * d.page_size);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.tickets = tickets;
  a.partials = partials;
  a.total = (long long)plan.units * plan.tiles;
  a.tiles = plan.tiles;
  a.grid = plan.grid;
  a.n_kv = d.n_kv_heads;
  a.page_size = d.page_size;
  a.width = d.width;
  a.sm_scale = d.sm_scale > 0.f ? d.sm_scale : 1.0f / sqrtf((float)d.head_dim);
  a.cl = 0;
  const bool fp8 = d.kv_dtype == QSA_KV_FP8_E4M3;
  if (plan.cl > 1 && plan.cl <= kMaxCluster && plan.cl <= plan.tiles) {
    // one cluster of cl CTAs per unit, if the device can place such clusters
    // (checked once per device and size; else the stream-K form below)
    auto kern = fp8 ? attn_kernel<true, true> : attn_kernel<false, true>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.units * plan.cl);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = plan.cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    const int placeable = cluster_ok[fp8 ? 1 : 0][plan.cl].get([&] {
      if (plan.cl > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        (void)cudaGetLastError();
        return 2;
      }
      cudaLaunchConfig_t one = cfg;
      one.numAttrs = 1;  // the cluster shape alone
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &one) != cudaSuccess) {
        (void)cudaGetLastError();
        return 2;
      }
      return n > 0 ? 1 : 2;  // 1: placeable, 2: not (both cached)
    });
    if (placeable == 1) {
      a.cl = plan.cl;
      return cudaLaunchKernelEx(&cfg, kern, a);
    }
  }
  if (fp8) return launch_k(attn_kernel<true, false>, dim3(plan.grid), dim3(kThreads), 0, s, pdl, a);
  return launch_k(attn_kernel<false, false>, dim3(plan.grid), dim3(kThreads), 0, s, pdl, a);
}

}  // namespace qsa
