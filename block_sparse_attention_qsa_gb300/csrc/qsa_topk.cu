// Top-512 block selection and the 2,051-wide selection buffer.
//
// The pages (arex-research.com, section "四类优化", bullet 1) say a persistent
// radix selector takes the top-k of the FP32 block-score buffer, that each
// query keeps at most 512 full blocks, and that the current unfilled block is
// appended without selection for a fixed width of 2,051.
//
// Design: one 1024-thread CTA per (request, query) row, persistent over rows.
// Scores map to order-preserving 32-bit keys (-0.0 folded onto +0.0, NaN
// below everything), so "largest score, lower index on ties" becomes "largest
// key, lower index on ties". A radix select on the keys finds the threshold
// key T (the 512th largest) and how many blocks equal to T are still needed.
//
// Rows of up to kFastCap blocks whose threshold bin holds at most kCandCap
// blocks - every 50K-token verify row - take the bitmap path: a first pass
// (8 loads in flight per thread) histograms the top 11 key bits; a second
// pass turns each 32 consecutive scores into one word of a "surely selected"
// bitmap (a higher bin) by warp ballot and appends the threshold bin's blocks
// to a candidate list; only those candidates - typically a few hundred - go
// through the two remaining radix passes. Selection is then two bitmaps
// (surely selected, equal to T) and one block-wide scan over 32-block words
// writes the block ids and positions in ascending order, the lowest-index
// ties first. Longer rows, and rows whose threshold bin is crowded, run the
// radix passes over the whole row (keys cached in shared memory when they
// fit) and compact in index order tile by tile.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kFastCap = 24576;  // longest row on the bitmap path (n/32 words <= kThreads)
constexpr int kKeyCap = 53248;   // keys cached in shared memory on the long-row path
constexpr int kHdrWords = 2048 + 64 + 8;
constexpr int kBatch = 8;        // score loads in flight per thread
constexpr int kCandCap = 8192;   // threshold-bin candidates held on the bitmap path

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Block-wide exclusive scan of one value per thread; returns the exclusive
// prefix and writes the total to *total. Uses wsum[0..32); ends with a barrier.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan(v, lane);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) wsum[lane] = warp_incl_scan(wsum[lane], lane);
  __syncthreads();
  const uint32_t excl = incl - v + (warp > 0 ? wsum[warp - 1] : 0u);
  *total = wsum[31];
  __syncthreads();
  return excl;
}

// Finds, scanning bins from the top, the bin d with count(bins > d) < need <=
// count(bins >= d). Writes d and count(bins > d) to res[0], res[1]. Ends with
// a barrier, after which every thread may read res.
template <int NB>
__device__ __forceinline__ void find_bin(const uint32_t* hist, uint32_t need, uint32_t* wsum,
                                         int* res) {
  constexpr int PER = NB / kThreads;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t c[PER];
  uint32_t tot = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    c[i] = hist[NB - 1 - (t * PER + i)];
    tot += c[i];
  }
  const uint32_t v = warp_incl_scan(tot, lane);
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) wsum[lane] = warp_incl_scan(wsum[lane], lane);
  __syncthreads();
  const uint32_t excl = v - tot + (warp > 0 ? wsum[warp - 1] : 0u);
  if (excl < need && need <= excl + tot) {
    uint32_t run = excl;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (run + c[i] >= need) {
        res[0] = NB - 1 - (t * PER + i);
        res[1] = (int)run;
        break;
      }
      run += c[i];
    }
  }
  __syncthreads();
}

// Reads the row's scores with kBatch loads in flight and calls f(index, key).
template <typename F>
__device__ __forceinline__ void for_each_score(const float* srow, int n, F&& f) {
  for (int base = threadIdx.x; base < n; base += kThreads * kBatch) {
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kThreads;
      v[u] = i < n ? srow[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kThreads;
      if (i < n) f(i, order_key(v[u]));
    }
  }
}

// Optional output inside qsa_decode: the cache row (for KV head 0) of every
// selected position, so the attention kernel needs no page lookup.
struct RowOut {
  const int32_t* page_table;  // [B][max_pages], or null: no rows written
  int32_t* sel_row;           // [rows][kWidth]
  int max_pages, num_pages, page_shift, n_kv;
};

// cache row of position pos of request r (KV head 0), or -1 for a bad page
__device__ __forceinline__ int row_of(const RowOut& ro, int r, int pos, int32_t* err, int j) {
  const int page = ro.page_table[(size_t)r * ro.max_pages + (pos >> ro.page_shift)];
  if (page < 0 || page >= ro.num_pages) {
    record_error(err, kErrPage, r, j, page);
    return -1;
  }
  return (page * ro.n_kv << ro.page_shift) + (pos & ((1 << ro.page_shift) - 1));
}

__device__ __forceinline__ void write_block(int32_t* ob, int32_t* op, int32_t* orow, const RowOut& ro,
                                            int32_t* err, int r, int j, uint32_t slot, int b) {
  if (slot >= (uint32_t)kTopK) return;  // exactly kTopK are selected; the bound is a guard
  ob[slot] = b;
  int32_t* o4 = op + kBlock * slot;
  o4[0] = kBlock * b;
  o4[1] = kBlock * b + 1;
  o4[2] = kBlock * b + 2;
  o4[3] = kBlock * b + 3;
  if (orow) {
    const int base = row_of(ro, r, kBlock * b, err, j);  // a block never straddles a page
    int32_t* w4 = orow + kBlock * slot;
    w4[0] = base;
    w4[1] = base < 0 ? -1 : base + 1;
    w4[2] = base < 0 ? -1 : base + 2;
    w4[3] = base < 0 ? -1 : base + 3;
  }
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const float* __restrict__ scores,
                                                           const int32_t* __restrict__ q_pos,
                                                           int32_t* __restrict__ sel_blk,
                                                           int32_t* __restrict__ sel_pos,
                                                           int32_t* err, const RowOut ro, int rows,
                                                           int n_q, int max_blocks, int fast_cap,
                                                           int key_cap) {
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;                           // [2048]
  uint32_t* wsum = hist + 2048;                  // [2][32]
  int* res = reinterpret_cast<int*>(wsum + 64);  // [8]
  // bitmap path: cand_idx[kCandCap], cand_key[kCandCap], 2 bitmaps[fast_cap / 32]
  // long-row path: keys[key_cap]
  uint32_t* body = sm + kHdrWords;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;

  pdl_wait();  // the scores come from the previous kernel
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int p = q_pos[row];
    int32_t* ob = sel_blk + (size_t)row * kTopK;
    int32_t* op = sel_pos + (size_t)row * kWidth;
    int32_t* orow = ro.page_table ? ro.sel_row + (size_t)row * kWidth : nullptr;
    const int r = row / n_q, j = row - r * n_q;
    const bool p_ok = p >= 0 && n_full_of(p) <= max_blocks && (!orow || (p >> ro.page_shift) < ro.max_pages);
    const int n = p_ok ? n_full_of(p) : 0;
    if (!p_ok || n <= kTopK) {
      if (!p_ok && tid == 0) record_error(err, kErrQueryPos, r, j, p);
      // every full block is kept (positions 0..p), or nothing for a bad position
      for (int i = tid; i < kTopK; i += kThreads) ob[i] = i < n ? i : -1;
      for (int i = tid; i < kWidth; i += kThreads) op[i] = (p_ok && i <= p) ? i : -1;
      if (orow)
        for (int i = tid; i < kWidth; i += kThreads) orow[i] = (p_ok && i <= p) ? row_of(ro, r, i, err, j) : -1;
      continue;
    }
    const int npart = (p + 1) & 3;
    const float* srow = scores + (size_t)row * max_blocks;

    // pass 1: histogram of the top 11 key bits
    const bool in_smem = n > fast_cap && n <= key_cap;  // long rows cache their keys
    uint32_t* keys = body;
    for (int i = tid; i < kHistBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for_each_score(srow, n, [&](int i, uint32_t k) {
      if (in_smem) keys[i] = k;
      atomicAdd(&hist[k >> 21], 1u);
    });
    __syncthreads();
    uint32_t need = kTopK;
    find_bin<2048>(hist, need, wsum, res);
    const uint32_t d1 = (uint32_t)res[0];
    need -= (uint32_t)res[1];
    const uint32_t nb = hist[d1];  // blocks in the threshold bin

    if (n <= fast_cap && nb <= (uint32_t)kCandCap) {
      // ---- bitmap path: one pass over the scores, candidates = the threshold bin ----
      const int nwords = (n + 31) >> 5;
      uint32_t* cand_idx = body;
      uint32_t* cand_key = cand_idx + kCandCap;
      uint32_t* sel_bits = cand_key + kCandCap;       // surely selected, one bit per block
      uint32_t* tie_bits = sel_bits + fast_cap / 32;  // equal to the threshold
      if (tid == 0) res[4] = 0;
      __syncthreads();
      for (int w0 = warp; w0 < nwords; w0 += (kThreads / 32) * kBatch) {
        float v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int i = ((w0 + u * (kThreads / 32)) << 5) + lane;
          v[u] = i < n ? srow[i] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int w = w0 + u * (kThreads / 32);
          if (w >= nwords) break;  // warp-uniform
          const int i = (w << 5) + lane;
          const uint32_t k = order_key(v[u]);
          const uint32_t d = k >> 21;
          const uint32_t gtm = __ballot_sync(kFull, i < n && d > d1);
          const uint32_t cm = __ballot_sync(kFull, i < n && d == d1);
          if (lane == 0) {
            sel_bits[w] = gtm;
            tie_bits[w] = 0u;
          }
          if (cm) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(reinterpret_cast<uint32_t*>(&res[4]), (uint32_t)__popc(cm));
            base = __shfl_sync(kFull, base, 0);
            const uint32_t slot = base + (uint32_t)__popc(cm & lt_mask);
            if ((cm & (1u << lane)) && slot < (uint32_t)kCandCap) {
              cand_idx[slot] = (uint32_t)i;
              cand_key[slot] = k;
            }
          }
        }
      }
      for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
      __syncthreads();
      const int nc = min(res[4], kCandCap);
      // pass 2 over the candidates: key bits 20..10
      for (int c = tid; c < nc; c += kThreads) atomicAdd(&hist[(cand_key[c] >> 10) & 2047u], 1u);
      __syncthreads();
      find_bin<2048>(hist, need, wsum, res);
      const uint32_t prefix = (d1 << 11) | (uint32_t)res[0];
      need -= (uint32_t)res[1];
      for (int i = tid; i < 1024; i += kThreads) hist[i] = 0;
      __syncthreads();
      // pass 3: key bits 9..0
      for (int c = tid; c < nc; c += kThreads) {
        const uint32_t k = cand_key[c];
        if ((k >> 10) == prefix) atomicAdd(&hist[k & 1023u], 1u);
      }
      __syncthreads();
      find_bin<1024>(hist, need, wsum, res);
      const uint32_t T = (prefix << 10) | (uint32_t)res[0];
      need -= (uint32_t)res[1];  // blocks equal to T still to take, >= 1
      for (int c = tid; c < nc; c += kThreads) {
        const uint32_t i = cand_idx[c];
        const uint32_t k = cand_key[c];
        if (k > T) atomicOr(&sel_bits[i >> 5], 1u << (i & 31));
        else if (k == T) atomicOr(&tie_bits[i >> 5], 1u << (i & 31));
      }
      __syncthreads();
      // one word of 32 blocks per thread, in index order
      uint32_t s = 0, e = 0;
      if (tid < nwords) {
        s = sel_bits[tid];
        e = tie_bits[tid];
      }
      uint32_t total;
      const uint32_t excl = block_excl_scan(((uint32_t)__popc(e) << 16) | (uint32_t)__popc(s), wsum, &total);
      const uint32_t e_before = excl >> 16, s_before = excl & 0xffffu;
      const uint32_t taken_before = min(e_before, need);
      uint32_t take = need > e_before ? min(need - e_before, (uint32_t)__popc(e)) : 0u;
      uint32_t rest = e;
      for (uint32_t t = 0; t < take; ++t) rest &= rest - 1u;  // drop the lowest `take` ties
      uint32_t word = s | (e ^ rest);
      uint32_t slot = s_before + taken_before;
      while (word) {
        const int b = __ffs(word) - 1;
        write_block(ob, op, orow, ro, err, r, j, slot++, (tid << 5) + b);
        word &= word - 1u;
      }
    } else {
      // ---- long rows (or a crowded threshold bin): radix passes over the whole row ----
      __syncthreads();  // every thread has read hist[d1]
      for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
      __syncthreads();
      auto key_at = [&](int i) { return in_smem ? keys[i] : order_key(srow[i]); };
      if (in_smem) {
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t k = keys[i];
          if ((k >> 21) == d1) atomicAdd(&hist[(k >> 10) & 2047u], 1u);
        }
      } else {
        for_each_score(srow, n, [&](int, uint32_t k) {
          if ((k >> 21) == d1) atomicAdd(&hist[(k >> 10) & 2047u], 1u);
        });
      }
      __syncthreads();
      find_bin<2048>(hist, need, wsum, res);
      const uint32_t prefix = (d1 << 11) | (uint32_t)res[0];
      need -= (uint32_t)res[1];
      for (int i = tid; i < 1024; i += kThreads) hist[i] = 0;
      __syncthreads();
      if (in_smem) {
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t k = keys[i];
          if ((k >> 10) == prefix) atomicAdd(&hist[k & 1023u], 1u);
        }
      } else {
        for_each_score(srow, n, [&](int, uint32_t k) {
          if ((k >> 10) == prefix) atomicAdd(&hist[k & 1023u], 1u);
        });
      }
      __syncthreads();
      find_bin<1024>(hist, need, wsum, res);
      const uint32_t T = (prefix << 10) | (uint32_t)res[0];
      need -= (uint32_t)res[1];

      // ordered compaction: keys > T, then the first `need` keys == T
      uint32_t n_sel = 0, n_tie = 0;
      int buf = 0;
      for (int base = 0; base < n; base += kThreads) {
        const int i = base + tid;
        const uint32_t k = (i < n) ? key_at(i) : 0u;
        const bool gt = (i < n) && k > T;
        const bool eq = (i < n) && k == T;
        const uint32_t gtm = __ballot_sync(kFull, gt);
        const uint32_t eqm = __ballot_sync(kFull, eq);
        uint32_t* wc = wsum + 32 * buf;
        if (lane == 0) wc[warp] = ((uint32_t)__popc(eqm) << 16) | (uint32_t)__popc(gtm);
        __syncthreads();
        const uint32_t c = wc[lane];
        const uint32_t incl = warp_incl_scan(c, lane);
        const uint32_t excl_w = __shfl_sync(kFull, incl - c, warp);
        const uint32_t total = __shfl_sync(kFull, incl, 31);
        const uint32_t E_w = excl_w >> 16, G_w = excl_w & 0xffffu;
        const uint32_t E_t = total >> 16, G_t = total & 0xffffu;
        const uint32_t rem_tile = need > n_tie ? need - n_tie : 0u;
        const uint32_t taken_before = min(rem_tile, E_w);
        const uint32_t rem_w = rem_tile > E_w ? rem_tile - E_w : 0u;
        const uint32_t my_eq = (uint32_t)__popc(eqm & lt_mask);
        if (gt || (eq && my_eq < rem_w))
          write_block(ob, op, orow, ro, err, r, j,
                      n_sel + G_w + taken_before + (uint32_t)__popc(gtm & lt_mask) + min(my_eq, rem_w), i);
        n_sel += G_t + min(rem_tile, E_t);
        n_tie += E_t;
        buf ^= 1;
      }
    }
    if (tid < kBlock - 1) {
      op[kBlock * kTopK + tid] = tid < npart ? kBlock * n + tid : -1;
      if (orow) orow[kBlock * kTopK + tid] = tid < npart ? row_of(ro, r, kBlock * n + tid, err, j) : -1;
    }
    __syncthreads();  // shared memory is reused by the next row
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_topk(const qsa_dims& d, const float* scores, const int32_t* q_pos,
                        int32_t* sel_blk, int32_t* sel_pos, int32_t* err, const int32_t* page_table,
                        int32_t* sel_row, cudaStream_t s, bool pdl) {
  const int rows = d.batch * d.n_q;
  // shared memory: header + either the bitmap path's candidates and two
  // bitmaps, or the long-row path's keys
  const int mb = d.max_blocks;
  const int mb32 = (mb + 31) / 32 * 32;
  const int fast_cap = mb <= kTopK ? 0 : (mb32 < kFastCap ? mb32 : kFastCap);
  const int key_cap = mb > kFastCap ? (mb < kKeyCap ? mb : kKeyCap) : 0;
  const size_t fast_words = fast_cap ? (size_t)2 * kCandCap + 2 * (fast_cap / 32) : 0;
  const size_t long_words = (size_t)key_cap;
  const size_t body = fast_words > long_words ? fast_words : long_words;
  const size_t smem = (kHdrWords + body) * sizeof(uint32_t);
  static size_t set_bytes[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || set_bytes[dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) set_bytes[dev] = smem;
  }
  int grid = rows < device_sm_count() ? rows : device_sm_count();
  if (grid < 1) grid = 1;
  RowOut ro;
  ro.page_table = page_table;
  ro.sel_row = sel_row;
  ro.max_pages = d.max_pages;
  ro.num_pages = d.num_pages;
  int shift = 0;
  while ((1 << shift) < d.page_size) ++shift;
  ro.page_shift = shift;
  ro.n_kv = d.n_kv_heads;
  return launch_k(topk_kernel, dim3(grid), dim3(kThreads), smem, s, pdl, scores, q_pos, sel_blk,
                  sel_pos, err, ro, rows, d.n_q, d.max_blocks, fast_cap, key_cap);
}

}  // namespace qsa
