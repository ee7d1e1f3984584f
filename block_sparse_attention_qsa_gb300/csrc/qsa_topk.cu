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
// Rows of up to kFastCap blocks - every 50K-token verify row - take the
// register path: thread t loads the scores of a contiguous run of at most
// kKpt blocks (16-byte loads when the buffer allows) and keeps their keys in
// registers. Pass 1 histograms the top 11 key bits; pass 2 classifies each
// key against the threshold bin into two register bit masks (above it, in
// it) and histograms the next 11 bits of the keys in it; a third digit is
// needed only when digit 2's bin is not taken whole. Because thread order is
// index order, one block-wide scan of the per-thread counts then lists the
// selected blocks ascending, the lowest-index ties first, and all threads
// write the outputs from that list with coalesced stores. Longer rows run the
// radix passes over the whole row (keys cached in shared memory when they
// fit, else read with several loads in flight), mark the selected and tied
// blocks in two shared bitmaps with warp ballots, and list them with one
// block scan over contiguous bitmap words per thread. The request's
// page table is staged in shared memory (before waiting on the score kernel,
// for a CTA's first row) so the cache rows written inside qsa_decode need no
// dependent global loads.
#include "qsa_internal.cuh"
#include "qsa_trace.cuh"

namespace qsa {
namespace {

QSA_TRACE_TABLE

constexpr int kThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kKpt = 24;         // most keys per thread on the register path
constexpr int kMaxCluster = 8;   // CTAs per row for small batches (portable cluster size)
constexpr int kFastCap = kKpt * kThreads - 4;  // longest row on it (3 blocks of alignment slack)
constexpr int kKeyCap = 49152;   // keys cached in shared memory on the long-row path
constexpr int kPtCap = 4096;     // page-table entries staged in shared memory
// header: hist[2048], hist2[2048], wsum[64], res[8], blk[512], pt[kPtCap]
constexpr int kHdrWords = 2048 + 2048 + 64 + 8 + kTopK + kPtCap;
constexpr int kBatch = 8;        // score loads in flight per thread (long-row path)

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

// Reads the row's scores with kBatch loads in flight and calls f(index,
// valid, key) on all lanes of a warp together (index >= n: valid false).
template <typename F>
__device__ __forceinline__ void for_each_score(const float* srow, int n, F&& f) {
  const int lane = threadIdx.x & 31;
  for (int wb = threadIdx.x & ~31; wb < n; wb += kThreads * kBatch) {  // warp-uniform
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = wb + lane + u * kThreads;
      v[u] = i < n ? srow[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (wb + u * kThreads >= n) break;  // warp-uniform
      const int i = wb + lane + u * kThreads;
      f(i, i < n, order_key(v[u]));
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

// cache row of position pos of request r (KV head 0), or -1 for a bad page;
// pt: the request's page table staged in shared memory, or null
__device__ __forceinline__ int row_of(const RowOut& ro, const int32_t* pt, int r, int pos, int32_t* err, int j) {
  const int pi = pos >> ro.page_shift;
  const int page = pt ? pt[pi] : ro.page_table[(size_t)r * ro.max_pages + pi];
  if (page < 0 || page >= ro.num_pages) {
    record_error(err, kErrPage, r, j, page);
    return -1;
  }
  return (page * ro.n_kv << ro.page_shift) + (pos & ((1 << ro.page_shift) - 1));
}

// histogram update (plain shared-memory atomics: measured on GB300, grouping
// equal bins of a warp with match.any first costs several times more)
__device__ __forceinline__ void hist_add(uint32_t* hist, bool valid, uint32_t bin, int) {
  if (valid) atomicAdd(&hist[bin], 1u);
}

// The register path for one row: thread t holds the keys of blocks
// [t KPT, t KPT + KPT) in "virtual" indices v = i + off, where off makes the
// 16-byte loads aligned. Lists the row's kTopK selected blocks, ascending,
// in blk. Starts after a barrier (zeroed histograms); ends with one.
template <int KPT>
__device__ __forceinline__ void select_regs(const float* srow, int n, int off, bool vec, uint32_t* hist,
                                            uint32_t* hist2, uint32_t* wsum, int* res, int32_t* blk) {
  const int tid = threadIdx.x;
  const int span = n + off;
  const int v0 = tid * KPT;
  const int lo = max(0, off - v0), hi = min(KPT, span - v0);  // valid entries [lo, hi)
  constexpr uint32_t kAll = (1u << KPT) - 1u;
  const uint32_t valid_m = hi > lo ? (kAll >> (KPT - hi)) & ~((1u << lo) - 1u) : 0u;
  const float* abase = srow - off;

  // pass 1: keys into registers, histogram of the top 11 bits
  uint32_t key[KPT];
#pragma unroll
  for (int q = 0; q < KPT / 4; ++q) {
    const int v = v0 + 4 * q;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (vec) {
      if (v < span && v + 4 > off) f = *reinterpret_cast<const float4*>(abase + v);
    } else {
      if (v < span) f.x = abase[v];
      if (v + 1 < span) f.y = abase[v + 1];
      if (v + 2 < span) f.z = abase[v + 2];
      if (v + 3 < span) f.w = abase[v + 3];
    }
    key[4 * q + 0] = order_key(f.x);
    key[4 * q + 1] = order_key(f.y);
    key[4 * q + 2] = order_key(f.z);
    key[4 * q + 3] = order_key(f.w);
  }
  if (valid_m == kAll) {
#pragma unroll
    for (int e = 0; e < KPT; ++e) atomicAdd(&hist[key[e] >> 21], 1u);
  } else if (valid_m) {
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if ((valid_m >> e) & 1u) atomicAdd(&hist[key[e] >> 21], 1u);
  }
  __syncthreads();
  uint32_t need = kTopK;
  find_bin<2048>(hist, need, wsum, res);
  const uint32_t d1 = (uint32_t)res[0];
  need -= (uint32_t)res[1];

  // pass 2: keys above the threshold bin / in it; digit 2 of the latter
  const uint32_t lo_key = d1 << 21;                                 // first key of bin d1
  const uint32_t hi_key = d1 == 2047u ? 0xffffffffu : ((d1 + 1u) << 21) - 1u;  // its last key
  uint32_t gt_m = 0, eq_m = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    gt_m |= (uint32_t)(key[e] > hi_key) << e;
    eq_m |= (uint32_t)(key[e] >= lo_key) << e;
  }
  gt_m &= valid_m;
  eq_m &= valid_m & ~gt_m;
  if (eq_m) {
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if ((eq_m >> e) & 1u) atomicAdd(&hist2[(key[e] >> 10) & 2047u], 1u);
  }
  for (int i = tid; i < 1024; i += kThreads) hist[i] = 0;
  __syncthreads();
  find_bin<2048>(hist2, need, wsum, res);
  const uint32_t d2 = (uint32_t)res[0];
  need -= (uint32_t)res[1];
  const uint32_t prefix = (d1 << 11) | d2;
  // when digit 2's bin is taken whole, no third digit is needed
  const bool whole = hist2[d2] == need;
  uint32_t T = prefix << 10;
  if (!whole) {
    // pass 3: digit 3 of the candidates sharing the prefix
    if (eq_m) {
#pragma unroll
      for (int e = 0; e < KPT; ++e)
        if (((eq_m >> e) & 1u) && (key[e] >> 10) == prefix) atomicAdd(&hist[key[e] & 1023u], 1u);
    }
    __syncthreads();
    find_bin<1024>(hist, need, wsum, res);
    T |= (uint32_t)res[0];
    need -= (uint32_t)res[1];  // blocks equal to T still to take, >= 1
  } else {
    need = 0;
  }
  // selected (above T, or the whole digit-2 bin) and tied (equal to T)
  uint32_t sel_m = gt_m, tie_m = 0;
  if (eq_m) {
    const uint32_t cut = whole ? T : T + 1u;  // selected: key >= cut (T < 2^32 - 1 here)
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const bool in = (eq_m >> e) & 1u;
      sel_m |= (uint32_t)(in && key[e] >= cut) << e;
      tie_m |= (uint32_t)(in && !whole && key[e] == T) << e;
    }
  }
  // thread order is index order: one scan lists the selection ascending,
  // the lowest-index ties first
  uint32_t total;
  const uint32_t excl = block_excl_scan(((uint32_t)__popc(tie_m) << 16) | (uint32_t)__popc(sel_m), wsum, &total);
  const uint32_t e_before = excl >> 16, s_before = excl & 0xffffu;
  uint32_t take = need > e_before ? min(need - e_before, (uint32_t)__popc(tie_m)) : 0u;
  uint32_t rest = tie_m;
  for (; take > 0; --take) rest &= rest - 1u;  // drop the lowest `take` ties: they are taken
  uint32_t pick = sel_m | (tie_m ^ rest);
  uint32_t slot = s_before + min(e_before, need);
  while (pick) {
    const int e = __ffs(pick) - 1;
    if (slot < (uint32_t)kTopK) blk[slot] = v0 + e - off;  // exactly kTopK; the bound is a guard
    ++slot;
    pick &= pick - 1u;
  }
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const float* __restrict__ scores,
                                                           const int32_t* __restrict__ q_pos,
                                                           int32_t* __restrict__ sel_blk,
                                                           int32_t* __restrict__ sel_pos,
                                                           int32_t* err, const RowOut ro, int rows,
                                                           int n_q, int max_blocks, int fast_cap,
                                                           int key_cap, bool vec) {
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* hist = sm;                                // [2048] digits 1 and 3
  uint32_t* hist2 = hist + 2048;                      // [2048] digit 2
  uint32_t* wsum = hist2 + 2048;                      // [2][32]
  int* res = reinterpret_cast<int*>(wsum + 64);       // [8]
  int32_t* blk = res + 8;                             // [512] the selection, ascending
  int32_t* pt_s = blk + kTopK;                        // [kPtCap] the request's page table
  // long-row path: keys[key_cap]
  uint32_t* body = sm + kHdrWords;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  QSA_MARK(0);

  // Inputs of a row that do not come from the score kernel: its position and
  // its request's page table (staged when it fits).
  int p = 0;
  bool pt_ok = false;
  auto stage_row = [&](int row) {
    p = q_pos[row];
    const int r = row / n_q;
    pt_ok = false;
    if (ro.page_table && p >= 0) {
      const int pages = min((p >> ro.page_shift) + 1, ro.max_pages);
      if (pages <= kPtCap) {
        pt_ok = true;
        for (int i = tid; i < pages; i += kThreads) pt_s[i] = ro.page_table[(size_t)r * ro.max_pages + i];
      }
    }
  };
  for (int i = tid; i < 2 * kHistBins; i += kThreads) hist[i] = 0;
  if (blockIdx.x < rows) stage_row(blockIdx.x);

  pdl_wait();  // the scores come from the previous kernel
  QSA_MARK(1);
  // Let the attention kernel launch now: its CTAs wait on the SMs this grid
  // leaves free, and their own wait still covers every selection written here.
  pdl_trigger();
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    if (row != (int)blockIdx.x) stage_row(row);
    __syncthreads();  // staged page table and zeroed histograms
    int32_t* ob = sel_blk ? sel_blk + (size_t)row * kTopK : nullptr;
    int32_t* op = sel_pos ? sel_pos + (size_t)row * kWidth : nullptr;
    int32_t* orow = ro.page_table ? ro.sel_row + (size_t)row * kWidth : nullptr;
    const int32_t* pt = pt_ok ? pt_s : nullptr;
    const int r = row / n_q, j = row - r * n_q;
    const bool p_ok = p >= 0 && n_full_of(p) <= max_blocks && (!orow || (p >> ro.page_shift) < ro.max_pages);
    const int n = p_ok ? n_full_of(p) : 0;
    if (!p_ok || n <= kTopK) {
      if (!p_ok && tid == 0) record_error(err, kErrQueryPos, r, j, p);
      // every full block is kept (positions 0..p), or nothing for a bad position
      if (ob)
        for (int i = tid; i < kTopK; i += kThreads) ob[i] = i < n ? i : -1;
      if (op)
        for (int i = tid; i < kWidth; i += kThreads) op[i] = (p_ok && i <= p) ? i : -1;
      if (orow)
        for (int i = tid; i < kWidth; i += kThreads) orow[i] = (p_ok && i <= p) ? row_of(ro, pt, r, i, err, j) : -1;
      __syncthreads();  // shared memory is reused by the next row
      continue;
    }
    const int npart = (p + 1) & 3;
    const float* srow = scores + (size_t)row * max_blocks;

    if (n <= fast_cap) {
      // ---- register path ----
      const int off = vec ? (int)(((size_t)row * max_blocks) & 3) : 0;
      const int span = n + off;
      if (span <= 4 * kThreads) select_regs<4>(srow, n, off, vec, hist, hist2, wsum, res, blk);
      else if (span <= 8 * kThreads) select_regs<8>(srow, n, off, vec, hist, hist2, wsum, res, blk);
      else if (span <= 12 * kThreads) select_regs<12>(srow, n, off, vec, hist, hist2, wsum, res, blk);
      else if (span <= 16 * kThreads) select_regs<16>(srow, n, off, vec, hist, hist2, wsum, res, blk);
      else if (span <= 20 * kThreads) select_regs<20>(srow, n, off, vec, hist, hist2, wsum, res, blk);
      else select_regs<24>(srow, n, off, vec, hist, hist2, wsum, res, blk);
    } else {
      // ---- long rows: radix passes over the whole row ----
      const bool in_smem = n <= key_cap;  // keys cached in shared memory
      uint32_t* keys = body;
      // f(i, valid, key) for the blocks [c0, c0 + cn), on all lanes of a warp
      // together (a warp's lanes take 32 consecutive blocks); global scores are
      // read with kBatch loads in flight
      auto each_key = [&](int c0, int cn, auto&& f) {
        if (in_smem) {
          for (int wb = tid & ~31; wb < cn; wb += kThreads) {  // warp-uniform
            const int i = wb + lane;
            f(i, i < cn, i < cn ? keys[c0 + i] : 0u);
          }
        } else {
          for_each_score(srow + c0, cn, f);
        }
      };
      for_each_score(srow, n, [&](int i, bool ok, uint32_t k) {
        if (in_smem && ok) keys[i] = k;
        hist_add(hist, ok, k >> 21, lane);
      });
      __syncthreads();
      uint32_t need = kTopK;
      find_bin<2048>(hist, need, wsum, res);
      const uint32_t d1 = (uint32_t)res[0];
      need -= (uint32_t)res[1];
      for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
      __syncthreads();
      each_key(0, n, [&](int, bool ok, uint32_t k) {
        if (ok && (k >> 21) == d1) atomicAdd(&hist[(k >> 10) & 2047u], 1u);
      });
      __syncthreads();
      find_bin<2048>(hist, need, wsum, res);
      const uint32_t d2 = (uint32_t)res[0];
      need -= (uint32_t)res[1];
      const uint32_t prefix = (d1 << 11) | d2;
      // when digit 2's bin is taken whole, no third digit is needed
      const bool whole = hist[d2] == need;
      uint32_t T = prefix << 10;
      __syncthreads();  // every thread has read hist[d2]
      if (!whole) {
        for (int i = tid; i < 1024; i += kThreads) hist[i] = 0;
        __syncthreads();
        each_key(0, n, [&](int, bool ok, uint32_t k) {
          if (ok && (k >> 10) == prefix) atomicAdd(&hist[k & 1023u], 1u);
        });
        __syncthreads();
        find_bin<1024>(hist, need, wsum, res);
        T |= (uint32_t)res[0];
        need -= (uint32_t)res[1];  // blocks equal to T still to take, >= 1
      } else {
        need = 0;
      }

      // ordered listing, 65,536 blocks at a time: one ballot pass marks the
      // selected blocks (key >= cut) and the tied ones (key == T, unless digit
      // 2's bin is taken whole) in two shared bitmaps (the histograms' space);
      // then each thread owns a contiguous run of bitmap words, and one block
      // scan of the per-thread counts gives every pick its slot: ascending
      // blocks, the lowest-index ties first
      uint32_t* sel_bits = hist2;  // [2048]
      uint32_t* tie_bits = hist;   // [2048]
      const uint32_t cut = whole ? T : T + 1u;  // T < 2^32 - 1 here
      uint32_t sel_done = 0, tie_done = 0;  // counts in the chunks before (the same in every thread)
      for (int c0 = 0; c0 < n; c0 += 65536) {
        const int cn = min(65536, n - c0);
        const int nw = (cn + 31) >> 5;
        __syncthreads();  // the histograms / previous chunk's bitmaps are no longer read
        each_key(c0, cn, [&](int i, bool ok, uint32_t k) {
          const uint32_t sb = __ballot_sync(kFull, ok && k >= cut);
          const uint32_t tb = __ballot_sync(kFull, ok && !whole && k == T);
          if (lane == 0) {
            sel_bits[i >> 5] = sb;
            tie_bits[i >> 5] = tb;
          }
        });
        __syncthreads();
        const int wpt = (nw + kThreads - 1) / kThreads;  // bitmap words per thread
        const int w0 = min(nw, tid * wpt), w1 = min(nw, w0 + wpt);
        uint32_t cs = 0, ce = 0;
        for (int w = w0; w < w1; ++w) {
          cs += (uint32_t)__popc(sel_bits[w]);
          ce += (uint32_t)__popc(tie_bits[w]);
        }
        // selected blocks number at most kTopK (< 2^11); ties at most 65,536
        uint32_t total;
        const uint32_t excl = block_excl_scan((ce << 11) | cs, wsum, &total);
        const uint32_t e_before = tie_done + (excl >> 11), s_before = sel_done + (excl & 2047u);
        uint32_t take = need > e_before ? min(need - e_before, ce) : 0u;
        uint32_t slot = s_before + min(e_before, need);
        for (int w = w0; w < w1; ++w) {
          uint32_t tb = tie_bits[w], keep = 0;
          for (; take > 0 && tb; --take) {  // the lowest ties are taken
            keep |= tb & (0u - tb);
            tb &= tb - 1u;
          }
          uint32_t pick = sel_bits[w] | keep;
          while (pick) {
            const int bit = __ffs(pick) - 1;
            if (slot < (uint32_t)kTopK) blk[slot] = c0 + 32 * w + bit;  // exactly kTopK; the bound is a guard
            ++slot;
            pick &= pick - 1u;
          }
        }
        sel_done += total & 2047u;
        tie_done += total >> 11;
      }
    }
    __syncthreads();  // the selection list is complete
    QSA_MARK(2);
    // outputs, coalesced: block ids, their positions (then the unfilled block's), cache rows
    if (ob)
      for (int i = tid; i < kTopK; i += kThreads) ob[i] = blk[i];
    if (op || orow)
      for (int i = tid; i < kWidth; i += kThreads) {
        int pos;
        if (i < kBlock * kTopK) pos = kBlock * blk[i >> 2] + (i & 3);
        else pos = (i - kBlock * kTopK < npart) ? kBlock * n + (i - kBlock * kTopK) : -1;
        if (op) op[i] = pos;
        if (orow) orow[i] = pos < 0 ? -1 : row_of(ro, pt, r, pos, err, j);
      }
    for (int i = tid; i < 2 * kHistBins; i += kThreads) hist[i] = 0;
    __syncthreads();  // shared memory is reused by the next row
  }
  QSA_MARK(3);
}


// ---------------------------------------------------------------------------
// Small batches: a thread-block cluster of C CTAs per row. CTA k of the
// cluster keeps the keys of blocks [n k / C, n (k+1) / C) in registers (a
// contiguous run of at most KPT per thread); each radix digit's histogram is
// counted per CTA and summed through distributed shared memory between
// cluster barriers; a cluster-level prefix of the per-CTA counts gives every
// CTA the global slots of its picks, which it writes directly. The hardware
// cluster barrier is the only wait.
// ---------------------------------------------------------------------------

constexpr int kClHdrWords = 2048 + 2048 + 2048 + 64 + 8 + 8 + kPtCap;  // hist, hist2, sum, wsum, res, cnt, pt

template <int KPT>
__global__ void __launch_bounds__(kThreads, 1) topk_cluster_kernel(const float* __restrict__ scores,
                                                                   const int32_t* __restrict__ q_pos,
                                                                   int32_t* __restrict__ sel_blk,
                                                                   int32_t* __restrict__ sel_pos, int32_t* err,
                                                                   const RowOut ro, int n_q, int max_blocks) {
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* hist = sm;             // [2048] this CTA's digit-1 (then digit-3) counts
  uint32_t* hist2 = hist + 2048;   // [2048] this CTA's digit-2 counts
  uint32_t* gsum = hist2 + 2048;   // [2048] the cluster's sums
  uint32_t* wsum = gsum + 2048;    // [2][32]
  int* res = reinterpret_cast<int*>(wsum + 64);  // [8]
  uint32_t* cnt = wsum + 64 + 8;   // [8]: this CTA's selected and tied counts
  int32_t* pt_s = reinterpret_cast<int32_t*>(cnt + 8);
  const int tid = threadIdx.x;
  const uint32_t crank = cluster_rank(), C = cluster_size();
  const int row = blockIdx.x / (int)C;
  const int r = row / n_q, j = row - r * n_q;
  QSA_MARK(0);

  // inputs that do not come from the score kernel
  const int p = q_pos[row];
  bool pt_ok = false;
  if (ro.page_table && p >= 0) {
    const int pages = min((p >> ro.page_shift) + 1, ro.max_pages);
    if (pages <= kPtCap) {
      pt_ok = true;
      for (int i = tid; i < pages; i += kThreads) pt_s[i] = ro.page_table[(size_t)r * ro.max_pages + i];
    }
  }
  for (int i = tid; i < 4096; i += kThreads) hist[i] = 0;  // hist and hist2
  pdl_wait();  // the scores come from the previous kernel
  QSA_MARK(1);
  pdl_trigger();
  __syncthreads();

  int32_t* ob = sel_blk ? sel_blk + (size_t)row * kTopK : nullptr;
  int32_t* op = sel_pos ? sel_pos + (size_t)row * kWidth : nullptr;
  int32_t* orow = ro.page_table ? ro.sel_row + (size_t)row * kWidth : nullptr;
  const int32_t* pt = pt_ok ? pt_s : nullptr;
  const bool p_ok = p >= 0 && n_full_of(p) <= max_blocks && (!orow || (p >> ro.page_shift) < ro.max_pages);
  const int n = p_ok ? n_full_of(p) : 0;
  if (!p_ok || n <= kTopK) {
    if (crank == 0) {
      if (!p_ok && tid == 0) record_error(err, kErrQueryPos, r, j, p);
      if (ob)
        for (int i = tid; i < kTopK; i += kThreads) ob[i] = i < n ? i : -1;
      if (op)
        for (int i = tid; i < kWidth; i += kThreads) op[i] = (p_ok && i <= p) ? i : -1;
      if (orow)
        for (int i = tid; i < kWidth; i += kThreads) orow[i] = (p_ok && i <= p) ? row_of(ro, pt, r, i, err, j) : -1;
    }
    QSA_MARK(3);
    cluster_sync();
    return;
  }
  const int npart = (p + 1) & 3;
  const float* srow = scores + (size_t)row * max_blocks;
  const int b0 = (int)((long long)n * crank / C), b1 = (int)((long long)n * (crank + 1) / C);
  const int v0 = b0 + tid * KPT;
  const int cnt_here = min(KPT, max(0, b1 - v0));
  constexpr uint32_t kAll = KPT >= 32 ? 0xffffffffu : (1u << KPT) - 1u;
  const uint32_t valid_m = cnt_here >= KPT ? kAll : ((1u << cnt_here) - 1u);

  // the cluster's sum of a per-CTA histogram, into gsum
  auto cluster_sum = [&](const uint32_t* local, int nbins) {
    for (int i = tid; i < nbins; i += kThreads) {
      uint32_t acc = 0;
      for (uint32_t k = 0; k < C; ++k) acc += ld_peer(peer_addr(local + i, k));
      gsum[i] = acc;
    }
    __syncthreads();
  };

  // pass 1: keys into registers, this CTA's histogram of the top 11 bits
  uint32_t key[KPT];
#pragma unroll
  for (int e = 0; e < KPT; ++e) key[e] = ((valid_m >> e) & 1u) ? order_key(srow[v0 + e]) : 0u;
#pragma unroll
  for (int e = 0; e < KPT; ++e)
    if ((valid_m >> e) & 1u) atomicAdd(&hist[key[e] >> 21], 1u);
  cluster_sync();
  cluster_sum(hist, 2048);
  uint32_t need = kTopK;
  find_bin<2048>(gsum, need, wsum, res);
  const uint32_t d1 = (uint32_t)res[0];
  need -= (uint32_t)res[1];

  // pass 2: above the threshold bin / in it; digit 2 of the latter
  const uint32_t lo_key = d1 << 21;
  const uint32_t hi_key = d1 == 2047u ? 0xffffffffu : ((d1 + 1u) << 21) - 1u;
  uint32_t gt_m = 0, eq_m = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    gt_m |= (uint32_t)(key[e] > hi_key) << e;
    eq_m |= (uint32_t)(key[e] >= lo_key) << e;
  }
  gt_m &= valid_m;
  eq_m &= valid_m & ~gt_m;
  if (eq_m) {
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if ((eq_m >> e) & 1u) atomicAdd(&hist2[(key[e] >> 10) & 2047u], 1u);
  }
  cluster_sync();  // every CTA's digit-1 reads are done; digit-2 counts are complete
  cluster_sum(hist2, 2048);
  find_bin<2048>(gsum, need, wsum, res);
  const uint32_t d2 = (uint32_t)res[0];
  need -= (uint32_t)res[1];
  const uint32_t prefix = (d1 << 11) | d2;
  const bool whole = gsum[d2] == need;  // the same in every CTA
  uint32_t T = prefix << 10;
  if (!whole) {
    // pass 3: digit 3 of the keys sharing the prefix
    for (int i = tid; i < 1024; i += kThreads) hist[i] = 0;
    __syncthreads();
    if (eq_m) {
#pragma unroll
      for (int e = 0; e < KPT; ++e)
        if (((eq_m >> e) & 1u) && (key[e] >> 10) == prefix) atomicAdd(&hist[key[e] & 1023u], 1u);
    }
    cluster_sync();
    cluster_sum(hist, 1024);
    find_bin<1024>(gsum, need, wsum, res);
    T |= (uint32_t)res[0];
    need -= (uint32_t)res[1];
  } else {
    need = 0;
  }
  uint32_t sel_m = gt_m, tie_m = 0;
  if (eq_m) {
    const uint32_t cut = whole ? T : T + 1u;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const bool in = (eq_m >> e) & 1u;
      sel_m |= (uint32_t)(in && key[e] >= cut) << e;
      tie_m |= (uint32_t)(in && !whole && key[e] == T) << e;
    }
  }
  QSA_MARK(2);
  // this CTA's counts in index order, then the CTAs before it in the cluster.
  // Inside one CTA the packed (ties << 16 | selected) scan cannot overflow: a
  // CTA holds at most 32 x 1024 keys and selects at most kTopK. Summed over
  // the lower-ranked CTAs the ties can pass 65,535 (a row of 131,073 equal
  // scores puts 65,536 in the first four CTAs of eight), so the cluster-level
  // counts are kept in two separate words.
  uint32_t total;
  const uint32_t excl = block_excl_scan(((uint32_t)__popc(tie_m) << 16) | (uint32_t)__popc(sel_m), wsum, &total);
  if (tid == 0) {
    cnt[0] = total & 0xffffu;  // selected
    cnt[1] = total >> 16;      // tied
  }
  cluster_sync();
  uint32_t s_peer = 0, e_peer = 0;  // selected and tied counts of the lower-ranked CTAs
  for (uint32_t k = 0; k < crank; ++k) {
    s_peer += ld_peer(peer_addr(cnt, k));
    e_peer += ld_peer(peer_addr(cnt + 1, k));
  }
  const uint32_t e_before = e_peer + (excl >> 16), s_before = s_peer + (excl & 0xffffu);
  uint32_t take = need > e_before ? min(need - e_before, (uint32_t)__popc(tie_m)) : 0u;
  uint32_t rest = tie_m;
  for (; take > 0; --take) rest &= rest - 1u;
  uint32_t pick = sel_m | (tie_m ^ rest);
  uint32_t slot = s_before + min(e_before, need);
  while (pick) {
    const int e = __ffs(pick) - 1;
    if (slot < (uint32_t)kTopK) {  // exactly kTopK; the bound is a guard
      const int b = v0 + e;
      if (ob) ob[slot] = b;
      const int pos = kBlock * b;
      const int base = orow ? row_of(ro, pt, r, pos, err, j) : 0;  // a block never straddles a page
#pragma unroll
      for (int k = 0; k < kBlock; ++k) {
        if (op) op[kBlock * slot + k] = pos + k;
        if (orow) orow[kBlock * slot + k] = base < 0 ? -1 : base + k;
      }
    }
    ++slot;
    pick &= pick - 1u;
  }
  if (crank == 0 && tid < kBlock - 1) {
    const int pos = tid < npart ? kBlock * n + tid : -1;
    if (op) op[kBlock * kTopK + tid] = pos;
    if (orow) orow[kBlock * kTopK + tid] = pos < 0 ? -1 : row_of(ro, pt, r, pos, err, j);
  }
  QSA_MARK(3);
  cluster_sync();  // no CTA leaves while another may still read its counts
}

template <int KPT>
cudaError_t launch_topk_cluster(int C, int rows, const float* scores, const int32_t* q_pos, int32_t* sel_blk,
                                int32_t* sel_pos, int32_t* err, const RowOut& ro, int n_q, int max_blocks,
                                cudaStream_t s, bool pdl) {
  const size_t smem = (size_t)kClHdrWords * sizeof(uint32_t);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows * C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<KPT>, scores, q_pos, sel_blk, sel_pos, err, ro, n_q,
                            max_blocks);
}

}  // namespace

QSA_TRACE_HOST(trace_topk)

cudaError_t launch_topk(const qsa_dims& d, const float* scores, const int32_t* q_pos,
                        int32_t* sel_blk, int32_t* sel_pos, int32_t* err, const int32_t* page_table,
                        int32_t* sel_row, cudaStream_t s, bool pdl) {
  const int rows = d.batch * d.n_q;
  // shared memory: the header, and the long-row path's keys (the register
  // path keeps its keys in registers)
  const int mb = d.max_blocks;
  const int mb32 = (mb + 31) / 32 * 32;
  const int fast_cap = mb <= kTopK ? 0 : (mb32 < kFastCap ? mb32 : kFastCap);
  const int key_cap = mb > kFastCap ? (mb < kKeyCap ? mb : kKeyCap) : 0;
  const size_t body = (size_t)key_cap;  // the register path needs no body
  const size_t smem = (kHdrWords + body) * sizeof(uint32_t);
  static DeviceSlots smem_slots;
  if (const cudaError_t e = smem_slots.raise_smem(topk_kernel, smem); e != cudaSuccess) return e;
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
  // Long rows (beyond the register path) and few of them: a cluster of C
  // CTAs per row, the largest C with every CTA on its own SM, when each CTA's
  // share of the longest row fits KPT <= 32 keys per thread (a batch-1
  // 262,144-token row takes the step from 121.6 us to 51.3 us). Rows the
  // register path holds are split in two only when the rows are very few:
  // measured at 15K blocks, a pair of CTAs per row takes a batch-1 step from
  // 33.1 to 31.2 us and batch 4 from 37.6 to 36.6 us, makes no difference
  // from 32 rows on, and 4 or 8 CTAs per row gain nothing more (their
  // barriers and reductions cost what the split saves).
  const int sms = device_sm_count();
  int C = 1;
  for (int c = kMaxCluster; c >= 2; c >>= 1)
    if ((long long)rows * c <= sms) {
      C = c;
      break;
    }
  if (mb <= kFastCap) C = (mb > 4096 && (long long)rows * 8 <= sms) ? 2 : 1;
  if (C > 1) {
    const int per_thread = ((mb + C - 1) / C + kThreads - 1) / kThreads;
    cudaError_t e = cudaErrorNotSupported;
    if (per_thread <= 4)
      e = launch_topk_cluster<4>(C, rows, scores, q_pos, sel_blk, sel_pos, err, ro, d.n_q, mb, s, pdl);
    else if (per_thread <= 8)
      e = launch_topk_cluster<8>(C, rows, scores, q_pos, sel_blk, sel_pos, err, ro, d.n_q, mb, s, pdl);
    else if (per_thread <= 16)
      e = launch_topk_cluster<16>(C, rows, scores, q_pos, sel_blk, sel_pos, err, ro, d.n_q, mb, s, pdl);
    else if (per_thread <= 32)
      e = launch_topk_cluster<32>(C, rows, scores, q_pos, sel_blk, sel_pos, err, ro, d.n_q, mb, s, pdl);
    if (e == cudaSuccess) return e;
    cudaGetLastError();  // a cluster the device cannot place: one CTA per row below
  }
  return launch_k(topk_kernel, dim3(grid), dim3(kThreads), smem, s, pdl, scores, q_pos, sel_blk,
                  sel_pos, err, ro, rows, d.n_q, d.max_blocks, fast_cap, key_cap,
                  (reinterpret_cast<uintptr_t>(scores) & 15u) == 0);
}

}  // namespace qsa
