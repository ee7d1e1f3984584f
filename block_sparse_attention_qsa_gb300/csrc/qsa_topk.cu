// Top-512 block selection and the 2,051-wide selection buffer.
//
// The pages (arex-research.com, section "四类优化", bullet 1) say a persistent
// radix selector takes the top-k of the FP32 block-score buffer, that each
// query keeps at most 512 full blocks, and that the current unfilled block is
// appended without selection for a fixed width of 2,051.
//
// Design: one 1024-thread CTA per (request, query) row, persistent over rows.
// Scores map to order-preserving 32-bit keys (-0.0 folded onto +0.0, NaN
// below everything). Three radix passes of 11, 11 and 10 bits narrow the
// threshold key T and the number of blocks equal to T still needed; each pass
// histograms only the keys that match the prefix found so far. The row's keys
// stay in shared memory when they fit, so the scores are read from HBM once.
// A final ordered pass keeps every key above T and the lowest-index keys equal
// to T, and writes block ids and positions in ascending order through
// ballot/popcount ranks, so the result is deterministic and bit-exact.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kKeyCap = 53248;  // keys held in shared memory (208 KB)
constexpr int kHdrWords = 2048 + 64 + 4;

__device__ __forceinline__ uint32_t to_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN ranks last
  if (u == 0x80000000u) u = 0u;                      // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
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

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const float* __restrict__ scores,
                                                           const int32_t* __restrict__ q_pos,
                                                           int32_t* __restrict__ sel_blk,
                                                           int32_t* __restrict__ sel_pos,
                                                           int32_t* err, int rows, int n_q,
                                                           int max_blocks, int key_cap) {
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;                                  // [2048]
  uint32_t* wsum = hist + 2048;                         // [2][32]
  int* res = reinterpret_cast<int*>(wsum + 64);         // [4]
  uint32_t* keys = sm + kHdrWords;                      // [key_cap]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;

  pdl_wait();  // the scores come from the previous kernel
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int p = q_pos[row];
    int32_t* ob = sel_blk + (size_t)row * kTopK;
    int32_t* op = sel_pos + (size_t)row * kWidth;
    if (p < 0 || n_full_of(p) > max_blocks) {
      if (tid == 0) record_error(err, kErrQueryPos, row / n_q, row % n_q, p);
      for (int i = tid; i < kTopK; i += kThreads) ob[i] = -1;
      for (int i = tid; i < kWidth; i += kThreads) op[i] = -1;
      continue;
    }
    const int n = n_full_of(p);
    const int npart = (p + 1) & 3;
    if (n <= kTopK) {  // every full block is kept: positions 0..p
      for (int i = tid; i < kTopK; i += kThreads) ob[i] = i < n ? i : -1;
      for (int i = tid; i < kWidth; i += kThreads) op[i] = i <= p ? i : -1;
      continue;
    }
    const float* srow = scores + (size_t)row * max_blocks;
    const bool in_smem = n <= key_cap;

    // pass 1: top 11 bits of every key (keys cached in shared memory)
    for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t k = to_key(srow[i]);
      if (in_smem) keys[i] = k;
      atomicAdd(&hist[k >> 21], 1u);
    }
    __syncthreads();
    uint32_t need = kTopK;
    find_bin<2048>(hist, need, wsum, res);
    uint32_t prefix = (uint32_t)res[0];
    need -= (uint32_t)res[1];

    // pass 2: next 11 bits of the keys in the threshold bin
    for (int i = tid; i < 2048; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t k = in_smem ? keys[i] : to_key(srow[i]);
      if ((k >> 21) == prefix) atomicAdd(&hist[(k >> 10) & 2047u], 1u);
    }
    __syncthreads();
    find_bin<2048>(hist, need, wsum, res);
    prefix = (prefix << 11) | (uint32_t)res[0];
    need -= (uint32_t)res[1];

    // pass 3: last 10 bits
    for (int i = tid; i < 1024; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t k = in_smem ? keys[i] : to_key(srow[i]);
      if ((k >> 10) == prefix) atomicAdd(&hist[k & 1023u], 1u);
    }
    __syncthreads();
    find_bin<1024>(hist, need, wsum, res);
    const uint32_t T = (prefix << 10) | (uint32_t)res[0];
    need -= (uint32_t)res[1];  // blocks equal to T still to take, >= 1

    // ordered compaction: keys > T, then the first `need` keys == T
    uint32_t n_sel = 0, n_tie = 0;
    int buf = 0;
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + tid;
      const uint32_t k = (i < n) ? (in_smem ? keys[i] : to_key(srow[i])) : 0u;
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
      const bool sel = gt || (eq && my_eq < rem_w);
      const uint32_t slot = n_sel + G_w + taken_before + (uint32_t)__popc(gtm & lt_mask) + min(my_eq, rem_w);
      if (sel && slot < (uint32_t)kTopK) {  // exactly kTopK are selected; the bound is a guard
        ob[slot] = i;
        int32_t* o4 = op + 4 * slot;
        o4[0] = 4 * i;
        o4[1] = 4 * i + 1;
        o4[2] = 4 * i + 2;
        o4[3] = 4 * i + 3;
      }
      n_sel += G_t + min(rem_tile, E_t);
      n_tie += E_t;
      buf ^= 1;
    }
    if (tid < kBlock - 1) op[kBlock * kTopK + tid] = tid < npart ? kBlock * n + tid : -1;
    __syncthreads();  // shared memory is reused by the next row
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_topk(const qsa_dims& d, const float* scores, const int32_t* q_pos,
                        int32_t* sel_blk, int32_t* sel_pos, int32_t* err, cudaStream_t s,
                        bool pdl) {
  const int rows = d.batch * d.n_q;
  const int key_cap = d.max_blocks < kKeyCap ? d.max_blocks : kKeyCap;
  const size_t smem = (size_t)(kHdrWords + key_cap) * sizeof(uint32_t);
  static size_t set_bytes[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || set_bytes[dev] < smem) {
    const size_t want = (size_t)(kHdrWords + kKeyCap) * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)want);
    if (e != cudaSuccess) return e;
    if (dev < 64) set_bytes[dev] = want;
  }
  int grid = rows < device_sm_count() ? rows : device_sm_count();
  if (grid < 1) grid = 1;
  return launch_k(topk_kernel, dim3(grid), dim3(kThreads), smem, s, pdl, scores, q_pos, sel_blk,
                  sel_pos, err, rows, d.n_q, d.max_blocks, key_cap);
}

}  // namespace qsa
