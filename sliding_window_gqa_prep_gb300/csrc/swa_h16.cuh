// Device helpers of the f16 hi/lo tensor-core attention kernel on split-once operand
// blocks: power-of-two block scales, f16 hi/lo pairs, the row-block units a persistent
// CTA walks and their longest-first order.
#pragma once
#include <cuda_fp16.h>

#include "swa_internal.cuh"

namespace swa {
namespace h16 {

constexpr int kHM = 128;               // query vectors per unit (MMA M)
constexpr int kHN = 32;                // keys per tile
constexpr int kHG = 4;                 // tiles per S product (N = 128)
constexpr float kHLazyMax = 8.0f;      // log2 headroom before the running max is raised
constexpr int kVHead = 4;              // P = p * 2^(e_v - E + kVHead)
constexpr int kVSlack = 3;             // E is raised when e_v > E + kVSlack (P < 2^15)
constexpr int kZeroExp = -127;         // exponent of a block of zeros
constexpr unsigned kFull = 0xffffffffu;

// Tiles of row block rb: the sink blocks, then logical blocks kb0 .. (len0 + r_last) / 32,
// where kb0 holds the first key of the block's first row's window
__device__ __forceinline__ int row_block_tiles(const AttendParams& p, const SeqState& st, int rb) {
  const int r0 = rb * p.rows, r_last = min(r0 + p.rows, p.t) - 1;
  const int xlo = st.len0 + r0 + 1 - min(st.W, st.len0 + r0 + 1);
  return p.ops_nsb + (st.len0 + r_last) / kHN - xlo / kHN + 1;
}

// exact 2^k for k in [-126, 127]; 0 below (the block exponents are clamped to +-100)
__device__ __forceinline__ float pow2i(int k) {
  return k < -126 ? 0.f : __int_as_float((127 + min(k, 127)) << 23);
}

// exact 2^k for k in [-252, 254] (a product of two normal powers; tiny results round to
// subnormals or 0)
__device__ __forceinline__ float pow2w(int k) {
  const int a = k >> 1;
  return pow2i(a) * pow2i(k - a);
}

// 2^x by the MUFU instruction (relative error about 2^-22; -inf -> +0, results below
// 2^-126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exponent e with max |x| * 2^-e in [2^14, 2^15) (clamped to +-100); kZeroExp if max |x| = 0
__device__ __forceinline__ int block_exp(float amax) {
  return amax > 0.f ? max(-100, min(100, ilogbf(amax) - 14)) : kZeroExp;
}

// bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) from global memory into L2
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// x = hi + lo as f16 pairs: hi = RN(x), lo = RN(x - hi); element 2c in the low half
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - f.x, x1 - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// A unit: (sequence b, KV head g, row block rb) at rank `rank` of the order
struct Unit {
  int b, g, bg, rb, r0, rows_eff, xlo, kb0, ntiles;
  SeqState st;
};

// rank of this CTA's k-th unit (boustrophedon over the longest-first order)
__device__ __forceinline__ long long unit_rank(int k) {
  const long long P = gridDim.x;
  return (long long)k * P + ((k & 1) ? (P - 1 - blockIdx.x) : blockIdx.x);
}

// the unit of row-block id `id` (index (b * nk + g) * n_rb + rb) with its sequence's meta
__device__ __forceinline__ Unit unit_from(const AttendParams& p, int id, const swa_meta m, bool report) {
  Unit u;
  u.rb = id % p.n_rb;
  u.bg = id / p.n_rb;
  u.b = u.bg / p.nk;
  u.g = u.bg % p.nk;
  bool bad = false;
  u.st = sanitize_state(m, p.cap, &bad);
  if (bad && report && u.g == 0 && u.rb == 0) set_err(p.err, SWA_DERR_META);
  u.r0 = u.rb * p.rows;
  const int r_last = min(u.r0 + p.rows, p.t) - 1;
  u.rows_eff = r_last - u.r0 + 1;
  u.xlo = u.st.len0 + u.r0 + 1 - min(u.st.W, u.st.len0 + u.r0 + 1);
  u.kb0 = u.xlo / kHN;
  u.ntiles = row_block_tiles(p, u.st, u.rb);
  return u;
}

__device__ __forceinline__ Unit load_unit(const AttendParams& p, long long rank, bool report) {
  const int id = p.ws_order[rank];
  return unit_from(p, id, p.meta[id / p.n_rb / p.nk], report);
}

// The token path's row blocks ordered by their tile count, longest first, by one CTA
// of 256 threads (a counting sort; equal counts in any order). Every order gives the
// same results.
__device__ void order_row_blocks_h16(const AttendParams& p) {
  constexpr int kBins = 2048;
  __shared__ int cnt[kBins];
  const int U = p.B * p.nk * p.n_rb;
  const int nb = min(kBins, p.ops_nblk + 1);   // a row block has at most ops_nblk tiles
  auto key = [&](int u) {                       // bin nb - 1 - tiles: longest first
    const SeqState st = sanitize_state(p.meta[u / p.n_rb / p.nk], p.cap, nullptr);
    const int tiles = min(max(row_block_tiles(p, st, u % p.n_rb), 0), nb - 1);
    return nb - 1 - tiles;
  };
  for (int i = threadIdx.x; i < nb; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  for (int u = threadIdx.x; u < U; u += blockDim.x) atomicAdd(&cnt[key(u)], 1);
  __syncthreads();
  // exclusive prefix over the bins by warp 0: lane l sums bins l * per .. l * per + per - 1
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x, per = (nb + 31) / 32;
    const int lo = min(lane * per, nb), hi = min(lo + per, nb);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += cnt[i];
    int incl = sum;
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - sum;
    for (int i = lo; i < hi; ++i) {
      const int c = cnt[i];
      cnt[i] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int u = threadIdx.x; u < U; u += blockDim.x) p.ws_order[atomicAdd(&cnt[key(u)], 1)] = u;
}

}  // namespace h16
}  // namespace swa
