// Device helpers of the f16 hi/lo tensor-core attention kernel on split-once operand
// blocks: power-of-two block scales, f16 hi/lo pairs, the row-block units a persistent
// CTA walks (token-path row blocks, or row blocks of full-sequence segments and pieces
// of them) and their longest-first order.
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

// x = hi + lo as f16 pairs: hi = RN(x), lo = RN(x - hi); element 2c in the low half
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - f.x, x1 - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// packed pairs of f32 (element 0 in the low half) and their f32x2 arithmetic
using u64 = unsigned long long;
__device__ __forceinline__ u64 pack2(float lo, float hi) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(u64 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// split_pair of a packed pair, the remainder x - hi as one packed fma by -1 (exact, as
// the subtraction)
__device__ __forceinline__ void split_pair2(u64 x, uint32_t& hi, uint32_t& lo) {
  const float2 v = unpack2(x);
  const __half2 h = __floats2half2_rn(v.x, v.y);
  const float2 f = __half22float2(h);
  const float2 d = unpack2(fma2(pack2(f.x, f.y), pack2(-1.f, -1.f), x));
  const __half2 l = __floats2half2_rn(d.x, d.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// A unit: (sequence or segment b, KV head g, row block rb), or one piece of it. Its
// tiles are operand blocks i >= ops_nsb ? kb0 + i : i (i < ntiles) of (b, g).
struct Unit {
  int b, g, bg, rb, r0, rows_eff, xlo, kb0, ntiles;
  SeqState st;                   // token path: the sequence's ring state
  int s0, len;                   // full-sequence segments: first row and length
  int piece, npiece, tail_at;    // piece `piece` of npiece; tail_at: its number in the launch tail
};

// rank of this CTA's k-th item (boustrophedon over the longest-first order)
__device__ __forceinline__ long long unit_rank(int k) {
  const long long P = gridDim.x;
  return (long long)k * P + ((k & 1) ? (P - 1 - blockIdx.x) : blockIdx.x);
}

// An item: a whole unit (the unit of rank urank in the order) or a piece of one. The
// units of ranks U - flash_tail .. U - 1 (the shortest) run as flash_q pieces each,
// piece j taking the j-th of flash_q equal runs of the unit's tiles, so that the last
// round of the persistent CTAs is spread over the whole grid.
struct ItemRef {
  long long urank;
  int piece, npiece, tail_at;
};

// this CTA's k-th item; false past the last one (the token path has no pieces)
template <bool FLASH>
__device__ __forceinline__ bool item_of(const AttendParams& p, long long U, int k, ItemRef& it) {
  const long long r = unit_rank(k);
  const long long full = FLASH ? U - p.flash_tail : U;
  if (r < full) {
    it = ItemRef{r, 0, 1, 0};
    return true;
  }
  const long long pc = r - full;
  if (!FLASH || pc >= (long long)p.flash_tail * p.flash_q) return false;
  it = ItemRef{full + pc / p.flash_q, (int)(pc % p.flash_q), p.flash_q, (int)pc};
  return true;
}

// segment (first row s0, length len) of unit id as (s0, length), the length 0 for a
// segment past row T or longer than max_len (reported once, by the segment's first
// unit, when `report`)
__device__ __forceinline__ int2 flash_segment_check(const AttendParams& p, int id, uint32_t s0, uint32_t len,
                                                    bool report) {
  if ((uint64_t)s0 + len > (uint64_t)p.T || len > (uint32_t)p.max_len) {
    if (report && id % (p.n_rb * p.nk) == 0) set_err(p.err, SWA_DERR_SEGMENT);
    return make_int2(0, 0);
  }
  return make_int2((int)s0, (int)len);
}
__device__ __forceinline__ int2 flash_segment(const AttendParams& p, int id, bool report) {
  const int b = id / p.n_rb / p.nk;
  return flash_segment_check(p, id, p.segs[2 * b], p.segs[2 * b + 1], report);
}

// tiles of a full-sequence unit: every key block of its segment, 0 for a row block
// past the segment's end
__device__ __forceinline__ int flash_unit_tiles(const AttendParams& p, int rb, int len) {
  return rb * p.rows < len ? (len + kHN - 1) / kHN : 0;
}

// the full-sequence unit of id `id` ((segment * nk + g) * n_rb + rb), piece it.piece
__device__ __forceinline__ Unit flash_unit_from(const AttendParams& p, int id, int2 seg, const ItemRef& it) {
  Unit u{};
  u.rb = id % p.n_rb;
  u.bg = id / p.n_rb;
  u.b = u.bg / p.nk;
  u.g = u.bg % p.nk;
  u.s0 = seg.x;
  u.len = seg.y;
  u.r0 = u.rb * p.rows;
  u.rows_eff = max(0, min(u.r0 + p.rows, u.len) - u.r0);
  const int n = flash_unit_tiles(p, u.rb, u.len);
  u.piece = it.piece;
  u.npiece = it.npiece;
  u.tail_at = it.tail_at;
  u.kb0 = (int)((long long)n * it.piece / it.npiece);
  u.ntiles = (int)((long long)n * (it.piece + 1) / it.npiece) - u.kb0;
  return u;
}

// the unit of row-block id `id` (index (b * nk + g) * n_rb + rb) with its sequence's meta
__device__ __forceinline__ Unit unit_from(const AttendParams& p, int id, const swa_meta m, bool report) {
  Unit u{};
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
  u.npiece = 1;
  return u;
}

// this CTA's k-th item as a unit (token-path row block, or full-sequence unit or piece);
// false past the last item
template <bool FLASH>
__device__ __forceinline__ bool unit_at(const AttendParams& p, long long U, int k, bool report, Unit& u) {
  ItemRef it;
  if (!item_of<FLASH>(p, U, k, it)) return false;
  const int id = p.ws_order[it.urank];
  if constexpr (FLASH)
    u = flash_unit_from(p, id, flash_segment(p, id, report), it);
  else
    u = unit_from(p, id, p.meta[id / p.n_rb / p.nk], report);
  return true;
}

// Units 0 .. U - 1 ordered by tile count, longest first, equal counts by index (a
// stable counting sort by one CTA of 256 threads), into order[0 .. U - 1]; tiles(u) is
// clamped to [0, nb - 1]. The order is the same on every call.
template <class Tiles>
__device__ void order_units_h16(int U, int nb, int* order, Tiles tiles) {
  constexpr int kBins = 2048;
  __shared__ int cnt[kBins];
  nb = max(1, min(kBins, nb));
  auto key = [&](int u) {                       // bin nb - 1 - tiles: longest first
    return nb - 1 - min(max(tiles(u), 0), nb - 1);
  };
  for (int i = threadIdx.x; i < nb; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  for (int u = threadIdx.x; u < U; u += blockDim.x) atomicAdd(&cnt[key(u)], 1);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // exclusive prefix over the bins by warp 0: lane l sums bins l * per .. l * per + per - 1
  if (warp == 0) {
    const int per = (nb + 31) / 32;
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
  // stable scatter: blockDim.x units at a time in index order, one warp after another;
  // within a warp the lanes of one bin take consecutive places in lane order
  for (int c0 = 0; c0 < U; c0 += blockDim.x) {
    const int u = c0 + threadIdx.x;
    const int k = u < U ? key(u) : -1;
    const unsigned peers = __match_any_sync(kFull, k);
    const int before = __popc(peers & ((1u << lane) - 1u));
    for (int w = 0; w < nw; ++w) {
      if (warp == w) {
        const int pos = u < U ? cnt[k] + before : 0;
        __syncwarp();
        if (u < U && before == 0) cnt[k] += __popc(peers);
        if (u < U) order[pos] = u;
      }
      __syncthreads();
    }
  }
}

// The token path's row blocks, longest first
__device__ inline void order_row_blocks_h16(const AttendParams& p) {
  order_units_h16(p.B * p.nk * p.n_rb, p.ops_nblk + 1, p.ws_order, [&](int u) {
    const SeqState st = sanitize_state(p.meta[u / p.n_rb / p.nk], p.cap, nullptr);
    return row_block_tiles(p, st, u % p.n_rb);
  });
}

// The full-sequence units, longest first (units of longer segments first)
__device__ inline void order_flash_units_h16(const AttendParams& p) {
  order_units_h16(p.B * p.nk * p.n_rb, p.ops_nblk + 1, p.ws_order, [&](int u) {
    return flash_unit_tiles(p, u % p.n_rb, flash_segment(p, u, false).y);
  });
}

}  // namespace h16
}  // namespace swa
