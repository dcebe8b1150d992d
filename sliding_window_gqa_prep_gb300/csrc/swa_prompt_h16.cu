// Prompt-chunk attention of the token path on the 5th-generation tensor cores
// (tcgen05, TMEM) with f16 hi/lo operands: the GEMM path of "o1c_msl.metal"
// (cortiq-engine 0.8.79: o1c_gather, o1c_cols, o1c_gmax, o1c_gsoft, o1c_gadd and
// the engine GEMMs Q K^T and P V they feed) as one persistent kernel.
//
// Precision. Every operand block is scaled by a power of two 2^-e so that its
// largest magnitude lies in [2^14, 2^15), then split x = hi + lo with hi = x
// rounded to f16 and lo = (x - hi) rounded to f16 (x - hi is exact in f32). Each
// product is hi*hi' + hi*lo' + lo*hi' accumulated in f32 (three tcgen05.mma
// kind::f16): 11 + 11 significand bits per operand, the same as a TF32 hi/lo
// split, at twice the TF32 rate and half its bytes. The scales are undone
// exactly: a score tile is multiplied by 2^(e_q + e_k) (e_q per query vector,
// e_k per K block); P is written as p * 2^(e_v - E + 4), where e_v is the V
// block's exponent and E a running V exponent that is raised (with O rescaled)
// only when a block exceeds it by more than 3, so P < 2^15 and O accumulates in
// units of 2^(E - 4). A block of zeros has e_v = -127 (its P underflows to 0).
//
// Work: one unit = 128 query vectors (rows x heads of one KV head) of a row
// block against its tiles of 32 keys (sink blocks, then the logical blocks that
// hold its window). The grid has one CTA per SM; CTA c takes the units of ranks
// c, 2P - 1 - c, 2P + c, ... of the longest-first order (P = grid size), so the
// SMs finish close together, and tensor memory, barriers and the pipelines stay
// up from one unit to the next.
//
// With FLASH the same kernel is swa_flash's full-sequence attention
// ("egemma2_msl.metal", cortiq-engine 0.8.17: eg_flash64 / eg_flash_staged): a
// unit is a row block of one segment of packed q|k|v rows, its tiles are every
// key block of the segment (only the segment's tail is masked), and o = O / l is
// written straight to the output. When the units leave a short last round, the
// shortest of them run as pieces (runs of their tiles) whose records the last
// piece to finish combines.
//
// CTA = 12 warps (13 at hd 64):
//   warps 0-7  two threads per query vector = per TMEM lane (warps w and w + 4 share
//              lanes 32 (w % 4) .. + 31, each taking half of every tile's keys and half
//              of the features): Q of each unit into TMEM, softmax of its score row,
//              P (f16 hi | lo) written over the row's own S columns, rare O rescales,
//              the unit's record;
//   warp 8     K producer: per group of 4 tiles, the K halves (hi, lo) of their
//              split-once blocks as bulk copies into one of two 4-slot halves;
//   warp 9     one lane issues the P V MMAs and their commits;
//   warp 10    V producer: the V^T halves of each tile into one of 4 slots;
//   warp 11    one lane issues the S MMAs and their commits;
//   warp 12    (hd 64) one lane issues the P V MMAs of the odd tiles of each unit into a
//              second O accumulator (warp 9 takes the even ones); the epilogue adds them.
// Tensor memory (512 columns at hd 128): Q_hi | Q_lo (f16 pairs, hd/2 columns
// each) | S buffer 0 | S buffer 1 (128 columns = 4 tiles each) | O (hd; at hd 64 two
// of them). S of a
// group of 4 tiles is one N = 128 product. Both S buffers are in flight: the MMA
// lane issues S of group g + 2 once P V of group g is done, so the tensor cores
// compute scores two groups ahead, and P V of tile j runs while the softmax warps
// work on tile j + 1 (P lives in its tile's S columns: no P buffer to wait for).
// Every hand-off is an mbarrier; all waits are bounded (1 s) and report
// SWA_DERR_TIMEOUT; tensor memory is released on every path.
#include <cuda_fp16.h>

#include "swa_internal.cuh"
#include "swa_tcgen05.cuh"
#include "swa_h16.cuh"

namespace swa {
namespace {

using namespace h16;


template <int HD>
struct HCfg {
  static constexpr int LAND = kHN * HD * 2;                 // one f16 half-tile (hi or lo), bytes
  static constexpr int NSV = 4;                             // V slots
  // shared memory: K_hi [2 halves x 4 slots], K_lo [8], V^T_hi [4], V^T_lo [4]
  static constexpr int OFF_KHI = 0, OFF_KLO = 8 * LAND, OFF_VHI = 16 * LAND, OFF_VLO = 16 * LAND + NSV * LAND;
  static constexpr int OFF_BAR = 16 * LAND + 2 * NSV * LAND;
  static constexpr int NBAR = 48;
  // softmax pair exchange: one (sequence, value) word per softmax thread
  static constexpr int OFF_XCH = OFF_BAR + NBAR * 8 + 16;
  static constexpr size_t USED = (size_t)OFF_XCH + 256 * 8;
  // at least 116 KB, so that one CTA (and one 512-column TMEM allocation) runs per SM
  static constexpr size_t BYTES = USED > 118784 ? USED : 118784;
  static_assert(BYTES <= 232448, "227 KB of shared memory per CTA");
  // TMEM columns
  // O accumulators: at hd 64 two (tiles of even / odd index within the unit, each issued
  // by its own P V lane: an N = 64 product costs the issuing thread as much as one of
  // N = 128, so one lane could not keep up), summed in the epilogue; at hd 128 one
  static constexpr int NO = HD == 64 ? 2 : 1;
  static constexpr int THREADS = (12 + NO - 1) * 32;       // warp 12: the second P V lane
  static constexpr uint32_t C_QHI = 0, C_QLO = HD / 2, C_S0 = HD, C_S1 = HD + kHG * kHN, C_O = HD + 2 * kHG * kHN;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(C_O + NO * HD <= TMEM_COLS, "tensor memory budget");
  // K-major core-matrix layouts (8 rows x 16 bytes): LBO = next core matrix along K, SBO = next 8 rows
  static constexpr uint32_t K_SBO = (HD / 8) * 128;        // K: rows = keys, K = features
  static constexpr uint32_t V_SBO = (kHN / 8) * 128;       // V^T: rows = features, K = keys
};

// barrier block
// (a commit costs the issuing thread about as much as three MMAs, so each event has
// one barrier: "S of group g done" also frees K half g % 2, "P V of tile T done" also
// frees V slot T % 4 and, for a group's last tile, the group's S buffer)
enum : int {
  B_KFULL = 0,     // [2] K half h landed (bytes)
  B_VFULL = 4,     // [4] V slot landed (bytes)
  B_SFULL = 12,    // [2] MMA commit: S of the group in buffer b is done (K half b is free)
  B_PREADY = 16,   // [8] softmax warps (8 arrivals): P of tile T % 8 written (and O rescaled)
  B_PVDONE = 24,   // [8] MMA commit: P V of tile T % 8 done (V slot T % 4 is free)
  B_QREADY = 32,   // softmax warps (4 arrivals): Q of the next unit in TMEM
  B_FIN = 33,      // [3] MMA commits: every MMA issued by the P V lane / the S lane / the second P V lane is done
};

template <int HD, bool FLASH>
__global__ void __launch_bounds__(HCfg<HD>::THREADS, 1) attend_prompt_h16_kernel(AttendParams p) {
  using C = HCfg<HD>;
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(1024) unsigned char sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + C::NBAR);
  volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(reinterpret_cast<int*>(bars + C::NBAR) + 1);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long U = (long long)p.B * p.nk * p.n_rb;
  const unsigned char* ops = reinterpret_cast<const unsigned char*>(p.ops);

  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars[B_KFULL + k], 1);
      mbar_init(&bars[B_SFULL + k], 1);
    }
    for (int k = 0; k < C::NSV; ++k) {
      mbar_init(&bars[B_VFULL + k], 1);
    }
    for (int k = 0; k < 8; ++k) {
      mbar_init(&bars[B_PREADY + k], 8);
      mbar_init(&bars[B_PVDONE + k], 1);
    }
    mbar_init(&bars[B_QREADY], 8);
    mbar_init(&bars[B_FIN], 1);
    mbar_init(&bars[B_FIN + 1], 1);
    mbar_init(&bars[B_FIN + 2], 1);
    mbar_fence_init();
    *s_abort = 0;
  }
  if (tid < 256) reinterpret_cast<unsigned long long*>(sm + C::OFF_XCH)[tid] = 0ull;
  if (warp == 0) tc_alloc(const_cast<uint32_t*>(s_tmem), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  auto abort_now = [&]() {
    *s_abort = 1;
    set_err(p.err, SWA_DERR_TIMEOUT);
  };

  // ------------------------------------------------------------------ K producer
  if (warp == 8 && lane == 0) {
    long long GR = 0;              // groups issued so far (this CTA)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!unit_at<FLASH>(p, U, k, false, u)) break;
      const unsigned char* blocks = ops + (size_t)u.bg * p.ops_nblk * 4 * C::LAND;
      // the unit's Q rows into L2 ahead of the softmax warps (hpg heads of a row are contiguous)
      for (int j = 0; j < u.rows_eff; ++j)
        bulk_prefetch_l2(FLASH ? p.qkv + (size_t)(u.s0 + u.r0 + j) * p.ld + p.q_off + (size_t)u.g * p.hpg * HD
                               : p.q + (((size_t)u.b * p.t + u.r0 + j) * p.nh + (size_t)u.g * p.hpg) * HD,
                         (uint32_t)(p.hpg * HD * 4));
      for (int i0 = 0; i0 < u.ntiles; i0 += kHG, ++GR) {
        const int h = (int)(GR & 1);
        if (GR >= 2 && (!mbar_wait_bounded(&bars[B_SFULL + h], (uint32_t)(((GR - 2) >> 1) & 1), kWaitLimitNs) ||
                        *s_abort)) {
          ok = false;
          break;
        }
        const int cnt = min(kHG, u.ntiles - i0);
        mbar_arrive_expect_tx(&bars[B_KFULL + h], (uint32_t)(cnt * 2 * C::LAND));
        for (int j = 0; j < cnt; ++j) {
          const int i = i0 + j;
          const int blk = i >= p.ops_nsb ? i + u.kb0 : i;
          const unsigned char* src = blocks + (size_t)blk * 4 * C::LAND;
          bulk_g2s(sm + C::OFF_KHI + (size_t)(h * kHG + j) * C::LAND, src, (uint32_t)C::LAND, &bars[B_KFULL + h]);
          bulk_g2s(sm + C::OFF_KLO + (size_t)(h * kHG + j) * C::LAND, src + C::LAND, (uint32_t)C::LAND,
                   &bars[B_KFULL + h]);
        }
      }
    }
    if (!ok) abort_now();
    // copies still in flight land before the CTA exits (bounded; on the normal path
    // the MMA lane has already seen them)
    for (long long g2 = GR - 2 < 0 ? 0 : GR - 2; g2 < GR; ++g2)
      mbar_wait_bounded(&bars[B_KFULL + (g2 & 1)], (uint32_t)((g2 >> 1) & 1), kWaitLimitNs);
  }

  // ------------------------------------------------------------------ V producer
  if (warp == 10 && lane == 0) {
    long long T = 0;               // tiles issued so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!unit_at<FLASH>(p, U, k, false, u)) break;
      const unsigned char* blocks = ops + (size_t)u.bg * p.ops_nblk * 4 * C::LAND;
      for (int i = 0; i < u.ntiles; ++i, ++T) {
        const int slot = (int)(T % C::NSV);
        if (T >= C::NSV &&
            (!mbar_wait_bounded(&bars[B_PVDONE + (int)((T - C::NSV) & 7)], (uint32_t)(((T - C::NSV) >> 3) & 1),
                                kWaitLimitNs) ||
             *s_abort)) {
          ok = false;
          break;
        }
        const int blk = i >= p.ops_nsb ? i + u.kb0 : i;
        const unsigned char* src = blocks + (size_t)blk * 4 * C::LAND + 2 * C::LAND;
        mbar_arrive_expect_tx(&bars[B_VFULL + slot], (uint32_t)(2 * C::LAND));
        bulk_g2s(sm + C::OFF_VHI + (size_t)slot * C::LAND, src, (uint32_t)C::LAND, &bars[B_VFULL + slot]);
        bulk_g2s(sm + C::OFF_VLO + (size_t)slot * C::LAND, src + C::LAND, (uint32_t)C::LAND, &bars[B_VFULL + slot]);
      }
    }
    if (!ok) abort_now();
    for (long long t2 = T - C::NSV < 0 ? 0 : T - C::NSV; t2 < T; ++t2)
      mbar_wait_bounded(&bars[B_VFULL + (int)(t2 % C::NSV)], (uint32_t)((t2 / C::NSV) & 1), kWaitLimitNs);
  }

  // ------------------------------------------------------------------ MMA issuers
  // Two lanes issue the MMAs (an MMA costs its issuing thread about 60 cycles and a
  // commit about 200, and the issuers share their schedulers with softmax warps): warp
  // 11 the S products, warp 9 the P V products. They write different accumulators; S
  // of group g waits for P V of the last tile of group g - 2 (the P it overwrites).
  // Shared-memory descriptors are a base plus (byte offset >> 4): every operand lies in
  // this CTA's window (< 2^18 bytes), so the 14-bit address field never carries.
  if (warp == 11 && lane == 0) {
    const uint32_t id_s = tc_idesc_f16(kHM, kHG * kHN);
    const uint64_t kd0 = smem_desc(sm, 128, C::K_SBO);
    long long T = 0, GR = 0;
    // the latest group in S buffer 0 / 1: its last tile, and the last tile of the other
    // P V lane in it (the same tile with one lane or a one-tile group); each lane's
    // commits are in order, so these two cover every P V that reads the buffer's P
    long long last0 = 0, last1 = 0, prev0 = 0, prev1 = 0;
    bool ok = true;
    for (int k = 0, un = 0; ok; ++k, ++un) {
      Unit u;
      if (!unit_at<FLASH>(p, U, k, false, u)) break;
      // Q of this unit is in tensor memory (the previous unit's S are all done)
      if (!mbar_wait_bounded(&bars[B_QREADY], (uint32_t)(un & 1), kWaitLimitNs) || *s_abort) {
        ok = false;
        break;
      }
      for (int i0 = 0; ok && i0 < u.ntiles; i0 += kHG) {
        const long long gr = GR + i0 / kHG;
        const int h = (int)(gr & 1);
        // S of group gr (K half h into S buffer h): Q_lo K_hi + Q_hi K_lo + Q_hi K_hi
        if (!mbar_wait_bounded(&bars[B_KFULL + h], (uint32_t)((gr >> 1) & 1), kWaitLimitNs) || *s_abort) {
          ok = false;
          break;
        }
        if (gr >= 2) {
          const long long tl = h ? last1 : last0, tp = h ? prev1 : prev0;
          if (!mbar_wait_bounded(&bars[B_PVDONE + (int)(tl & 7)], (uint32_t)((tl >> 3) & 1), kWaitLimitNs) ||
              !mbar_wait_bounded(&bars[B_PVDONE + (int)(tp & 7)], (uint32_t)((tp >> 3) & 1), kWaitLimitNs) ||
              *s_abort) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        const uint32_t d = tmem + (h ? C::C_S1 : C::C_S0);
        const uint64_t kd = kd0 + (uint64_t)((h * kHG * C::LAND) >> 4);
#pragma unroll
        for (int term = 0; term < 3; ++term) {
          const uint32_t qa = tmem + (term == 0 ? C::C_QLO : C::C_QHI);
          const uint32_t kofs = term == 1 ? C::OFF_KLO : C::OFF_KHI;
#pragma unroll
          for (int ks = 0; ks < HD / 16; ++ks)
            tc_mma_f16(d, qa + ks * 8, kd + ((kofs + ks * 256) >> 4), id_s, term > 0 || ks > 0);
        }
        tc_commit(&bars[B_SFULL + h]);
        const long long tlast = T + min(i0 + kHG, u.ntiles) - 1;
        (h ? last1 : last0) = tlast;
        (h ? prev1 : prev0) = C::NO == 2 && min(kHG, u.ntiles - i0) >= 2 ? tlast - 1 : tlast;
      }
      T += u.ntiles;
      GR += (u.ntiles + kHG - 1) / kHG;
    }
    if (!ok) abort_now();
    tc_commit(&bars[B_FIN + 1]);
    mbar_wait_bounded(&bars[B_FIN + 1], 0, kWaitLimitNs);
  }
  // P V lanes: warp 9 (and at hd 64 warp 12) issue the P V products of the unit's tiles
  // i = lane k, k + NO, ... into accumulator O_k
  if ((warp == 9 || (C::NO == 2 && warp == 12)) && lane == 0) {
    const int kl = warp == 9 ? 0 : 1;
    const uint32_t id_o = tc_idesc_f16(kHM, HD);
    const uint64_t vd0 = smem_desc(sm, 128, C::V_SBO);
    const uint32_t od = tmem + C::C_O + (uint32_t)(kl * HD);
    long long T = 0, GR = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!unit_at<FLASH>(p, U, k, false, u)) break;
      for (int i = kl; ok && i < u.ntiles; i += C::NO) {
        const long long t = T + i;
        const int h = (int)((GR + i / kHG) & 1);
        const int vs = (int)(t % C::NSV);
        if (!mbar_wait_bounded(&bars[B_PREADY + (int)(t & 7)], (uint32_t)((t >> 3) & 1), kWaitLimitNs) ||
            *s_abort || !mbar_wait_bounded(&bars[B_VFULL + vs], (uint32_t)((t / C::NSV) & 1), kWaitLimitNs) ||
            *s_abort) {
          ok = false;
          break;
        }
        tc_fence_after();
        // O_k += P_lo V_hi + P_hi V_lo + P_hi V_hi; P of tile i in its S columns: for keys
        // 0-15 and then 16-31, 8 columns of hi pairs and 8 of lo pairs
        const uint32_t pa = tmem + (h ? C::C_S1 : C::C_S0) + (uint32_t)((i % kHG) * kHN);
        const uint64_t vd = vd0 + (uint64_t)((vs * C::LAND) >> 4);
#pragma unroll
        for (int term = 0; term < 3; ++term) {
          const uint32_t vofs = term == 1 ? C::OFF_VLO : C::OFF_VHI;
#pragma unroll
          for (int ks = 0; ks < kHN / 16; ++ks)
            tc_mma_f16(od, pa + ks * 16 + (term == 0 ? 8 : 0), vd + ((vofs + ks * 256) >> 4), id_o,
                       i >= C::NO || term > 0 || ks > 0);
        }
        tc_commit(&bars[B_PVDONE + (int)(t & 7)]);
      }
      T += u.ntiles;
      GR += (u.ntiles + kHG - 1) / kHG;
    }
    if (!ok) abort_now();
    uint64_t* fin = &bars[kl == 0 ? B_FIN : B_FIN + 2];
    tc_commit(fin);
    mbar_wait_bounded(fin, 0, kWaitLimitNs);
  }

  // ------------------------------------------------------------------ softmax warps
  // Warps w and w + 4 share TMEM lanes 32 (w % 4) .. + 31 (one query vector each per
  // lane): warp w takes keys 0-15 of every tile, features 0 .. hd/2 - 1 of Q and O,
  // warp w + 4 the other halves. The pair exchanges row maxima (and at the end l)
  // through shared memory with a 64-thread named barrier; both then take the same
  // decisions (running max, V exponent, rescale) from the same values.
  if (warp < 8) {
    const int quarter = warp & 3, half = warp >> 2;
    const int q = quarter * 32 + lane;                   // query vector = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int rr = q / p.hpg, hq = q % p.hpg;
    constexpr int HH = HD / 2;                           // features per half
    const uint32_t xmine = smem_u32(sm + C::OFF_XCH + tid * 8);
    const uint32_t xpair = smem_u32(sm + C::OFF_XCH + (tid ^ 128) * 8);
    uint32_t xseq = 0;                                   // exchanges so far
    long long T = 0, GR = 0;
    bool dead = false;
    auto fail = [&]() {
      if (lane == 0) abort_now();
      dead = true;
    };
    // v to the thread of the same query vector in the pair's other warp (softmax thread
    // tid ^ 128) and its value back, as one 64-bit shared word (sequence number, value)
    // per thread: a single-copy-atomic store and polled loads, no fence (a fence would
    // wait for this thread's global loads and stores in flight). The partner cannot be
    // more than one exchange ahead: it waits for this thread's previous word first.
    // Polled a bounded number of times; on a timeout the warp is marked dead.
    auto swap_with_pair = [&](float v) -> float {
      ++xseq;
      const unsigned long long word = ((unsigned long long)xseq << 32) | __float_as_uint(v);
      asm volatile("st.relaxed.cta.shared.u64 [%0], %1;" :: "r"(xmine), "l"(word) : "memory");
      uint32_t sq = 0, val = 0;
      for (int n = 0; n < (1 << 24); ++n) {
        unsigned long long got;
        asm volatile("ld.relaxed.cta.shared.u64 %0, [%1];" : "=l"(got) : "r"(xpair) : "memory");
        sq = (uint32_t)(got >> 32);
        val = (uint32_t)got;
        if (sq >= xseq) break;
      }
      if (!__all_sync(kFull, sq >= xseq)) {
        fail();
        return v;
      }
      return __uint_as_float(val);
    };
    const int2* exps = reinterpret_cast<const int2*>(p.ops_exp);
    // this half of Q of unit u into TMEM: q * qmul * 2^-e_q as f16 hi / lo pairs
    // (returns e_q); the S products of the previous unit are all done when this runs
    auto put_q = [&](const Unit& u) -> int {
      const bool q_ok = rr < u.rows_eff && q < p.rows * p.hpg;
      float x[HH];
      const float* src =
          (FLASH ? p.qkv + (size_t)(u.s0 + u.r0 + rr) * p.ld + p.q_off + ((size_t)u.g * p.hpg + hq) * HD
                 : p.q + (((size_t)u.b * p.t + u.r0 + rr) * p.nh + (size_t)u.g * p.hpg + hq) * HD) +
          half * HH;
#pragma unroll
      for (int c = 0; c < HH; c += 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q_ok) v = *reinterpret_cast<const float4*>(src + c);
        x[c] = v.x * p.qmul;
        x[c + 1] = v.y * p.qmul;
        x[c + 2] = v.z * p.qmul;
        x[c + 3] = v.w * p.qmul;
      }
      float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < HH; ++c) am[c & 3] = fmaxf(am[c & 3], fabsf(x[c]));
      float amax = fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3]));
      amax = fmaxf(amax, swap_with_pair(amax));
      const int e = amax > 0.f ? max(-100, min(100, ilogbf(amax) - 14)) : 0;
      const float sq = pow2i(-e);
      if constexpr (HH == 64) {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) split_pair(x[2 * c] * sq, x[2 * c + 1] * sq, hi[c], lo[c]);
        tc_st32(tmem + lane_off + C::C_QHI + half * 32, hi);
        tc_st32(tmem + lane_off + C::C_QLO + half * 32, lo);
      } else {
        static_assert(HH == 32, "hd 64 or 128");
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) split_pair(x[2 * c] * sq, x[2 * c + 1] * sq, hi[c], lo[c]);
        tc_st16(tmem + lane_off + C::C_QHI + half * 16, hi);
        tc_st16(tmem + lane_off + C::C_QLO + half * 16, lo);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_QREADY]);
      return e;
    };
    // block exponents (e_k, e_v) of tiles base .. base + 31 of unit u, lane l holding tile
    // base + l (loaded a window ahead, read per tile by shuffle: no global load is in
    // flight at the per-tile hand-offs)
    auto exp_window = [&](const Unit& u, int base) -> int2 {
      const int i = base + lane;
      if (i >= u.ntiles) return make_int2(0, kZeroExp);
      return __ldg(exps + (size_t)u.bg * p.ops_nblk + (i >= p.ops_nsb ? i + u.kb0 : i));
    };
    // this half of O times s into dst[0 .. HH - 1] (zeros for a unit without tiles);
    // `store` false: tensor memory is read (warp-collective) but nothing is written
    auto store_o = [&](float* dst, bool have_o, float s, bool store, bool n_o1) {
      if (have_o) {
        for (int c0 = 0; c0 < HH; c0 += 32) {
          uint32_t o[32];
          tc_ld32(tmem + lane_off + C::C_O + half * HH + c0, o);
          if constexpr (C::NO == 2) {
            // O = O_0 + O_1 (O_1 holds tiles 1, 3, ...: nothing with a single tile)
            uint32_t o1[32];
            tc_ld32(tmem + lane_off + C::C_O + HD + half * HH + c0, o1);
            tc_wait_ld();
            if (n_o1)
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) + __uint_as_float(o1[e]));
          } else {
            tc_wait_ld();
          }
          if (store) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + c0 + e) =
                  make_float4(__uint_as_float(o[e]) * s, __uint_as_float(o[e + 1]) * s,
                              __uint_as_float(o[e + 2]) * s, __uint_as_float(o[e + 3]) * s);
          }
        }
      } else if (store) {
        for (int c0 = 0; c0 < HH; c0 += 4) *reinterpret_cast<float4*>(dst + c0) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    Unit u{};
    int e_q = 0;
    int2 exw = make_int2(0, kZeroExp);
    bool have = unit_at<FLASH>(p, U, 0, true, u);
    if (have) {
      exw = exp_window(u, 0);
      e_q = put_q(u);
    }
    for (int k = 0; have && !dead; ++k) {
      if (__any_sync(kFull, *s_abort)) { fail(); break; }
      // the next item's unit id now, its meta (its segment) after the first tile: both
      // arrive during this unit
      ItemRef nit{};
      const bool has_next = item_of<FLASH>(p, U, k + 1, nit);
      const int nid = has_next ? p.ws_order[nit.urank] : 0;
      swa_meta nmeta{};
      uint32_t nseg0 = 0, nseg1 = 0;
      auto load_next = [&]() {
        if constexpr (FLASH) {
          const int b = nid / p.n_rb / p.nk;
          nseg0 = p.segs[2 * b];
          nseg1 = p.segs[2 * b + 1];
        } else {
          nmeta = p.meta[nid / p.n_rb / p.nk];
        }
      };
      const bool q_ok = rr < u.rows_eff && q < p.rows * p.hpg;
      const int r = u.r0 + rr;
      // this row's keys x: q_lo <= x <= q_hi (its window; for FLASH its whole segment)
      int q_lo = 0, q_hi = u.len - 1;
      if constexpr (!FLASH) {
        q_lo = u.st.len0 + r + 1 - min(u.st.W, u.st.len0 + r + 1);
        q_hi = u.st.len0 + r;
        if (u.g == 0 && tid == 0) {
          p.ws_nsplit[u.b * p.n_rb + u.rb] = 1;
          if (u.rb == 0) p.ws_meta[u.b] = p.meta[u.b];
        }
      }
      float m_run = -INFINITY, l_run = 0.f;              // l_run: this half's keys
      int E = kZeroExp;
      const int nsb = p.ops_nsb;
      int2 exn = make_int2(0, kZeroExp);
      // one group of (up to) 4 tiles per step: one S wait, one row maximum over the
      // group (one pair exchange), one running-max / V-exponent decision and at most one
      // O rescale; then P of each tile and its hand-off to the MMA lane
      for (int i0 = 0; i0 < u.ntiles; i0 += kHG) {
        const long long gr = GR + i0 / kHG;
        const int h = (int)(gr & 1);
        const int cnt = min(kHG, u.ntiles - i0);
        if ((i0 & 31) == 16) exn = exp_window(u, i0 + 16);
        if ((i0 & 31) == 0 && i0 > 0) exw = exn;
        if (!__all_sync(kFull, mbar_wait_bounded(&bars[B_SFULL + h], (uint32_t)((gr >> 1) & 1), kWaitLimitNs))) {
          fail();
          break;
        }
        if (__any_sync(kFull, *s_abort)) { fail(); break; }
        tc_fence_after();
        // this half's 16 columns of each tile's S, later its P (a missing tile's are unused)
        const uint32_t gcol = (h ? C::C_S1 : C::C_S0) + (uint32_t)(half * 16);
        uint32_t sr[kHG][16];
#pragma unroll
        for (int j = 0; j < kHG; ++j) tc_ld16(tmem + lane_off + gcol + j * kHN, sr[j]);
        tc_wait_ld();
        int ev[kHG];
        float f[kHG];
        float gmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < kHG; ++j) {
          const int i = i0 + j;
          const int ek = __shfl_sync(kFull, exw.x, i & 31);
          ev[j] = __shfl_sync(kFull, exw.y, i & 31);
          // f undoes the Q and K block scales (> 0: the sum is clamped at the smallest subnormal)
          f[j] = pow2w(max(e_q + ek, -149));
          // window mask; a tile wholly inside this row's window skips it. A sink tile
          // holds sinks j0 .. j0 + 31 (valid below ns), a logical tile keys x0 .. x0 + 31.
          const bool sink_tile = i < nsb;
          const int j0 = i * kHN + half * 16;
          const int x0 = (u.kb0 + i - nsb) * kHN + half * 16;
          const bool inside =
              j < cnt && (sink_tile ? q_ok && p.ns - j0 >= 16 : q_ok && x0 >= q_lo && x0 + 15 <= q_hi);
          if (!__all_sync(kFull, inside)) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const bool v = j < cnt && q_ok && (sink_tile ? j0 + c < p.ns : (x0 + c >= q_lo && x0 + c <= q_hi));
              if (!v) sr[j][c] = __float_as_uint(-INFINITY);
            }
          }
          float mx[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            mx[c] = fmaxf(fmaxf(__uint_as_float(sr[j][c]), __uint_as_float(sr[j][c + 4])),
                          fmaxf(__uint_as_float(sr[j][c + 8]), __uint_as_float(sr[j][c + 12])));
          gmax = fmaxf(gmax, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * f[j]);
        }
        gmax = fmaxf(gmax, swap_with_pair(gmax));
        if (dead) break;
        // The running max m_run moves only when the group exceeds it by more than
        // kHLazyMax (log2 units): below that p = 2^(s - m_run) <= 2^kHLazyMax, and
        // O and l keep one common scale, so o = O / l is unchanged.
        const bool raise = gmax > m_run + kHLazyMax;
        const float m_new = raise ? gmax : m_run;
        const float c1 = raise ? ex2(m_run - m_new) : 1.f;
        // the V exponent after this group's tiles (every e_v <= E_new + kVSlack)
        int E_new = E;
#pragma unroll
        for (int j = 0; j < kHG; ++j)
          if (j < cnt && (i0 + j == 0 || ev[j] > E_new + kVSlack)) E_new = ev[j];
        const float c2 = i0 == 0 ? 1.f : pow2w(max(E - E_new, -252));
        // O rescale (warp-uniform; the pair decides alike): O holds P V of the tiles
        // before this group, all done first; none of this group's P is handed off yet
        const float c = c1 * c2;
        if (i0 > 0 && __any_sync(kFull, c != 1.f && m_run != -INFINITY)) {
          // the last tile of each P V lane (i0 >= 4: both lanes have one)
          const long long tp = T + i0 - 1, tq = T + i0 - C::NO;
          if (!__all_sync(kFull, mbar_wait_bounded(&bars[B_PVDONE + (int)(tp & 7)], (uint32_t)((tp >> 3) & 1),
                                                   kWaitLimitNs) &&
                                     mbar_wait_bounded(&bars[B_PVDONE + (int)(tq & 7)], (uint32_t)((tq >> 3) & 1),
                                                       kWaitLimitNs))) {
            fail();
            break;
          }
          tc_fence_after();
          for (int ko = 0; ko < C::NO; ++ko) {
#pragma unroll 1
            for (int c0 = ko * HD + half * HH; c0 < ko * HD + half * HH + HH; c0 += 16) {
              uint32_t o[16];
              tc_ld16(tmem + lane_off + C::C_O + c0, o);
              tc_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * c);
              tc_st16(tmem + lane_off + C::C_O + c0, o);
            }
          }
        }
        const float mref = m_new == -INFINITY ? 0.f : m_new;   // no valid key yet: every s is -inf, p = 0
        float lsum = 0.f;
#pragma unroll
        for (int j = 0; j < kHG; ++j) {
          if (j < cnt) {
            const long long t = T + i0 + j;
            // P = p * 2^kp with kp = e_v - E + kVHead, as one exp2 of s f - (m - kp). kp
            // is clamped at -100 (the row sum then keeps every p above 2^-26); a tile
            // with e_v that far below E holds V values 2^-89 times the largest, whose
            // products this scales by at most 2^27.
            const int kp = max(ev[j] - E_new + kVHead, -100);
            const float moff = mref - (float)kp;
            uint32_t w[16];                                      // 8 hi pairs | 8 lo pairs
            // two scores per packed f32x2 instruction: the scale FMA, the row sum and the
            // lo remainder p - hi (an exact fma by -1)
            const u64 f2 = pack2(f[j], f[j]), m2 = pack2(-moff, -moff);
            u64 ps2[2] = {0ull, 0ull};
#pragma unroll
            for (int c = 0; c < 16; c += 2) {
              const float2 x = unpack2(fma2(pack2(__uint_as_float(sr[j][c]), __uint_as_float(sr[j][c + 1])), f2, m2));
              const u64 pp = pack2(ex2(x.x), ex2(x.y));
              ps2[(c >> 1) & 1] = fma2(pp, pack2(1.f, 1.f), ps2[(c >> 1) & 1]);
              split_pair2(pp, w[c / 2], w[8 + c / 2]);
            }
            const float2 sa = unpack2(ps2[0]), sb = unpack2(ps2[1]);
            lsum += ((sa.x + sa.y) + (sb.x + sb.y)) * pow2i(-kp);
            tc_st16(tmem + lane_off + gcol + j * kHN, w);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_PREADY + (int)(t & 7)]);
          }
        }
        l_run = l_run * c1 + lsum;
        m_run = m_new;
        E = E_new;
        if (i0 == 0 && has_next) load_next();
      }
      if (dead) break;
      if (u.ntiles == 0 && has_next) load_next();
      // ---- the next unit's Q: its first S products run while this unit's output is written
      Unit nu{};
      int e_qn = 0;
      int2 exw_n = make_int2(0, kZeroExp);
      if (has_next) {
        if constexpr (FLASH)
          nu = flash_unit_from(p, nid, flash_segment_check(p, nid, nseg0, nseg1, true), nit);
        else
          nu = unit_from(p, nid, nmeta, true);
        exw_n = exp_window(nu, 0);
        e_qn = put_q(nu);
      }
      if (dead) break;
      const float l_other = swap_with_pair(l_run);
      if (dead) break;
      if (u.ntiles > 0) {
        // the last tile of each P V lane that has one
        const long long tl = T + u.ntiles - 1, tm = T + max(u.ntiles - C::NO, 0);
        if (!__all_sync(kFull, mbar_wait_bounded(&bars[B_PVDONE + (int)(tl & 7)], (uint32_t)((tl >> 3) & 1),
                                                 kWaitLimitNs) &&
                                   mbar_wait_bounded(&bars[B_PVDONE + (int)(tm & 7)], (uint32_t)((tm >> 3) & 1),
                                                     kWaitLimitNs))) {
          fail();
          break;
        }
        tc_fence_after();
      }
      const float os = pow2w(E - kVHead);                 // O is in units of 2^(E - kVHead)
      if constexpr (!FLASH) {
        // ---- the unit's record: O * 2^(E - kVHead) (unnormalised), m, l (both halves' keys)
        const size_t item = (size_t)u.bg * p.n_rb + u.rb;
        store_o(p.ws_acc + (item * (size_t)p.nq + q) * HD + half * HH, u.ntiles > 0, os, true, u.ntiles > 1);
        if (half == 0) p.ws_ml[item * p.nq + q] = make_float2(m_run, l_run + l_other);
      } else {
        float* dst = p.out + (size_t)(u.s0 + r) * p.ldo + ((size_t)u.g * p.hpg + hq) * HD + half * HH;
        if (u.npiece == 1) {
          // ---- o = O / l straight to the output row (a row block past its segment's end
          // has no tiles and no rows)
          if (u.ntiles > 0) store_o(dst, true, os / (l_run + l_other), q_ok, u.ntiles > 1);
        } else {
          // ---- a piece: its record (O, then (m, l) per half) and, by the last piece of
          // the unit to get here (per softmax warp: its 32 query vectors and half of the
          // features), the combination of all of them. No wait on another CTA.
          const size_t rstride = (size_t)kHM * (HD + 4);
          float* rec = p.ws_rec + (size_t)u.tail_at * rstride;
          store_o(rec + (size_t)q * HD + half * HH, u.ntiles > 0, os, true, u.ntiles > 1);
          reinterpret_cast<float2*>(rec + (size_t)kHM * HD)[half * kHM + q] =
              u.ntiles > 0 ? make_float2(m_run, l_run + l_other) : make_float2(-INFINITY, 0.f);
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0)
            last = atomicAdd(p.ws_cnt + (size_t)(u.tail_at / u.npiece) * 8 + warp, 1) == u.npiece - 1;
          if (__shfl_sync(kFull, last, 0)) {
            __threadfence();
            const float* rec0 = p.ws_rec + (size_t)(u.tail_at - u.piece) * rstride;
            auto ml_of = [&](int j) {
              return __ldcg(reinterpret_cast<const float2*>(rec0 + j * rstride + (size_t)kHM * HD) + half * kHM + q);
            };
            float M = -INFINITY;
            for (int j = 0; j < u.npiece; ++j) M = fmaxf(M, ml_of(j).x);
            float den = 0.f;
            for (int j = 0; j < u.npiece; ++j) {
              const float2 ml = ml_of(j);
              if (ml.x != -INFINITY) den += ml.y * exp2f(ml.x - M);   // a piece without keys weighs 0
            }
            if (q_ok) {
              const float inv = 1.0f / den;
              for (int c = 0; c < HH; c += 4) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int j = 0; j < u.npiece; ++j) {
                  const float2 ml = ml_of(j);
                  if (ml.x == -INFINITY) continue;
                  const float w = exp2f(ml.x - M);
                  const float4 v =
                      __ldcg(reinterpret_cast<const float4*>(rec0 + j * rstride + (size_t)q * HD + half * HH + c));
                  acc.x += v.x * w;
                  acc.y += v.y * w;
                  acc.z += v.z * w;
                  acc.w += v.w * w;
                }
                *reinterpret_cast<float4*>(dst + c) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
              }
            }
          }
        }
      }
      T += u.ntiles;
      GR += (u.ntiles + kHG - 1) / kHG;
      u = nu;
      e_q = e_qn;
      exw = exw_n;
      have = has_next;
    }
  }

  // ------------------------------------------------------------------ teardown
  // every role has waited for what it issued (copies, MMAs) before it got here
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tc_dealloc(tmem, C::TMEM_COLS);
  }
}

// One split-once operand block of 32 keys by a CTA of 256 threads: K_hi | K_lo (keys x
// features, K-major core matrices: (key / 8) * K_SBO + (f / 8) * 128 + (key % 8) * 16 +
// (f % 8) * 2 bytes) | V^T_hi | V^T_lo ((f / 8) * V_SBO + (key / 8) * 128 + (f % 8) * 16
// + (key % 8) * 2), each f16 of 2^-e times the block's rows, into block blk of (sequence
// or segment, KV head) bg; ops_exp gets (e_k, e_v). fetch(key, kr, vr) points kr / vr at
// the key's K and V rows, or leaves them null for a missing key (zeros).
template <int HD, class Fetch>
__device__ __forceinline__ void split_block_h16(const AttendParams& p, int bg, int blk, Fetch fetch) {
  using C = HCfg<HD>;
  __shared__ __align__(16) float ks[kHN][HD + 4];
  __shared__ __align__(16) float vs[kHN][HD + 4];
  __shared__ float red[2][8];
  constexpr int D4 = HD / 4;
  float ak = 0.f, av = 0.f;
  for (int idx = threadIdx.x; idx < kHN * D4; idx += blockDim.x) {
    const int key = idx / D4, f4 = idx % D4;
    const float* kr = nullptr;
    const float* vr = nullptr;
    fetch(key, kr, vr);
    float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
    if (kr) {
      kv = *reinterpret_cast<const float4*>(kr + f4 * 4);
      vv = *reinterpret_cast<const float4*>(vr + f4 * 4);
    }
    *reinterpret_cast<float4*>(&ks[key][f4 * 4]) = kv;
    *reinterpret_cast<float4*>(&vs[key][f4 * 4]) = vv;
    ak = fmaxf(ak, fmaxf(fmaxf(fabsf(kv.x), fabsf(kv.y)), fmaxf(fabsf(kv.z), fabsf(kv.w))));
    av = fmaxf(av, fmaxf(fmaxf(fabsf(vv.x), fabsf(vv.y)), fmaxf(fabsf(vv.z), fabsf(vv.w))));
  }
  for (int d = 16; d > 0; d >>= 1) {
    ak = fmaxf(ak, __shfl_xor_sync(kFull, ak, d));
    av = fmaxf(av, __shfl_xor_sync(kFull, av, d));
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = ak;
    red[1][threadIdx.x >> 5] = av;
  }
  __syncthreads();
  ak = 0.f;
  av = 0.f;
  for (int w = 0; w < 8; ++w) {
    ak = fmaxf(ak, red[0][w]);
    av = fmaxf(av, red[1][w]);
  }
  const int e_k = block_exp(ak), e_v = block_exp(av);
  const float sk = pow2i(-(e_k == kZeroExp ? 0 : e_k)), sv = pow2i(-(e_v == kZeroExp ? 0 : e_v));
  unsigned char* dst = reinterpret_cast<unsigned char*>(p.ops) + ((size_t)bg * p.ops_nblk + blk) * 4 * C::LAND;
  if (threadIdx.x == 0) reinterpret_cast<int2*>(p.ops_exp)[(size_t)bg * p.ops_nblk + blk] = make_int2(e_k, e_v);
  // K: thread -> (key, 8 features): one 16-byte store each of hi and lo
  for (int idx = threadIdx.x; idx < kHN * (HD / 8); idx += blockDim.x) {
    const int key = idx % kHN, f8 = idx / kHN;
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      split_pair(ks[key][f8 * 8 + 2 * e] * sk, ks[key][f8 * 8 + 2 * e + 1] * sk, hw[e], lw[e]);
    const size_t off = (size_t)(key >> 3) * C::K_SBO + f8 * 128 + (key & 7) * 16;
    *reinterpret_cast<uint4*>(dst + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(dst + C::LAND + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  // V^T: thread -> (feature, 8 keys)
  for (int idx = threadIdx.x; idx < HD * (kHN / 8); idx += blockDim.x) {
    const int f = idx % HD, k8 = idx / HD;
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      split_pair(vs[k8 * 8 + 2 * e][f] * sv, vs[k8 * 8 + 2 * e + 1][f] * sv, hw[e], lw[e]);
    const size_t off = (size_t)(f >> 3) * C::V_SBO + k8 * 128 + (f & 7) * 16;
    *reinterpret_cast<uint4*>(dst + 2 * C::LAND + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(dst + 3 * C::LAND + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

// Token path: one CTA per (sequence, KV head, block). Blocks 0 .. nsb - 1 hold the
// sinks, block nsb + k the logical keys x = 32k .. 32k + 31 below len0 + t (ring slot
// (head0 + x) % W for x < len0, chunk row x - len0 after), read before the commit
// rewrites the ring; missing keys are zeros. The extra row blockIdx.y = B * nk orders
// the row blocks.
template <int HD>
__global__ void __launch_bounds__(256) token_presplit_h16_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  if (blockIdx.y == (unsigned)(p.B * p.nk)) {
    if (blockIdx.x == 0) order_row_blocks_h16(p);
    return;
  }
  const int blk = blockIdx.x, bg = blockIdx.y;
  const int b = bg / p.nk, g = bg % p.nk;
  const SeqState st = sanitize_state(p.meta[b], p.cap, nullptr);   // the attention reports bad metas
  const size_t kv_head = (size_t)b * p.nk + g;
  const bool sink = blk < p.ops_nsb;
  const int j0 = blk * kHN;                                        // first sink of a sink block
  const int x0 = (blk - p.ops_nsb) * kHN;                          // first logical key otherwise
  if (!sink && x0 >= st.len0 + p.t) return;                        // past every row's window
  split_block_h16<HD>(p, bg, blk, [&](int key, const float*& kr, const float*& vr) {
    if (sink) {
      if (j0 + key < p.ns) {
        const size_t at = (kv_head * p.ns + j0 + key) * HD;
        kr = p.sink_k + at;
        vr = p.sink_v + at;
      }
    } else {
      const int x = x0 + key;
      if (x < st.len0) {
        int slot = st.head0 + x;
        if (slot >= st.W) slot -= st.W;
        const size_t at = (kv_head * p.cap + (size_t)slot) * HD;
        kr = p.ring_k + at;
        vr = p.ring_v + at;
      } else if (x < st.len0 + p.t) {
        const size_t at = (((size_t)b * p.t + (x - st.len0)) * p.nk + g) * HD;
        kr = p.k_chunk + at;
        vr = p.v_chunk + at;
      }
    }
  });
}

// swa_flash: one CTA per (segment, KV head, block): block k holds the segment's rows
// 32k .. 32k + 31 (zeros past its end). The extra row blockIdx.y = nseg * nk orders the
// units and clears the combine counters of the launch tail.
template <int HD>
__global__ void __launch_bounds__(256) flash_presplit_h16_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  if (blockIdx.y == (unsigned)(p.B * p.nk)) {
    if (blockIdx.x == 0) {
      for (int i = threadIdx.x; i < 8 * p.flash_tail; i += blockDim.x) p.ws_cnt[i] = 0;
      order_flash_units_h16(p);
    }
    return;
  }
  const int blk = blockIdx.x, bg = blockIdx.y;
  const int g = bg % p.nk;
  const int2 seg = flash_segment(p, bg * p.n_rb, false);           // the attention reports bad segments
  const int j0 = blk * kHN;
  if (j0 >= seg.y) return;
  const int cnt = min(kHN, seg.y - j0);
  split_block_h16<HD>(p, bg, blk, [&](int key, const float*& kr, const float*& vr) {
    if (key < cnt) {
      const float* row = p.qkv + (size_t)(seg.x + j0 + key) * p.ld + (size_t)g * HD;
      kr = row + p.k_off;
      vr = row + p.v_off;
    }
  });
}

template <int HD, bool FLASH>
int launch_h16(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = HCfg<HD>;
  auto kern = attend_prompt_h16_kernel<HD, FLASH>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const dim3 pgrid((unsigned)p.ops_nblk, (unsigned)(p.B * p.nk + 1));
  int rc = finish_launch(FLASH ? launch_pdl(flash_presplit_h16_kernel<HD>, pgrid, dim3(256), 0, s, p)
                               : launch_pdl(token_presplit_h16_kernel<HD>, pgrid, dim3(256), 0, s, p));
  if (rc != SWA_OK) return rc;
  // items: whole units, then the launch tail's pieces; one persistent CTA per SM
  const long long items = (long long)p.B * p.nk * p.n_rb - p.flash_tail + (long long)p.flash_tail * p.flash_q;
  const int sms = num_sms();
  const unsigned grid = (unsigned)(items < sms ? items : (sms > 0 ? sms : 148));
  if (e0) cudaEventRecord(e0, s);
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::BYTES, s, p);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e1) cudaEventRecord(e1, s);
  return cuda_status(e);
}

}  // namespace

int launch_attend_prompt_h16(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  switch (p.hd) {
    case 64: return launch_h16<64, false>(p, s, e0, e1);
    case 128: return launch_h16<128, false>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

int launch_flash_h16(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  switch (p.hd) {
    case 64: return launch_h16<64, true>(p, s, e0, e1);
    case 128: return launch_h16<128, true>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

}  // namespace swa
