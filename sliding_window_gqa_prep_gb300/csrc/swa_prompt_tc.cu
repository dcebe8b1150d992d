// Prompt-chunk attention on the 5th-generation tensor cores (tcgen05, TMEM) with
// TF32 hi/lo operands that the kernel stages and splits itself: the GEMM path of
// "o1c_msl.metal" (cortiq-engine 0.8.79: o1c_gather, o1c_cols, o1c_gmax, o1c_gsoft,
// o1c_gadd and the engine GEMMs Q K^T and P V they feed) as one flash-style kernel
// per block of 128 query vectors. The token path takes it for prompt chunks given
// the minimum workspace (with room for split-once operand blocks the persistent f16
// kernel of swa_prompt_h16.cu runs instead); swa_flash takes it always (below).
//
// Precision: every operand is split a = a_hi + a_lo with a_hi = a rounded to
// TF32 and a_lo = (a - a_hi) rounded to TF32; each product is
// a_hi b_hi + a_hi b_lo + a_lo b_hi accumulated in f32 (three tcgen05.mma
// kind::tf32), which keeps f32 accuracy (the dropped a_lo b_lo is ~2^-22 of
// the product).
//
// CTA = 10 warps:
//   warps 0-3  one thread per query vector = per TMEM lane (the 128-row MMA
//              accumulator rows): softmax of the thread's own score row (read
//              from TMEM), P into TMEM, rescale of O, final record;
//   warp 4     producer: keys with contiguous sources (ring runs, sinks) as one
//              cp.async.bulk per run into fp32 landing tiles of 32 keys;
//   warp 5     one elected lane issues every tcgen05.mma and tcgen05.commit;
//   warps 6-9  split of the landed K/V tiles into TF32 hi/lo shared-memory
//              operands, in parallel with the softmax warps.
// Tensor memory (512 columns): Q_hi, Q_lo (A operands of S = Q K^T), S,
// O (the P V accumulator), P_hi, P_lo (A operands of P V).
// Shared memory: two fp32 landing stages, K_hi/K_lo (32 keys x hd, K-major
// canonical core-matrix layout: 8 rows x 16 bytes per core matrix) and
// V^T_hi/V^T_lo (hd x 32 keys, K-major): TF32 operands must be K-major, so V
// is transposed while it is split.
// Pipelining: the hi/lo operand sets and the S accumulator are double
// buffered, so the MMA lane issues S of tile i+1 before P V of tile i and the
// tensor cores compute the next scores while the softmax warps work on the
// current ones; the K half of split j waits for S of tile j-2 (the last reader
// of its buffer), the V half for P V of tile j-2.
//
// The same kernel with MODE 1 or 2 is swa_flash's full-sequence attention
// ("egemma2_msl.metal", cortiq-engine 0.8.17: eg_flash64 / eg_flash_staged):
// the keys of a row block are the rows of its segment of a packed q|k|v buffer,
// only the segment's tail is masked, and o = O / l is written directly. In
// MODE 2 flash_presplit_kernel has already split each KV head's K/V rows into
// the four operand blocks of every 32-key tile (the split warps' output layout),
// once per call: the producer lands them straight in the operand set (four
// contiguous copies per tile) and the split warps sit idle.
// Every hand-off is an mbarrier; all waits are bounded (1 s) and report
// SWA_DERR_TIMEOUT; tensor memory is released on every path.
#include "swa_internal.cuh"
#include "swa_tcgen05.cuh"

namespace swa {
namespace {

constexpr int kTM = 128;               // query vectors per CTA (MMA M)
constexpr int kTN = 32;                // keys per tile
constexpr int kTThreads = 10 * 32;
constexpr int kSoftThreads = 128;
constexpr unsigned kTF = 0xffffffffu;
constexpr float kLazyMax = 8.0f;       // log2 headroom before the running max is raised

template <int HD, int MODE = 0>
struct TCfg {
  // operand sets behind the split warps (MODE 0 / 1)
  static constexpr int NSETS = 2;
  // split-once blocks (MODE 2): separate pools of K (hi, lo) and V^T (hi, lo)
  // slots, consecutive K slots adjacent so that one S product spans G tiles
  static constexpr int NSK = HD == 64 ? 8 : 4, NSV = HD == 64 ? 4 : 2;
  // MODE 2: S of G consecutive tiles is one product of N = 32 G keys (the MMA
  // time of S follows its instruction count, not N). At hd 128 the 128 S columns
  // leave no room for P in tensor memory: P (hi, lo) sits in shared memory and is
  // the A operand of P V.
  static constexpr bool PRE = MODE >= 2;
  static constexpr int G = PRE ? (HD == 64 ? 8 : 4) : 1;
  static constexpr bool P_SMEM = PRE && HD == 128;
  // TMEM columns: Q_hi | Q_lo | S (MODE 0 / 1: buffers S0, S1 of 32; MODE 2: 32 G) | O | P_hi | P_lo
  static constexpr uint32_t SCOLS = PRE ? G * kTN : 2 * kTN;
  static constexpr uint32_t C_QHI = 0, C_QLO = HD, C_S0 = 2 * HD, C_S1 = 2 * HD + kTN;
  static constexpr uint32_t C_O = 2 * HD + SCOLS, C_PHI = 3 * HD + SCOLS, C_PLO = 3 * HD + SCOLS + kTN;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert((P_SMEM ? C_O + HD : C_PLO + kTN) <= TMEM_COLS, "tensor memory budget");
  // shared memory (bytes)
  static constexpr int LAND = kTN * HD * 4;                 // one fp32 tile of K or V
  static constexpr int OFF_LK = 0;                          // [2 stages] K landing
  static constexpr int OFF_LV = 2 * LAND;                   // [2 stages] V landing
  static constexpr int OFF_OPS = 4 * LAND;                  // [NSETS] K_hi, K_lo, V^T_hi, V^T_lo
  static constexpr int SET = 4 * LAND;
  // MODE 2 pools: K_hi [NSK], K_lo [NSK], V^T_hi [NSV], V^T_lo [NSV]
  static constexpr int OFF_KHI = 0, OFF_KLO = NSK * LAND, OFF_VHI = 2 * NSK * LAND;
  static constexpr int OFF_VLO = (2 * NSK + NSV) * LAND;
  // P_SMEM: P_hi, P_lo after the pools, K-major (rows = query vectors, K = keys)
  static constexpr int OFF_PHI = 2 * (NSK + NSV) * LAND, OFF_PLO = OFF_PHI + kTM * kTN * 4;
  static constexpr int OFF_BAR = MODE < 2 ? OFF_OPS + NSETS * SET
                                          : 2 * (NSK + NSV) * LAND + (P_SMEM ? 2 * kTM * kTN * 4 : 0);   // mbarriers
  static constexpr int NBAR = 32;
  // at least 116 KB, so that one CTA (and one 512-column TMEM allocation) runs per SM
  static constexpr size_t USED = (size_t)OFF_BAR + NBAR * 8 + 16;
  static constexpr size_t BYTES = USED > 118784 ? USED : 118784;
  static_assert(BYTES <= 232448, "227 KB of shared memory per CTA");
  // K-major core-matrix layouts: LBO = next core matrix along K, SBO = next 8 rows
  static constexpr uint32_t K_LBO = 128, K_SBO = (HD / 4) * 128;   // K_hi: rows = keys, K = features
  static constexpr uint32_t V_LBO = 128, V_SBO = (kTN / 4) * 128;  // V^T: rows = features, K = keys
  static constexpr uint32_t P_LBO = 128, P_SBO = (kTN / 4) * 128;  // P: rows = query vectors, K = keys
  static_assert(!P_SMEM || (OFF_PLO + (int)(kTM / 8 * P_SBO) <= OFF_BAR && OFF_PHI % 16 == 0 && P_LBO == 128),
                "P_hi, P_lo: 16-byte aligned, below the barriers");
};

__device__ __forceinline__ uint32_t tf32_hi(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// MODE 0: a row block of the token path (sinks, ring window, chunk rows; split
// record to the workspace). MODE 1 / 2: a row block of one segment of packed
// q|k|v rows attending all of the segment's rows (swa_flash); blockIdx.z =
// segment * nk + KV head, and the normalised output is written directly. MODE 2
// takes split-once operand blocks of the segment's rows from p.ops.

template <int HD, int MODE>
__global__ void __launch_bounds__(kTThreads, 1) attend_prompt_tc_kernel(AttendParams p) {
  constexpr bool FLASH = MODE == 1 || MODE == 2;
  constexpr bool PRESPLIT = MODE >= 2;
  constexpr int NS = TCfg<HD, MODE>::NSETS;    // MODE 0 / 1 operand sets: tile j uses set j % NS
  constexpr int NSK = TCfg<HD, MODE>::NSK, NSV = TCfg<HD, MODE>::NSV;
  constexpr int G = TCfg<HD, MODE>::G;
  constexpr bool P_SMEM = TCfg<HD, MODE>::P_SMEM;
  static_assert(NSK % G == 0, "S of a tile group spans G adjacent K slots");
  static_assert(NSK <= 8 && NSV <= 4, "the barrier block holds 8 K and 4 V slots (kfull/kfree, vfull/vfree)");
  pdl_trigger();
  pdl_wait();
  using C = TCfg<HD, MODE>;
  extern __shared__ __align__(1024) unsigned char sm[];
  float* landK = reinterpret_cast<float*>(sm + C::OFF_LK);
  float* landV = reinterpret_cast<float*>(sm + C::OFF_LV);
  // operand set k (k = tile % 2): K_hi, K_lo, V^T_hi, V^T_lo
  auto op = [&](int set, int which) {
    return reinterpret_cast<uint32_t*>(sm + C::OFF_OPS + set * C::SET + which * C::LAND);
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  // MODE 0 / 1
  uint64_t* land_full = bars + 0;    // [2] producer -> split warps (bytes)
  uint64_t* land_empty = bars + 2;   // [2] split warps -> producer (4 arrivals)
  uint64_t* split_done = bars + 4;   // [2 sets] split warps -> MMA (4 arrivals)
  uint64_t* v_free = bars + 12;      // [2 sets] MMA commit (P V of the set done) -> split warps
  // MODE 2
  uint64_t* kfull = bars + 0;        // [NSK] K copies landed (bytes)
  uint64_t* kfree = bars + 8;        // [NSK] MMA commit: S that read the slot is done
  uint64_t* vfull = bars + 16;       // [NSV] V copies landed (bytes)
  uint64_t* vfree = bars + 20;       // [NSV] MMA commit: P V that read the slot is done
  uint64_t* s_empty = bars + 25;     // softmax warps: every tile of the group's S read (4 arrivals)
  // both: S (MODE 0 / 1: [2 buffers]; MODE 2: one buffer of a tile group)
  uint64_t* s_full = PRESPLIT ? bars + 24 : bars + 8;
  uint64_t* p_ready = PRESPLIT ? bars + 26 : bars + 10;   // softmax warps -> MMA (4 arrivals)
  uint64_t* pv_done = PRESPLIT ? bars + 27 : bars + 11;   // MMA commit -> softmax warps
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + C::NBAR);
  volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(reinterpret_cast<int*>(bars + C::NBAR) + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int rb = blockIdx.y, bg = blockIdx.z;
  // MODE 2 launch tail (swa_flash): the last flash_tail units of the 1-D grid run as
  // flash_q pieces each, piece j taking the j-th of flash_q equal runs of the
  // unit's tiles; tail_at numbers the pieces of the tail in launch order
  int piece = 0, npiece = 1, tail_at = 0;
  if constexpr (MODE == 2) {
    if (p.flash_q > 1) {
      const long long full = (long long)p.n_rb * p.B * p.nk - p.flash_tail;
      long long u = blockIdx.x;
      if (u >= full) {
        const long long pc = u - full;
        u = full + pc / p.flash_q;
        piece = (int)(pc % p.flash_q);
        npiece = p.flash_q;
        tail_at = (int)pc;
      }
      rb = (int)(u % p.n_rb);
      bg = (int)(u / p.n_rb);
    }
  }
  const int b = bg / p.nk, g = bg % p.nk;
  const int r0 = rb * p.rows;
  SeqState st{0, 0, 0};
  int s0 = 0, r_last, xlo = 0, n;
  if constexpr (FLASH) {
    // segment b: rows s0 .. s0 + len - 1 of the packed buffer; keys = its rows
    s0 = (int)p.segs[2 * b];
    const uint32_t len = p.segs[2 * b + 1];
    if ((uint64_t)(uint32_t)s0 + len > (uint64_t)p.T || len > (uint32_t)p.max_len) {
      if (tid == 0 && g == 0 && rb == 0) set_err(p.err, SWA_DERR_SEGMENT);
      return;
    }
    if (r0 >= (int)len) return;
    r_last = min(r0 + p.rows, (int)len) - 1;
    n = (int)len;
  } else {
    st = load_state(p, b, tid == 0 && g == 0 && rb == 0);
    r_last = min(r0 + p.rows, p.t) - 1;
    const int win0 = min(st.W, st.len0 + r0 + 1);
    xlo = st.len0 + r0 + 1 - win0;
    n = p.ns + (st.len0 + r_last - xlo + 1);
    if (g == 0 && tid == 0) p.ws_nsplit[b * p.n_rb + rb] = 1;
    if (g == 0 && rb == 0 && tid == 0) p.ws_meta[b] = p.meta[b];
  }
  const int rows_eff = r_last - r0 + 1;
  // a piece takes tiles tile0 .. tile0 + ntiles - 1 of the unit's ceil(n / 32) (may be none)
  const int nt_all = (n + kTN - 1) / kTN;
  const int tile0 = npiece > 1 ? (int)((long long)piece * nt_all / npiece) : 0;
  const int ntiles = npiece > 1 ? (int)((long long)(piece + 1) * nt_all / npiece) - tile0 : nt_all;
  const size_t kv_head = (size_t)b * p.nk + g;

  if (tid == 0) {
    if constexpr (PRESPLIT) {
      for (int k = 0; k < NSK; ++k) {
        mbar_init(&kfull[k], 1);
        mbar_init(&kfree[k], 1);
      }
      for (int k = 0; k < NSV; ++k) {
        mbar_init(&vfull[k], 1);
        mbar_init(&vfree[k], 1);
      }
      mbar_init(s_full, 1);
      mbar_init(s_empty, 4);
    } else {
      mbar_init(&land_full[0], 1);
      mbar_init(&land_full[1], 1);
      mbar_init(&land_empty[0], 4);
      mbar_init(&land_empty[1], 4);
      for (int k = 0; k < NS; ++k) {
        mbar_init(&split_done[k], 4);
        mbar_init(&v_free[k], 1);
      }
      mbar_init(&s_full[0], 1);
      mbar_init(&s_full[1], 1);
    }
    mbar_init(p_ready, 4);
    mbar_init(pv_done, 1);
    mbar_fence_init();
    *s_abort = 0;
  }
  if (warp == 0) tc_alloc(const_cast<uint32_t*>(s_tmem), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // Q rows of the block -> TMEM (hi and lo parts), times scale * log2 e; done by
  // the softmax warps before any role starts, so the first S finds Q in place.
  if (warp < 4) {
    const int q = tid;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int rr = q / p.hpg, h = q % p.hpg;
    const bool q_ok = rr < rows_eff && q < p.rows * p.hpg;
    const int r = r0 + rr;
    {
      const float* src = FLASH ? p.qkv + (size_t)(s0 + r) * p.ld + p.q_off + ((size_t)g * p.hpg + h) * HD
                               : p.q + (((size_t)b * p.t + r) * p.nh + (size_t)g * p.hpg + h) * HD;
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (q_ok) v = *reinterpret_cast<const float4*>(src + c0 + c);
          const float x[4] = {v.x * p.qmul, v.y * p.qmul, v.z * p.qmul, v.w * p.qmul};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[c + e] = tf32_hi(x[e]);
            lo[c + e] = tf32_hi(x[e] - __uint_as_float(hi[c + e]));
          }
        }
        tc_st32(tmem + lane_off + C::C_QHI + c0, hi);
        tc_st32(tmem + lane_off + C::C_QLO + c0, lo);
      }
      tc_wait_st();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ------------------------------------------------------------------ producer
  if (PRESPLIT && (warp == 4 || warp == 6)) {
    // MODE 2 producers: warp 4 lands the K half (hi, lo) of tile i's block in K
    // slot i % NSK once the S that last read the slot is done; warp 6 (a split warp,
    // idle here) lands the V^T half in V slot i % NSV once its P V is done.
    const bool kside = warp == 4;
    const int nslot = kside ? NSK : NSV;
    uint64_t* fullb = kside ? kfull : vfull;
    uint64_t* freeb = kside ? kfree : vfree;
    unsigned char* hi_pool = sm + (kside ? C::OFF_KHI : C::OFF_VHI);
    unsigned char* lo_pool = sm + (kside ? C::OFF_KLO : C::OFF_VLO);
    const float* blocks = p.ops + (size_t)bg * p.ops_nblk * 4 * (kTN * HD) + (kside ? 0 : 2 * kTN * HD);
    int issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int slot = i % nslot;
      bool ok = i < nslot || mbar_wait_bounded(&freeb[slot], (uint32_t)(((i - nslot) / nslot) & 1), kWaitLimitNs);
      ok = __all_sync(kTF, ok);
      if (!ok) {
        if (lane == 0) { *s_abort = 1; set_err(p.err, SWA_DERR_TIMEOUT); }
        break;
      }
      if (__shfl_sync(kTF, *s_abort, 0)) break;
      if (lane == 0) {
        const int blk = i + tile0;
        const float* src = blocks + (size_t)blk * 4 * (kTN * HD);
        mbar_arrive_expect_tx(&fullb[slot], (uint32_t)(2 * C::LAND));
        bulk_g2s(hi_pool + (size_t)slot * C::LAND, src, (uint32_t)C::LAND, &fullb[slot]);
        bulk_g2s(lo_pool + (size_t)slot * C::LAND, src + kTN * HD, (uint32_t)C::LAND, &fullb[slot]);
      }
      __syncwarp();
      issued = i + 1;
    }
    // copies still in flight after an abort land before the CTA exits (bounded; on
    // the normal path the MMA lane has already seen them)
    if (lane == 0)
      for (int i = max(0, issued - nslot); i < issued; ++i)
        mbar_wait_bounded(&fullb[i % nslot], (uint32_t)((i / nslot) & 1), kWaitLimitNs);
  }
  if (!PRESPLIT && warp == 4) {
    for (int i = 0; i < ntiles; ++i) {
      const int stage = i & 1;
      const int use = i >> 1;
      bool ok = use == 0 || mbar_wait_bounded(&land_empty[stage], (uint32_t)((use - 1) & 1), kWaitLimitNs);
      ok = __all_sync(kTF, ok);
      if (!ok) {
        if (lane == 0) { *s_abort = 1; set_err(p.err, SWA_DERR_TIMEOUT); }
        break;
      }
      if (__shfl_sync(kTF, *s_abort, 0)) break;
      fence_proxy_async_smem();
      const int j0 = i * kTN;
      const int cnt = min(kTN, n - j0);
      if (lane == 0) mbar_arrive_expect_tx(&land_full[stage], (uint32_t)(cnt * HD * 4 * 2));
      __syncwarp();
      const float* sk = nullptr;
      const float* sv = nullptr;
      if (lane < cnt) {
        const int j = j0 + lane;
        if constexpr (FLASH) {
          const size_t at = (size_t)(s0 + j) * p.ld + (size_t)g * HD;
          sk = p.qkv + at + p.k_off;
          sv = p.qkv + at + p.v_off;
        } else if (j < p.ns) {
          const size_t at = (kv_head * p.ns + j) * HD;
          sk = p.sink_k + at;
          sv = p.sink_v + at;
        } else {
          const int x = xlo + (j - p.ns);
          if (x < st.len0) {
            int slot = st.head0 + x;
            if (slot >= st.W) slot -= st.W;
            const size_t at = (kv_head * p.cap + (size_t)slot) * HD;
            sk = p.ring_k + at;
            sv = p.ring_v + at;
          } else {
            const size_t at = (((size_t)b * p.t + (x - st.len0)) * p.nk + g) * HD;
            sk = p.k_chunk + at;
            sv = p.v_chunk + at;
          }
        }
      }
      const unsigned long long pk = __shfl_up_sync(kTF, reinterpret_cast<unsigned long long>(sk), 1);
      const unsigned long long pv = __shfl_up_sync(kTF, reinterpret_cast<unsigned long long>(sv), 1);
      const bool start = lane < cnt && (lane == 0 || reinterpret_cast<unsigned long long>(sk) != pk + HD * 4 ||
                                        reinterpret_cast<unsigned long long>(sv) != pv + HD * 4);
      const unsigned starts = __ballot_sync(kTF, start);
      if (start) {
        const unsigned later = starts & ~((2u << lane) - 1u);
        const int end = later ? __ffs(later) - 1 : cnt;
        const uint32_t bytes = (uint32_t)((end - lane) * HD * 4);
        bulk_g2s(landK + ((size_t)stage * kTN + lane) * HD, sk, bytes, &land_full[stage]);
        bulk_g2s(landV + ((size_t)stage * kTN + lane) * HD, sv, bytes, &land_full[stage]);
      }
    }
  }

  // ------------------------------------------------------------------ MMA issuer
  if (PRESPLIT && warp == 5 && lane == 0) {
    // MODE 2: S of a group of G tiles (their K slots are adjacent) as one product
    // of N = 32 G keys; S of group g + 1 is issued right after P V of group g's
    // second-to-last tile, so it runs while the softmax warps work on the last one.
    const uint32_t id_s = tc_idesc(kTM, G * kTN);
    const uint32_t id_o = tc_idesc(kTM, HD);
    const int ngroups = (ntiles + G - 1) / G;
    auto issue_s = [&](int gr) -> bool {
      const int t0 = G * gr;
      // missing tiles of the last group leave their columns undefined; nothing reads them
      for (int k = 0; k < G; ++k) {
        const int t = t0 + k;
        if (t < ntiles && (!mbar_wait_bounded(&kfull[t % NSK], (uint32_t)((t / NSK) & 1), kWaitLimitNs) || *s_abort))
          return false;
      }
      // the softmax warps have read every tile of the previous group
      if (gr >= 1 && (!mbar_wait_bounded(s_empty, (uint32_t)((gr - 1) & 1), kWaitLimitNs) || *s_abort))
        return false;
      tc_fence_after();
      const int slot = t0 % NSK;
      const uint32_t dcol = C::C_S0;
#pragma unroll 1
      for (int term = 0; term < 3; ++term) {
        const uint32_t qcol = term == 0 ? C::C_QLO : C::C_QHI;
        const uint32_t* kb =
            reinterpret_cast<const uint32_t*>(sm + (term == 1 ? C::OFF_KLO : C::OFF_KHI) + (size_t)slot * C::LAND);
        for (int ks = 0; ks < HD / 8; ++ks) {
          const uint64_t bd = smem_desc(kb + ks * 64, C::K_LBO, C::K_SBO);   // 4 G groups of 8 keys
          tc_mma(tmem + dcol, tmem + qcol + ks * 8, bd, id_s, term > 0 || ks > 0);
        }
      }
      tc_commit(s_full);
      for (int k = 0; k < G; ++k)
        if (t0 + k < ntiles) tc_commit(&kfree[(t0 + k) % NSK]);
      return true;
    };
    auto issue_pv = [&](int i) -> bool {
      if (!mbar_wait_bounded(p_ready, (uint32_t)(i & 1), kWaitLimitNs) || *s_abort) return false;
      if (!mbar_wait_bounded(&vfull[i % NSV], (uint32_t)((i / NSV) & 1), kWaitLimitNs) || *s_abort) return false;
      tc_fence_after();
      const int slot = i % NSV;
#pragma unroll 1
      for (int term = 0; term < 3; ++term) {
        const uint32_t* vb =
            reinterpret_cast<const uint32_t*>(sm + (term == 1 ? C::OFF_VLO : C::OFF_VHI) + (size_t)slot * C::LAND);
        if constexpr (P_SMEM) {
          const uint32_t* pb = reinterpret_cast<const uint32_t*>(sm + (term == 0 ? C::OFF_PLO : C::OFF_PHI));
          for (int ks = 0; ks < kTN / 8; ++ks) {
            const uint64_t ad = smem_desc(pb + ks * 64, C::P_LBO, C::P_SBO);
            const uint64_t bd = smem_desc(vb + ks * 64, C::V_LBO, C::V_SBO);
            tc_mma_ss(tmem + C::C_O, ad, bd, id_o, i > 0 || term > 0 || ks > 0);
          }
        } else {
          const uint32_t pcol = term == 0 ? C::C_PLO : C::C_PHI;
          for (int ks = 0; ks < kTN / 8; ++ks) {
            const uint64_t bd = smem_desc(vb + ks * 64, C::V_LBO, C::V_SBO);
            tc_mma(tmem + C::C_O, tmem + pcol + ks * 8, bd, id_o, i > 0 || term > 0 || ks > 0);
          }
        }
      }
      tc_commit(pv_done);
      tc_commit(&vfree[slot]);
      return true;
    };
    bool ok = ntiles == 0 || issue_s(0);
    for (int i = 0; ok && i < ntiles; ++i) {
      ok = issue_pv(i);
      if (ok && i % G == G - 2 && i / G + 1 < ngroups) ok = issue_s(i / G + 1);
    }
    if (!ok) {
      *s_abort = 1;
      set_err(p.err, SWA_DERR_TIMEOUT);
    }
  }
  if (!PRESPLIT && warp == 5 && lane == 0) {
    const uint32_t id_s = tc_idesc(kTM, kTN);
    const uint32_t id_o = tc_idesc(kTM, HD);
    // S(j) = Q_lo K_hi + Q_hi K_lo + Q_hi K_hi of tile j into S buffer j % 2
    auto issue_s = [&](int j) -> bool {
      const int set = j % NS, sb = j & 1;          // operand set, S buffer
      if (!mbar_wait_bounded(&split_done[set], (uint32_t)((j / NS) & 1), kWaitLimitNs) || *s_abort)
        return false;
      tc_fence_after();
      const uint32_t dcol = sb ? C::C_S1 : C::C_S0;
#pragma unroll 1
      for (int term = 0; term < 3; ++term) {
        const uint32_t qcol = term == 0 ? C::C_QLO : C::C_QHI;
        const uint32_t* kb = op(set, term == 1 ? 1 : 0);
        for (int ks = 0; ks < HD / 8; ++ks) {
          const uint64_t bd = smem_desc(kb + ks * 64, C::K_LBO, C::K_SBO);   // 2 core matrices along K
          tc_mma(tmem + dcol, tmem + qcol + ks * 8, bd, id_s, term > 0 || ks > 0);
        }
      }
      tc_commit(&s_full[sb]);
      return true;
    };
    bool ok = ntiles == 0 || issue_s(0);
    for (int i = 0; ok && i < ntiles; ++i) {
      if (i + 1 < ntiles && !issue_s(i + 1)) { ok = false; break; }
      if (!mbar_wait_bounded(p_ready, (uint32_t)(i & 1), kWaitLimitNs) || *s_abort) { ok = false; break; }
      tc_fence_after();
      // O += P_lo V_hi + P_hi V_lo + P_hi V_hi over 32 / 8 steps of K = 8
      const int set = i % NS;
#pragma unroll 1
      for (int term = 0; term < 3; ++term) {
        const uint32_t pcol = term == 0 ? C::C_PLO : C::C_PHI;
        const uint32_t* vb = op(set, term == 1 ? 3 : 2);
        for (int ks = 0; ks < kTN / 8; ++ks) {
          const uint64_t bd = smem_desc(vb + ks * 64, C::V_LBO, C::V_SBO);
          tc_mma(tmem + C::C_O, tmem + pcol + ks * 8, bd, id_o, i > 0 || term > 0 || ks > 0);
        }
      }
      tc_commit(pv_done);
      tc_commit(&v_free[set]);
    }
    if (!ok) {
      *s_abort = 1;
      set_err(p.err, SWA_DERR_TIMEOUT);
    }
  }

  // ------------------------------------------------------------------ split warps
  if (!PRESPLIT && warp >= 6) {
    const int sidx = tid - 6 * 32;                     // 0 .. 127
    // fp32 landing tile j -> TF32 hi/lo operands of set j % 2.
    // K: element (key, f) -> (key/8)*K_SBO + (f/4)*128 + (key%8)*16 + (f%4)*4 bytes. Lane t of an
    // 8-lane phase takes key 8kg + t and feature chunk (fb + t) mod hd/4, so the 8 reads hit 8
    // different chunks of 8 rows and the 8 writes 8 consecutive 16-byte slots: no bank conflicts.
    auto split_k = [&](int j) {
      const float* lk = landK + (size_t)(j & 1) * kTN * HD;
      uint32_t* kh = op(j & 1, 0);
      uint32_t* kl = op(j & 1, 1);
      const int cnt = min(kTN, n - j * kTN);
      constexpr int D4 = HD / 4;
      for (int idx = sidx; idx < kTN * D4; idx += kSoftThreads) {
        const int t8 = idx & 7, rest = idx >> 3;
        const int kg = rest % (kTN / 8), fb = rest / (kTN / 8);
        const int key = kg * 8 + t8, f4 = (fb + t8) % D4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (key < cnt) v = *reinterpret_cast<const float4*>(lk + key * HD + f4 * 4);
        const float x[4] = {v.x, v.y, v.z, v.w};
        uint4 hv, lv4;
        uint32_t* hp = &hv.x;
        uint32_t* lp = &lv4.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hp[e] = tf32_hi(x[e]);
          lp[e] = tf32_hi(x[e] - __uint_as_float(hp[e]));
        }
        const int off = ((key >> 3) * (int)C::K_SBO + f4 * 128 + (key & 7) * 16) / 4;
        *reinterpret_cast<uint4*>(kh + off) = hv;
        *reinterpret_cast<uint4*>(kl + off) = lv4;
      }
    };
    // V^T: element (f, key) -> (f/8)*V_SBO + (key/4)*128 + (f%8)*16 + (key%4)*4 bytes
    auto split_v = [&](int j) {
      const float* lv = landV + (size_t)(j & 1) * kTN * HD;
      uint32_t* vh = op(j & 1, 2);
      uint32_t* vl = op(j & 1, 3);
      const int cnt = min(kTN, n - j * kTN);
      for (int idx = sidx; idx < HD * kTN / 4; idx += kSoftThreads) {
        const int f = idx % HD, k4 = idx / HD;
        uint4 hv, lv4;
        uint32_t* hp = &hv.x;
        uint32_t* lp = &lv4.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = k4 * 4 + e;
          const float x = key < cnt ? lv[key * HD + f] : 0.f;
          hp[e] = tf32_hi(x);
          lp[e] = tf32_hi(x - __uint_as_float(hp[e]));
        }
        const int off = ((f >> 3) * (int)C::V_SBO + k4 * 128 + (f & 7) * 16) / 4;
        *reinterpret_cast<uint4*>(vh + off) = hv;
        *reinterpret_cast<uint4*>(vl + off) = lv4;
      }
    };
    // tile j: K half (once S of tile j - 2 has read the set), then V half (once P V of
    // tile j - 2 has). For j >= 3 the S wait is already met by the v_free wait of tile
    // j - 3 (that commit follows S of tile j - 2); for j == 2 it is the only guard. S of
    // tile j cannot commit before this iteration arrives on split_done, so the parity
    // names S of tile j - 2 and no later phase.
    for (int j = 0; j < ntiles; ++j) {
      bool ok = mbar_wait_bounded(&land_full[j & 1], (uint32_t)((j >> 1) & 1), kWaitLimitNs);
      if (ok && j >= 2) ok = mbar_wait_bounded(&s_full[j & 1], (uint32_t)(((j - 2) >> 1) & 1), kWaitLimitNs);
      ok = __all_sync(kTF, ok) && !*s_abort;
      if (ok) split_k(j);
      if (ok && j >= 2)
        ok = __all_sync(kTF, mbar_wait_bounded(&v_free[j & 1], (uint32_t)(((j - 2) >> 1) & 1), kWaitLimitNs));
      if (!ok) {
        if (lane == 0) { *s_abort = 1; set_err(p.err, SWA_DERR_TIMEOUT); }
        break;
      }
      split_v(j);
      fence_proxy_async_smem();               // generic writes -> tensor-core reads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&land_empty[j & 1]);
        mbar_arrive(&split_done[j & 1]);
      }
    }
  }

  // ------------------------------------------------------------------ softmax warps
  if (warp < 4) {
    const int q = tid;                                   // query vector = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int rr = q / p.hpg;
    const bool q_ok = rr < rows_eff && q < p.rows * p.hpg;
    const int r = r0 + rr;
    const int q_lo = st.len0 + r + 1 - min(st.W, st.len0 + r + 1);
    const int q_hi = st.len0 + r;
    float m_run = -INFINITY, l_run = 0.f;
    bool dead = false;
    auto fail = [&]() {
      if (lane == 0) { *s_abort = 1; set_err(p.err, SWA_DERR_TIMEOUT); }
      dead = true;
    };
    for (int i = 0; !dead && i < ntiles; ++i) {
      if (*s_abort) { fail(); break; }
      const int cnt = min(kTN, n - (tile0 + i) * kTN);
      // S of tile i: MODE 0 / 1 buffer i % 2; MODE 2 the group's buffer, tile i in
      // its 32 columns i % G
      if (!__all_sync(kTF, mbar_wait_bounded(PRESPLIT ? s_full : &s_full[i & 1],
                                             PRESPLIT ? (uint32_t)((i / G) & 1) : (uint32_t)((i >> 1) & 1),
                                             kWaitLimitNs))) {
        fail();
        break;
      }
      tc_fence_after();
      uint32_t sr[32];
      tc_ld32(tmem + lane_off + (PRESPLIT ? C::C_S0 + (uint32_t)((i % G) * kTN) : ((i & 1) ? C::C_S1 : C::C_S0)),
              sr);
      tc_wait_ld();
      if (PRESPLIT && (i % G == G - 1 || i == ntiles - 1)) {
        // every tile of the group's S is read: S of the next group may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty);
      }
      // window mask; a tile wholly inside this row's window skips it (a whole
      // segment row sees every key of its segment: only the tail is masked)
      const int j0 = (tile0 + i) * kTN;
      const bool inside = FLASH ? q_ok && cnt == kTN
                                : q_ok && cnt == kTN && j0 >= p.ns && xlo + (j0 - p.ns) >= q_lo &&
                                      xlo + (j0 + kTN - 1 - p.ns) <= q_hi;
      float tmax = -INFINITY;
      float s[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        bool v = true;
        if (!inside) {
          const int j = j0 + k;
          v = q_ok && k < cnt;
          if (!FLASH && v && j >= p.ns) {
            const int x = xlo + (j - p.ns);
            v = x >= q_lo && x <= q_hi;
          }
        }
        s[k] = v ? __uint_as_float(sr[k]) : -INFINITY;
        tmax = fmaxf(tmax, s[k]);
      }
      // The running max m_run moves only when a tile exceeds it by more than
      // kLazyMax (log2 units): below that, p = 2^(s - m_run) <= 2^kLazyMax and
      // O and l keep one common scale, so o = O / l is unchanged while the
      // O rescale in tensor memory is skipped.
      const bool raise = tmax > m_run + kLazyMax;
      const float m_new = raise ? tmax : m_run;
      const float c = raise ? exp2f(m_run - m_new) : 1.f;
      uint32_t phi[32], plo[32];
      float psum = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float pv = m_new == -INFINITY ? 0.f : exp2f(s[k] - m_new);
        psum += pv;
        phi[k] = tf32_hi(pv);
        plo[k] = tf32_hi(pv - __uint_as_float(phi[k]));
      }
      l_run = l_run * c + psum;
      m_run = m_new;
      // P V of tile i - 1 must be complete before P and O are rewritten; the
      // work above overlapped it
      if (i >= 1 && !__all_sync(kTF, mbar_wait_bounded(pv_done, (uint32_t)((i - 1) & 1), kWaitLimitNs))) {
        fail();
        break;
      }
      tc_fence_after();
      if constexpr (P_SMEM) {
        // row q of P in the K-major layout: (q / 8) * P_SBO + (k / 4) * 128 + (q % 8) * 16 +
        // (k % 4) * 4 bytes (8 lanes write 128 contiguous bytes per store)
        const int prow = (q >> 3) * (int)C::P_SBO + (q & 7) * 16;
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
          *reinterpret_cast<uint4*>(sm + C::OFF_PHI + prow + k4 * 128) =
              make_uint4(phi[4 * k4], phi[4 * k4 + 1], phi[4 * k4 + 2], phi[4 * k4 + 3]);
          *reinterpret_cast<uint4*>(sm + C::OFF_PLO + prow + k4 * 128) =
              make_uint4(plo[4 * k4], plo[4 * k4 + 1], plo[4 * k4 + 2], plo[4 * k4 + 3]);
        }
        // the generic-proxy stores become visible to the MMA's (async-proxy) reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      } else {
        tc_st32(tmem + lane_off + C::C_PHI, phi);
        tc_st32(tmem + lane_off + C::C_PLO, plo);
      }
      // rescale this row of O when its max moved (warp-uniform decision)
      if (i > 0 && __any_sync(kTF, c != 1.f)) {
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t o[32];
          tc_ld32(tmem + lane_off + C::C_O + c0, o);
          tc_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * c);
          tc_st32(tmem + lane_off + C::C_O + c0, o);
        }
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
    }
    // ---- the block's record: m, l, O (unnormalised)
    if (!dead && !*s_abort) {
      const bool ok = __all_sync(kTF, ntiles == 0 ||
                                          mbar_wait_bounded(pv_done, (uint32_t)((ntiles - 1) & 1), kWaitLimitNs));
      if (ok && FLASH && npiece > 1) {
        // a piece of a split unit: its record (O unnormalised, then m, l) to the
        // workspace; per softmax warp (32 query vectors), the last of the unit's
        // pieces to get there combines all of them. No wait on another CTA.
        tc_fence_after();
        const size_t rstride = (size_t)kTM * (HD + 2);
        float* rec = p.ws_rec + (size_t)tail_at * rstride;
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t o[32];
          tc_ld32(tmem + lane_off + C::C_O + c0, o);
          tc_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(rec + (size_t)q * HD + c0 + k) =
                ntiles > 0 ? make_float4(__uint_as_float(o[k]), __uint_as_float(o[k + 1]),
                                         __uint_as_float(o[k + 2]), __uint_as_float(o[k + 3]))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        reinterpret_cast<float2*>(rec + kTM * HD)[q] =
            ntiles > 0 ? make_float2(m_run, l_run) : make_float2(-INFINITY, 0.f);
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(p.ws_cnt + (size_t)(tail_at / npiece) * 4 + warp, 1) == npiece - 1;
        if (__shfl_sync(kTF, last, 0)) {
          __threadfence();
          const float* rec0 = p.ws_rec + (size_t)(tail_at - piece) * rstride;
          auto ml_of = [&](int j) { return __ldcg(reinterpret_cast<const float2*>(rec0 + j * rstride + kTM * HD) + q); };
          float M = -INFINITY;
          for (int j = 0; j < npiece; ++j) M = fmaxf(M, ml_of(j).x);
          float den = 0.f;
          for (int j = 0; j < npiece; ++j) {
            const float2 ml = ml_of(j);
            if (ml.x != -INFINITY) den += ml.y * exp2f(ml.x - M);   // a piece without keys weighs 0
          }
          const float inv = 1.0f / den;
          if (q_ok) {
            float* dst = p.out + (size_t)(s0 + r) * p.ldo + ((size_t)g * p.hpg + (q % p.hpg)) * HD;
            for (int c = 0; c < HD; c += 4) {
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int j = 0; j < npiece; ++j) {
                const float2 ml = ml_of(j);
                if (ml.x == -INFINITY) continue;
                const float w = exp2f(ml.x - M);
                const float4 v = __ldcg(reinterpret_cast<const float4*>(rec0 + j * rstride + (size_t)q * HD + c));
                acc.x += v.x * w; acc.y += v.y * w; acc.z += v.z * w; acc.w += v.w * w;
              }
              *reinterpret_cast<float4*>(dst + c) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            }
          }
        }
      } else if (ok && FLASH) {
        // o = O / l straight to the output row of this query vector
        tc_fence_after();
        const float inv = 1.0f / l_run;
        float* dst = p.out + (size_t)(s0 + r) * p.ldo + ((size_t)g * p.hpg + (q % p.hpg)) * HD;
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t o[32];
          tc_ld32(tmem + lane_off + C::C_O + c0, o);
          tc_wait_ld();
          if (q_ok) {
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              *reinterpret_cast<float4*>(dst + c0 + k) =
                  make_float4(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                              __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
          }
        }
      } else if (ok) {
        tc_fence_after();
        const size_t item = ((size_t)bg * p.n_rb + rb) * p.splits;
        float* dst = p.ws_acc + (item * (size_t)p.nq + q) * HD;
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t o[32];
          tc_ld32(tmem + lane_off + C::C_O + c0, o);
          tc_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(dst + c0 + k) =
                make_float4(__uint_as_float(o[k]), __uint_as_float(o[k + 1]), __uint_as_float(o[k + 2]),
                            __uint_as_float(o[k + 3]));
        }
        p.ws_ml[item * p.nq + q] = make_float2(m_run, l_run);
      } else if (lane == 0) {
        *s_abort = 1;
        set_err(p.err, SWA_DERR_TIMEOUT);
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  // Outstanding MMAs of an aborted run finish on their own; wait (bounded) for
  // the last commit before the tensor memory is released.
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    if (*s_abort && ntiles > 0) mbar_wait_bounded(pv_done, (uint32_t)((ntiles - 1) & 1), kWaitLimitNs);
    tc_fence_after();
    tc_dealloc(tmem, C::TMEM_COLS);
  }
}

// One 32-key block as TF32 hi/lo operands, by a CTA of 256 threads: the K rows in
// the K-major layout of the kernel's K operand ((key / 8) * K_SBO + (f / 4) * 128 +
// (key % 8) * 16 + (f % 4) * 4 bytes) and the V rows transposed likewise ((f / 8) *
// V_SBO + (key / 4) * 128 + (f % 8) * 16 + (key % 4) * 4); keys whose source is
// null are zeros. Same arithmetic as the split warps: bit-identical operands.
// src(key, &k, &v) gives the key's K and V rows (nullptr: none).
template <int HD, class Src>
__device__ __forceinline__ void split_block(uint32_t* dst, Src src) {
  using C = TCfg<HD>;
  constexpr int D4 = HD / 4;
  __shared__ __align__(16) float vs[kTN][HD + 4];
  // K: thread -> (key, f4) with key % 8 fastest, so 8 threads write 128 contiguous bytes
  for (int idx = threadIdx.x; idx < kTN * D4; idx += blockDim.x) {
    const int key = (idx & 7) + 8 * (idx / (8 * D4)), f4 = (idx >> 3) % D4;
    const float* kr = nullptr;
    const float* vr = nullptr;
    src(key, &kr, &vr);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 w = v;
    if (kr) {
      v = *reinterpret_cast<const float4*>(kr + f4 * 4);
      w = *reinterpret_cast<const float4*>(vr + f4 * 4);
    }
    *reinterpret_cast<float4*>(&vs[key][f4 * 4]) = w;
    const float x[4] = {v.x, v.y, v.z, v.w};
    uint4 hv, lv;
    uint32_t* hp = &hv.x;
    uint32_t* lp = &lv.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hp[e] = tf32_hi(x[e]);
      lp[e] = tf32_hi(x[e] - __uint_as_float(hp[e]));
    }
    const int off = ((key >> 3) * (int)C::K_SBO + f4 * 128 + (key & 7) * 16) / 4;
    *reinterpret_cast<uint4*>(dst + off) = hv;
    *reinterpret_cast<uint4*>(dst + kTN * HD + off) = lv;
  }
  __syncthreads();
  // V^T: thread -> (f, 4 keys) with f % 8 fastest
  for (int idx = threadIdx.x; idx < HD * kTN / 4; idx += blockDim.x) {
    const int f = idx % HD, k4 = idx / HD;
    uint4 hv, lv;
    uint32_t* hp = &hv.x;
    uint32_t* lp = &lv.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = vs[k4 * 4 + e][f];
      hp[e] = tf32_hi(x);
      lp[e] = tf32_hi(x - __uint_as_float(hp[e]));
    }
    const int off = ((f >> 3) * (int)C::V_SBO + k4 * 128 + (f & 7) * 16) / 4;
    *reinterpret_cast<uint4*>(dst + 2 * kTN * HD + off) = hv;
    *reinterpret_cast<uint4*>(dst + 3 * kTN * HD + off) = lv;
  }
}

// swa_flash: one CTA per (segment, KV head, 32-key block) of the segment's rows.
template <int HD>
__global__ void __launch_bounds__(256) flash_presplit_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  // the attention's combine counters of a split launch tail (4 per tail unit)
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < 4 * p.flash_tail; i += blockDim.x) p.ws_cnt[i] = 0;
  const int blk = blockIdx.x, bg = blockIdx.y;
  const int b = bg / p.nk, g = bg % p.nk;
  const uint32_t s0 = p.segs[2 * b], len = p.segs[2 * b + 1];
  if ((uint64_t)s0 + len > (uint64_t)p.T || len > (uint32_t)p.max_len) return;   // the attention reports it
  const int j0 = blk * kTN;
  if (j0 >= (int)len) return;
  const int cnt = min(kTN, (int)len - j0);
  uint32_t* dst = reinterpret_cast<uint32_t*>(p.ops + ((size_t)bg * p.ops_nblk + blk) * 4 * (kTN * HD));
  split_block<HD>(dst, [&](int key, const float** kr, const float** vr) {
    if (key < cnt) {
      const float* row = p.qkv + (size_t)(s0 + j0 + key) * p.ld + (size_t)g * HD;
      *kr = row + p.k_off;
      *vr = row + p.v_off;
    }
  });
}

template <int HD, int MODE>
int launch_tc(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = TCfg<HD, MODE>;
  auto kern = attend_prompt_tc_kernel<HD, MODE>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  if (MODE == 2) {
    const dim3 pgrid((unsigned)p.ops_nblk, (unsigned)(p.B * p.nk));
    const int rc = finish_launch(launch_pdl(flash_presplit_kernel<HD>, pgrid, dim3(256), 0, s, p));
    if (rc != SWA_OK) return rc;
  }
  dim3 grid(1u, (unsigned)p.n_rb, (unsigned)(p.B * p.nk));
  if (MODE == 2 && p.flash_q > 1)   // 1-D: whole units, then the tail's pieces
    grid = dim3((unsigned)((long long)p.n_rb * p.B * p.nk - p.flash_tail + (long long)p.flash_tail * p.flash_q));
  if (e0) cudaEventRecord(e0, s);
  cudaError_t e = launch_pdl(kern, grid, dim3(kTThreads), C::BYTES, s, p);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e1) cudaEventRecord(e1, s);
  return cuda_status(e);
}

}  // namespace

int launch_attend_prompt_tc(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  switch (p.hd) {
    case 64: return launch_tc<64, 0>(p, s, e0, e1);
    case 128: return launch_tc<128, 0>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

int launch_flash_tc(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  switch (p.hd) {
    case 64: return p.ops ? launch_tc<64, 2>(p, s, e0, e1) : launch_tc<64, 1>(p, s, e0, e1);
    case 128: return p.ops ? launch_tc<128, 2>(p, s, e0, e1) : launch_tc<128, 1>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

}  // namespace swa
