// Prompt-chunk attention on the 5th-generation tensor cores (tcgen05, TMEM) with
// TF32 hi/lo operands that the kernel stages and splits itself: the GEMM path of
// "o1c_msl.metal" (cortiq-engine 0.8.79: o1c_gather, o1c_cols, o1c_gmax, o1c_gsoft,
// o1c_gadd and the engine GEMMs Q K^T and P V they feed) as one flash-style kernel
// per block of 128 query vectors. The token path takes it for prompt chunks given
// the minimum workspace (with room for split-once operand blocks the persistent f16
// kernel of swa_prompt_h16.cu runs instead); swa_flash takes it without a workspace
// (below).
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
// The same kernel with FLASH is swa_flash's full-sequence attention
// ("egemma2_msl.metal", cortiq-engine 0.8.17: eg_flash64 / eg_flash_staged):
// the keys of a row block are the rows of its segment of a packed q|k|v buffer,
// only the segment's tail is masked, and o = O / l is written directly.
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

template <int HD>
struct TCfg {
  static constexpr int NSETS = 2;                           // operand sets behind the split warps
  // TMEM columns: Q_hi | Q_lo | S buffers S0, S1 of 32 | O | P_hi | P_lo
  static constexpr uint32_t SCOLS = 2 * kTN;
  static constexpr uint32_t C_QHI = 0, C_QLO = HD, C_S0 = 2 * HD, C_S1 = 2 * HD + kTN;
  static constexpr uint32_t C_O = 2 * HD + SCOLS, C_PHI = 3 * HD + SCOLS, C_PLO = 3 * HD + SCOLS + kTN;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(C_PLO + kTN <= TMEM_COLS, "tensor memory budget");
  // shared memory (bytes)
  static constexpr int LAND = kTN * HD * 4;                 // one fp32 tile of K or V
  static constexpr int OFF_LK = 0;                          // [2 stages] K landing
  static constexpr int OFF_LV = 2 * LAND;                   // [2 stages] V landing
  static constexpr int OFF_OPS = 4 * LAND;                  // [NSETS] K_hi, K_lo, V^T_hi, V^T_lo
  static constexpr int SET = 4 * LAND;
  static constexpr int OFF_BAR = OFF_OPS + NSETS * SET;     // mbarriers
  static constexpr int NBAR = 16;
  // at least 116 KB, so that one CTA (and one 512-column TMEM allocation) runs per SM
  static constexpr size_t USED = (size_t)OFF_BAR + NBAR * 8 + 16;
  static constexpr size_t BYTES = USED > 118784 ? USED : 118784;
  static_assert(BYTES <= 232448, "227 KB of shared memory per CTA");
  // K-major core-matrix layouts: LBO = next core matrix along K, SBO = next 8 rows
  static constexpr uint32_t K_LBO = 128, K_SBO = (HD / 4) * 128;   // K_hi: rows = keys, K = features
  static constexpr uint32_t V_LBO = 128, V_SBO = (kTN / 4) * 128;  // V^T: rows = features, K = keys
};

__device__ __forceinline__ uint32_t tf32_hi(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// Without FLASH: a row block of the token path (sinks, ring window, chunk rows;
// split record to the workspace). With FLASH: a row block of one segment of packed
// q|k|v rows attending all of the segment's rows (swa_flash); blockIdx.z = segment *
// nk + KV head, and the normalised output is written directly.

template <int HD, bool FLASH>
__global__ void __launch_bounds__(kTThreads, 1) attend_prompt_tc_kernel(AttendParams p) {
  constexpr int NS = TCfg<HD>::NSETS;    // operand sets: tile j uses set j % NS
  pdl_trigger();
  pdl_wait();
  using C = TCfg<HD>;
  extern __shared__ __align__(1024) unsigned char sm[];
  float* landK = reinterpret_cast<float*>(sm + C::OFF_LK);
  float* landV = reinterpret_cast<float*>(sm + C::OFF_LV);
  // operand set k (k = tile % 2): K_hi, K_lo, V^T_hi, V^T_lo
  auto op = [&](int set, int which) {
    return reinterpret_cast<uint32_t*>(sm + C::OFF_OPS + set * C::SET + which * C::LAND);
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* land_full = bars + 0;    // [2] producer -> split warps (bytes)
  uint64_t* land_empty = bars + 2;   // [2] split warps -> producer (4 arrivals)
  uint64_t* split_done = bars + 4;   // [2 sets] split warps -> MMA (4 arrivals)
  uint64_t* s_full = bars + 8;       // [2 buffers] MMA commit: S of the tile done
  uint64_t* p_ready = bars + 10;     // softmax warps -> MMA (4 arrivals)
  uint64_t* pv_done = bars + 11;     // MMA commit -> softmax warps
  uint64_t* v_free = bars + 12;      // [2 sets] MMA commit (P V of the set done) -> split warps
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + C::NBAR);
  volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(reinterpret_cast<int*>(bars + C::NBAR) + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rb = blockIdx.y, bg = blockIdx.z;
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
  const int ntiles = (n + kTN - 1) / kTN;
  const size_t kv_head = (size_t)b * p.nk + g;

  if (tid == 0) {
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
  if (warp == 4) {
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
  if (warp == 5 && lane == 0) {
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
  if (warp >= 6) {
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
      const int cnt = min(kTN, n - i * kTN);
      // S of tile i in buffer i % 2
      if (!__all_sync(kTF, mbar_wait_bounded(&s_full[i & 1], (uint32_t)((i >> 1) & 1), kWaitLimitNs))) {
        fail();
        break;
      }
      tc_fence_after();
      uint32_t sr[32];
      tc_ld32(tmem + lane_off + ((i & 1) ? C::C_S1 : C::C_S0), sr);
      tc_wait_ld();
      // window mask; a tile wholly inside this row's window skips it (a whole
      // segment row sees every key of its segment: only the tail is masked)
      const int j0 = i * kTN;
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
      tc_st32(tmem + lane_off + C::C_PHI, phi);
      tc_st32(tmem + lane_off + C::C_PLO, plo);
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
      if (ok && FLASH) {
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

template <int HD, bool FLASH>
int launch_tc(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = TCfg<HD>;
  auto kern = attend_prompt_tc_kernel<HD, FLASH>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const dim3 grid(1u, (unsigned)p.n_rb, (unsigned)(p.B * p.nk));
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
    case 64: return launch_tc<64, false>(p, s, e0, e1);
    case 128: return launch_tc<128, false>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

int launch_flash_tc(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  switch (p.hd) {
    case 64: return launch_tc<64, true>(p, s, e0, e1);
    case 128: return launch_tc<128, true>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

}  // namespace swa
