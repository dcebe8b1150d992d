// Attention of a row block with 16 or 32 query vectors (speculative verify
// and other short chunks) on CUDA cores: o1c_score / o1c_soft / o1c_sum of
// "o1c_msl.metal" (cortiq-engine 0.8.79) for several rows at once, as one
// split-KV kernel writing the shared partial-record format (or, for ordered
// single-split blocks, the finished rows).
//
// With 32 query vectors per key the path does 16 flops per K/V byte, so the
// FP32 FMA pipe, not HBM, bounds it, and the design is about feeding that
// pipe: every FMA is a packed fma.rn.f32x2 and shared-memory wavefronts stay
// near half the FMA cycles in both products.
//  - 32-key tiles stream through STAGES shared-memory stages. Keys whose
//    sources are contiguous (a run of ring slots up to the wrap, the sinks,
//    the chunk rows) travel as ONE cp.async.bulk per run for K and one for V
//    into consecutive unpadded rows (4-16 KB copies run at the HBM read rate;
//    one 512-byte copy per row would cap the stream far below it). Warp 0
//    issues them: the first STAGES tiles up front, then each stage again as
//    soon as all four warps have released it. There is no separate producer
//    warp, so two CTAs put exactly two warps on each SM sub-partition and
//    every thread may hold the 128 accumulator registers the tiles need.
//  - Consumer warp w owns a group of QW query vectors and a range of KW keys of
//    every tile, with its own online softmax state for them; warps that share
//    query vectors combine their states once, after the key loop, so no CTA
//    barrier runs inside it.
//  - Scores: lane (kq, e) = (lane / 8, lane % 8) takes keys kq + 4j of the
//    warp's range and the float4 feature chunks e, e + 8, ...: each 8-lane
//    shared-memory phase reads one contiguous 128-byte piece of a K row. The
//    query vectors sit transposed ([feature][query], chunk-rotated by feature
//    so the 8 chunk lanes hit distinct banks) and are read as pairs of query
//    vectors, so one packed FMA updates the scores of two query vectors.
//    Transposed shuffles over the 8 chunk lanes leave each lane the full
//    scores of QW / 8 query vectors for its keys.
//  - P V: lane = (query group, feature group): all 16 query vectors of the
//    warp and 4 features at hd 128 (8 x 4 at hd 64, 8 x 8 at hd 256); P is
//    handed over through a per-warp shared slice as plain floats read as
//    natural pairs of query vectors, V is duplicated in a register (one pair
//    feeds QPL / 2 packed FMAs), and each lane accumulates its QPL x FPL tile
//    of the numerator as pairs (O[q][f], O[q + 1][f]).
//  - Ordered blocks (p.ws_order): one split per block and a 1-D grid over the
//    order order_verify_kernel writes (longest first); with p.fused the CTA, the
//    only reader of its KV head's ring, normalises, gates and writes its rows and
//    commits its KV head's chunk rows (and, for KV head 0, the meta) itself.
#include "swa_internal.cuh"
#include "swa_h16.cuh"

namespace swa {
namespace {

constexpr int kVCW = 4;                        // warps (all consume; warp 0 also issues copies)
constexpr int kVThreads = kVCW * 32;
constexpr unsigned kVFull = 0xffffffffu;

typedef unsigned long long u64;

__device__ __forceinline__ u64 ffma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
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
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  u64 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float comp(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

template <int HD, int NQ>
struct VCfg {
  static constexpr int QW = HD == 256 ? 8 : 16;   // query vectors per consumer warp
  static constexpr int QG = NQ / QW;              // query groups
  static constexpr int KG = kVCW / QG;            // key groups (warps per query group)
  static constexpr int KW = TK / KG;              // keys per warp per tile
  static constexpr int KPL = KW / 4;              // keys per lane in the scores
  static constexpr int CH = HD / 32;              // float4 chunks per lane in the scores
  static constexpr int QO = QW / 8;               // query vectors a lane owns after the reduction
  // feature lanes in P V: 32 (every lane takes all QW query vectors) unless a
  // lane would hold fewer than 4 features
  static constexpr int FG = QW == 16 && HD == 64 ? 16 : 32;
  static constexpr int QGL = 32 / FG;             // query lanes in P V
  static constexpr int QPL = QW / QGL;            // query vectors per lane in P V
  static constexpr int FPL = HD / FG;             // features per lane in P V
  static constexpr int FCH = FPL / 4;
  static constexpr int STAGES = HD == 64 ? 4 : 2;
  static constexpr int OFF_K = 0;                             // [STAGES][TK][HD]
  static constexpr int OFF_V = STAGES * TK * HD;              // [STAGES][TK][HD]
  static constexpr int OFF_QT = 2 * STAGES * TK * HD;         // [HD][32] rotated chunks
  static constexpr int OFF_P = OFF_QT + HD * 32;              // [kVCW][KW][QW] (p, p)
  static constexpr int OFF_C = OFF_P + kVCW * KW * QW * 2;    // [kVCW][QW] (c, c)
  static constexpr int OFF_ML = OFF_C + kVCW * QW * 2;        // [kVCW][QW] (m, l)
  static constexpr int OFF_FLAG = OFF_ML + kVCW * QW * 2;
  static constexpr int FLOATS = ((OFF_FLAG + 4 + 1) / 2) * 2;
  static constexpr size_t BYTES = (size_t)FLOATS * 4 + 2 * STAGES * sizeof(uint64_t);
  static constexpr int MIN_BLOCKS = HD == 256 ? 1 : 2;
  static_assert(NQ == 16 || NQ == 32, "16 or 32 query vectors");
  static_assert(QG * KG == kVCW && KPL >= 1 && (QPL == 8 || QPL == 16) && FCH >= 1, "warp arrangement");
  static_assert(kVCW * QW * HD <= 2 * STAGES * TK * HD, "warp states fit the stage buffers");
};

template <int HD, int NQ>
__global__ void __launch_bounds__(kVThreads, VCfg<HD, NQ>::MIN_BLOCKS)
attend_verify_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  using C = VCfg<HD, NQ>;
  extern __shared__ __align__(128) float smem[];
  float* Ks = smem + C::OFF_K;
  float* Vs = smem + C::OFF_V;
  float* QT = smem + C::OFF_QT;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::FLOATS);
  uint64_t* empty = full + C::STAGES;

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  int s = blockIdx.x, rb = blockIdx.y, bg = blockIdx.z;
  if (p.ws_order) {           // ordered blocks: one split each, a 1-D grid over the order
    const int u = p.ws_order[blockIdx.x];
    s = 0;
    rb = u % p.n_rb;
    bg = u / p.n_rb;
  }
  const int b = bg / p.nk, g = bg % p.nk;

  const SeqState st = load_state(p, b, tid == 0 && g == 0 && rb == 0 && s == 0);
  const int r0 = rb * p.rows;
  const int r_last = min(r0 + p.rows, p.t) - 1;
  const int rows_eff = r_last - r0 + 1;
  const int win0 = min(st.W, st.len0 + r0 + 1);
  const int xlo = st.len0 + r0 + 1 - win0;       // first logical key of the block
  const int n = p.ns + (st.len0 + r_last - xlo + 1);
  if (!p.fused) {
    if (g == 0 && s == 0 && tid == 0) p.ws_nsplit[b * p.n_rb + rb] = (n + p.chunk - 1) / p.chunk;
    if (g == 0 && s == 0 && rb == 0 && tid == 0) p.ws_meta[b] = p.meta[b];
  }
  const int jb = s * p.chunk;
  if (jb >= n) return;
  const int je = min(n, jb + p.chunk);
  const int ntiles = (je - jb + TK - 1) / TK;

  if (tid == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kVCW);
    }
    mbar_fence_init();
    *s_abort = 0;
  }
  // Query vectors of the block (rows then heads) times scale * log2 e, stored
  // transposed: feature f holds the 32 query slots as 8 float4 chunks, chunk
  // c at position c ^ ((f / 4) mod 8).
  {
    constexpr int PER = 32 * (HD / 4) / kVThreads;   // float4 loads per thread
    const int q = tid % 32;                           // a warp covers the 32 query slots of a chunk
    const int rr = q / p.hpg, h = q % p.hpg;
    const bool live = q < NQ && rr < rows_eff && q < p.rows * p.hpg;
    const float* qsrc = p.q + (((size_t)b * p.t + r0 + rr) * p.nh + (size_t)g * p.hpg + h) * HD;
    float4 v[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {                   // all loads in flight before the stores
      const int d4 = tid / 32 + k * (kVThreads / 32);
      v[k] = live ? *reinterpret_cast<const float4*>(qsrc + d4 * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int d4 = tid / 32 + k * (kVThreads / 32);
      const int pos = (((q >> 2) ^ d4) & 7) * 4 + (q & 3);
      QT[(d4 * 4 + 0) * 32 + pos] = v[k].x * p.qmul;
      QT[(d4 * 4 + 1) * 32 + pos] = v[k].y * p.qmul;
      QT[(d4 * 4 + 2) * 32 + pos] = v[k].z * p.qmul;
      QT[(d4 * 4 + 3) * 32 + pos] = v[k].w * p.qmul;
    }
  }
  __syncthreads();
  const size_t kv_head = (size_t)b * p.nk + g;

  // ------------------------------------------------------------ copy issue
  // Warp 0 copies tile `it` into its stage: the source row of key `lane`; a
  // lane whose row does not follow its left neighbour's starts a run and
  // issues one copy of the whole run.
  auto issue_tile = [&](int it) {
    const int stage = it % C::STAGES;
    const int j0 = jb + it * TK;
    const int cnt = min(TK, je - j0);
    if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)(cnt * HD * 4 * 2));
    __syncwarp();
    const float* sk = nullptr;
    const float* sv = nullptr;
    if (lane < cnt) {
      const int j = j0 + lane;
      if (j < p.ns) {
        const size_t at = (kv_head * p.ns + j) * HD;
        sk = p.sink_k + at;
        sv = p.sink_v + at;
      } else {
        const int x = xlo + (j - p.ns);
        if (x < st.len0) {
          int slot = st.head0 + x;
          if (slot >= st.W) slot -= st.W;        // head0 < W and x < W
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
    const u64 prev_k = __shfl_up_sync(kVFull, reinterpret_cast<u64>(sk), 1);
    const u64 prev_v = __shfl_up_sync(kVFull, reinterpret_cast<u64>(sv), 1);
    const bool start = lane < cnt &&
                       (lane == 0 || reinterpret_cast<u64>(sk) != prev_k + HD * 4 ||
                        reinterpret_cast<u64>(sv) != prev_v + HD * 4);
    const unsigned starts = __ballot_sync(kVFull, start);
    if (start) {
      const unsigned later = starts & ~((2u << lane) - 1u);
      const int end = later ? __ffs(later) - 1 : cnt;
      const uint32_t bytes = (uint32_t)((end - lane) * HD * 4);
      bulk_g2s(Ks + ((size_t)stage * TK + lane) * HD, sk, bytes, &full[stage]);
      bulk_g2s(Vs + ((size_t)stage * TK + lane) * HD, sv, bytes, &full[stage]);
    }
  };
  int issued = 0;                                 // tiles warp 0 has issued
  if (warp == 0) {
    for (; issued < C::STAGES && issued < ntiles; ++issued) issue_tile(issued);
  }

  // ------------------------------------------------------------------ consumers
  const int e = lane & 7, kq = lane >> 3;
  const int qgrp = warp % C::QG, kgrp = warp / C::QG;
  const int kbase = kgrp * C::KW;                 // the warp's first key of every tile
  // query vectors this lane owns after the score reduction: qgrp*QW + e*QO + o
  int q_lo[C::QO], q_hi[C::QO];
  bool q_ok[C::QO];
#pragma unroll
  for (int o = 0; o < C::QO; ++o) {
    const int q = qgrp * C::QW + e * C::QO + o;
    const int rr = q / p.hpg;
    const int r = r0 + rr;
    q_ok[o] = rr < rows_eff && q < p.rows * p.hpg;
    q_lo[o] = st.len0 + r + 1 - min(st.W, st.len0 + r + 1);
    q_hi[o] = st.len0 + r;
  }
  // logical keys inside the window of every row of the block
  const int x_in_lo = st.len0 + r_last + 1 - min(st.W, st.len0 + r_last + 1);
  const int x_in_hi = st.len0 + r0;
  float m[C::QO], l[C::QO];
#pragma unroll
  for (int o = 0; o < C::QO; ++o) {
    m[o] = -INFINITY;
    l[o] = 0.f;
  }
  // P V lane arrangement
  const int fg = lane % C::FG, qgl = lane / C::FG;
  // O as pairs of query vectors: acc[k2][f] = (O[q][f], O[q + 1][f]) for the
  // lane's query vectors q = qgl * QPL + 2 k2 and its features f
  u64 acc[C::QPL / 2][C::FPL];
#pragma unroll
  for (int k = 0; k < C::QPL / 2; ++k)
#pragma unroll
    for (int d = 0; d < C::FPL; ++d) acc[k][d] = 0ull;

  float* Pw = smem + C::OFF_P + warp * C::KW * C::QW;     // [KW][QW] P of the warp's keys
  float* Cw = smem + C::OFF_C + warp * C::QW;             // [QW] rescale factors
  const u64 one2 = pack2(1.f, 1.f);
  const bool b1 = (e & 2) != 0, b0 = (e & 1) != 0;
  // Visit order of the warp's query chunks: after the chunk-level reduction
  // rounds (lane bits 2 and 1 when QW = 16, bit 2 when QW = 8) a lane keeps
  // the chunk whose index bits equal those lane bits.
  const int uperm = C::QW == 16 ? (e >> 1) : (e >> 2);

  int consumed = 0;                               // tiles whose copies have landed
  for (int i = 0; i < ntiles; ++i) {
    const int stage = i % C::STAGES;
    const bool ok = __all_sync(kVFull, mbar_wait_bounded(&full[stage], (uint32_t)((i / C::STAGES) & 1),
                                                       kWaitLimitNs));
    if (!ok) {
      if (lane == 0) {
        *s_abort = 1;
        set_err(p.err, SWA_DERR_TIMEOUT);
      }
      break;
    }
    consumed = i + 1;
    if (__shfl_sync(kVFull, *s_abort, 0)) break;
    const int j0 = jb + i * TK;
    const int cnt = min(TK, je - j0);
    const float* Kt = Ks + (size_t)stage * TK * HD;
    const float* Vt = Vs + (size_t)stage * TK * HD;

    // ---- partial scores: keys kbase + kq + 4j, query pairs of the warp's group
    u64 sp[C::KPL][C::QW / 2];
#pragma unroll
    for (int j = 0; j < C::KPL; ++j)
#pragma unroll
      for (int u = 0; u < C::QW / 2; ++u) sp[j][u] = 0ull;
#pragma unroll
    for (int c = 0; c < C::CH; ++c) {
      const int ch = e + 8 * c;
      float4 kv[C::KPL];
#pragma unroll
      for (int j = 0; j < C::KPL; ++j)
        kv[j] = *reinterpret_cast<const float4*>(Kt + (size_t)(kbase + kq + 4 * j) * HD + ch * 4);
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const float* qrow = QT + (ch * 4 + f) * 32;
        u64 kd[C::KPL];
#pragma unroll
        for (int j = 0; j < C::KPL; ++j) {
          const float kf = comp(kv[j], f);
          kd[j] = pack2(kf, kf);
        }
#pragma unroll
        for (int u = 0; u < C::QW / 4; ++u) {
          const int lc = qgrp * (C::QW / 4) + (u ^ uperm);
          const ulonglong2 qv = *reinterpret_cast<const ulonglong2*>(qrow + ((lc ^ e) & 7) * 4);
#pragma unroll
          for (int j = 0; j < C::KPL; ++j) {
            sp[j][2 * u] = ffma2(qv.x, kd[j], sp[j][2 * u]);
            sp[j][2 * u + 1] = ffma2(qv.y, kd[j], sp[j][2 * u + 1]);
          }
        }
      }
    }
    // ---- transposed reduction over the 8 chunk lanes (lane bits 2, 1, 0).
    // The lane's query chunks were visited in the order u ^ uperm, so at the
    // chunk-level rounds the half a lane keeps is always its first half: no
    // selects there.
    constexpr int P0 = C::QW / 2;                 // query pairs before the reduction
    u64 r1[C::KPL][P0 / 2];
#pragma unroll
    for (int j = 0; j < C::KPL; ++j)
#pragma unroll
      for (int k = 0; k < P0 / 2; ++k)
        r1[j][k] = ffma2(sp[j][k], one2, __shfl_xor_sync(kVFull, sp[j][P0 / 2 + k], 4));
    u64 r2[C::KPL][P0 / 4];
#pragma unroll
    for (int j = 0; j < C::KPL; ++j)
#pragma unroll
      for (int k = 0; k < P0 / 4; ++k) {
        if constexpr (C::QW == 16) {
          r2[j][k] = ffma2(r1[j][k], one2, __shfl_xor_sync(kVFull, r1[j][P0 / 4 + k], 2));
        } else {
          const u64 send = b1 ? r1[j][k] : r1[j][P0 / 4 + k];
          const u64 keep = b1 ? r1[j][P0 / 4 + k] : r1[j][k];
          r2[j][k] = ffma2(keep, one2, __shfl_xor_sync(kVFull, send, 2));
        }
      }
    float sc[C::KPL][C::QO];
#pragma unroll
    for (int j = 0; j < C::KPL; ++j) {
      if constexpr (C::QO == 2) {                 // one pair left per lane: queries 2e, 2e + 1
        const u64 send = b0 ? r2[j][0] : r2[j][1];
        const u64 keep = b0 ? r2[j][1] : r2[j][0];
        const float2 v = unpack2(ffma2(keep, one2, __shfl_xor_sync(kVFull, send, 1)));
        sc[j][0] = v.x;
        sc[j][1] = v.y;
      } else {                                    // split the last pair: query e
        const float2 v = unpack2(r2[j][0]);
        const float send = b0 ? v.x : v.y;
        const float keep = b0 ? v.y : v.x;
        sc[j][0] = keep + __shfl_xor_sync(kVFull, send, 1);
      }
    }
    // ---- window mask, online softmax of the owned query vectors over the
    // warp's keys of this tile, P and the rescale factors to shared memory
    // A tile whose keys are all present and inside every row's window needs
    // no mask (warp-uniform test; query slots past the block's rows hold zero
    // vectors and their records are never read).
    const bool inside = cnt == TK && xlo + (max(j0, p.ns) - p.ns) >= x_in_lo &&
                        xlo + (j0 + TK - 1 - p.ns) <= x_in_hi;
    float cq[C::QO];
#pragma unroll
    for (int o = 0; o < C::QO; ++o) {
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < C::KPL; ++j) {
        if (!inside) {
          const int kl = kbase + kq + 4 * j;
          const int jj = j0 + kl;
          bool v = kl < cnt && q_ok[o];
          if (v && jj >= p.ns) {
            const int x = xlo + (jj - p.ns);
            v = x >= q_lo[o] && x <= q_hi[o];
          }
          sc[j][o] = v ? sc[j][o] : -INFINITY;
        }
        tmax = fmaxf(tmax, sc[j][o]);
      }
      tmax = fmaxf(tmax, __shfl_xor_sync(kVFull, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(kVFull, tmax, 16));
      const float m_new = fmaxf(m[o], tmax);
      float c = 1.f, lsum = 0.f;
      if (m_new != -INFINITY) {
        c = h16::ex2(m[o] - m_new);
#pragma unroll
        for (int j = 0; j < C::KPL; ++j) {
          sc[j][o] = h16::ex2(sc[j][o] - m_new);
          lsum += sc[j][o];
        }
      } else {
#pragma unroll
        for (int j = 0; j < C::KPL; ++j) sc[j][o] = 0.f;
      }
      l[o] = l[o] * c + lsum;
      m[o] = m_new;
      cq[o] = c;
    }
#pragma unroll
    for (int j = 0; j < C::KPL; ++j) {
      float* dst = Pw + (size_t)(kq + 4 * j) * C::QW + e * C::QO;
      if constexpr (C::QO == 2) {
        *reinterpret_cast<float2*>(dst) = make_float2(sc[j][0], sc[j][1]);
      } else {
        *dst = sc[j][0];
      }
    }
    if (kq == 0) {
#pragma unroll
      for (int o = 0; o < C::QO; ++o) Cw[e * C::QO + o] = cq[o];
    }
    __syncwarp();

    // ---- P V: lane = (query group qgl of 8, feature group fg)
    bool moved = false;
#pragma unroll
    for (int o = 0; o < C::QO; ++o) moved |= cq[o] != 1.f;
    if (__any_sync(kVFull, moved)) {                // some running max moved: rescale
#pragma unroll
      for (int k2 = 0; k2 < C::QPL / 2; ++k2) {
        const u64 cc = *reinterpret_cast<const u64*>(Cw + qgl * C::QPL + 2 * k2);
#pragma unroll
        for (int d = 0; d < C::FPL; ++d) acc[k2][d] = mul2(acc[k2][d], cc);
      }
    }
    const int nkv = min(C::KW, cnt - kbase);
    auto pv_key = [&](int kk) {
      // P of the lane's query vectors as natural pairs (q, q + 1); V once per feature
      u64 pk[C::QPL / 2];
#pragma unroll
      for (int k4 = 0; k4 < C::QPL / 4; ++k4) {
        const ulonglong2 a =
            *reinterpret_cast<const ulonglong2*>(Pw + (size_t)kk * C::QW + qgl * C::QPL + 4 * k4);
        pk[2 * k4] = a.x;
        pk[2 * k4 + 1] = a.y;
      }
      const float* vr = Vt + (size_t)(kbase + kk) * HD;
      float vf[C::FPL];
#pragma unroll
      for (int u = 0; u < C::FCH; ++u) {
        const float4 a = *reinterpret_cast<const float4*>(vr + (fg + C::FG * u) * 4);
        vf[4 * u] = a.x;
        vf[4 * u + 1] = a.y;
        vf[4 * u + 2] = a.z;
        vf[4 * u + 3] = a.w;
      }
#pragma unroll
      for (int d = 0; d < C::FPL; ++d) {
        const u64 vd = pack2(vf[d], vf[d]);
#pragma unroll
        for (int k2 = 0; k2 < C::QPL / 2; ++k2) acc[k2][d] = ffma2(pk[k2], vd, acc[k2][d]);
      }
    };
    // A full share of keys runs fully unrolled: every P and V load can be hoisted
    // ahead of the products (5 % of the kernel against two keys a trip)
    if (nkv == C::KW) {
#pragma unroll
      for (int kk = 0; kk < C::KW; ++kk) pv_key(kk);
    } else {
#pragma unroll 2
      for (int kk = 0; kk < nkv; ++kk) pv_key(kk);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (warp == 0 && issued < ntiles) {           // refill this stage with tile i + STAGES
      bool ok2 = mbar_wait_bounded(&empty[stage], (uint32_t)((i / C::STAGES) & 1), kWaitLimitNs);
      ok2 = __all_sync(kVFull, ok2);
      if (!ok2) {
        if (lane == 0) {
          *s_abort = 1;
          set_err(p.err, SWA_DERR_TIMEOUT);
        }
        break;
      }
      fence_proxy_async_smem();
      issue_tile(issued);
      ++issued;
    }
  }
  // No copy may still be landing in shared memory when the CTA ends: on an
  // early exit warp 0 waits (bounded) for the tiles it issued beyond the
  // last one it consumed.
  if (warp == 0) {
    for (int it = max(consumed, issued - C::STAGES); it < issued; ++it)
      mbar_wait_bounded(&full[it % C::STAGES], (uint32_t)((it / C::STAGES) & 1), kWaitLimitNs);
  }

  // ---- combine the states of the warps sharing a query group into the
  // CTA's partial record
#pragma unroll
  for (int o = 0; o < C::QO; ++o) {
    l[o] += __shfl_xor_sync(kVFull, l[o], 8);
    l[o] += __shfl_xor_sync(kVFull, l[o], 16);
  }
  named_barrier(1, kVCW * 32);                 // every consumer is past its last tile
  if (*s_abort) return;
  float* MLs = smem + C::OFF_ML;
  if (kq == 0) {
#pragma unroll
    for (int o = 0; o < C::QO; ++o) {
      MLs[(warp * C::QW + e * C::QO + o) * 2 + 0] = m[o];
      MLs[(warp * C::QW + e * C::QO + o) * 2 + 1] = l[o];
    }
  }
  float* red = smem;                           // [kVCW][QW][HD], reuses the stage buffers
#pragma unroll
  for (int k2 = 0; k2 < C::QPL / 2; ++k2) {
    float* row0 = red + ((size_t)warp * C::QW + qgl * C::QPL + 2 * k2) * HD;
    float* row1 = row0 + HD;
#pragma unroll
    for (int u = 0; u < C::FCH; ++u) {
      const float2 a0 = unpack2(acc[k2][4 * u]);
      const float2 a1 = unpack2(acc[k2][4 * u + 1]);
      const float2 a2 = unpack2(acc[k2][4 * u + 2]);
      const float2 a3 = unpack2(acc[k2][4 * u + 3]);
      *reinterpret_cast<float4*>(row0 + (fg + C::FG * u) * 4) = make_float4(a0.x, a1.x, a2.x, a3.x);
      *reinterpret_cast<float4*>(row1 + (fg + C::FG * u) * 4) = make_float4(a0.y, a1.y, a2.y, a3.y);
    }
  }
  named_barrier(1, kVCW * 32);

  if (p.fused) {
    // ---- the block's rows finished here (the only split of a (sequence, KV head)):
    // o = O / l, gated, to the output (what the merge computes for one split, bit for
    // bit); then this KV head's chunk rows committed to its ring, which no other CTA
    // reads, and the sequence's meta by the CTA of KV head 0 (meta_out is not meta)
    for (int idx = tid; idx < NQ * HD / 4; idx += kVCW * 32) {
      const int q = idx / (HD / 4), d4 = idx % (HD / 4);
      const int rr = q / p.hpg, h = q % p.hpg;
      if (rr >= rows_eff || q >= p.rows * p.hpg) continue;
      const int qg = q / C::QW, ql = q % C::QW;
      float M = -INFINITY;
#pragma unroll
      for (int kg = 0; kg < C::KG; ++kg) M = fmaxf(M, MLs[((qg + C::QG * kg) * C::QW + ql) * 2]);
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      float L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int kg = 0; kg < C::KG; ++kg) {
          const int w = qg + C::QG * kg;
          const float mw = MLs[(w * C::QW + ql) * 2];
          if (mw == -INFINITY) continue;
          const float f = exp2f(mw - M);
          L += MLs[(w * C::QW + ql) * 2 + 1] * f;
          const float4 a = *reinterpret_cast<const float4*>(red + ((size_t)w * C::QW + ql) * HD + d4 * 4);
          sum.x += a.x * f; sum.y += a.y * f; sum.z += a.z * f; sum.w += a.w * f;
        }
      }
      const size_t row = ((size_t)b * p.t + r0 + rr) * p.nh + (size_t)g * p.hpg + h;
      const float4 gt = *reinterpret_cast<const float4*>(p.gate + row * HD + d4 * 4);
      const float4 gs = *reinterpret_cast<const float4*>(p.gate_scale + ((size_t)g * p.hpg + h) * HD + d4 * 4);
      const float inv = 1.0f / L;
      *reinterpret_cast<float4*>(p.out + row * HD + d4 * 4) =
          make_float4(gated(sum.x, inv, gt.x, gs.x), gated(sum.y, inv, gt.y, gs.y), gated(sum.z, inv, gt.z, gs.z),
                      gated(sum.w, inv, gt.w, gs.w));
    }
    if (p.commit) {
      const int first = max(0, p.t - st.W);        // only the last W rows survive
      const int nrow = p.t - first;
      for (int idx = tid; idx < nrow * (HD / 4); idx += kVCW * 32) {
        const int j = first + idx / (HD / 4), d4 = idx % (HD / 4);
        const int slot = (int)(((long long)st.head0 + st.len0 + j) % st.W);
        const size_t src = (((size_t)b * p.t + j) * p.nk + g) * HD + d4 * 4;
        const size_t dst = (kv_head * p.cap + (size_t)slot) * HD + d4 * 4;
        *reinterpret_cast<float4*>(p.ring_k + dst) = *reinterpret_cast<const float4*>(p.k_chunk + src);
        *reinterpret_cast<float4*>(p.ring_v + dst) = *reinterpret_cast<const float4*>(p.v_chunk + src);
      }
      if (g == 0 && tid == 0) p.meta_out[b] = advance_meta(p.meta[b], st, p.t);
    }
    return;
  }

  const size_t item = (((size_t)bg * p.n_rb + rb) * p.splits + s);
  float* wacc = p.ws_acc + item * (size_t)p.nq * HD;
  for (int idx = tid; idx < NQ * HD / 4; idx += kVCW * 32) {
    const int q = idx / (HD / 4), d4 = idx % (HD / 4);
    const int qg = q / C::QW, ql = q % C::QW;
    float M = -INFINITY;
#pragma unroll
    for (int kg = 0; kg < C::KG; ++kg) M = fmaxf(M, MLs[((qg + C::QG * kg) * C::QW + ql) * 2]);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int kg = 0; kg < C::KG; ++kg) {
        const int w = qg + C::QG * kg;
        const float mw = MLs[(w * C::QW + ql) * 2];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - M);
        const float4 a = *reinterpret_cast<const float4*>(red + ((size_t)w * C::QW + ql) * HD + d4 * 4);
        sum.x += a.x * f; sum.y += a.y * f; sum.z += a.z * f; sum.w += a.w * f;
      }
    }
    *reinterpret_cast<float4*>(wacc + (size_t)q * HD + d4 * 4) = sum;
  }
  if (tid < NQ) {
    const int qg = tid / C::QW, ql = tid % C::QW;
    float M = -INFINITY;
#pragma unroll
    for (int kg = 0; kg < C::KG; ++kg) M = fmaxf(M, MLs[((qg + C::QG * kg) * C::QW + ql) * 2]);
    float L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int kg = 0; kg < C::KG; ++kg) {
        const int w = qg + C::QG * kg;
        const float mw = MLs[(w * C::QW + ql) * 2];
        if (mw != -INFINITY) L += MLs[(w * C::QW + ql) * 2 + 1] * exp2f(mw - M);
      }
    }
    p.ws_ml[item * p.nq + tid] = make_float2(M, L);
  }
}

// The order of ordered verify blocks: (sequence, KV head, row block) units by key
// tile count, longest first, by one CTA of 256 threads.
__global__ void __launch_bounds__(256) order_verify_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  h16::order_units_h16(p.B * p.nk * p.n_rb, p.chunk / TK + 1, p.ws_order, [&](int u) {
    const SeqState st = sanitize_state(p.meta[u / p.n_rb / p.nk], p.cap, nullptr);
    const int r0 = (u % p.n_rb) * p.rows, r_last = min(r0 + p.rows, p.t) - 1;
    const int xlo = st.len0 + r0 + 1 - min(st.W, st.len0 + r0 + 1);
    return (p.ns + (st.len0 + r_last - xlo + 1) + TK - 1) / TK;
  });
}

template <int HD, int NQ>
int launch_v(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = VCfg<HD, NQ>;
  auto kern = attend_verify_kernel<HD, NQ>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  dim3 grid((unsigned)p.splits, (unsigned)p.n_rb, (unsigned)(p.B * p.nk));
  if (p.ws_order) {
    const int rc = finish_launch(launch_pdl(order_verify_kernel, dim3(1), dim3(256), 0, s, p));
    if (rc != SWA_OK) return rc;
    grid = dim3((unsigned)(p.B * p.nk * p.n_rb));
  }
  if (e0) cudaEventRecord(e0, s);
  cudaError_t e = launch_pdl(kern, grid, dim3(kVThreads), C::BYTES, s, p);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e1) cudaEventRecord(e1, s);
  return cuda_status(e);
}

template <int HD, int NQ>
int occ_v() {
  using C = VCfg<HD, NQ>;
  auto kern = attend_verify_kernel<HD, NQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES) != cudaSuccess)
    return 1;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kVThreads, C::BYTES) != cudaSuccess)
    return 1;
  return blocks > 0 ? blocks : 1;
}

}  // namespace

int launch_attend_verify(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  switch (p.hd * 100 + p.nq) {
    case 6416: return launch_v<64, 16>(p, s, e0, e1);
    case 6432: return launch_v<64, 32>(p, s, e0, e1);
    case 12816: return launch_v<128, 16>(p, s, e0, e1);
    case 12832: return launch_v<128, 32>(p, s, e0, e1);
    case 25616: return launch_v<256, 16>(p, s, e0, e1);
    case 25632: return launch_v<256, 32>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

int attend_verify_occupancy(int hd, int nq) {
  switch (hd * 100 + nq) {
    case 6416: return occ_v<64, 16>();
    case 6432: return occ_v<64, 32>();
    case 12816: return occ_v<128, 16>();
    case 12832: return occ_v<128, 32>();
    case 25616: return occ_v<256, 16>();
    case 25632: return occ_v<256, 32>();
  }
  return 1;
}

}  // namespace swa
