// Attention of a row block with 16 or 32 query vectors (speculative verify
// and other short chunks) on CUDA cores: o1c_score / o1c_soft / o1c_sum of
// "o1c_msl.metal" (cortiq-engine 0.8.79) for several rows at once, as one
// warp-specialised split-KV kernel writing the shared partial-record format.
//
// With 32 query vectors per key the path does 16 flops per K/V byte, so FP32
// FMA throughput, not HBM, bounds it. The layout is chosen to keep the FMA
// pipe fed:
//  - a producer warp streams 32-key tiles into shared memory (one
//    cp.async.bulk per K row into rows padded to hd + 4 floats, and per V row)
//    through full/empty mbarriers;
//  - consumer warp w owns query vectors [w * nq/4, (w + 1) * nq/4) and runs
//    their complete softmax rows over every key, so warps never combine
//    states and no CTA barrier runs in the key loop;
//  - scores: lane = key; each lane reads its K row (the padding puts the 8
//    lanes of a shared-memory phase on distinct banks) and the query rows by
//    broadcast, accumulating with packed fma.rn.f32x2 over feature pairs;
//  - P V: lane = a slice of hd/32 features; P goes through a per-warp shared
//    slice stored as (p, p) pairs so the packed FMA needs no shuffles.
#include "swa_internal.cuh"

namespace swa {
namespace {

constexpr int kVCW = 4;                        // consumer warps
constexpr int kVThreads = (kVCW + 1) * 32;     // + one producer warp
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

template <int HD, int NQ>
struct VCfg {
  static constexpr int KP = HD + 4;            // padded K row (floats)
  static constexpr int QW = NQ / kVCW;         // query vectors per consumer warp
  static constexpr int D4 = HD / 4;
  static constexpr int DPL = HD / 32;          // features per lane in P V (2, 4 or 8)
  static constexpr int STAGES = 2;
  static constexpr int OFF_K = 0;                              // [STAGES][TK][KP]
  static constexpr int OFF_V = STAGES * TK * KP;               // [STAGES][TK][HD]
  static constexpr int OFF_Q = OFF_V + STAGES * TK * HD;       // [NQ][HD]
  static constexpr int OFF_P = OFF_Q + NQ * HD;                // [kVCW][TK][QW] x (p, p)
  static constexpr int OFF_FLAG = OFF_P + kVCW * TK * QW * 2;
  static constexpr int FLOATS = ((OFF_FLAG + 4 + 1) / 2) * 2;
  static constexpr size_t BYTES = (size_t)FLOATS * 4 + 2 * STAGES * sizeof(uint64_t);
  static_assert(QW == 4 || QW == 8, "4 or 8 query vectors per warp");
};

template <int HD, int NQ>
__global__ void __launch_bounds__(kVThreads) attend_verify_kernel(AttendParams p) {
  using C = VCfg<HD, NQ>;
  extern __shared__ __align__(128) float smem[];
  float* Ks = smem + C::OFF_K;
  float* Vs = smem + C::OFF_V;
  float* Qs = smem + C::OFF_Q;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::FLOATS);
  uint64_t* empty = full + C::STAGES;

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x, rb = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.nk, g = bg % p.nk;

  const SeqState st = load_state(p, b, tid == 0 && g == 0 && rb == 0 && s == 0);
  const int r0 = rb * p.rows;
  const int r_last = min(r0 + p.rows, p.t) - 1;
  const int rows_eff = r_last - r0 + 1;
  const int win0 = min(st.W, st.len0 + r0 + 1);
  const int xlo = st.len0 + r0 + 1 - win0;
  const int n = p.ns + (st.len0 + r_last - xlo + 1);
  if (g == 0 && s == 0 && tid == 0) p.ws_nsplit[b * p.n_rb + rb] = (n + p.chunk - 1) / p.chunk;
  if (g == 0 && s == 0 && rb == 0 && tid == 0) p.ws_meta[b] = p.meta[b];
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
  for (int idx = tid; idx < NQ * C::D4; idx += kVThreads) {
    const int q = idx / C::D4, d4 = idx % C::D4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    const int rr = q / p.hpg, h = q % p.hpg;
    if (rr < rows_eff && q < p.rows * p.hpg) {
      v = *reinterpret_cast<const float4*>(
          p.q + (((size_t)b * p.t + r0 + rr) * p.nh + (size_t)g * p.hpg + h) * HD + d4 * 4);
      v.x *= p.qmul; v.y *= p.qmul; v.z *= p.qmul; v.w *= p.qmul;
    }
    *reinterpret_cast<float4*>(Qs + q * HD + d4 * 4) = v;
  }
  __syncthreads();
  const size_t kv_head = (size_t)b * p.nk + g;

  // ------------------------------------------------------------------ producer
  if (warp == kVCW) {
    int last = -1;
    for (int i = 0; i < ntiles; ++i) {
      const int stage = i % C::STAGES;
      const int use = i / C::STAGES;
      bool ok = use == 0 || mbar_wait_bounded(&empty[stage], (uint32_t)((use - 1) & 1), kWaitLimitNs);
      ok = __all_sync(kVFull, ok);
      if (!ok) {
        if (lane == 0) {
          *s_abort = 1;
          set_err(p.err, SWA_DERR_TIMEOUT);
        }
        break;
      }
      if (__shfl_sync(kVFull, *s_abort, 0)) break;
      fence_proxy_async_smem();
      const int j0 = jb + i * TK;
      const int cnt = min(TK, je - j0);
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)(cnt * HD * 4 * 2));
      __syncwarp();
      if (lane < cnt) {
        const int j = j0 + lane;
        const float* sk;
        const float* sv;
        if (j < p.ns) {
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
        bulk_g2s(Ks + ((size_t)stage * TK + lane) * C::KP, sk, HD * 4, &full[stage]);
        bulk_g2s(Vs + ((size_t)stage * TK + lane) * HD, sv, HD * 4, &full[stage]);
      }
      last = i;
    }
    for (int st_i = 0; st_i < C::STAGES && st_i <= last; ++st_i) {
      const int lt = last - ((last - st_i) % C::STAGES);
      mbar_wait_bounded(&full[st_i], (uint32_t)((lt / C::STAGES) & 1), kWaitLimitNs);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int q0 = warp * C::QW;                     // this warp's first query vector
  int q_lo[C::QW], q_hi[C::QW];
  bool q_ok[C::QW];
#pragma unroll
  for (int k = 0; k < C::QW; ++k) {
    const int q = q0 + k;
    const int rr = q / p.hpg;
    const int r = r0 + rr;
    q_ok[k] = rr < rows_eff && q < p.rows * p.hpg;
    q_lo[k] = st.len0 + r + 1 - min(st.W, st.len0 + r + 1);
    q_hi[k] = st.len0 + r;
  }
  float m[C::QW], l[C::QW];
  u64 acc[C::QW][C::DPL / 2];
#pragma unroll
  for (int k = 0; k < C::QW; ++k) {
    m[k] = -INFINITY;
    l[k] = 0.f;
#pragma unroll
    for (int d = 0; d < C::DPL / 2; ++d) acc[k][d] = 0ull;
  }
  u64* Pw = reinterpret_cast<u64*>(smem + C::OFF_P) + warp * TK * C::QW;
  const u64 zero2 = 0ull;

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
    if (__shfl_sync(kVFull, *s_abort, 0)) break;
    const int j0 = jb + i * TK;
    const int cnt = min(TK, je - j0);

    // ---- scores of key `lane` against the warp's query vectors
    // two independent accumulator chains per query vector (features 4i..4i+1
    // and 4i+2..4i+3) keep consecutive packed FMAs from waiting on each other
    u64 sacc[C::QW], sacc2[C::QW];
#pragma unroll
    for (int k = 0; k < C::QW; ++k) sacc[k] = sacc2[k] = 0ull;
    const float* krow = Ks + ((size_t)stage * TK + lane) * C::KP;
    const float* qrow = Qs + (size_t)q0 * HD;
#pragma unroll 8
    for (int d4 = 0; d4 < C::D4; ++d4) {
      const ulonglong2 kv = *reinterpret_cast<const ulonglong2*>(krow + d4 * 4);
#pragma unroll
      for (int k = 0; k < C::QW; ++k) {
        const ulonglong2 qv = *reinterpret_cast<const ulonglong2*>(qrow + k * HD + d4 * 4);
        sacc[k] = ffma2(qv.x, kv.x, sacc[k]);
        sacc2[k] = ffma2(qv.y, kv.y, sacc2[k]);
      }
    }
    const int j = j0 + lane;
    const bool key_in = lane < cnt;
    const int x = xlo + (j - p.ns);
    u64 cc[C::QW];
#pragma unroll
    for (int k = 0; k < C::QW; ++k) {
      const float2 sp = unpack2(sacc[k]);
      const float2 sp2 = unpack2(sacc2[k]);
      bool v = key_in && q_ok[k];
      if (v && j >= p.ns) v = x >= q_lo[k] && x <= q_hi[k];
      const float sv = v ? (sp.x + sp.y) + (sp2.x + sp2.y) : -INFINITY;
      float tmax = sv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kVFull, tmax, o));
      const float m_new = fmaxf(m[k], tmax);
      float c = 1.f, pv = 0.f;
      if (m_new != -INFINITY) {
        c = exp2f(m[k] - m_new);
        pv = exp2f(sv - m_new);
      }
      l[k] = l[k] * c + pv;
      m[k] = m_new;
      cc[k] = pack2(c, c);
      Pw[lane * C::QW + k] = pack2(pv, pv);
    }
    __syncwarp();

    // ---- P V: lane = features [lane * DPL, lane * DPL + DPL)
#pragma unroll
    for (int k = 0; k < C::QW; ++k)
#pragma unroll
      for (int d = 0; d < C::DPL / 2; ++d) acc[k][d] = ffma2(acc[k][d], cc[k], zero2);
#pragma unroll 4
    for (int kk = 0; kk < cnt; ++kk) {
      u64 pk[C::QW];
#pragma unroll
      for (int k2 = 0; k2 < C::QW / 2; ++k2) {
        const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(Pw + kk * C::QW + 2 * k2);
        pk[2 * k2] = a.x;
        pk[2 * k2 + 1] = a.y;
      }
      const float* vr = Vs + ((size_t)stage * TK + kk) * HD + lane * C::DPL;
      u64 vv[C::DPL / 2];
      if constexpr (C::DPL == 2) {
        vv[0] = *reinterpret_cast<const u64*>(vr);
      } else {
#pragma unroll
        for (int c4 = 0; c4 < C::DPL / 4; ++c4) {
          const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(vr + 4 * c4);
          vv[2 * c4] = a.x;
          vv[2 * c4 + 1] = a.y;
        }
      }
#pragma unroll
      for (int k = 0; k < C::QW; ++k)
#pragma unroll
        for (int d = 0; d < C::DPL / 2; ++d) acc[k][d] = ffma2(pk[k], vv[d], acc[k][d]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
  if (__shfl_sync(kVFull, *s_abort, 0)) return;

  // ---- this warp's query vectors of the partial record
  const size_t item = (((size_t)bg * p.n_rb + rb) * p.splits + s);
  float* wacc = p.ws_acc + item * (size_t)p.nq * HD;
#pragma unroll
  for (int k = 0; k < C::QW; ++k) {
    float lt = l[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(kVFull, lt, o);
    float* dst = wacc + (size_t)(q0 + k) * HD + lane * C::DPL;
#pragma unroll
    for (int d = 0; d < C::DPL / 2; ++d) *reinterpret_cast<float2*>(dst + 2 * d) = unpack2(acc[k][d]);
    if (lane == 0) p.ws_ml[item * p.nq + q0 + k] = make_float2(m[k], lt);
  }
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
  if (e0) cudaEventRecord(e0, s);
  kern<<<grid, kVThreads, C::BYTES, s>>>(p);
  note_launch();
  cudaError_t e = cudaGetLastError();
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
