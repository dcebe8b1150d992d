// Attention of a row block with at most 8 query vectors (decode tokens and
// short chunks): the near window of "o1c_msl.metal" (cortiq-engine 0.8.79),
// o1c_tok_near and o1c_score / o1c_soft / o1c_sum, as one warp-specialised
// split-KV kernel. It writes the same partial records as the block kernel in
// swa_attend.cu, which the merge kernel there reduces.
//
// One CTA per (sequence, KV head, row block, split) with 4 consumer warps and
// 1 producer warp:
//  - the producer streams the split's keys through STAGES shared-memory tiles
//    of 32 key rows. Keys whose sources are contiguous (a run of ring slots up
//    to the wrap, the sinks) travel as ONE cp.async.bulk per run for K and one
//    for V, landing in consecutive (unpadded) rows: copies of 4-16 KB stream at
//    the HBM read rate, where one 512-byte copy per row saturates the copy
//    engine's per-request cost far below it. A tile completes on its `full`
//    barrier and is refilled when the 4 consumer warps arrive on its `empty`
//    barrier;
//  - consumer warp w owns keys [8w, 8w + 8) of every tile and keeps its own
//    online softmax (max, sum, numerator) for all query vectors of the block,
//    so no CTA-wide barrier runs inside the key loop. Scores: lane (kq, e) =
//    (lane / 8, lane % 8) takes key kq of a group of 4 and the float4 chunks
//    e, e + 8, ... of the features, so each 8-lane shared-memory phase reads
//    one contiguous 128-byte segment of a row (conflict-free without padding);
//    transposed shuffles over the 8 chunk lanes leave each lane with the full
//    score of one query vector. P goes through a per-warp shared slice and P V
//    runs with lane = a slice of hd/32 features.
// At the end the 4 warps' states are combined (max, rescaled sums) into the
// CTA's partial record.
#include "swa_internal.cuh"

namespace swa {
namespace {

constexpr int kCW = 4;                         // consumer warps
constexpr int kDecThreads = (kCW + 1) * 32;    // + one producer warp
constexpr int kKPW = TK / kCW;                 // keys per consumer warp per tile (8)
constexpr unsigned kFull = 0xffffffffu;

template <int HD, int NQ>
struct DCfg {
  static constexpr int CH = HD / 32;           // float4 chunks per lane in the scores (stride 8)
  static constexpr int DPL = HD / 32;          // features per lane in P V
  static constexpr int STAGES = HD == 64 ? 6 : (HD == 128 ? 3 : 2);
  static constexpr int OFF_K = 0;                          // [STAGES][TK][HD]
  static constexpr int OFF_V = STAGES * TK * HD;           // [STAGES][TK][HD]
  static constexpr int OFF_Q = 2 * STAGES * TK * HD;       // [NQ][HD]
  static constexpr int OFF_P = OFF_Q + NQ * HD;            // [kCW][kKPW][NQ]
  static constexpr int OFF_ML = OFF_P + kCW * kKPW * NQ;   // [kCW][NQ] x (m, l)
  static constexpr int OFF_FLAG = OFF_ML + kCW * NQ * 2;   // abort flag
  static constexpr int FLOATS = ((OFF_FLAG + 4 + 1) / 2) * 2;
  static constexpr size_t BYTES = (size_t)FLOATS * 4 + 2 * STAGES * sizeof(uint64_t);
  // one-launch decode step only, after the barriers (the attention-only kernel
  // does not allocate them): the row's cos | sin, its own k-hat and v rows, the
  // gate rows and gate scales of the KV head's query heads, then the barrier of
  // the gate copies
  static constexpr int OFF_STEP = (FLOATS + 4 * STAGES + 3) / 4 * 4;
  static constexpr int STEP_FLOATS = (3 + 2 * NQ) * HD;
  static constexpr size_t STEP_BYTES = (size_t)(OFF_STEP + STEP_FLOATS) * sizeof(float) + sizeof(uint64_t);
  static_assert(NQ == 4 || NQ == 8, "decode kernel serves 4 or 8 query vectors");
  static_assert(kCW * NQ * HD <= 2 * STAGES * TK * HD, "warp states fit the stage buffers");
  static_assert(DPL == 2 || DPL % 4 == 0, "feature slice per lane");
};

template <int DPL>
__device__ __forceinline__ void load_slice(const float* row, int lane, float (&v)[DPL]) {
  if constexpr (DPL == 2) {
    const float2 a = *reinterpret_cast<const float2*>(row + lane * 2);
    v[0] = a.x; v[1] = a.y;
  } else {
#pragma unroll
    for (int c = 0; c < DPL / 4; ++c) {
      const float4 a = *reinterpret_cast<const float4*>(row + (lane + 32 * c) * 4);
      v[4 * c + 0] = a.x; v[4 * c + 1] = a.y; v[4 * c + 2] = a.z; v[4 * c + 3] = a.w;
    }
  }
}

template <int DPL>
__device__ __forceinline__ void store_slice(float* row, int lane, const float (&v)[DPL]) {
  if constexpr (DPL == 2) {
    *reinterpret_cast<float2*>(row + lane * 2) = make_float2(v[0], v[1]);
  } else {
#pragma unroll
    for (int c = 0; c < DPL / 4; ++c)
      *reinterpret_cast<float4*>(row + (lane + 32 * c) * 4) =
          make_float4(v[4 * c + 0], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  }
}

template <int HD, int NQ>
__global__ void __launch_bounds__(kDecThreads) attend_decode_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  using C = DCfg<HD, NQ>;
  extern __shared__ __align__(128) float smem[];
  float* Ks = smem + C::OFF_K;
  float* Vs = smem + C::OFF_V;
  float* Qs = smem + C::OFF_Q;
  float* Ps = smem + C::OFF_P;
  float* MLs = smem + C::OFF_ML;
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
  const int xlo = st.len0 + r0 + 1 - win0;       // first logical key of the block
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
      mbar_init(&empty[i], kCW);
    }
    mbar_fence_init();
    *s_abort = 0;
  }
  // Query vectors of the block (row-major: rows then heads), times scale * log2 e.
  for (int idx = tid; idx < NQ * (HD / 4); idx += kDecThreads) {
    const int q = idx / (HD / 4), d4 = idx % (HD / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    const int rr = q / p.hpg, h = q % p.hpg;
    if (rr < rows_eff) {
      v = *reinterpret_cast<const float4*>(
          p.q + (((size_t)b * p.t + r0 + rr) * p.nh + (size_t)g * p.hpg + h) * HD + d4 * 4);
      v.x *= p.qmul; v.y *= p.qmul; v.z *= p.qmul; v.w *= p.qmul;
    }
    *reinterpret_cast<float4*>(Qs + q * HD + d4 * 4) = v;
  }
  __syncthreads();

  const size_t kv_head = (size_t)b * p.nk + g;

  // ------------------------------------------------------------------ producer
  if (warp == kCW) {
    int last = -1;
    for (int i = 0; i < ntiles; ++i) {
      const int stage = i % C::STAGES;
      const int use = i / C::STAGES;
      bool ok = use == 0 || mbar_wait_bounded(&empty[stage], (uint32_t)((use - 1) & 1), kWaitLimitNs);
      ok = __all_sync(kFull, ok);                 // one decision per warp
      if (!ok) {
        if (lane == 0) {
          *s_abort = 1;
          set_err(p.err, SWA_DERR_TIMEOUT);
        }
        break;
      }
      if (__shfl_sync(kFull, *s_abort, 0)) break;
      fence_proxy_async_smem();
      const int j0 = jb + i * TK;
      const int cnt = min(TK, je - j0);
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)(cnt * HD * 4 * 2));
      __syncwarp();
      // Source row of key `lane`; a lane whose row does not follow its left
      // neighbour's starts a run, and issues one copy of the whole run.
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
      const unsigned long long prev_k =
          __shfl_up_sync(kFull, reinterpret_cast<unsigned long long>(sk), 1);
      const unsigned long long prev_v =
          __shfl_up_sync(kFull, reinterpret_cast<unsigned long long>(sv), 1);
      const bool start = lane < cnt &&
                         (lane == 0 ||
                          reinterpret_cast<unsigned long long>(sk) != prev_k + HD * 4 ||
                          reinterpret_cast<unsigned long long>(sv) != prev_v + HD * 4);
      const unsigned starts = __ballot_sync(kFull, start);
      if (start) {
        const unsigned later = starts & ~((2u << lane) - 1u);   // run starts after this lane
        const int end = later ? __ffs(later) - 1 : cnt;
        const uint32_t bytes = (uint32_t)((end - lane) * HD * 4);
        bulk_g2s(Ks + ((size_t)stage * TK + lane) * HD, sk, bytes, &full[stage]);
        bulk_g2s(Vs + ((size_t)stage * TK + lane) * HD, sv, bytes, &full[stage]);
      }
      last = i;
    }
    // No copy may still be landing in shared memory when the CTA ends: wait
    // (bounded) for the last tile issued into every stage.
    for (int st_i = 0; st_i < C::STAGES && st_i <= last; ++st_i) {
      const int lt = last - ((last - st_i) % C::STAGES);
      mbar_wait_bounded(&full[st_i], (uint32_t)((lt / C::STAGES) & 1), kWaitLimitNs);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int e = lane & 7, kq = lane >> 3;
  // after the reduction lane (kq, e) holds query vector ql (NQ = 8: e; NQ = 4: e / 2)
  const int ql = NQ == 8 ? e : (e >> 1);
  const int q_rr = ql / p.hpg;
  const bool q_ok = q_rr < rows_eff;
  const int q_r = r0 + q_rr;
  const int q_lo = st.len0 + q_r + 1 - min(st.W, st.len0 + q_r + 1);
  const int q_hi = st.len0 + q_r;
  float m = -INFINITY, l = 0.f;
  float acc[NQ][C::DPL];
#pragma unroll
  for (int q = 0; q < NQ; ++q)
#pragma unroll
    for (int d = 0; d < C::DPL; ++d) acc[q][d] = 0.f;

  float* Pw = Ps + warp * kKPW * NQ;
  for (int i = 0; i < ntiles; ++i) {
    const int stage = i % C::STAGES;
    const bool ok = __all_sync(kFull, mbar_wait_bounded(&full[stage], (uint32_t)((i / C::STAGES) & 1),
                                                      kWaitLimitNs));
    if (!ok) {
      if (lane == 0) {
        *s_abort = 1;
        set_err(p.err, SWA_DERR_TIMEOUT);
      }
      break;
    }
    if (__shfl_sync(kFull, *s_abort, 0)) break;
    const int j0 = jb + i * TK;
    const int cnt = min(TK, je - j0);

    // ---- scores of the warp's 8 keys, two groups of 4 (key kq of each group)
    float sc[2];
#pragma unroll
    for (int rd = 0; rd < 2; ++rd) {
      const int kl = warp * kKPW + rd * 4 + kq;
      float sp[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) sp[q] = 0.f;
      const float* krow = Ks + ((size_t)stage * TK + kl) * HD;
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        const int off = (e + 8 * c) * 4;
        const float4 kv = *reinterpret_cast<const float4*>(krow + off);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const float4 qv = *reinterpret_cast<const float4*>(Qs + q * HD + off);
          sp[q] += qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
        }
      }
      // transposed reduction over the 8 chunk lanes (lane bits 2, 1, 0)
      float t4[NQ / 2];
      const bool b2 = (e & 4) != 0, b1 = (e & 2) != 0, b0 = (e & 1) != 0;
#pragma unroll
      for (int k = 0; k < NQ / 2; ++k) {
        const float send = b2 ? sp[k] : sp[NQ / 2 + k];
        const float keep = b2 ? sp[NQ / 2 + k] : sp[k];
        t4[k] = keep + __shfl_xor_sync(kFull, send, 4);
      }
      float t2[NQ / 4];
#pragma unroll
      for (int k = 0; k < NQ / 4; ++k) {
        const float send = b1 ? t4[k] : t4[NQ / 4 + k];
        const float keep = b1 ? t4[NQ / 4 + k] : t4[k];
        t2[k] = keep + __shfl_xor_sync(kFull, send, 2);
      }
      float full_s;
      if constexpr (NQ == 8) {
        const float send = b0 ? t2[0] : t2[1];
        const float keep = b0 ? t2[1] : t2[0];
        full_s = keep + __shfl_xor_sync(kFull, send, 1);
      } else {
        full_s = t2[0] + __shfl_xor_sync(kFull, t2[0], 1);
      }
      const int j = j0 + kl;
      bool v = kl < cnt && q_ok;
      if (v && j >= p.ns) {
        const int x = xlo + (j - p.ns);
        v = x >= q_lo && x <= q_hi;
      }
      sc[rd] = v ? full_s : -INFINITY;
    }
    // ---- tile max of query ql over the warp's 8 keys, online update
    float tmax = fmaxf(sc[0], sc[1]);
    tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
    tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
    const float m_new = fmaxf(m, tmax);
    float c = 1.f, p0 = 0.f, p1 = 0.f;
    if (m_new != -INFINITY) {
      c = exp2f(m - m_new);
      p0 = exp2f(sc[0] - m_new);
      p1 = exp2f(sc[1] - m_new);
    }
    l = l * c + p0 + p1;
    m = m_new;
    if (NQ == 8 || (e & 1) == 0) {
      Pw[kq * NQ + ql] = p0;
      Pw[(4 + kq) * NQ + ql] = p1;
    }
    float call[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) call[q] = __shfl_sync(kFull, c, NQ == 8 ? q : 2 * q);
    __syncwarp();

    // ---- P V over the warp's keys, lane = feature slice
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
      for (int d = 0; d < C::DPL; ++d) acc[q][d] *= call[q];
    const int nk = min(kKPW, cnt - warp * kKPW);
#pragma unroll
    for (int kk = 0; kk < kKPW; ++kk) {
      if (kk < nk) {
        float pk[NQ];
#pragma unroll
        for (int q4 = 0; q4 < NQ / 4; ++q4) {
          const float4 a = *reinterpret_cast<const float4*>(Pw + kk * NQ + q4 * 4);
          pk[q4 * 4 + 0] = a.x; pk[q4 * 4 + 1] = a.y; pk[q4 * 4 + 2] = a.z; pk[q4 * 4 + 3] = a.w;
        }
        float v[C::DPL];
        load_slice<C::DPL>(Vs + ((size_t)stage * TK + warp * kKPW + kk) * HD, lane, v);
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
          for (int d = 0; d < C::DPL; ++d) acc[q][d] += pk[q] * v[d];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  // ---- combine the 4 warps' states into the CTA's partial record
  l += __shfl_xor_sync(kFull, l, 8);
  l += __shfl_xor_sync(kFull, l, 16);
  named_barrier(1, kCW * 32);                  // every consumer is past its last tile
  if (*s_abort) return;
  if (kq == 0 && (NQ == 8 || (e & 1) == 0)) {
    MLs[(warp * NQ + ql) * 2 + 0] = m;
    MLs[(warp * NQ + ql) * 2 + 1] = l;
  }
  float* red = smem;                              // [kCW][NQ][HD], reuses the stage buffers
#pragma unroll
  for (int q = 0; q < NQ; ++q) store_slice<C::DPL>(red + ((size_t)warp * NQ + q) * HD, lane, acc[q]);
  named_barrier(1, kCW * 32);

  const size_t item = (((size_t)bg * p.n_rb + rb) * p.splits + s);
  float* wacc = p.ws_acc + item * (size_t)p.nq * HD;
  for (int idx = tid; idx < NQ * HD / 4; idx += kCW * 32) {
    const int q = idx / (HD / 4);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) M = fmaxf(M, MLs[(w * NQ + q) * 2]);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float mw = MLs[(w * NQ + q) * 2];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - M);
        const float4 a = *reinterpret_cast<const float4*>(red + ((size_t)w * NQ) * HD + (size_t)idx * 4);
        sum.x += a.x * f; sum.y += a.y * f; sum.z += a.z * f; sum.w += a.w * f;
      }
    }
    *reinterpret_cast<float4*>(wacc + (size_t)idx * 4) = sum;
  }
  if (tid < NQ) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) M = fmaxf(M, MLs[(w * NQ + tid) * 2]);
    float L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float mw = MLs[(w * NQ + tid) * 2];
        if (mw != -INFINITY) L += MLs[(w * NQ + tid) * 2 + 1] * exp2f(mw - M);
      }
    }
    p.ws_ml[item * p.nq + tid] = make_float2(M, L);
  }
}

// The prep inputs a one-launch decode step folds into the attention.
struct StepExtra {
  const float* yq;            // [B][nh][hd]
  const float* yk;            // [B][nk][hd]
  const float* yv;            // [B][nk][hd]
  const float* q_scale;       // [nh][hd]
  const uint32_t* pos0;       // [B]
  float eps;
  double inv_freq[128];       // theta^(-2e/hd)
};

// A whole decode step of one row (t = 1) in one launch, for calls whose plan
// has one split per (sequence, KV head), on the structure of the attention
// kernel above: the CTA of (sequence, KV head) first preps the
// row's query heads of that KV head and its own k and v head ("dory_msl.metal"
// dory_prep; angles from pos0 in f64, as the prep kernel), attends the window
// with its own row taken from shared memory instead of a copy, writes the
// gated output itself (dory_gate) and commits its k-hat / v row into the ring
// slot (win_head + win_len) % W and, for KV head 0, the advanced meta
// (o1c_ring_commit, o1c_meta). That slot never holds a key of the row's window
// (it is the evicted key's, or past the last key of a ring not yet full), so
// the write races with no read.
template <int HD, int NQ>
__device__ __forceinline__ void step_body(const AttendParams& p, const StepExtra* x) {
  using C = DCfg<HD, NQ>;
  extern __shared__ __align__(128) float smem[];
  float* Ks = smem + C::OFF_K;
  float* Vs = smem + C::OFF_V;
  float* Qs = smem + C::OFF_Q;
  float* Ps = smem + C::OFF_P;
  float* MLs = smem + C::OFF_ML;
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
  const int xlo = st.len0 + r0 + 1 - win0;       // first logical key of the block
  const int n = p.ns + (st.len0 + r_last - xlo + 1);
  const int jb = s * p.chunk;
  if (jb >= n) return;
  const int je = min(n, jb + p.chunk);
  const int ntiles = (je - jb + TK - 1) / TK;
  // the step's own row: the last key (logical key len0), held in shared memory
  float* s_cs = smem + C::OFF_STEP;               // [HD] cos | sin
  float* own_k = s_cs + HD;                       // [HD]
  float* own_v = own_k + HD;                      // [HD]
  float* s_gate = own_v + HD;                     // [hpg][HD] gate rows
  float* s_gs = s_gate + NQ * HD;                 // [hpg][HD] gate scales
  uint64_t* gbar = reinterpret_cast<uint64_t*>(smem + C::OFF_STEP + C::STEP_FLOATS);

  if (tid == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    mbar_init(gbar, 1);
    mbar_fence_init();
    *s_abort = 0;
  }
  // The producer starts the ring copies (and the gate's) at once; the
  // consumer warps prep the row meanwhile (t = 1): each warp requests the
  // inputs of its heads, the angles are evaluated once (f64, as the prep
  // kernel), then query heads g*hpg .. g*hpg + hpg - 1 go to Qs (q-hat, then
  // times scale * log2 e, as the attention reads the prep's output), k head
  // g to own_k and its v row to own_v.
  __syncthreads();
  if (warp < kCW) {
    constexpr int P = HD / 64;
    constexpr int HALF = HD / 2;
    constexpr int HEADS = (NQ + 1 + kCW - 1) / kCW;   // heads per consumer warp, at most
    const int e = lane * P;
    float xv[HEADS][P], yv[HEADS][P], sa[HEADS][P], sb[HEADS][P];
#pragma unroll
    for (int k = 0; k < HEADS; ++k) {
      const int a = warp + k * kCW;
      if (a > p.hpg) continue;
      const bool is_q = a < p.hpg;
      const float* src = is_q ? x->yq + ((size_t)b * p.nh + (size_t)g * p.hpg + a) * HD
                              : x->yk + ((size_t)b * p.nk + g) * HD;
      const float* ext = is_q ? x->q_scale + ((size_t)g * p.hpg + a) * HD
                              : x->yv + ((size_t)b * p.nk + g) * HD;
#pragma unroll
      for (int i = 0; i < P; ++i) {
        xv[k][i] = src[e + i];
        yv[k][i] = src[HALF + e + i];
        sa[k][i] = ext[e + i];
        sb[k][i] = ext[HALF + e + i];
      }
    }
    const uint64_t pos = (uint64_t)x->pos0[b];
    for (int e2 = tid; e2 < HALF; e2 += kCW * 32) {
      double sn, cs;
      sincos((double)pos * x->inv_freq[e2], &sn, &cs);
      s_cs[e2] = (float)cs;
      s_cs[HALF + e2] = (float)sn;
    }
    for (int idx = tid; idx < (NQ - p.hpg) * (HD / 4); idx += kCW * 32)
      *reinterpret_cast<float4*>(Qs + p.hpg * HD + idx * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
    named_barrier(2, kCW * 32);
    float c[P], sn[P];
#pragma unroll
    for (int i = 0; i < P; ++i) {
      c[i] = s_cs[e + i];
      sn[i] = s_cs[HALF + e + i];
    }
#pragma unroll
    for (int k = 0; k < HEADS; ++k) {
      const int a = warp + k * kCW;
      if (a > p.hpg) continue;
      float u[P], v[P];
      const float inv = rotate_unit<P>(xv[k], yv[k], c, sn, x->eps, u, v);
      if (a < p.hpg) {
#pragma unroll
        for (int i = 0; i < P; ++i) {
          const float qa = u[i] * inv * sa[k][i];
          const float qb = v[i] * inv * sb[k][i];
          Qs[a * HD + e + i] = qa * p.qmul;
          Qs[a * HD + HALF + e + i] = qb * p.qmul;
        }
      } else {
#pragma unroll
        for (int i = 0; i < P; ++i) {
          own_k[e + i] = u[i] * inv;
          own_k[HALF + e + i] = v[i] * inv;
          own_v[e + i] = sa[k][i];
          own_v[HALF + e + i] = sb[k][i];
        }
      }
    }
    named_barrier(2, kCW * 32);
  }

  const size_t kv_head = (size_t)b * p.nk + g;

  // ------------------------------------------------------------------ producer
  if (warp == kCW) {
    // the gate rows and gate scales of the KV head's query heads (contiguous)
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)(p.hpg * HD * 4);
      mbar_arrive_expect_tx(gbar, 2 * bytes);
      bulk_g2s(s_gate, p.gate + ((size_t)b * p.nh + (size_t)g * p.hpg) * HD, bytes, gbar);
      bulk_g2s(s_gs, p.gate_scale + (size_t)g * p.hpg * HD, bytes, gbar);
    }
    __syncwarp();
    int last = -1;
    for (int i = 0; i < ntiles; ++i) {
      const int stage = i % C::STAGES;
      const int use = i / C::STAGES;
      bool ok = use == 0 || mbar_wait_bounded(&empty[stage], (uint32_t)((use - 1) & 1), kWaitLimitNs);
      ok = __all_sync(kFull, ok);                 // one decision per warp
      if (!ok) {
        if (lane == 0) {
          *s_abort = 1;
          set_err(p.err, SWA_DERR_TIMEOUT);
        }
        break;
      }
      if (__shfl_sync(kFull, *s_abort, 0)) break;
      fence_proxy_async_smem();
      const int j0 = jb + i * TK;
      // a step's last key (its own row) stays in shared memory: not copied
      const int cnt = min(TK, je - j0) - (j0 + TK >= n ? 1 : 0);
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)(cnt * HD * 4 * 2));
      __syncwarp();
      // Source row of key `lane`; a lane whose row does not follow its left
      // neighbour's starts a run, and issues one copy of the whole run.
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
      const unsigned long long prev_k =
          __shfl_up_sync(kFull, reinterpret_cast<unsigned long long>(sk), 1);
      const unsigned long long prev_v =
          __shfl_up_sync(kFull, reinterpret_cast<unsigned long long>(sv), 1);
      const bool start = lane < cnt &&
                         (lane == 0 ||
                          reinterpret_cast<unsigned long long>(sk) != prev_k + HD * 4 ||
                          reinterpret_cast<unsigned long long>(sv) != prev_v + HD * 4);
      const unsigned starts = __ballot_sync(kFull, start);
      if (start) {
        const unsigned later = starts & ~((2u << lane) - 1u);   // run starts after this lane
        const int end = later ? __ffs(later) - 1 : cnt;
        const uint32_t bytes = (uint32_t)((end - lane) * HD * 4);
        bulk_g2s(Ks + ((size_t)stage * TK + lane) * HD, sk, bytes, &full[stage]);
        bulk_g2s(Vs + ((size_t)stage * TK + lane) * HD, sv, bytes, &full[stage]);
      }
      last = i;
    }
    // No copy may still be landing in shared memory when the CTA ends: wait
    // (bounded) for the last tile issued into every stage.
    for (int st_i = 0; st_i < C::STAGES && st_i <= last; ++st_i) {
      const int lt = last - ((last - st_i) % C::STAGES);
      mbar_wait_bounded(&full[st_i], (uint32_t)((lt / C::STAGES) & 1), kWaitLimitNs);
    }
    mbar_wait_bounded(gbar, 0, kWaitLimitNs);
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int e = lane & 7, kq = lane >> 3;
  // after the reduction lane (kq, e) holds query vector ql (NQ = 8: e; NQ = 4: e / 2)
  const int ql = NQ == 8 ? e : (e >> 1);
  const int q_rr = ql / p.hpg;
  const bool q_ok = q_rr < rows_eff;
  const int q_r = r0 + q_rr;
  const int q_lo = st.len0 + q_r + 1 - min(st.W, st.len0 + q_r + 1);
  const int q_hi = st.len0 + q_r;
  float m = -INFINITY, l = 0.f;
  float acc[NQ][C::DPL];
#pragma unroll
  for (int q = 0; q < NQ; ++q)
#pragma unroll
    for (int d = 0; d < C::DPL; ++d) acc[q][d] = 0.f;

  float* Pw = Ps + warp * kKPW * NQ;
  for (int i = 0; i < ntiles; ++i) {
    const int stage = i % C::STAGES;
    const bool ok = __all_sync(kFull, mbar_wait_bounded(&full[stage], (uint32_t)((i / C::STAGES) & 1),
                                                      kWaitLimitNs));
    if (!ok) {
      if (lane == 0) {
        *s_abort = 1;
        set_err(p.err, SWA_DERR_TIMEOUT);
      }
      break;
    }
    if (__shfl_sync(kFull, *s_abort, 0)) break;
    const int j0 = jb + i * TK;
    const int cnt = min(TK, je - j0);

    // ---- scores of the warp's 8 keys, two groups of 4 (key kq of each group)
    float sc[2];
#pragma unroll
    for (int rd = 0; rd < 2; ++rd) {
      const int kl = warp * kKPW + rd * 4 + kq;
      float sp[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) sp[q] = 0.f;
      const float* krow = j0 + kl == n - 1 ? own_k : Ks + ((size_t)stage * TK + kl) * HD;
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        const int off = (e + 8 * c) * 4;
        const float4 kv = *reinterpret_cast<const float4*>(krow + off);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const float4 qv = *reinterpret_cast<const float4*>(Qs + q * HD + off);
          sp[q] += qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
        }
      }
      // transposed reduction over the 8 chunk lanes (lane bits 2, 1, 0)
      float t4[NQ / 2];
      const bool b2 = (e & 4) != 0, b1 = (e & 2) != 0, b0 = (e & 1) != 0;
#pragma unroll
      for (int k = 0; k < NQ / 2; ++k) {
        const float send = b2 ? sp[k] : sp[NQ / 2 + k];
        const float keep = b2 ? sp[NQ / 2 + k] : sp[k];
        t4[k] = keep + __shfl_xor_sync(kFull, send, 4);
      }
      float t2[NQ / 4];
#pragma unroll
      for (int k = 0; k < NQ / 4; ++k) {
        const float send = b1 ? t4[k] : t4[NQ / 4 + k];
        const float keep = b1 ? t4[NQ / 4 + k] : t4[k];
        t2[k] = keep + __shfl_xor_sync(kFull, send, 2);
      }
      float full_s;
      if constexpr (NQ == 8) {
        const float send = b0 ? t2[0] : t2[1];
        const float keep = b0 ? t2[1] : t2[0];
        full_s = keep + __shfl_xor_sync(kFull, send, 1);
      } else {
        full_s = t2[0] + __shfl_xor_sync(kFull, t2[0], 1);
      }
      const int j = j0 + kl;
      bool v = kl < cnt && q_ok;
      if (v && j >= p.ns) {
        const int x = xlo + (j - p.ns);
        v = x >= q_lo && x <= q_hi;
      }
      sc[rd] = v ? full_s : -INFINITY;
    }
    // ---- tile max of query ql over the warp's 8 keys, online update
    float tmax = fmaxf(sc[0], sc[1]);
    tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
    tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
    const float m_new = fmaxf(m, tmax);
    float c = 1.f, p0 = 0.f, p1 = 0.f;
    if (m_new != -INFINITY) {
      c = exp2f(m - m_new);
      p0 = exp2f(sc[0] - m_new);
      p1 = exp2f(sc[1] - m_new);
    }
    l = l * c + p0 + p1;
    m = m_new;
    if (NQ == 8 || (e & 1) == 0) {
      Pw[kq * NQ + ql] = p0;
      Pw[(4 + kq) * NQ + ql] = p1;
    }
    float call[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) call[q] = __shfl_sync(kFull, c, NQ == 8 ? q : 2 * q);
    __syncwarp();

    // ---- P V over the warp's keys, lane = feature slice
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
      for (int d = 0; d < C::DPL; ++d) acc[q][d] *= call[q];
    const int nk = min(kKPW, cnt - warp * kKPW);
#pragma unroll
    for (int kk = 0; kk < kKPW; ++kk) {
      if (kk < nk) {
        float pk[NQ];
#pragma unroll
        for (int q4 = 0; q4 < NQ / 4; ++q4) {
          const float4 a = *reinterpret_cast<const float4*>(Pw + kk * NQ + q4 * 4);
          pk[q4 * 4 + 0] = a.x; pk[q4 * 4 + 1] = a.y; pk[q4 * 4 + 2] = a.z; pk[q4 * 4 + 3] = a.w;
        }
        float v[C::DPL];
        const int kv_l = warp * kKPW + kk;
        load_slice<C::DPL>(j0 + kv_l == n - 1 ? own_v : Vs + ((size_t)stage * TK + kv_l) * HD,
                           lane, v);
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
          for (int d = 0; d < C::DPL; ++d) acc[q][d] += pk[q] * v[d];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  // ---- combine the 4 warps' states into the CTA's partial record
  l += __shfl_xor_sync(kFull, l, 8);
  l += __shfl_xor_sync(kFull, l, 16);
  named_barrier(1, kCW * 32);                  // every consumer is past its last tile
  if (*s_abort) return;
  if (kq == 0 && (NQ == 8 || (e & 1) == 0)) {
    MLs[(warp * NQ + ql) * 2 + 0] = m;
    MLs[(warp * NQ + ql) * 2 + 1] = l;
  }
  float* red = smem;                              // [kCW][NQ][HD], reuses the stage buffers
#pragma unroll
  for (int q = 0; q < NQ; ++q) store_slice<C::DPL>(red + ((size_t)warp * NQ + q) * HD, lane, acc[q]);
  named_barrier(1, kCW * 32);

  // ---- gated output of the row's query heads (the merge's arithmetic for a
  // single split), then the commit
  if (!__all_sync(kFull, mbar_wait_bounded(gbar, 0, kWaitLimitNs))) {
    if (lane == 0) set_err(p.err, SWA_DERR_TIMEOUT);
    return;
  }
  for (int idx = tid; idx < p.hpg * (HD / 4); idx += kCW * 32) {
    const int q = idx / (HD / 4), d4 = idx % (HD / 4);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) M = fmaxf(M, MLs[(w * NQ + q) * 2]);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) {
      const float mw = MLs[(w * NQ + q) * 2];
      if (mw == -INFINITY) continue;
      const float f = exp2f(mw - M);
      const float4 a = *reinterpret_cast<const float4*>(red + ((size_t)w * NQ) * HD + (size_t)idx * 4);
      sum.x += a.x * f; sum.y += a.y * f; sum.z += a.z * f; sum.w += a.w * f;
      L += MLs[(w * NQ + q) * 2 + 1] * f;
    }
    const int h = g * p.hpg + q;
    const size_t row = (size_t)b * p.nh + h;
    const float4 gt = *reinterpret_cast<const float4*>(s_gate + q * HD + d4 * 4);
    const float4 gs = *reinterpret_cast<const float4*>(s_gs + q * HD + d4 * 4);
    const float inv = 1.0f / L;
    float4 o;
    o.x = gated(sum.x, inv, gt.x, gs.x);
    o.y = gated(sum.y, inv, gt.y, gs.y);
    o.z = gated(sum.z, inv, gt.z, gs.z);
    o.w = gated(sum.w, inv, gt.w, gs.w);
    *reinterpret_cast<float4*>(p.out + row * HD + d4 * 4) = o;
  }
  const int slot = (int)(((long long)st.head0 + st.len0) % st.W);
  const size_t dst = (((size_t)b * p.nk + g) * p.cap + slot) * HD;
  for (int d4 = tid; d4 < HD / 4; d4 += kCW * 32) {
    *reinterpret_cast<float4*>(p.ring_k + dst + d4 * 4) = *reinterpret_cast<const float4*>(own_k + d4 * 4);
    *reinterpret_cast<float4*>(p.ring_v + dst + d4 * 4) = *reinterpret_cast<const float4*>(own_v + d4 * 4);
  }
  if (g == 0 && tid == 0) p.meta_out[b] = advance_meta(p.meta[b], st, 1);
}

template <int HD, int NQ>
__global__ void __launch_bounds__(kDecThreads) decode_step_kernel(AttendParams p, StepExtra x) {
  pdl_trigger();
  pdl_wait();
  step_body<HD, NQ>(p, &x);
}

template <int HD, int NQ>
int launch_step(const AttendParams& p, const StepExtra& x, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = DCfg<HD, NQ>;
  auto kern = decode_step_kernel<HD, NQ>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::STEP_BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  dim3 grid(1u, 1u, (unsigned)(p.B * p.nk));
  if (e0) cudaEventRecord(e0, s);
  cudaError_t e = launch_pdl(kern, grid, dim3(kDecThreads), C::STEP_BYTES, s, p, x);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e1) cudaEventRecord(e1, s);
  return cuda_status(e);
}

template <int HD, int NQ>
int launch_t(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = DCfg<HD, NQ>;
  auto kern = attend_decode_kernel<HD, NQ>;
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
  cudaError_t e = launch_pdl(kern, grid, dim3(kDecThreads), C::BYTES, s, p);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e1) cudaEventRecord(e1, s);
  return cuda_status(e);
}

template <int HD, int NQ>
int occ_t() {
  using C = DCfg<HD, NQ>;
  auto kern = attend_decode_kernel<HD, NQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES) != cudaSuccess)
    return 1;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kDecThreads, C::BYTES) != cudaSuccess)
    return 1;
  return blocks > 0 ? blocks : 1;
}

}  // namespace

int launch_attend_decode(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  const int key = p.hd * 100 + p.nq;
  switch (key) {
    case 6404: return launch_t<64, 4>(p, s, e0, e1);
    case 6408: return launch_t<64, 8>(p, s, e0, e1);
    case 12804: return launch_t<128, 4>(p, s, e0, e1);
    case 12808: return launch_t<128, 8>(p, s, e0, e1);
    case 25604: return launch_t<256, 4>(p, s, e0, e1);
    case 25608: return launch_t<256, 8>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

int launch_decode_step(const AttendParams& p, const double* inv_freq, const float* yq, const float* yk,
                       const float* yv, const float* q_scale, const uint32_t* pos0, float eps, cudaStream_t s,
                       cudaEvent_t e0, cudaEvent_t e1) {
  StepExtra x;
  x.yq = yq; x.yk = yk; x.yv = yv; x.q_scale = q_scale; x.pos0 = pos0; x.eps = eps;
  for (int e = 0; e < 128; ++e) x.inv_freq[e] = inv_freq[e];
  switch (p.hd * 100 + p.nq) {
    case 6404: return launch_step<64, 4>(p, x, s, e0, e1);
    case 6408: return launch_step<64, 8>(p, x, s, e0, e1);
    case 12804: return launch_step<128, 4>(p, x, s, e0, e1);
    case 12808: return launch_step<128, 8>(p, x, s, e0, e1);
    case 25604: return launch_step<256, 4>(p, x, s, e0, e1);
    case 25608: return launch_step<256, 8>(p, x, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

int attend_decode_occupancy(int hd, int nq) {
  switch (hd * 100 + nq) {
    case 6404: return occ_t<64, 4>();
    case 6408: return occ_t<64, 8>();
    case 12804: return occ_t<128, 4>();
    case 12808: return occ_t<128, 8>();
    case 25604: return occ_t<256, 4>();
    case 25608: return occ_t<256, 8>();
  }
  return 1;
}

}  // namespace swa
