// Attend stage: sinks + causal window over the ring and the chunk, GQA, f32
// softmax, split-KV value sums, their reduction, the sigmoid gate and the
// commit ("o1c_msl.metal", cortiq-engine 0.8.79: o1c_score, o1c_max,
// o1c_soft, o1c_sum, o1c_add, o1c_tok_near, o1c_tok_merge, o1c_ring_commit,
// o1c_meta; "dory_msl.metal", cortiq-engine 0.8.57: dory_gate).
//
// Kernel 1 (attend_partial_kernel): one CTA per (sequence b, KV head g, row
// block rb, split s). A row block is `rows` consecutive chunk rows; its nq =
// rows * hpg query vectors (all query heads of g) share every K/V byte, so
// each byte of the block's key range is read from HBM once per split. The
// key range of a row block is the sinks followed by the logical keys
// [lo(r0), len0 + r_last]; split s takes keys [s*chunk, (s+1)*chunk) of it.
// Keys stream through a ring of STAGES shared-memory tiles of TK rows; each
// key row is one bulk copy (cp.async.bulk, the TMA's non-tensor form) from
// the sink buffer, the ring slot (head0 + x) % W, or the chunk row x - len0,
// so the ring's wrap-around lives in the address map, not in the data. Per
// tile: scores Q K^T (register-blocked on CUDA cores), row max, exp2 with
// online rescaling (scores carry scale * log2 e), P V accumulation. The CTA
// writes its (m, l, acc) record to the workspace.
//
// Kernel 2 (attend_merge_kernel): per output (b, row, head, 4 features):
// max over the valid splits, rescale-and-sum of l and acc, o = acc / den,
// times sigmoid(gate * gate_scale). Extra CTAs (one per sequence) commit the
// chunk into the ring and advance the meta; they run after kernel 1 has
// finished every read of the ring (stream order).
#include "swa_internal.cuh"

#include <cfloat>

namespace swa {
namespace {

constexpr int kNT = 128;                   // threads per attention CTA

template <int HD, int NQ>
struct Cfg {
  static constexpr int HDP = HD + 4;       // padded shared row (floats): conflict-free row reads
  // scores: thread = (q-group of 4, key group, d-split)
  static constexpr int QG = NQ / 4;
  static constexpr int KT = (NQ == 32) ? 2 : 1;
  static constexpr int KG = TK / KT;
  static constexpr int DS = kNT / (QG * KG);
  static constexpr int DSPAN = HD / DS;
  // P V: thread = (q-group of 4, feature group, key split)
  static constexpr int NDC4 = (NQ / 4) * (HD / 4);
  static constexpr int KS = NDC4 <= kNT ? kNT / NDC4 : 1;
  static constexpr int DT = NDC4 <= kNT ? 4 : 4 * NDC4 / kNT;
  static constexpr int NDC = HD / DT;
  static constexpr int STAGES = (HD == 64) ? 4 : (HD == 128 ? (NQ >= 16 ? 2 : 3) : 2);
  static constexpr int SROW = TK + 1;      // padded score row
  static constexpr int PROW = NQ + 4;      // P^T row (keeps 16-byte alignment)
  // shared-memory layout (floats, then barriers)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * TK * HDP;
  static constexpr int OFF_QT = OFF_V + STAGES * TK * HDP;
  static constexpr int OFF_S = OFF_QT + HD * NQ;
  static constexpr int OFF_P = OFF_S + DS * NQ * SROW;
  static constexpr int OFF_M = OFF_P + TK * PROW;
  static constexpr int OFF_L = OFF_M + NQ;
  static constexpr int OFF_C = OFF_L + NQ;
  static constexpr int OFF_MISC = OFF_C + NQ;          // [0]: abort flag
  static constexpr int FLOATS = ((OFF_MISC + 4 + 1) / 2) * 2;   // 8-byte align barriers
  static constexpr size_t BYTES = (size_t)FLOATS * 4 + STAGES * sizeof(uint64_t);
  static_assert(QG * KG * DS == kNT, "score layout must cover the CTA");
  static_assert(QG * NDC * KS == kNT, "P V layout must cover the CTA");
  static_assert(DT % 4 == 0, "feature chunks are float4");
  static_assert(KS * NQ * HD <= 2 * STAGES * TK * HDP, "split reduction fits the stage buffers");
};

template <int HD, int NQ>
__global__ void __launch_bounds__(kNT) attend_partial_kernel(AttendParams p) {
  using C = Cfg<HD, NQ>;
  extern __shared__ __align__(128) float smem[];
  float* Ks = smem + C::OFF_K;
  float* Vs = smem + C::OFF_V;
  float* QT = smem + C::OFF_QT;
  float* Sp = smem + C::OFF_S;
  float* PT = smem + C::OFF_P;
  float* s_m = smem + C::OFF_M;
  float* s_l = smem + C::OFF_L;
  float* s_c = smem + C::OFF_C;
  int* s_abort = reinterpret_cast<int*>(smem + C::OFF_MISC);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::FLOATS);

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x;                      // split
  const int rb = blockIdx.y;                     // row block
  const int bg = blockIdx.z;                     // b * nk + g
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
    for (int i = 0; i < C::STAGES; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
    *s_abort = 0;
  }
  if (tid < NQ) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  __syncthreads();

  const size_t kv_head = (size_t)b * p.nk + g;
  // Producer: warp 0 issues one bulk copy per key row (K and V) of tile i.
  auto issue = [&](int i) {
    const int stage = i % C::STAGES;
    const int j0 = jb + i * TK;
    const int cnt = min(TK, je - j0);
    if (lane == 0) mbar_arrive_expect_tx(&bars[stage], (uint32_t)(cnt * HD * 4 * 2));
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
          const size_t at = (kv_head * p.cap + (size_t)((st.head0 + x) % st.W)) * HD;
          sk = p.ring_k + at;
          sv = p.ring_v + at;
        } else {
          const size_t at = (((size_t)b * p.t + (x - st.len0)) * p.nk + g) * HD;
          sk = p.k_chunk + at;
          sv = p.v_chunk + at;
        }
      }
      float* dk = Ks + ((size_t)stage * TK + lane) * C::HDP;
      float* dv = Vs + ((size_t)stage * TK + lane) * C::HDP;
      bulk_g2s(dk, sk, HD * 4, &bars[stage]);
      bulk_g2s(dv, sv, HD * 4, &bars[stage]);
    }
  };
  if (warp == 0) {
    fence_proxy_async_smem();
    for (int i = 0; i < C::STAGES && i < ntiles; ++i) issue(i);
  }

  // Q^T [HD][NQ], pre-multiplied by scale * log2(e); unused query slots are 0.
  for (int idx = tid; idx < NQ * (HD / 4); idx += kNT) {
    const int q = idx / (HD / 4), d4 = idx % (HD / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    const int rr = q / p.hpg, h = q % p.hpg;
    if (rr < rows_eff) {
      v = *reinterpret_cast<const float4*>(
          p.q + (((size_t)b * p.t + r0 + rr) * p.nh + (size_t)g * p.hpg + h) * HD + d4 * 4);
      v.x *= p.qmul; v.y *= p.qmul; v.z *= p.qmul; v.w *= p.qmul;
    }
    QT[(d4 * 4 + 0) * NQ + q] = v.x;
    QT[(d4 * 4 + 1) * NQ + q] = v.y;
    QT[(d4 * 4 + 2) * NQ + q] = v.z;
    QT[(d4 * 4 + 3) * NQ + q] = v.w;
  }
  __syncthreads();   // Q^T visible to every thread

  // thread roles
  const int sq_g = tid % C::QG;
  const int sk_g = (tid / C::QG) % C::KG;
  const int s_ds = tid / (C::QG * C::KG);
  const int pq_g = tid % C::QG;
  const int p_dc = (tid / C::QG) % C::NDC;
  const int p_ks = tid / (C::QG * C::NDC);

  float acc[4][C::DT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int d = 0; d < C::DT; ++d) acc[i][d] = 0.f;

  bool aborted = false;
  int last_issued = min(ntiles, C::STAGES) - 1;   // highest tile index handed to the copy engine
  for (int i = 0; i < ntiles; ++i) {
    const int stage = i % C::STAGES;
    const uint32_t parity = (uint32_t)((i / C::STAGES) & 1);
    if (!mbar_wait_bounded(&bars[stage], parity, kWaitLimitNs)) *s_abort = 1;
    const int j0 = jb + i * TK;
    const int cnt = min(TK, je - j0);
    const float* Kt = Ks + (size_t)stage * TK * C::HDP;
    const float* Vt = Vs + (size_t)stage * TK * C::HDP;

    // ---- scores: S[q][k] = sum_d QT[d][q] * K[k][d] over this thread's d-span
    {
      float sacc[C::KT][4];
#pragma unroll
      for (int kt = 0; kt < C::KT; ++kt)
#pragma unroll
        for (int qi = 0; qi < 4; ++qi) sacc[kt][qi] = 0.f;
      const float* qb = QT + (size_t)(s_ds * C::DSPAN) * NQ + sq_g * 4;
      const float* kb = Kt + (size_t)sk_g * C::HDP + s_ds * C::DSPAN;
#pragma unroll 4
      for (int d = 0; d < C::DSPAN; d += 4) {
        const float4 q0 = *reinterpret_cast<const float4*>(qb + (d + 0) * NQ);
        const float4 q1 = *reinterpret_cast<const float4*>(qb + (d + 1) * NQ);
        const float4 q2 = *reinterpret_cast<const float4*>(qb + (d + 2) * NQ);
        const float4 q3 = *reinterpret_cast<const float4*>(qb + (d + 3) * NQ);
#pragma unroll
        for (int kt = 0; kt < C::KT; ++kt) {
          const float4 kv = *reinterpret_cast<const float4*>(kb + (size_t)kt * C::KG * C::HDP + d);
          sacc[kt][0] += q0.x * kv.x + q1.x * kv.y + q2.x * kv.z + q3.x * kv.w;
          sacc[kt][1] += q0.y * kv.x + q1.y * kv.y + q2.y * kv.z + q3.y * kv.w;
          sacc[kt][2] += q0.z * kv.x + q1.z * kv.y + q2.z * kv.z + q3.z * kv.w;
          sacc[kt][3] += q0.w * kv.x + q1.w * kv.y + q2.w * kv.z + q3.w * kv.w;
        }
      }
#pragma unroll
      for (int kt = 0; kt < C::KT; ++kt)
#pragma unroll
        for (int qi = 0; qi < 4; ++qi)
          Sp[((size_t)s_ds * NQ + sq_g * 4 + qi) * C::SROW + sk_g + kt * C::KG] = sacc[kt][qi];
    }
    __syncthreads();   // scores visible; every thread is done with tile i-1
    if (*s_abort) { aborted = true; break; }
    if (i >= 1 && i - 1 + C::STAGES < ntiles) {
      last_issued = i - 1 + C::STAGES;
      if (warp == 0) {
        fence_proxy_async_smem();
        issue(i - 1 + C::STAGES);
      }
    }

    // ---- softmax of the tile: warp w owns queries w, w+4, ...; lane = key
    for (int q = warp; q < NQ; q += kNT / 32) {
      const int rr = q / p.hpg;
      const int j = j0 + lane;
      bool valid = lane < cnt && rr < rows_eff;
      if (valid && j >= p.ns) {
        const int r = r0 + rr;
        const int x = xlo + (j - p.ns);
        const int lo = st.len0 + r + 1 - min(st.W, st.len0 + r + 1);
        valid = x >= lo && x <= st.len0 + r;
      }
      float sv = 0.f;
#pragma unroll
      for (int ds = 0; ds < C::DS; ++ds) sv += Sp[((size_t)ds * NQ + q) * C::SROW + lane];
      sv = valid ? sv : -INFINITY;
      float tmax = sv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_old = s_m[q];
      const float m_new = fmaxf(m_old, tmax);
      float pv, corr;
      if (m_new == -INFINITY) {
        pv = 0.f;
        corr = 1.f;
      } else {
        pv = exp2f(sv - m_new);
        corr = exp2f(m_old - m_new);
      }
      float psum = pv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      PT[(size_t)lane * C::PROW + q] = pv;
      __syncwarp();
      if (lane == 0) {
        s_l[q] = s_l[q] * corr + psum;
        s_m[q] = m_new;
        s_c[q] = corr;
      }
    }
    __syncthreads();   // P^T and corrections visible

    // ---- P V: acc[q][d] = acc * corr + sum_k P[k][q] V[k][d]
    {
      const float4 c4 = *reinterpret_cast<const float4*>(s_c + pq_g * 4);
#pragma unroll
      for (int d = 0; d < C::DT; ++d) {
        acc[0][d] *= c4.x;
        acc[1][d] *= c4.y;
        acc[2][d] *= c4.z;
        acc[3][d] *= c4.w;
      }
      for (int k = p_ks; k < cnt; k += C::KS) {
        const float4 pk = *reinterpret_cast<const float4*>(PT + (size_t)k * C::PROW + pq_g * 4);
        const float* vr = Vt + (size_t)k * C::HDP;
#pragma unroll
        for (int c = 0; c < C::DT / 4; ++c) {
          const float4 v = *reinterpret_cast<const float4*>(vr + (p_dc + c * C::NDC) * 4);
          acc[0][c * 4 + 0] += pk.x * v.x; acc[0][c * 4 + 1] += pk.x * v.y;
          acc[0][c * 4 + 2] += pk.x * v.z; acc[0][c * 4 + 3] += pk.x * v.w;
          acc[1][c * 4 + 0] += pk.y * v.x; acc[1][c * 4 + 1] += pk.y * v.y;
          acc[1][c * 4 + 2] += pk.y * v.z; acc[1][c * 4 + 3] += pk.y * v.w;
          acc[2][c * 4 + 0] += pk.z * v.x; acc[2][c * 4 + 1] += pk.z * v.y;
          acc[2][c * 4 + 2] += pk.z * v.z; acc[2][c * 4 + 3] += pk.z * v.w;
          acc[3][c * 4 + 0] += pk.w * v.x; acc[3][c * 4 + 1] += pk.w * v.y;
          acc[3][c * 4 + 2] += pk.w * v.z; acc[3][c * 4 + 3] += pk.w * v.w;
        }
      }
    }
  }

  if (aborted) {
    // Let copies still in flight land (bounded) before the CTA's shared memory goes away.
    if (tid == 0) {
      set_err(p.err, SWA_DERR_TIMEOUT);
      for (int st_i = 0; st_i < C::STAGES && st_i <= last_issued; ++st_i) {
        const int last = last_issued - ((last_issued - st_i) % C::STAGES);   // last tile of this stage
        mbar_wait_bounded(&bars[st_i], (uint32_t)((last / C::STAGES) & 1), kWaitLimitNs);
      }
    }
    return;
  }

  // ---- epilogue: reduce the key splits of P V, write (m, l, acc)
  const size_t item = (((size_t)bg * p.n_rb + rb) * p.splits + s);
  float* wacc = p.ws_acc + item * (size_t)p.nq * HD;
  if (C::KS == 1) {
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) {
      float* dst = wacc + (size_t)(pq_g * 4 + qi) * HD;
#pragma unroll
      for (int c = 0; c < C::DT / 4; ++c)
        *reinterpret_cast<float4*>(dst + (p_dc + c * C::NDC) * 4) =
            make_float4(acc[qi][c * 4 + 0], acc[qi][c * 4 + 1], acc[qi][c * 4 + 2], acc[qi][c * 4 + 3]);
    }
  } else {
    __syncthreads();   // every thread is past its last read of the stage buffers
    float* red = smem;  // [KS][NQ][HD], reuses the K/V stages
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) {
      float* dst = red + ((size_t)p_ks * NQ + pq_g * 4 + qi) * HD;
#pragma unroll
      for (int c = 0; c < C::DT / 4; ++c)
        *reinterpret_cast<float4*>(dst + (p_dc + c * C::NDC) * 4) =
            make_float4(acc[qi][c * 4 + 0], acc[qi][c * 4 + 1], acc[qi][c * 4 + 2], acc[qi][c * 4 + 3]);
    }
    __syncthreads();
    for (int idx = tid; idx < NQ * HD / 4; idx += kNT) {
      float4 sum = *reinterpret_cast<const float4*>(red + (size_t)idx * 4);
#pragma unroll
      for (int k = 1; k < C::KS; ++k) {
        const float4 o = *reinterpret_cast<const float4*>(red + ((size_t)k * NQ * HD) + (size_t)idx * 4);
        sum.x += o.x; sum.y += o.y; sum.z += o.z; sum.w += o.w;
      }
      *reinterpret_cast<float4*>(wacc + (size_t)idx * 4) = sum;
    }
  }
  if (tid < NQ) p.ws_ml[item * p.nq + tid] = make_float2(s_m[tid], s_l[tid]);
}

// Merge of the split records + gate; trailing CTAs commit the chunk.
template <int HD>
__global__ void __launch_bounds__(256) attend_merge_kernel(AttendParams p, int out_blocks) {
  if ((int)blockIdx.x >= out_blocks) {
    // ---- commit of sequence b, spread over commit_blocks CTAs: the last
    // min(t, W) chunk rows into their ring slots (o1c_ring_commit), then the
    // meta (o1c_meta). The ring map comes from the copy of the meta the
    // attention kernel saved, so meta_out may alias meta.
    const int cb = (blockIdx.x - out_blocks) % p.commit_blocks;
    const int b = (blockIdx.x - out_blocks) / p.commit_blocks;
    const swa_meta m0 = p.ws_meta[b];
    const SeqState st = sanitize_state(m0, p.cap, nullptr);
    const int first = max(0, p.t - st.W);      // only the last W rows survive
    const int nrow = p.t - first;
    const int per_row = p.nk * (HD / 4);
    const int stride = p.commit_blocks * blockDim.x;
    for (int idx = cb * blockDim.x + threadIdx.x; idx < nrow * per_row; idx += stride) {
      const int j = first + idx / per_row;
      const int g = (idx % per_row) / (HD / 4);
      const int d4 = idx % (HD / 4);
      int slot = (int)(((long long)st.head0 + st.len0 + j) % st.W);
      const size_t src = (((size_t)b * p.t + j) * p.nk + g) * HD + d4 * 4;
      const size_t dst = (((size_t)b * p.nk + g) * p.cap + slot) * HD + d4 * 4;
      *reinterpret_cast<float4*>(p.ring_k + dst) = *reinterpret_cast<const float4*>(p.k_chunk + src);
      *reinterpret_cast<float4*>(p.ring_v + dst) = *reinterpret_cast<const float4*>(p.v_chunk + src);
    }
    if (cb == 0 && threadIdx.x == 0) {
      swa_meta m1 = m0;
      const long long tot = (long long)st.len0 + p.t;
      if (tot <= st.W) {
        m1.win_len = (uint32_t)tot;
      } else {
        const long long ev = tot - st.W;
        m1.win_len = (uint32_t)st.W;
        m1.win_head = (uint32_t)((st.head0 + ev) % st.W);
        m1.far_len = (uint32_t)(m0.far_len + (uint32_t)ev);
      }
      p.meta_out[b] = m1;
    }
    return;
  }
  constexpr int D4 = HD / 4;
  const size_t total = (size_t)p.B * p.t * p.nh * D4;
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int d4 = (int)(idx % D4);
  const size_t row = idx / D4;                 // (b * t + r) * nh + h
  const int h = (int)(row % p.nh);
  const size_t br = row / p.nh;
  const int r = (int)(br % p.t);
  const int b = (int)(br / p.t);
  const int g = h / p.hpg;
  const int rb = r / p.rows;
  const int q = (r - rb * p.rows) * p.hpg + (h - g * p.hpg);
  const size_t item0 = (((size_t)b * p.nk + g) * p.n_rb + rb) * p.splits;
  const int nval = p.ws_nsplit[b * p.n_rb + rb];
  float M = -INFINITY;
  for (int sidx = 0; sidx < nval; ++sidx) M = fmaxf(M, p.ws_ml[(item0 + sidx) * p.nq + q].x);
  float den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sidx = 0; sidx < nval; ++sidx) {
    const float2 ml = p.ws_ml[(item0 + sidx) * p.nq + q];
    if (ml.x == -INFINITY) continue;           // a split with no key of this row
    const float w = exp2f(ml.x - M);
    den += ml.y * w;
    const float4 a = *reinterpret_cast<const float4*>(
        p.ws_acc + ((item0 + sidx) * p.nq + q) * (size_t)HD + d4 * 4);
    acc.x += a.x * w; acc.y += a.y * w; acc.z += a.z * w; acc.w += a.w * w;
  }
  const float inv = 1.0f / den;
  const float4 gt = *reinterpret_cast<const float4*>(p.gate + row * HD + d4 * 4);
  const float4 gs = *reinterpret_cast<const float4*>(p.gate_scale + (size_t)h * HD + d4 * 4);
  float4 o;
  o.x = acc.x * inv / (1.0f + expf(-(gt.x * gs.x)));
  o.y = acc.y * inv / (1.0f + expf(-(gt.y * gs.y)));
  o.z = acc.z * inv / (1.0f + expf(-(gt.z * gs.z)));
  o.w = acc.w * inv / (1.0f + expf(-(gt.w * gs.w)));
  *reinterpret_cast<float4*>(p.out + row * HD + d4 * 4) = o;
}

template <int HD, int NQ>
int launch_partial_t(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = Cfg<HD, NQ>;
  auto kern = attend_partial_kernel<HD, NQ>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    attr_set[dev] = true;
  }
  dim3 grid((unsigned)p.splits, (unsigned)p.n_rb, (unsigned)(p.B * p.nk));
  if (e0) cudaEventRecord(e0, s);
  kern<<<grid, kNT, C::BYTES, s>>>(p);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e1) cudaEventRecord(e1, s);
  return cuda_status(e);
}

template <int HD, int NQ>
int occupancy_t() {
  using C = Cfg<HD, NQ>;
  auto kern = attend_partial_kernel<HD, NQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES) != cudaSuccess)
    return 1;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kNT, C::BYTES) != cudaSuccess) return 1;
  return blocks > 0 ? blocks : 1;
}

template <int HD>
int launch_partial_hd(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  switch (p.nq) {
    case 4: return launch_partial_t<HD, 4>(p, s, e0, e1);
    case 8: return launch_partial_t<HD, 8>(p, s, e0, e1);
    case 16: return launch_partial_t<HD, 16>(p, s, e0, e1);
    case 32: return launch_partial_t<HD, 32>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

template <int HD>
int occupancy_hd(int nq) {
  switch (nq) {
    case 4: return occupancy_t<HD, 4>();
    case 8: return occupancy_t<HD, 8>();
    case 16: return occupancy_t<HD, 16>();
    case 32: return occupancy_t<HD, 32>();
  }
  return 1;
}

}  // namespace

int launch_attend_partial(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  if (p.nq <= 8) return launch_attend_decode(p, s, e0, e1);
  if (p.nq == 64) return launch_attend_prompt(p, s, e0, e1);
  if (p.nq == 16 || p.nq == 32) return launch_attend_verify(p, s, e0, e1);
  switch (p.hd) {
    case 64: return launch_partial_hd<64>(p, s, e0, e1);
    case 128: return launch_partial_hd<128>(p, s, e0, e1);
    case 256: return launch_partial_hd<256>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

int attend_partial_occupancy(int hd, int nq) {
  if (nq <= 8) return attend_decode_occupancy(hd, nq);
  if (nq == 16 || nq == 32) return attend_verify_occupancy(hd, nq);
  switch (hd) {
    case 64: return occupancy_hd<64>(nq);
    case 128: return occupancy_hd<128>(nq);
    case 256: return occupancy_hd<256>(nq);
  }
  return 1;
}

int launch_attend_merge(const AttendParams& p, cudaStream_t s) {
  const size_t total = (size_t)p.B * p.t * p.nh * (p.hd / 4);
  const int block = 256;
  const int out_blocks = (int)((total + block - 1) / block);
  const int grid = out_blocks + (p.commit ? p.B * p.commit_blocks : 0);
  switch (p.hd) {
    case 64: attend_merge_kernel<64><<<grid, block, 0, s>>>(p, out_blocks); break;
    case 128: attend_merge_kernel<128><<<grid, block, 0, s>>>(p, out_blocks); break;
    case 256: attend_merge_kernel<256><<<grid, block, 0, s>>>(p, out_blocks); break;
    default: return SWA_E_SHAPE;
  }
  note_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace swa
