// Far field of a decode row ("o1c_msl.metal", cortiq-engine 0.8.79:
// o1c_tok_far, the far half of o1c_tok_commit; "dory_msl.metal",
// cortiq-engine 0.8.57: the clip of dory_ofar).
//
// One warp per (sequence, query head), lane a = landmark a (m <= 32), for
// every row of the chunk (o1c_far_e, o1c_far, o1c_far_commit for chunks):
//  1. once the window is full, row j evicts the oldest key still held (ring
//     slot (win_head + j - j0) % W, j0 = W - win_len): every landmark scores
//     the chunk's evicted keys (fe_j = s <q~_a, k_j>) and takes the chunk's
//     max mx', the rescale rr = exp(mx - mx') and e_j = exp(fe_j - mx');
//  2. row i sees the evictions of rows 0..i: landmark scores
//     fs_a = s <q_i, k~_a>, weights w_b = sum_a exp(fs_a - f) mu[a][b]
//     (clipped at 0 with rect), gains gain_b = w_b exp(f + mx'_b - fm),
//     fm = max_b (f + mx'_b), far mass sum_b gain_b (z_b rr_b + sum_j e_bj)
//     (negative: no far part), and the numerator, lanes over features,
//     sum_b gain_b rr_b t_b + sum_j (sum_b gain_b e_bj) v_j;
//  3. with commit, every eviction into the landmarks' numerators, max and mass.
// The record per (sequence, row, query head) — fm in log2 units, far mass, keep
// flag, numerator — is what the merge kernel adds to the row. The kernel runs
// before the attention and the merge, so the evicted ring slot still holds
// the evicted key when it is read here.
#include "swa_internal.cuh"

namespace swa {
namespace {

constexpr unsigned kFFull = 0xffffffffu;
constexpr int kFarWarps = 4;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFFull, v, o);
  return v;
}

template <int HD, int MAXT>
__global__ void __launch_bounds__(kFarWarps * 32, 1) far_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int D4 = HD / 4;
  constexpr int PER = (D4 + 31) / 32;
  constexpr int RG = MAXT < 8 ? MAXT : 8;               // rows per numerator sweep
  extern __shared__ __align__(16) float far_smem[];     // [kFarWarps][m][HD] landmark numerators
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * kFarWarps + warp;        // b * nh + h
  if (idx >= p.B * p.nh) return;
  const int b = idx / p.nh, h = idx % p.nh, g = h / p.hpg;
  const int m = p.far_m;
  const int t = p.t;
  const bool live = lane < m;
  bool bad = false;
  const swa_meta meta = p.meta[b];
  const SeqState st = sanitize_state(meta, p.cap, &bad);
  // rows j >= j0 = W - win_len evict logical key j - j0 (ring slot
  // (win_head + j - j0) % W); a far chunk holds at most W rows
  const int j0 = st.W - st.len0;
  int n_ev = t - j0;
  if (n_ev < 0) n_ev = 0;
  if (n_ev > st.W) {
    n_ev = st.W;
    bad = true;
  }
  if (bad && lane == 0 && h == 0) set_err(p.err, SWA_DERR_META);
  const size_t ghi = (size_t)b * p.nh + h;
  const size_t kvh = (size_t)b * p.nk + g;
  float* mz = p.mz + ghi * 2 * m;
  const float* ring_k = p.ring_k + kvh * p.cap * HD;
  const float* ring_v = p.ring_v + kvh * p.cap * HD;
  auto ev_slot = [&](int e) { return (st.head0 + e) % st.W; };
  auto n_upto = [&](int i) {                            // evictions of rows 0..i
    int n = i - j0 + 1;
    return n < 0 ? 0 : (n > n_ev ? n_ev : n);
  };

  // the head's landmark numerators into shared memory, once (lanes over features)
  float* th_s = far_smem + (size_t)warp * m * HD;
  for (int a0 = 0; a0 < m; a0 += 8) {                   // 8 rows' loads in flight before the stores
    float4 tmp[8][PER];
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        tmp[k][c] = (a0 + k < m && d4 < D4)
                        ? reinterpret_cast<const float4*>(p.t_hat + (ghi * m + a0 + k) * HD)[d4]
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        if (a0 + k < m && d4 < D4) reinterpret_cast<float4*>(th_s + (a0 + k) * HD)[d4] = tmp[k][c];
      }
  }
  // the lane's column of mu, fetched up front (independent loads)
  const bool any_far = meta.far_len + (uint32_t)n_ev > 0u;
  float mu_col[32];
  {
    const float* mu = p.mu + ghi * m * m;
#pragma unroll
    for (int a = 0; a < 32; ++a) mu_col[a] = (any_far && live && a < m) ? mu[a * m + lane] : 0.f;
  }

  // 1. every eviction of the chunk against landmark `lane` and every row's
  // landmark score, in one pass over the features (the lane's q~ and k~ rows
  // are read once; the evicted keys and the rows' queries are broadcast)
  float mx = live ? mz[lane] : 0.f;
  float z = live ? mz[m + lane] : 0.f;
  float ev[MAXT], fs[MAXT];                             // MAXT >= t >= evictions
#pragma unroll
  for (int j = 0; j < MAXT; ++j) ev[j] = fs[j] = 0.f;
  if (live && any_far) {
    const float* qt = p.q_tilde + (ghi * m + lane) * HD;
    const float* kt = p.k_tilde + (kvh * m + lane) * HD;
    const float* qrow = p.q + ((size_t)b * t * p.nh + h) * HD;   // row i at qrow + i * nh * HD
#pragma unroll 2
    for (int d4 = 0; d4 < D4; ++d4) {
      const float4 x = *reinterpret_cast<const float4*>(qt + d4 * 4);
      const float4 k = *reinterpret_cast<const float4*>(kt + d4 * 4);
#pragma unroll
      for (int j = 0; j < MAXT; ++j) {
        if (j < n_ev) {
          const float4 y = *reinterpret_cast<const float4*>(ring_k + (size_t)ev_slot(j) * HD + d4 * 4);
          ev[j] += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
        }
        if (j < t) {
          const float4 u = *reinterpret_cast<const float4*>(qrow + (size_t)j * p.nh * HD + d4 * 4);
          fs[j] += u.x * k.x + u.y * k.y + u.z * k.z + u.w * k.w;
        }
      }
    }
  }
  float rr = 1.f;
  if (n_ev > 0 && live) {                               // the chunk's max, rescale and e_j
    float mx2 = mx;
#pragma unroll
    for (int j = 0; j < MAXT; ++j)
      if (j < n_ev) {
        ev[j] *= p.scale;
        mx2 = fmaxf(mx2, ev[j]);
      }
    rr = mx2 == mx ? 1.f : expf(mx - mx2);             // an empty landmark (-inf) gives 0
#pragma unroll
    for (int j = 0; j < MAXT; ++j) ev[j] = j < n_ev ? expf(ev[j] - mx2) : 0.f;
    mx = mx2;
  }
  const float z_base = z * rr;                          // mass before the chunk, rescaled
  __syncwarp();                                         // th_s is complete

  // 2. each row's gains and far mass (the record's header); gn[i] = gain_i
  float gn[MAXT];
#pragma unroll
  for (int i = 0; i < MAXT; ++i) {
    gn[i] = 0.f;
    if (i >= t) continue;
    const int n_i = n_upto(i);
    float fm = -INFINITY, far_den = 0.f;
    bool have = false;
    if (meta.far_len + (uint32_t)n_i > 0u) {
      const float fsi = live ? fs[i] * p.scale : -INFINITY;
      const float f = warp_max(fsi);
      const float ea = live ? expf(fsi - f) : 0.f;
      float w = 0.f;
#pragma unroll
      for (int a = 0; a < 32; ++a) w += __shfl_sync(kFFull, ea, a) * mu_col[a];   // mu_col[a] = 0 past m
      if (p.far_rect) w = fmaxf(w, 0.f);
      const float fb = live ? f + mx : -INFINITY;
      fm = warp_max(fb);
      float gain = (live && fm != -INFINITY) ? w * expf(fb - fm) : 0.f;
      float zi = z_base;
#pragma unroll
      for (int j = 0; j < MAXT; ++j) zi += j < n_i ? ev[j] : 0.f;
      far_den = warp_sum(gain * zi);
      have = fm != -INFINITY && far_den >= 0.f;          // a NaN or negative mass drops the far part
      if (!have) far_den = 0.f;
      gn[i] = have ? gain : 0.f;
    }
    if (lane == 0) {
      float* rec = p.ws_far + (((size_t)b * t + i) * p.nh + h) * (4 + HD);
      rec[0] = have ? fm * 1.4426950408889634f : -INFINITY;  // log2 units, as the near records
      rec[1] = far_den;
      rec[2] = have ? 1.f : 0.f;
      rec[3] = 0.f;
    }
  }

  // 3. numerators, RG rows at a time, lanes over features:
  // sum_b gain_b rr_b t_b + sum_{j < n_i} (sum_b gain_b e_bj) v_j
  for (int i0 = 0; i0 < t; i0 += RG) {
    float4 num[RG][PER];
#pragma unroll
    for (int k = 0; k < RG; ++k)
#pragma unroll
      for (int c = 0; c < PER; ++c) num[k][c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float grr[RG];
#pragma unroll
    for (int k = 0; k < RG; ++k) {
      float v = 0.f;
#pragma unroll
      for (int i = 0; i < MAXT; ++i) v = i == i0 + k ? gn[i] : v;  // static register indices
      grr[k] = v * rr;
    }
    for (int a = 0; a < m; ++a) {
      float4 ta[PER];
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        ta[c] = d4 < D4 ? reinterpret_cast<const float4*>(th_s + a * HD)[d4] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < RG; ++k) {
        const float ga = __shfl_sync(kFFull, grr[k], a);
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          num[k][c].x += ga * ta[c].x; num[k][c].y += ga * ta[c].y;
          num[k][c].z += ga * ta[c].z; num[k][c].w += ga * ta[c].w;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < MAXT; ++j) {
      if (j >= n_ev) continue;
      float4 vj[PER];
      const float* vr = ring_v + (size_t)ev_slot(j) * HD;
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        vj[c] = d4 < D4 ? *reinterpret_cast<const float4*>(vr + d4 * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < RG; ++k) {
        const int i = i0 + k;
        if (i >= t || j >= n_upto(i)) continue;
        float gi = 0.f;
#pragma unroll
        for (int ii = 0; ii < MAXT; ++ii) gi = ii == i ? gn[ii] : gi;
        const float cf = warp_sum(gi * ev[j]);          // the evicted row's weight in row i
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          num[k][c].x += cf * vj[c].x; num[k][c].y += cf * vj[c].y;
          num[k][c].z += cf * vj[c].z; num[k][c].w += cf * vj[c].w;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < RG; ++k) {
      const int i = i0 + k;
      if (i >= t) continue;
      float* rec = p.ws_far + (((size_t)b * t + i) * p.nh + h) * (4 + HD);
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        if (d4 < D4) *reinterpret_cast<float4*>(rec + 4 + d4 * 4) = num[k][c];
      }
    }
  }

  // 4. the commit: every eviction of the chunk into the landmark numerators,
  // the max and the mass (o1c_far_commit)
  if (p.commit && n_ev > 0) {
    for (int a = 0; a < m; ++a) {
      const float ra = __shfl_sync(kFFull, rr, a);
      float4 tv[PER];
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        tv[c] = d4 < D4 ? reinterpret_cast<const float4*>(th_s + a * HD)[d4] : make_float4(0.f, 0.f, 0.f, 0.f);
        tv[c].x *= ra; tv[c].y *= ra; tv[c].z *= ra; tv[c].w *= ra;
      }
#pragma unroll
      for (int j = 0; j < MAXT; ++j) {
        if (j >= n_ev) continue;
        const float ej = __shfl_sync(kFFull, ev[j], a);     // landmark a's e_j
        const float* vr = ring_v + (size_t)ev_slot(j) * HD;
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          const int d4 = lane + 32 * c;
          if (d4 < D4) {
            const float4 v = *reinterpret_cast<const float4*>(vr + d4 * 4);
            tv[c].x += ej * v.x; tv[c].y += ej * v.y; tv[c].z += ej * v.z; tv[c].w += ej * v.w;
          }
        }
      }
      float4* th = reinterpret_cast<float4*>(p.t_hat + (ghi * m + a) * HD);
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        if (d4 < D4) th[d4] = tv[c];
      }
    }
    if (live) {
      float zf = z_base;
#pragma unroll
      for (int j = 0; j < MAXT; ++j) zf += j < n_ev ? ev[j] : 0.f;
      mz[lane] = mx;
      mz[m + lane] = zf;
    }
  }
}

template <int HD, int MAXT>
int run_far(const AttendParams& p, dim3 grid, dim3 block, size_t smem, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(far_kernel<HD, MAXT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(kFarWarps * 32 * HD * sizeof(float)));
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  far_kernel<HD, MAXT><<<grid, block, smem, s>>>(p);
  return finish_launch(cudaSuccess);
}

// the row and eviction arrays are sized by the chunk: 1, 8 or 32 rows
template <int HD>
int run_far_t(const AttendParams& p, dim3 grid, dim3 block, size_t smem, cudaStream_t s) {
  if (p.t == 1) return run_far<HD, 1>(p, grid, block, smem, s);
  if (p.t <= 8) return run_far<HD, 8>(p, grid, block, smem, s);
  return run_far<HD, 32>(p, grid, block, smem, s);
}

}  // namespace

int launch_far(const AttendParams& p, cudaStream_t s) {
  const int warps = p.B * p.nh;
  const dim3 grid((unsigned)((warps + kFarWarps - 1) / kFarWarps));
  const dim3 block(kFarWarps * 32);
  // An ordinary launch (after the prep in full stream order): launched
  // programmatically its CTAs were resident early and the step took 237.5 us
  // instead of 210 us on batched_decode_far. It still triggers its dependents,
  // so the attention's CTAs are scheduled during its tail.
  const size_t smem = (size_t)kFarWarps * p.far_m * p.hd * sizeof(float);
  switch (p.hd) {
    case 64: return run_far_t<64>(p, grid, block, smem, s);
    case 128: return run_far_t<128>(p, grid, block, smem, s);
    case 256: return run_far_t<256>(p, grid, block, smem, s);
    default: return SWA_E_SHAPE;
  }
}

}  // namespace swa
