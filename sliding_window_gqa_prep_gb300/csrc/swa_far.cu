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

template <int HD>
__global__ void __launch_bounds__(kFarWarps * 32, 1) far_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int D4 = HD / 4;
  constexpr int PER = (D4 + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * kFarWarps + warp;        // b * nh + h
  if (idx >= p.B * p.nh) return;
  const int b = idx / p.nh, h = idx % p.nh, g = h / p.hpg;
  const int m = p.far_m;
  const bool live = lane < m;
  bool bad = false;
  const swa_meta meta = p.meta[b];
  const SeqState st = sanitize_state(meta, p.cap, &bad);
  // rows j >= j0 = W - win_len evict logical key j - j0 (ring slot
  // (win_head + j - j0) % W); a far chunk holds at most W rows
  const int j0 = st.W - st.len0;
  int n_ev = p.t - j0;
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

  // the lane's column of mu, fetched up front (independent loads)
  const bool any_far = meta.far_len + (uint32_t)n_ev > 0u;
  float mu_col[32];
  {
    const float* mu = p.mu + ghi * m * m;
#pragma unroll
    for (int a = 0; a < 32; ++a) mu_col[a] = (any_far && live && a < m) ? mu[a * m + lane] : 0.f;
  }

  // 1. every eviction of the chunk against landmark `lane`: scores in one
  // pass over the features, then the chunk's max, the rescale rr and e_j
  float mx = live ? mz[lane] : 0.f;
  float z = live ? mz[m + lane] : 0.f;
  float ev[32];                                         // e_j after the pass below
#pragma unroll
  for (int j = 0; j < 32; ++j) ev[j] = 0.f;
  if (n_ev > 0 && live) {
    const float* qt = p.q_tilde + (ghi * m + lane) * HD;
#pragma unroll 4
    for (int d4 = 0; d4 < D4; ++d4) {
      const float4 x = *reinterpret_cast<const float4*>(qt + d4 * 4);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < n_ev) {
          const float4 y = *reinterpret_cast<const float4*>(ring_k + (size_t)ev_slot(j) * HD + d4 * 4);
          ev[j] += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
        }
      }
    }
  }
  float rr = 1.f;
  if (n_ev > 0 && live) {
    float mx2 = mx;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n_ev) {
        ev[j] *= p.scale;
        mx2 = fmaxf(mx2, ev[j]);
      }
    rr = mx2 == mx ? 1.f : expf(mx - mx2);             // an empty landmark (-inf) gives 0
#pragma unroll
    for (int j = 0; j < 32; ++j) ev[j] = j < n_ev ? expf(ev[j] - mx2) : 0.f;
    mx = mx2;
  }
  const float z_base = z * rr;                          // mass before the chunk, rescaled

  // 2. each row: landmark weights, gains, far mass, numerator
  for (int i = 0; i < p.t; ++i) {
    int n_i = i - j0 + 1;                               // evictions of rows 0..i
    if (n_i < 0) n_i = 0;
    if (n_i > n_ev) n_i = n_ev;
    float fm = -INFINITY, far_den = 0.f, gain = 0.f;
    bool have = false;
    if (meta.far_len + (uint32_t)n_i > 0u) {
      float fs = -INFINITY;
      if (live) {
        const float* q = p.q + (((size_t)b * p.t + i) * p.nh + h) * HD;
        const float* kt = p.k_tilde + (kvh * m + lane) * HD;
        float acc = 0.f;
#pragma unroll 8
        for (int d4 = 0; d4 < D4; ++d4) {
          const float4 u = *reinterpret_cast<const float4*>(q + d4 * 4);
          const float4 v = *reinterpret_cast<const float4*>(kt + d4 * 4);
          acc += u.x * v.x + u.y * v.y + u.z * v.z + u.w * v.w;
        }
        fs = acc * p.scale;
      }
      const float f = warp_max(fs);
      const float ea = live ? expf(fs - f) : 0.f;
      float w = 0.f;
#pragma unroll
      for (int a = 0; a < 32; ++a) w += __shfl_sync(kFFull, ea, a) * mu_col[a];   // mu_col[a] = 0 past m
      if (p.far_rect) w = fmaxf(w, 0.f);
      const float fb = live ? f + mx : -INFINITY;
      fm = warp_max(fb);
      gain = (live && fm != -INFINITY) ? w * expf(fb - fm) : 0.f;
      float zi = z_base;
#pragma unroll
      for (int j = 0; j < 32; ++j) zi += j < n_i ? ev[j] : 0.f;
      far_den = warp_sum(gain * zi);
      have = fm != -INFINITY && far_den >= 0.f;          // a NaN or negative mass drops the far part
      if (!have) {
        far_den = 0.f;
        gain = 0.f;
      }
    }
    // numerator: sum_b gain_b (rr_b t_b + sum_{j < n_i} e_bj v_j), lanes over features
    float4 num[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c) num[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (have) {
      const float grr = gain * rr;
      for (int a0 = 0; a0 < m; a0 += 8) {
        float4 tl[8][PER];
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
          for (int c = 0; c < PER; ++c) {
            const int d4 = lane + 32 * c;
            tl[k][c] = (a0 + k < m && d4 < D4)
                           ? reinterpret_cast<const float4*>(p.t_hat + (ghi * m + a0 + k) * HD)[d4]
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float ga = __shfl_sync(kFFull, grr, (a0 + k) & 31);   // 0 past m
#pragma unroll
          for (int c = 0; c < PER; ++c) {
            num[c].x += ga * tl[k][c].x; num[c].y += ga * tl[k][c].y;
            num[c].z += ga * tl[k][c].z; num[c].w += ga * tl[k][c].w;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {                   // static indices keep ev[] in registers
        if (j < n_i) {
          const float cf = warp_sum(gain * ev[j]);      // the evicted row's weight in this row
          const float* vr = ring_v + (size_t)ev_slot(j) * HD;
#pragma unroll
          for (int c = 0; c < PER; ++c) {
            const int d4 = lane + 32 * c;
            if (d4 < D4) {
              const float4 v = *reinterpret_cast<const float4*>(vr + d4 * 4);
              num[c].x += cf * v.x; num[c].y += cf * v.y; num[c].z += cf * v.z; num[c].w += cf * v.w;
            }
          }
        }
      }
    }
    float* rec = p.ws_far + (((size_t)b * p.t + i) * p.nh + h) * (4 + HD);
#pragma unroll
    for (int c = 0; c < PER; ++c) {
      const int d4 = lane + 32 * c;
      if (d4 < D4) *reinterpret_cast<float4*>(rec + 4 + d4 * 4) = num[c];
    }
    if (lane == 0) {
      rec[0] = have ? fm * 1.4426950408889634f : -INFINITY;  // log2 units, as the near records
      rec[1] = far_den;
      rec[2] = have ? 1.f : 0.f;
      rec[3] = 0.f;
    }
  }

  // 3. the commit: every eviction of the chunk into the landmark numerators,
  // the max and the mass (o1c_far_commit)
  if (p.commit && n_ev > 0) {
    for (int a = 0; a < m; ++a) {
      const float ra = __shfl_sync(kFFull, rr, a);
      float4* th = reinterpret_cast<float4*>(p.t_hat + (ghi * m + a) * HD);
      float4 t[PER];
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        t[c] = d4 < D4 ? th[d4] : make_float4(0.f, 0.f, 0.f, 0.f);
        t[c].x *= ra; t[c].y *= ra; t[c].z *= ra; t[c].w *= ra;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {                   // static indices keep ev[] in registers
        if (j < n_ev) {
          const float ej = __shfl_sync(kFFull, ev[j], a);   // landmark a's e_j
          const float* vr = ring_v + (size_t)ev_slot(j) * HD;
#pragma unroll
          for (int c = 0; c < PER; ++c) {
            const int d4 = lane + 32 * c;
            if (d4 < D4) {
              const float4 v = *reinterpret_cast<const float4*>(vr + d4 * 4);
              t[c].x += ej * v.x; t[c].y += ej * v.y; t[c].z += ej * v.z; t[c].w += ej * v.w;
            }
          }
        }
      }
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        if (d4 < D4) th[d4] = t[c];
      }
    }
    if (live) {
      float zf = z_base;
#pragma unroll
      for (int j = 0; j < 32; ++j) zf += j < n_ev ? ev[j] : 0.f;
      mz[lane] = mx;
      mz[m + lane] = zf;
    }
  }
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
  switch (p.hd) {
    case 64: far_kernel<64><<<grid, block, 0, s>>>(p); break;
    case 128: far_kernel<128><<<grid, block, 0, s>>>(p); break;
    case 256: far_kernel<256><<<grid, block, 0, s>>>(p); break;
    default: return SWA_E_SHAPE;
  }
  return finish_launch(cudaSuccess);
}

}  // namespace swa
