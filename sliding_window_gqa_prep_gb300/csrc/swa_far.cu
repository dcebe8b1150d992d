// Far field of a decode row ("o1c_msl.metal", cortiq-engine 0.8.79:
// o1c_tok_far, the far half of o1c_tok_commit; "dory_msl.metal",
// cortiq-engine 0.8.57: the clip of dory_ofar).
//
// One warp per (sequence, query head), lane a = landmark a (m <= 32):
//  1. a full window evicts its oldest key (ring slot win_head): every landmark
//     takes it into its running max and mass (fe = s <q~_a, k>, mx' = max,
//     rr = exp(mx - mx'), e = exp(fe - mx'), z' = z rr + e);
//  2. the row's far part: landmark scores fs_a = s <q, k~_a>, weights
//     w_b = sum_a exp(fs_a - f) mu[a][b] (clipped at 0 with rect), gains
//     gain_b = w_b exp(f + mx'_b - fm) with fm = max_b (f + mx'_b), far mass
//     sum_b gain_b z'_b (negative: no far part);
//  3. lanes over features: the landmarks' numerators after the eviction,
//     t'_b = t_b rr_b + e_b v, their gain-weighted sum (the row's far
//     numerator) and, with commit, t' and (mx', z') written back.
// The record per (sequence, query head) — fm in log2 units, far mass, keep
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
__global__ void __launch_bounds__(kFarWarps * 32) far_kernel(AttendParams p) {
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
  const swa_meta meta = p.meta[b];
  const SeqState st = sanitize_state(meta, p.cap, nullptr);
  const bool evict = st.len0 == st.W;
  const size_t ghi = (size_t)b * p.nh + h;
  const size_t kvh = (size_t)b * p.nk + g;
  float* mz = p.mz + ghi * 2 * m;

  // 1-2. the eviction score s <q~_a, k_ev> and the landmark score
  // s <q, k~_a> of landmark `lane`: one pass over the features with both
  // rows' loads in flight
  float mx = live ? mz[lane] : 0.f;
  float z = live ? mz[m + lane] : 0.f;
  const float* k_ev = p.ring_k + (kvh * p.cap + st.head0) * HD;
  const float* v_ev = p.ring_v + (kvh * p.cap + st.head0) * HD;
  const bool any_far = meta.far_len + (evict ? 1u : 0u) > 0u;
  // the lane's column of mu, fetched up front (independent loads)
  float mu_col[32];
  {
    const float* mu = p.mu + ghi * m * m;
#pragma unroll
    for (int a = 0; a < 32; ++a) mu_col[a] = (any_far && live && a < m) ? mu[a * m + lane] : 0.f;
  }
  float fe_acc = 0.f, fs_acc = 0.f;
  if (live && (evict || any_far)) {
    const float* qt = p.q_tilde + (ghi * m + lane) * HD;
    const float* kt = p.k_tilde + (kvh * m + lane) * HD;
    const float* q = p.q + ghi * HD;                    // t = 1: row 0 of sequence b
#pragma unroll 16
    for (int d4 = 0; d4 < HD / 4; ++d4) {
      if (evict) {
        const float4 x = *reinterpret_cast<const float4*>(qt + d4 * 4);
        const float4 y = *reinterpret_cast<const float4*>(k_ev + d4 * 4);
        fe_acc += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
      }
      const float4 u = *reinterpret_cast<const float4*>(q + d4 * 4);
      const float4 v = *reinterpret_cast<const float4*>(kt + d4 * 4);
      fs_acc += u.x * v.x + u.y * v.y + u.z * v.z + u.w * v.w;
    }
  }
  float rr = 1.f, e = 0.f;
  if (evict && live) {                                  // the key joins landmark `lane`
    const float fe = fe_acc * p.scale;
    const float mx2 = fmaxf(mx, fe);
    rr = mx2 == mx ? 1.f : expf(mx - mx2);              // an empty landmark (-inf) gives 0
    e = expf(fe - mx2);
    z = z * rr + e;
    mx = mx2;
  }

  // landmark weights, gains, far mass
  float fm = -INFINITY, far_den = 0.f, gain = 0.f;
  bool have = false;
  if (any_far) {
    const float fs = live ? fs_acc * p.scale : -INFINITY;
    const float f = warp_max(fs);
    const float ea = live ? expf(fs - f) : 0.f;
    float w = 0.f;
#pragma unroll
    for (int a = 0; a < 32; ++a) w += __shfl_sync(kFFull, ea, a) * mu_col[a];   // mu_col[a] = 0 past m
    if (p.far_rect) w = fmaxf(w, 0.f);
    const float fb = live ? f + mx : -INFINITY;
    fm = warp_max(fb);
    gain = (live && fm != -INFINITY) ? w * expf(fb - fm) : 0.f;
    far_den = warp_sum(gain * z);
    have = fm != -INFINITY && far_den >= 0.f;            // a NaN or negative mass drops the far part
    if (!have) {
      far_den = 0.f;
      gain = 0.f;
    }
  }

  // 3. numerators after the eviction, the row's far numerator, the write-back
  const bool write_back = p.commit && evict;
  float4 num[PER], vv[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) {
    num[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    vv[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int d4 = lane + 32 * c;
    if (evict && d4 < D4) vv[c] = *reinterpret_cast<const float4*>(v_ev + d4 * 4);
  }
  if (have || write_back) {
    // landmarks 8 at a time: their numerator rows are loaded before any is used
    for (int a0 = 0; a0 < m; a0 += 8) {
      float4 t[8][PER];
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          const int d4 = lane + 32 * c;
          t[k][c] = (a0 + k < m && d4 < D4)
                        ? reinterpret_cast<const float4*>(p.t_hat + (ghi * m + a0 + k) * HD)[d4]
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int a = a0 + k;                            // lanes past m hold gain = rr = e = 0
        const float ga = __shfl_sync(kFFull, gain, a & 31);
        const float ra = __shfl_sync(kFFull, rr, a & 31);
        const float eb = __shfl_sync(kFFull, e, a & 31);
        if (a >= m) continue;
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          const int d4 = lane + 32 * c;
          if (d4 >= D4) continue;
          float4 u = t[k][c];
          if (evict) {
            u.x = u.x * ra + eb * vv[c].x;
            u.y = u.y * ra + eb * vv[c].y;
            u.z = u.z * ra + eb * vv[c].z;
            u.w = u.w * ra + eb * vv[c].w;
            if (write_back) reinterpret_cast<float4*>(p.t_hat + (ghi * m + a) * HD)[d4] = u;
          }
          num[c].x += ga * u.x; num[c].y += ga * u.y; num[c].z += ga * u.z; num[c].w += ga * u.w;
        }
      }
    }
  }
  float* rec = p.ws_far + ghi * (4 + HD);
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
  if (write_back && live) {
    mz[lane] = mx;
    mz[m + lane] = z;
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
