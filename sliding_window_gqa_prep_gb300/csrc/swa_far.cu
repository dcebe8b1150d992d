// Far field of a chunk ("o1c_msl.metal", cortiq-engine 0.8.79: o1c_far_e,
// o1c_far, o1c_far_commit and, for a decode row, o1c_tok_far and the far half
// of o1c_tok_commit; "dory_msl.metal", cortiq-engine 0.8.57: the clip of
// dory_ofar).
//
// One CTA per (sequence, query head), one warp per chunk row (chunks of up to
// 64 rows, the pages' OB_K: 32 warps, two rows each past 32); lane a is
// landmark a (m <= 32) in the scalar steps and lanes run over features in the
// numerators:
//  1. the head's landmark numerators go to shared memory once; once the window
//     is full, row j evicts the oldest key still held (ring slot
//     (win_head + j - j0) % W, j0 = W - win_len), and warp j scores that key
//     against every landmark (fe_j = s <q~_a, k_j>);
//  2. the chunk's max per landmark mx', the rescale rr = exp(mx - mx') and
//     e_j = exp(fe_j - mx');
//  3. row i sees the evictions of rows 0..i: landmark scores
//     fs_a = s <q_i, k~_a>, weights w_b = sum_a exp(fs_a - f) mu[a][b]
//     (clipped at 0 with rect), gains gain_b = w_b exp(f + mx'_b - fm) with
//     fm = max_b (f + mx'_b), far mass sum_b gain_b (z_b rr_b + sum_j e_bj)
//     (negative: no far part), numerator
//     sum_b gain_b rr_b t_b + sum_j (sum_b gain_b e_bj) v_j;
//  4. with commit, every eviction into the landmarks' numerators, max and mass.
// The record per (sequence, row, query head) — fm in log2 units, far mass,
// keep flag, numerator — is what the merge kernel adds to the row. The kernel
// runs before the attention and the merge, so the evicted ring slots still
// hold the evicted keys when they are read here.
#include "swa_internal.cuh"

namespace swa {
namespace {

constexpr unsigned kFFull = 0xffffffffu;
constexpr int kFarRows = 64;                            // longest chunk with a far field (OB_K)

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

template <int HD, int MAXW>
__global__ void __launch_bounds__(MAXW * 32) far_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int D4 = HD / 4;
  constexpr int PER = (D4 + 31) / 32;
  extern __shared__ __align__(16) float far_smem[];
  const int m = p.far_m, t = p.t;
  float* th_s = far_smem;                               // [m][HD]  landmark numerators before the chunk
  float* fe_s = th_s + (size_t)m * HD;                  // [64][32] eviction scores, e_j after step 2
  float* rr_s = fe_s + kFarRows * 32;                   // [32]     rescale of each landmark
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int b = blockIdx.x / p.nh, h = blockIdx.x % p.nh, g = h / p.hpg;
  const bool live = lane < m;
  bool bad = false;
  const swa_meta meta = p.meta[b];
  const SeqState st = sanitize_state(meta, p.cap, &bad);
  // rows j >= j0 = W - win_len evict logical key j - j0; a far chunk holds at
  // most W rows
  const int j0 = st.W - st.len0;
  int n_ev = t - j0;
  if (n_ev < 0) n_ev = 0;
  if (n_ev > st.W) {
    n_ev = st.W;
    bad = true;
  }
  if (bad && threadIdx.x == 0 && h == 0) set_err(p.err, SWA_DERR_META);
  const size_t ghi = (size_t)b * p.nh + h;
  const size_t kvh = (size_t)b * p.nk + g;
  float* mz = p.mz + ghi * 2 * m;
  const float* ring_k = p.ring_k + kvh * p.cap * HD;
  const float* ring_v = p.ring_v + kvh * p.cap * HD;
  auto ev_slot = [&](int e) { return (st.head0 + e) % st.W; };

  // 1. the landmark numerators into shared memory (warps share the
  // landmarks, lanes over features) and eviction j = warp against every landmark
  for (int a = warp; a < m; a += nwarps)
#pragma unroll
    for (int c = 0; c < PER; ++c) {
      const int d4 = lane + 32 * c;
      if (d4 < D4)
        reinterpret_cast<float4*>(th_s + a * HD)[d4] =
            reinterpret_cast<const float4*>(p.t_hat + (ghi * m + a) * HD)[d4];
    }
  for (int j = warp; j < n_ev; j += nwarps) {
    float acc = 0.f;
    if (live) {
      const float* qt = p.q_tilde + (ghi * m + lane) * HD;
      const float* kj = ring_k + (size_t)ev_slot(j) * HD;
#pragma unroll 8
      for (int d4 = 0; d4 < D4; ++d4) {
        const float4 x = *reinterpret_cast<const float4*>(qt + d4 * 4);
        const float4 y = *reinterpret_cast<const float4*>(kj + d4 * 4);
        acc += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
      }
    }
    fe_s[j * 32 + lane] = acc * p.scale;
  }
  __syncthreads();

  // 2. every warp: the chunk's max per landmark and the rescale; warp 0 turns
  // the scores into e_j (shared) and keeps rr for the commit
  float mx = live ? mz[lane] : 0.f;
  const float z = live ? mz[m + lane] : 0.f;
  float mx2 = mx;
  for (int j = 0; j < n_ev; ++j) mx2 = fmaxf(mx2, fe_s[j * 32 + lane]);
  const float rr = (!live || mx2 == mx) ? 1.f : expf(mx - mx2);   // an empty landmark (-inf) gives 0
  mx = mx2;
  __syncthreads();                                      // every warp has read the raw scores
  if (warp == 0) {
    for (int j = 0; j < n_ev; ++j) fe_s[j * 32 + lane] = live ? expf(fe_s[j * 32 + lane] - mx) : 0.f;
    rr_s[lane] = rr;
  }
  __syncthreads();                                      // fe_s holds e_j
  const float z_base = z * rr;

  // 3. row i = warp: landmark weights, gains, far mass, numerator
  for (int i = warp; i < t; i += nwarps) {
    int n_i = i - j0 + 1;                               // evictions of rows 0..i
    n_i = n_i < 0 ? 0 : (n_i > n_ev ? n_ev : n_i);
    float fm = -INFINITY, far_den = 0.f, gain = 0.f;
    bool have = false;
    if (meta.far_len + (uint32_t)n_i > 0u) {
      float fs = -INFINITY;
      if (live) {
        const float* q = p.q + (((size_t)b * t + i) * p.nh + h) * HD;
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
      // w_b = sum_a exp(fs_a - f) mu[a][b]: the lane's column of mu, 8 rows in flight
      const float* mu = p.mu + ghi * m * m;
      float w = 0.f;
      for (int a0 = 0; a0 < m; a0 += 8) {
        float mu8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mu8[k] = (live && a0 + k < m) ? mu[(a0 + k) * m + lane] : 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) w += __shfl_sync(kFFull, ea, (a0 + k) & 31) * mu8[k];
      }
      if (p.far_rect) w = fmaxf(w, 0.f);
      const float fb = live ? f + mx : -INFINITY;
      fm = warp_max(fb);
      gain = (live && fm != -INFINITY) ? w * expf(fb - fm) : 0.f;
      float zi = z_base;
      for (int j = 0; j < n_i; ++j) zi += live ? fe_s[j * 32 + lane] : 0.f;
      far_den = warp_sum(gain * zi);
      have = fm != -INFINITY && far_den >= 0.f;          // a NaN or negative mass drops the far part
      if (!have) {
        far_den = 0.f;
        gain = 0.f;
      }
    }
    float4 num[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c) num[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (have) {
      const float grr = gain * rr;
      for (int a = 0; a < m; ++a) {
        const float ga = __shfl_sync(kFFull, grr, a);
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          const int d4 = lane + 32 * c;
          if (d4 < D4) {
            const float4 ta = reinterpret_cast<const float4*>(th_s + a * HD)[d4];
            num[c].x += ga * ta.x; num[c].y += ga * ta.y; num[c].z += ga * ta.z; num[c].w += ga * ta.w;
          }
        }
      }
      for (int j = 0; j < n_i; ++j) {
        const float cf = warp_sum(gain * (live ? fe_s[j * 32 + lane] : 0.f));   // eviction j's weight
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
    float* rec = p.ws_far + (((size_t)b * t + i) * p.nh + h) * (4 + HD);
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

  // 4. the commit: every eviction into the landmark numerators (warps share
  // the landmarks, lanes over features), the max and the mass
  if (p.commit && n_ev > 0) {
    for (int a = warp; a < m; a += nwarps) {
      const float ra = rr_s[a];
      float4 tv[PER];
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = lane + 32 * c;
        tv[c] = d4 < D4 ? reinterpret_cast<const float4*>(th_s + a * HD)[d4] : make_float4(0.f, 0.f, 0.f, 0.f);
        tv[c].x *= ra; tv[c].y *= ra; tv[c].z *= ra; tv[c].w *= ra;
      }
      for (int j = 0; j < n_ev; ++j) {
        const float ej = fe_s[j * 32 + a];
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
    if (warp == 0 && live) {
      float zf = z_base;
      for (int j = 0; j < n_ev; ++j) zf += fe_s[j * 32 + lane];
      mz[lane] = mx;
      mz[m + lane] = zf;
    }
  }
}

template <int HD, int MAXW>
int run_far_w(const AttendParams& p, dim3 grid, dim3 block, size_t smem, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(far_kernel<HD, MAXW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)((32 * HD + kFarRows * 32 + 32) * sizeof(float)));
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  far_kernel<HD, MAXW><<<grid, block, smem, s>>>(p);
  return finish_launch(cudaSuccess);
}

// blocks of up to 8 warps get the full register budget; longer chunks up to 32
// warps (a warp takes rows warp and warp + 32 of a chunk longer than 32)
template <int HD>
int run_far(const AttendParams& p, dim3 grid, dim3 block, size_t smem, cudaStream_t s) {
  return p.t <= 8 ? run_far_w<HD, 8>(p, grid, block, smem, s) : run_far_w<HD, 32>(p, grid, block, smem, s);
}

}  // namespace

int launch_far(const AttendParams& p, cudaStream_t s) {
  const dim3 grid((unsigned)(p.B * p.nh));               // a CTA per (sequence, query head)
  const dim3 block((unsigned)(32 * (p.t < 32 ? p.t : 32)));   // a warp per chunk row, at most 32
  const size_t smem = ((size_t)p.far_m * p.hd + kFarRows * 32 + 32) * sizeof(float);
  // An ordinary launch (after the prep in full stream order): launched
  // programmatically, its CTAs were resident early and the step was slower
  // (237.5 vs 210 us on batched_decode_far). It still triggers its dependents,
  // so the attention's CTAs are scheduled during its tail.
  switch (p.hd) {
    case 64: return run_far<64>(p, grid, block, smem, s);
    case 128: return run_far<128>(p, grid, block, smem, s);
    case 256: return run_far<256>(p, grid, block, smem, s);
    default: return SWA_E_SHAPE;
  }
}

}  // namespace swa
