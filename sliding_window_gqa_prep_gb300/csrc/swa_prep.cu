// Prep stage: rotation, unit heads, query scale, ring write ("dory_msl.metal",
// cortiq-engine 0.8.57, kernel dory_prep), and the RoPE table it consumes.
//
// One CTA per row, one warp per head at a time: the q heads of a row come
// first, then its k heads (the same split of the head index as dory_prep).
// Lane l owns the hd/64 rotated pairs (e, e + hd/2) with e in
// [l*hd/64, (l+1)*hd/64), so both halves of a head are read and written as
// contiguous, coalesced vectors. The sum of squares is a butterfly over the
// warp. Every byte moves once. The row's angles, when the kernel computes
// them, cost f64 sine/cosine evaluations, which are slow on this GPU: one CTA
// per row evaluates them once for all of the row's heads (several rows per CTA,
// sharing the angle work, measured slower: fewer warps in flight).
#include "swa_internal.cuh"

namespace swa {
namespace {

template <int P> struct VecT;
template <> struct VecT<1> { using T = float; };
template <> struct VecT<2> { using T = float2; };
template <> struct VecT<4> { using T = float4; };

template <int P>
__device__ __forceinline__ void ldv(const float* p, float (&r)[P]) {
  typename VecT<P>::T v = *reinterpret_cast<const typename VecT<P>::T*>(p);
  const float* f = reinterpret_cast<const float*>(&v);
#pragma unroll
  for (int i = 0; i < P; ++i) r[i] = f[i];
}

template <int P>
__device__ __forceinline__ void stv(float* p, const float (&r)[P]) {
  typename VecT<P>::T v;
  float* f = reinterpret_cast<float*>(&v);
#pragma unroll
  for (int i = 0; i < P; ++i) f[i] = r[i];
  *reinterpret_cast<typename VecT<P>::T*>(p) = v;
}

constexpr int kPrepWarps = 8;
constexpr int kPrepBatch = 4;      // heads a warp loads before it stores any

// Inputs of one head: both halves of the rotated vector and, for a q head, both
// halves of its per-feature scale, for a k head both halves of its v row.
template <int HD>
struct HeadIn {
  float x[HD / 64], y[HD / 64], sa[HD / 64], sb[HD / 64];
};

template <int HD>
__device__ __forceinline__ void load_head(const PrepParams& p, int row, int a, int lane, HeadIn<HD>& in) {
  constexpr int P = HD / 64;
  constexpr int HALF = HD / 2;
  const int e = lane * P;
  if (a < p.nh) {
    const float* src = p.yq + ((size_t)row * p.nh + a) * HD;
    ldv<P>(src + e, in.x);
    ldv<P>(src + HALF + e, in.y);
    ldv<P>(p.q_scale + (size_t)a * HD + e, in.sa);
    ldv<P>(p.q_scale + (size_t)a * HD + HALF + e, in.sb);
  } else {
    const int kh = a - p.nh;
    const float* src = p.yk + ((size_t)row * p.nk + kh) * HD;
    ldv<P>(src + e, in.x);
    ldv<P>(src + HALF + e, in.y);
    if (p.v_out || p.ring_k) {
      const float* vs = p.yv + ((size_t)row * p.nk + kh) * HD;
      ldv<P>(vs + e, in.sa);
      ldv<P>(vs + HALF + e, in.sb);
    }
  }
}

// One head of one row: rotation, unit norm, query scale / ring write (to `slot`).
template <int HD>
__device__ __forceinline__ void prep_head(const PrepParams& p, int row, int a, int lane, uint32_t slot,
                                          const float (&c)[HD / 64], const float (&s)[HD / 64],
                                          const HeadIn<HD>& in) {
  constexpr int P = HD / 64;
  constexpr int HALF = HD / 2;
  const int e = lane * P;
  float u[P], v[P];
  const float inv = rotate_unit<P>(in.x, in.y, c, s, p.eps, u, v);

  if (a < p.nh) {
#pragma unroll
    for (int i = 0; i < P; ++i) {
      u[i] = u[i] * inv * in.sa[i];
      v[i] = v[i] * inv * in.sb[i];
    }
    float* dst = p.q_out + ((size_t)row * p.nh + a) * HD;
    stv<P>(dst + e, u);
    stv<P>(dst + HALF + e, v);
    return;
  }
  const int kh = a - p.nh;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    u[i] *= inv;
    v[i] *= inv;
  }
  float* kd = p.k_out + ((size_t)row * p.nk + kh) * HD;
  stv<P>(kd + e, u);
  stv<P>(kd + HALF + e, v);
  if (p.v_out) {
    float* vd = p.v_out + ((size_t)row * p.nk + kh) * HD;
    stv<P>(vd + e, in.sa);
    stv<P>(vd + HALF + e, in.sb);
  }
  if (p.ring_k) {
    const int b = row / p.t;
    const size_t at = (((size_t)b * p.nk + kh) * p.cap + slot) * HD;
    stv<P>(p.ring_k + at + e, u);
    stv<P>(p.ring_k + at + HALF + e, v);
    stv<P>(p.ring_v + at + e, in.sa);
    stv<P>(p.ring_v + at + HALF + e, in.sb);
  }
}

template <int HD>
__global__ void __launch_bounds__(kPrepWarps * 32) prep_kernel(PrepParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int P = HD / 64;       // pairs per lane
  constexpr int HALF = HD / 2;
  const int row = blockIdx.x;      // b * t + j
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = row / p.t, j = row % p.t;
  // heads a = warp, warp + kPrepWarps, ...: q heads first, then k heads (the
  // head split of dory_prep); kPrepBatch heads' inputs are in flight at once.
  // The first batch is requested before the angles are evaluated, so its load
  // latency overlaps them.
  const int nheads = p.nh + p.nk;
  HeadIn<HD> in[kPrepBatch];
  auto load_batch = [&](int a0) {
#pragma unroll
    for (int k = 0; k < kPrepBatch; ++k) {
      const int a = a0 + k * kPrepWarps;
      if (a < nheads) load_head<HD>(p, row, a, lane, in[k]);
    }
  };
  load_batch(warp);
  const bool need_pos = p.rope == nullptr || p.ring_k != nullptr;
  const uint64_t pos = need_pos ? (uint64_t)p.pos0[b] + (uint64_t)j : 0;
  const uint32_t slot = p.ring_k ? (uint32_t)(pos % (uint64_t)p.cap) : 0u;
  // Without a table, the row's cos/sin are computed once per CTA (the CTA
  // covers every head of the row), with the same f64 expression as
  // rope_table_kernel (bit-identical f32 values).
  __shared__ __align__(16) float s_cs[HD];
  if (p.rope == nullptr) {
    for (int e2 = threadIdx.x; e2 < HALF; e2 += blockDim.x) {
      double sn, cs;
      sincos((double)pos * p.inv_freq[e2], &sn, &cs);
      s_cs[e2] = (float)cs;
      s_cs[HALF + e2] = (float)sn;
    }
    __syncthreads();
  }
  const int e = lane * P;
  float c[P], s[P];
  const float* rope = p.rope ? p.rope + (size_t)row * HD : s_cs;
  ldv<P>(rope + e, c);
  ldv<P>(rope + HALF + e, s);

  for (int a0 = warp; a0 < nheads; a0 += kPrepWarps * kPrepBatch) {
    if (a0 != warp) load_batch(a0);
#pragma unroll
    for (int k = 0; k < kPrepBatch; ++k) {
      const int a = a0 + k * kPrepWarps;
      if (a < nheads) prep_head<HD>(p, row, a, lane, slot, c, s, in[k]);
    }
  }
}

struct RopeFreq {
  double inv_freq[128];
};

// One thread per (row, pair e): angle in f64 from the absolute position and the
// host-computed frequency theta^(-2e/hd); cos/sin in f64, stored as f32.
__global__ void rope_table_kernel(float* rope, const uint32_t* pos0, int B, int t, int hd,
                                  RopeFreq f) {
  const int half = hd / 2;
  const size_t n = (size_t)B * t * half;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(idx % half);
    const size_t r = idx / half;
    const int b = (int)(r / t), j = (int)(r % t);
    const double pos = (double)pos0[b] + (double)j;
    double sn, cs;
    sincos(pos * f.inv_freq[e], &sn, &cs);
    rope[r * hd + e] = (float)cs;
    rope[r * hd + half + e] = (float)sn;
  }
}

}  // namespace

int launch_prep(const PrepParams& p, cudaStream_t s) {
  dim3 grid((unsigned)(p.B * p.t));
  dim3 block(kPrepWarps * 32);
  switch (p.hd) {
    case 64: return finish_launch(launch_pdl(prep_kernel<64>, grid, block, 0, s, p));
    case 128: return finish_launch(launch_pdl(prep_kernel<128>, grid, block, 0, s, p));
    case 256: return finish_launch(launch_pdl(prep_kernel<256>, grid, block, 0, s, p));
    default: return SWA_E_SHAPE;
  }
}

int launch_rope_table(float* rope, const uint32_t* pos0, int B, int t, int hd,
                      const double* inv_freq, cudaStream_t s) {
  RopeFreq f;
  for (int e = 0; e < 128; ++e) f.inv_freq[e] = e < hd / 2 ? inv_freq[e] : 0.0;
  const size_t n = (size_t)B * t * (hd / 2);
  const int block = 256;
  const size_t want = (n + block - 1) / block;
  const unsigned grid = (unsigned)(want < 4096 ? (want ? want : 1) : 4096);
  rope_table_kernel<<<grid, block, 0, s>>>(rope, pos0, B, t, hd, f);
  note_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace swa
