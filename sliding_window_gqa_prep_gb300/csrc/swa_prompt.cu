// Prompt-chunk attention on tensor cores: the GEMM path of "o1c_msl.metal"
// (cortiq-engine 0.8.79: o1c_gather, o1c_cols, o1c_gmax, o1c_gsoft, o1c_gadd
// and the engine GEMMs Q K^T and P V they feed), as one flash-style kernel per
// row block, without materialising the gathered key panel.
//
// A CTA takes 64 query vectors (rows x query heads of one KV head: 16 rows
// for 4 heads per KV head) and streams the block's key range (sinks, then the
// logical keys [lo(r0), len0 + r_last] from the ring slot (head0 + x) % W or
// the chunk row x - len0) through 3 shared-memory tiles of 32 keys, filled
// with cp.async (per-row source addresses, so the ring wrap lives in the
// address map). Each of 4 warps owns 16 query vectors:
//   S = Q K^T with mma.sync m16n8k8 TF32, split three ways for f32 accuracy:
//       a = a_hi + a_lo (a_hi = a rounded to TF32, a_lo = the rest rounded to
//       TF32); a b ~ a_hi b_hi + a_hi b_lo + a_lo b_hi, accumulated in f32
//       (the dropped a_lo b_lo term is ~2^-22 of the product);
//   the per-row window mask, an online max / exp2 / sum on the accumulator
//   fragments (scores carry scale * log2 e), the rescale of O;
//   O += P V with the same 3-way split (P through a per-warp shared slice).
// The CTA writes one partial record (m, l, O) per query vector, which the
// merge kernel normalises, gates and commits like every other path.
#include "swa_internal.cuh"

namespace swa {
namespace {

constexpr int kPW = 4;                 // warps
constexpr int kPThreads = kPW * 32;
constexpr int kPTK = 32;               // keys per tile
constexpr int kPStages = 3;
constexpr unsigned kFullMask = 0xffffffffu;

template <int HD>
struct PCfg {
  static constexpr int KP = HD + 4;     // K row stride: B-fragment reads (key g, feature t) hit bank 4g + t
  static constexpr int VP = HD + 8;     // V row stride: B-fragment reads (key t, feature g) hit bank 8t + g
  static constexpr int PP = kPTK + 4;   // P row stride: A-fragment reads (row g, key t) hit bank 4g + t
  static constexpr int KS = HD / 8;     // k-steps of Q K^T
  static constexpr int NB = HD / 8;     // n-blocks of P V
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + kPStages * kPTK * KP;
  static constexpr int OFF_P = OFF_V + kPStages * kPTK * VP;
  static constexpr int FLOATS = OFF_P + kPW * 16 * PP;
  static constexpr size_t BYTES = (size_t)FLOATS * 4;
};

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// x = hi + lo with both parts representable in TF32
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// three-term product accumulation: d += a_hi b_hi + a_hi b_lo + a_lo b_hi
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                     uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  mma_tf32(d, al, bh0, bh1);
  mma_tf32(d, ah, bl0, bl1);
  mma_tf32(d, ah, bh0, bh1);
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool fill) {
  const uint32_t bytes = fill ? 16u : 0u;     // 0: zero-fill the 16 bytes
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(smem_u32(dst)), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <int HD>
__global__ void __launch_bounds__(kPThreads, 2) attend_prompt_kernel(AttendParams p) {
  pdl_trigger();
  pdl_wait();
  using C = PCfg<HD>;
  extern __shared__ __align__(128) float smem[];
  float* Ks = smem + C::OFF_K;
  float* Vs = smem + C::OFF_V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;     // mma fragment coordinates
  float* Pw = smem + C::OFF_P + warp * 16 * C::PP;

  const int rb = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.nk, g = bg % p.nk;
  const SeqState st = load_state(p, b, tid == 0 && g == 0 && rb == 0);
  const int r0 = rb * p.rows;
  const int r_last = min(r0 + p.rows, p.t) - 1;
  const int rows_eff = r_last - r0 + 1;
  const int win0 = min(st.W, st.len0 + r0 + 1);
  const int xlo = st.len0 + r0 + 1 - win0;
  const int n = p.ns + (st.len0 + r_last - xlo + 1);
  if (g == 0 && tid == 0) p.ws_nsplit[b * p.n_rb + rb] = 1;
  if (g == 0 && rb == 0 && tid == 0) p.ws_meta[b] = p.meta[b];
  const int ntiles = (n + kPTK - 1) / kPTK;
  const size_t kv_head = (size_t)b * p.nk + g;

  // cp.async of tile i: 32 rows x HD floats of K and of V, 16 bytes per copy
  auto issue = [&](int i) {
    const int stage = i % kPStages;
    constexpr int per_row = HD / 4;
    for (int idx = tid; idx < kPTK * per_row; idx += kPThreads) {
      const int k = idx / per_row, c4 = idx % per_row;
      const int j = i * kPTK + k;
      const bool in = j < n;
      const float* sk = p.q;          // any valid address when zero-filling
      const float* sv = p.q;
      if (in) {
        size_t at;
        if (j < p.ns) {
          at = (kv_head * p.ns + j) * HD;
          sk = p.sink_k + at;
          sv = p.sink_v + at;
        } else {
          const int x = xlo + (j - p.ns);
          if (x < st.len0) {
            int slot = st.head0 + x;
            if (slot >= st.W) slot -= st.W;
            at = (kv_head * p.cap + (size_t)slot) * HD;
            sk = p.ring_k + at;
            sv = p.ring_v + at;
          } else {
            at = (((size_t)b * p.t + (x - st.len0)) * p.nk + g) * HD;
            sk = p.k_chunk + at;
            sv = p.v_chunk + at;
          }
        }
      }
      cp_async16(Ks + ((size_t)stage * kPTK + k) * C::KP + c4 * 4, sk + c4 * 4, in);
      cp_async16(Vs + ((size_t)stage * kPTK + k) * C::VP + c4 * 4, sv + c4 * 4, in);
    }
  };
  issue(0);
  cp_async_commit();
  if (ntiles > 1) issue(1);
  cp_async_commit();

  // Q fragments of this warp's 16 query vectors (rows qa = warp*16 + gq and
  // qa + 8), kept in f32 and multiplied by scale * log2 e.
  float qf[C::KS][4];
  int qrow[2];
  bool qvalid[2];
  int qlo[2], qhi[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int q = warp * 16 + gq + 8 * hh;
    const int rr = q / p.hpg, h = q % p.hpg;
    qvalid[hh] = rr < rows_eff && q < p.rows * p.hpg;
    const int r = r0 + rr;
    qrow[hh] = r;
    qlo[hh] = st.len0 + r + 1 - min(st.W, st.len0 + r + 1);
    qhi[hh] = st.len0 + r;
    const float* src = p.q + (((size_t)b * p.t + r) * p.nh + (size_t)g * p.hpg + h) * HD;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      qf[ks][hh] = qvalid[hh] ? src[ks * 8 + tq] * p.qmul : 0.f;
      qf[ks][2 + hh] = qvalid[hh] ? src[ks * 8 + tq + 4] * p.qmul : 0.f;
    }
  }
  // fragment register order: a0 (row g, col t), a1 (row g+8, col t), a2 (row g, col t+4), a3 (row g+8, col t+4)
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[C::NB][4];
#pragma unroll
  for (int nb = 0; nb < C::NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;

  for (int i = 0; i < ntiles; ++i) {
    const int stage = i % kPStages;
    cp_async_wait_1();
    __syncthreads();   // tile i visible to all; every warp is done with tile i-1
    if (i + 2 < ntiles) issue(i + 2);
    cp_async_commit();
    const float* Kt = Ks + (size_t)stage * kPTK * C::KP;
    const float* Vt = Vs + (size_t)stage * kPTK * C::VP;

    // ---- S (16 x 32) = Q K^T
    float s[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      uint32_t ah[4], al[4];
      // a0 = (g, t), a1 = (g+8, t), a2 = (g, t+4), a3 = (g+8, t+4)
      split_tf32(qf[ks][0], ah[0], al[0]);
      split_tf32(qf[ks][1], ah[1], al[1]);
      split_tf32(qf[ks][2], ah[2], al[2]);
      split_tf32(qf[ks][3], ah[3], al[3]);
#pragma unroll
      for (int nb = 0; nb < 4; ++nb) {
        const float* kr = Kt + (size_t)(nb * 8 + gq) * C::KP + ks * 8 + tq;
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(kr[0], bh0, bl0);
        split_tf32(kr[4], bh1, bl1);
        mma3(s[nb], ah, al, bh0, bh1, bl0, bl1);
      }
    }
    // ---- mask, online softmax on the fragments (rows gq and gq + 8)
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hh = e >> 1;
        const int j = i * kPTK + nb * 8 + 2 * tq + (e & 1);
        bool v = qvalid[hh] && j < n;
        if (v && j >= p.ns) {
          const int x = xlo + (j - p.ns);
          v = x >= qlo[hh] && x <= qhi[hh];
        }
        s[nb][e] = v ? s[nb][e] : -INFINITY;
        tmax[hh] = fmaxf(tmax[hh], s[nb][e]);
      }
    }
    float corr[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(kFullMask, tmax[hh], 1));
      tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(kFullMask, tmax[hh], 2));
      const float m_new = fmaxf(m_run[hh], tmax[hh]);
      corr[hh] = m_new == -INFINITY ? 1.f : exp2f(m_run[hh] - m_new);
      m_run[hh] = m_new;
    }
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hh = e >> 1;
        const float pv = m_run[hh] == -INFINITY ? 0.f : exp2f(s[nb][e] - m_run[hh]);
        psum[hh] += pv;
        Pw[(gq + 8 * hh) * C::PP + nb * 8 + 2 * tq + (e & 1)] = pv;
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) l_run[hh] = l_run[hh] * corr[hh] + psum[hh];
#pragma unroll
    for (int nb = 0; nb < C::NB; ++nb) {
      o[nb][0] *= corr[0]; o[nb][1] *= corr[0];
      o[nb][2] *= corr[1]; o[nb][3] *= corr[1];
    }
    __syncwarp();

    // ---- O (16 x HD) += P (16 x 32) V (32 x HD)
#pragma unroll
    for (int ks = 0; ks < kPTK / 8; ++ks) {
      uint32_t ah[4], al[4];
      split_tf32(Pw[gq * C::PP + ks * 8 + tq], ah[0], al[0]);
      split_tf32(Pw[(gq + 8) * C::PP + ks * 8 + tq], ah[1], al[1]);
      split_tf32(Pw[gq * C::PP + ks * 8 + tq + 4], ah[2], al[2]);
      split_tf32(Pw[(gq + 8) * C::PP + ks * 8 + tq + 4], ah[3], al[3]);
      const float* v0 = Vt + (size_t)(ks * 8 + tq) * C::VP + gq;
      const float* v1 = v0 + 4 * C::VP;
#pragma unroll
      for (int nb = 0; nb < C::NB; ++nb) {
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(v0[nb * 8], bh0, bl0);
        split_tf32(v1[nb * 8], bh1, bl1);
        mma3(o[nb], ah, al, bh0, bh1, bl0, bl1);
      }
    }
    __syncwarp();      // P slice is rewritten by the next tile
  }
  cp_async_wait_0();

  // ---- partial record: m, l (summed over the 4 lanes of a row), O unnormalised
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(kFullMask, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(kFullMask, l_run[hh], 2);
  }
  const size_t item = ((size_t)bg * p.n_rb + rb) * p.splits;
  float* wacc = p.ws_acc + item * (size_t)p.nq * HD;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int q = warp * 16 + gq + 8 * hh;
    float* dst = wacc + (size_t)q * HD;
#pragma unroll
    for (int nb = 0; nb < C::NB; ++nb)
      *reinterpret_cast<float2*>(dst + nb * 8 + 2 * tq) = make_float2(o[nb][2 * hh], o[nb][2 * hh + 1]);
    if (tq == 0) p.ws_ml[item * p.nq + q] = make_float2(m_run[hh], l_run[hh]);
  }
}

template <int HD>
int launch_prompt_t(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = PCfg<HD>;
  auto kern = attend_prompt_kernel<HD>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  dim3 grid(1u, (unsigned)p.n_rb, (unsigned)(p.B * p.nk));
  if (e0) cudaEventRecord(e0, s);
  cudaError_t e = launch_pdl(kern, grid, dim3(kPThreads), C::BYTES, s, p);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e1) cudaEventRecord(e1, s);
  return cuda_status(e);
}

}  // namespace

int launch_attend_prompt(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  switch (p.hd) {
    case 64: return launch_prompt_t<64>(p, s, e0, e1);
    case 128: return launch_prompt_t<128>(p, s, e0, e1);
  }
  return SWA_E_SHAPE;
}

}  // namespace swa
