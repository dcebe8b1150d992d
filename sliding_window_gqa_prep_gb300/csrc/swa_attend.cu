// Attend stage, second half: dispatch of the attention kernels and the
// reduction of their split records ("o1c_msl.metal", cortiq-engine 0.8.79:
// o1c_add, o1c_tok_merge, o1c_ring_commit, o1c_meta; "dory_msl.metal",
// cortiq-engine 0.8.57: dory_gate).
//
// The attention of a row block runs in one of three kernels, chosen by the
// number of query vectors (rows x query heads of a KV head) a CTA serves:
//   <= 8       attend_decode_kernel (swa_decode.cu), HBM-bound;
//   16 or 32   attend_verify_kernel (swa_verify.cu), FP32-bound;
//   64         attend_prompt_kernel (swa_prompt.cu), mma.sync TF32 (3xTF32);
//   128        attend_prompt_tc_kernel (swa_prompt_tc.cu), tcgen05 + TMEM (3xTF32).
// Each writes, per (sequence, KV head, row block, split) and query vector, a
// record (m in log2 units, l, unnormalised numerator). attend_merge_kernel
// then takes, per output (b, row, head, 4 features), the max over the valid
// splits, the rescaled sums of l and of the numerators, o = acc / den and the
// sigmoid gate; its trailing CTAs commit the chunk into the ring and advance
// the meta, after every read of the ring (stream order).
#include "swa_internal.cuh"

#include <cfloat>

namespace swa {
namespace {

// One output row (b, r, h) by a whole CTA of 8 warps: every warp finds the
// max over the valid splits, warp w adds the rescaled records of splits
// w, w + 8, ... (lanes over features), and the CTA sums the 8 partials.
template <int HD, bool BATCH>
__device__ void merge_row_wide(const AttendParams& p, unsigned blk) {
  constexpr int D4 = HD / 4;
  constexpr int PER = (D4 + 31) / 32;
  __shared__ float4 s_acc[8][D4];
  __shared__ float s_den[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t row = blk;                    // (b * t + r) * nh + h (< 2^31)
  if (row >= (uint32_t)p.B * p.t * p.nh) return;
  const int h = (int)(row % (uint32_t)p.nh);
  const uint32_t br = row / (uint32_t)p.nh;
  const int r = (int)(br % (uint32_t)p.t);
  const int b = (int)(br / (uint32_t)p.t);
  const int g = h / p.hpg;
  const int rb = r / p.rows;
  const int q = (r - rb * p.rows) * p.hpg + (h - g * p.hpg);
  const size_t item0 = (((size_t)b * p.nk + g) * p.n_rb + rb) * p.splits;
  // the gate of the features this thread writes at the end, loaded up front
  float4 gt = make_float4(0.f, 0.f, 0.f, 0.f), gs = gt;
  if ((int)threadIdx.x < D4) {
    gt = *reinterpret_cast<const float4*>(p.gate + (size_t)row * HD + threadIdx.x * 4);
    gs = *reinterpret_cast<const float4*>(p.gate_scale + (size_t)h * HD + threadIdx.x * 4);
  }
  const int nval = p.ws_nsplit[b * p.n_rb + rb];
  float M = -INFINITY;
  for (int s0 = lane; s0 < nval; s0 += 32) M = fmaxf(M, p.ws_ml[(item0 + s0) * p.nq + q].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float* far_rec = p.far ? p.ws_far + (((size_t)b * p.t + r) * p.nh + h) * (4 + HD) : nullptr;
  const bool far_on = far_rec && far_rec[2] > 0.5f;
  if (far_on) M = fmaxf(M, far_rec[0]);
  float4 acc[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if constexpr (BATCH) {
    // each warp's splits warp, warp + 8, ... eight at a time with every load in flight
    // (the same order of additions as one at a time)
    constexpr int KW = 8;
    for (int sp0 = warp; sp0 < nval; sp0 += 8 * KW) {
      float2 mlk[KW];
      float4 ak[KW][PER];
#pragma unroll
      for (int kk = 0; kk < KW; ++kk) {
        const int sp = sp0 + 8 * kk;
        const bool ok = sp < nval;
        mlk[kk] = ok ? p.ws_ml[(item0 + sp) * p.nq + q] : make_float2(-INFINITY, 0.f);
        const float* src = p.ws_acc + ((item0 + sp) * p.nq + q) * (size_t)HD;
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          const int d4 = c * 32 + lane;
          ak[kk][c] = (ok && d4 < D4) ? *reinterpret_cast<const float4*>(src + d4 * 4)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int kk = 0; kk < KW; ++kk) {
        if (mlk[kk].x == -INFINITY) continue;      // a split with no key of this row weighs 0
        const float w = exp2f(mlk[kk].x - M);
        den += mlk[kk].y * w;
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          acc[c].x += ak[kk][c].x * w; acc[c].y += ak[kk][c].y * w; acc[c].z += ak[kk][c].z * w;
          acc[c].w += ak[kk][c].w * w;
        }
      }
    }
  } else {
#pragma unroll 4
    for (int sp = warp; sp < nval; sp += 8) {
      const float2 ml = p.ws_ml[(item0 + sp) * p.nq + q];
      if (ml.x == -INFINITY) continue;            // a split with no key of this row weighs 0
      const float w = exp2f(ml.x - M);
      den += ml.y * w;
      const float* src = p.ws_acc + ((item0 + sp) * p.nq + q) * (size_t)HD;
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        const int d4 = c * 32 + lane;
        if (d4 < D4) {
          const float4 a = *reinterpret_cast<const float4*>(src + d4 * 4);
          acc[c].x += a.x * w; acc[c].y += a.y * w; acc[c].z += a.z * w; acc[c].w += a.w * w;
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < PER; ++c) {
    const int d4 = c * 32 + lane;
    if (d4 < D4) s_acc[warp][d4] = acc[c];
  }
  if (lane == 0) s_den[warp] = den;
  __syncthreads();
  if ((int)threadIdx.x < D4) {
    const int d4 = threadIdx.x;
    float4 t = s_acc[0][d4];
    float dsum = s_den[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
      const float4 a = s_acc[w][d4];
      t.x += a.x; t.y += a.y; t.z += a.z; t.w += a.w;
      dsum += s_den[w];
    }
    if (far_on) {
      const float sf = exp2f(far_rec[0] - M);
      const float4 a = *reinterpret_cast<const float4*>(far_rec + 4 + d4 * 4);
      t.x += a.x * sf; t.y += a.y * sf; t.z += a.z * sf; t.w += a.w * sf;
      dsum += far_rec[1] * sf;
    }
    const float inv = 1.0f / dsum;
    float4 o;
    o.x = gated(t.x, inv, gt.x, gs.x);
    o.y = gated(t.y, inv, gt.y, gs.y);
    o.z = gated(t.z, inv, gt.z, gs.z);
    o.w = gated(t.w, inv, gt.w, gs.w);
    *reinterpret_cast<float4*>(p.out + (size_t)row * HD + d4 * 4) = o;
  }
}

// Elementwise merge for calls with S <= 4 splits and no far field: a thread per
// (output row, 4 features), kMergeVec of them per thread with all their loads
// in flight at once; each thread takes the max over the row's valid splits, the
// rescaled sums and the gate itself (the (m, l) and split-count reads of the 32
// threads of a row are broadcasts). With one split this is bit-identical to the
// warp path (the weight is exp2(0) = 1).
constexpr int kMergeVec = 2;
constexpr int kMergeFewSplits = 4;

template <int HD, int S>
__device__ __forceinline__ void merge_elementwise(const AttendParams& p, unsigned blk) {
  // 32-bit index math: the host takes this path only when the element count fits
  constexpr int D4 = HD / 4;
  const uint32_t total = (uint32_t)p.B * p.t * p.nh * D4;
  const uint32_t base = blk * blockDim.x * kMergeVec + threadIdx.x;
  float4 gt[kMergeVec], gs[kMergeVec], a[kMergeVec][S];
  float2 ml[kMergeVec][S];
  int nval[kMergeVec];
#pragma unroll
  for (int k = 0; k < kMergeVec; ++k) {
    const uint32_t idx = base + k * blockDim.x;
    nval[k] = 0;
    if (idx >= total) continue;
    const uint32_t row = idx / D4;                   // (b * t + r) * nh + h
    const int d4 = (int)(idx % D4);
    const int h = (int)(row % (uint32_t)p.nh);
    const uint32_t br = row / (uint32_t)p.nh;
    const int r = (int)(br % (uint32_t)p.t);
    const int b = (int)(br / (uint32_t)p.t);
    const int g = h / p.hpg;
    const int rb = r / p.rows;
    const int q = (r - rb * p.rows) * p.hpg + (h - g * p.hpg);
    const size_t item0 = (((size_t)b * p.nk + g) * p.n_rb + rb) * S;
    nval[k] = p.ws_nsplit[b * p.n_rb + rb];
    gt[k] = *reinterpret_cast<const float4*>(p.gate + (size_t)row * HD + d4 * 4);
    gs[k] = *reinterpret_cast<const float4*>(p.gate_scale + (size_t)h * HD + d4 * 4);
    // every split's record is allocated: read them all, use the valid ones
#pragma unroll
    for (int sp = 0; sp < S; ++sp) {
      ml[k][sp] = p.ws_ml[(item0 + sp) * p.nq + q];
      a[k][sp] = *reinterpret_cast<const float4*>(p.ws_acc + ((item0 + sp) * p.nq + q) * (size_t)HD + d4 * 4);
    }
  }
#pragma unroll
  for (int k = 0; k < kMergeVec; ++k) {
    const uint32_t idx = base + k * blockDim.x;
    if (idx >= total) continue;
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < S; ++sp)
      if (sp < nval[k]) M = fmaxf(M, ml[k][sp].x);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sp = 0; sp < S; ++sp) {
      if (sp < nval[k] && ml[k][sp].x != -INFINITY) {  // a split with no key of this row weighs 0
        const float w = exp2f(ml[k][sp].x - M);
        den += ml[k][sp].y * w;
        acc.x += a[k][sp].x * w; acc.y += a[k][sp].y * w; acc.z += a[k][sp].z * w; acc.w += a[k][sp].w * w;
      }
    }
    const float inv = 1.0f / den;
    float4 o;
    o.x = gated(acc.x, inv, gt[k].x, gs[k].x);
    o.y = gated(acc.y, inv, gt[k].y, gs[k].y);
    o.z = gated(acc.z, inv, gt[k].z, gs[k].z);
    o.w = gated(acc.w, inv, gt[k].w, gs[k].w);
    *reinterpret_cast<float4*>(p.out + (size_t)idx * 4) = o;
  }
}

// Commit of sequence b, spread over commit_blocks CTAs (cta = index among the
// trailing CTAs of a merge launch).
template <int HD>
__device__ void commit_chunk(const AttendParams& p, int cta) {
  // ---- commit of sequence b, spread over commit_blocks CTAs: the last
  // min(t, W) chunk rows into their ring slots (o1c_ring_commit), then the
  // meta (o1c_meta). The ring map comes from the copy of the meta the
  // attention kernel saved, so meta_out may alias meta.
  const int cb = cta % p.commit_blocks;
  const int b = cta / p.commit_blocks;
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
  if (cb == 0 && threadIdx.x == 0) p.meta_out[b] = advance_meta(m0, st, p.t);
}

// Merge of few split records (elementwise) + gate; trailing CTAs commit the chunk.
template <int HD, int S>
__global__ void __launch_bounds__(256) attend_merge_few_kernel(AttendParams p, int out_blocks) {
  pdl_trigger();
  pdl_wait();
  if ((int)blockIdx.x >= out_blocks) {
    commit_chunk<HD>(p, (int)blockIdx.x - out_blocks);
    return;
  }
  merge_elementwise<HD, S>(p, blockIdx.x);
}

// Merge of the split records + gate; trailing CTAs commit the chunk. With
// `wide`, one CTA per output row whose 8 warps share the splits (calls with
// many splits per row); otherwise one warp per output row.
// BATCH: the splits' numerators are loaded many at a time (calls with more than
// kMergeFewSplits splits, which have few rows); without it the kernel keeps far
// fewer registers, so that calls with many rows keep more CTAs resident.
template <int HD, bool BATCH>
__global__ void __launch_bounds__(256) attend_merge_kernel(AttendParams p, int out_blocks, int wide) {
  pdl_trigger();
  pdl_wait();
  if ((int)blockIdx.x >= out_blocks) {
    commit_chunk<HD>(p, (int)blockIdx.x - out_blocks);
    return;
  }
  if (wide) {
    merge_row_wide<HD, BATCH>(p, blockIdx.x);
    return;
  }
  // ---- one warp per output row (b, r, h): lane s of each group of 32 splits
  // takes that split's (m, l); the weights exp2(m_s - M) are broadcast and each
  // lane adds its features of every split's numerator (independent loads).
  constexpr int D4 = HD / 4;
  constexpr int PER = (D4 + 31) / 32;          // float4 chunks per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t row = blockIdx.x * (blockDim.x / 32) + warp;   // (b * t + r) * nh + h (< 2^31)
  if (row >= (uint32_t)p.B * p.t * p.nh) return;
  const int h = (int)(row % (uint32_t)p.nh);
  const uint32_t br = row / (uint32_t)p.nh;
  const int r = (int)(br % (uint32_t)p.t);
  const int b = (int)(br / (uint32_t)p.t);
  const int g = h / p.hpg;
  const int rb = r / p.rows;
  const int q = (r - rb * p.rows) * p.hpg + (h - g * p.hpg);
  const size_t item0 = (((size_t)b * p.nk + g) * p.n_rb + rb) * p.splits;
  // Loads that wait for nothing go out together: the gate and its scale, the
  // valid-split count, the (m, l) of split `lane` and the numerator of split 0
  // (every split's record is allocated, so reads past the valid splits stay in
  // bounds; split 0 always exists, a row sees at least its own key).
  float4 gt[PER], gs[PER], a0[PER];
  const float* src0 = p.ws_acc + (item0 * p.nq + q) * (size_t)HD;
#pragma unroll
  for (int c = 0; c < PER; ++c) {
    const int d4 = c * 32 + lane;
    if (d4 < D4) {
      gt[c] = *reinterpret_cast<const float4*>(p.gate + (size_t)row * HD + d4 * 4);
      gs[c] = *reinterpret_cast<const float4*>(p.gate_scale + (size_t)h * HD + d4 * 4);
      a0[c] = *reinterpret_cast<const float4*>(src0 + d4 * 4);
    }
  }
  const int nval = p.ws_nsplit[b * p.n_rb + rb];
  float2 ml0 = make_float2(-INFINITY, 0.f);
  if (lane < p.splits) ml0 = p.ws_ml[(item0 + lane) * p.nq + q];
  if (lane >= nval) ml0 = make_float2(-INFINITY, 0.f);
  float M = ml0.x;
  for (int s0 = 32; s0 < nval; s0 += 32)
    if (s0 + lane < nval) M = fmaxf(M, p.ws_ml[(item0 + s0 + lane) * p.nq + q].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  // the far part of a decode row joins under the common exponent (o1c_tok_merge)
  const float* far_rec = p.far ? p.ws_far + (((size_t)b * p.t + r) * p.nh + h) * (4 + HD) : nullptr;
  const bool far_on = far_rec && far_rec[2] > 0.5f;
  if (far_on) M = fmaxf(M, far_rec[0]);
  float den = 0.f;
  float4 acc[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < nval; s0 += 32) {
    float2 ml = ml0;
    if (s0 > 0) {
      ml = make_float2(-INFINITY, 0.f);
      if (s0 + lane < nval) ml = p.ws_ml[(item0 + s0 + lane) * p.nq + q];
    }
    float w = 0.f;
    if (ml.x != -INFINITY) {                   // a split with no key of this row weighs 0
      w = exp2f(ml.x - M);                     // (its numerator is 0, so 0 x it is exact)
      den += ml.y * w;
    }
    const int cnt = min(32, nval - s0);
    int k = 0;
    if (s0 == 0) {
      const float wk = __shfl_sync(0xffffffffu, w, 0);
#pragma unroll
      for (int c = 0; c < PER; ++c) {
        acc[c].x += a0[c].x * wk; acc[c].y += a0[c].y * wk; acc[c].z += a0[c].z * wk; acc[c].w += a0[c].w * wk;
      }
      k = 1;
    }
    if constexpr (BATCH) {
      // up to 16 splits' numerators in flight at once (a runtime trip count let the
      // compiler keep only a few loads ahead)
      constexpr int KB = 16;
      for (; k < cnt; k += KB) {
        float4 ak[KB][PER];
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
          const float* src = p.ws_acc + ((item0 + s0 + k + kk) * p.nq + q) * (size_t)HD;
#pragma unroll
          for (int c = 0; c < PER; ++c) {
            const int d4 = c * 32 + lane;
            ak[kk][c] = (k + kk < cnt && d4 < D4) ? *reinterpret_cast<const float4*>(src + d4 * 4)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
          const float wk = __shfl_sync(0xffffffffu, w, (k + kk) & 31);
          if (k + kk < cnt) {
#pragma unroll
            for (int c = 0; c < PER; ++c) {
              acc[c].x += ak[kk][c].x * wk; acc[c].y += ak[kk][c].y * wk;
              acc[c].z += ak[kk][c].z * wk; acc[c].w += ak[kk][c].w * wk;
            }
          }
        }
      }
    } else {
#pragma unroll 4
      for (; k < cnt; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        const float* src = p.ws_acc + ((item0 + s0 + k) * p.nq + q) * (size_t)HD;
#pragma unroll
        for (int c = 0; c < PER; ++c) {
          const int d4 = c * 32 + lane;
          if (d4 < D4) {
            const float4 a = *reinterpret_cast<const float4*>(src + d4 * 4);
            acc[c].x += a.x * wk; acc[c].y += a.y * wk; acc[c].z += a.z * wk; acc[c].w += a.w * wk;
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  if (far_on) {
    const float sf = exp2f(far_rec[0] - M);
    den += far_rec[1] * sf;
#pragma unroll
    for (int c = 0; c < PER; ++c) {
      const int d4 = c * 32 + lane;
      if (d4 < D4) {
        const float4 a = *reinterpret_cast<const float4*>(far_rec + 4 + d4 * 4);
        acc[c].x += a.x * sf; acc[c].y += a.y * sf; acc[c].z += a.z * sf; acc[c].w += a.w * sf;
      }
    }
  }
  const float inv = 1.0f / den;
#pragma unroll
  for (int c = 0; c < PER; ++c) {
    const int d4 = c * 32 + lane;
    if (d4 >= D4) continue;
    float4 o;
    o.x = gated(acc[c].x, inv, gt[c].x, gs[c].x);
    o.y = gated(acc[c].y, inv, gt[c].y, gs[c].y);
    o.z = gated(acc[c].z, inv, gt[c].z, gs[c].z);
    o.w = gated(acc[c].w, inv, gt[c].w, gs[c].w);
    *reinterpret_cast<float4*>(p.out + (size_t)row * HD + d4 * 4) = o;
  }
}

}  // namespace

int launch_attend_partial(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  if (p.nq <= 8) return launch_attend_decode(p, s, e0, e1);
  if (p.nq == 16 || p.nq == 32) return launch_attend_verify(p, s, e0, e1);
  if (p.nq == 64) return launch_attend_prompt(p, s, e0, e1);
  if (p.nq == 128) return p.ops ? launch_attend_prompt_h16(p, s, e0, e1) : launch_attend_prompt_tc(p, s, e0, e1);
  return SWA_E_SHAPE;
}

int attend_partial_occupancy(int hd, int nq) {
  if (nq <= 8) return attend_decode_occupancy(hd, nq);
  if (nq == 16 || nq == 32) return attend_verify_occupancy(hd, nq);
  return 1;
}

int launch_attend_merge(const AttendParams& p, cudaStream_t s) {
  const size_t rows = (size_t)p.B * p.t * p.nh;
  const int block = 256;
  // many splits per row: a CTA per row (8 warps share the splits); else a warp per row
  const int commit_ctas = p.commit ? p.B * p.commit_blocks : 0;
  const size_t elems = rows * (size_t)(p.hd / 4);
  if (!p.far && p.splits <= kMergeFewSplits && elems + (size_t)block * kMergeVec < (1ull << 32)) {
    // few splits, no far field: elementwise
    const size_t per_cta = (size_t)block * kMergeVec;
    const int out_blocks = (int)((rows * (size_t)(p.hd / 4) + per_cta - 1) / per_cta);
    const dim3 grid(out_blocks + commit_ctas);
#define SWA_FEW(HDV, SV) case HDV * 10 + SV: \
    return finish_launch(launch_pdl(attend_merge_few_kernel<HDV, SV>, grid, dim3(block), 0, s, p, out_blocks));
    switch (p.hd * 10 + p.splits) {
      SWA_FEW(64, 1) SWA_FEW(64, 2) SWA_FEW(64, 3) SWA_FEW(64, 4)
      SWA_FEW(128, 1) SWA_FEW(128, 2) SWA_FEW(128, 3) SWA_FEW(128, 4)
      SWA_FEW(256, 1) SWA_FEW(256, 2) SWA_FEW(256, 3) SWA_FEW(256, 4)
      default: return SWA_E_SHAPE;
    }
#undef SWA_FEW
  }
  // many splits: a CTA per row (8 warps share the splits); else a warp per row
  const int wide = p.splits >= 16 ? 1 : 0;
  const int out_blocks = wide ? (int)rows : (int)((rows + block / 32 - 1) / (block / 32));
  const int grid = out_blocks + commit_ctas;
  const bool batch = p.splits > kMergeFewSplits;
#define SWA_MERGE(HDV) case HDV: \
    return finish_launch(batch ? launch_pdl(attend_merge_kernel<HDV, true>, dim3(grid), dim3(block), 0, s, p, out_blocks, wide) \
                               : launch_pdl(attend_merge_kernel<HDV, false>, dim3(grid), dim3(block), 0, s, p, out_blocks, wide));
  switch (p.hd) {
    SWA_MERGE(64) SWA_MERGE(128) SWA_MERGE(256)
    default: return SWA_E_SHAPE;
  }
#undef SWA_MERGE
}

}  // namespace swa
