// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>

#include "swa.h"

namespace swa {

// ---------------------------------------------------------------------------
// Launch bookkeeping (swa_api.cu)
// ---------------------------------------------------------------------------
void note_launch(int n = 1);
int cuda_status(cudaError_t e);   // records the error text, returns SWA_E_CUDA / SWA_OK
int num_sms();                    // SM count of the current device (cached per device)

// ---------------------------------------------------------------------------
// Attention plan: how a call is cut into CTAs (host side, swa_api.cu).
// ---------------------------------------------------------------------------
constexpr int TK = 32;            // keys per shared-memory tile
struct AttendPlan {
  int nq;          // query vectors per CTA: 4, 8, 16 or 32 (rows_per_block * hpg, rounded up)
  int rows;        // chunk rows per CTA (row block)
  int n_rb;        // row blocks per sequence
  int keys_max;    // upper bound of keys a row block reads (sinks + window + rows - 1)
  int chunk;       // keys per split (multiple of TK)
  int splits;      // splits per (sequence, KV head, row block)
  size_t items;    // B * nk * n_rb * splits partial records
  size_t ws_bytes; // workspace bytes
  size_t off_ml;   // byte offset of the (m, l) records
  size_t off_nsplit; // byte offset of the per-(b, rb) valid-split counts
  size_t off_meta;   // byte offset of the per-sequence copy of the meta before the chunk
  size_t off_far;    // byte offset of the far records [B][nh] x (4 + hd) floats (far field only)
  size_t ws_min;     // the smallest workspace swa_attend accepts (no split-once operand blocks)
  size_t off_ops;    // byte offset of the split-once operand blocks (tensor-core prompt kernel)
  int ops_nblk;      // their blocks per (sequence, KV head), 0 if the plan has none
  int ops_nsb;       // sink blocks among them
  size_t off_order;  // byte offset of the row-block order (tensor-core blocks, or ordered verify)
  size_t off_exp;    // byte offset of the operand blocks' exponents (with the operand blocks)
  int ordered;       // verify blocks: one split each, CTAs take them longest first (off_order)
};
bool make_plan(const swa_attend_args* a, AttendPlan* p);
// swa_attend's argument checks short of the workspace (SWA_OK or the first error)
int attend_args_status(const swa_attend_args* a);

// Kernel parameters of the attention (one struct, passed by value).
struct AttendParams {
  int B, t, nh, nk, hd, cap, ns, hpg;
  float qmul;                 // scale * log2(e): scores are kept in log2 units
  const swa_meta* meta;
  const float* q;
  const float* k_chunk;
  const float* v_chunk;
  float* ring_k;
  float* ring_v;
  const float* sink_k;
  const float* sink_v;
  const float* gate;
  const float* gate_scale;
  float* out;
  float* ws_acc;              // [items][nq][hd]
  float2* ws_ml;              // [items][nq] (m in log2 units, l)
  int* ws_nsplit;             // [B][n_rb]
  swa_meta* ws_meta;          // [B]: meta before the chunk, saved by the attention kernel
  int commit;
  int commit_blocks;          // CTAs per sequence of the commit
  swa_meta* meta_out;
  uint32_t* err;
  int nq, rows, n_rb, chunk, splits;
  // far field (decode rows): far == 0 means none
  int far, far_m, far_rect;
  const float* k_tilde;       // [B][nk][m][hd]
  const float* q_tilde;       // [B][nh][m][hd]
  const float* mu;            // [B][nh][m][m]
  float* mz;                  // [B][nh][2m]
  float* t_hat;               // [B][nh][m][hd]
  float* ws_far;              // [B][nh] x (fm in log2 units, far mass, have, 0, numerator[hd])
  float scale;                // score scale in natural units (the far state's units)
  // full-sequence attention (swa_flash): packed q|k|v rows and segments; B is
  // the segment count there
  const float* qkv;
  const uint32_t* segs;       // [B][2]: first row, length
  int T, ld, q_off, k_off, v_off, ldo, max_len;
  // split-once operand blocks [B][nk][ops_nblk] of 32 keys (K hi, K lo, V^T hi, V^T lo;
  // f16 with ops_exp, TF32 without), or null: swa_flash's segment rows, or the token
  // path's sink blocks then its logical keys 0 .. len0 + t - 1 (tensor-core prompt kernels)
  float* ops;
  int ops_nblk;               // blocks per (sequence or segment, KV head)
  int ops_nsb;                // token path: sink blocks among them (ceil(ns / 32))
  int flash_tail, flash_q;    // swa_flash: the last flash_tail units run as flash_q pieces each
  float* ws_rec;              // their records: [tail * q] x (O[128][hd], then [2][128] (m, l))
  int* ws_cnt;                // [tail][8] pieces done per unit and softmax warp
  int* ws_order;              // with f16 ops, or ordered verify blocks: [B * nk * n_rb] units (index
                              // (b * nk + g) * n_rb + rb), longest first
  int fused;                  // ordered verify blocks: the attention kernel also normalises, gates,
                              // writes out and commits (no records, no merge)
  int* ops_exp;               // [B][nk][ops_nblk] x (e_k, e_v), the power-of-two exponents of
                              // the f16 operand blocks (ops then holds f16 blocks)
};

int launch_attend_partial(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1);
int launch_attend_merge(const AttendParams& p, cudaStream_t s);
int launch_far(const AttendParams& p, cudaStream_t s);
int launch_rollback(swa_meta* meta, const int32_t* n_back, int B, int cap, uint32_t* err,
                    cudaStream_t s);
int attend_partial_occupancy(int hd, int nq);   // resident CTAs per SM
// decode kernel (nq <= 8 query vectors per CTA), swa_decode.cu
int launch_attend_decode(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1);
int attend_decode_occupancy(int hd, int nq);
// one-launch decode step (t = 1, one split per (sequence, KV head), nq <= 8): prep,
// attention with the row's own key from shared memory, gate and commit, swa_decode.cu
int launch_decode_step(const AttendParams& p, const double* inv_freq, const float* yq, const float* yk,
                       const float* yv, const float* q_scale, const uint32_t* pos0, float eps, cudaStream_t s,
                       cudaEvent_t e0, cudaEvent_t e1);
// prompt-chunk kernel (64 query vectors per CTA, tensor cores), swa_prompt.cu
int launch_attend_prompt(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1);
// prompt-chunk kernel on tcgen05 / TMEM (128 query vectors per CTA), swa_prompt_tc.cu
int launch_attend_prompt_tc(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1);
// prompt-chunk kernel of the token path with split-once f16 operand blocks (a workspace
// of plan.ws_bytes): persistent, tcgen05 kind::f16, swa_prompt_h16.cu
int launch_attend_prompt_h16(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1);
// the same kernel over whole segments of packed q|k|v rows (swa_flash, p.ops with f16
// blocks, p.ops_exp, p.ws_order), swa_prompt_h16.cu
int launch_flash_h16(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1);
// the TF32 kernel over whole segments of packed q|k|v rows (swa_flash without a
// workspace: each CTA splits the rows it stages), swa_prompt_tc.cu
int launch_flash_tc(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1);
constexpr int kOpsBlockKeys = 32;   // keys per split-once operand block (= the kernel's key tile)
// verify kernel (16 or 32 query vectors per CTA, CUDA cores), swa_verify.cu
int launch_attend_verify(const AttendParams& p, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1);
int attend_verify_occupancy(int hd, int nq);

struct PrepParams {
  int B, t, nh, nk, hd, cap;
  float eps;
  const float* yq;
  const float* yk;
  const float* yv;
  const float* rope;
  const float* q_scale;
  const uint32_t* pos0;
  float* q_out;
  float* k_out;
  float* v_out;
  float* ring_k;
  float* ring_v;
  double inv_freq[128];       // theta^(-2e/hd), used when rope == nullptr
};
int launch_prep(const PrepParams& p, cudaStream_t s);
void fill_inv_freq(double theta, int hd, double* inv_freq);   // theta^(-2e/hd), e < hd/2
int launch_rope_table(float* rope, const uint32_t* pos0, int B, int t, int hd,
                      const double* inv_freq, cudaStream_t s);

// ---------------------------------------------------------------------------
// Device helpers: mbarrier, bulk copies into shared memory, bounded waits.
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for the barrier's phase `parity` to complete, for at most `limit_ns`
// nanoseconds of wall time. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Order this thread's earlier shared-memory accesses (generic proxy) before
// later bulk copies (async proxy) that overwrite the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) from global memory into L2
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// Bulk copy (TMA, non-tensor) of `bytes` (multiple of 16, both addresses
// 16-byte aligned) from global memory into this CTA's shared memory; the
// transaction count of `bar` is decremented by `bytes` when it lands.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void set_err(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// 16-byte asynchronous copy global -> shared (L2 only), tracked by cp.async groups
// or, after cp_async_arrive_noinc, by an mbarrier.
__device__ __forceinline__ void cp_async16_cg(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               :: "r"(smem_u32(dst_smem)), "l"(src_gmem) : "memory");
}

// The barrier receives one arrival from this thread once all of the thread's
// earlier cp.async copies have landed (the arrival is counted in the barrier's
// expected count: no pending-count increment).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// Plain arrival (no transaction bytes) on a barrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// Barrier among `nthreads` threads (whole warps) of the CTA on hardware barrier `id`.
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// A sequence's ring state with the window, length and head clamped into range
// (window <= cap, win_len <= window, win_head < window); out-of-range meta is
// reported through the error word when `report` is set.
struct SeqState {
  int W, len0, head0;
};

__device__ __forceinline__ SeqState sanitize_state(const swa_meta m, int cap, bool* bad_out) {
  int W = m.window ? (int)m.window : cap;
  bool bad = false;
  if (W > cap) { W = cap; bad = true; }
  int len0 = (int)m.win_len;
  if (len0 > W) { len0 = W; bad = true; }
  int head0 = (int)m.win_head;
  if (head0 >= W) { head0 %= W; bad = true; }
  if (bad_out) *bad_out = bad;
  return {W, len0, head0};
}

// The meta after a commit of t rows ("o1c_msl.metal", o1c_meta): the window grows
// to at most W; past it the head advances by the evicted rows and far_len counts
// them.
__device__ __forceinline__ swa_meta advance_meta(const swa_meta m0, const SeqState& st, int t) {
  swa_meta m1 = m0;
  const long long tot = (long long)st.len0 + t;
  if (tot <= st.W) {
    m1.win_len = (uint32_t)tot;
  } else {
    const long long ev = tot - st.W;
    m1.win_len = (uint32_t)st.W;
    m1.win_head = (uint32_t)((st.head0 + ev) % st.W);
    m1.far_len = (uint32_t)(m0.far_len + (uint32_t)ev);
  }
  return m1;
}

__device__ __forceinline__ SeqState load_state(const AttendParams& p, int b, bool report) {
  bool bad = false;
  const SeqState st = sanitize_state(p.meta[b], p.cap, &bad);
  if (bad && report) set_err(p.err, SWA_DERR_META);
  return st;
}

// One head of the prep ("dory_msl.metal" dory_prep) as a warp sees it: lane l
// holds the P = hd/64 pairs (e, e + hd/2) with e in [l*P, (l+1)*P). Rotates
// (u = x c - y s, v = y c + x s) and returns 1 / sqrt(sum over the head of
// u^2 + v^2 + eps), summed across the warp. Shared by the prep kernel and the
// one-launch decode step so that both produce the same bits.
template <int P>
__device__ __forceinline__ float rotate_unit(const float (&x)[P], const float (&y)[P], const float (&c)[P],
                                             const float (&s)[P], float eps, float (&u)[P], float (&v)[P]) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    u[i] = x[i] * c[i] - y[i] * s[i];
    v[i] = y[i] * c[i] + x[i] * s[i];
    ss += u[i] * u[i] + v[i] * v[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return 1.0f / sqrtf(ss + eps);
}

#endif  // __CUDACC__

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s per bounded wait

// Programmatic dependent launch. A kernel started by launch_pdl may be
// scheduled while the previous kernel of the stream is still running: it calls
// pdl_wait() before its first global memory access, which returns once that
// kernel has completed and its writes are visible (so stream order holds for
// every byte), and pdl_trigger() to let the next kernel's CTAs be scheduled as
// soon as all of its own CTAs have started. Without a programmatic dependency
// (an ordinary launch, another preceding operation) both are no-ops.
#ifdef __CUDACC__
// The output gate: o * inv * sigma(g * s) with sigma(x) = 1 / (1 + e^-x) from the MUFU
// exp2 and reciprocal (relative error about 2^-21; x -> -inf gives 0, x -> inf 1). Every
// kernel that applies the gate uses this one function, so their results agree bit for bit.
__device__ __forceinline__ float gated(float o, float inv, float g, float s) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"((g * s) * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return (o * inv) * r;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

// Bookkeeping after a launch: count it and fold the launch error into a status.
inline int finish_launch(cudaError_t e) {
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace swa
