// C ABI of the sliding-window GQA token path: argument checks, the split
// planner and the kernel launches (declarations and contracts in swa.h).
#include "swa_internal.cuh"

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>

namespace swa {

static std::atomic<uint64_t> g_launches{0};
static thread_local char g_cuda_err[256] = "";

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SWA_OK;
  std::snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return SWA_E_CUDA;
}

int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = sms;
  return sms;
}

static bool hd_ok(int hd) { return hd == 64 || hd == 128 || hd == 256; }

void fill_inv_freq(double theta, int hd, double* inv_freq) {
  for (int e = 0; e < 128; ++e) inv_freq[e] = e < hd / 2 ? std::pow(theta, -2.0 * e / hd) : 0.0;
}
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int attend_shape_ok(const swa_attend_args* a) {
  if (a->B < 1 || a->t < 1 || a->nh < 1 || a->nk < 1 || a->cap < 1 || a->ns < 0) return 0;
  if (!hd_ok(a->hd)) return 0;
  if (a->nh % a->nk != 0) return 0;
  if (a->nh / a->nk > 32) return 0;
  if (a->num_splits < 0) return 0;
  if (a->far && (a->t > 64 || a->t > a->cap || a->far->m < 1 || a->far->m > 32)) return 0;
  // output rows are indexed in 32 bits (q alone would exceed device memory first)
  if ((long long)a->B * a->t * a->nh >= (1LL << 31)) return 0;
  // grid y / z extents: (sequence, KV head) pairs (one more row in the split-once pass)
  if ((long long)a->B * a->nk > 65534) return 0;
  return 1;
}

// Resident attention CTAs per SM for (hd, nq) on the current device, queried
// once and cached (the first call per device should precede any stream capture).
static int cached_occupancy(int hd, int nq) {
  static int cache[64][3][8] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return attend_partial_occupancy(hd, nq);
  const int hi = hd == 64 ? 0 : (hd == 128 ? 1 : 2);
  int qi = 0;
  while ((4 << qi) < nq && qi < 7) ++qi;
  int& c = cache[dev][hi][qi];
  if (c == 0) c = attend_partial_occupancy(hd, nq);
  return c;
}

// Cut a call into CTAs. A row block holds `rows` chunk rows so that its
// rows * hpg query vectors fit one CTA (<= 32); the split count balances the
// CTAs over the SMs: it minimises (waves of resident CTAs) x (keys per CTA +
// a fixed per-CTA cost), with the keys of a row block bounded by
// ns + cap + rows - 1 (the window never exceeds cap).
// Far records after the rest of the workspace: per (sequence, row, query head) the
// far exponent, mass, a keep flag and the far numerator.
static void add_far_records(const swa_attend_args* a, AttendPlan* p) {
  p->off_far = p->ws_bytes;
  if (a->far) p->ws_bytes += (((size_t)a->B * a->t * a->nh * (4 + a->hd) * sizeof(float)) + 255) & ~(size_t)255;
}

bool make_plan(const swa_attend_args* a, AttendPlan* p) {
  if (!attend_shape_ok(a)) return false;
  p->off_ops = 0;
  p->off_order = 0;
  p->off_exp = 0;
  p->ops_nblk = 0;
  p->ops_nsb = 0;
  p->ordered = 0;
  const int hpg = a->nh / a->nk;
  // Prompt-sized chunks run on tensor cores, one split per row block: blocks of
  // 128 query vectors on tcgen05 when a chunk has at least 128 query vectors
  // per KV head, else blocks of 64 on mma.sync (hd <= 128 in both).
  if (a->hd <= 128 && (long long)a->t * hpg >= 64) {
    const int block = (long long)a->t * hpg >= 128 ? 128 : 64;
    const int rows = block / hpg;
    p->nq = block;
    p->rows = rows;
    p->n_rb = (a->t + rows - 1) / rows;
    if (p->n_rb > 65535) return false;
    const long long keys_max = (long long)a->ns + a->cap + rows - 1;
    if (keys_max > (1LL << 30)) return false;
    p->keys_max = (int)keys_max;
    p->chunk = (int)((keys_max + TK - 1) / TK * TK);
    p->splits = 1;
    p->items = (size_t)a->B * a->nk * p->n_rb;
    const size_t acc_bytes = p->items * p->nq * (size_t)a->hd * sizeof(float);
    const size_t ml_bytes = p->items * p->nq * sizeof(float2);
    const size_t ns_bytes = (size_t)a->B * p->n_rb * sizeof(int);
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    p->off_ml = up(acc_bytes);
    p->off_nsplit = p->off_ml + up(ml_bytes);
    p->off_meta = p->off_nsplit + up(ns_bytes);
    p->ws_bytes = p->off_meta + up((size_t)a->B * sizeof(swa_meta));
    add_far_records(a, p);
    p->ws_min = p->ws_bytes;
    if (block == 128) {
      // split-once operand blocks for the tcgen05 kernel: per (sequence, KV head) the
      // sinks' blocks, then blocks of the logical keys 0 .. len0 + t - 1 (< cap + t)
      p->ops_nsb = (a->ns + kOpsBlockKeys - 1) / kOpsBlockKeys;
      const long long nlog = ((long long)a->cap + a->t + kOpsBlockKeys - 1) / kOpsBlockKeys;
      p->ops_nblk = (int)(p->ops_nsb + nlog);
      // (f16 K hi, K lo, V^T hi, V^T lo of 32 keys each) and their exponents (e_k, e_v)
      p->off_ops = p->ws_bytes;
      p->ws_bytes += up((size_t)a->B * a->nk * p->ops_nblk * 4 * kOpsBlockKeys * a->hd * 2);
      p->off_exp = p->ws_bytes;
      p->ws_bytes += up((size_t)a->B * a->nk * p->ops_nblk * 2 * sizeof(int));
      // the order in which the kernel's CTAs take the row blocks (longest first)
      p->off_order = p->ws_bytes;
      p->ws_bytes += up(p->items * sizeof(int));
    }
    return true;
  }
  int rows = 32 / hpg;
  if (rows < 1) rows = 1;
  if (rows > a->t) rows = a->t;
  const int used = rows * hpg;
  int nq = 4;
  while (nq < used) nq *= 2;
  p->nq = nq;
  p->rows = rows;
  p->n_rb = (a->t + rows - 1) / rows;
  if (p->n_rb > 65535) return false;
  const long long keys_max = (long long)a->ns + a->cap + rows - 1;
  if (keys_max > (1LL << 30)) return false;
  p->keys_max = (int)keys_max;
  const int max_splits = (int)((keys_max + TK - 1) / TK);
  const long long units = (long long)a->B * a->nk * p->n_rb;
  int best_s = 1;
  // Verify blocks (16 / 32 query vectors) of one row block per (sequence, KV head),
  // far more of them than resident CTAs: one split each, taken longest first (the
  // longest-processing-time rule balances the SMs without splitting), so that the
  // attention kernel can finish them itself: no records, no merge (with a far field
  // the single-split records still go to the merge, which joins the far part).
  const int sms_now = num_sms();
  const long long slots_now =
      (long long)(sms_now > 0 ? sms_now : 148) * cached_occupancy(a->hd, nq);
  const bool ordered = (nq == 16 || nq == 32) && a->num_splits == 0 && p->n_rb == 1 &&
                       sms_now > 0 && units >= 2 * slots_now;
  if (ordered) {
    best_s = 1;
  } else if (a->num_splits > 0) {
    best_s = a->num_splits < max_splits ? a->num_splits : max_splits;
  } else {
    // About 8 waves of resident CTAs (a short tail and enough key streams in
    // flight to cover HBM latency), but at least 4 tiles of keys per split.
    const int sms = num_sms();
    const int occ = cached_occupancy(a->hd, nq);
    const long long slots = (long long)(sms > 0 ? sms : 148) * (occ > 0 ? occ : 1);
    long long want = (8 * slots + units - 1) / units;
    const long long cap_s = (keys_max + 4 * TK - 1) / (4 * TK);
    if (want > cap_s) want = cap_s;
    if (want < 1) want = 1;
    best_s = (int)want;
  }
  long long chunk = ((keys_max + best_s - 1) / best_s + TK - 1) / TK * TK;
  p->chunk = (int)chunk;
  p->splits = (int)((keys_max + chunk - 1) / chunk);
  p->items = (size_t)units * p->splits;
  const size_t acc_bytes = p->items * nq * (size_t)a->hd * sizeof(float);
  const size_t ml_bytes = p->items * nq * sizeof(float2);
  const size_t ns_bytes = (size_t)a->B * p->n_rb * sizeof(int);
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  p->off_ml = up(acc_bytes);
  p->off_nsplit = p->off_ml + up(ml_bytes);
  p->off_meta = p->off_nsplit + up(ns_bytes);
  p->ws_bytes = p->off_meta + up((size_t)a->B * sizeof(swa_meta));
  add_far_records(a, p);
  if (ordered) {
    p->ordered = 1;
    p->off_order = p->ws_bytes;
    p->ws_bytes += up((size_t)units * sizeof(int));
  }
  p->ws_min = p->ws_bytes;
  return true;
}

// Every check of swa_attend's arguments that does not depend on the workspace,
// in the order swa_attend applies them: NULL pointers, sizes, alignment.
int attend_args_status(const swa_attend_args* a) {
  if (!a) return SWA_E_NULL;
  if (!a->meta || !a->q || !a->k_chunk || !a->v_chunk || !a->ring_k || !a->ring_v || !a->gate ||
      !a->gate_scale || !a->out)
    return SWA_E_NULL;
  if (a->ns > 0 && (!a->sink_k || !a->sink_v)) return SWA_E_NULL;
  if (a->commit && !a->meta_out) return SWA_E_NULL;
  if (a->far && (!a->far->k_tilde || !a->far->q_tilde || !a->far->mu || !a->far->mz || !a->far->t_hat))
    return SWA_E_NULL;
  if (!attend_shape_ok(a)) return SWA_E_SHAPE;
  if (a->far && (!aligned16(a->far->k_tilde) || !aligned16(a->far->q_tilde) || !aligned16(a->far->t_hat) ||
                 (reinterpret_cast<uintptr_t>(a->far->mu) & 3u) || (reinterpret_cast<uintptr_t>(a->far->mz) & 3u)))
    return SWA_E_ALIGN;
  if (!(a->scale == a->scale) || std::isinf(a->scale)) return SWA_E_SHAPE;
  const void* ptrs[] = {a->q, a->k_chunk, a->v_chunk, a->ring_k, a->ring_v, a->sink_k,
                        a->sink_v, a->gate, a->gate_scale, a->out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return SWA_E_ALIGN;
  return SWA_OK;
}

}  // namespace swa

using namespace swa;

extern "C" {

const char* swa_status_string(int status) {
  switch (status) {
    case SWA_OK: return "ok";
    case SWA_E_NULL: return "a required pointer is NULL";
    case SWA_E_SHAPE: return "unsupported or inconsistent sizes";
    case SWA_E_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case SWA_E_WORKSPACE: return "workspace missing or too small";
    case SWA_E_HAZARD: return "prep ring write needs t == 1 (commit chunks through swa_attend)";
    case SWA_E_CUDA: return "a CUDA launch or query failed";
  }
  return "unknown status";
}

const char* swa_last_cuda_error(void) { return g_cuda_err; }

const char* swa_version(void) { return "swa-gb300 0.1 (sm_103a)"; }

uint64_t swa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int swa_rope_table(float* rope, const uint32_t* pos0, int B, int t, int hd, double theta,
                   cudaStream_t stream) {
  if (!rope || !pos0) return SWA_E_NULL;
  if (B < 1 || t < 1 || !hd_ok(hd) || !(theta > 0.0)) return SWA_E_SHAPE;
  if (!aligned16(rope)) return SWA_E_ALIGN;
  double inv_freq[128];
  fill_inv_freq(theta, hd, inv_freq);
  return launch_rope_table(rope, pos0, B, t, hd, inv_freq, stream);
}

int swa_rollback(swa_meta* meta, const int32_t* n_back, int B, int cap, uint32_t* err,
                 cudaStream_t stream) {
  if (!meta || !n_back) return SWA_E_NULL;
  if (B < 1 || cap < 1) return SWA_E_SHAPE;
  if (!aligned16(meta)) return SWA_E_ALIGN;
  return launch_rollback(meta, n_back, B, cap, err, stream);
}

int swa_prep(const swa_prep_args* a, cudaStream_t stream) {
  if (!a) return SWA_E_NULL;
  if (!a->yq || !a->yk || !a->yv || !a->q_scale || !a->q_out || !a->k_out) return SWA_E_NULL;
  if (!a->rope) {
    if (!a->pos0) return SWA_E_NULL;
    if (!(a->theta > 0.0)) return SWA_E_SHAPE;
  }
  if (a->B < 1 || a->t < 1 || a->nh < 1 || a->nk < 1 || !hd_ok(a->hd)) return SWA_E_SHAPE;
  if (!(a->eps >= 0.0f)) return SWA_E_SHAPE;
  const bool ring = a->ring_k || a->ring_v;
  if (ring) {
    if (!a->ring_k || !a->ring_v || !a->pos0) return SWA_E_NULL;
    if (a->cap < 1) return SWA_E_SHAPE;
    if (a->t > 1) return SWA_E_HAZARD;
  }
  const void* ptrs[] = {a->yq, a->yk, a->yv, a->rope, a->q_scale, a->q_out, a->k_out,
                        a->v_out, a->ring_k, a->ring_v};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return SWA_E_ALIGN;
  PrepParams p;
  p.B = a->B; p.t = a->t; p.nh = a->nh; p.nk = a->nk; p.hd = a->hd; p.cap = a->cap;
  p.eps = a->eps;
  p.yq = a->yq; p.yk = a->yk; p.yv = a->yv; p.rope = a->rope; p.q_scale = a->q_scale;
  p.pos0 = a->pos0;
  p.q_out = a->q_out; p.k_out = a->k_out; p.v_out = a->v_out;
  p.ring_k = ring ? a->ring_k : nullptr;
  p.ring_v = ring ? a->ring_v : nullptr;
  fill_inv_freq(a->rope ? 10000.0 : a->theta, a->hd, p.inv_freq);
  return launch_prep(p, stream);
}

size_t swa_attend_workspace_size(const swa_attend_args* a) {
  if (!a) return 0;
  AttendPlan plan;
  if (!make_plan(a, &plan)) return 0;
  return plan.ws_bytes;
}

size_t swa_attend_workspace_min(const swa_attend_args* a) {
  if (!a) return 0;
  AttendPlan plan;
  if (!make_plan(a, &plan)) return 0;
  return plan.ws_min;
}

// Kernel parameters of an attention call with plan `plan` (workspace regions
// only when the call has a workspace).
static void fill_attend_params(const swa_attend_args* a, const AttendPlan& plan, AttendParams& p) {
  p.B = a->B; p.t = a->t; p.nh = a->nh; p.nk = a->nk; p.hd = a->hd; p.cap = a->cap;
  p.ns = a->ns; p.hpg = a->nh / a->nk;
  p.qmul = a->scale * 1.4426950408889634f;
  p.meta = a->meta;
  p.q = a->q; p.k_chunk = a->k_chunk; p.v_chunk = a->v_chunk;
  p.ring_k = a->ring_k; p.ring_v = a->ring_v;
  p.sink_k = a->sink_k; p.sink_v = a->sink_v;
  p.gate = a->gate; p.gate_scale = a->gate_scale; p.out = a->out;
  char* ws = static_cast<char*>(a->workspace);
  if (ws) {
    p.ws_acc = reinterpret_cast<float*>(ws);
    p.ws_ml = reinterpret_cast<float2*>(ws + plan.off_ml);
    p.ws_nsplit = reinterpret_cast<int*>(ws + plan.off_nsplit);
    p.ws_meta = reinterpret_cast<swa_meta*>(ws + plan.off_meta);
    p.ws_far = reinterpret_cast<float*>(ws + plan.off_far);
  }
  {
    // commit CTAs per sequence: about 4 float4 pairs per thread of 256
    const long long rows = a->t < a->cap ? a->t : a->cap;
    const long long work = rows * a->nk * (a->hd / 4);
    long long cb = (work + 1023) / 1024;
    p.commit_blocks = (int)(cb < 1 ? 1 : (cb > 4096 ? 4096 : cb));
  }
  p.commit = a->commit ? 1 : 0;
  p.meta_out = a->meta_out;
  p.err = a->err;
  p.nq = plan.nq; p.rows = plan.rows; p.n_rb = plan.n_rb; p.chunk = plan.chunk;
  p.splits = plan.splits;
  p.scale = a->scale;
  p.far = a->far ? 1 : 0;
  p.far_m = a->far ? a->far->m : 0;
  p.far_rect = a->far ? (a->far->rect != 0) : 0;
  p.k_tilde = a->far ? a->far->k_tilde : nullptr;
  p.q_tilde = a->far ? a->far->q_tilde : nullptr;
  p.mu = a->far ? a->far->mu : nullptr;
  p.mz = a->far ? a->far->mz : nullptr;
  p.t_hat = a->far ? a->far->t_hat : nullptr;
  // the split-once operand blocks when the workspace holds them
  p.ops = (ws && plan.ops_nblk > 0 && a->workspace_bytes >= plan.ws_bytes)
              ? reinterpret_cast<float*>(ws + plan.off_ops) : nullptr;
  p.ops_nblk = plan.ops_nblk;
  p.ops_nsb = plan.ops_nsb;
  p.ws_order = p.ops ? reinterpret_cast<int*>(ws + plan.off_order) : nullptr;
  p.ops_exp = p.ops ? reinterpret_cast<int*>(ws + plan.off_exp) : nullptr;
  if (ws && plan.ordered) {
    // ordered verify blocks; the kernel finishes them itself unless the commit's meta
    // aliases the meta other CTAs still read, the gate may still be arriving, or a far
    // field joins the rows in the merge
    p.ws_order = reinterpret_cast<int*>(ws + plan.off_order);
    const bool aliased = a->commit && (const void*)a->meta_out == (const void*)a->meta;
    p.fused = !aliased && !a->gate_ready && !a->far ? 1 : 0;
  }
}

int swa_attend(const swa_attend_args* a, cudaStream_t stream) {
  const int rc0 = attend_args_status(a);
  if (rc0 != SWA_OK) return rc0;
  AttendPlan plan;
  if (!make_plan(a, &plan)) return SWA_E_SHAPE;
  if (!a->workspace || a->workspace_bytes < plan.ws_min) return SWA_E_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0) return SWA_E_ALIGN;
  AttendParams p{};
  fill_attend_params(a, plan, p);
  int rc = SWA_OK;
  if (p.far) {            // before the attention: it reads the evicted ring slot, which the commit overwrites
    rc = launch_far(p, stream);
    if (rc != SWA_OK) return rc;
  }
  rc = launch_attend_partial(p, stream, a->ev_start, a->ev_stop);
  if (rc != SWA_OK) return rc;
  if (p.fused) return SWA_OK;   // the attention kernel wrote out and committed
  if (a->gate_ready) {    // the gate may still be arriving: only the merge reads it
    const cudaError_t e = cudaStreamWaitEvent(stream, a->gate_ready, 0);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return launch_attend_merge(p, stream);
}

// ---------------------------------------------------------------------------
// swa_decode_step: prep + attend + commit of one token, one kernel when the plan
// runs each (sequence, KV head) as a single CTA
// ---------------------------------------------------------------------------
static void decode_as_attend(const swa_decode_args* a, swa_attend_args* t) {
  std::memset(t, 0, sizeof(*t));
  t->B = a->B; t->t = 1; t->nh = a->nh; t->nk = a->nk; t->hd = a->hd; t->cap = a->cap; t->ns = a->ns;
  t->scale = a->scale;
  t->meta = a->meta;
  t->ring_k = a->ring_k; t->ring_v = a->ring_v;
  t->sink_k = a->sink_k; t->sink_v = a->sink_v;
  t->gate = a->gate; t->gate_scale = a->gate_scale;
  t->out = a->out;
  t->commit = 1;
  t->meta_out = a->meta_out;
  t->err = a->err;
  t->ev_start = a->ev_start; t->ev_stop = a->ev_stop;
}

static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// K/V bytes of one (sequence, KV head) up to which a decode step runs as one
// kernel even where the split planner would cut the window: below it the CTA
// streams its window in a few microseconds, less than the two launches saved.
constexpr size_t kStepOneCtaBytes = 512 * 1024;

// 1: one kernel (the plan then has one split per (sequence, KV head)),
// 3: prep + attention + merge, 0: invalid sizes.
static int decode_form(const swa_decode_args* a, AttendPlan* plan) {
  swa_attend_args t;
  decode_as_attend(a, &t);
  if (a->B < 1 || a->nh < 1 || a->nk < 1 || a->cap < 1 || a->ns < 0 || !hd_ok(a->hd)) return 0;
  if (!make_plan(&t, plan)) return 0;
  const bool aliased = a->meta_out != nullptr && (const void*)a->meta_out == (const void*)a->meta;
  const bool short_window = (size_t)plan->keys_max * a->hd * 8 <= kStepOneCtaBytes;
  if (plan->nq > 8 || aliased || (plan->splits != 1 && !short_window)) return 3;
  plan->splits = 1;
  plan->chunk = (plan->keys_max + TK - 1) / TK * TK;
  return 1;
}

size_t swa_decode_workspace_size(const swa_decode_args* a) {
  if (!a) return 0;
  AttendPlan plan;
  const int form = decode_form(a, &plan);
  if (form != 3) return 0;
  return up256((size_t)a->B * a->nh * a->hd * sizeof(float)) +
         up256((size_t)a->B * a->nk * a->hd * sizeof(float)) + plan.ws_bytes;
}

int swa_decode_launches(const swa_decode_args* a) {
  if (!a) return 0;
  AttendPlan plan;
  return decode_form(a, &plan);
}

int swa_decode_step(const swa_decode_args* a, cudaStream_t stream) {
  if (!a) return SWA_E_NULL;
  if (!a->yq || !a->yk || !a->yv || !a->q_scale || !a->pos0 || !a->meta || !a->ring_k || !a->ring_v ||
      !a->gate || !a->gate_scale || !a->out || !a->meta_out)
    return SWA_E_NULL;
  if (a->ns > 0 && (!a->sink_k || !a->sink_v)) return SWA_E_NULL;
  swa_attend_args t;
  decode_as_attend(a, &t);
  if (!attend_shape_ok(&t)) return SWA_E_SHAPE;
  if (!(a->eps >= 0.0f) || !(a->theta > 0.0) || !(a->scale == a->scale) || std::isinf(a->scale))
    return SWA_E_SHAPE;
  const void* ptrs[] = {a->yq, a->yk, a->yv, a->q_scale, a->ring_k, a->ring_v, a->sink_k,
                        a->sink_v, a->gate, a->gate_scale, a->out, a->meta, a->meta_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return SWA_E_ALIGN;
  AttendPlan plan;
  const int form = decode_form(a, &plan);
  if (form == 0) return SWA_E_SHAPE;
  double inv_freq[128];
  fill_inv_freq(a->theta, a->hd, inv_freq);
  if (form == 1) {
    AttendParams p{};
    fill_attend_params(&t, plan, p);
    return launch_decode_step(p, inv_freq, a->yq, a->yk, a->yv, a->q_scale, a->pos0, a->eps, stream,
                              a->ev_start, a->ev_stop);
  }
  // prep (q-hat, k-hat into the workspace; v read in place) + attention + merge
  const size_t qb = up256((size_t)a->B * a->nh * a->hd * sizeof(float));
  const size_t kb = up256((size_t)a->B * a->nk * a->hd * sizeof(float));
  if (!a->workspace || a->workspace_bytes < qb + kb + plan.ws_min) return SWA_E_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return SWA_E_ALIGN;
  char* ws = static_cast<char*>(a->workspace);
  swa_prep_args pa;
  std::memset(&pa, 0, sizeof pa);
  pa.B = a->B; pa.t = 1; pa.nh = a->nh; pa.nk = a->nk; pa.hd = a->hd; pa.cap = a->cap; pa.eps = a->eps;
  pa.yq = a->yq; pa.yk = a->yk; pa.yv = a->yv; pa.rope = nullptr; pa.q_scale = a->q_scale;
  pa.pos0 = a->pos0; pa.theta = a->theta;
  pa.q_out = reinterpret_cast<float*>(ws);
  pa.k_out = reinterpret_cast<float*>(ws + qb);
  int rc = swa_prep(&pa, stream);
  if (rc != SWA_OK) return rc;
  t.q = pa.q_out;
  t.k_chunk = pa.k_out;
  t.v_chunk = a->yv;
  t.workspace = ws + qb + kb;
  t.workspace_bytes = a->workspace_bytes - qb - kb;
  return swa_attend(&t, stream);
}

static bool flash_shape_ok(const swa_flash_args* a) {
  if (a->T < 1 || a->nseg < 1 || a->nh < 1 || a->nk < 1 || a->max_len < 1 || a->max_len > a->T) return false;
  if (a->hd != 64 && a->hd != 128) return false;
  return a->nh % a->nk == 0 && a->nh / a->nk <= 32;
}

// The split-once workspace of swa_flash: f16 operand blocks [nseg][nk][ceil(max_len /
// 32)] of 4 x 32 x hd halves (K hi, K lo, V^T hi, V^T lo), their exponents (2 ints a
// block), the unit order (an int per unit), then, optionally, the launch tail's records
// and counters. Each part starts on a 256-byte boundary.
struct FlashWs {
  size_t off_exp = 0, off_order = 0, bytes = 0;
};
static FlashWs flash_ws(const swa_flash_args* a) {
  FlashWs f;
  const size_t nblk = ((size_t)a->max_len + kOpsBlockKeys - 1) / kOpsBlockKeys;
  const size_t nbg = (size_t)a->nseg * a->nk;
  const size_t rows = 128 / (a->nh / a->nk);
  const size_t n_rb = (a->max_len + rows - 1) / rows;
  f.off_exp = nbg * nblk * 4 * kOpsBlockKeys * a->hd * 2;   // a multiple of 256 bytes
  f.off_order = f.off_exp + up256(nbg * nblk * 2 * sizeof(int));
  f.bytes = f.off_order + up256(nbg * n_rb * sizeof(int));
  return f;
}
static size_t ops_bytes(const swa_flash_args* a) { return flash_ws(a).bytes; }

// The tail of a flash launch. The attention runs one CTA (one row block of one
// segment and KV head, a "unit") per SM at a time; when the units fill at least
// one wave of SMs and leave a remainder of at most half of one, the last `tail`
// units are cut into q = sms / tail pieces each (key ranges of the unit, combined
// by the last piece), so that the last wave keeps every SM busy.
struct FlashTail {
  int tail = 0, q = 1;
  size_t rec_bytes = 0;   // piece records [tail * q] x (128 x hd, then 2 x 128 x 2) floats
  size_t bytes = 0;       // + combine counters [tail][8] ints
};
static FlashTail flash_tail(const swa_flash_args* a) {
  FlashTail ft;
  const int rows = 128 / (a->nh / a->nk);
  const long long units = (long long)((a->max_len + rows - 1) / rows) * a->nseg * a->nk;
  const int n = num_sms();
  const long long sms = n > 0 ? n : 148;
  if (units < sms) return ft;
  const long long rem = units % sms;
  if (rem == 0 || 2 * rem > sms) return ft;
  const long long q = sms / rem;
  if (units - rem + rem * q >= (1LL << 31)) return ft;
  ft.tail = (int)rem;
  ft.q = (int)q;
  ft.rec_bytes = up256((size_t)rem * q * 128 * (a->hd + 4) * sizeof(float));
  ft.bytes = ft.rec_bytes + up256((size_t)rem * 8 * sizeof(int));
  return ft;
}

size_t swa_flash_workspace_size(const swa_flash_args* a) {
  if (!a || !flash_shape_ok(a)) return 0;
  return ops_bytes(a) + flash_tail(a).bytes;
}

int swa_flash(const swa_flash_args* a, cudaStream_t stream) {
  if (!a) return SWA_E_NULL;
  if (!a->qkv || !a->segs || !a->out) return SWA_E_NULL;
  if (!flash_shape_ok(a)) return SWA_E_SHAPE;
  if (a->ld < 1 || a->ldo < 1 || a->q_off < 0 || a->k_off < 0 || a->v_off < 0) return SWA_E_SHAPE;
  const long long qh = (long long)a->nh * a->hd, kh = (long long)a->nk * a->hd;
  if (a->q_off + qh > a->ld || a->k_off + kh > a->ld || a->v_off + kh > a->ld || qh > a->ldo)
    return SWA_E_SHAPE;
  if (!(a->scale == a->scale) || std::isinf(a->scale)) return SWA_E_SHAPE;
  const int hpg = a->nh / a->nk;
  const int rows = 128 / hpg;                   // query vectors of a CTA: rows x hpg <= 128
  const long long n_rb = (a->max_len + rows - 1) / rows;
  // grids: (n_rb, nseg * nk) CTAs, or (blocks, nseg * nk + 1) and one per SM over the units
  if (n_rb > 65535 || (long long)a->nseg * a->nk > 65534 || n_rb * a->nseg * a->nk >= (1LL << 31))
    return SWA_E_SHAPE;
  if ((a->ld | a->ldo | a->q_off | a->k_off | a->v_off) & 3) return SWA_E_ALIGN;
  if (!aligned16(a->qkv) || !aligned16(a->out) || (reinterpret_cast<uintptr_t>(a->segs) & 3u))
    return SWA_E_ALIGN;
  if (a->workspace) {
    if (a->workspace_bytes < ops_bytes(a)) return SWA_E_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return SWA_E_ALIGN;
  }
  AttendParams p{};
  p.B = a->nseg; p.t = 0; p.nh = a->nh; p.nk = a->nk; p.hd = a->hd; p.cap = 0; p.ns = 0; p.hpg = hpg;
  p.qmul = a->scale * 1.4426950408889634f;
  p.scale = a->scale;
  p.out = a->out;
  p.err = a->err;
  p.nq = 128; p.rows = rows; p.n_rb = (int)n_rb; p.chunk = 0; p.splits = 1;
  p.qkv = a->qkv; p.segs = a->segs;
  p.T = a->T; p.ld = a->ld; p.q_off = a->q_off; p.k_off = a->k_off; p.v_off = a->v_off; p.ldo = a->ldo;
  p.max_len = a->max_len;
  p.ops_nblk = (a->max_len + kOpsBlockKeys - 1) / kOpsBlockKeys;
  p.ops_nsb = 0;
  if (!a->workspace) return launch_flash_tc(p, stream, a->ev_start, a->ev_stop);   // TF32, in-kernel split
  // f16 split-once blocks; the split tail when the workspace has room for its records
  unsigned char* ws = static_cast<unsigned char*>(a->workspace);
  const FlashWs fw = flash_ws(a);
  p.ops = reinterpret_cast<float*>(ws);
  p.ops_exp = reinterpret_cast<int*>(ws + fw.off_exp);
  p.ws_order = reinterpret_cast<int*>(ws + fw.off_order);
  const FlashTail ft = flash_tail(a);
  if (ft.tail > 0 && a->workspace_bytes >= fw.bytes + ft.bytes) {
    p.flash_tail = ft.tail;
    p.flash_q = ft.q;
    p.ws_rec = reinterpret_cast<float*>(ws + fw.bytes);
    p.ws_cnt = reinterpret_cast<int*>(ws + fw.bytes + ft.rec_bytes);
  }
  return launch_flash_h16(p, stream, a->ev_start, a->ev_stop);
}

}  // extern "C"
