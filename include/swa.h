/*
 * swa.h — C ABI of the sliding-window GQA token path on GB300 (sm_103a).
 *
 * Two stages of a sealed sliding-window attention layer, as defined on the
 * Metal shader pages of the cortiq-engine crate:
 *   prep   — "dory_msl.metal" (cortiq-engine 0.8.57), kernel dory_prep:
 *            rotate-half RoPE of every q/k head, unit heads with eps, the
 *            per-feature query scale, K/V into the ring at slot (pos0+j) % cap.
 *   attend — "o1c_msl.metal" (cortiq-engine 0.8.79), kernels o1c_score,
 *            o1c_max, o1c_soft, o1c_sum, o1c_add, o1c_tok_near, o1c_tok_merge,
 *            o1c_ring_commit, o1c_meta; "dory_msl.metal" dory_gate:
 *            each chunk row attends the sinks plus its causal window over the
 *            ring and the chunk's own earlier rows, all query heads of a KV
 *            head together (GQA), max-subtracted f32 softmax, value sums split
 *            across key ranges and reduced, then out = o * sigmoid(g * s_g).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, f32 unless
 *     stated, densely packed in the row-major layout given beside each field,
 *     and 16-byte aligned (SWA_E_ALIGN otherwise).
 *   - Work is enqueued on `stream` (0 = legacy default stream). No entry point
 *     synchronises the device, allocates device memory or keeps state between
 *     calls besides cached device attributes.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     negative status means nothing was enqueued, except SWA_E_CUDA, which
 *     reports a failed launch (the CUDA error text is kept for
 *     swa_status_string / swa_last_cuda_error).
 *   - Sizes are ints; hd must be 64, 128 or 256; nh must be a multiple of nk
 *     with nh / nk <= 32.
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every int entry point. */
#define SWA_OK            0
#define SWA_E_NULL       -1  /* a required pointer is NULL */
#define SWA_E_SHAPE      -2  /* unsupported or inconsistent sizes */
#define SWA_E_ALIGN      -3  /* a tensor pointer is not 16-byte aligned */
#define SWA_E_WORKSPACE  -4  /* workspace missing or smaller than swa_attend_workspace_min */
#define SWA_E_HAZARD     -5  /* prep ring write requested for t > 1 (see swa_prep) */
#define SWA_E_CUDA       -6  /* a CUDA launch or query failed */

/* Bits a kernel ORs into the optional device error word (`err`). The kernels
 * never trap: on such an event they clamp or stop and report it here. */
#define SWA_DERR_META     1u /* meta out of range: window > cap, win_len > window
                                or win_head >= window (values were clamped) */
#define SWA_DERR_TIMEOUT  2u /* a bounded wait on a copy into shared memory
                                expired; the kernel stopped without output */
#define SWA_DERR_SEGMENT  4u /* swa_flash: a segment reaches past row T or is
                                longer than max_len (its rows are not written) */

/* Per-sequence ring state, as the per-group meta of o1c_msl.metal:
 *   win_len  — keys held in the ring (<= window)
 *   win_head — slot of the oldest held key (< window)
 *   far_len  — keys that have left the window (advanced by the commit, read
 *              by nothing on this path)
 *   window   — the window W, which is also the ring modulus; 0 means cap. */
typedef struct swa_meta {
  uint32_t win_len, win_head, far_len, window;
} swa_meta;

/* Human-readable text of a status code (static storage). */
const char* swa_status_string(int status);
/* Text of the last CUDA error seen by this library in this thread ("" if none). */
const char* swa_last_cuda_error(void);
/* Library version string (static storage). */
const char* swa_version(void);
/* Number of kernels this library has launched in this process. */
uint64_t swa_launch_count(void);

/*
 * swa_rope_table — fill the RoPE table that swa_prep consumes.
 *   rope [B][t][hd]: row (b, j) holds cos(a_e) for e < hd/2, then sin(a_e),
 *   a_e = (pos0[b] + j) * theta^(-2e/hd), angles and cos/sin in f64, stored
 *   rounded to f32. The pages consume such a table (dory_prep reads cos at e
 *   and sin at hd/2 + e; eg_qkv_prep in "egemma2_msl.metal" the same pairing)
 *   but do not show how it is built: this is the standard rotate-half
 *   schedule.
 *   pos0 [B] (device, uint32): absolute position of chunk row 0.
 * Errors: SWA_E_NULL, SWA_E_SHAPE (B, t < 1 or hd unsupported, theta <= 0),
 *         SWA_E_ALIGN, SWA_E_CUDA.
 */
int swa_rope_table(float* rope, const uint32_t* pos0, int B, int t, int hd,
                   double theta, cudaStream_t stream);

/*
 * swa_prep — rotation, unit heads, query scale and ring write of a chunk
 * ("dory_msl.metal", dory_prep). For every sequence b, row j, head:
 *   x = head[0:hd/2], y = head[hd/2:hd], c/s = rope[b][j] halves
 *   u = x*c - y*s, v = y*c + x*s, inv = 1 / sqrt(sum(u^2 + v^2) + eps)
 *   q_out[b][j][h] = (u, v) * inv * q_scale[h]          (h < nh)
 *   k_out[b][j][g] = (u, v) * inv                       (g < nk)
 *   v_out[b][j][g] = yv[b][j][g]                        (unchanged)
 * and, when ring_k/ring_v are non-NULL, k_out/v_out rows also go to ring
 * slot (pos0[b] + j) % cap.
 *
 * rope may be NULL: the kernel then computes each row's cos/sin itself from
 * pos0 and theta exactly as swa_rope_table does (same f64 angles, same f32
 * rounding, bit-identical values) and no table is read or written.
 *
 * The ring write is only accepted for t == 1 (SWA_E_HAZARD otherwise): with a
 * full ring a chunk's later rows land on slots that its earlier rows still
 * read. For t > 1 pass NULL rings here and let swa_attend commit the chunk
 * after its reads (commit = 1). For t == 1 the written slot is the evicted
 * one, which the row does not read. The ring slot (pos0 + j) % cap agrees
 * with swa_attend's slot map when the sequence's window equals cap and
 * win_head == (pos0 - win_len) % cap (a ring grown from position 0).
 */
typedef struct swa_prep_args {
  int B, t, nh, nk, hd, cap;     /* cap only read when rings are given      */
  float eps;                     /* added to the sum of squares             */
  const float* yq;               /* [B][t][nh][hd]                          */
  const float* yk;               /* [B][t][nk][hd]                          */
  const float* yv;               /* [B][t][nk][hd]                          */
  const float* rope;             /* [B][t][hd] (swa_rope_table) or NULL     */
  const float* q_scale;          /* [nh][hd]                                */
  const uint32_t* pos0;          /* [B]; required with rings or rope NULL   */
  float* q_out;                  /* [B][t][nh][hd]                          */
  float* k_out;                  /* [B][t][nk][hd]                          */
  float* v_out;                  /* [B][t][nk][hd] or NULL (no copy)        */
  float* ring_k;                 /* [B][nk][cap][hd] or NULL                */
  float* ring_v;                 /* [B][nk][cap][hd] or NULL (with ring_k)  */
  double theta;                  /* RoPE base, read only when rope is NULL  */
} swa_prep_args;

int swa_prep(const swa_prep_args* args, cudaStream_t stream);

/*
 * swa_attend — attention of a chunk of t rows of a sealed sliding-window
 * layer; a decode token (t = 1), a speculative verify and a prompt chunk take
 * the same call ("o1c_msl.metal" o1c_score ... o1c_add and o1c_tok_*;
 * "dory_msl.metal" dory_gate).
 *
 * Row i of sequence b (len0 = win_len, head0 = win_head, W = window before
 * the chunk) attends, for each query head h of KV head g = h / (nh/nk):
 *   the ns sinks sink_k/v[b][g][0..ns), always, and
 *   logical keys x in [lo_i, len0 + i], win_i = min(W, len0 + i + 1),
 *   lo_i = len0 + i + 1 - win_i; x < len0 reads ring slot (head0 + x) % W,
 *   x >= len0 reads chunk row x - len0 from k_chunk/v_chunk.
 *   s = scale * <q, key>, p = exp(s - max s), o = sum p v / sum p,
 *   out[b][i][h] = o * 1 / (1 + exp(-gate[b][i][h] * gate_scale[h])).
 * The ring is read per the meta BEFORE the chunk; chunk rows always come
 * from k_chunk / v_chunk.
 *
 * commit = 1 additionally, after every read of the call: writes chunk row j
 * (the last min(t, W) rows) into ring slot (head0 + len0 + j) % W
 * (o1c_ring_commit) and writes the advanced meta to meta_out (o1c_meta):
 * win_len = min(len0 + t, W); on an overflow by ev keys win_head advances by
 * ev (mod W) and far_len grows by ev. meta_out may alias meta.
 *
 * The value sums run split across key ranges (split-KV) with partial
 * (max, sum, numerator) records in `workspace`, reduced by a second kernel
 * that also applies the gate and the commit. num_splits = 0 lets the library
 * choose; a positive value caps the splits per (sequence, KV head, row block)
 * (results agree within f32 rounding for any split count). Calls of 16 or 32
 * query vectors per (sequence, KV head) (one row block each, e.g. speculative
 * verify) with at least twice as many of them as the attention kernel has
 * resident CTAs on the device, and num_splits = 0, run one split each, taken
 * longest first (a one-CTA kernel sorts them first; the order is in the
 * workspace); unless meta_out aliases meta, gate_ready is set or a far field is
 * given (its part joins in the second kernel), the attention kernel then gates,
 * writes and commits them itself and no second kernel runs (the same bits as
 * through the second kernel).
 *
 * Workspace: device memory, 256-byte aligned, no initial contents needed;
 * overlapping calls must not share it. `workspace_bytes` must be at least
 * swa_attend_workspace_min(args). swa_attend_workspace_size(args) (larger for
 * chunks with at least 128 query vectors per KV head) also holds, for the
 * tensor-core prompt kernel, every KV head's sink and window keys split once
 * into operand blocks of 32 keys (f16 hi/lo pairs under a power-of-two scale per
 * block, with the blocks' exponents), which the kernel then copies in whole
 * blocks, and the order in which its CTAs take the row blocks (longest first);
 * with less, a TF32 kernel splits the keys it stages itself (same results within
 * f32 rounding). ev_start / ev_stop, when non-NULL, are recorded on the
 * stream right before and after the main attention kernel (for timing it).
 * gate_ready, when non-NULL, is an event the stream waits for after the
 * attention and before the merge, then the only kernel that reads gate: a caller
 * may still be copying the gate in (on another stream) while the attention
 * runs, and record gate_ready after that copy.
 * err, when non-NULL, is a device word the kernels OR SWA_DERR_* bits into.
 *
 * Errors: SWA_E_NULL, SWA_E_SHAPE (also B * nk > 65534, or more than 65535
 * row blocks: grid limits), SWA_E_ALIGN, SWA_E_WORKSPACE, SWA_E_CUDA.
 */
/* Far field of a chunk ("o1c_msl.metal", cortiq-engine 0.8.79: o1c_far_e,
 * o1c_far, o1c_far_commit and the token path's o1c_tok_far, o1c_tok_merge,
 * o1c_tok_commit; the clip of "dory_msl.metal" dory_ofar). Keys that leave the window are not dropped: every query head
 * keeps m landmarks, each with a running max, mass and numerator of the keys
 * evicted so far, scored against the landmark's query. A row adds to its
 * window the far part: landmark scores s * <q, k~_a> give weights
 * w_b = sum_a exp(fs_a - f) mu[a][b] (clipped at 0 when rect), gains
 * gain_b = w_b exp(f + max_b - fm), far mass sum_b gain_b mass_b and far
 * numerator sum_b gain_b num_b, joined to the near softmax under a common
 * exponent; a negative far mass drops the far part. The row of a full window
 * evicts its oldest key (ring slot win_head) into every landmark first.
 * Per sequence (the pages hold one), all f32, device memory:
 *   k_tilde [B][nk][m][hd]  landmark keys (16-byte aligned)
 *   q_tilde [B][nh][m][hd]  landmark queries (16-byte aligned)
 *   mu      [B][nh][m][m]   landmark weight matrix, row a, column b
 *   mz      [B][nh][2m]     per landmark: running max (score units, -inf when
 *                           empty), then mass; rewritten iff commit = 1
 *   t_hat   [B][nh][m][hd]  per landmark numerator (16-byte aligned);
 *                           rewritten iff commit = 1
 * 1 <= m <= 32. A chunk with a far field has t <= 64 rows (the pages size
 * their far scratch for OB_K = 64) and t <= cap;
 * once the window is full, row j evicts the oldest key still held, and row i
 * sees the evictions of rows 0..i (o1c_far_e / o1c_far). The evicted keys
 * must still be in the ring: do not let swa_prep write the ring in such a
 * step (pass ring_k = ring_v = NULL there) and commit through swa_attend.
 * A sequence whose window is shorter than t sets SWA_DERR_META.
 * meta.far_len counts the evicted keys; with far_len = 0 and no eviction the
 * far part is empty. */
typedef struct swa_far_args {
  int m;                         /* landmarks per query head, 1..32          */
  int rect;                      /* 1: clip negative landmark weights at 0   */
  const float* k_tilde;
  const float* q_tilde;
  const float* mu;
  float* mz;
  float* t_hat;
} swa_far_args;

typedef struct swa_attend_args {
  int B, t, nh, nk, hd, cap, ns;
  float scale;                   /* score scale (e.g. 1/sqrt(hd))           */
  const swa_meta* meta;          /* [B], state before the chunk             */
  const float* q;                /* [B][t][nh][hd] (q_out of swa_prep)      */
  const float* k_chunk;          /* [B][t][nk][hd]                          */
  const float* v_chunk;          /* [B][t][nk][hd]                          */
  float* ring_k;                 /* [B][nk][cap][hd]; written iff commit    */
  float* ring_v;                 /* [B][nk][cap][hd]; written iff commit    */
  const float* sink_k;           /* [B][nk][ns][hd]; NULL allowed if ns = 0 */
  const float* sink_v;           /* [B][nk][ns][hd]; NULL allowed if ns = 0 */
  const float* gate;             /* [B][t][nh][hd]                          */
  const float* gate_scale;       /* [nh][hd]                                */
  float* out;                    /* [B][t][nh][hd]                          */
  void* workspace;               /* split-KV partials                       */
  size_t workspace_bytes;
  int commit;                    /* 1: ring + meta commit after the reads   */
  swa_meta* meta_out;            /* [B]; required when commit = 1           */
  int num_splits;                /* 0: automatic                            */
  uint32_t* err;                 /* optional device error word              */
  cudaEvent_t ev_start;          /* optional                                */
  cudaEvent_t ev_stop;           /* optional                                */
  const swa_far_args* far;       /* optional far field (t <= 64), host struct */
  cudaEvent_t gate_ready;        /* optional: the merge waits for it        */
} swa_attend_args;

/* Bytes of workspace swa_attend needs for these sizes (reads B, t, nh, nk,
 * hd, cap, ns, num_splits; 0 if the sizes are invalid). Queries the current
 * device's SM count on first use. */
size_t swa_attend_workspace_size(const swa_attend_args* args);
/* The smallest workspace swa_attend accepts for these sizes (0 if unsupported). */
size_t swa_attend_workspace_min(const swa_attend_args* args);

int swa_attend(const swa_attend_args* args, cudaStream_t stream);

/*
 * swa_decode_step — one decode token (t = 1) of every sequence in one call:
 * the prep of swa_prep (RoPE angles from pos0 and theta in the kernel, no
 * table) followed by swa_attend with commit = 1 ("dory_msl.metal",
 * cortiq-engine 0.8.57, dory_prep and dory_gate; "o1c_msl.metal",
 * cortiq-engine 0.8.79, o1c_tok_near / o1c_tok_merge / o1c_tok_commit, the
 * page's fused token path: for one token the number of dispatches, not the
 * arithmetic, was the layer's cost).
 *
 * Results are those of swa_prep(rope = NULL, ring_k = ring_v = NULL) and then
 * swa_attend(commit = 1) on the same tensors (bit for bit with the split count
 * the form uses: one per (sequence, KV head) in the one-kernel form, the
 * planner's otherwise; split counts change only the f32 rounding): out[b][h] for every
 * query head; the row's k-hat / v row written to ring slot
 * (win_head + win_len) % W (the evicted key's slot, or the next free one); the
 * advanced meta in meta_out. The ring is read per the meta before the call.
 *
 * When a KV head has at most 8 query heads, meta_out does not alias meta, and
 * either the library's split planner gives every (sequence, KV head) a single
 * CTA or one CTA's keys (sinks + window) hold at most 512 KB of K and V (512
 * keys at hd 128: the launch-bound regime), the whole step is ONE kernel:
 * the CTA of (sequence, KV head) preps that KV head's query heads and its own
 * k / v head, attends with its own row held in shared memory, writes the gated
 * output and commits its row (the committed slot is never a key of the row's
 * window). Otherwise the step runs the prep kernel, the attention and the merge,
 * with q-hat and k-hat in the workspace. swa_decode_launches tells which.
 *
 *   yq [B][nh][hd], yk, yv [B][nk][hd], gate [B][nh][hd]    the row's inputs
 *   q_scale, gate_scale [nh][hd]
 *   pos0 [B] u32 device: the row's absolute position (angles)
 *   meta [B] device, before the step; meta_out [B] device, after it
 *   ring_k, ring_v [B][nk][cap][hd]; sink_k, sink_v [B][nk][ns][hd] (NULL if ns = 0)
 *   out [B][nh][hd]
 *   workspace   swa_decode_workspace_size(args) bytes, 256-byte aligned (may be
 *               NULL when that is 0); no initial contents; not shared by
 *               overlapping calls
 *   err         optional device error word (SWA_DERR_META, SWA_DERR_TIMEOUT)
 *   ev_start / ev_stop   optional, recorded around the attention kernel (the
 *               whole step in the one-kernel form)
 * Errors: SWA_E_NULL, SWA_E_SHAPE, SWA_E_ALIGN, SWA_E_WORKSPACE, SWA_E_CUDA
 * (as swa_prep and swa_attend; eps < 0, theta <= 0 or a non-finite scale are
 * SWA_E_SHAPE).
 */
typedef struct swa_decode_args {
  int B, nh, nk, hd, cap, ns;
  float scale;                   /* score scale (e.g. 1/sqrt(hd))           */
  float eps;                     /* added to the sum of squares             */
  double theta;                  /* RoPE base                               */
  const float* yq;               /* [B][nh][hd]                             */
  const float* yk;               /* [B][nk][hd]                             */
  const float* yv;               /* [B][nk][hd]                             */
  const float* q_scale;          /* [nh][hd]                                */
  const uint32_t* pos0;          /* [B]                                     */
  const swa_meta* meta;          /* [B], state before the step              */
  float* ring_k;                 /* [B][nk][cap][hd], read and committed    */
  float* ring_v;                 /* [B][nk][cap][hd], read and committed    */
  const float* sink_k;           /* [B][nk][ns][hd]; NULL allowed if ns = 0 */
  const float* sink_v;           /* [B][nk][ns][hd]; NULL allowed if ns = 0 */
  const float* gate;             /* [B][nh][hd]                             */
  const float* gate_scale;       /* [nh][hd]                                */
  float* out;                    /* [B][nh][hd]                             */
  swa_meta* meta_out;            /* [B], state after the step               */
  void* workspace;               /* see swa_decode_workspace_size           */
  size_t workspace_bytes;
  uint32_t* err;                 /* optional device error word              */
  cudaEvent_t ev_start;          /* optional                                */
  cudaEvent_t ev_stop;           /* optional                                */
} swa_decode_args;

/* Workspace bytes swa_decode_step needs for these sizes: 0 in the one-kernel
 * form, else room for q-hat, k-hat and swa_attend's workspace (reads B, nh,
 * nk, hd, cap, ns and whether meta_out aliases meta; 0 also when the sizes are
 * invalid). */
size_t swa_decode_workspace_size(const swa_decode_args* args);
/* Kernels one swa_decode_step call with these arguments launches: 1 (one
 * kernel) or 3 (prep, attention, merge); 0 if the sizes are invalid. */
int swa_decode_launches(const swa_decode_args* args);
int swa_decode_step(const swa_decode_args* args, cudaStream_t stream);

/* Speculative rollback of the ring meta ("dory_msl.metal", cortiq-engine
 * 0.8.57, kernel dory_o1_back). After a verify step committed t draft rows
 * (swa_attend with commit = 1) and only the first a were accepted, pass
 * n_back[b] = t - a to rewind sequence b's meta by that many tokens, one
 * token at a time as the page does:
 *   - window full (win_len == W, W = window or cap when window is 0): the
 *     length stays W, win_head steps back one slot mod W and far_len drops
 *     by one (modulo 2^32). A full window stays full, and its oldest slots
 *     keep the rejected rows' keys: the keys those rows evicted are gone.
 *   - otherwise: win_len drops by one. Exact: the rejected rows' slots fall
 *     outside the window again.
 * The ring contents are not touched.
 *   meta    [B] device, updated in place (state after the verify's commit)
 *   n_back  [B] int32 device, >= 0
 *   cap     ring capacity the meta refers to
 *   err     optional device error word: SWA_DERR_META when a meta is out of
 *           range, n_back is negative, or a window that is not full would
 *           drop below zero keys; that sequence's meta is left unchanged.
 * Errors: SWA_E_NULL (meta or n_back NULL), SWA_E_SHAPE (B < 1 or cap < 1),
 * SWA_E_ALIGN (meta not 16-byte aligned), SWA_E_CUDA. One launch, no
 * synchronisation. */
int swa_rollback(swa_meta* meta, const int32_t* n_back, int B, int cap, uint32_t* err,
                 cudaStream_t stream);

/*
 * swa_attend_noalloc — swa_attend for callers that cannot allocate device
 * memory. The pages have no counterpart: it is a deployment convenience of
 * this library, not part of the method.
 *
 * Some callers cannot call cudaMalloc at all: a plugin that its host program
 * hands only the input and output buffers, a serving engine whose device
 * memory is reserved up front by its own allocator, or a latency-critical loop
 * that must not take the device-wide synchronisation an allocation can cause.
 * This entry point runs exactly what swa_attend runs, with the split-KV
 * scratch (per-split partial records and valid-split counts) taken from a
 * fixed array of SWA_NOALLOC_SCRATCH_BYTES that the library owns; every GPU
 * that loads the library holds that array until the process exits.
 *
 * args->workspace and args->workspace_bytes are ignored; every other field
 * means what it means for swa_attend, and the caller still passes all inputs
 * and outputs. Nothing is allocated: no cudaMalloc, cudaFree or allocating
 * library call.
 *   - Sizes whose scratch need (swa_attend_workspace_min) exceeds
 *     SWA_NOALLOC_SCRATCH_BYTES are refused with SWA_E_WORKSPACE before
 *     anything is enqueued; use swa_attend with your own workspace for them.
 *     The split-once operand blocks of the tensor-core prompt kernel are used
 *     when swa_attend_workspace_size fits the array too.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it with the
 *     id of the device's context; make that first call before any stream
 *     capture. A call that finds another context current (after
 *     cudaDeviceReset, for instance) looks the address up again, so make the
 *     first call after a reset outside any capture as well.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Nothing in it needs to start at zero (every record is written before it
 *     is read within a call), but calls that overlap on the GPU (different
 *     streams, or different host threads, without ordering between them)
 *     race on it and corrupt each other's results: order them.
 * Errors: those of swa_attend, in the same order (NULL pointers, sizes,
 * alignment), then SWA_E_WORKSPACE for oversized calls and SWA_E_CUDA if the
 * address lookup fails.
 */
#define SWA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int swa_attend_noalloc(const swa_attend_args* args, cudaStream_t stream);

/*
 * swa_flash — full-sequence attention over packed q|k|v rows, the second
 * workload beside the token path ("egemma2_msl.metal", cortiq-engine 0.8.17,
 * kernels eg_flash64 / eg_flash_staged): every query row of a segment attends
 * every key row of the same segment (no window, no causal mask, no sinks, no
 * gate), q head h reads K/V head h / (nh / nk), scores are multiplied by
 * `scale`, the softmax is max-subtracted in f32 and the value sum is divided by
 * the weight sum. Both products run on the tensor cores with f32 accuracy (f16
 * hi/lo operands under power-of-two block scales with a workspace, 3xTF32
 * without), with each K/V block of a KV head staged in shared memory once per
 * 128 query vectors (the rows x query heads of that KV head).
 *
 *   qkv      [T][ld] f32: row r holds q head h at qkv + r*ld + q_off + h*hd and
 *            K / V head g at k_off + g*hd / v_off + g*hd; read in place.
 *   segs     [nseg][2] u32 on the device: first row and length of each segment.
 *            A segment with first + length > T or length > max_len is skipped
 *            and sets SWA_DERR_SEGMENT; empty segments are allowed. Segments
 *            must not overlap (their outputs would race); this is not checked.
 *   out      [T][ldo] f32: row r of a segment receives head h at
 *            out + r*ldo + h*hd (nh * hd <= ldo); other rows are not written.
 *   max_len  an upper bound of the segment lengths (>= 1); it sizes the grid.
 *   ld, ldo, q_off, k_off, v_off   in floats, multiples of 4 (16-byte rows).
 *   hd       64 or 128.  nh % nk == 0 and nh / nk <= 32.
 *   scale    finite.
 *   err      optional device word (SWA_DERR_SEGMENT, SWA_DERR_TIMEOUT).
 *   ev_start, ev_stop  optional events recorded on `stream` right before and
 *            after the attention kernel (NULL: none).
 *   workspace, workspace_bytes  optional device scratch (256-byte aligned) of
 *            at least swa_flash_workspace_size(args) bytes, no initial contents
 *            needed, not shared by calls that overlap on the GPU. With it, a first
 *            kernel splits each KV head's K and V rows into f16 hi/lo operand
 *            blocks of 32 keys (each block scaled by a power of two) once per
 *            call and orders the blocks of 128 query vectors longest first; one
 *            persistent CTA per SM then walks them, copying operand blocks whole.
 *            When those blocks leave a last round of at most half the SMs, and
 *            the workspace has room for it, the last (shortest) blocks run as
 *            several key ranges each whose partial sums the last range combines.
 *            Without a workspace (NULL), one CTA per block of query vectors
 *            splits the rows it stages into TF32 hi/lo itself. Both forms are
 *            deterministic and agree within f32 rounding.
 * The call allocates nothing. Errors: SWA_E_NULL (qkv, segs or out NULL),
 * SWA_E_SHAPE (sizes, offsets past ld, nh * hd > ldo, nseg < 1, max_len < 1,
 * scale not finite, nseg * nk > 65534, more than 65535 blocks of query vectors
 * per segment and KV head, or 2^31 of them in all), SWA_E_ALIGN (pointers not 16-byte aligned, workspace not
 * 256-byte aligned, or ld / ldo / offsets not multiples of 4),
 * SWA_E_WORKSPACE (a workspace smaller than needed), SWA_E_CUDA.
 */
typedef struct swa_flash_args {
  int T, nseg, hd, nh, nk;
  int ld, q_off, k_off, v_off, ldo;
  int max_len;
  float scale;
  const float* qkv;            /* [T][ld] */
  const uint32_t* segs;        /* [nseg][2]: first row, length */
  float* out;                  /* [T][ldo] */
  uint32_t* err;               /* optional */
  cudaEvent_t ev_start, ev_stop;  /* optional */
  void* workspace;             /* optional */
  size_t workspace_bytes;
} swa_flash_args;
/* Workspace bytes of the split-once form of swa_flash: nseg * nk *
 * ceil(max_len / 32) blocks of 4 x 32 x hd halves and their two exponents, an
 * int per block of query vectors (the order), plus, when the launch has a split
 * tail on the current device, its partial records (128 x (hd + 4) floats per
 * key range, at most one range per SM) and counters; each part rounded up to
 * 256 bytes; 0 for unsupported sizes. Queries the current device's SM count on
 * first use. */
size_t swa_flash_workspace_size(const swa_flash_args* args);
int swa_flash(const swa_flash_args* args, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SWA_H */
