"""CPU oracle of the sliding-window GQA token path: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import or run this module. The product path (the CUDA
library and its Python binding) never touches it, and this module imports
nothing from the product package.

Everything is computed in float64 with plain NumPy, one (sequence, row, head)
at a time, with the key list of each row written out explicitly, so a reader
can check it against the pages' definitions by eye. Sources (Metal shader
pages of the ``cortiq-engine`` crate on docs.rs):

* "dory_msl.metal" (cortiq-engine 0.8.57): ``dory_prep`` (rotation, unit heads,
  query scale, ring write), ``low_key`` (first key of a window),
  ``dory_gate`` (sigmoid output gate).
* "o1c_msl.metal" (cortiq-engine 0.8.79): header comment (meta and buffer
  layouts), ``o1c_score`` (a row's key list: sinks, ring, chunk rows),
  ``o1c_soft`` / ``o1c_add`` (softmax and value sum), ``o1c_cols`` (a row's
  readable columns), ``o1c_ring_commit`` and ``o1c_meta`` (state after a chunk).
* "egemma2_msl.metal" (cortiq-engine 0.8.17): ``eg_qkv_prep`` (rotate-half
  pairing of a head and the [*, hd/2] cos/sin tables).

Readings where the pages are silent:
* the RoPE table holds, per row, cos of the hd/2 angles then their sines,
  angle_e = pos * theta^(-2e/hd), pos = pos0 + row (the pages consume the
  table but do not build it);
* the attend reads chunk rows from the chunk buffers and ring rows only for
  logical keys older than the chunk; the chunk is committed to the ring after
  every read (o1c_ring_commit runs after the attention);
* without a far field (``attend``) no far terms enter the denominator and
  far_len is only advanced by the commit, as o1c_meta does; the far field
  below gives a row a far part only when far_len plus its own evictions is
  positive;
* softmax starts from -inf and has no denominator clamp (every row attends at
  least its own key, so the sum is >= 1).

The far field of a decode row (``far_*``, ``attend_far*``) follows
"o1c_msl.metal" ``o1c_tok_far`` / ``o1c_tok_merge`` / ``o1c_tok_commit`` and the
optional clip of "dory_msl.metal" ``dory_ofar`` (``rect``). Reading: the state
(landmark keys and queries, the m x m matrix mu, per-landmark max / mass /
numerator) is per sequence; the pages hold one sequence and never build it.

The full-sequence attention (``flash_row``, ``flash_attention``) follows
"egemma2_msl.metal" (cortiq-engine 0.8.17) ``eg_flash64`` / ``eg_flash_staged``:
every row of a segment attends every row of the same segment (no window, no
causal mask), grouped query heads, Q/K/V read in place from a packed row
buffer; pinned against a masked dense attention over the whole buffer, closed
forms (one key, two keys, zero query) and row-permutation / segment
independence.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, a library attention routine on a materialised sequence,
invariants, hand-derived integer fixtures under ``tests/golden/``) except the
RoPE frequency schedule beyond the closed-form entries it checks and the
default score scale 1/sqrt(hd) for workloads whose scale the pages leave
open: those two readings are "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# meta = win_len | win_head | far_len | window  (o1c_msl.metal, header comment)
# ---------------------------------------------------------------------------
WIN_LEN, WIN_HEAD, FAR_LEN, WINDOW = 0, 1, 2, 3


def ring_modulus(meta_b, cap):
    """The ring wraps modulo the sequence's window; a zero window means the
    ring capacity (o1c_msl.metal, ``wgf``)."""
    w = int(meta_b[WINDOW])
    return w if w != 0 else int(cap)


# ---------------------------------------------------------------------------
# Prep: rotation, unit heads, query scale, ring write (dory_msl.metal, dory_prep)
# ---------------------------------------------------------------------------
def rope_table(pos0, t, hd, theta=10000.0):
    """[B][t][hd] table: cos(angle_e) for e < hd/2, then sin(angle_e),
    angle_e = (pos0[b] + j) * theta^(-2e/hd). Reading of the table that
    dory_prep and eg_qkv_prep consume (they read cos at [e], sin at [hd/2 + e])."""
    pos0 = np.asarray(pos0, dtype=np.int64).reshape(-1)
    B = pos0.shape[0]
    half = hd // 2
    tab = np.zeros((B, t, hd), dtype=np.float64)
    for b in range(B):
        for j in range(t):
            pos = float(pos0[b] + j)
            for e in range(half):
                ang = pos * theta ** (-2.0 * e / hd)
                tab[b, j, e] = np.cos(ang)
                tab[b, j, half + e] = np.sin(ang)
    return tab


def rotate_head(head, cos_half, sin_half):
    """Rotate-half RoPE of one head: feature e pairs with e + hd/2,
    u = x*cos - y*sin, v = y*cos + x*sin (dory_prep)."""
    half = head.shape[-1] // 2
    x = head[:half]
    y = head[half:]
    u = x * cos_half - y * sin_half
    v = y * cos_half + x * sin_half
    return np.concatenate([u, v])


def unit_head(rot, eps):
    """rot / sqrt(sum(rot^2) + eps): eps inside the root of the SUM of squares
    (dory_prep: ``1/sqrt(simd_sum(dot(u,u)+dot(v,v)) + eps)``)."""
    return rot / np.sqrt(np.sum(rot * rot) + eps)


def prep(yq, yk, yv, rope, q_scale, eps):
    """Prep of a chunk (dory_prep).

    yq [B][t][nh][hd], yk/yv [B][t][nk][hd], rope [B][t][hd], q_scale [nh][hd].
    Returns (q_hat [B][t][nh][hd], k_hat [B][t][nk][hd], v [B][t][nk][hd]) in f64:
      q_hat = unit(rotate(yq)) * q_scale[h]   (per head and feature)
      k_hat = unit(rotate(yk))
      v     = yv unchanged (no rotation, no norm)
    """
    yq = np.asarray(yq, np.float64)
    yk = np.asarray(yk, np.float64)
    yv = np.asarray(yv, np.float64)
    rope = np.asarray(rope, np.float64)
    q_scale = np.asarray(q_scale, np.float64)
    B, t, nh, hd = yq.shape
    nk = yk.shape[2]
    half = hd // 2
    q_hat = np.zeros_like(yq)
    k_hat = np.zeros_like(yk)
    for b in range(B):
        for j in range(t):
            c = rope[b, j, :half]
            s = rope[b, j, half:]
            for h in range(nh):
                q_hat[b, j, h] = unit_head(rotate_head(yq[b, j, h], c, s), eps) * q_scale[h]
            for g in range(nk):
                k_hat[b, j, g] = unit_head(rotate_head(yk[b, j, g], c, s), eps)
    return q_hat, k_hat, yv.copy()


def prep_ring_slot(pos0_b, j, cap):
    """Ring slot of chunk row j in the prep's ring write: (pos0 + j) % cap
    (dory_prep)."""
    return (int(pos0_b) + j) % int(cap)


def prep_ring_write(ring_k, ring_v, k_hat, v, pos0, cap):
    """Returns copies of the rings with every chunk row written at its prep slot
    (rows in order, so a later row that lands on the same slot wins)."""
    rk = np.array(ring_k, dtype=np.float64, copy=True)
    rv = np.array(ring_v, dtype=np.float64, copy=True)
    B, t, nk, _ = k_hat.shape
    for b in range(B):
        for j in range(t):
            slot = prep_ring_slot(pos0[b], j, cap)
            for g in range(nk):
                rk[b, g, slot] = k_hat[b, j, g]
                rv[b, g, slot] = v[b, j, g]
    return rk, rv


# ---------------------------------------------------------------------------
# Attend (o1c_msl.metal: o1c_score, o1c_max, o1c_soft, o1c_sum, o1c_add, o1c_cols;
# dory_msl.metal: low_key, dory_gate)
# ---------------------------------------------------------------------------
def row_window(meta_b, i, cap):
    """Logical key range [lo, hi] of chunk row i (inclusive). The window counts
    the row itself: win = min(W, len0 + i + 1), lo = len0 + i + 1 - win,
    hi = len0 + i (o1c_score; dory_msl.metal low_key)."""
    len0 = int(meta_b[WIN_LEN])
    W = ring_modulus(meta_b, cap)
    win = min(W, len0 + i + 1)
    lo = len0 + i + 1 - win
    hi = len0 + i
    return lo, hi


def row_key_list(meta_b, i, ns, cap):
    """The keys of row i, in the pages' order: the sinks, then logical keys
    x = lo..hi; x < len0 is ring slot (win_head + x) % W, x >= len0 is chunk
    row x - len0 (o1c_score)."""
    len0 = int(meta_b[WIN_LEN])
    head0 = int(meta_b[WIN_HEAD])
    W = ring_modulus(meta_b, cap)
    keys = [("sink", s) for s in range(ns)]
    lo, hi = row_window(meta_b, i, cap)
    for x in range(lo, hi + 1):
        if x < len0:
            keys.append(("ring", (head0 + x) % W))
        else:
            keys.append(("chunk", x - len0))
    return keys


def sigmoid_gate(gate_value, gate_scale_value):
    """1 / (1 + exp(-g * s_g)) (dory_gate)."""
    return 1.0 / (1.0 + np.exp(-(gate_value * gate_scale_value)))


def attend_row(b, i, h, inp, scale, hpg, return_weights=False):
    """Output of query head h of chunk row i of sequence b.

    inp holds: meta [B][4], q [B][t][nh][hd], k_chunk/v_chunk [B][t][nk][hd],
    ring_k/ring_v [B][nk][cap][hd], sink_k/sink_v [B][nk][ns][hd],
    gate [B][t][nh][hd], gate_scale [nh][hd].
    s_k = scale * <q, key_k>; m = max s; p_k = exp(s_k - m);
    o = sum p_k v_k / sum p_k; out = o * sigmoid(gate * gate_scale).
    """
    meta_b = inp["meta"][b]
    g = h // hpg
    cap = inp["ring_k"].shape[2]
    ns = inp["sink_k"].shape[2]
    keys = row_key_list(meta_b, i, ns, cap)
    q = np.asarray(inp["q"][b, i, h], np.float64)
    K = []
    V = []
    for kind, idx in keys:
        if kind == "sink":
            K.append(inp["sink_k"][b, g, idx])
            V.append(inp["sink_v"][b, g, idx])
        elif kind == "ring":
            K.append(inp["ring_k"][b, g, idx])
            V.append(inp["ring_v"][b, g, idx])
        else:
            K.append(inp["k_chunk"][b, idx, g])
            V.append(inp["v_chunk"][b, idx, g])
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    s = scale * (K @ q)
    m = np.max(s)
    p = np.exp(s - m)
    o = (p @ V) / np.sum(p)
    out = o * sigmoid_gate(np.asarray(inp["gate"][b, i, h], np.float64),
                           np.asarray(inp["gate_scale"][h], np.float64))
    if return_weights:
        return out, p / np.sum(p), keys
    return out


def attend(inp, scale, hpg):
    """Every output row: out [B][t][nh][hd] (f64)."""
    B, t, nh, hd = inp["q"].shape
    out = np.zeros((B, t, nh, hd), np.float64)
    for b in range(B):
        for i in range(t):
            for h in range(nh):
                out[b, i, h] = attend_row(b, i, h, inp, scale, hpg)
    return out


# ---------------------------------------------------------------------------
# State after the chunk (o1c_ring_commit, o1c_meta)
# ---------------------------------------------------------------------------
def commit_slot(meta_b, j, cap):
    """Chunk row j lands in slot (win_head + win_len + j) % W: where the key it
    evicts was (o1c_ring_commit)."""
    W = ring_modulus(meta_b, cap)
    return (int(meta_b[WIN_HEAD]) + int(meta_b[WIN_LEN]) + j) % W


def commit_meta(meta_b, t, cap):
    """Meta after t pushes (o1c_meta): len = min(len0 + t, W); on overflow by
    ev keys the head moves by ev (mod W) and far_len grows by ev."""
    len0 = int(meta_b[WIN_LEN])
    head0 = int(meta_b[WIN_HEAD])
    far = int(meta_b[FAR_LEN])
    wfield = int(meta_b[WINDOW])
    W = ring_modulus(meta_b, cap)
    tot = len0 + t
    if tot <= W:
        return np.array([tot, head0, far, wfield], dtype=np.int64)
    ev = tot - W
    return np.array([W, (head0 + ev) % W, far + ev, wfield], dtype=np.int64)


def commit(meta, ring_k, ring_v, k_chunk, v_chunk):
    """Ring and meta after the chunk, rows written in order (a later row that
    lands on the same slot wins, as a sequence of single-row commits would)."""
    rk = np.array(ring_k, dtype=np.float64, copy=True)
    rv = np.array(ring_v, dtype=np.float64, copy=True)
    B, t, nk, _ = k_chunk.shape
    cap = rk.shape[2]
    new_meta = np.zeros((B, 4), dtype=np.int64)
    for b in range(B):
        for j in range(t):
            slot = commit_slot(meta[b], j, cap)
            for g in range(nk):
                rk[b, g, slot] = k_chunk[b, j, g]
                rv[b, g, slot] = v_chunk[b, j, g]
        new_meta[b] = commit_meta(meta[b], t, cap)
    return rk, rv, new_meta


# ---------------------------------------------------------------------------
# Speculative rollback (dory_msl.metal, dory_o1_back)
# ---------------------------------------------------------------------------
def rollback_meta(meta_b, n, cap):
    """Meta after rejecting the last ``n`` pushed tokens, one token at a time
    as dory_o1_back does: while the window is full (win_len equals the ring
    modulus) the head steps back one slot (mod W) and far_len drops by one in
    32-bit unsigned arithmetic; otherwise win_len drops by one. A full window
    therefore stays full. Returns None when a non-full window would have to
    drop below zero keys (an invalid request)."""
    W = ring_modulus(meta_b, cap)
    length = int(meta_b[WIN_LEN])
    head = int(meta_b[WIN_HEAD])
    far = int(meta_b[FAR_LEN])
    for _ in range(int(n)):
        if length == W:
            head = (head + W - 1) % W
            far = (far - 1) % (1 << 32)
        else:
            if length == 0:
                return None
            length -= 1
    return np.array([length, head, far, int(meta_b[WINDOW])], dtype=np.int64)


def rollback(meta, n_back, cap):
    """rollback_meta over a batch; a sequence whose request is invalid keeps
    its meta and is flagged. Returns (new_meta, bad[B])."""
    meta = np.asarray(meta, dtype=np.int64)
    out = meta.copy()
    bad = np.zeros(meta.shape[0], dtype=bool)
    for b in range(meta.shape[0]):
        r = rollback_meta(meta[b], n_back[b], cap)
        if r is None:
            bad[b] = True
        else:
            out[b] = r
    return out, bad


# ---------------------------------------------------------------------------
# Far field of a decode row ("o1c_msl.metal": o1c_tok_far, o1c_tok_merge,
# o1c_tok_commit; "dory_msl.metal": dory_ofar for the optional clip `rect`)
#
# far = {"m": landmarks, "rect": 0/1,
#        "k_tilde": [B][nk][m][hd]  landmark keys of each KV group,
#        "q_tilde": [B][nh][m][hd]  landmark queries of each query head,
#        "mu":      [B][nh][m][m]   the landmark weights' matrix,
#        "mz":      [B][nh][2m]     per landmark: running max, then mass,
#        "t_hat":   [B][nh][m][hd]  per landmark: far numerator}
# One decode row (t = 1) of sequence b. Keys leave the window only when it is
# full (win_len == W): the oldest, ring slot win_head, is evicted by the row.
# ---------------------------------------------------------------------------
def far_evict(mx_b, z_b, k_ev, q_tilde_b, scale):
    """One landmark's running max and mass after an evicted key, as
    o1c_tok_far does: fe = scale * <q~, k>, mx' = max(mx, fe),
    rr = exp(mx - mx') (1 when the max stays; an empty field, mx = -inf,
    gives 0), e = exp(fe - mx'), z' = z * rr + e. Returns (mx', z', rr, e)."""
    fe = scale * float(np.dot(np.asarray(q_tilde_b, np.float64), np.asarray(k_ev, np.float64)))
    mx2 = max(mx_b, fe)
    rr = 1.0 if mx2 == mx_b else math.exp(mx_b - mx2)
    e = math.exp(fe - mx2)
    return mx2, z_b * rr + e, rr, e


def far_part(q, far, b, h, g, mx2, z2, scale):
    """The far part of a row for query head h with the far state mx2, z2 (after
    this row's eviction): landmark scores fs_a = scale * <q, k~_a>, f = max fs;
    w_b = sum_a exp(fs_a - f) mu[a][b] (clipped at 0 with rect); fm = max_b
    (f + mx2_b); gain_b = w_b exp(f + mx2_b - fm); far_den = sum_b gain_b z2_b.
    A negative far_den drops the far part (have = False). Returns
    (have, fm, far_den, gain[m])."""
    m = far["m"]
    kt = np.asarray(far["k_tilde"][b, g], np.float64)
    mu = np.asarray(far["mu"][b, h], np.float64)
    fs = scale * (kt @ np.asarray(q, np.float64))
    f = np.max(fs)
    w = np.exp(fs - f) @ mu                      # w[b] = sum_a exp(fs_a - f) mu[a][b]
    if far["rect"]:
        w = np.maximum(w, 0.0)
    fb = f + np.asarray(mx2, np.float64)
    fm = np.max(fb)
    gain = w * np.exp(fb - fm)
    far_den = float(np.sum(gain * np.asarray(z2, np.float64)))
    if not far_den >= 0.0:
        return False, fm, 0.0, np.zeros(m)
    return True, fm, far_den, gain


def far_evictions(meta_b, t, cap):
    """The chunk rows that evict a key and the ring slot each evicts: with a
    full window (win_len + row + 1 > W) row j evicts the oldest key still held,
    logical key j - j0 with j0 = W - win_len, i.e. ring slot
    (win_head + j - j0) % W (o1c_far_e). Chunks with a far field are at most W
    rows long, so every evicted key is a ring key."""
    W = ring_modulus(meta_b, cap)
    j0 = W - int(meta_b[WIN_LEN])
    head0 = int(meta_b[WIN_HEAD])
    return [(j, (head0 + j - j0) % W) for j in range(max(j0, 0), t)]


def far_row_state(meta_b, far, b, h, g, inp, scale, row=0):
    """The far state of head h as row `row` of the chunk sees it: every
    eviction of rows 0..row applied in order (far_evict per landmark), with
    the landmark numerators t_hat * rr + e * v. Returns (evictions, mx, z,
    t_hat) after them."""
    cap = inp["ring_k"].shape[2]
    m = far["m"]
    mx = np.array(far["mz"][b, h, :m], np.float64)
    z = np.array(far["mz"][b, h, m:], np.float64)
    th = np.array(far["t_hat"][b, h], np.float64)
    t = inp["q"].shape[1]
    n_ev = 0
    for j, slot in far_evictions(meta_b, t, cap):
        if j > row:
            break
        n_ev += 1
        k_ev = inp["ring_k"][b, g, slot]
        v_ev = np.asarray(inp["ring_v"][b, g, slot], np.float64)
        for a in range(m):
            mx[a], z[a], rr, e = far_evict(float(mx[a]), float(z[a]), k_ev, far["q_tilde"][b, h, a], scale)
            th[a] = th[a] * rr + e * v_ev
    return n_ev, mx, z, th


def attend_far_row(b, h, inp, far, scale, hpg, i=0):
    """Output of query head h of chunk row i of sequence b with the far field
    (o1c_far / o1c_tok_far, o1c_tok_merge, then dory_gate): with c the larger
    of the near max and (when the far part is kept) fm,
    o = (sum_near exp(s - c) v + exp(fm - c) sum_b gain_b t_hat_b)
        / (sum_near exp(s - c) + exp(fm - c) far_den),
    over the far state after the evictions of rows 0..i."""
    meta_b = inp["meta"][b]
    g = h // hpg
    cap = inp["ring_k"].shape[2]
    ns = inp["sink_k"].shape[2]
    keys = row_key_list(meta_b, i, ns, cap)
    q = np.asarray(inp["q"][b, i, h], np.float64)
    K, V = [], []
    for kind, idx in keys:
        if kind == "sink":
            K.append(inp["sink_k"][b, g, idx])
            V.append(inp["sink_v"][b, g, idx])
        elif kind == "ring":
            K.append(inp["ring_k"][b, g, idx])
            V.append(inp["ring_v"][b, g, idx])
        else:
            K.append(inp["k_chunk"][b, idx, g])
            V.append(inp["v_chunk"][b, idx, g])
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    s = scale * (K @ q)
    n_ev, mx2, z2, th2 = far_row_state(meta_b, far, b, h, g, inp, scale, row=i)
    farl = int(meta_b[FAR_LEN]) + n_ev
    have, fm, far_den, gain = (False, -np.inf, 0.0, None)
    if farl > 0:
        have, fm, far_den, gain = far_part(q, far, b, h, g, mx2, z2, scale)
    c = max(np.max(s), fm) if have else np.max(s)
    p = np.exp(s - c)
    num = p @ V
    den = np.sum(p)
    if have:
        sf = math.exp(fm - c)
        num = num + sf * (gain @ th2)
        den = den + sf * far_den
    o = num / den
    return o * sigmoid_gate(np.asarray(inp["gate"][b, i, h], np.float64),
                            np.asarray(inp["gate_scale"][h], np.float64))


def attend_far(inp, far, scale, hpg):
    """Every output of a chunk with the far field: out [B][t][nh][hd]. Far
    chunks are at most min(W, 64) rows ("o1c_msl.metal" sizes its far scratch
    for OB_K = 64 rows; within W rows every evicted key is a ring key)."""
    B, t, nh, hd = inp["q"].shape
    out = np.zeros((B, t, nh, hd), np.float64)
    for b in range(B):
        for i in range(t):
            for h in range(nh):
                out[b, i, h] = attend_far_row(b, h, inp, far, scale, hpg, i)
    return out


def far_commit(inp, far, scale, hpg):
    """The far state after the chunk (o1c_far_commit / o1c_tok_commit, far
    part): every key the chunk evicts joins every landmark of every head, in
    row order. Returns (mz, t_hat)."""
    B, t, nh, _ = inp["q"].shape
    m = far["m"]
    mz = np.array(far["mz"], np.float64, copy=True)
    th = np.array(far["t_hat"], np.float64, copy=True)
    for b in range(B):
        for h in range(nh):
            n_ev, mx2, z2, th2 = far_row_state(inp["meta"][b], far, b, h, h // hpg, inp, scale, row=t - 1)
            if n_ev:
                mz[b, h, :m] = mx2
                mz[b, h, m:] = z2
                th[b, h] = th2
    return mz, th


# ---------------------------------------------------------------------------
# Full-sequence attention ("egemma2_msl.metal", cortiq-engine 0.8.17:
# eg_flash64 / eg_flash_staged). Every query row of a segment attends every key
# row of the same segment: no window, no causal mask, no sinks, no gate.
# Grouped query heads (q head h reads K/V head h // group), scores scaled by
# `scale`, max-subtracted softmax, value sum divided by the weight sum.
# Q, K and V are read in place from the rows of one packed buffer qkv[T][ld]:
# q head h at columns q_off + h*hd .. +hd, K/V head g at k_off / v_off + g*hd.
# A segment is (first row, length). Output rows are [nq*hd], head h at h*hd.
# ---------------------------------------------------------------------------
def flash_row(qkv, s0, length, r, h, hd, group, q_off, k_off, v_off, scale):
    """Output of query row s0 + r, head h: softmax over the segment's keys."""
    g = h // group
    q = np.asarray(qkv[s0 + r, q_off + h * hd:q_off + (h + 1) * hd], dtype=np.float64)
    keys = np.asarray(qkv[s0:s0 + length, k_off + g * hd:k_off + (g + 1) * hd], dtype=np.float64)
    vals = np.asarray(qkv[s0:s0 + length, v_off + g * hd:v_off + (g + 1) * hd], dtype=np.float64)
    s = scale * (keys @ q)
    p = np.exp(s - s.max())
    return (p @ vals) / p.sum()


def flash_attention(qkv, segs, hd, nq, group, q_off, k_off, v_off, scale):
    """All segments' rows, every q head: out[T][nq*hd] (rows outside every
    segment stay zero)."""
    out = np.zeros((qkv.shape[0], nq * hd))
    for s0, length in segs:
        for r in range(int(length)):
            for h in range(nq):
                out[s0 + r, h * hd:(h + 1) * hd] = flash_row(qkv, int(s0), int(length), r, h, hd, group,
                                                             q_off, k_off, v_off, scale)
    return out
