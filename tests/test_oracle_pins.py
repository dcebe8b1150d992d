"""Pins of the CPU oracle to things other than itself (CPU only).

Each pin is chosen so that a plausible mistake in the oracle fails it:
  * hand-derived integer fixtures (tests/golden/ring_window_cases.json) for the
    key list, the window bounds, the prep and commit ring slots and the meta
    update (off-by-one in the window, wrong modulus, wrong head advance);
  * closed forms of the rotation (sign, pairing e <-> e + hd/2, frequency of the
    first pair and of pair hd/4), of the unit norm (eps inside the root of the
    sum), of a two-key softmax, of a one-key window and of uniform scores;
  * a library attention routine (torch scaled_dot_product_attention in float64
    with an explicit sliding-window mask) on a materialised logical sequence;
  * invariants: softmax weights sum to 1, ring-rotation invariance, a t-row
    chunk equals t single-row steps with commits, the RoPE relative-position
    identity;
  * for the full-sequence attention: a block-diagonally masked dense attention
    over the whole packed buffer, one-key / two-key / zero-query closed forms,
    row permutation and segment / KV-head independence.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ring_window_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


# ---------------------------------------------------------------------------
# integer fixtures
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_key_lists_and_windows_match_hand_derivation(case):
    meta_b = np.array(case["meta"])
    for row in case["rows"]:
        lo, hi = oracle.row_window(meta_b, row["i"], case["cap"])
        assert (lo, hi) == (row["lo"], row["hi"])
        keys = oracle.row_key_list(meta_b, row["i"], case["ns"], case["cap"])
        assert [[k, int(v)] for k, v in keys] == row["keys"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_commit_slots_ring_and_meta_match_hand_derivation(case):
    meta_b = np.array(case["meta"])
    t, cap = case["t"], case["cap"]
    slots = [oracle.commit_slot(meta_b, j, cap) for j in range(t)]
    assert slots == case["commit_slots"]
    # Tag each chunk row's key with its row index to read back the final ring.
    ring = np.full((1, 1, cap, 1), -1.0)
    kc = np.arange(t, dtype=np.float64).reshape(1, t, 1, 1)
    rk, rv, new_meta = oracle.commit(meta_b.reshape(1, 4), ring, ring, kc, kc)
    expect = np.full(cap, -1.0)
    for slot, row in case["final_ring"].items():
        expect[int(slot)] = row
    np.testing.assert_array_equal(rk[0, 0, :, 0], expect)
    np.testing.assert_array_equal(rv[0, 0, :, 0], expect)
    assert new_meta[0].tolist() == case["meta_after"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_prep_slots_match_hand_derivation(case):
    slots = [oracle.prep_ring_slot(case["pos0"], j, case["cap"]) for j in range(case["t"])]
    assert slots == case["prep_slots"]


# ---------------------------------------------------------------------------
# rotation and unit heads
# ---------------------------------------------------------------------------
def test_rope_table_closed_forms():
    hd, theta = 64, 10000.0
    pos0 = np.array([0, 7, 12345])
    tab = oracle.rope_table(pos0, 3, hd, theta)
    half = hd // 2
    # position 0: the identity rotation
    np.testing.assert_array_equal(tab[0, 0, :half], np.ones(half))
    np.testing.assert_array_equal(tab[0, 0, half:], np.zeros(half))
    for b, p0 in enumerate(pos0):
        for j in range(3):
            pos = int(p0) + j
            # pair 0 turns by pos radians; pair hd/4 by pos / sqrt(theta) = pos / 100
            assert tab[b, j, 0] == pytest.approx(math.cos(pos), abs=1e-12)
            assert tab[b, j, half] == pytest.approx(math.sin(pos), abs=1e-12)
            assert tab[b, j, hd // 4] == pytest.approx(math.cos(pos / 100.0), abs=1e-12)
            assert tab[b, j, half + hd // 4] == pytest.approx(math.sin(pos / 100.0), abs=1e-12)
    # frequencies fall with the pair index
    ang = np.arctan2(oracle.rope_table(np.array([1]), 1, hd, theta)[0, 0, half:],
                     oracle.rope_table(np.array([1]), 1, hd, theta)[0, 0, :half])
    assert np.all(np.diff(ang) < 0)


def test_rotation_sign_and_pairing():
    hd = 8
    c = np.cos(np.array([0.3, 0.5, 0.7, 0.9]))
    s = np.sin(np.array([0.3, 0.5, 0.7, 0.9]))
    x = np.zeros(hd)
    x[1] = 1.0            # first half, pair 1
    r = oracle.rotate_head(x, c, s)
    expect = np.zeros(hd)
    expect[1] = c[1]
    expect[1 + hd // 2] = s[1]   # a rotation by +angle of (1, 0)
    np.testing.assert_allclose(r, expect, atol=1e-15)
    y = np.zeros(hd)
    y[1 + hd // 2] = 1.0  # second half of pair 1
    r = oracle.rotate_head(y, c, s)
    expect = np.zeros(hd)
    expect[1] = -s[1]
    expect[1 + hd // 2] = c[1]
    np.testing.assert_allclose(r, expect, atol=1e-15)


def test_rope_relative_position_identity():
    rng = np.random.default_rng(5)
    hd = 32
    a = rng.standard_normal(hd)
    k = rng.standard_normal(hd)
    tab = oracle.rope_table(np.array([0]), 40, hd)
    half = hd // 2

    def rot(v, p):
        return oracle.rotate_head(v, tab[0, p, :half], tab[0, p, half:])

    for p, q in [(9, 4), (30, 25), (17, 12)]:
        assert np.dot(rot(a, p), rot(k, q)) == pytest.approx(np.dot(rot(a, p - q), k), rel=1e-12)
    # rotation preserves the norm
    assert np.linalg.norm(rot(a, 33)) == pytest.approx(np.linalg.norm(a), rel=1e-12)


def test_unit_norm_puts_eps_inside_root_of_sum():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(64)
    S = float(np.sum(v * v))
    # eps == S halves the squared norm: |v|^2 / (S + eps) = 1/2
    assert np.sum(oracle.unit_head(v, S) ** 2) == pytest.approx(0.5, rel=1e-12)
    assert np.sum(oracle.unit_head(v, 1e-6) ** 2) == pytest.approx(S / (S + 1e-6), rel=1e-12)


def test_prep_norms_scale_and_value_copy():
    w = workloads.custom(B=2, t=3, nh=4, nk=2, hd=32, window=8, cap=8, pos_lo=5)
    inp = workloads.make_inputs(w)
    rope = oracle.rope_table(inp["pos0"].numpy(), w.t, w.hd)
    eps = 1e-6
    q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                          inp["q_scale"].numpy(), eps)
    S_k = np.sum(inp["yk"].numpy().astype(np.float64) ** 2, axis=-1)
    np.testing.assert_allclose(np.sum(k * k, axis=-1), S_k / (S_k + eps), rtol=1e-12)
    S_q = np.sum(inp["yq"].numpy().astype(np.float64) ** 2, axis=-1)
    q_unscaled = q / inp["q_scale"].numpy().astype(np.float64)[None, None]
    np.testing.assert_allclose(np.sum(q_unscaled ** 2, axis=-1), S_q / (S_q + eps), rtol=1e-12)
    np.testing.assert_array_equal(v, inp["yv"].numpy().astype(np.float64))
    # a one-hot query scale keeps exactly that feature
    sq = np.zeros((w.nh, w.hd))
    sq[:, 3] = 2.0
    q1, _, _ = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope, sq, eps)
    assert np.count_nonzero(q1[..., np.arange(w.hd) != 3]) == 0
    np.testing.assert_allclose(q1[..., 3], 2.0 * q_unscaled[..., 3], rtol=1e-12)


# ---------------------------------------------------------------------------
# attention: closed forms
# ---------------------------------------------------------------------------
def _attend_inputs(w, inp, q=None):
    """Oracle attend inputs from the generator's tensors (q from prep unless given)."""
    rope = oracle.rope_table(inp["pos0"].numpy(), w.t, w.hd, w.theta)
    qh, kh, vv = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                             inp["q_scale"].numpy(), w.eps)
    return {
        "meta": inp["meta"].numpy(),
        "q": qh if q is None else q,
        "k_chunk": kh, "v_chunk": vv,
        "ring_k": inp["ring_k"].numpy().astype(np.float64),
        "ring_v": inp["ring_v"].numpy().astype(np.float64),
        "sink_k": inp["sink_k"].numpy().astype(np.float64),
        "sink_v": inp["sink_v"].numpy().astype(np.float64),
        "gate": inp["gate"].numpy().astype(np.float64),
        "gate_scale": inp["gate_scale"].numpy().astype(np.float64),
    }


def test_two_key_softmax_closed_form():
    hd = 4
    inp = {
        "meta": np.array([[0, 0, 0, 1]]),
        "q": np.array([[[[math.log(3.0), 0, 0, 0]]]]),
        "k_chunk": np.zeros((1, 1, 1, hd)),
        "v_chunk": np.array([[[[0.0, 4.0, 0.0, 8.0]]]]),
        "ring_k": np.zeros((1, 1, 1, hd)), "ring_v": np.zeros((1, 1, 1, hd)),
        "sink_k": np.array([[[[1.0, 0, 0, 0]]]]),
        "sink_v": np.array([[[[4.0, 0.0, 8.0, 0.0]]]]),
        "gate": np.array([[[[0.0, 0.0, 1.0, -1.0]]]]),
        "gate_scale": np.array([[1.0, 2.0, 2.0, 2.0]]),
    }
    out = oracle.attend(inp, scale=1.0, hpg=1)
    # weights 3/4 (sink, score ln 3) and 1/4 (chunk row, score 0)
    o = np.array([3.0, 1.0, 6.0, 2.0])
    gate = np.array([0.5, 0.5, expit(2.0), expit(-2.0)])
    np.testing.assert_allclose(out[0, 0, 0], o * gate, rtol=1e-14)


def test_one_key_window_returns_gated_value():
    w = workloads.custom(B=2, t=3, nh=8, nk=2, hd=16, window=1, cap=1, ns=0, pos_lo=9)
    inp = workloads.make_inputs(w)
    a = _attend_inputs(w, inp)
    out = oracle.attend(a, w.score_scale, w.hpg)
    for b in range(w.B):
        for i in range(w.t):
            for h in range(w.nh):
                expect = a["v_chunk"][b, i, h // w.hpg] * expit(a["gate"][b, i, h] * a["gate_scale"][h])
                np.testing.assert_allclose(out[b, i, h], expect, rtol=1e-13, atol=1e-15)


def _textbook_masked_attention(w, a):
    """Materialise each sequence's logical keys (ring un-rotated, then the chunk),
    build the sliding-window causal mask position-wise, and run torch's
    scaled_dot_product_attention in float64."""
    B, t, nh, hd = a["q"].shape
    out = np.zeros_like(a["q"])
    for b in range(B):
        len0, head0, _, wf = (int(x) for x in a["meta"][b])
        W = wf if wf else a["ring_k"].shape[2]
        ring_k = np.stack([a["ring_k"][b, :, (head0 + x) % W] for x in range(len0)], 1) \
            if len0 else np.zeros((w.nk, 0, hd))
        ring_v = np.stack([a["ring_v"][b, :, (head0 + x) % W] for x in range(len0)], 1) \
            if len0 else np.zeros((w.nk, 0, hd))
        seq_k = np.concatenate([a["sink_k"][b], ring_k, a["k_chunk"][b].transpose(1, 0, 2)], 1)
        seq_v = np.concatenate([a["sink_v"][b], ring_v, a["v_chunk"][b].transpose(1, 0, 2)], 1)
        n = seq_k.shape[1]
        mask = np.zeros((t, n), dtype=bool)
        for i in range(t):
            qpos = len0 + i          # logical position of row i
            for col in range(n):
                if col < w.ns:
                    mask[i, col] = True
                else:
                    kpos = col - w.ns
                    mask[i, col] = kpos <= qpos and qpos - kpos < W
        for h in range(nh):
            g = h // w.hpg
            q = torch.tensor(a["q"][b, :, h][None, None])           # [1,1,t,hd]
            k = torch.tensor(seq_k[g][None, None])
            v = torch.tensor(seq_v[g][None, None])
            o = torch.nn.functional.scaled_dot_product_attention(
                q, k, v, attn_mask=torch.tensor(mask)[None, None], scale=w.score_scale)
            gate = expit(a["gate"][b, :, h] * a["gate_scale"][h][None])
            out[b, :, h] = o[0, 0].numpy() * gate
    return out


SDPA_CASES = [
    dict(B=2, t=1, nh=8, nk=2, hd=16, window=12, cap=12, ns=0, pos_mode="fixed", pos_lo=29),
    dict(B=3, t=4, nh=6, nk=2, hd=8, window=10, cap=10, ns=2, pos_mode="partial", pos_lo=1, pos_hi=10),
    dict(B=2, t=7, nh=4, nk=1, hd=8, window=5, cap=5, ns=1, pos_mode="prompt", pos_lo=0, pos_hi=9),
    dict(B=2, t=9, nh=4, nk=2, hd=8, window=3, cap=3, ns=3, pos_mode="full", pos_lo=3, pos_hi=40),
    dict(B=1, t=5, nh=2, nk=2, hd=4, window=16, cap=16, ns=0, pos_mode="fixed", pos_lo=0),
]


@pytest.mark.parametrize("kw", SDPA_CASES)
@pytest.mark.parametrize("sharp", [False, True])
def test_attend_matches_library_attention_on_materialised_sequence(kw, sharp):
    w = workloads.custom(scale=3.0 if sharp else None, **kw)
    inp = workloads.make_inputs(w)
    a = _attend_inputs(w, inp)
    out = oracle.attend(a, w.score_scale, w.hpg)
    ref = _textbook_masked_attention(w, a)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_softmax_weights_sum_to_one_and_follow_scores():
    w = workloads.custom(B=1, t=3, nh=4, nk=1, hd=16, window=9, cap=9, ns=2, pos_mode="full",
                         pos_lo=9, pos_hi=30, scale=2.0)
    a = _attend_inputs(w, workloads.make_inputs(w))
    for i in range(w.t):
        for h in range(w.nh):
            _, p, keys = oracle.attend_row(0, i, h, a, w.score_scale, w.hpg, return_weights=True)
            assert p.sum() == pytest.approx(1.0, abs=1e-14)
            assert len(p) == w.ns + min(9, int(a["meta"][0][0]) + i + 1)


def test_uniform_scores_return_window_mean():
    w = workloads.custom(B=2, t=4, nh=4, nk=2, hd=8, window=6, cap=6, ns=1, pos_mode="full",
                         pos_lo=6, pos_hi=50)
    inp = workloads.make_inputs(w)
    a = _attend_inputs(w, inp, q=np.zeros((w.B, w.t, w.nh, w.hd)))
    out = oracle.attend(a, w.score_scale, w.hpg)
    for b in range(w.B):
        len0, head0 = int(a["meta"][b][0]), int(a["meta"][b][1])
        for i in range(w.t):
            for h in range(w.nh):
                g = h // w.hpg
                vals = [a["sink_v"][b, g, 0]]
                qpos = len0 + i
                for kpos in range(qpos - 6 + 1, qpos + 1):   # the 6 newest positions
                    vals.append(a["ring_v"][b, g, (head0 + kpos) % 6] if kpos < len0
                                else a["v_chunk"][b, kpos - len0, g])
                expect = np.mean(vals, axis=0) * expit(a["gate"][b, i, h] * a["gate_scale"][h])
                np.testing.assert_allclose(out[b, i, h], expect, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
def test_ring_rotation_invariance():
    w = workloads.custom(B=2, t=3, nh=4, nk=2, hd=8, window=7, cap=7, ns=2, pos_mode="full",
                         pos_lo=7, pos_hi=60, scale=2.0)
    a = _attend_inputs(w, workloads.make_inputs(w))
    base = oracle.attend(a, w.score_scale, w.hpg)
    for r in (1, 3, 6):
        b2 = dict(a)
        b2["ring_k"] = np.roll(a["ring_k"], r, axis=2)
        b2["ring_v"] = np.roll(a["ring_v"], r, axis=2)
        m = a["meta"].copy()
        m[:, 1] = (m[:, 1] + r) % 7
        b2["meta"] = m
        np.testing.assert_allclose(oracle.attend(b2, w.score_scale, w.hpg), base, rtol=1e-13,
                                   atol=1e-15)


@pytest.mark.parametrize("kw", [
    dict(B=2, t=5, nh=4, nk=2, hd=8, window=4, cap=4, ns=1, pos_mode="full", pos_lo=4, pos_hi=30),
    dict(B=2, t=6, nh=2, nk=1, hd=8, window=8, cap=8, ns=0, pos_mode="partial", pos_lo=1, pos_hi=8),
])
def test_chunk_equals_sequential_single_row_steps(kw):
    w = workloads.custom(scale=2.0, **kw)
    a = _attend_inputs(w, workloads.make_inputs(w))
    out_chunk = oracle.attend(a, w.score_scale, w.hpg)
    rk_c, rv_c, meta_c = oracle.commit(a["meta"], a["ring_k"], a["ring_v"], a["k_chunk"], a["v_chunk"])
    meta = a["meta"].copy()
    rk, rv = a["ring_k"].copy(), a["ring_v"].copy()
    for i in range(w.t):
        step = {
            "meta": meta, "q": a["q"][:, i:i + 1], "k_chunk": a["k_chunk"][:, i:i + 1],
            "v_chunk": a["v_chunk"][:, i:i + 1], "ring_k": rk, "ring_v": rv,
            "sink_k": a["sink_k"], "sink_v": a["sink_v"], "gate": a["gate"][:, i:i + 1],
            "gate_scale": a["gate_scale"],
        }
        o = oracle.attend(step, w.score_scale, w.hpg)
        np.testing.assert_allclose(o[:, 0], out_chunk[:, i], rtol=1e-13, atol=1e-15)
        rk, rv, meta = oracle.commit(meta, rk, rv, step["k_chunk"], step["v_chunk"])
    np.testing.assert_array_equal(rk, rk_c)
    np.testing.assert_array_equal(rv, rv_c)
    np.testing.assert_array_equal(meta, meta_c)


def test_commit_after_prep_grown_ring_matches_prep_slots():
    """For a ring grown from position 0 (win_head = (pos0 - win_len) % W, W = cap),
    the commit slot equals the prep slot (pos0 + j) % cap."""
    for name in ("tiny_decode", "batched_decode", "spec_verify", "prompt_chunk", "long_decode"):
        w = workloads.WORKLOADS[name]
        pos0, meta = workloads.make_meta(w, torch.Generator().manual_seed(w.seed))
        for b in range(meta.shape[0]):
            for j in (0, w.t - 1):
                assert oracle.commit_slot(meta[b].numpy(), j, w.cap) == \
                    oracle.prep_ring_slot(int(pos0[b]), j, w.cap)


# ---------------------------------------------------------------------------
# speculative rollback (dory_msl.metal, dory_o1_back)
# ---------------------------------------------------------------------------
ROLLBACK_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rollback_cases.json")
with open(ROLLBACK_GOLDEN) as _f:
    ROLLBACK_CASES = json.load(_f)["cases"]


@pytest.mark.parametrize("case", ROLLBACK_CASES, ids=[c["name"] for c in ROLLBACK_CASES])
def test_rollback_matches_hand_derivation(case):
    got = oracle.rollback_meta(np.array(case["meta"]), case["n"], case["cap"])
    if case["after"] is None:
        assert got is None
    else:
        assert got is not None and got.tolist() == case["after"]


@pytest.mark.parametrize("len0,t,W", [(0, 5, 16), (3, 12, 16), (16, 5, 16), (16, 40, 16), (6, 1, 8)])
def test_rollback_undoes_a_commit_that_never_changes_fullness(len0, t, W):
    # a window that stays below W, or is full throughout, returns exactly to
    # the meta before the commit (o1c_meta forward, dory_o1_back backward)
    meta = np.array([len0, 5 % W, 11, W])
    fwd = oracle.commit_meta(meta, t, W)
    back = oracle.rollback_meta(fwd, t, W)
    assert back.tolist() == meta.tolist()


def test_rollback_after_a_commit_that_fills_the_window_stays_full():
    # len0 + t crosses W: the forward commit evicts ev keys; rewinding t tokens
    # keeps the window full and moves the head back t slots from where the
    # commit left it, so it ends t - ev slots before the original head
    W, len0, t, head0 = 16, 12, 7, 3
    fwd = oracle.commit_meta(np.array([len0, head0, 0, W]), t, W)
    ev = len0 + t - W
    assert fwd.tolist() == [W, (head0 + ev) % W, ev, W]
    back = oracle.rollback_meta(fwd, t, W)
    assert back.tolist() == [W, (head0 + ev - t) % W, (ev - t) % (1 << 32), W]


def test_rollback_batch_flags_only_invalid_sequences():
    meta = np.array([[5, 0, 0, 8], [8, 3, 2, 8], [2, 1, 0, 8]])
    out, bad = oracle.rollback(meta, [2, 1, 3], 8)
    assert bad.tolist() == [False, False, True]
    assert out.tolist() == [[3, 0, 0, 8], [8, 2, 1, 8], [2, 1, 0, 8]]


# ---------------------------------------------------------------------------
# far field of a decode row (o1c_msl.metal: o1c_tok_far, o1c_tok_merge,
# o1c_tok_commit; dory_msl.metal: dory_ofar)
# ---------------------------------------------------------------------------
def test_far_eviction_running_max_and_mass_closed_forms():
    q = np.array([1.0, 0.0, 0.0, 0.0])
    k1, k2 = np.array([0.5, 0, 0, 0]), np.array([2.0, 0, 0, 0])
    mx, z, rr, e = oracle.far_evict(-np.inf, 0.0, k1, q, 1.0)    # empty field
    assert (mx, z, rr, e) == (0.5, 1.0, 0.0, 1.0)
    mx, z, rr, e = oracle.far_evict(mx, z, k2, q, 1.0)           # larger score moves the max
    assert mx == 2.0 and rr == pytest.approx(math.exp(-1.5)) and e == 1.0
    assert z == pytest.approx(1.0 + math.exp(-1.5))
    mx, z, rr, e = oracle.far_evict(mx, z, k1, q, 1.0)           # smaller score keeps it
    assert mx == 2.0 and rr == 1.0 and e == pytest.approx(math.exp(-1.5))
    assert z == pytest.approx(1.0 + 2 * math.exp(-1.5))


def _far_decode_case(seed, W=6, ns=1, hd=16, nh=2, m=4):
    g = np.random.default_rng(seed)
    cap = W
    pos0 = 3 * W + 2
    meta = np.array([[W, pos0 % W, 0, W]], dtype=np.int64)
    ring_k, ring_v = g.normal(size=(1, 1, cap, hd)), g.normal(size=(1, 1, cap, hd))
    inp = {"meta": meta, "ring_k": ring_k, "ring_v": ring_v,
           "sink_k": g.normal(size=(1, 1, ns, hd)), "sink_v": g.normal(size=(1, 1, ns, hd)),
           "gate_scale": g.normal(size=(nh, hd))}
    scale = hd ** -0.5
    # landmark keys = the first m keys the coming steps evict (slots head0, head0 + 1, ...)
    head0 = int(meta[0, 1])
    kt = np.stack([ring_k[0, 0, (head0 + j) % W] for j in range(m)])[None, None]
    qt = 2.5 * g.normal(size=(1, nh, m, hd))
    mu = np.zeros((1, nh, m, m))
    for h in range(nh):
        Bm = np.exp(scale * qt[0, h] @ kt[0, 0].T)          # Bm[b][j] = exp(s <q~_b, k_j>)
        assert np.linalg.cond(Bm) < 1e8
        mu[0, h] = np.linalg.inv(Bm)
    far = {"m": m, "rect": 0, "k_tilde": kt, "q_tilde": qt, "mu": mu,
           "mz": np.concatenate([np.full((1, nh, m), -np.inf), np.zeros((1, nh, m))], axis=2),
           "t_hat": np.zeros((1, nh, m, hd))}
    return g, inp, far, scale


def test_far_field_is_exact_when_the_landmarks_are_the_evicted_keys():
    """Nystrom reconstruction is exact on its own landmarks: with k~ = the keys
    the steps evict and mu = [exp(s <q~_b, k_j>)]^-1, every decode step equals
    full softmax attention over the sinks, every key evicted so far and the
    window (the far field then loses nothing)."""
    hd, nh, hpg = 16, 2, 2
    g, inp, far, scale = _far_decode_case(7, hd=hd, nh=nh)
    W = 6
    evicted_k, evicted_v = [], []
    for step in range(far["m"]):
        inp["q"] = g.normal(size=(1, 1, nh, hd))
        inp["k_chunk"] = g.normal(size=(1, 1, 1, hd))
        inp["v_chunk"] = g.normal(size=(1, 1, 1, hd))
        inp["gate"] = g.normal(size=(1, 1, nh, hd))
        got = oracle.attend_far(inp, far, scale, hpg)
        meta_b = inp["meta"][0]
        slot = int(meta_b[1]) % W
        evicted_k.append(inp["ring_k"][0, 0, slot].copy())
        evicted_v.append(inp["ring_v"][0, 0, slot].copy())
        for h in range(nh):
            keys = oracle.row_key_list(meta_b, 0, 1, W)
            K = [inp["sink_k"][0, 0, 0]] + evicted_k
            V = [inp["sink_v"][0, 0, 0]] + evicted_v
            for kind, idx in keys[1:]:
                src = (inp["ring_k"], inp["ring_v"]) if kind == "ring" else None
                K.append(src[0][0, 0, idx] if src else inp["k_chunk"][0, idx, 0])
                V.append(src[1][0, 0, idx] if src else inp["v_chunk"][0, idx, 0])
            s = scale * (np.asarray(K) @ inp["q"][0, 0, h])
            p = np.exp(s - s.max())
            ref = (p @ np.asarray(V)) / p.sum() * oracle.sigmoid_gate(inp["gate"][0, 0, h], inp["gate_scale"][h])
            np.testing.assert_allclose(got[0, 0, h], ref, rtol=1e-7, atol=1e-9)
        far["mz"], far["t_hat"] = oracle.far_commit(inp, far, scale, hpg)
        inp["ring_k"], inp["ring_v"], inp["meta"] = oracle.commit(inp["meta"], inp["ring_k"], inp["ring_v"],
                                                                 inp["k_chunk"], inp["v_chunk"])
        assert int(inp["meta"][0, 2]) == step + 1          # far_len counts the evictions


def test_far_single_landmark_closed_form():
    """m = 1: the far part is mu exp(s <q, k~>) * sum_j exp(s <q~, k_j>) (v_j, 1)
    over the evicted keys, next to the near terms."""
    hd, nh, hpg = 8, 1, 1
    g, inp, far, scale = _far_decode_case(11, hd=hd, nh=nh, m=1)
    far["mu"] = np.full((1, 1, 1, 1), 0.37)
    inp["q"] = g.normal(size=(1, 1, nh, hd))
    inp["k_chunk"], inp["v_chunk"] = g.normal(size=(1, 1, 1, hd)), g.normal(size=(1, 1, 1, hd))
    inp["gate"] = np.zeros((1, 1, nh, hd))                  # sigmoid(0) = 1/2
    got = oracle.attend_far(inp, far, scale, hpg)[0, 0, 0]
    W = 6
    meta_b = inp["meta"][0]
    slot = int(meta_b[1]) % W
    kev, vev = inp["ring_k"][0, 0, slot], inp["ring_v"][0, 0, slot]
    q = inp["q"][0, 0, 0]
    wfar = 0.37 * math.exp(scale * q @ far["k_tilde"][0, 0, 0]) * math.exp(scale * far["q_tilde"][0, 0, 0] @ kev)
    num, den = wfar * vev, wfar
    for kind, idx in oracle.row_key_list(meta_b, 0, 1, W):
        if kind == "sink":
            kk, vv = inp["sink_k"][0, 0, idx], inp["sink_v"][0, 0, idx]
        elif kind == "ring":
            kk, vv = inp["ring_k"][0, 0, idx], inp["ring_v"][0, 0, idx]
        else:
            kk, vv = inp["k_chunk"][0, idx, 0], inp["v_chunk"][0, idx, 0]
        e = math.exp(scale * q @ kk)
        num, den = num + e * vv, den + e
    np.testing.assert_allclose(got, 0.5 * num / den, rtol=1e-10)


def test_far_part_with_negative_mass_is_dropped_and_empty_field_adds_nothing():
    hd, nh, hpg = 8, 2, 2
    g, inp, far, scale = _far_decode_case(13, hd=hd, nh=nh)
    inp["q"] = g.normal(size=(1, 1, nh, hd))
    inp["k_chunk"], inp["v_chunk"] = g.normal(size=(1, 1, 1, hd)), g.normal(size=(1, 1, 1, hd))
    inp["gate"] = g.normal(size=(1, 1, nh, hd))
    near = oracle.attend(inp, scale, hpg)
    far["mu"] = -np.abs(far["mu"]) - 0.1                    # every gain negative: far_den < 0
    np.testing.assert_allclose(oracle.attend_far(inp, far, scale, hpg), near, rtol=1e-12)
    inp["meta"] = np.array([[4, 0, 0, 6]])                  # not full: no eviction, far_len 0
    near = oracle.attend(inp, scale, hpg)
    far["mu"] = np.abs(far["mu"])
    np.testing.assert_allclose(oracle.attend_far(inp, far, scale, hpg), near, rtol=1e-12)


def test_far_rect_clips_negative_landmark_weights():
    """rect (dory_ofar): w_b = max(w_b, 0). Two landmarks, mu = diag(2, -1):
    w = (2 e^{fs_0 - f}, -e^{fs_1 - f}); clipped, only landmark 0 feeds the far
    part, so the result equals the same state with landmark 1's mu column 0."""
    hd, nh, hpg = 8, 1, 1
    g, inp, far, scale = _far_decode_case(17, hd=hd, nh=nh, m=2)
    inp["q"] = g.normal(size=(1, 1, nh, hd))
    inp["k_chunk"], inp["v_chunk"] = g.normal(size=(1, 1, 1, hd)), g.normal(size=(1, 1, 1, hd))
    inp["gate"] = g.normal(size=(1, 1, nh, hd))
    far["mu"] = np.array([[[[2.0, 0.0], [0.0, -1.0]]]])
    clipped = dict(far, rect=1)
    zeroed = dict(far, mu=np.array([[[[2.0, 0.0], [0.0, 0.0]]]]))
    a = oracle.attend_far(inp, clipped, scale, hpg)
    b = oracle.attend_far(inp, zeroed, scale, hpg)
    np.testing.assert_allclose(a, b, rtol=1e-12)
    assert not np.allclose(oracle.attend_far(inp, far, scale, hpg), a)


@pytest.mark.parametrize("len0", [6, 3])        # full window; one that fills during the chunk
def test_far_chunk_equals_sequential_decode_steps(len0):
    """A t-row chunk with the far field (o1c_far_e / o1c_far: row i sees the
    evictions of rows 0..i) equals t single-row steps each committing ring,
    meta and far state (o1c_tok_*), row by row, and leaves the same state."""
    hd, nh, hpg, W, t = 8, 2, 2, 6, 5
    g, inp, far, scale = _far_decode_case(19, W=W, hd=hd, nh=nh, m=3)
    far["mu"] = np.abs(far["mu"]) + 0.1
    inp["meta"] = np.array([[len0, 2, 4 if len0 == W else 0, W]])
    if len0 < W:
        far["mz"][0, :, :3] = -np.inf
        far["mz"][0, :, 3:] = 0.0
    inp["q"] = g.normal(size=(1, t, nh, hd))
    inp["k_chunk"], inp["v_chunk"] = g.normal(size=(1, t, 1, hd)), g.normal(size=(1, t, 1, hd))
    inp["gate"] = g.normal(size=(1, t, nh, hd))
    chunk = oracle.attend_far(inp, far, scale, hpg)
    mz_c, th_c = oracle.far_commit(inp, far, scale, hpg)
    rk_c, rv_c, meta_c = oracle.commit(inp["meta"], inp["ring_k"], inp["ring_v"], inp["k_chunk"], inp["v_chunk"])
    st = dict(inp)
    fs = dict(far)
    for i in range(t):
        step = dict(st, q=inp["q"][:, i:i + 1], k_chunk=inp["k_chunk"][:, i:i + 1],
                    v_chunk=inp["v_chunk"][:, i:i + 1], gate=inp["gate"][:, i:i + 1])
        np.testing.assert_allclose(oracle.attend_far(step, fs, scale, hpg)[:, 0], chunk[:, i], rtol=1e-10)
        fs["mz"], fs["t_hat"] = oracle.far_commit(step, fs, scale, hpg)
        st["ring_k"], st["ring_v"], st["meta"] = oracle.commit(step["meta"], step["ring_k"], step["ring_v"],
                                                               step["k_chunk"], step["v_chunk"])
    np.testing.assert_allclose(fs["mz"], mz_c, rtol=1e-12)
    np.testing.assert_allclose(fs["t_hat"], th_c, rtol=1e-12)
    np.testing.assert_array_equal(st["meta"], meta_c)
    np.testing.assert_array_equal(st["ring_k"], rk_c)


@pytest.mark.parametrize("t,len0", [(64, 80), (48, 40)])  # OB_K = 64 rows: full window; one that fills mid-chunk
def test_far_chunk_of_up_to_64_rows_equals_sequential_decode_steps(t, len0):
    """The chunk length the pages size their far scratch for ("o1c_msl.metal"
    OB_K = 64, o1c_far_e / o1c_far): a 64- or 48-row chunk with the far field
    equals as many single-row steps, each committing ring, meta and far state,
    row by row, and leaves the same state."""
    hd, nh, hpg, W, m = 8, 2, 2, 80, 3
    g, inp, far, scale = _far_decode_case(23, W=W, hd=hd, nh=nh, m=m)
    far["mu"] = np.abs(far["mu"]) + 0.1
    inp["meta"] = np.array([[len0, 5, 9 if len0 == W else 0, W]])
    if len0 < W:
        far["mz"][0, :, :m] = -np.inf
        far["mz"][0, :, m:] = 0.0
    inp["q"] = g.normal(size=(1, t, nh, hd))
    inp["k_chunk"], inp["v_chunk"] = g.normal(size=(1, t, 1, hd)), g.normal(size=(1, t, 1, hd))
    inp["gate"] = g.normal(size=(1, t, nh, hd))
    assert len(oracle.far_evictions(inp["meta"][0], t, W)) == t - (W - len0)
    chunk = oracle.attend_far(inp, far, scale, hpg)
    mz_c, th_c = oracle.far_commit(inp, far, scale, hpg)
    rk_c, rv_c, meta_c = oracle.commit(inp["meta"], inp["ring_k"], inp["ring_v"], inp["k_chunk"], inp["v_chunk"])
    st = dict(inp)
    fs = dict(far)
    for i in range(t):
        step = dict(st, q=inp["q"][:, i:i + 1], k_chunk=inp["k_chunk"][:, i:i + 1],
                    v_chunk=inp["v_chunk"][:, i:i + 1], gate=inp["gate"][:, i:i + 1])
        np.testing.assert_allclose(oracle.attend_far(step, fs, scale, hpg)[:, 0], chunk[:, i], rtol=1e-10)
        fs["mz"], fs["t_hat"] = oracle.far_commit(step, fs, scale, hpg)
        st["ring_k"], st["ring_v"], st["meta"] = oracle.commit(step["meta"], step["ring_k"], step["ring_v"],
                                                               step["k_chunk"], step["v_chunk"])
    np.testing.assert_allclose(fs["mz"], mz_c, rtol=1e-12)
    np.testing.assert_allclose(fs["t_hat"], th_c, rtol=1e-12)
    np.testing.assert_array_equal(st["meta"], meta_c)
    np.testing.assert_array_equal(st["ring_k"], rk_c)


def test_far_chunk_of_64_rows_is_exact_with_landmarks_at_its_evictions():
    """Nystrom exactness over a whole 64-row chunk: a ring of 46 keys in a
    window of 80 fills at row 34, so rows 34..63 evict the 30 oldest keys. With
    those keys as the 30 landmarks and mu = [exp(s <q~_b, k_j>)]^-1, every row
    equals full softmax attention over the sinks, every ring key and the
    chunk's rows up to itself: the far field returns exactly what the window
    dropped."""
    hd, nh, hpg, W, t, len0, head0, m = 32, 2, 2, 80, 64, 46, 10, 30
    g = np.random.default_rng(29)
    ns = 2
    ring_k, ring_v = g.normal(size=(1, 1, W, hd)), g.normal(size=(1, 1, W, hd))
    inp = {"meta": np.array([[len0, head0, 0, W]], dtype=np.int64), "ring_k": ring_k, "ring_v": ring_v,
           "sink_k": g.normal(size=(1, 1, ns, hd)), "sink_v": g.normal(size=(1, 1, ns, hd)),
           "gate_scale": g.normal(size=(nh, hd)), "q": g.normal(size=(1, t, nh, hd)),
           "k_chunk": g.normal(size=(1, t, 1, hd)), "v_chunk": g.normal(size=(1, t, 1, hd)),
           "gate": g.normal(size=(1, t, nh, hd))}
    scale = hd ** -0.5
    ev = oracle.far_evictions(inp["meta"][0], t, W)
    assert [j for j, _ in ev] == list(range(34, 64))
    assert [slot for _, slot in ev] == [(head0 + x) % W for x in range(m)]
    kt = np.stack([ring_k[0, 0, slot] for _, slot in ev])[None, None]
    qt = 2.5 * g.normal(size=(1, nh, m, hd))
    mu = np.zeros((1, nh, m, m))
    for h in range(nh):
        Bm = np.exp(scale * qt[0, h] @ kt[0, 0].T)
        assert np.linalg.cond(Bm) < 1e8
        mu[0, h] = np.linalg.inv(Bm)
    far = {"m": m, "rect": 0, "k_tilde": kt, "q_tilde": qt, "mu": mu,
           "mz": np.concatenate([np.full((1, nh, m), -np.inf), np.zeros((1, nh, m))], axis=2),
           "t_hat": np.zeros((1, nh, m, hd))}
    got = oracle.attend_far(inp, far, scale, hpg)
    ring_keys = [(head0 + x) % W for x in range(len0)]
    for i in range(t):
        K = np.concatenate([inp["sink_k"][0, 0], ring_k[0, 0, ring_keys], inp["k_chunk"][0, :i + 1, 0]])
        V = np.concatenate([inp["sink_v"][0, 0], ring_v[0, 0, ring_keys], inp["v_chunk"][0, :i + 1, 0]])
        for h in range(nh):
            sc = scale * (K @ inp["q"][0, i, h])
            p = np.exp(sc - sc.max())
            ref = (p @ V) / p.sum() * oracle.sigmoid_gate(inp["gate"][0, i, h], inp["gate_scale"][h])
            np.testing.assert_allclose(got[0, i, h], ref, rtol=1e-7, atol=1e-9)


# ---------------------------------------------------------------------------
# full-sequence attention (egemma2_msl.metal eg_flash64 / eg_flash_staged)
# ---------------------------------------------------------------------------
def _flash_case(seed, segs, hd=8, nq=4, group=2, pad=4):
    """Packed rows [q heads | k heads | v heads | pad]: offsets not at 0 and a
    row stride larger than the three blocks, so a slip in either shows."""
    g = np.random.default_rng(seed)
    nk = nq // group
    q_off, k_off = pad, pad + nq * hd
    v_off = k_off + nk * hd
    ld = v_off + nk * hd + pad
    T = max(s0 + n for s0, n in segs) + 2
    return g.normal(size=(T, ld)), dict(hd=hd, nq=nq, group=group, q_off=q_off, k_off=k_off, v_off=v_off)


def test_flash_matches_masked_dense_attention_over_the_whole_buffer():
    """One dense score matrix over all T rows per head with a block-diagonal
    segment mask (torch scaled_dot_product_attention in float64), against the
    oracle's per-segment, per-row loops."""
    segs = [(0, 5), (5, 1), (7, 9)]                 # row 6 belongs to no segment
    qkv, c = _flash_case(1, segs)
    hd, nq, group, scale = c["hd"], c["nq"], c["group"], 0.7
    got = oracle.flash_attention(qkv, segs, scale=scale, **c)
    T = qkv.shape[0]
    seg_id = np.full(T, -1)
    for k, (s0, n) in enumerate(segs):
        seg_id[s0:s0 + n] = k
    mask = (seg_id[:, None] == seg_id[None, :]) & (seg_id[:, None] >= 0)
    mask[seg_id < 0, :] = True                        # rows outside segments: any finite value
    for h in range(nq):
        g = h // group
        q = torch.tensor(qkv[:, c["q_off"] + h * hd:c["q_off"] + (h + 1) * hd])
        k = torch.tensor(qkv[:, c["k_off"] + g * hd:c["k_off"] + (g + 1) * hd])
        v = torch.tensor(qkv[:, c["v_off"] + g * hd:c["v_off"] + (g + 1) * hd])
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, None], k[None, None], v[None, None], attn_mask=torch.tensor(mask)[None, None],
            scale=scale)[0, 0].numpy()
        for s0, n in segs:
            np.testing.assert_allclose(got[s0:s0 + n, h * hd:(h + 1) * hd], ref[s0:s0 + n], rtol=1e-12, atol=1e-13)
    assert not got[6].any()


def test_flash_one_key_segment_returns_its_value_row():
    segs = [(2, 1)]
    qkv, c = _flash_case(2, segs)
    got = oracle.flash_attention(qkv, segs, scale=3.0, **c)
    for h in range(c["nq"]):
        g = h // c["group"]
        np.testing.assert_array_equal(got[2, h * c["hd"]:(h + 1) * c["hd"]],
                                      qkv[2, c["v_off"] + g * c["hd"]:c["v_off"] + (g + 1) * c["hd"]])


def test_flash_zero_query_gives_the_mean_of_the_segment_values():
    segs = [(0, 7)]
    qkv, c = _flash_case(3, segs)
    qkv[:, c["q_off"]:c["q_off"] + c["nq"] * c["hd"]] = 0.0
    got = oracle.flash_attention(qkv, segs, scale=1.0, **c)
    for h in range(c["nq"]):
        g = h // c["group"]
        mean = qkv[0:7, c["v_off"] + g * c["hd"]:c["v_off"] + (g + 1) * c["hd"]].mean(axis=0)
        np.testing.assert_allclose(got[0:7, h * c["hd"]:(h + 1) * c["hd"]], np.tile(mean, (7, 1)), rtol=1e-13)


def test_flash_two_key_closed_form():
    """Two keys: o = (e^{s1} v1 + e^{s2} v2) / (e^{s1} + e^{s2}), s_k = scale <q, k_k>,
    written out by hand for one head with hd = 2 and group = 1."""
    qkv = np.array([[1.0, 2.0, 0.5, -1.0, 3.0, 4.0],
                    [-2.0, 0.0, 2.0, 1.0, -5.0, 6.0]])    # per row: q (2) | k (2) | v (2)
    scale = 0.25
    got = oracle.flash_attention(qkv, [(0, 2)], hd=2, nq=1, group=1, q_off=0, k_off=2, v_off=4, scale=scale)
    for r in range(2):
        q = qkv[r, 0:2]
        s1 = scale * (q[0] * 0.5 + q[1] * -1.0)
        s2 = scale * (q[0] * 2.0 + q[1] * 1.0)
        e1, e2 = math.exp(s1), math.exp(s2)
        want = [(e1 * 3.0 + e2 * -5.0) / (e1 + e2), (e1 * 4.0 + e2 * 6.0) / (e1 + e2)]
        np.testing.assert_allclose(got[r], want, rtol=1e-14)


def test_flash_row_permutation_permutes_the_outputs():
    segs = [(1, 8)]
    qkv, c = _flash_case(4, segs)
    got = oracle.flash_attention(qkv, segs, scale=0.9, **c)
    perm = np.random.default_rng(5).permutation(8)
    qkv2 = qkv.copy()
    qkv2[1:9] = qkv[1:9][perm]
    got2 = oracle.flash_attention(qkv2, segs, scale=0.9, **c)
    np.testing.assert_allclose(got2[1:9], got[1:9][perm], rtol=1e-12, atol=1e-14)


def test_flash_segments_are_independent_and_heads_share_kv_by_group():
    segs = [(0, 4), (4, 5)]
    qkv, c = _flash_case(6, segs)
    got = oracle.flash_attention(qkv, segs, scale=1.1, **c)
    qkv2 = qkv.copy()
    qkv2[4:9] = np.random.default_rng(7).normal(size=(5, qkv.shape[1]))
    got2 = oracle.flash_attention(qkv2, segs, scale=1.1, **c)
    np.testing.assert_array_equal(got2[0:4], got[0:4])
    # group = 2: q heads 0 and 1 read K/V head 0; swapping the K/V of head 1
    # changes heads 2 and 3 only
    qkv3 = qkv.copy()
    hd, k1 = c["hd"], c["k_off"] + c["hd"]
    qkv3[:, k1:k1 + hd] = np.random.default_rng(8).normal(size=(qkv.shape[0], hd))
    got3 = oracle.flash_attention(qkv3, segs, scale=1.1, **c)
    np.testing.assert_array_equal(got3[:, 0:2 * hd], got[:, 0:2 * hd])
    assert np.abs(got3[0:9, 2 * hd:] - got[0:9, 2 * hd:]).max() > 1e-3
