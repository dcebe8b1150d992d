"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the GPU.

Floating point: max_abs <= 2e-5 and max_abs / max|oracle| <= 1e-4 per tensor.
Ring slots, window bounds and meta: exact.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
import sliding_window_gqa_prep_gb300 as swa
from swa_harness import (assert_close, check_commit_placement, check_commit_placement_full,
                         far_to_dev, far_to_np, oracle_rows,
                         gpu_full_path, oracle_inputs, to_dev)

pytestmark = pytest.mark.gpu

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a GPU")
    yield


# ---------------------------------------------------------------------------
# rope table and prep
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("hd", [64, 128, 256])
def test_rope_table_matches_oracle_to_one_ulp(hd):
    pos0 = np.array([0, 1, 99, 4095, 20000, 131071, 262143], dtype=np.int64)
    t = 3
    gpu = swa.rope_table(torch.tensor(pos0, dtype=torch.int32, device="cuda"), t, hd).cpu().numpy()
    ref = oracle.rope_table(pos0, t, hd)
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(gpu.astype(np.float64) - ref) <= ulp + 1e-30)


PREP_CASES = [
    dict(B=3, t=1, nh=8, nk=2, hd=64, window=32, cap=32, pos_mode="full", pos_lo=32, pos_hi=500),
    dict(B=2, t=5, nh=16, nk=4, hd=128, window=64, cap=64, pos_mode="full", pos_lo=64, pos_hi=9000),
    dict(B=2, t=1, nh=8, nk=2, hd=256, window=16, cap=16, pos_mode="full", pos_lo=16, pos_hi=130000),
    dict(B=1, t=7, nh=6, nk=3, hd=64, window=16, cap=16, pos_mode="prompt", pos_lo=0, pos_hi=40),
]


@pytest.mark.parametrize("kw", PREP_CASES)
def test_prep_matches_oracle_and_writes_ring_slots_exactly(kw):
    w = workloads.custom(seed=11, **kw)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=False)
    rope = oracle.rope_table(inp["pos0"].numpy(), w.t, w.hd, w.theta)
    q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                          inp["q_scale"].numpy(), w.eps)
    assert_close(res["q"], q, "q_hat")
    assert_close(res["k"], k, "k_hat")
    np.testing.assert_array_equal(res["v"], inp["yv"].numpy())
    if w.t == 1:
        # prep's ring write: slot (pos0 + j) % cap holds the GPU's k row bit for bit,
        # every other slot is untouched
        ring = res["ring_after_prep_k"]
        for b in range(w.B):
            slot = oracle.prep_ring_slot(int(inp["pos0"][b]), 0, w.cap)
            for s in range(w.cap):
                want = res["k"][b, 0] if s == slot else inp["ring_k"].numpy()[b, :, s]
                np.testing.assert_array_equal(ring[b, :, s], want)


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_prep_with_in_kernel_angles_equals_table_prep_bit_for_bit(hd):
    w = workloads.custom(B=3, t=4, nh=8, nk=2, hd=hd, window=64, cap=64, pos_mode="full",
                         pos_lo=64, pos_hi=131000, seed=19)
    d = to_dev(workloads.make_inputs(w))
    rope = swa.rope_table(d["pos0"], w.t, w.hd, w.theta)
    q1, k1, _ = swa.prep(d["yq"], d["yk"], d["yv"], rope, d["q_scale"], w.eps)
    q2, k2, _ = swa.prep(d["yq"], d["yk"], d["yv"], None, d["q_scale"], w.eps, pos0=d["pos0"],
                         theta=w.theta)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(k1, k2)


# ---------------------------------------------------------------------------
# attend: full path (generator -> rope -> prep -> attend -> commit) vs oracle
# ---------------------------------------------------------------------------
ATTEND_CASES = [
    # decode, wrapped ring, several tiles + ragged tail, sinks
    dict(B=3, t=1, nh=8, nk=2, hd=128, window=200, cap=200, ns=3, pos_mode="full", pos_lo=200, pos_hi=5000),
    # tiny decode shape
    dict(B=1, t=1, nh=8, nk=2, hd=64, window=32, cap=32, ns=0, pos_mode="fixed", pos_lo=100),
    # long head dim, one KV head
    dict(B=2, t=1, nh=4, nk=1, hd=256, window=300, cap=300, ns=8, pos_mode="full", pos_lo=300, pos_hi=99999),
    # verify: partially filled rings, causal chunk
    dict(B=4, t=8, nh=16, nk=4, hd=128, window=150, cap=150, ns=4, pos_mode="partial", pos_lo=1, pos_hi=150),
    # prompt chunk longer than the window, empty ring in sequence 0
    dict(B=2, t=40, nh=8, nk=2, hd=64, window=24, cap=24, ns=2, pos_mode="prompt", pos_lo=0, pos_hi=60),
    # one key window
    dict(B=2, t=3, nh=4, nk=1, hd=64, window=1, cap=1, ns=0, pos_mode="full", pos_lo=1, pos_hi=50),
    # ragged query block (t * hpg not a power of two), hpg = 6
    dict(B=2, t=3, nh=12, nk=2, hd=128, window=70, cap=70, ns=1, pos_mode="full", pos_lo=70, pos_hi=999),
    # hpg = 1 and hpg = 32
    dict(B=2, t=2, nh=2, nk=2, hd=64, window=40, cap=40, ns=0, pos_mode="partial", pos_lo=1, pos_hi=40),
    dict(B=1, t=1, nh=32, nk=1, hd=128, window=90, cap=90, ns=2, pos_mode="full", pos_lo=90, pos_hi=400),
    # hd 256, verify-sized block
    dict(B=2, t=8, nh=8, nk=2, hd=256, window=64, cap=64, ns=4, pos_mode="full", pos_lo=64, pos_hi=700),
    # tensor-core prompt path: hpg 8 (8 rows per block, ragged last block), partial rings
    dict(B=3, t=37, nh=16, nk=2, hd=128, window=100, cap=100, ns=3, pos_mode="partial", pos_lo=1, pos_hi=100),
    # tensor-core prompt path: hpg 6 (10 rows = 60 of 64 query slots), wrapped rings, window < t
    dict(B=2, t=33, nh=12, nk=2, hd=64, window=20, cap=20, ns=1, pos_mode="full", pos_lo=20, pos_hi=900),
    # tensor-core prompt path: empty ring, hpg 4, several key tiles
    dict(B=2, t=70, nh=8, nk=2, hd=128, window=64, cap=64, ns=0, pos_mode="prompt", pos_lo=0, pos_hi=200),
    # every remaining attention-kernel instance: decode with 8 query vectors
    # (hd 64 / 128 / 256), verify with 16 and 32 (hd 64) and 16 (hd 256)
    dict(B=2, t=2, nh=8, nk=2, hd=64, window=80, cap=80, ns=2, pos_mode="full", pos_lo=80, pos_hi=900),
    dict(B=2, t=2, nh=8, nk=2, hd=128, window=70, cap=70, ns=1, pos_mode="partial", pos_lo=1, pos_hi=70),
    dict(B=2, t=2, nh=8, nk=2, hd=256, window=50, cap=50, ns=3, pos_mode="full", pos_lo=50, pos_hi=700),
    dict(B=3, t=8, nh=8, nk=2, hd=64, window=120, cap=120, ns=4, pos_mode="partial", pos_lo=1, pos_hi=120),
    dict(B=2, t=4, nh=8, nk=2, hd=64, window=90, cap=90, ns=0, pos_mode="full", pos_lo=90, pos_hi=999),
    dict(B=2, t=4, nh=8, nk=2, hd=256, window=75, cap=75, ns=2, pos_mode="full", pos_lo=75, pos_hi=800),
    # mid-size chunks (64 <= rows x heads < 128): the 64-vector mma.sync path
    dict(B=2, t=20, nh=8, nk=2, hd=128, window=90, cap=90, ns=2, pos_mode="full", pos_lo=90, pos_hi=900),
    dict(B=2, t=12, nh=16, nk=2, hd=64, window=30, cap=30, ns=1, pos_mode="partial", pos_lo=1, pos_hi=30),
    # verify blocks of 32 query vectors at hd 128 with other head groupings:
    # hpg 2 (16 rows), a window of three 128-key spans with a ragged tail, wrapped rings
    dict(B=2, t=16, nh=4, nk=2, hd=128, window=300, cap=300, ns=4, pos_mode="full", pos_lo=300, pos_hi=5000),
    # hpg 8 (4 rows), a window of 129 keys
    dict(B=2, t=4, nh=16, nk=2, hd=128, window=129, cap=129, ns=1, pos_mode="partial", pos_lo=1, pos_hi=129),
    # hpg 16 (2 rows), one KV head, no sinks
    dict(B=1, t=2, nh=16, nk=1, hd=128, window=512, cap=512, ns=0, pos_mode="full", pos_lo=512, pos_hi=3000),
    # hpg 4, two row blocks (8 + 3 rows), a window shorter than the block
    dict(B=2, t=11, nh=8, nk=2, hd=128, window=6, cap=6, ns=2, pos_mode="full", pos_lo=6, pos_hi=400),
    # hpg 6 (5 rows = 30 of 32 query slots), prompt-style rings (some empty)
    dict(B=3, t=5, nh=12, nk=2, hd=128, window=260, cap=260, ns=3, pos_mode="prompt", pos_lo=0, pos_hi=300),
]


@pytest.mark.parametrize("kw", ATTEND_CASES)
@pytest.mark.parametrize("sharp", [False, True])
def test_full_path_matches_oracle(kw, sharp):
    w = workloads.custom(seed=5, scale=4.0 if sharp else None, **kw)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=True)
    assert res["err"] == 0
    a = oracle_inputs(w, inp)
    ref = oracle.attend(a, w.score_scale, w.hpg)
    assert_close(res["out"], ref, "out")
    check_commit_placement(w, inp, res)


@pytest.mark.parametrize("kw", [c for c in ATTEND_CASES if c["hd"] <= 128 and c["t"] * c["nh"] // c["nk"] >= 128])
def test_tensor_core_prompt_with_the_minimum_workspace(kw):
    """The tcgen05 prompt kernel staging and splitting K/V itself (a workspace of
    swa_attend_workspace_min bytes, no split-once operand blocks)."""
    w = workloads.custom(seed=5, **kw)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=True, min_workspace=True)
    assert res["err"] == 0
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    assert_close(res["out"], ref, "out")
    check_commit_placement(w, inp, res)


@pytest.mark.parametrize("meta_alias", [False, True])
def test_ordered_verify_blocks_finish_in_the_attention_kernel(meta_alias):
    """Far more verify blocks (16 query vectors, one row block per (sequence, KV
    head)) than resident CTAs: one split each, taken longest first from an order a
    one-CTA kernel sorts; the attention kernel itself normalises, gates, writes the
    output and commits (two launches). With meta_out aliasing meta it writes records
    and the merge commits (three launches). Every output row against the oracle;
    ring and meta exact."""
    w = workloads.custom(B=600, t=4, nh=8, nk=2, hd=128, window=64, cap=64, ns=2, pos_mode="partial",
                         pos_lo=1, pos_hi=64, seed=47)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=True, meta_alias=meta_alias)
    assert res["err"] == 0
    assert res["attend_launches"] == (3 if meta_alias else 2)
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    assert_close(res["out"], ref, "out")
    check_commit_placement(w, inp, res)


@pytest.mark.parametrize("hd,t,B", [(64, 8, 320), (256, 4, 160), (256, 8, 160)])
def test_ordered_verify_blocks_at_other_head_dims(hd, t, B):
    """The ordered blocks finished in the attention kernel at hd 64 (32 query
    vectors) and hd 256 (16 and 32; one CTA per SM, so fewer blocks suffice):
    every output row against the oracle, ring and meta exact."""
    w = workloads.custom(B=B, t=t, nh=8, nk=2, hd=hd, window=48, cap=48, ns=3, pos_mode="partial",
                         pos_lo=1, pos_hi=48, seed=60 + hd + t)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=True)
    assert res["err"] == 0 and res["attend_launches"] == 2
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    assert_close(res["out"], ref, "out")
    check_commit_placement(w, inp, res)


def test_ordered_verify_blocks_without_commit_leave_ring_and_meta_alone():
    w = workloads.custom(B=600, t=4, nh=8, nk=2, hd=128, window=64, cap=64, ns=2, pos_mode="full",
                         pos_lo=64, pos_hi=900, seed=49)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=False)
    assert res["err"] == 0 and res["attend_launches"] == 2
    assert_close(res["out"], oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg), "out")
    np.testing.assert_array_equal(res["ring_k"], inp["ring_k"].numpy())
    np.testing.assert_array_equal(res["ring_v"], inp["ring_v"].numpy())


def test_ordered_verify_blocks_kernel_finish_equals_the_merge():
    """The block finished in the attention kernel and the same block written as a
    record and finished by the merge (meta_out aliasing meta) give the same bits:
    for one split the merge's weight is exp2(0) = 1."""
    w = workloads.custom(B=600, t=4, nh=8, nk=2, hd=128, window=64, cap=64, ns=2, pos_mode="partial",
                         pos_lo=1, pos_hi=64, seed=48)
    inp = workloads.make_inputs(w)
    a = gpu_full_path(w, inp, commit=True)
    b = gpu_full_path(w, inp, commit=True, meta_alias=True)
    assert a["attend_launches"] == 2 and b["attend_launches"] == 3
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["ring_k"], b["ring_k"])
    np.testing.assert_array_equal(a["ring_v"], b["ring_v"])
    np.testing.assert_array_equal(a["meta_out"], b["meta_out"])


def test_attend_only_matches_oracle_on_shared_q_k():
    """Attend fed the same (generator-drawn) q and chunk k/v on both sides."""
    w = workloads.custom(B=3, t=8, nh=16, nk=4, hd=128, window=100, cap=100, ns=4,
                         pos_mode="partial", pos_lo=1, pos_hi=100, seed=21, scale=1.0)
    inp = workloads.make_inputs(w)
    g = torch.Generator().manual_seed(99)
    q = torch.randn(w.B, w.t, w.nh, w.hd, generator=g)
    k = torch.randn(w.B, w.t, w.nk, w.hd, generator=g)
    v = torch.randn(w.B, w.t, w.nk, w.hd, generator=g)
    d = to_dev(inp)
    meta_out = torch.empty_like(d["meta"])
    out = swa.attend(d["meta"], q.cuda(), k.cuda(), v.cuda(), d["ring_k"], d["ring_v"],
                     d["sink_k"], d["sink_v"], d["gate"], d["gate_scale"], w.score_scale,
                     commit=False, meta_out=meta_out)
    ref = oracle.attend(oracle_inputs(w, inp, q.numpy(), k.numpy(), v.numpy()), w.score_scale, w.hpg)
    assert_close(out.cpu().numpy(), ref, "out")


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_split_count_invariance(splits):
    w = workloads.custom(B=2, t=4, nh=8, nk=2, hd=128, window=500, cap=500, ns=4,
                         pos_mode="full", pos_lo=500, pos_hi=9000, seed=3, scale=3.0)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=False, num_splits=splits)
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    assert_close(res["out"], ref, f"out (splits={splits})")


@pytest.mark.parametrize("splits", [1, 2, 5])
def test_split_count_invariance_verify_block(splits):
    """hd 128 blocks of 32 query vectors (the verify kernel) under several split counts."""
    w = workloads.custom(B=2, t=8, nh=8, nk=2, hd=128, window=700, cap=700, ns=4,
                         pos_mode="full", pos_lo=700, pos_hi=9000, seed=4, scale=3.0)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=False, num_splits=splits)
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    assert_close(res["out"], ref, f"out (splits={splits})")


def test_window_bounds_exact_via_one_hot_values():
    """Uniform scores (q = 0) and one-hot values that name each key: the set of
    keys each row attends is read back exactly and compared with the oracle's
    key list (sinks, ring slots, chunk rows)."""
    B, t, nh, nk, hd, cap, ns = 3, 8, 4, 1, 128, 100, 4
    w = workloads.custom(B=B, t=t, nh=nh, nk=nk, hd=hd, window=cap, cap=cap, ns=ns,
                         pos_mode="partial", pos_lo=1, pos_hi=cap, seed=8)
    inp = workloads.make_inputs(w)
    ring_v = torch.zeros(B, nk, cap, hd)
    for s in range(cap):
        ring_v[:, :, s, s] = 1.0
    sink_v = torch.zeros(B, nk, ns, hd)
    for s in range(ns):
        sink_v[:, :, s, cap + s] = 1.0
    v_chunk = torch.zeros(B, t, nk, hd)
    for j in range(t):
        v_chunk[:, j, :, cap + ns + j] = 1.0
    d = to_dev(inp)
    q = torch.zeros(B, t, nh, hd, device="cuda")
    k = torch.randn(B, t, nk, hd, device="cuda")
    gate = torch.zeros(B, t, nh, hd, device="cuda")          # sigmoid(0) = 1/2
    meta_out = torch.empty_like(d["meta"])
    out = swa.attend(d["meta"], q, k, v_chunk.cuda(), d["ring_k"], ring_v.cuda(), d["sink_k"],
                     sink_v.cuda(), gate, d["gate_scale"], w.score_scale, meta_out=meta_out)
    out = out.cpu().numpy() * 2.0
    meta = inp["meta"].numpy()
    for b in range(B):
        for i in range(t):
            keys = oracle.row_key_list(meta[b], i, ns, cap)
            want = set()
            for kind, idx in keys:
                want.add(idx if kind == "ring" else (cap + idx if kind == "sink" else cap + ns + idx))
            for h in range(nh):
                got = set(np.nonzero(out[b, i, h] > 0.5 / len(keys))[0].tolist())
                assert got == want, (b, i, h)
                np.testing.assert_allclose(out[b, i, h][sorted(want)], 1.0 / len(keys), rtol=1e-5)


def test_out_of_window_ring_slots_are_never_read():
    """NaN in every ring slot outside the pre-chunk window (and in the slots the
    chunk will overwrite): outputs stay finite, so no such slot is loaded."""
    w = workloads.custom(B=4, t=8, nh=8, nk=2, hd=128, window=64, cap=96, ns=2,
                         pos_mode="partial", pos_lo=1, pos_hi=64, seed=4)
    inp = workloads.make_inputs(w)
    meta = inp["meta"].numpy()
    for b in range(w.B):
        len0, head0 = int(meta[b][0]), int(meta[b][1])
        live = {(head0 + x) % 64 for x in range(len0)}
        for s in range(w.cap):
            if s not in live:
                inp["ring_k"][b, :, s] = float("nan")
                inp["ring_v"][b, :, s] = float("nan")
    res = gpu_full_path(w, inp, commit=False)
    assert np.all(np.isfinite(res["out"]))
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    assert_close(res["out"], ref, "out")


def test_window_smaller_than_cap_and_zero_window_field():
    w = workloads.custom(B=2, t=4, nh=8, nk=2, hd=64, window=40, cap=64, ns=1,
                         pos_mode="full", pos_lo=40, pos_hi=3000, seed=12)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=True)
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    assert_close(res["out"], ref, "out")
    check_commit_placement(w, inp, res)
    # window field 0 means cap
    w0 = workloads.custom(B=2, t=2, nh=4, nk=1, hd=64, window=48, cap=48, ns=0,
                          pos_mode="full", pos_lo=48, pos_hi=3000, seed=13)
    inp0 = workloads.make_inputs(w0)
    inp0["meta"][:, 3] = 0
    res0 = gpu_full_path(w0, inp0, commit=True)
    ref0 = oracle.attend(oracle_inputs(w0, inp0), w0.score_scale, w0.hpg)
    assert_close(res0["out"], ref0, "out")
    check_commit_placement(w0, inp0, res0)


def test_commit_with_meta_out_aliasing_meta():
    w = workloads.custom(B=3, t=5, nh=8, nk=2, hd=128, window=32, cap=32, ns=0,
                         pos_mode="full", pos_lo=32, pos_hi=900, seed=14)
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=True, meta_alias=True)
    check_commit_placement(w, inp, res)


def test_chunk_equals_sequential_decode_steps_on_gpu():
    """A t-row chunk with commit == t single-row steps, each committing and
    advancing the meta: outputs within tolerance, final ring and meta exact."""
    w = workloads.custom(B=2, t=6, nh=8, nk=2, hd=128, window=48, cap=48, ns=2,
                         pos_mode="full", pos_lo=48, pos_hi=2000, seed=15)
    inp = workloads.make_inputs(w)
    chunk = gpu_full_path(w, inp, commit=True)
    d = to_dev(inp)
    rope = swa.rope_table(d["pos0"], w.t, w.hd, w.theta)
    q, k, v = swa.prep(d["yq"], d["yk"], d["yv"], rope, d["q_scale"], w.eps)
    ring_k, ring_v = d["ring_k"].clone(), d["ring_v"].clone()
    meta = d["meta"].clone()
    outs = []
    for i in range(w.t):
        meta_next = torch.empty_like(meta)
        o = swa.attend(meta, q[:, i:i + 1].contiguous(), k[:, i:i + 1].contiguous(),
                       v[:, i:i + 1].contiguous(), ring_k, ring_v, d["sink_k"], d["sink_v"],
                       d["gate"][:, i:i + 1].contiguous(), d["gate_scale"], w.score_scale,
                       commit=True, meta_out=meta_next)
        outs.append(o.clone())
        meta = meta_next
    seq_out = torch.cat(outs, dim=1).cpu().numpy()
    assert_close(seq_out, chunk["out"], "sequential vs chunk")
    np.testing.assert_array_equal(ring_k.cpu().numpy(), chunk["ring_k"])
    np.testing.assert_array_equal(ring_v.cpu().numpy(), chunk["ring_v"])
    np.testing.assert_array_equal(meta.cpu().numpy(), chunk["meta_out"])


def test_bad_meta_sets_error_word_without_fault():
    w = workloads.custom(B=2, t=1, nh=4, nk=1, hd=64, window=16, cap=16, ns=0,
                         pos_mode="full", pos_lo=16, pos_hi=100, seed=16)
    inp = workloads.make_inputs(w)
    inp["meta"][0, 0] = 50       # win_len > window
    inp["meta"][1, 3] = 1000     # window > cap
    res = gpu_full_path(w, inp, commit=False)
    assert res["err"] & swa.SWA_DERR_META
    assert np.all(np.isfinite(res["out"]))


def test_token_path_host_step_matches_device_step():
    w = workloads.custom(B=2, t=1, nh=8, nk=2, hd=128, window=64, cap=64, ns=2,
                         pos_mode="full", pos_lo=64, pos_hi=900, seed=17)
    inp = workloads.make_inputs(w)
    mk = lambda: swa.TokenPath(B=w.B, t=w.t, nh=w.nh, nk=w.nk, hd=w.hd, cap=w.cap, ns=w.ns,
                               q_scale=inp["q_scale"], gate_scale=inp["gate_scale"],
                               ring_k=inp["ring_k"], ring_v=inp["ring_v"], sink_k=inp["sink_k"],
                               sink_v=inp["sink_v"], meta=inp["meta"], pos0=inp["pos0"])
    host = mk().step(inp["yq"].pin_memory(), inp["yk"].pin_memory(), inp["yv"].pin_memory(),
                     inp["gate"].pin_memory(), out_host=torch.empty(w.B, w.t, w.nh, w.hd).pin_memory())
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    assert_close(host.numpy(), ref, "out")


def test_token_path_captured_graph_matches_oracle_twice():
    w = workloads.custom(B=3, t=1, nh=8, nk=2, hd=128, window=96, cap=96, ns=2,
                         pos_mode="full", pos_lo=96, pos_hi=5000, seed=23)
    inp = workloads.make_inputs(w)
    tp = swa.TokenPath(B=w.B, t=w.t, nh=w.nh, nk=w.nk, hd=w.hd, cap=w.cap, ns=w.ns,
                       q_scale=inp["q_scale"], gate_scale=inp["gate_scale"],
                       ring_k=inp["ring_k"], ring_v=inp["ring_v"], sink_k=inp["sink_k"],
                       sink_v=inp["sink_v"], meta=inp["meta"], pos0=inp["pos0"])
    tp.capture()
    ref = oracle.attend(oracle_inputs(w, inp), w.score_scale, w.hpg)
    for _ in range(2):
        for k in ("yq", "yk", "yv", "gate"):
            tp.h_in[k].copy_(inp[k])
        out = tp.replay()
        assert_close(out.numpy(), ref, "graph replay out")


def test_prompt_chunk_captured_graph_follows_each_steps_inputs():
    # a tensor-core chunk (64 rows x 4 query heads per KV head): the copies of yv and
    # the gate overlap the prep and the attention. Every window stays below W - t,
    # so one replay's commit never lands in the next one's window.
    w = workloads.custom(B=2, t=64, nh=8, nk=2, hd=128, window=200, cap=200, ns=3,
                         pos_mode="prompt", pos_lo=0, pos_hi=100, seed=29)
    inp = workloads.make_inputs(w)
    g = torch.Generator().manual_seed(30)
    other = dict(inp, **{k: torch.randn(inp[k].shape, generator=g) for k in ("yq", "yk", "yv", "gate")})
    tp = swa.TokenPath(B=w.B, t=w.t, nh=w.nh, nk=w.nk, hd=w.hd, cap=w.cap, ns=w.ns,
                       q_scale=inp["q_scale"], gate_scale=inp["gate_scale"],
                       ring_k=inp["ring_k"], ring_v=inp["ring_v"], sink_k=inp["sink_k"],
                       sink_v=inp["sink_v"], meta=inp["meta"], pos0=inp["pos0"])
    tp.capture()
    for cur in (inp, other, inp):
        for k in ("yq", "yk", "yv", "gate"):
            tp.h_in[k].copy_(cur[k])
        out = tp.replay()
        assert_close(out.numpy(), oracle.attend(oracle_inputs(w, cur), w.score_scale, w.hpg),
                     "graph replay out")


def test_ordered_verify_blocks_in_a_captured_graph_with_the_gate_arriving_late():
    """Ordered verify blocks inside the captured host-to-host step: the gate is still
    being copied in while the attention runs, so the blocks write records and the
    merge (which waits for the gate) finishes them. Two replays with different inputs;
    every window stays below W - t, so a replay's commit never lands in the next one's
    window."""
    w = workloads.custom(B=600, t=4, nh=8, nk=2, hd=128, window=64, cap=64, ns=2,
                         pos_mode="prompt", pos_lo=1, pos_hi=60, seed=33)   # sequence 0: empty ring
    inp = workloads.make_inputs(w)
    g = torch.Generator().manual_seed(34)
    other = dict(inp, **{k: torch.randn(inp[k].shape, generator=g) for k in ("yq", "yk", "yv", "gate")})
    tp = swa.TokenPath(B=w.B, t=w.t, nh=w.nh, nk=w.nk, hd=w.hd, cap=w.cap, ns=w.ns,
                       q_scale=inp["q_scale"], gate_scale=inp["gate_scale"],
                       ring_k=inp["ring_k"], ring_v=inp["ring_v"], sink_k=inp["sink_k"],
                       sink_v=inp["sink_v"], meta=inp["meta"], pos0=inp["pos0"])
    tp.capture()
    for cur in (inp, other):
        for k in ("yq", "yk", "yv", "gate"):
            tp.h_in[k].copy_(cur[k])
        out = tp.replay()
        assert_close(out.numpy(), oracle.attend(oracle_inputs(w, cur), w.score_scale, w.hpg),
                     "graph replay out")


def test_rollback_matches_oracle_bit_for_bit():
    g = torch.Generator().manual_seed(31)
    B, cap = 300, 64
    W = torch.randint(1, cap + 1, (B,), generator=g)
    W[::7] = 0                                            # window 0 means cap
    Wm = torch.where(W == 0, torch.full_like(W, cap), W)
    full = torch.rand(B, generator=g) < 0.5
    length = torch.where(full, Wm, (torch.rand(B, generator=g) * Wm.double()).long())
    head = (torch.rand(B, generator=g) * Wm.double()).long()
    far = torch.randint(0, 50, (B,), generator=g)
    meta = torch.stack([length, head, far, W], 1).to(torch.int32)
    n_back = torch.randint(0, 3 * cap, (B,), generator=g).to(torch.int32)
    n_back[:20] = length[:20].to(torch.int32)             # exactly to empty (or full: any)
    ref, bad = oracle.rollback(meta.numpy().astype(np.int64) % (1 << 32), n_back.numpy(), cap)
    d_meta, err = meta.cuda(), torch.zeros(1, dtype=torch.int32, device="cuda")
    swa.rollback(d_meta, n_back.cuda(), cap, err=err)
    got = d_meta.cpu().numpy().astype(np.int64) % (1 << 32)
    assert (got == ref % (1 << 32)).all()
    assert bad.any() and (int(err.item()) & 1) == 1


def test_rollback_after_verify_commit_equals_committing_the_accepted_prefix():
    # a window that does not fill: verify t rows with commit, reject t - a,
    # then the meta and the logical window's ring rows equal those of a
    # commit of only the first a rows
    w = workloads.custom(B=4, t=6, nh=8, nk=2, hd=64, window=64, cap=64, ns=0,
                         pos_mode="partial", pos_lo=1, pos_hi=40, seed=37)
    inp = workloads.make_inputs(w)
    acc = torch.tensor([0, 2, 5, 6], dtype=torch.int32)
    d = to_dev(inp)
    meta_out = torch.empty_like(d["meta"])
    q, k, v = swa.prep(d["yq"], d["yk"], d["yv"], None, d["q_scale"], w.eps, pos0=d["pos0"])
    swa.attend(d["meta"], q, k, v, d["ring_k"], d["ring_v"], None, None, d["gate"],
               d["gate_scale"], w.score_scale, commit=True, meta_out=meta_out)
    swa.rollback(meta_out, (w.t - acc).cuda(), w.cap)
    got_meta = meta_out.cpu().numpy()
    rk = d["ring_k"].cpu().numpy()
    for b in range(w.B):
        a = int(acc[b])
        len0, head0 = int(inp["meta"][b][0]), int(inp["meta"][b][1])
        W = int(inp["meta"][b][3]) or w.cap
        ref_meta = oracle.commit_meta(inp["meta"][b].numpy(), a, w.cap)
        assert got_meta[b].tolist() == ref_meta.tolist()
        written = {(head0 + len0 + j) % W for j in range(w.t)}
        L, H = int(ref_meta[0]), int(ref_meta[1])
        for x in range(L):
            slot = (H + x) % W
            if x < len0 and slot not in written:          # untouched key of the old window
                np.testing.assert_array_equal(rk[b, :, slot], inp["ring_k"][b, :, slot].numpy())
            elif len0 + w.t <= W and x >= len0:           # an accepted row (window never filled)
                np.testing.assert_array_equal(rk[b, :, slot], k[b, x - len0].cpu().numpy())


# ---------------------------------------------------------------------------
# far field of decode rows (o1c_tok_far, o1c_tok_merge, o1c_tok_commit)
# ---------------------------------------------------------------------------
def _far_case(seed, **kw):
    base = dict(B=4, t=1, nh=8, nk=2, hd=128, window=96, cap=96, ns=3, pos_mode="partial",
                pos_lo=40, pos_hi=96, far_m=16, seed=seed)
    base.update(kw)
    w = workloads.custom(**base)
    inp = workloads.make_inputs(w)
    # sequences 1.. are partial (no eviction); give one of them evictions behind it
    inp["meta"][1, 2] = 7
    inp["far"]["mz"][1, :, :w.far_m] = torch.randn(w.nh, w.far_m, generator=torch.Generator().manual_seed(seed))
    inp["far"]["mz"][1, :, w.far_m:] = 3.0
    return w, inp


def _check_far_state(w, inp, res, atol=2e-5):
    far_ref = far_to_np(inp["far"])
    mz_ref, th_ref = oracle.far_commit(oracle_inputs(w, inp, *_gpu_prepped(res)), far_ref, w.score_scale, w.hpg)
    got_mz, got_th = res["far"]["mz"].astype(np.float64), res["far"]["t_hat"].astype(np.float64)
    fin = np.isfinite(mz_ref)
    assert np.array_equal(fin, np.isfinite(got_mz))
    assert_close(got_mz[fin], mz_ref[fin], "far max / mass", max_abs=2e-4, max_rel=1e-5)
    assert_close(got_th, th_ref, "far numerators", max_abs=1e-3, max_rel=1e-5)


def _gpu_prepped(res):
    return res["q"], res["k"], res["v"]


@pytest.mark.parametrize("rect", [0, 1])
@pytest.mark.parametrize("splits", [0, 1, 64])
def test_far_decode_step_matches_oracle(rect, splits):
    w, inp = _far_case(41)
    _far_step_check(w, inp, rect, splits)


@pytest.mark.parametrize("t,hd,nh,nk,W", [(4, 128, 8, 2, 96), (8, 128, 16, 4, 96), (8, 256, 8, 2, 40),
                                          (32, 64, 8, 2, 64), (48, 128, 8, 2, 96), (64, 128, 16, 4, 80),
                                          (48, 256, 8, 2, 64), (64, 256, 4, 2, 70)])
def test_far_chunk_matches_oracle(t, hd, nh, nk, W):
    """Chunks with the far field (row i sees the evictions of rows 0..i), up to
    the pages' 64 rows (OB_K): verify-sized blocks on the CUDA-core kernel,
    chunks of 4 heads per KV head on the tcgen05 kernel, hd 256 chunks of 48 and
    64 rows on the CUDA-core kernel (two far rows per warp past 32); one
    sequence starts evicting mid-chunk."""
    w, inp = _far_case(53 + t, t=t, hd=hd, nh=nh, nk=nk, window=W, cap=W, pos_lo=max(1, W // 2), pos_hi=W)
    inp["meta"][2, 0] = W - 2                           # fills after two rows of the chunk
    inp["meta"][2, 1] = 0
    _far_step_check(w, inp, 0, 0)


def test_ordered_verify_blocks_with_a_far_field():
    """Far more verify blocks (32 query vectors) than resident CTAs with a far
    field: one split each, taken longest first; the blocks write records and the
    merge joins the far part, gates and commits (far kernel, order, attention,
    merge: four launches). Every output row against the oracle; ring, meta and
    far state after the commit."""
    w, inp = _far_case(71, B=600, t=8)
    inp["meta"][2, 0] = w.window - 2                    # fills after two rows of the chunk
    inp["meta"][2, 1] = 0
    inp["far"]["mu"] = inp["far"]["mu"] - 0.05
    res = gpu_full_path(w, inp, commit=True, far=inp["far"])
    assert res["err"] == 0 and res["attend_launches"] == 4
    a = oracle_inputs(w, inp, *_gpu_prepped(res))
    assert_close(res["out"], oracle.attend_far(a, far_to_np(inp["far"]), w.score_scale, w.hpg), "out (far field)")
    check_commit_placement(w, inp, res)
    _check_far_state(w, inp, res)


def test_far_decode_with_odd_landmark_count():
    """m = 7: the per-head shared-memory sections of a CTA that serves several
    decode heads stay aligned; heads past nh in the last CTA write nothing."""
    w, inp = _far_case(61, nh=6, nk=2, far_m=7)
    _far_step_check(w, inp, 1, 0)


def _far_step_check(w, inp, rect, splits):
    inp["far"]["rect"] = rect
    inp["far"]["mu"] = inp["far"]["mu"] - 0.05       # some negative landmark weights for the clip
    res = gpu_full_path(w, inp, commit=True, num_splits=splits, far=inp["far"])
    assert res["err"] == 0
    a = oracle_inputs(w, inp, *_gpu_prepped(res))
    ref = oracle.attend_far(a, far_to_np(inp["far"]), w.score_scale, w.hpg)
    assert_close(res["out"], ref, "out (far field)")
    check_commit_placement(w, inp, res)
    _check_far_state(w, inp, res)


def test_far_part_with_negative_mass_is_dropped_on_gpu():
    w, inp = _far_case(43)
    inp["far"]["mu"] = -inp["far"]["mu"].abs() - 0.1
    res = gpu_full_path(w, inp, commit=False, far=inp["far"])
    a = oracle_inputs(w, inp, *_gpu_prepped(res))
    assert_close(res["out"], oracle.attend(a, w.score_scale, w.hpg), "out (far mass < 0)")
    # without commit the far state is left as it was
    np.testing.assert_array_equal(res["far"]["t_hat"], inp["far"]["t_hat"].numpy())


def test_far_field_exact_over_decode_steps_with_landmarks_at_the_evicted_keys():
    """GPU version of the Nystrom pin: the landmarks are the keys the next
    steps evict and mu inverts their kernel matrix, so every step must equal
    the oracle's far-field step (itself pinned to full attention over every
    evicted key) while the far state advances through the GPU's commits."""
    hd, nh, nk, m, W = 64, 4, 2, 4, 12
    w = workloads.custom(B=2, t=1, nh=nh, nk=nk, hd=hd, window=W, cap=W, ns=1, pos_mode="full",
                         pos_lo=W, pos_hi=5 * W, seed=47)
    inp = workloads.make_inputs(w)
    inp["meta"][:, 2] = 0                               # nothing evicted yet
    rng = np.random.default_rng(5)
    scale = w.score_scale
    kt = np.zeros((w.B, nk, m, hd))
    qt = 1.5 * rng.normal(size=(w.B, nh, m, hd))
    mu = np.zeros((w.B, nh, m, m))
    for b in range(w.B):
        head0 = int(inp["meta"][b, 1])
        for g in range(nk):
            kt[b, g] = inp["ring_k"][b, g, [(head0 + j) % W for j in range(m)]].numpy()
        for h in range(nh):
            mu[b, h] = np.linalg.inv(np.exp(scale * qt[b, h] @ kt[b, h // w.hpg].T))
    far_np = {"m": m, "rect": 0, "k_tilde": kt, "q_tilde": qt, "mu": mu,
              "mz": np.concatenate([np.full((w.B, nh, m), -np.inf), np.zeros((w.B, nh, m))], axis=2),
              "t_hat": np.zeros((w.B, nh, m, hd))}
    far_d = {k: (torch.tensor(v, dtype=torch.float32).cuda() if isinstance(v, np.ndarray) else v)
             for k, v in far_np.items()}
    d = to_dev({k: v for k, v in inp.items() if k != "far"})
    ring_k, ring_v, meta = d["ring_k"].clone(), d["ring_v"].clone(), d["meta"].clone()
    g = torch.Generator().manual_seed(9)
    for step in range(m):
        q = torch.randn(w.B, 1, nh, hd, generator=g)
        k = torch.randn(w.B, 1, nk, hd, generator=g)
        v = torch.randn(w.B, 1, nk, hd, generator=g)
        gate = torch.randn(w.B, 1, nh, hd, generator=g)
        a = {"meta": meta.cpu().numpy().astype(np.int64), "q": q.numpy(), "k_chunk": k.numpy(),
             "v_chunk": v.numpy(), "ring_k": ring_k.cpu().numpy(), "ring_v": ring_v.cpu().numpy(),
             "sink_k": inp["sink_k"].numpy(), "sink_v": inp["sink_v"].numpy(), "gate": gate.numpy(),
             "gate_scale": inp["gate_scale"].numpy()}
        ref = oracle.attend_far(a, far_np, scale, w.hpg)
        meta_next = torch.empty_like(meta)
        out = swa.attend(meta, q.cuda(), k.cuda(), v.cuda(), ring_k, ring_v, d["sink_k"], d["sink_v"],
                         gate.cuda(), d["gate_scale"], scale, commit=True, meta_out=meta_next, far=far_d)
        assert_close(out.cpu().numpy(), ref, f"far step {step}")
        far_np["mz"], far_np["t_hat"] = oracle.far_commit(a, far_np, scale, w.hpg)
        meta = meta_next
        assert int(meta[0, 2].item()) == step + 1


# ---------------------------------------------------------------------------
# the named workloads at full size, in the launch configuration the bench times
# (automatic splits): every prep output, the ring and meta after the commit bit
# for bit for every sequence, and the attention output of every vector of the
# decode workloads and of every row of whole sequences of the chunk workloads
# (the oracle runs in a pool of worker processes)
# ---------------------------------------------------------------------------
def _full_size_rows(w, meta):
    """(b, i, h) of the output vectors checked against the oracle: all of them
    for decode rows; for chunks, every row and head of a few whole sequences:
    a full wrapped ring, an empty or the shortest ring, the longest of the
    others and one more."""
    W = w.window
    if w.t == 1:
        seqs = list(range(w.B))
    else:
        lens = [int(meta[b][0]) for b in range(w.B)]
        full = [b for b in range(w.B) if lens[b] == W]
        seqs = [full[0] if full else 0, int(np.argmin(lens))]
        if w.B > 2:
            rest = [b for b in range(w.B) if b not in seqs]
            seqs.append(max(rest, key=lambda b: lens[b]))
            rest = [b for b in rest if b not in seqs]
            if rest:
                seqs.append(rest[len(rest) // 2])
        seqs = sorted(set(seqs))
    return [(b, i, h) for b in seqs for i in range(w.t) for h in range(w.nh)], seqs


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_named_workload_full_size(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w)
    res = gpu_full_path(w, inp, commit=True, far=inp.get("far"))
    assert res["err"] == 0
    rope = oracle.rope_table(inp["pos0"].numpy(), w.t, w.hd, w.theta)
    q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                          inp["q_scale"].numpy(), w.eps)
    assert_close(res["q"], q, "q_hat")
    assert_close(res["k"], k, "k_hat")
    # every output is finite; ring and meta after the commit exact for every sequence
    assert np.all(np.isfinite(res["out"]))
    check_commit_placement_full(w, inp, res)
    a = oracle_inputs(w, inp, q, k, v)
    rows, seqs = _full_size_rows(w, inp["meta"].numpy())
    if w.t > 1:
        assert len(seqs) >= 2
    ref = oracle_rows(a, rows, w.score_scale, w.hpg, far=far_to_np(inp["far"]) if w.far_m else None)
    got = np.stack([res["out"][b, i, h] for b, i, h in rows])
    assert_close(got, ref, f"{name}: {len(rows)} output vectors of sequences {seqs[:4]}...")
