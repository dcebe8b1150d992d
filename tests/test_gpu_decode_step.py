"""swa_decode_step: one decode token (t = 1) in one call, against the oracle
and against swa_prep + swa_attend with commit on the same tensors (the same
bits: output, ring and meta; the one-kernel form attends each (sequence, KV
head) as one split, so it is compared with swa_attend at one split). The
one-kernel form is taken for at most 8 query heads per KV head, meta_out not
aliasing meta, and short windows or a one-split plan; the other calls run prep,
attention and merge."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import sliding_window_gqa_prep_gb300 as swa
from swa_harness import assert_close, oracle_inputs, oracle_rows, to_dev

pytestmark = pytest.mark.gpu

# (case, kernels the call is expected to launch)
CASES = [
    # the tiny decode shape: wrapped ring of 32, two KV heads of 4 query heads
    (dict(B=1, nh=8, nk=2, hd=64, window=32, cap=32, ns=0, pos_mode="fixed", pos_lo=100), 1),
    # wrapped rings with sinks, several tiles and a ragged tail
    (dict(B=3, nh=8, nk=2, hd=128, window=200, cap=200, ns=3, pos_mode="full", pos_lo=200, pos_hi=5000), 1),
    # one query head per KV head, partially filled rings
    (dict(B=2, nh=2, nk=2, hd=64, window=40, cap=40, ns=0, pos_mode="partial", pos_lo=1, pos_hi=40), 1),
    # eight query heads per KV head (8 query vectors)
    (dict(B=2, nh=16, nk=2, hd=128, window=64, cap=64, ns=2, pos_mode="full", pos_lo=64, pos_hi=900), 1),
    # hd 256, one KV head, eight sinks
    (dict(B=2, nh=4, nk=1, hd=256, window=100, cap=100, ns=8, pos_mode="full", pos_lo=100, pos_hi=99999), 1),
    # an empty ring (position 0: the row's own key and the sinks only) beside a partial one
    (dict(B=2, nh=8, nk=2, hd=64, window=48, cap=48, ns=2, pos_mode="prompt", pos_lo=0, pos_hi=30), 1),
    # a window shorter than the ring's capacity
    (dict(B=2, nh=8, nk=2, hd=128, window=20, cap=32, ns=1, pos_mode="full", pos_lo=20, pos_hi=500), 1),
    # 32 query heads per KV head: the attention takes the 32-vector kernel, three launches
    (dict(B=1, nh=32, nk=1, hd=128, window=90, cap=90, ns=2, pos_mode="full", pos_lo=90, pos_hi=400), 3),
    # a window of 513 keys with 8 sinks at hd 64 (265 KB per KV head): one kernel
    (dict(B=2, nh=8, nk=2, hd=64, window=513, cap=513, ns=8, pos_mode="full", pos_lo=513, pos_hi=9000), 1),
    # a long window over few (sequence, KV head) pairs: split-KV, three launches
    (dict(B=2, nh=4, nk=1, hd=128, window=3000, cap=3000, ns=4, pos_mode="full", pos_lo=3000, pos_hi=9000), 3),
]


def _oracle_step(w, inp):
    rope = oracle.rope_table(inp["pos0"].numpy(), 1, w.hd, w.theta)
    q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                          inp["q_scale"].numpy(), w.eps)
    a = oracle_inputs(w, inp, q, k, v)
    return oracle.attend(a, w.score_scale, w.hpg), k


def _gpu_step(w, d, meta_alias=False):
    ring_k, ring_v = d["ring_k"].clone(), d["ring_v"].clone()
    meta = d["meta"].clone()
    meta_out = meta if meta_alias else torch.full_like(meta, -1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B, nh, nk, hd = w.B, w.nh, w.nk, w.hd
    n0 = swa.launch_count()
    out = swa.decode_step(d["yq"].view(B, nh, hd), d["yk"].view(B, nk, hd), d["yv"].view(B, nk, hd),
                          d["q_scale"], d["pos0"], meta, ring_k, ring_v,
                          d["sink_k"] if w.ns else None, d["sink_v"] if w.ns else None,
                          d["gate"].view(B, nh, hd), d["gate_scale"], w.score_scale, eps=w.eps,
                          theta=w.theta, meta_out=meta_out, err=err)
    torch.cuda.synchronize()
    return {"out": out, "ring_k": ring_k, "ring_v": ring_v, "meta_out": meta_out,
            "launches": swa.launch_count() - n0, "err": int(err.item())}


def _reference_path(w, d, num_splits=0):
    """swa_prep (angles in the kernel, no ring write) + swa_attend (commit)."""
    ring_k, ring_v = d["ring_k"].clone(), d["ring_v"].clone()
    meta_out = torch.full_like(d["meta"], -1)
    q, k, v = swa.prep(d["yq"], d["yk"], d["yv"], None, d["q_scale"], w.eps, pos0=d["pos0"],
                       theta=w.theta, copy_v=False)
    out = swa.attend(d["meta"], q, k, v, ring_k, ring_v, d["sink_k"] if w.ns else None,
                     d["sink_v"] if w.ns else None, d["gate"], d["gate_scale"], w.score_scale,
                     commit=True, meta_out=meta_out, num_splits=num_splits)
    torch.cuda.synchronize()
    return {"out": out.view(w.B, w.nh, w.hd), "ring_k": ring_k, "ring_v": ring_v, "meta_out": meta_out}


@pytest.mark.parametrize("kw,launches", CASES)
def test_decode_step_matches_oracle_and_the_prep_attend_path(kw, launches):
    w = workloads.custom(t=1, seed=41, **kw)
    inp = workloads.make_inputs(w)
    d = to_dev(inp)
    assert swa.decode_launches(w.B, w.nh, w.nk, w.hd, w.cap, w.ns, meta=d["meta"],
                               meta_out=torch.empty_like(d["meta"])) == launches
    res = _gpu_step(w, d)
    assert res["err"] == 0
    assert res["launches"] == launches
    ref_out, ref_k = _oracle_step(w, inp)
    assert_close(res["out"].cpu().numpy(), ref_out[:, 0], "decode_step out vs oracle")
    # the same bits as prep + attend with commit (one split for the one-kernel form)
    two = _reference_path(w, d, num_splits=1 if launches == 1 else 0)
    assert torch.equal(res["out"], two["out"])
    assert torch.equal(res["ring_k"], two["ring_k"]) and torch.equal(res["ring_v"], two["ring_v"])
    assert torch.equal(res["meta_out"], two["meta_out"])
    # ring and meta against the oracle: the committed slot holds the row's k-hat
    # (oracle within tolerance) and v (exact); every other slot is untouched
    meta = inp["meta"].numpy()
    ring_k, ring_v = res["ring_k"].cpu().numpy(), res["ring_v"].cpu().numpy()
    for b in range(w.B):
        slot = oracle.commit_slot(meta[b], 0, w.cap)
        assert_close(ring_k[b, :, slot], ref_k[b, 0], "committed k-hat")
        np.testing.assert_array_equal(ring_v[b, :, slot], inp["yv"].numpy()[b, 0])
        others = [s for s in range(w.cap) if s != slot]
        np.testing.assert_array_equal(ring_k[b][:, others], inp["ring_k"].numpy()[b][:, others])
        np.testing.assert_array_equal(ring_v[b][:, others], inp["ring_v"].numpy()[b][:, others])
        assert res["meta_out"][b].cpu().numpy().astype(np.int64).tolist() == \
            oracle.commit_meta(meta[b], 1, w.cap).tolist()


def test_decode_step_with_meta_out_aliasing_meta_takes_the_three_launch_form():
    kw, _ = CASES[0]
    w = workloads.custom(t=1, seed=42, **kw)
    inp = workloads.make_inputs(w)
    d = to_dev(inp)
    m = d["meta"].clone()
    assert swa.decode_launches(w.B, w.nh, w.nk, w.hd, w.cap, w.ns, meta=m, meta_out=m) == 3
    res = _gpu_step(w, d, meta_alias=True)
    assert res["launches"] == 3 and res["err"] == 0
    two = _reference_path(w, d)
    assert torch.equal(res["out"], two["out"])
    assert torch.equal(res["ring_k"], two["ring_k"]) and torch.equal(res["ring_v"], two["ring_v"])
    assert torch.equal(res["meta_out"], two["meta_out"])


def test_decode_steps_in_sequence_equal_a_chunk():
    """Four one-kernel steps, each committing its row, give the ring and meta of
    one 4-row chunk committed by swa_attend, and each step's output matches the
    oracle's row of that chunk."""
    w = workloads.custom(B=2, t=4, nh=8, nk=2, hd=64, window=24, cap=24, ns=2, pos_mode="full",
                         pos_lo=24, pos_hi=300, seed=43)
    inp = workloads.make_inputs(w)
    d = to_dev(inp)
    rope = oracle.rope_table(inp["pos0"].numpy(), w.t, w.hd, w.theta)
    q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                          inp["q_scale"].numpy(), w.eps)
    ref = oracle.attend(oracle_inputs(w, inp, q, k, v), w.score_scale, w.hpg)
    ring_k, ring_v = d["ring_k"].clone(), d["ring_v"].clone()
    meta = d["meta"].clone()
    B, nh, nk, hd = w.B, w.nh, w.nk, w.hd
    for j in range(w.t):
        pos = (d["pos0"] + j).contiguous()
        meta_out = torch.empty_like(meta)
        assert swa.decode_launches(B, nh, nk, hd, w.cap, w.ns, meta=meta, meta_out=meta_out) == 1
        out = swa.decode_step(d["yq"][:, j].contiguous(), d["yk"][:, j].contiguous(),
                              d["yv"][:, j].contiguous(), d["q_scale"], pos, meta, ring_k, ring_v,
                              d["sink_k"], d["sink_v"], d["gate"][:, j].contiguous(), d["gate_scale"],
                              w.score_scale, eps=w.eps, theta=w.theta, meta_out=meta_out)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref[:, j], f"step {j}")
        meta = meta_out
    meta0 = inp["meta"].numpy()
    for b in range(B):
        assert meta[b].cpu().numpy().astype(np.int64).tolist() == oracle.commit_meta(meta0[b], w.t, w.cap).tolist()
        for j in range(w.t):
            slot = oracle.commit_slot(meta0[b], j, w.cap)
            assert_close(ring_k[b, :, slot].cpu().numpy(), k[b, j], f"ring k row {j}")
            np.testing.assert_array_equal(ring_v[b, :, slot].cpu().numpy(), inp["yv"].numpy()[b, j])


def _check_step(w, inp, d, launches, rows=None):
    """The step against the oracle (every output vector, or `rows`), and against
    swa_prep + swa_attend on the same tensors: the same bits for the output, the
    ring and the meta."""
    res = _gpu_step(w, d)
    assert res["err"] == 0 and res["launches"] == launches
    rope = oracle.rope_table(inp["pos0"].numpy(), 1, w.hd, w.theta)
    q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                          inp["q_scale"].numpy(), w.eps)
    rows = rows or [(b, 0, h) for b in range(w.B) for h in range(w.nh)]
    ref = oracle_rows(oracle_inputs(w, inp, q, k, v), rows, w.score_scale, w.hpg)
    out = res["out"].cpu().numpy()
    assert_close(np.stack([out[b, h] for b, _, h in rows]), ref, f"{w.name}: {len(rows)} output vectors")
    two = _reference_path(w, d, num_splits=1 if launches == 1 else 0)
    assert torch.equal(res["out"], two["out"])
    assert torch.equal(res["ring_k"], two["ring_k"]) and torch.equal(res["ring_v"], two["ring_v"])
    assert torch.equal(res["meta_out"], two["meta_out"])
    meta = inp["meta"].numpy()
    for b in range(w.B):
        assert res["meta_out"][b].cpu().numpy().astype(np.int64).tolist() == \
            oracle.commit_meta(meta[b], 1, w.cap).tolist()
    return res, k


@pytest.mark.parametrize("name", ["tiny_decode", "batched_decode", "long_decode"])
def test_decode_step_full_size(name):
    """The decode workloads at full size through swa_decode_step, the call the
    benchmark times: every output vector against the oracle, and output, ring and
    meta bit for bit against swa_prep + swa_attend."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w)
    d = to_dev({k: v for k, v in inp.items() if k != "far"})
    launches = swa.decode_launches(w.B, w.nh, w.nk, w.hd, w.cap, w.ns, meta=d["meta"],
                                   meta_out=torch.empty_like(d["meta"]))
    assert launches in (1, 3)
    _check_step(w, inp, d, launches)
