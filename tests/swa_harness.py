"""Shared helpers of the parity tests: run the CUDA path and the CPU oracle on
the same seeded inputs and compare them.

Tolerance (floating point outputs, per tensor): max |gpu - oracle| <= 2e-5 and
max |gpu - oracle| / max |oracle| <= 1e-4. Integer results (ring slots, meta)
are compared exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads
import sliding_window_gqa_prep_gb300 as swa

MAX_ABS = 2e-5
MAX_REL = 1e-4


def assert_close(gpu, ref, what, max_abs=MAX_ABS, max_rel=MAX_REL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    err = np.max(np.abs(gpu - ref)) if gpu.size else 0.0
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    rel = err / scale if scale > 0 else err
    assert err <= max_abs and rel <= max_rel, f"{what}: max_abs {err:.3e}, rel {rel:.3e}"
    return err, rel


def to_dev(inp, dev="cuda"):
    out = {}
    for k, v in inp.items():
        if k in ("meta", "pos0"):
            out[k] = v.to(torch.int32).to(dev).contiguous()
        else:
            out[k] = v.to(dev).contiguous()
    return out


def far_to_dev(far, dev="cuda"):
    return {k: (v.to(dev).contiguous() if torch.is_tensor(v) else v) for k, v in far.items()}


def far_to_np(far):
    return {k: (v.numpy().astype(np.float64) if torch.is_tensor(v) else v) for k, v in far.items()}


def gpu_full_path(w, inp, *, commit=True, num_splits=0, prep_ring=None, meta_alias=False, far=None,
                  min_workspace=False):
    """rope table -> prep -> attend (+ commit) on the GPU. The prep writes the
    ring only for t == 1 with window == cap (prep's slot map) and no far field;
    otherwise the attend's commit does. far: the generator's far state (CPU);
    the result then holds the far state after the call."""
    d = {k: v for k, v in to_dev({k: v for k, v in inp.items() if k != "far"}).items()}
    far_d = far_to_dev(far) if far is not None else None
    if prep_ring is None:
        prep_ring = w.t == 1 and w.window == w.cap and far is None
    rope = swa.rope_table(d["pos0"], w.t, w.hd, w.theta)
    ring_k, ring_v = d["ring_k"].clone(), d["ring_v"].clone()
    q, k, v = swa.prep(d["yq"], d["yk"], d["yv"], rope, d["q_scale"], w.eps, pos0=d["pos0"],
                       ring_k=ring_k if prep_ring else None,
                       ring_v=ring_v if prep_ring else None)
    ring_after_prep_k = ring_k.clone() if prep_ring else None
    meta = d["meta"].clone()
    n_launch = swa.launch_count()
    meta_out = meta if meta_alias else torch.full_like(meta, -1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = swa.attend(meta, q, k, v, ring_k, ring_v, d["sink_k"] if w.ns else None,
                     d["sink_v"] if w.ns else None, d["gate"], d["gate_scale"], w.score_scale,
                     commit=commit, meta_out=meta_out, num_splits=num_splits, err=err, far=far_d,
                     workspace=(torch.empty(swa.attend_workspace_min(w.B, w.t, w.nh, w.nk, w.hd, w.cap, w.ns,
                                                                     num_splits, w.far_m),
                                            dtype=torch.uint8, device="cuda") if min_workspace else None))
    torch.cuda.synchronize()
    return {
        "rope": rope.cpu().numpy(), "q": q.cpu().numpy(), "k": k.cpu().numpy(),
        "attend_launches": swa.launch_count() - n_launch,
        "v": v.cpu().numpy(), "out": out.cpu().numpy(), "ring_k": ring_k.cpu().numpy(),
        "ring_v": ring_v.cpu().numpy(), "meta_out": meta_out.cpu().numpy(),
        "err": int(err.item()),
        "far": None if far_d is None else {k: (v.cpu().numpy() if torch.is_tensor(v) else v)
                                          for k, v in far_d.items()},
        "ring_after_prep_k": None if ring_after_prep_k is None else ring_after_prep_k.cpu().numpy(),
    }


def oracle_inputs(w, inp, q=None, k=None, v=None):
    """The oracle's attend inputs: its own prep unless q/k/v are given."""
    if q is None:
        rope = oracle.rope_table(inp["pos0"].numpy(), w.t, w.hd, w.theta)
        q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                              inp["q_scale"].numpy(), w.eps)
    return {
        "meta": inp["meta"].numpy(), "q": q, "k_chunk": k, "v_chunk": v,
        "ring_k": inp["ring_k"].numpy(), "ring_v": inp["ring_v"].numpy(),
        "sink_k": inp["sink_k"].numpy(), "sink_v": inp["sink_v"].numpy(),
        "gate": inp["gate"].numpy(), "gate_scale": inp["gate_scale"].numpy(),
    }


def check_commit_placement(w, inp, res):
    """Ring after the commit: each slot the oracle's slot map assigns to chunk
    row j holds the GPU's own k/v row j bit for bit; every other slot is
    unchanged (bit for bit). Meta after the commit equals the oracle's."""
    meta = inp["meta"].numpy()
    ring0_k = inp["ring_k"].numpy()
    ring0_v = inp["ring_v"].numpy()
    for b in range(w.B):
        final = {}
        for j in range(w.t):
            final[oracle.commit_slot(meta[b], j, w.cap)] = j
        for slot in range(w.cap):
            if slot in final:
                j = final[slot]
                np.testing.assert_array_equal(res["ring_k"][b, :, slot], res["k"][b, j])
                np.testing.assert_array_equal(res["ring_v"][b, :, slot], res["v"][b, j])
            else:
                np.testing.assert_array_equal(res["ring_k"][b, :, slot], ring0_k[b, :, slot])
                np.testing.assert_array_equal(res["ring_v"][b, :, slot], ring0_v[b, :, slot])
        expect = oracle.commit_meta(meta[b], w.t, w.cap)
        assert res["meta_out"][b].astype(np.int64).tolist() == expect.tolist(), (b, res["meta_out"][b], expect)


def check_commit_placement_full(w, inp, res):
    """check_commit_placement for large batches, vectorised: the expected ring
    is the ring before the call with chunk row j of sequence b written to the
    oracle's slot for (b, j), rows in order (a later row that lands on the
    same slot wins); it must equal the GPU's ring bit for bit, as must the
    meta after the commit."""
    meta = inp["meta"].numpy()
    exp_k = inp["ring_k"].numpy().copy()
    exp_v = inp["ring_v"].numpy().copy()
    for b in range(w.B):
        for j in range(w.t):
            slot = oracle.commit_slot(meta[b], j, w.cap)
            exp_k[b, :, slot] = res["k"][b, j]
            exp_v[b, :, slot] = res["v"][b, j]
        expect = oracle.commit_meta(meta[b], w.t, w.cap)
        assert res["meta_out"][b].astype(np.int64).tolist() == expect.tolist(), (b, res["meta_out"][b], expect)
    np.testing.assert_array_equal(res["ring_k"], exp_k)
    np.testing.assert_array_equal(res["ring_v"], exp_v)


# ---------------------------------------------------------------------------
# The oracle over many output vectors: a pool of single-threaded worker
# processes (spawn start, safe after CUDA is initialised), each sent the slices
# of the sequences it computes, calling oracle.attend_row /
# oracle.attend_far_row as they are.
# ---------------------------------------------------------------------------
_PER_SEQ = ("meta", "q", "k_chunk", "v_chunk", "ring_k", "ring_v", "sink_k", "sink_v", "gate")
_FAR_PER_SEQ = ("k_tilde", "q_tilde", "mu", "mz", "t_hat")


def _oracle_task(job):
    sub, far, rows, scale, hpg = job
    if far is None:
        return np.stack([oracle.attend_row(b, i, h, sub, scale, hpg) for b, i, h in rows])
    return np.stack([oracle.attend_far_row(b, h, sub, far, scale, hpg, i) for b, i, h in rows])


def oracle_rows(a, rows, scale, hpg, far=None, procs=None):
    """oracle.attend_row (or attend_far_row with `far`) for every (b, i, h) in
    `rows`, in that order, computed by a process pool; each task holds whole
    sequences, re-indexed from 0."""
    import os
    import multiprocessing as mp
    procs = procs or max(1, min(16, os.cpu_count() or 1))
    seqs = sorted({b for b, _, _ in rows})
    groups = [seqs[k::procs] for k in range(procs) if seqs[k::procs]]
    jobs, where = [], []
    for grp in groups:
        idx = {b: n for n, b in enumerate(grp)}
        sub = {k: (np.ascontiguousarray(v[grp]) if k in _PER_SEQ else v) for k, v in a.items()}
        fsub = None
        if far is not None:
            fsub = {k: (np.ascontiguousarray(v[grp]) if k in _FAR_PER_SEQ else v) for k, v in far.items()}
        mine = [(n, r) for n, r in enumerate(rows) if r[0] in idx]
        jobs.append((sub, fsub, [(idx[b], i, h) for _, (b, i, h) in mine], scale, hpg))
        where.append([n for n, _ in mine])
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v in saved:
        os.environ[v] = "1"
    try:
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            parts = pool.map(_oracle_task, jobs, chunksize=1)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    out = np.empty((len(rows), parts[0].shape[1]), np.float64)
    for part, pos in zip(parts, where):
        out[pos] = part
    return out
