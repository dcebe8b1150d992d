"""swa_attend_noalloc: the attention for callers that cannot allocate device memory.

A plugin handed only its input and output buffers, a serving engine whose
device memory is all reserved by its own allocator, or a latency-critical
loop that must avoid the synchronisation an allocation can cause cannot give
swa_attend a workspace. swa_attend_noalloc takes its scratch from a fixed
array inside the library instead. These tests call it through the C ABI and
check it against swa_attend (caller-owned workspace): twice in a row, on
different shapes and data, so results left in the shared array by one call
cannot leak into the next; and an oversized call is refused up front.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
import sliding_window_gqa_prep_gb300 as swa
from sliding_window_gqa_prep_gb300 import _abi
from swa_harness import assert_close, to_dev

pytestmark = pytest.mark.gpu


def _noalloc():
    lib = swa.library()
    fn = lib.swa_attend_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(_abi.AttendArgs), ctypes.c_void_p]
    return fn


def _struct(w, d, q, k, v, ring_k, ring_v, out, meta_out, commit):
    a = _abi.AttendArgs()
    a.B, a.t, a.nh, a.nk, a.hd, a.cap, a.ns = w.B, w.t, w.nh, w.nk, w.hd, w.cap, w.ns
    a.scale = w.score_scale
    a.meta = d["meta"].data_ptr()
    a.q, a.k_chunk, a.v_chunk = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.ring_k, a.ring_v = ring_k.data_ptr(), ring_v.data_ptr()
    a.sink_k = d["sink_k"].data_ptr() if w.ns else 0
    a.sink_v = d["sink_v"].data_ptr() if w.ns else 0
    a.gate, a.gate_scale = d["gate"].data_ptr(), d["gate_scale"].data_ptr()
    a.out = out.data_ptr()
    a.workspace, a.workspace_bytes = None, 0       # ignored by swa_attend_noalloc
    a.commit = 1 if commit else 0
    a.meta_out = meta_out.data_ptr()
    a.num_splits = 0
    return a


CASES = [
    # decode: wrapped rings, sinks, several splits per (sequence, KV head)
    dict(B=8, t=1, nh=16, nk=4, hd=128, window=1024, cap=1024, ns=4, pos_mode="full",
         pos_lo=1024, pos_hi=20000, seed=31),
    # verify-shaped chunk with commit: a different plan and scratch layout
    dict(B=4, t=8, nh=16, nk=4, hd=64, window=300, cap=300, ns=2, pos_mode="partial",
         pos_lo=1, pos_hi=300, seed=32),
    # prompt chunk on the tensor-core kernel whose split-once operand blocks fit
    # the fixed scratch as well (swa_attend_workspace_size <= 16 MiB)
    dict(B=2, t=128, nh=8, nk=2, hd=64, window=256, cap=256, ns=4, pos_mode="full",
         pos_lo=256, pos_hi=2000, seed=33),
    # prompt chunk whose operand blocks do not fit: only swa_attend_workspace_min
    # does, and the kernel stages and splits K/V itself
    dict(B=2, t=128, nh=32, nk=8, hd=128, window=2048, cap=2048, ns=4, pos_mode="full",
         pos_lo=2048, pos_hi=6000, seed=34),
]


def _fits(kw):
    w = workloads.custom(**kw)
    a = _abi.AttendArgs()
    a.B, a.t, a.nh, a.nk, a.hd, a.cap, a.ns = w.B, w.t, w.nh, w.nk, w.hd, w.cap, w.ns
    a.scale = w.score_scale
    lib = swa.library()
    return (lib.swa_attend_workspace_min(ctypes.byref(a)) <= (16 << 20),
            lib.swa_attend_workspace_size(ctypes.byref(a)) <= (16 << 20))


def test_noalloc_prompt_cases_cover_both_scratch_layouts():
    assert _fits(CASES[2]) == (True, True)
    assert _fits(CASES[3]) == (True, False)


def test_noalloc_matches_swa_attend_on_two_calls_in_a_row():
    fn = _noalloc()
    stream = torch.cuda.current_stream()
    for kw in CASES:
        w = workloads.custom(**kw)
        d = to_dev(workloads.make_inputs(w))
        rope = swa.rope_table(d["pos0"], w.t, w.hd, w.theta)
        q, k, v = swa.prep(d["yq"], d["yk"], d["yv"], rope, d["q_scale"], w.eps)
        commit = w.t > 1
        # existing entry point, caller-owned workspace
        rk_ref, rv_ref = d["ring_k"].clone(), d["ring_v"].clone()
        meta_ref = torch.empty_like(d["meta"])
        ref = swa.attend(d["meta"], q, k, v, rk_ref, rv_ref, d["sink_k"] if w.ns else None,
                         d["sink_v"] if w.ns else None, d["gate"], d["gate_scale"],
                         w.score_scale, commit=commit, meta_out=meta_ref)
        # allocation-free entry point
        rk, rv = d["ring_k"].clone(), d["ring_v"].clone()
        meta_out = torch.empty_like(d["meta"])
        out = torch.full_like(q, float("nan"))
        a = _struct(w, d, q, k, v, rk, rv, out, meta_out, commit)
        rc = fn(ctypes.byref(a), stream.cuda_stream)
        assert rc == _abi.SWA_OK, swa.library().swa_status_string(rc)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref.cpu().numpy(), f"noalloc vs swa_attend ({kw})")
        if commit:
            np.testing.assert_array_equal(rk.cpu().numpy(), rk_ref.cpu().numpy())
            np.testing.assert_array_equal(rv.cpu().numpy(), rv_ref.cpu().numpy())
            np.testing.assert_array_equal(meta_out.cpu().numpy(), meta_ref.cpu().numpy())


def test_noalloc_refuses_sizes_beyond_its_scratch():
    fn = _noalloc()
    # 256 sequences x 32 KV heads x 32 query vectors x 128 features of partial
    # records is far beyond the fixed scratch
    a = _abi.AttendArgs()
    a.B, a.t, a.nh, a.nk, a.hd, a.cap, a.ns = 256, 8, 128, 32, 128, 4096, 4
    a.scale = 0.1
    # aligned stand-ins that are never dereferenced: the call is refused first
    for f in ("meta", "q", "k_chunk", "v_chunk", "ring_k", "ring_v", "sink_k", "sink_v", "gate",
              "gate_scale", "out"):
        setattr(a, f, 0x10000)
    need = swa.library().swa_attend_workspace_size(ctypes.byref(a))
    assert need > (16 << 20)
    n0 = swa.launch_count()
    assert fn(ctypes.byref(a), None) == _abi.SWA_E_WORKSPACE
    assert swa.launch_count() == n0
