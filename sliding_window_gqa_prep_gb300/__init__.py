"""Sliding-window GQA token path on GB300: Python binding of libswa_gb300.so.

The binding only checks tensors and passes their device addresses to the C ABI
(include/swa.h); every step of the path runs in the library's CUDA kernels.
PyTorch provides device memory and streams. There is no CPU fallback: on a
machine without the built library or without a GPU the calls raise.

Public calls (same names as the C ABI):
  rope_table(pos0, t, hd, theta)                 -> rope [B][t][hd]
  prep(yq, yk, yv, rope, q_scale, eps, ...)      -> (q, k, v) chunk tensors
  attend(meta, q, k_chunk, v_chunk, ring_k, ring_v, sink_k, sink_v,
         gate, gate_scale, scale, ...)           -> out [B][t][nh][hd]
  attend_workspace_size(B, t, nh, nk, hd, cap, ns, num_splits=0)
  decode_step(yq, yk, yv, q_scale, pos0, meta, ring_k, ring_v, sink_k, sink_v,
              gate, gate_scale, scale, ...)      -> out [B][nh][hd] (t = 1, one call)
  TokenPath: holds a batch's ring state and runs whole steps
Meta tensors are int32 [B][4] = (win_len, win_head, far_len, window), read by
the kernels as uint32; pos0 tensors are int32 [B].
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _abi
from ._abi import SwaError, SWA_DERR_META, SWA_DERR_TIMEOUT  # noqa: F401

__all__ = ["rope_table", "prep", "attend", "attend_workspace_size", "decode_step",
           "decode_workspace_size", "decode_launches", "rollback", "launch_count",
           "TokenPath", "SwaError", "library"]


def library() -> ctypes.CDLL:
    return _abi.load()


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(library().swa_launch_count())


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(x: Optional[torch.Tensor], name: str, shape=None, dtype=torch.float32,
         required: bool = True) -> int:
    if x is None:
        if required:
            raise ValueError(f"{name} is required")
        return 0
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(x.shape)}, expected {tuple(shape)}")
    return x.data_ptr()


def rope_table(pos0: torch.Tensor, t: int, hd: int, theta: float = 10000.0,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """RoPE table [B][t][hd] (cos | sin of (pos0[b] + j) * theta^(-2e/hd))."""
    B = pos0.shape[0]
    if out is None:
        out = torch.empty(B, t, hd, device=pos0.device, dtype=torch.float32)
    lib = library()
    rc = lib.swa_rope_table(_ptr(out, "out", (B, t, hd)), _ptr(pos0, "pos0", (B,), torch.int32),
                            B, t, hd, float(theta), _stream(stream))
    _abi.check(rc, "swa_rope_table")
    return out


def prep(yq, yk, yv, rope, q_scale, eps: float = 1e-6, *, pos0=None, ring_k=None,
         ring_v=None, q_out=None, k_out=None, v_out=None, copy_v: bool = True,
         theta: float = 10000.0, stream=None):
    """Rotation, unit heads, query scale and (t == 1 only) the ring write.

    rope=None computes the RoPE angles in the kernel from pos0 and theta
    (bit-identical to rope_table). Returns (q_out, k_out, v) where v is v_out
    when copy_v, else yv itself."""
    B, t, nh, hd = yq.shape
    nk = yk.shape[2]
    if q_out is None:
        q_out = torch.empty_like(yq)
    if k_out is None:
        k_out = torch.empty_like(yk)
    if copy_v and v_out is None:
        v_out = torch.empty_like(yv)
    cap = ring_k.shape[2] if ring_k is not None else 0
    a = _abi.PrepArgs()
    a.B, a.t, a.nh, a.nk, a.hd, a.cap = B, t, nh, nk, hd, cap
    a.eps = float(eps)
    a.yq = _ptr(yq, "yq", (B, t, nh, hd))
    a.yk = _ptr(yk, "yk", (B, t, nk, hd))
    a.yv = _ptr(yv, "yv", (B, t, nk, hd))
    a.rope = _ptr(rope, "rope", (B, t, hd), required=False)
    a.theta = float(theta)
    a.q_scale = _ptr(q_scale, "q_scale", (nh, hd))
    a.pos0 = _ptr(pos0, "pos0", (B,), torch.int32, required=ring_k is not None or rope is None)
    a.q_out = _ptr(q_out, "q_out", (B, t, nh, hd))
    a.k_out = _ptr(k_out, "k_out", (B, t, nk, hd))
    a.v_out = _ptr(v_out, "v_out", (B, t, nk, hd), required=False) if copy_v else 0
    a.ring_k = _ptr(ring_k, "ring_k", (B, nk, cap, hd), required=False)
    a.ring_v = _ptr(ring_v, "ring_v", (B, nk, cap, hd), required=ring_k is not None)
    rc = library().swa_prep(ctypes.byref(a), _stream(stream))
    _abi.check(rc, "swa_prep")
    return q_out, k_out, (v_out if copy_v else yv)


def _attend_struct(B, t, nh, nk, hd, cap, ns, num_splits=0) -> _abi.AttendArgs:
    a = _abi.AttendArgs()
    a.B, a.t, a.nh, a.nk, a.hd, a.cap, a.ns = B, t, nh, nk, hd, cap, ns
    a.num_splits = int(num_splits)
    return a


def attend_workspace_size(B, t, nh, nk, hd, cap, ns, num_splits: int = 0, far_m: int = 0) -> int:
    """Workspace bytes of swa_attend; far_m > 0 sizes it for a far field."""
    a = _attend_struct(B, t, nh, nk, hd, cap, ns, num_splits)
    fa = _abi.FarArgs()
    if far_m:
        fa.m = int(far_m)
        a.far = ctypes.pointer(fa)
    n = int(library().swa_attend_workspace_size(ctypes.byref(a)))
    if n == 0:
        raise SwaError(_abi.SWA_E_SHAPE, "swa_attend_workspace_size")
    return n


def attend_workspace_min(B, t, nh, nk, hd, cap, ns, num_splits: int = 0, far_m: int = 0) -> int:
    """The smallest workspace swa_attend accepts (without the split-once operand
    blocks of the tensor-core prompt kernel, which attend_workspace_size includes)."""
    a = _attend_struct(B, t, nh, nk, hd, cap, ns, num_splits)
    fa = _abi.FarArgs()
    if far_m:
        fa.m = int(far_m)
        a.far = ctypes.pointer(fa)
    n = int(library().swa_attend_workspace_min(ctypes.byref(a)))
    if n == 0:
        raise SwaError(_abi.SWA_E_SHAPE, "swa_attend_workspace_min")
    return n


def attend(meta, q, k_chunk, v_chunk, ring_k, ring_v, sink_k, sink_v, gate, gate_scale,
           scale: float, *, out=None, workspace=None, commit: bool = False, meta_out=None,
           num_splits: int = 0, err=None, ev_start=None, ev_stop=None, far=None, stream=None,
           gate_ready=None):
    """Attention of a chunk (decode, verify or prompt); see include/swa.h.

    gate_ready: optional recorded torch CUDA event that the merge (the only
    kernel that reads ``gate``) waits for, so the gate may still be copied in
    on another stream while the attention runs.

    far: optional far field of a decode step (t = 1), a dict with m, rect and
    the device tensors k_tilde [B][nk][m][hd], q_tilde [B][nh][m][hd],
    mu [B][nh][m][m], mz [B][nh][2m], t_hat [B][nh][m][hd] (mz and t_hat are
    updated in place when commit)."""
    B, t, nh, hd = q.shape
    nk = k_chunk.shape[2]
    cap = ring_k.shape[2]
    ns = sink_k.shape[2] if sink_k is not None else 0
    if out is None:
        out = torch.empty_like(q)
    far_m = int(far["m"]) if far is not None else 0
    if workspace is None:
        need = attend_workspace_size(B, t, nh, nk, hd, cap, ns, num_splits, far_m)
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    a = _attend_struct(B, t, nh, nk, hd, cap, ns, num_splits)
    a.scale = float(scale)
    a.meta = _ptr(meta, "meta", (B, 4), torch.int32)
    a.q = _ptr(q, "q", (B, t, nh, hd))
    a.k_chunk = _ptr(k_chunk, "k_chunk", (B, t, nk, hd))
    a.v_chunk = _ptr(v_chunk, "v_chunk", (B, t, nk, hd))
    a.ring_k = _ptr(ring_k, "ring_k", (B, nk, cap, hd))
    a.ring_v = _ptr(ring_v, "ring_v", (B, nk, cap, hd))
    a.sink_k = _ptr(sink_k, "sink_k", (B, nk, ns, hd), required=ns > 0) if ns else 0
    a.sink_v = _ptr(sink_v, "sink_v", (B, nk, ns, hd), required=ns > 0) if ns else 0
    a.gate = _ptr(gate, "gate", (B, t, nh, hd))
    a.gate_scale = _ptr(gate_scale, "gate_scale", (nh, hd))
    a.out = _ptr(out, "out", (B, t, nh, hd))
    a.workspace = _ptr(workspace, "workspace", None, torch.uint8)
    a.workspace_bytes = workspace.numel()
    a.commit = 1 if commit else 0
    a.meta_out = _ptr(meta_out, "meta_out", (B, 4), torch.int32, required=commit)
    a.err = _ptr(err, "err", (1,), torch.int32, required=False)
    a.ev_start = ctypes.c_void_p(ev_start.cuda_event) if ev_start is not None else None
    a.ev_stop = ctypes.c_void_p(ev_stop.cuda_event) if ev_stop is not None else None
    a.gate_ready = ctypes.c_void_p(gate_ready.cuda_event) if gate_ready is not None else None
    fa = None
    if far is not None:
        m = far_m
        fa = _abi.FarArgs()
        fa.m, fa.rect = m, 1 if far.get("rect") else 0
        fa.k_tilde = _ptr(far["k_tilde"], "k_tilde", (B, nk, m, hd))
        fa.q_tilde = _ptr(far["q_tilde"], "q_tilde", (B, nh, m, hd))
        fa.mu = _ptr(far["mu"], "mu", (B, nh, m, m))
        fa.mz = _ptr(far["mz"], "mz", (B, nh, 2 * m))
        fa.t_hat = _ptr(far["t_hat"], "t_hat", (B, nh, m, hd))
        a.far = ctypes.pointer(fa)
    rc = library().swa_attend(ctypes.byref(a), _stream(stream))
    _abi.check(rc, "swa_attend")
    return out


def _decode_struct(B, nh, nk, hd, cap, ns, meta=None, meta_out=None) -> _abi.DecodeArgs:
    a = _abi.DecodeArgs()
    a.B, a.nh, a.nk, a.hd, a.cap, a.ns = B, nh, nk, hd, cap, ns
    if meta is not None:
        a.meta = meta.data_ptr()
    if meta_out is not None:
        a.meta_out = meta_out.data_ptr()
    return a


def decode_workspace_size(B, nh, nk, hd, cap, ns, *, meta=None, meta_out=None) -> int:
    """Workspace bytes of decode_step (0 when the step runs as one kernel; that
    form needs meta_out distinct from meta, so pass both to decide)."""
    a = _decode_struct(B, nh, nk, hd, cap, ns, meta, meta_out)
    return int(library().swa_decode_workspace_size(ctypes.byref(a)))


def decode_launches(B, nh, nk, hd, cap, ns, *, meta=None, meta_out=None) -> int:
    """Kernels one decode_step call launches: 1 (one kernel) or 3."""
    a = _decode_struct(B, nh, nk, hd, cap, ns, meta, meta_out)
    n = int(library().swa_decode_launches(ctypes.byref(a)))
    if n == 0:
        raise SwaError(_abi.SWA_E_SHAPE, "swa_decode_launches")
    return n


def decode_step(yq, yk, yv, q_scale, pos0, meta, ring_k, ring_v, sink_k, sink_v, gate, gate_scale,
                scale: float, *, eps: float = 1e-6, theta: float = 10000.0, out=None, meta_out=None,
                workspace=None, err=None, ev_start=None, ev_stop=None, stream=None):
    """One decode token of every sequence (t = 1): prep, attention, gate and
    commit in one call (one kernel when the plan allows it); see include/swa.h.
    yq [B][nh][hd], yk / yv [B][nk][hd], gate [B][nh][hd]; the ring gets the
    row's k-hat / v and meta_out the advanced meta. Returns out [B][nh][hd]."""
    B, nh, hd = yq.shape
    nk = yk.shape[1]
    cap = ring_k.shape[2]
    ns = sink_k.shape[2] if sink_k is not None else 0
    if out is None:
        out = torch.empty_like(yq)
    if meta_out is None:
        raise ValueError("meta_out is required")
    if workspace is None:
        need = decode_workspace_size(B, nh, nk, hd, cap, ns, meta=meta, meta_out=meta_out)
        workspace = torch.empty(max(need, 1), device=yq.device, dtype=torch.uint8)
    a = _decode_struct(B, nh, nk, hd, cap, ns)
    a.scale, a.eps, a.theta = float(scale), float(eps), float(theta)
    a.yq = _ptr(yq, "yq", (B, nh, hd))
    a.yk = _ptr(yk, "yk", (B, nk, hd))
    a.yv = _ptr(yv, "yv", (B, nk, hd))
    a.q_scale = _ptr(q_scale, "q_scale", (nh, hd))
    a.pos0 = _ptr(pos0, "pos0", (B,), torch.int32)
    a.meta = _ptr(meta, "meta", (B, 4), torch.int32)
    a.ring_k = _ptr(ring_k, "ring_k", (B, nk, cap, hd))
    a.ring_v = _ptr(ring_v, "ring_v", (B, nk, cap, hd))
    a.sink_k = _ptr(sink_k, "sink_k", (B, nk, ns, hd)) if ns else 0
    a.sink_v = _ptr(sink_v, "sink_v", (B, nk, ns, hd)) if ns else 0
    a.gate = _ptr(gate, "gate", (B, nh, hd))
    a.gate_scale = _ptr(gate_scale, "gate_scale", (nh, hd))
    a.out = _ptr(out, "out", (B, nh, hd))
    a.meta_out = _ptr(meta_out, "meta_out", (B, 4), torch.int32)
    a.workspace = _ptr(workspace, "workspace", None, torch.uint8)
    a.workspace_bytes = workspace.numel()
    a.err = _ptr(err, "err", (1,), torch.int32, required=False)
    a.ev_start = ctypes.c_void_p(ev_start.cuda_event) if ev_start is not None else None
    a.ev_stop = ctypes.c_void_p(ev_stop.cuda_event) if ev_stop is not None else None
    rc = library().swa_decode_step(ctypes.byref(a), _stream(stream))
    _abi.check(rc, "swa_decode_step")
    return out


def rollback(meta: torch.Tensor, n_back: torch.Tensor, cap: int, err=None, stream=None):
    """Rewind each sequence's meta (in place) by n_back[b] rejected draft
    tokens, one token at a time as dory_o1_back does. Returns meta."""
    B = meta.shape[0]
    rc = library().swa_rollback(_ptr(meta, "meta", (B, 4), torch.int32),
                                _ptr(n_back, "n_back", (B,), torch.int32), B, int(cap),
                                _ptr(err, "err", (1,), torch.int32, required=False),
                                _stream(stream))
    _abi.check(rc, "swa_rollback")
    return meta


def _flash_struct(T, nseg, hd, nh, nk, ld, q_off, k_off, v_off, ldo, max_len, scale) -> _abi.FlashArgs:
    a = _abi.FlashArgs()
    a.T, a.nseg, a.hd, a.nh, a.nk = T, nseg, hd, nh, nk
    a.ld, a.q_off, a.k_off, a.v_off, a.ldo, a.max_len = ld, q_off, k_off, v_off, ldo, int(max_len)
    a.scale = float(scale)
    return a


def flash_workspace_size(T, nseg, hd, nh, nk, max_len) -> int:
    """Bytes of swa_flash's split-once workspace (0 for unsupported sizes)."""
    a = _flash_struct(T, nseg, hd, nh, nk, 3 * nh * hd, 0, nh * hd, (nh + nk) * hd, nh * hd, max_len, 1.0)
    return int(library().swa_flash_workspace_size(ctypes.byref(a)))


def flash(qkv: torch.Tensor, segs: torch.Tensor, *, hd: int, nh: int, nk: int, q_off: int, k_off: int,
          v_off: int, scale: float, max_len: int, out: Optional[torch.Tensor] = None, ldo: Optional[int] = None,
          err=None, ev_start=None, ev_stop=None, workspace: Optional[torch.Tensor] = None,
          stream=None) -> torch.Tensor:
    """Full-sequence attention over packed q|k|v rows (swa_flash): qkv [T][ld],
    segs [nseg][2] int32 (first row, length), every row of a segment attends
    every row of the segment. Returns out [T][ldo] (rows outside every segment
    are left as they were; a new output starts zeroed). With `workspace` (a
    uint8 CUDA tensor of at least flash_workspace_size bytes) each KV head's
    K/V rows are split into f16 hi/lo operand blocks once per call and a
    persistent kernel attends them; without it the kernel splits its own tiles
    (TF32)."""
    if qkv.dim() != 2:
        raise ValueError("qkv must be [T][ld]")
    T, ld = qkv.shape
    nseg = segs.shape[0]
    if ldo is None:
        ldo = nh * hd
    if out is None:
        out = torch.zeros(T, ldo, device=qkv.device, dtype=torch.float32)
    a = _flash_struct(T, nseg, hd, nh, nk, ld, q_off, k_off, v_off, ldo, max_len, scale)
    if workspace is not None:
        a.workspace = _ptr(workspace, "workspace", dtype=torch.uint8)
        a.workspace_bytes = workspace.numel()
    a.qkv = _ptr(qkv, "qkv", (T, ld))
    a.segs = _ptr(segs, "segs", (nseg, 2), torch.int32)
    a.out = _ptr(out, "out", (T, ldo))
    a.err = _ptr(err, "err", (1,), torch.int32, required=False)
    a.ev_start = ctypes.c_void_p(ev_start.cuda_event) if ev_start is not None else None
    a.ev_stop = ctypes.c_void_p(ev_stop.cuda_event) if ev_stop is not None else None
    _abi.check(library().swa_flash(ctypes.byref(a), _stream(stream)), "swa_flash")
    return out


class TokenPath:
    """One batch of sequences of a sealed sliding-window layer, resident on the GPU.

    Holds the ring K/V, sinks, meta, the per-head scales and the workspace;
    ``step`` runs prep + attend (+ commit) for a chunk of t rows. With host
    (CPU, ideally pinned) inputs, ``step`` copies them in, runs the kernels and
    copies the gated output back (the end-to-end call); with device inputs it
    returns the device output.
    """

    def __init__(self, *, B, t, nh, nk, hd, cap, ns, window=None, q_scale, gate_scale,
                 ring_k, ring_v, sink_k, sink_v, meta, pos0, scale=None, eps=1e-6,
                 theta=10000.0, device="cuda", num_splits=0, far=None):
        self.B, self.t, self.nh, self.nk, self.hd, self.cap, self.ns = B, t, nh, nk, hd, cap, ns
        self.scale = float(scale) if scale is not None else hd ** -0.5
        self.eps, self.theta = float(eps), float(theta)
        dev = torch.device(device)
        f32 = dict(device=dev, dtype=torch.float32)
        self.q_scale = q_scale.to(**f32).contiguous()
        self.gate_scale = gate_scale.to(**f32).contiguous()
        self.ring_k = ring_k.to(**f32).contiguous()
        self.ring_v = ring_v.to(**f32).contiguous()
        self.sink_k = sink_k.to(**f32).contiguous()
        self.sink_v = sink_v.to(**f32).contiguous()
        self.meta = meta.to(device=dev, dtype=torch.int32).contiguous()
        self.meta_next = self.meta.clone()
        self.pos0 = pos0.to(device=dev, dtype=torch.int32).contiguous()
        self.num_splits = num_splits
        self.q = torch.empty(B, t, nh, hd, **f32)
        self.k = torch.empty(B, t, nk, hd, **f32)
        self.out = torch.empty(B, t, nh, hd, **f32)
        # far field of decode steps: landmark state on the device (mz and t_hat
        # advance with every committed step)
        self.far = None
        if far is not None:
            self.far = {"m": int(far["m"]), "rect": int(far.get("rect", 0))}
            for key in ("k_tilde", "q_tilde", "mu", "mz", "t_hat"):
                self.far[key] = far[key].to(**f32).contiguous()
        # single rows without a far field and with automatic splits run as
        # decode_step (one kernel when the plan gives each (sequence, KV head) a
        # single CTA)
        self.decode = t == 1 and far is None and num_splits == 0
        need = attend_workspace_size(B, t, nh, nk, hd, cap, ns, num_splits,
                                     self.far["m"] if self.far else 0)
        if self.decode:
            need = max(need, decode_workspace_size(B, nh, nk, hd, cap, ns, meta=self.meta,
                                                   meta_out=self.meta_next))
        self.workspace = torch.empty(need, device=dev, dtype=torch.uint8)
        self.err = torch.zeros(1, device=dev, dtype=torch.int32)
        self.in_bufs = {
            "yq": torch.empty(B, t, nh, hd, **f32), "yk": torch.empty(B, t, nk, hd, **f32),
            "yv": torch.empty(B, t, nk, hd, **f32), "gate": torch.empty(B, t, nh, hd, **f32),
        }

    def step(self, yq, yk, yv, gate, *, commit: bool = True, out_host=None,
             ev_start=None, ev_stop=None, prep_events=None, stream=None, v_ready=None,
             gate_ready=None):
        """One pass of the path. commit = True writes the chunk into the ring and
        the advanced meta into ``meta_next`` (the current ``meta`` is kept, so
        repeating a step repeats the same work). Host inputs are copied in and
        the output is copied back (into ``out_host`` when given, e.g. pinned).
        ev_start / ev_stop bracket the attention kernel, prep_events (a pair of
        torch CUDA events) the prep kernel, on the step's stream. v_ready and
        gate_ready are events of device inputs still being copied in: the
        attention waits for v_ready, the merge for gate_ready."""
        host = not yq.is_cuda
        if host:
            for name, x in (("yq", yq), ("yk", yk), ("yv", yv), ("gate", gate)):
                self.in_bufs[name].copy_(x, non_blocking=True)
            yq, yk, yv, gate = (self.in_bufs[n] for n in ("yq", "yk", "yv", "gate"))
        if self.decode and commit:
            # one decode token: prep, attention, gate and commit in one call
            cur = stream if stream is not None else torch.cuda.current_stream()
            for ev in (v_ready, gate_ready):
                if ev is not None:
                    cur.wait_event(ev)
            if prep_events is not None:
                prep_events[0].record(stream)
                prep_events[1].record(stream)
            B, nh, nk, hd = self.B, self.nh, self.nk, self.hd
            decode_step(yq.view(B, nh, hd), yk.view(B, nk, hd), yv.view(B, nk, hd), self.q_scale,
                        self.pos0, self.meta, self.ring_k, self.ring_v, self.sink_k, self.sink_v,
                        gate.view(B, nh, hd), self.gate_scale, self.scale, eps=self.eps,
                        theta=self.theta, out=self.out.view(B, nh, hd), meta_out=self.meta_next,
                        workspace=self.workspace, err=self.err, ev_start=ev_start, ev_stop=ev_stop,
                        stream=stream)
            if host:
                if out_host is None:
                    return self.out.to("cpu")
                out_host.copy_(self.out, non_blocking=True)
                cur.synchronize()
                return out_host
            return self.out
        # the prep writes the ring for single rows, except with a far field:
        # that step's eviction still reads the evicted slot, so the commit does
        ring = self.t == 1 and self.far is None
        if prep_events is not None:
            prep_events[0].record(stream)
        q, k, v = prep(yq, yk, yv, None, self.q_scale, self.eps, pos0=self.pos0, theta=self.theta,
                       ring_k=self.ring_k if ring else None, ring_v=self.ring_v if ring else None,
                       q_out=self.q, k_out=self.k, copy_v=False, stream=stream)
        if prep_events is not None:
            prep_events[1].record(stream)
        if v_ready is not None:
            (stream if stream is not None else torch.cuda.current_stream()).wait_event(v_ready)
        attend(self.meta, q, k, v, self.ring_k, self.ring_v, self.sink_k, self.sink_v, gate,
               self.gate_scale, self.scale, out=self.out, workspace=self.workspace,
               commit=commit, meta_out=self.meta_next, num_splits=self.num_splits, err=self.err,
               ev_start=ev_start, ev_stop=ev_stop, far=self.far, stream=stream,
               gate_ready=gate_ready)
        if host:
            if out_host is None:
                return self.out.to("cpu")
            out_host.copy_(self.out, non_blocking=True)
            (stream if stream is not None else torch.cuda.current_stream()).synchronize()
            return out_host
        return self.out

    def capture(self):
        """Record one host-to-host step as a CUDA graph: the copies of the
        pinned inputs ``h_in`` to the device, prep, attention, merge/gate/
        commit and the copy of the output into the pinned ``h_out``. Write a
        step's inputs into ``h_in`` and call ``replay``.

        The inputs travel on a copy stream in the order the kernels need them
        (yq and yk for the prep, then yv for the attention, then the gate for
        the merge), so the later copies overlap the prep and the attention."""
        self.h_in = {n: torch.empty(tuple(b.shape), dtype=b.dtype).pin_memory()
                     for n, b in self.in_bufs.items()}
        self.h_out = torch.empty(tuple(self.out.shape), dtype=self.out.dtype).pin_memory()
        self._copy_stream = torch.cuda.Stream()
        self._arrived = {n: torch.cuda.Event() for n in ("qk", "v", "gate")}
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):           # warm-up: attributes, plans, allocations
            self._graph_body()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._graph_body()
        self.graph = g
        return g

    def _graph_body(self):
        cur, cs, ev = torch.cuda.current_stream(), self._copy_stream, self._arrived
        cs.wait_stream(cur)
        with torch.cuda.stream(cs):
            for name, mark in (("yq", None), ("yk", "qk"), ("yv", "v"), ("gate", "gate")):
                self.in_bufs[name].copy_(self.h_in[name], non_blocking=True)
                if mark:
                    ev[mark].record(cs)
        cur.wait_event(ev["qk"])
        self.step(self.in_bufs["yq"], self.in_bufs["yk"], self.in_bufs["yv"], self.in_bufs["gate"],
                  v_ready=ev["v"], gate_ready=ev["gate"])
        self.h_out.copy_(self.out, non_blocking=True)
        cur.wait_stream(cs)

    def replay(self):
        """One captured step; returns the pinned host output."""
        self.graph.replay()
        torch.cuda.current_stream().synchronize()
        return self.h_out
