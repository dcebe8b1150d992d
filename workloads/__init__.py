"""Seeded synthetic inputs for the sliding-window GQA token path.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It only draws random numbers and lays out ring state; it holds none of
the method's arithmetic (no RoPE, no norms, no scores, no softmax).

Ring state follows the per-sequence meta of the sealed-layer attention page
(cortiq-engine 0.8.79, src/gpu_metal/o1c_msl.metal, header comment and
``o1c_meta``): ``win_len | win_head | far_len | window``. A ring that has grown
from position 0 holds ``win_len = min(pos0, window)`` keys and its oldest key
sits in slot ``(pos0 - win_len) % window``; the generator builds exactly that
state so that ``win_head`` and ``pos0`` agree.

Every tensor is float32 on the CPU, drawn from ``torch.Generator('cpu')``
seeded with the workload's seed, in the fixed order documented in
``make_inputs``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int          # sequences
    t: int          # chunk rows per sequence
    nh: int         # query heads
    nk: int         # KV heads
    hd: int         # head dim
    window: int     # window W (== ring capacity in every named workload)
    cap: int        # ring capacity
    ns: int         # sink keys per (sequence, KV head)
    seed: int
    pos_mode: str   # how pos0 / win_len are drawn (see make_meta)
    pos_lo: int = 0
    pos_hi: int = 0
    theta: float = 10000.0
    eps: float = 1e-6
    scale: Optional[float] = None   # None -> 1/sqrt(hd)
    far_m: int = 0                  # landmarks of a far field (decode rows), 0 = none

    @property
    def hpg(self) -> int:
        return self.nh // self.nk

    @property
    def score_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.hd)


# The five workloads of the method's token path (decode token, batched decode,
# speculative verify, prompt chunk, long-window decode), and batched decode with
# the far field of the sealed layer.
WORKLOADS: Dict[str, Workload] = {
    "tiny_decode": Workload("tiny_decode", B=1, t=1, nh=8, nk=2, hd=64, window=32, cap=32,
                            ns=0, seed=0, pos_mode="fixed", pos_lo=100),
    "batched_decode": Workload("batched_decode", B=64, t=1, nh=16, nk=4, hd=128, window=4096,
                               cap=4096, ns=4, seed=1, pos_mode="full", pos_lo=4096,
                               pos_hi=20000, scale=1.0 / math.sqrt(128.0)),
    "spec_verify": Workload("spec_verify", B=128, t=8, nh=32, nk=8, hd=128, window=2048,
                            cap=2048, ns=4, seed=2, pos_mode="partial", pos_lo=1, pos_hi=2048),
    "prompt_chunk": Workload("prompt_chunk", B=4, t=512, nh=32, nk=8, hd=128, window=1024,
                             cap=1024, ns=4, seed=3, pos_mode="prompt", pos_lo=0, pos_hi=3000),
    "long_decode": Workload("long_decode", B=16, t=1, nh=8, nk=2, hd=256, window=32768,
                            cap=32768, ns=8, seed=4, pos_mode="full", pos_lo=32768,
                            pos_hi=131072),
    # batched_decode with the sealed layer's far field: 32 landmarks per query head
    "batched_decode_far": Workload("batched_decode_far", B=64, t=1, nh=16, nk=4, hd=128,
                                   window=4096, cap=4096, ns=4, seed=5, pos_mode="full",
                                   pos_lo=4096, pos_hi=20000, scale=1.0 / math.sqrt(128.0),
                                   far_m=32),
    # spec_verify with the far field: 32 landmarks per query head
    "spec_verify_far": Workload("spec_verify_far", B=128, t=8, nh=32, nk=8, hd=128, window=2048,
                                cap=2048, ns=4, seed=6, pos_mode="partial", pos_lo=1, pos_hi=2048,
                                far_m=32),
}


def make_meta(w: Workload, g: torch.Generator):
    """Draw pos0[B] and build meta[B][4] = (win_len, win_head, far_len, window).

    pos_mode:
      fixed   -- every sequence at pos0 = pos_lo
      full    -- pos0 ~ U[pos_lo, pos_hi) (ring full and wrapped, random head)
      partial -- win_len ~ U[pos_lo, pos_hi] inclusive with pos0 = win_len, head 0;
                 sequence 0 is forced full: pos0 ~ U[W, 4W), win_len = W
      prompt  -- sequence 0 at pos0 = 0 (empty ring), the rest pos0 ~ U[pos_lo, pos_hi]
    far_len counts keys that left the window (pos0 - win_len).
    """
    W = w.window
    if w.pos_mode == "fixed":
        pos0 = torch.full((w.B,), w.pos_lo, dtype=torch.int64)
    elif w.pos_mode == "full":
        pos0 = torch.randint(w.pos_lo, w.pos_hi, (w.B,), generator=g, dtype=torch.int64)
    elif w.pos_mode == "partial":
        pos0 = torch.randint(w.pos_lo, w.pos_hi + 1, (w.B,), generator=g, dtype=torch.int64)
        full0 = torch.randint(W, 4 * W, (1,), generator=g, dtype=torch.int64)
        pos0[0] = full0[0]
    elif w.pos_mode == "prompt":
        pos0 = torch.randint(w.pos_lo, w.pos_hi + 1, (w.B,), generator=g, dtype=torch.int64)
        pos0[0] = 0
    else:
        raise ValueError(w.pos_mode)
    win_len = torch.clamp(pos0, max=W)
    win_head = (pos0 - win_len) % W
    far_len = pos0 - win_len
    meta = torch.stack([win_len, win_head, far_len, torch.full_like(pos0, W)], dim=1)
    return pos0, meta


def make_inputs(w: Workload, seed: Optional[int] = None, batch: Optional[int] = None) -> dict:
    """All inputs of one step of the token path, as CPU float32 / int64 tensors.

    Draw order (fixed): pos0/meta, yq, yk, yv, gate, q_scale, gate_scale,
    ring_k, ring_v, sink_k, sink_v.
      yq [B][t][nh][hd], yk/yv [B][t][nk][hd], gate [B][t][nh][hd]  ~ N(0, 1)
      q_scale [nh][hd] ~ U(0.5, 1.5), gate_scale [nh][hd] ~ N(0, 1)
      ring_k/ring_v [B][nk][cap][hd] ~ N(0, 1), sink_k/sink_v [B][nk][ns][hd] ~ N(0, 1)
    ``batch`` (optional) overrides B, keeping everything else (used to draw a
    bounded sample of a large workload).
    """
    if batch is not None:
        w = dataclasses.replace(w, B=batch)
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    pos0, meta = make_meta(w, g)
    B, t, nh, nk, hd = w.B, w.t, w.nh, w.nk, w.hd
    out = {
        "pos0": pos0,
        "meta": meta,
        "yq": torch.randn(B, t, nh, hd, generator=g),
        "yk": torch.randn(B, t, nk, hd, generator=g),
        "yv": torch.randn(B, t, nk, hd, generator=g),
        "gate": torch.randn(B, t, nh, hd, generator=g),
        "q_scale": torch.rand(nh, hd, generator=g) + 0.5,
        "gate_scale": torch.randn(nh, hd, generator=g),
        "ring_k": torch.randn(B, nk, w.cap, hd, generator=g),
        "ring_v": torch.randn(B, nk, w.cap, hd, generator=g),
        "sink_k": torch.randn(B, nk, w.ns, hd, generator=g),
        "sink_v": torch.randn(B, nk, w.ns, hd, generator=g),
    }
    if w.far_m:
        # far field state (drawn after everything above): landmark keys and
        # queries ~ N(0, 1); mu = identity + N(0, 0.02^2); per landmark a
        # running max ~ N(0, 1), a mass ~ U(1, 50) and a numerator ~ N(0, 1).
        # Sequences that have evicted nothing yet (far_len = 0) hold the empty
        # state: max -inf, mass 0, numerator 0.
        m = w.far_m
        mx = torch.randn(B, nh, m, generator=g)
        z = torch.rand(B, nh, m, generator=g) * 49.0 + 1.0
        far = {
            "m": m, "rect": 0,
            "k_tilde": torch.randn(B, nk, m, hd, generator=g),
            "q_tilde": torch.randn(B, nh, m, hd, generator=g),
            "mu": torch.eye(m).expand(B, nh, m, m) + 0.02 * torch.randn(B, nh, m, m, generator=g),
            "t_hat": torch.randn(B, nh, m, hd, generator=g),
        }
        empty = (meta[:, 2] == 0).view(B, 1, 1)
        mx = torch.where(empty, torch.full_like(mx, -math.inf), mx)
        z = torch.where(empty, torch.zeros_like(z), z)
        far["t_hat"] = torch.where(empty.unsqueeze(-1), torch.zeros_like(far["t_hat"]), far["t_hat"])
        far["mz"] = torch.cat([mx, z], dim=2).contiguous()
        far["mu"] = far["mu"].contiguous()
        out["far"] = far
    return out


def _seq_pos0(w: Workload, b: int, g: torch.Generator) -> int:
    """pos0 of global sequence b, by the rules of make_meta."""
    W = w.window
    if w.pos_mode == "fixed":
        return w.pos_lo
    if w.pos_mode == "full":
        return int(torch.randint(w.pos_lo, w.pos_hi, (1,), generator=g)[0])
    if w.pos_mode == "partial":
        if b == 0:
            return int(torch.randint(W, 4 * W, (1,), generator=g)[0])
        return int(torch.randint(w.pos_lo, w.pos_hi + 1, (1,), generator=g)[0])
    if w.pos_mode == "prompt":
        return 0 if b == 0 else int(torch.randint(w.pos_lo, w.pos_hi + 1, (1,), generator=g)[0])
    raise ValueError(w.pos_mode)


def make_shard_inputs(w: Workload, global_B: int, seqs, seed: Optional[int] = None) -> dict:
    """Inputs of sequences ``seqs`` of a batch of ``global_B`` sequences with the
    shapes of ``w``, each sequence drawn from a generator of its own, so that a
    sequence's inputs are the same whichever shard (rank) holds it.

    The shared tensors q_scale, gate_scale come from ``Generator(seed)``;
    sequence b draws, from ``Generator(seed * 1000003 + 1 + b)``, its pos0 (the
    rules of make_meta, by global index), then yq, yk, yv, gate, ring_k, ring_v,
    sink_k, sink_v with the distributions of make_inputs (and the far field
    state when ``w.far_m``). Returns the layout of make_inputs for B = len(seqs).
    """
    seqs = list(seqs)
    if any(b < 0 or b >= global_B for b in seqs):
        raise ValueError("sequence index outside the batch")
    base = w.seed if seed is None else seed
    g0 = torch.Generator(device="cpu")
    g0.manual_seed(base)
    t, nh, nk, hd, W = w.t, w.nh, w.nk, w.hd, w.window
    q_scale = torch.rand(nh, hd, generator=g0) + 0.5
    gate_scale = torch.randn(nh, hd, generator=g0)
    parts = {k: [] for k in ("yq", "yk", "yv", "gate", "ring_k", "ring_v", "sink_k", "sink_v")}
    far_parts = {k: [] for k in ("mx", "z", "k_tilde", "q_tilde", "mu", "t_hat")}
    pos = []
    for b in seqs:
        g = torch.Generator(device="cpu")
        g.manual_seed(base * 1000003 + 1 + b)
        pos.append(_seq_pos0(w, b, g))
        parts["yq"].append(torch.randn(1, t, nh, hd, generator=g))
        parts["yk"].append(torch.randn(1, t, nk, hd, generator=g))
        parts["yv"].append(torch.randn(1, t, nk, hd, generator=g))
        parts["gate"].append(torch.randn(1, t, nh, hd, generator=g))
        parts["ring_k"].append(torch.randn(1, nk, w.cap, hd, generator=g))
        parts["ring_v"].append(torch.randn(1, nk, w.cap, hd, generator=g))
        parts["sink_k"].append(torch.randn(1, nk, w.ns, hd, generator=g))
        parts["sink_v"].append(torch.randn(1, nk, w.ns, hd, generator=g))
        if w.far_m:
            m = w.far_m
            far_parts["mx"].append(torch.randn(1, nh, m, generator=g))
            far_parts["z"].append(torch.rand(1, nh, m, generator=g) * 49.0 + 1.0)
            far_parts["k_tilde"].append(torch.randn(1, nk, m, hd, generator=g))
            far_parts["q_tilde"].append(torch.randn(1, nh, m, hd, generator=g))
            far_parts["mu"].append(torch.eye(m).expand(1, nh, m, m)
                                   + 0.02 * torch.randn(1, nh, m, m, generator=g))
            far_parts["t_hat"].append(torch.randn(1, nh, m, hd, generator=g))
    pos0 = torch.tensor(pos, dtype=torch.int64)
    win_len = torch.clamp(pos0, max=W)
    meta = torch.stack([win_len, (pos0 - win_len) % W, pos0 - win_len, torch.full_like(pos0, W)], dim=1)
    out = {"pos0": pos0, "meta": meta, "q_scale": q_scale, "gate_scale": gate_scale}
    for k, v in parts.items():
        out[k] = torch.cat(v, dim=0)
    if w.far_m:
        B = len(seqs)
        f = {k: torch.cat(v, dim=0) for k, v in far_parts.items()}
        empty = (meta[:, 2] == 0).view(B, 1, 1)
        mx = torch.where(empty, torch.full_like(f["mx"], -math.inf), f["mx"])
        z = torch.where(empty, torch.zeros_like(f["z"]), f["z"])
        t_hat = torch.where(empty.unsqueeze(-1), torch.zeros_like(f["t_hat"]), f["t_hat"])
        out["far"] = {"m": w.far_m, "rect": 0, "k_tilde": f["k_tilde"], "q_tilde": f["q_tilde"],
                      "mu": f["mu"].contiguous(), "t_hat": t_hat,
                      "mz": torch.cat([mx, z], dim=2).contiguous()}
    return out


def custom(name="custom", **kw) -> Workload:
    """A workload with arbitrary shapes (parity cases, edge cases)."""
    base = dict(B=1, t=1, nh=4, nk=1, hd=64, window=16, cap=16, ns=0, seed=0,
                pos_mode="fixed", pos_lo=0)
    base.update(kw)
    return Workload(name, **base)


def kv_keys_and_bytes(w: Workload, meta) -> tuple:
    """Attended KV-keys and algorithmic KV bytes of one call (a measurement
    definition, not the method's arithmetic).

    keys  = sum over (sequence, row, KV head) of ns + min(window, win_len + i + 1)
    bytes = sum over (sequence, KV head) of the distinct keys the chunk reads,
            ns + min(win_len + t, window + t - 1), times 2 * hd * 4 bytes (K and V).
    """
    keys = 0
    distinct = 0
    for b in range(w.B):
        L = int(meta[b][0])
        W = int(meta[b][3])
        for i in range(w.t):
            keys += w.ns + min(W, L + i + 1)
        distinct += w.ns + min(L + w.t, W + w.t - 1)
    return keys * w.nk, distinct * w.nk * 2 * w.hd * 4


# ---------------------------------------------------------------------------
# Full-sequence attention over packed q|k|v rows (the second workload,
# "egemma2_msl.metal" eg_flash64 / eg_flash_staged: a vision tower's patch
# sequence with head dim 64). A row holds [pad | q heads | k heads | v heads |
# pad]; segments are (first row, length). qkv ~ N(0, 1), drawn in one call.
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class FlashWorkload:
    name: str
    segs: tuple      # ((first row, length), ...)
    T: int           # rows of the packed buffer
    nh: int          # query heads
    nk: int          # KV heads
    hd: int          # head dim
    seed: int
    scale: Optional[float] = None   # None -> 1/sqrt(hd)
    pad: int = 0                     # floats before the q heads and after the v heads (multiple of 4)

    @property
    def group(self) -> int:
        return self.nh // self.nk

    @property
    def q_off(self) -> int:
        return self.pad

    @property
    def k_off(self) -> int:
        return self.pad + self.nh * self.hd

    @property
    def v_off(self) -> int:
        return self.k_off + self.nk * self.hd

    @property
    def ld(self) -> int:
        return self.v_off + self.nk * self.hd + self.pad

    @property
    def max_len(self) -> int:
        return max(1, max(n for _, n in self.segs))

    @property
    def score_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.hd)


# one vision-tower image: 99 x 99 = 9801 patches, 16 heads of 64
FLASH_WORKLOADS: Dict[str, FlashWorkload] = {
    "vision_flash": FlashWorkload("vision_flash", segs=((0, 9801),), T=9801, nh=16, nk=16, hd=64, seed=7),
}


def make_flash_inputs(w: FlashWorkload) -> Dict[str, torch.Tensor]:
    g = torch.Generator().manual_seed(w.seed)
    return {"qkv": torch.randn(w.T, w.ld, generator=g),
            "segs": torch.tensor([list(s) for s in w.segs], dtype=torch.int32).reshape(len(w.segs), 2)}


def flash_keys_and_flops(w: FlashWorkload) -> tuple:
    """Attended keys of one call counted per (query row, KV head) as the token
    path counts them (each serves nh / nk query heads), and the useful flops
    (4 * hd per (query row, query head, key): the score and the value sum); a
    measurement definition."""
    pairs = sum(n * n for _, n in w.segs)
    return pairs * w.nk, 4 * w.hd * pairs * w.nh
