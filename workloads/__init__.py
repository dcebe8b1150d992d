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
