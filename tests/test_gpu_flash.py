"""Parity of swa_flash (full-sequence attention over packed q|k|v rows, on the
tensor cores: f16 hi/lo operand blocks split once per call with a workspace, 3xTF32
split in the kernel without one) with the CPU oracle, through the C ABI on the GPU.

Floating point: max_abs <= 2e-5 and max_abs / max|oracle| <= 1e-4 per tensor.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import sliding_window_gqa_prep_gb300 as swa
from swa_harness import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a GPU")
    yield


def _run(w, segs_dev=None, out=None, err=None, split_once=False, ws_bytes=None):
    inp = workloads.make_flash_inputs(w)
    qkv = inp["qkv"].cuda()
    segs = (segs_dev if segs_dev is not None else inp["segs"]).cuda()
    ws = None
    if split_once:
        n = ws_bytes or swa.flash_workspace_size(w.T, len(w.segs), w.hd, w.nh, w.nk, w.max_len)
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")      # NaN bit patterns
    res = swa.flash(qkv, segs, hd=w.hd, nh=w.nh, nk=w.nk, q_off=w.q_off, k_off=w.k_off, v_off=w.v_off,
                    scale=w.score_scale, max_len=w.max_len, out=out, err=err, workspace=ws)
    torch.cuda.synchronize()
    return inp, res.cpu().numpy()


def _oracle(w, inp, segs=None):
    return oracle.flash_attention(inp["qkv"].numpy(), segs if segs is not None else w.segs, w.hd, w.nh, w.group,
                                  w.q_off, w.k_off, w.v_off, w.score_scale)


FLASH_CASES = [
    # group 1 (128 rows per CTA): a one-row segment, exactly 128 rows, ragged tails
    dict(segs=((0, 1), (1, 37), (40, 128), (170, 300)), T=480, nh=4, nk=4, hd=64, seed=1),
    # group 4 (32 rows per CTA), hd 128, offsets inside a padded row
    dict(segs=((3, 200), (210, 33)), T=250, nh=8, nk=2, hd=128, seed=2, pad=8),
    # group 6 (21 rows = 126 of 128 query slots per CTA)
    dict(segs=((0, 90), (90, 64)), T=160, nh=12, nk=2, hd=64, seed=3, pad=4),
    # a sharp softmax (scores of several units), exercising the lazy running max
    dict(segs=((0, 257),), T=257, nh=2, nk=1, hd=128, seed=4, scale=0.5),
]


@pytest.mark.parametrize("split_once", [False, True])
@pytest.mark.parametrize("kw", FLASH_CASES)
def test_flash_matches_oracle(kw, split_once):
    """Both forms: K/V split in the attention kernel, and split once per call into a
    workspace (poisoned with NaN bit patterns first)."""
    w = workloads.FlashWorkload("case", **kw)
    inp, got = _run(w, split_once=split_once)
    ref = _oracle(w, inp)
    rows = np.concatenate([np.arange(s0, s0 + n) for s0, n in w.segs])
    assert_close(got[rows], ref[rows], "flash out")
    outside = np.setdiff1d(np.arange(w.T), rows)
    assert not got[outside].any()                       # rows outside every segment untouched


@pytest.mark.parametrize("kw", FLASH_CASES[:2])
def test_flash_split_once_is_deterministic(kw):
    """The split-once form gives the same bits on every call (the unit order is a
    stable sort), and agrees with the in-kernel TF32 form within the tolerance."""
    w = workloads.FlashWorkload("case", **kw)
    _, a = _run(w, split_once=True)
    _, b = _run(w, split_once=True)
    np.testing.assert_array_equal(a, b)
    _, c = _run(w)
    assert_close(a, c, "f16 split-once vs TF32")


def _split_tail(w, sms):
    """The (tail, pieces) of the launch: with at least one full wave of one-CTA-per-SM
    units (row block x segment x KV head) and a remainder of at most half a wave,
    the last `tail` units of the launch run as sms // tail key ranges each."""
    n_rb = -(-w.max_len // (128 // w.group))
    units = n_rb * len(w.segs) * w.nk
    tail = units % sms if units >= sms else 0
    return (tail, sms // tail) if 0 < 2 * tail <= sms else (0, 1)


def _tail_units(w, tail):
    """The units the launch tail cuts into pieces: the last `tail` of the order, units
    (index (segment * nk + g) * n_rb + rb) by tile count, longest first, then index."""
    rows = 128 // w.group
    n_rb = -(-w.max_len // rows)
    units = n_rb * len(w.segs) * w.nk
    def tiles(u):
        n = w.segs[u // n_rb // w.nk][1]
        return -(-n // 32) if (u % n_rb) * rows < n else 0
    return sorted(range(units), key=lambda u: (-tiles(u), u))[units - tail:]


def _tail_bytes(w, tail, q):
    up = lambda x: -(-x // 256) * 256
    return up(tail * q * 128 * (w.hd + 4) * 4) + up(tail * 8 * 4)


def _tail_cells(w, sms, tail):
    """(row, head) of every output the tail units write."""
    rows = 128 // w.group
    n_rb = -(-w.max_len // rows)
    cells = []
    for u in _tail_units(w, tail):
        rb, bg = u % n_rb, u // n_rb
        (s0, n), g = w.segs[bg // w.nk], bg % w.nk
        for r in range(rb * rows, min(rb * rows + rows, n)):
            cells += [(s0 + r, h) for h in range(g * w.group, (g + 1) * w.group)]
    return cells


@pytest.mark.parametrize("shape", ["one_head", "empty_pieces"])
def test_flash_split_launch_tail_matches_oracle(shape):
    """Two units past a whole round of the persistent CTAs: each is cut into sms // 2
    key ranges whose records the last piece combines. "one_head": one segment of
    (sms + 2) row blocks of 128. "empty_pieces": 32 query heads per KV head (4 rows per
    unit) over two segments of sms // 2 + 1 row blocks each, so the tail units have 10
    tiles for sms // 2 pieces and most pieces hold no key."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if shape == "one_head":
        T = 128 * (sms + 2)
        w = workloads.FlashWorkload("case", segs=((0, T),), T=T, nh=1, nk=1, hd=64, seed=8)
    else:
        n0 = 4 * (sms // 2 + 1)
        w = workloads.FlashWorkload("case", segs=((0, n0), (n0, n0 - 3)), T=2 * n0 - 3, nh=32, nk=1, hd=64, seed=9)
    tail, q = _split_tail(w, sms)
    assert tail == 2 and q == sms // 2
    inp, got = _run(w, split_once=True)
    # the same kernel without room for the tail's records: never split
    full = swa.flash_workspace_size(w.T, len(w.segs), w.hd, w.nh, w.nk, w.max_len)
    _, plain = _run(w, split_once=True, ws_bytes=full - _tail_bytes(w, tail, q))
    cells = _tail_cells(w, sms, tail)
    qkv = inp["qkv"].numpy()
    seg_of = lambda r: next((s0, n) for s0, n in w.segs if s0 <= r < s0 + n)
    ref = np.stack([oracle.flash_row(qkv, seg_of(r)[0], seg_of(r)[1], r - seg_of(r)[0], h, w.hd, w.group,
                                     w.q_off, w.k_off, w.v_off, w.score_scale) for r, h in cells])
    gpu = np.stack([got[r, h * w.hd:(h + 1) * w.hd] for r, h in cells])
    assert_close(gpu, ref, "split tail out")
    rows = np.concatenate([np.arange(s0, s0 + n) for s0, n in w.segs])
    assert_close(got[rows], plain[rows], "split launch vs unsplit")
    # every other output comes from a whole unit: bit-identical to the unsplit kernel
    mask = np.ones(got.shape, dtype=bool)
    for r, h in cells:
        mask[r, h * w.hd:(h + 1) * w.hd] = False
    np.testing.assert_array_equal(got[mask], plain[mask])


def test_flash_skips_bad_and_empty_segments_and_reports_them():
    w = workloads.FlashWorkload("case", segs=((0, 50), (50, 0), (60, 40)), T=100, nh=4, nk=2, hd=64, seed=5)
    bad = torch.tensor([[0, 50], [50, 0], [60, 41]], dtype=torch.int32)   # the last reaches row 101
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((w.T, w.nh * w.hd), 7.0, device="cuda")
    inp, got = _run(w, segs_dev=bad, out=out, err=err, split_once=True)
    assert int(err.item()) & 4                             # SWA_DERR_SEGMENT
    ref = _oracle(w, inp, segs=[(0, 50)])
    assert_close(got[0:50], ref[0:50], "flash out")
    assert np.all(got[50:] == 7.0)                         # the empty and the bad segment wrote nothing


def test_flash_full_size_workload_sampled():
    """The benchmark's workload (9801 patches, 16 heads of 64) in the launch the
    bench times, compared with the oracle on sampled rows."""
    w = workloads.FLASH_WORKLOADS["vision_flash"]
    inp, got = _run(w, split_once=True)
    qkv = inp["qkv"].numpy()
    rng = np.random.default_rng(11)
    picks = [(0, 0), (w.T - 1, w.nh - 1)] + [(int(rng.integers(w.T)), int(rng.integers(w.nh))) for _ in range(22)]
    ref = np.stack([oracle.flash_row(qkv, 0, w.T, r, h, w.hd, w.group, w.q_off, w.k_off, w.v_off, w.score_scale)
                    for r, h in picks])
    gpu = np.stack([got[r, h * w.hd:(h + 1) * w.hd] for r, h in picks])
    assert_close(gpu, ref, "flash sampled out")
    assert np.all(np.isfinite(got))
