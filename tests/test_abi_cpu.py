"""The C ABI without a GPU: the library builds, loads, exports every entry
point include/swa.h declares, and rejects bad arguments on the host before any
CUDA call (so these run on a machine with no GPU)."""
import ctypes
import os
import re

import pytest

from sliding_window_gqa_prep_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(swa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return _abi.load()


def test_header_declares_the_path(lib):
    names = declared_functions()
    for n in ("swa_prep", "swa_attend", "swa_attend_workspace_size", "swa_rope_table",
              "swa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.swa_status_string(code)
    assert b"unknown" in lib.swa_status_string(-99)
    assert b"sm_103a" in lib.swa_version()


FAKE = 0x10000  # an aligned address that is never dereferenced: checks fail first


def _prep(**kw):
    a = _abi.PrepArgs()
    a.B, a.t, a.nh, a.nk, a.hd, a.cap, a.eps = 2, 1, 8, 2, 128, 16, 1e-6
    for f in ("yq", "yk", "yv", "rope", "q_scale", "q_out", "k_out"):
        setattr(a, f, FAKE)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_prep_rejects_bad_arguments(lib):
    call = lambda a: lib.swa_prep(ctypes.byref(a), None)
    assert lib.swa_prep(None, None) == _abi.SWA_E_NULL
    assert call(_prep(yq=None)) == _abi.SWA_E_NULL
    assert call(_prep(hd=96)) == _abi.SWA_E_SHAPE
    assert call(_prep(B=0)) == _abi.SWA_E_SHAPE
    assert call(_prep(eps=-1.0)) == _abi.SWA_E_SHAPE
    assert call(_prep(yq=FAKE + 4)) == _abi.SWA_E_ALIGN
    # no table: the angles need pos0 and a positive theta
    assert call(_prep(rope=None, theta=1e4)) == _abi.SWA_E_NULL
    assert call(_prep(rope=None, pos0=FAKE, theta=0.0)) == _abi.SWA_E_SHAPE
    # ring write: both rings and pos0 needed, and only for t == 1
    assert call(_prep(ring_k=FAKE)) == _abi.SWA_E_NULL
    assert call(_prep(ring_k=FAKE, ring_v=FAKE)) == _abi.SWA_E_NULL
    assert call(_prep(t=4, ring_k=FAKE, ring_v=FAKE, pos0=FAKE)) == _abi.SWA_E_HAZARD
    assert call(_prep(cap=0, ring_k=FAKE, ring_v=FAKE, pos0=FAKE)) == _abi.SWA_E_SHAPE


def _attend(**kw):
    a = _abi.AttendArgs()
    a.B, a.t, a.nh, a.nk, a.hd, a.cap, a.ns = 2, 1, 8, 2, 128, 64, 2
    a.scale = 0.1
    for f in ("meta", "q", "k_chunk", "v_chunk", "ring_k", "ring_v", "sink_k", "sink_v", "gate",
              "gate_scale", "out", "workspace"):
        setattr(a, f, FAKE)
    a.workspace_bytes = 1 << 40
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_attend_rejects_bad_arguments(lib):
    call = lambda a: lib.swa_attend(ctypes.byref(a), None)
    assert lib.swa_attend(None, None) == _abi.SWA_E_NULL
    assert call(_attend(q=None)) == _abi.SWA_E_NULL
    assert call(_attend(sink_k=None)) == _abi.SWA_E_NULL          # ns > 0 needs sinks
    assert call(_attend(commit=1)) == _abi.SWA_E_NULL             # commit needs meta_out
    assert call(_attend(hd=100)) == _abi.SWA_E_SHAPE
    assert call(_attend(nh=9)) == _abi.SWA_E_SHAPE                # nh % nk
    assert call(_attend(nh=66)) == _abi.SWA_E_SHAPE               # 33 q heads per KV head
    assert call(_attend(cap=0)) == _abi.SWA_E_SHAPE
    assert call(_attend(ns=-1)) == _abi.SWA_E_SHAPE
    assert call(_attend(scale=float("nan"))) == _abi.SWA_E_SHAPE
    assert call(_attend(B=1 << 20, t=1024)) == _abi.SWA_E_SHAPE   # 2^33 output rows
    assert call(_attend(out=FAKE + 8)) == _abi.SWA_E_ALIGN
    assert call(_attend(workspace_bytes=16)) == _abi.SWA_E_WORKSPACE
    assert call(_attend(workspace=None)) == _abi.SWA_E_WORKSPACE
    assert call(_attend(workspace=FAKE + 16)) == _abi.SWA_E_ALIGN  # workspace wants 256 B


def test_noalloc_reports_the_errors_of_swa_attend_in_its_order(lib):
    """swa_attend_noalloc runs swa_attend's argument checks before its own size
    check, so a call that is wrong in several ways gets the same status from both."""
    noalloc = lambda a: lib.swa_attend_noalloc(ctypes.byref(a), None)
    attend = lambda a: lib.swa_attend(ctypes.byref(a), None)
    assert lib.swa_attend_noalloc(None, None) == _abi.SWA_E_NULL
    for kw in (dict(q=None), dict(q=None, hd=100), dict(q=None, B=256, t=8, nh=128, nk=32, cap=4096),
               dict(sink_k=None, hd=100), dict(commit=1, nh=9), dict(hd=100), dict(nh=9),
               dict(scale=float("inf")), dict(out=FAKE + 8), dict(out=FAKE + 8, B=256, t=8, nh=128, nk=32, cap=4096)):
        want = attend(_attend(**kw))
        assert want != _abi.SWA_OK
        assert noalloc(_attend(**kw)) == want, kw
    # valid arguments whose scratch need exceeds the fixed array: refused before any CUDA call
    big = _attend(B=256, t=8, nh=128, nk=32, hd=128, cap=4096, ns=4)
    assert lib.swa_attend_workspace_min(ctypes.byref(big)) > (16 << 20)
    assert noalloc(big) == _abi.SWA_E_WORKSPACE


def test_workspace_size_rejects_bad_sizes(lib):
    assert lib.swa_attend_workspace_size(None) == 0
    a = _attend(hd=100)
    assert lib.swa_attend_workspace_size(ctypes.byref(a)) == 0


def test_attend_rejects_shapes_past_the_grid_limits(lib):
    size = lambda **kw: lib.swa_attend_workspace_size(ctypes.byref(_attend(**kw)))
    call = lambda **kw: lib.swa_attend(ctypes.byref(_attend(**kw)), None)
    # (sequence, KV head) pairs index a grid dimension (65535), one more row for the ordering
    assert size(B=32767, nk=2) > 0
    assert size(B=32768, nk=2) == 0 and call(B=32768, nk=2) == _abi.SWA_E_SHAPE
    # row blocks of 4 rows (32 query heads per KV head, 128 query vectors) index another
    assert size(B=1, t=4 * 65535, nh=32, nk=1) > 0
    assert size(B=1, t=4 * 65535 + 1, nh=32, nk=1) == 0
    assert call(B=1, t=4 * 65535 + 1, nh=32, nk=1) == _abi.SWA_E_SHAPE


def test_rope_table_rejects_bad_arguments(lib):
    assert lib.swa_rope_table(None, FAKE, 1, 1, 64, 1e4, None) == _abi.SWA_E_NULL
    assert lib.swa_rope_table(FAKE, FAKE, 1, 1, 48, 1e4, None) == _abi.SWA_E_SHAPE
    assert lib.swa_rope_table(FAKE, FAKE, 1, 1, 64, -1.0, None) == _abi.SWA_E_SHAPE
    assert lib.swa_rope_table(FAKE + 4, FAKE, 1, 1, 64, 1e4, None) == _abi.SWA_E_ALIGN


def test_rollback_rejects_bad_arguments(lib):
    assert lib.swa_rollback(None, FAKE, 1, 8, None, None) == _abi.SWA_E_NULL
    assert lib.swa_rollback(FAKE, None, 1, 8, None, None) == _abi.SWA_E_NULL
    assert lib.swa_rollback(FAKE, FAKE, 0, 8, None, None) == _abi.SWA_E_SHAPE
    assert lib.swa_rollback(FAKE, FAKE, 1, 0, None, None) == _abi.SWA_E_SHAPE
    assert lib.swa_rollback(FAKE + 4, FAKE, 1, 8, None, None) == _abi.SWA_E_ALIGN


def _far(**kw):
    f = _abi.FarArgs()
    f.m, f.rect = 16, 0
    for k in ("k_tilde", "q_tilde", "mu", "mz", "t_hat"):
        setattr(f, k, FAKE)
    for k, v in kw.items():
        setattr(f, k, v)
    return f


def test_attend_rejects_bad_far_field_arguments(lib):
    call = lambda a: lib.swa_attend(ctypes.byref(a), None)
    for missing in ("k_tilde", "q_tilde", "mu", "mz", "t_hat"):
        f = _far(**{missing: None})
        assert call(_attend(far=ctypes.pointer(f))) == _abi.SWA_E_NULL, missing
    f = _far()
    # at most 64 rows (the pages' OB_K), even with room in the ring
    assert call(_attend(t=65, cap=128, far=ctypes.pointer(f))) == _abi.SWA_E_SHAPE
    assert lib.swa_attend_workspace_size(ctypes.byref(_attend(t=65, cap=128, far=ctypes.pointer(f)))) == 0
    assert lib.swa_attend_workspace_size(ctypes.byref(_attend(t=64, cap=128, far=ctypes.pointer(f)))) > 0
    assert call(_attend(t=8, cap=6, far=ctypes.pointer(f))) == _abi.SWA_E_SHAPE   # t <= cap
    for m in (0, 33):
        f = _far(m=m)
        assert call(_attend(far=ctypes.pointer(f))) == _abi.SWA_E_SHAPE, m
    f = _far(t_hat=FAKE + 4)
    assert call(_attend(far=ctypes.pointer(f))) == _abi.SWA_E_ALIGN
    f = _far(mz=FAKE + 2)
    assert call(_attend(far=ctypes.pointer(f))) == _abi.SWA_E_ALIGN


def test_workspace_minimum_and_split_once_blocks(lib):
    a = _attend()                                           # decode: no split-once blocks
    assert lib.swa_attend_workspace_min(ctypes.byref(a)) == lib.swa_attend_workspace_size(ctypes.byref(a))
    p = _attend(t=64, nh=8, nk=2, cap=100, ns=3)           # 256 query vectors per KV head: tcgen05
    lo = lib.swa_attend_workspace_min(ctypes.byref(p))
    hi = lib.swa_attend_workspace_size(ctypes.byref(p))
    blocks = 1 + (100 + 64 + 31) // 32                      # sink block + logical blocks
    ops = 2 * 2 * blocks * 4 * 32 * 128 * 2                 # B * nk * blocks * (K, V) x (hi, lo) x 32 x hd f16
    exps = 2 * 2 * blocks * 8                               # (e_k, e_v) per block
    order = 2 * 2 * (64 // 32) * 4                          # one int per row block (32 rows of 4 heads)
    assert hi - lo >= ops + exps + order and hi - lo < ops + exps + order + 3 * 256
    call = lambda a: lib.swa_attend(ctypes.byref(a), None)
    assert call(_attend(t=64, nh=8, nk=2, cap=100, ns=3, workspace_bytes=lo - 1)) == _abi.SWA_E_WORKSPACE
    assert lib.swa_attend_workspace_min(None) == 0


def test_workspace_grows_by_the_far_records(lib):
    a = _attend()
    base = lib.swa_attend_workspace_size(ctypes.byref(a))
    f = _far()
    a.far = ctypes.pointer(f)
    with_far = lib.swa_attend_workspace_size(ctypes.byref(a))
    need = 2 * 1 * 8 * (4 + 128) * 4                    # B * t * nh * (4 + hd) floats
    assert with_far - base >= need and with_far - base < need + 256


def _flash(**kw):
    a = _abi.FlashArgs()
    a.T, a.nseg, a.hd, a.nh, a.nk = 100, 2, 64, 8, 4
    a.ld, a.q_off, a.k_off, a.v_off, a.ldo, a.max_len = 1024, 0, 512, 768, 512, 60
    a.scale = 0.125
    for f in ("qkv", "segs", "out"):
        setattr(a, f, FAKE)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_flash_rejects_bad_arguments(lib):
    call = lambda a: lib.swa_flash(ctypes.byref(a), None)
    assert lib.swa_flash(None, None) == _abi.SWA_E_NULL
    for f in ("qkv", "segs", "out"):
        assert call(_flash(**{f: None})) == _abi.SWA_E_NULL, f
    assert call(_flash(hd=256)) == _abi.SWA_E_SHAPE               # tensor-core tiles: hd 64 or 128
    assert call(_flash(nh=9)) == _abi.SWA_E_SHAPE                 # nh % nk
    assert call(_flash(nh=132, nk=2, ld=20000, k_off=8448, v_off=8576, ldo=8448)) == _abi.SWA_E_SHAPE  # hpg 66
    assert call(_flash(nseg=0)) == _abi.SWA_E_SHAPE
    assert call(_flash(max_len=0)) == _abi.SWA_E_SHAPE
    assert call(_flash(max_len=101)) == _abi.SWA_E_SHAPE          # longer than the buffer
    assert call(_flash(v_off=800)) == _abi.SWA_E_SHAPE            # V heads past the row
    assert call(_flash(ldo=256)) == _abi.SWA_E_SHAPE              # output row too short
    assert call(_flash(scale=float("inf"))) == _abi.SWA_E_SHAPE
    assert call(_flash(nseg=70000)) == _abi.SWA_E_SHAPE           # grid z = nseg * nk
    assert call(_flash(k_off=514)) == _abi.SWA_E_ALIGN            # offsets in float4 units
    assert call(_flash(ld=1026)) == _abi.SWA_E_ALIGN
    assert call(_flash(qkv=FAKE + 4)) == _abi.SWA_E_ALIGN
    assert call(_flash(segs=FAKE + 2)) == _abi.SWA_E_ALIGN


def _up(x):
    return (x + 255) // 256 * 256


def _flash_ops_bytes(nseg, nh, nk, hd, max_len):
    """The split-once part of the flash workspace: f16 blocks of 4 x 32 x hd halves,
    two exponent ints per block, one order int per unit (row block of 128 // group
    rows), each part rounded up to 256 bytes."""
    nblk = -(-max_len // 32)
    units = nseg * nk * -(-max_len // (128 // (nh // nk)))
    return nseg * nk * nblk * 4 * 32 * hd * 2 + _up(nseg * nk * nblk * 8) + _up(units * 4)


def test_flash_workspace_size_and_checks(lib):
    a = _flash()
    need = lib.swa_flash_workspace_size(ctypes.byref(a))
    assert need == 2 * 4 * 2 * 4 * 32 * 64 * 2 + 256 + 256   # 16 blocks of 4 x 32 x hd halves, exponents, order
    assert need == _flash_ops_bytes(2, 8, 4, 64, 60)
    assert lib.swa_flash_workspace_size(None) == 0
    assert lib.swa_flash_workspace_size(ctypes.byref(_flash(hd=256))) == 0
    call = lambda a: lib.swa_flash(ctypes.byref(a), None)
    assert call(_flash(workspace=FAKE, workspace_bytes=need - 1)) == _abi.SWA_E_WORKSPACE
    assert call(_flash(workspace=FAKE + 16, workspace_bytes=need)) == _abi.SWA_E_ALIGN   # wants 256 B


def test_flash_workspace_holds_the_split_tail_records(lib):
    # 154 row blocks of 128 (one head) pass one wave of SMs (148 when no GPU is
    # visible): the size adds the tail pieces' records (128 x (hd + 4) floats each,
    # at most one per SM) and a 256-byte block of combine counters
    T = 128 * 154
    a = _flash(T=T, nseg=1, nh=1, nk=1, ld=192, q_off=0, k_off=64, v_off=128, ldo=64, max_len=T)
    need = lib.swa_flash_workspace_size(ctypes.byref(a))
    ops = _flash_ops_bytes(1, 1, 1, 64, T)
    rec = 128 * (64 + 4) * 4
    assert need > ops and (need - ops - 256) % rec == 0 and 0 < (need - ops - 256) // rec <= 152
    # one segment of 128 rows: far from a wave, no records
    b = _flash(T=128, nseg=1, nh=1, nk=1, ld=192, q_off=0, k_off=64, v_off=128, ldo=64, max_len=128)
    assert lib.swa_flash_workspace_size(ctypes.byref(b)) == _flash_ops_bytes(1, 1, 1, 64, 128)


def test_flash_split_tail_rule_over_shapes(lib):
    # the library's rule: with U units (row blocks of 128 query vectors x segments x
    # KV heads) and S SMs (148 when no GPU is visible), U >= S and 0 < U % S <= S / 2
    # give U % S tail units of S // (U % S) pieces, each with a 128 x (hd + 4)-float
    # record, plus 8 counters per tail unit
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    up = lambda x: (x + 255) // 256 * 256
    for nseg, nh, nk, hd, max_len in [(1, 1, 1, 64, 128 * 150), (1, 16, 16, 64, 9801), (3, 8, 2, 128, 1000),
                                      (2, 32, 1, 64, 308), (1, 4, 4, 128, 128 * 37), (5, 2, 1, 64, 128 * 31)]:
        rows = 128 // (nh // nk)
        units = -(-max_len // rows) * nseg * nk
        tail = units % sms if units >= sms else 0
        extra = 0
        if 0 < 2 * tail <= sms:
            extra = up(tail * (sms // tail) * 128 * (hd + 4) * 4) + up(tail * 8 * 4)
        ld = (nh + 2 * nk) * hd
        a = _flash(T=max_len * nseg, nseg=nseg, nh=nh, nk=nk, hd=hd, ld=ld, q_off=0, k_off=nh * hd,
                   v_off=(nh + nk) * hd, ldo=nh * hd, max_len=max_len)
        ops = _flash_ops_bytes(nseg, nh, nk, hd, max_len)
        assert lib.swa_flash_workspace_size(ctypes.byref(a)) == ops + extra, (nseg, nh, nk, hd, max_len)


def _decode(**kw):
    a = _abi.DecodeArgs()
    a.B, a.nh, a.nk, a.hd, a.cap, a.ns = 2, 8, 2, 128, 64, 2
    a.scale, a.eps, a.theta = 0.1, 1e-6, 1e4
    for f in ("yq", "yk", "yv", "q_scale", "pos0", "meta", "ring_k", "ring_v", "sink_k", "sink_v",
              "gate", "gate_scale", "out", "meta_out"):
        setattr(a, f, FAKE)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_decode_step_rejects_bad_arguments(lib):
    call = lambda a: lib.swa_decode_step(ctypes.byref(a), None)
    assert lib.swa_decode_step(None, None) == _abi.SWA_E_NULL
    for f in ("yq", "yk", "yv", "q_scale", "pos0", "meta", "ring_k", "gate", "out", "meta_out"):
        assert call(_decode(**{f: None})) == _abi.SWA_E_NULL, f
    assert call(_decode(sink_k=None)) == _abi.SWA_E_NULL           # ns > 0 needs sinks
    assert call(_decode(hd=96)) == _abi.SWA_E_SHAPE
    assert call(_decode(nh=9)) == _abi.SWA_E_SHAPE
    assert call(_decode(nh=66)) == _abi.SWA_E_SHAPE                 # 33 query heads per KV head
    assert call(_decode(eps=-1.0)) == _abi.SWA_E_SHAPE
    assert call(_decode(theta=0.0)) == _abi.SWA_E_SHAPE
    assert call(_decode(scale=float("inf"))) == _abi.SWA_E_SHAPE
    assert call(_decode(out=FAKE + 8)) == _abi.SWA_E_ALIGN
    assert lib.swa_decode_workspace_size(None) == 0
    assert lib.swa_decode_launches(None) == 0
    assert lib.swa_decode_launches(ctypes.byref(_decode(hd=96))) == 0
