#!/usr/bin/env python
"""Throughput of the sliding-window GQA token path on GB300: one JSON line.

A step is one pass of the whole path over one batch resident in HBM: prep
(RoPE with in-kernel angles, unit heads, query scale, ring write for t == 1),
the split-KV attention, the merge with the sigmoid gate, and the commit of the
chunk into the ring with the advanced meta written to a second meta buffer (so
every step repeats the same work on the same state). The end-to-end figure
(e2e) replays the same step captured as a CUDA graph together with the copy of
the step's inputs from pinned host memory and of its output back.

Metric: attended KV-keys/s = sum over (sequence, row, KV head) of
ns + min(window, win_len + row + 1), per second, over all GPUs. Also reported:
the algorithmic KV-read bandwidth (each distinct K/V byte of a
(sequence, KV head) once per step) and its fraction of the measured HBM peak.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       [--impl reference]
Under torchrun the batch has world x B sequences and every rank runs its shard
of B sequences on its own GPU (no collective on the data path; weak scaling);
rank 0 prints the line.
"""
from __future__ import annotations

import os

# Each oracle worker process is single-threaded (one per host core; see oracle_pool).
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import dataclasses  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

DEFAULT_WORKLOAD = "batched_decode"
PROFILE_DIR = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "sliding_window_gqa_prep_gb300", "csrc")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(workloads.WORKLOADS) + list(workloads.FLASH_WORKLOADS))
    ap.add_argument("--impl", default="swa", choices=["swa", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's sequence count (small profiling cases)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# measurement definitions
# ---------------------------------------------------------------------------
def keys_and_bytes(w, meta):
    return workloads.kv_keys_and_bytes(w, meta)


def attention_path(w):
    """Which attention kernel a workload's row blocks take (the library's
    planner rule, hd <= 128 for the tensor-core paths): >= 128 query vectors per
    KV head -> tcgen05 prompt kernel; >= 64 -> mma.sync prompt kernel; <= 8
    query vectors per row block -> decode kernel; else the verify kernel."""
    if w.hd <= 128 and w.t * w.hpg >= 128:
        return "prompt_tc"
    if w.hd <= 128 and w.t * w.hpg >= 64:
        return "prompt"
    rows = max(1, min(w.t, 32 // w.hpg))
    nq = 4
    while nq < rows * w.hpg:
        nq *= 2
    return "decode" if nq <= 8 else "verify"


def dominant_kernel(w):
    """The attention kernel a workload runs and its source file."""
    path = attention_path(w)
    name = {"decode": "attend_decode_kernel", "verify": "attend_verify_kernel",
            "prompt": "attend_prompt_kernel", "prompt_tc": "attend_prompt_h16_kernel"}[path]
    src = {"decode": "swa_decode.cu", "verify": "swa_verify.cu", "prompt": "swa_prompt.cu",
           "prompt_tc": "swa_prompt_h16.cu"}[path]
    return name, os.path.join(CSRC, src)


# the HBM figure the method's bandwidth target is stated against (GB300 HBM3e, nominal)
NOMINAL_HBM_GBS = 8000.0


def rank_inputs(w, rank, world):
    """The inputs rank `rank` of `world` works on: its shard (dist.shard_sequences)
    of one batch of world x B sequences with the workload's shapes, each sequence
    drawn from its own generator (workloads.make_shard_inputs), so the per-GPU
    work is the workload's B sequences at every world size (weak scaling)."""
    from sliding_window_gqa_prep_gb300.dist import shard_sequences
    global_b = world * w.B
    return workloads.make_shard_inputs(w, global_b, shard_sequences(global_b, rank, world))


def peaks():
    """Roofline denominators: measured HBM copy GB/s and bf16 TFLOP/s (or the
    fallback), the FP32 CUDA-core peak derived from unit counts and the max SM
    clock (152 SMs x 128 FMA/clk x 2 flop), and the TF32 tensor peak as the
    measured bf16 peak x the nominal TF32/bf16 ratio (1.1 / 2.25)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        hbm, bf16, kind = float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
        mhz = float(d.get("sm_max_mhz", 2070.0))
    else:
        hbm, bf16, kind, mhz = 6800.0, 1900.0, "fallback", 2070.0
    fp32 = 152 * 128 * 2 * mhz * 1e6 / 1e12
    return {"hbm_gbs": hbm, "bf16_tflops": bf16, "tf32_tflops": bf16 * 1.1 / 2.25,
            "fp32_tflops": fp32, "kind": kind}


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(w, kernel=None):
    """DRAM bytes per launch of the workload's attention kernel (or `kernel`, a
    kernel of the same source file) from the committed ncu summary, if it was
    taken on the current kernel source."""
    name, src = dominant_kernel(w)
    kernel = kernel or name
    path = os.path.join(PROFILE_DIR, f"{kernel}_{w.name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch\s*[:=]\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256_16\s*[:=]\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != source_hash(src):
        return None
    return float(m.group(1))


class _Nvml:
    """The few read-only NVML queries the clock record needs, through ctypes on
    the driver's libnvidia-ml (no Python package required)."""
    SM = 0x1                                   # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        try:                                   # the same GPU as the CUDA device, by UUID
            uuid = "GPU-" + str(torch.cuda.get_device_properties(cuda_index).uuid)
            ok = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            idx = int(vis.split(",")[cuda_index]) if vis else cuda_index
            if self.lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h)) != 0:
                raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        c = self.c
        sm, smax, mw, rs = c.c_uint(), c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, c.byref(sm)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, c.byref(smax))
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(mw))
        self.reasons_fn(self.h, c.byref(rs))
        return (float(sm.value), float(smax.value), mw.value / 1000.0,
                [n for bit, n in self.REASONS.items() if rs.value & bit])


class ClockSampler:
    """SM clock, power and throttle reasons sampled during the timed regions.

    A background thread polls NVML every 2 ms between start() and stop() (the
    calls are read-only and release the interpreter lock), plus one sample at
    each mark() taken right after a timed region's work is enqueued, when the
    GPU is certainly busy; so even a region of a few milliseconds has samples.
    Without NVML it falls back to ``nvidia-smi -lms 100``."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        import threading
        self.local_rank = local_rank
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.index = vis.split(",")[local_rank] if vis else str(local_rank)
        self.rows = []
        self.lock = threading.Lock()
        self.stop_ev = threading.Event()
        self.thread = None
        self.proc = None
        self.file = None
        self.source = None
        try:
            self.nvml = _Nvml(local_rank)
        except (OSError, AttributeError):
            self.nvml = None

    def _poll(self):
        while not self.stop_ev.is_set():
            self.mark()
            self.stop_ev.wait(0.002)

    def mark(self):
        if self.nvml is None:
            return
        r = self.nvml.sample()
        if r:
            with self.lock:
                self.rows.append(r)

    def start(self):
        import threading
        if self.nvml is not None:
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.source = "nvidia-smi"
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.index], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def _smi_rows(self):
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        raw = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for r in raw:
            if len(r) < 9:
                continue
            try:
                rows.append((float(r[1]), float(r[2]), float(r[3]),
                             [n for n, v in zip(names, r[5:9]) if v.strip().lower() == "active"]))
            except ValueError:
                continue
        return rows

    def stop(self):
        if self.thread is not None:
            self.stop_ev.set()
            self.thread.join(timeout=5)
            rows = self.rows
        elif self.proc is not None:
            rows = self._smi_rows()
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                    "reasons": [], "source": "unavailable (no NVML, no nvidia-smi)"}
        sm = [r[0] for r in rows]
        reasons = sorted({n for r in rows for n in r[3]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_min_mhz": min(sm) if sm else None,
                "sm_max_mhz": max(r[1] for r in rows) if rows else None,
                "power_w_max": max(r[2] for r in rows) if rows else None,
                "samples": len(sm), "reasons": reasons, "source": self.source}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_prep_seq(w, inp, b):
    """The oracle's rope table and prep of sequence b; returns its attend inputs."""
    import oracle
    rope = oracle.rope_table(inp["pos0"].numpy()[b:b + 1], w.t, w.hd, w.theta)
    q, k, v = oracle.prep(inp["yq"].numpy()[b:b + 1], inp["yk"].numpy()[b:b + 1],
                          inp["yv"].numpy()[b:b + 1], rope, inp["q_scale"].numpy(), w.eps)
    a = {"meta": inp["meta"].numpy()[b:b + 1], "q": q, "k_chunk": k, "v_chunk": v,
         "ring_k": inp["ring_k"].numpy()[b:b + 1], "ring_v": inp["ring_v"].numpy()[b:b + 1],
         "sink_k": inp["sink_k"].numpy()[b:b + 1], "sink_v": inp["sink_v"].numpy()[b:b + 1],
         "gate": inp["gate"].numpy()[b:b + 1], "gate_scale": inp["gate_scale"].numpy()}
    if "far" in inp:              # the sequence's far field state
        a["far"] = {k: (v.numpy()[b:b + 1].astype(np.float64) if torch.is_tensor(v) else v)
                    for k, v in inp["far"].items()}
    return a


def oracle_unit(w, a, i, g):
    """The oracle's attention of every query head of KV head g in row i;
    returns the attended KV-keys of the unit."""
    import oracle
    for h in range(g * w.hpg, (g + 1) * w.hpg):
        if "far" in a:
            oracle.attend_far_row(0, h, a, a["far"], w.score_scale, w.hpg, i)
        else:
            oracle.attend_row(0, i, h, a, w.score_scale, w.hpg)
    L, W = int(a["meta"][0][0]), int(a["meta"][0][3])
    return w.ns + min(W, L + i + 1)


def sample_inputs(w, nseq=4):
    """The first sequences of the batch the GPU arm runs at one GPU."""
    return workloads.make_shard_inputs(w, w.B, range(min(w.B, nseq)))


def _units_of(w, b, seed):
    units = [(i, g) for i in range(w.t) for g in range(w.nk)]
    np.random.default_rng(seed + b).shuffle(units)
    return units


# The oracle runs on every host core: one single-threaded worker process per core
# (spawn context, safe after CUDA is initialised), each holding the workload's
# seeded sample inputs; a task is one sequence, prepped and attended unit by unit
# (token path), or a batch of (query row, KV head) units (full-sequence attention).
_POOL_W = None
_POOL_INP = None


def host_cores():
    return max(1, min(32, os.cpu_count() or 1))


def host_cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _pool_init(kind, name, batch):
    global _POOL_W, _POOL_INP
    if kind == "token":
        w = workloads.WORKLOADS[name]
        if batch:
            w = dataclasses.replace(w, B=batch)
        _POOL_W, _POOL_INP = w, sample_inputs(w)
    else:
        w = workloads.FLASH_WORKLOADS[name]
        _POOL_W, _POOL_INP = w, workloads.make_flash_inputs(w)["qkv"].numpy()


def _token_task(job):
    """Sequence job[0] of the sample, prepped, then its first job[1] units;
    returns (attended KV-keys, units)."""
    b, limit, seed = job
    w, inp = _POOL_W, _POOL_INP
    b %= inp["meta"].shape[0]
    a = oracle_prep_seq(w, inp, b)
    units = _units_of(w, b, seed)[:limit]
    return sum(oracle_unit(w, a, i, g) for i, g in units), len(units)


def _flash_task(job):
    count, seed = job
    return flash_oracle_rows(_POOL_W, _POOL_INP, flash_units(_POOL_W, count, seed)), count


def oracle_pool(kind, w, batch=None):
    import multiprocessing as mp
    return mp.get_context("spawn").Pool(host_cores(), initializer=_pool_init, initargs=(kind, w.name, batch))


def cpu_baseline(w, budget_s, batch=None):
    """The oracle on a time-bounded sample, on every host core: rounds of one task
    per worker (a sequence of the sample, prepped, then attended unit by unit)."""
    n = host_cores()
    with oracle_pool("token", w, batch) as pool:
        pool.map(_token_task, [(k, 1, 0) for k in range(n)])        # warm the workers
        t0 = time.perf_counter()
        keys = units = seqs = 0
        r = 0
        while time.perf_counter() - t0 < budget_s:
            for k, u in pool.map(_token_task, [(r * n + k, 1 << 30, r) for k in range(n)]):
                keys += k
                units += u
            seqs += n
            r += 1
        dt = time.perf_counter() - t0
    return {"value": keys / dt, "unit": "keys/s", "cores": n, "kind": "oracle", "cpu": host_cpu_model(),
            "sample": f"{units} (sequence, row, KV head) units of {w.name} over {seqs} prepped sequences, "
                      f"all query heads of each unit ({keys} attended KV-keys, {dt:.1f} s, numpy float64, "
                      f"{n} single-threaded worker processes, one per host core)"}


def run_reference(args, w, rank):
    """Reference arm: the CPU oracle as it stands; each step preps one sequence
    of the workload and attends a bounded number of its units."""
    if rank != 0:
        return
    n = host_cores()
    with oracle_pool("token", w, args.batch) as pool:
        # size a step: every worker preps one sequence and attends per_step of its units
        t_a = time.perf_counter()
        pool.map(_token_task, [(k, 1, 1) for k in range(n)])
        t_unit = max(time.perf_counter() - t_a, 1e-4)
        budget_per_step = 150.0 / max(1, args.steps + args.warmup)
        per_step = int(max(1, min(w.t * w.nk, budget_per_step / t_unit)))
        state = {"r": 0}

        def step():
            r = state["r"]
            state["r"] += 1
            return sum(k for k, _ in pool.map(_token_task, [(r * n + k, per_step, 1) for k in range(n)]))

        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        keys = 0
        for _ in range(args.steps):
            keys += step()
        dt = time.perf_counter() - t0
    value = keys / dt
    sample = (f"per step: on each of {n} worker processes (one per host core), the rope table and prep "
              f"of one sequence of {w.name} and {per_step} of its (row, KV head) units with all their "
              f"query heads; numpy float64, single-threaded workers")
    line = {"impl": "reference", "metric": "attended KV-keys/s", "value": value, "unit": "keys/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "keys/s", "cores": n, "kind": "oracle",
                             "cpu": host_cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def prep_bytes(w):
    """Bytes the prep moves once per step (P1-P3): the q and k heads read and
    written; for single rows without a far field also the v heads read and
    the K/V rows written into the ring."""
    q = w.B * w.t * w.nh * w.hd * 4
    k = w.B * w.t * w.nk * w.hd * 4
    ring = 3 * k if (w.t == 1 and not w.far_m) else 0
    return 2 * q + 2 * k + ring


def prep_report(w, prep_ms, peak_gbs):
    """The prep stage timed on its own (CUDA events around its kernel)."""
    us = statistics.median(prep_ms) * 1e3
    b = prep_bytes(w)
    gbs = b / (us * 1e-6) / 1e9
    return {"us_median": us, "bytes": b, "gbs": gbs, "frac_of_hbm": gbs / peak_gbs,
            "note": "rotation, unit heads, query scale and (single rows) the ring write; "
                    "the RoPE angles are evaluated in the kernel (f64)"}


# the L2 flush between timed steps when the inputs fit in L2 (129 MB)
L2_FLUSH_BYTES = 256 << 20
# device-side spin (SM clock cycles, about 0.2 ms) after the flush, while the
# interpreter issues a step whose kernels take microseconds
SPIN_CYCLES = 400000


def rings_fit_l2(w):
    """Whether a token-path workload's K/V rings fit in L2: then bench.py flushes
    L2 between timed steps (outside the timed events) instead of relying on size."""
    return w.B * w.nk * w.cap * w.hd * 8 <= 129e6


def workload_config(w, n):
    return {"workload": w.name, "B": w.B, "t": w.t, "nh": w.nh, "nk": w.nk, "hd": w.hd,
            "window": w.window, "cap": w.cap, "ns": w.ns, "seed": w.seed,
            "far_landmarks": w.far_m,
            "global_batch": n * w.B,
            "parallelism": f"sequence shards x{n} of a {n * w.B}-sequence batch (no collective)"
            if n > 1 else "1 GPU",
            "l2": "inputs larger than L2: the K/V rings read each step exceed 129 MB"
            if not rings_fit_l2(w) else
            f"L2 flushed between timed steps (a {L2_FLUSH_BYTES >> 20} MB write outside the timed "
            "events, then a device-side spin while the step is issued; for e2e, outside the "
            "host-timed replays): the K/V rings fit in L2"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def make_events(n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:          # materialise the CUDA events before handing them to C
        e.record()
    torch.cuda.synchronize()
    return evs


def run_gpu(args, w, rank, world, local_rank):
    import sliding_window_gqa_prep_gb300 as swa
    from sliding_window_gqa_prep_gb300.dist import max_over_ranks

    dev = torch.device("cuda", local_rank)
    inp = rank_inputs(w, rank, world)
    keys, kv_bytes = keys_and_bytes(w, inp["meta"])
    tp = swa.TokenPath(B=w.B, t=w.t, nh=w.nh, nk=w.nk, hd=w.hd, cap=w.cap, ns=w.ns,
                       q_scale=inp["q_scale"], gate_scale=inp["gate_scale"],
                       ring_k=inp["ring_k"], ring_v=inp["ring_v"], sink_k=inp["sink_k"],
                       sink_v=inp["sink_v"], meta=inp["meta"], pos0=inp["pos0"],
                       scale=w.score_scale, eps=w.eps, theta=w.theta, device=dev,
                       far=inp.get("far"))
    d_in = {k: inp[k].to(dev).contiguous() for k in ("yq", "yk", "yv", "gate")}
    del inp["ring_k"], inp["ring_v"]
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev) if rings_fit_l2(w) else None

    def cold():
        if flush is not None:
            flush.zero_()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # warm-up
    for _ in range(args.warmup):
        cold()
        tp.step(d_in["yq"], d_in["yk"], d_in["yv"], d_in["gate"])
    torch.cuda.synchronize()

    # the timed steps: nothing between the kernels, so each kernel's CTAs can be
    # scheduled while its predecessor finishes (programmatic dependent launch)
    K = args.steps
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier()
    l0 = swa.launch_count()
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for s in range(K):
            tp.step(d_in["yq"], d_in["yk"], d_in["yv"], d_in["gate"])
        e1.record()
        if clocks:
            clocks.mark()
        barrier()
        ms = e0.elapsed_time(e1)
    else:
        # inputs that fit in L2: the flush runs between the steps, outside their
        # events. These steps take microseconds, less than the interpreter needs
        # to issue them, so a device-side spin after the flush keeps the device
        # busy while the step is issued: the events bracket device time only.
        sev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
        for s in range(K):
            cold()
            torch.cuda._sleep(SPIN_CYCLES)
            sev[2 * s].record()
            tp.step(d_in["yq"], d_in["yk"], d_in["yv"], d_in["gate"])
            sev[2 * s + 1].record()
        if clocks:
            clocks.mark()
        barrier()
        ms = sum(sev[2 * s].elapsed_time(sev[2 * s + 1]) for s in range(K))
    launches = swa.launch_count() - l0
    # the attention kernel alone: events the library records right before and
    # after it on the same stream, over the same number of steps
    kev = make_events(2 * K)
    pev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
    barrier()
    for s in range(K):
        cold()
        if flush is not None:
            torch.cuda._sleep(SPIN_CYCLES)
        tp.step(d_in["yq"], d_in["yk"], d_in["yv"], d_in["gate"], ev_start=kev[2 * s],
                ev_stop=kev[2 * s + 1], prep_events=(pev[2 * s], pev[2 * s + 1]))
    if clocks:
        clocks.mark()
    barrier()
    clk = clocks.stop() if clocks else None
    kern_ms = [kev[2 * s].elapsed_time(kev[2 * s + 1]) for s in range(K)]
    prep_ms = [pev[2 * s].elapsed_time(pev[2 * s + 1]) for s in range(K)]
    err = int(tp.err.item())
    ms = max_over_ranks(ms, dev)

    # end to end: pinned host inputs in, gated output back, every step
    e2e = None
    if not args.no_e2e:
        # the public end-to-end call: a captured step (pinned inputs -> device,
        # prep, attention, merge/gate/commit, output -> pinned host), replayed
        tp.capture()
        for k, v in d_in.items():
            tp.h_in[k].copy_(v)
        h_in, h_out = tp.h_in, tp.h_out
        for _ in range(max(args.warmup, 1)):
            cold()
            tp.replay()
        K2 = K
        barrier()
        if flush is None:
            t0 = time.perf_counter()
            for _ in range(K2):
                tp.replay()
            barrier()
            e2e_s = time.perf_counter() - t0
        else:
            # each replay timed on its own (it ends with the host holding the output),
            # the L2 flush before it outside the timed span
            e2e_s = 0.0
            for _ in range(K2):
                cold()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                tp.replay()
                e2e_s += time.perf_counter() - t0
            barrier()
        e2e_s = max_over_ranks(e2e_s, dev)
        e2e = {"value": keys * K2 * world / e2e_s, "unit": "keys/s",
               "h2d_bytes_per_step": sum(v.numel() * 4 for v in h_in.values()),
               "d2h_bytes_per_step": h_out.numel() * 4,
               "ms_per_step": e2e_s * 1e3 / K2}

    if rank != 0:
        return
    pk = peaks()
    peak = pk["hbm_gbs"]
    step_s = ms / 1e3 / K
    one_kernel = launches == K
    kern_avg_s = sum(kern_ms) / len(kern_ms) / 1e3
    traffic = recorded_traffic(w)
    kernel_name = dominant_kernel(w)[0]
    if one_kernel:              # the whole step is one kernel: prep, attention, gate, commit
        kernel_name = "decode_step_kernel"
        traffic = recorded_traffic(w, kernel_name)
    path = attention_path(w)
    useful_flop = keys * w.hpg * w.hd * 4          # Q K^T and P V, 2 flop per multiply-add
    if path == "decode":
        roof = {"bound": "hbm", "achieved": kv_bytes / kern_avg_s / 1e9, "peak": peak,
                "unit": "GB/s", "peak_kind": pk["kind"]}
    elif path == "verify":
        roof = {"bound": "alu", "achieved": useful_flop / kern_avg_s / 1e12,
                "peak": pk["fp32_tflops"], "unit": "TFLOP/s",
                "peak_kind": "derived: 152 SMs x 128 FP32 FMA/clk x 2 x max SM clock",
                "kv_gbs": kv_bytes / kern_avg_s / 1e9, "kv_frac_of_hbm": kv_bytes / kern_avg_s / 1e9 / peak}
    else:
        # f16 hi/lo operands: three kind::f16 products per multiply-add, at the bf16 rate
        roof = {"bound": "tensor", "achieved": 3 * useful_flop / kern_avg_s / 1e12,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "peak_kind": f"{pk['kind']} bf16 (the f16 rate); achieved counts the 3 f16 products of each "
                             "multiply-add",
                "useful_tflops": useful_flop / kern_avg_s / 1e12}
    if path == "decode":
        roof["frac_of_nominal_8tbs"] = roof["achieved"] / NOMINAL_HBM_GBS
    elif path == "verify":
        roof["kv_frac_of_nominal_8tbs"] = roof["kv_gbs"] / NOMINAL_HBM_GBS
    roof.update({"frac": roof["achieved"] / roof["peak"], "kernel": kernel_name,
                 "traffic": traffic, "algorithmic_bytes_per_launch": kv_bytes,
                 "launch_ms_avg": kern_avg_s * 1e3})
    line = {
        "metric": "attended KV-keys/s",
        "value": keys * world / step_s,
        "unit": "keys/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded generator, shapes of the named workload)",
        "config": workload_config(w, world),
        "kv_read_gbs_step": kv_bytes * world / step_s / 1e9,
        "kv_read_frac_of_peak_step": kv_bytes / step_s / 1e9 / peak,
        "kv_read_frac_of_nominal_8tbs_step": kv_bytes / step_s / 1e9 / NOMINAL_HBM_GBS,
        "roofline": roof,
        "prep": prep_report(w, prep_ms, pk["hbm_gbs"]) if not one_kernel else
        {"note": "folded into the one-kernel decode step (no separate prep launch)"},
        "gpu_launches": launches,
        "launches_per_step": launches / K,
        "device_errors": err,
        "clocks": clk,
    }
    if e2e:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, args.batch)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Full-sequence attention (swa_flash): the second workload
# ---------------------------------------------------------------------------


def flash_recorded_traffic(w):
    """DRAM bytes per launch of swa_flash's kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(PROFILE_DIR, f"attend_prompt_h16_kernel_{w.name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch\s*[:=]\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256_16\s*[:=]\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != source_hash(os.path.join(CSRC, "swa_prompt_h16.cu")):
        return None
    return float(m.group(1))


def flash_config(w, n):
    return {"workload": w.name, "segments": [list(s) for s in w.segs], "T": w.T, "nh": w.nh, "nk": w.nk,
            "hd": w.hd, "ld": w.ld, "seed": w.seed, "scale": w.score_scale,
            "parallelism": f"replicas x{n} (no collective)" if n > 1 else "1 GPU",
            "l2": f"L2 flushed between timed calls (a {L2_FLUSH_BYTES >> 20} MB write): "
                  "the packed rows fit in L2"}


def flash_oracle_rows(w, qkv, picks):
    """The oracle on (segment, row, KV head) units: all query heads of the unit."""
    import oracle
    keys = 0
    for (s0, n), r, g in picks:
        for h in range(g * w.group, (g + 1) * w.group):
            oracle.flash_row(qkv, s0, n, r, h, w.hd, w.group, w.q_off, w.k_off, w.v_off, w.score_scale)
        keys += n
    return keys


def flash_units(w, count, seed):
    rng = np.random.default_rng(seed)
    segs = [s for s in w.segs if s[1] > 0]
    out = []
    for _ in range(count):
        s0, n = segs[int(rng.integers(len(segs)))]
        out.append(((s0, n), int(rng.integers(n)), int(rng.integers(w.nk))))
    return out


def flash_cpu_baseline(w, budget_s):
    n = host_cores()
    with oracle_pool("flash", w) as pool:
        pool.map(_flash_task, [(1, k) for k in range(n)])             # warm the workers
        t0 = time.perf_counter()
        keys = units = r = 0
        while time.perf_counter() - t0 < budget_s:
            for k, u in pool.map(_flash_task, [(4, 1000 + r * n + k) for k in range(n)]):
                keys += k
                units += u
            r += 1
        dt = time.perf_counter() - t0
    return {"value": keys / dt, "unit": "keys/s", "cores": n, "kind": "oracle", "cpu": host_cpu_model(),
            "sample": f"{units} random (query row, KV head) units of {w.name}, all query heads of each "
                      f"({keys} attended keys, {dt:.1f} s, numpy float64, {n} single-threaded worker "
                      f"processes, one per host core)"}


def run_flash_reference(args, w, rank):
    """Reference arm for the full-sequence workload: the CPU oracle as it stands,
    each step a bounded sample of (query row, KV head) units."""
    if rank != 0:
        return
    n = host_cores()
    with oracle_pool("flash", w) as pool:
        t_a = time.perf_counter()
        pool.map(_flash_task, [(1, k) for k in range(n)])
        t_unit = max(time.perf_counter() - t_a, 1e-4)
        budget_per_step = 150.0 / max(1, args.steps + args.warmup)
        per_step = int(max(1, budget_per_step / t_unit))
        state = {"i": 0}

        def step():
            state["i"] += 1
            return sum(k for k, _ in pool.map(_flash_task, [(per_step, 100000 * state["i"] + k) for k in range(n)]))

        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        keys = 0
        for _ in range(args.steps):
            keys += step()
        dt = time.perf_counter() - t0
    value = keys / dt
    sample = (f"per step: on each of {n} worker processes (one per host core), {per_step} random (query row, "
              f"KV head) units of {w.name} with all their query heads; numpy float64, single-threaded workers")
    line = {"impl": "reference", "metric": "attended keys/s", "value": value, "unit": "keys/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": flash_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "keys/s", "cores": n, "kind": "oracle", "cpu": host_cpu_model(),
                             "sample": sample},
            "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_flash_gpu(args, w, rank, world, local_rank):
    """One step = one swa_flash call over the workload's packed rows (resident in
    HBM); an L2-sized write separates the timed calls."""
    import sliding_window_gqa_prep_gb300 as swa
    from sliding_window_gqa_prep_gb300.dist import max_over_ranks

    dev = torch.device("cuda", local_rank)
    inp = workloads.make_flash_inputs(dataclasses.replace(w, seed=w.seed + 1000 * rank))
    keys, useful_flop = workloads.flash_keys_and_flops(w)
    qkv = inp["qkv"].to(dev)
    segs = inp["segs"].to(dev)
    out = torch.zeros(w.T, w.nh * w.hd, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    # the split-once form: each KV head's K/V split into f16 hi/lo operand blocks once per call
    ws = torch.empty(swa.flash_workspace_size(w.T, len(w.segs), w.hd, w.nh, w.nk, w.max_len),
                     dtype=torch.uint8, device=dev)
    kw = dict(hd=w.hd, nh=w.nh, nk=w.nk, q_off=w.q_off, k_off=w.k_off, v_off=w.v_off,
              scale=w.score_scale, max_len=w.max_len, err=err, workspace=ws)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.zero_()
        swa.flash(qkv, segs, out=out, **kw)
    barrier()
    K = args.steps
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    kev = make_events(2 * K)                     # the library's, around the attention kernel
    sev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]   # around the whole call
    barrier()
    l0 = swa.launch_count()
    for s in range(K):
        flush.zero_()
        sev[2 * s].record()
        swa.flash(qkv, segs, out=out, ev_start=kev[2 * s], ev_stop=kev[2 * s + 1], **kw)
        sev[2 * s + 1].record()
    if clocks:
        clocks.mark()
    barrier()
    launches = swa.launch_count() - l0
    clk = clocks.stop() if clocks else None
    kern_ms = [kev[2 * s].elapsed_time(kev[2 * s + 1]) for s in range(K)]
    ms = max_over_ranks(sum(sev[2 * s].elapsed_time(sev[2 * s + 1]) for s in range(K)), dev)

    e2e = None
    if not args.no_e2e:
        # the public call on host buffers: pinned rows in, output rows back, every step
        h_qkv = inp["qkv"].pin_memory()
        h_out = torch.empty(w.T, w.nh * w.hd).pin_memory()
        d_qkv = torch.empty_like(qkv)

        def e2e_step():
            d_qkv.copy_(h_qkv, non_blocking=True)
            swa.flash(d_qkv, segs, out=out, **kw)
            h_out.copy_(out, non_blocking=True)

        for _ in range(max(args.warmup, 1)):
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        barrier()
        e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
        e2e = {"value": keys * K * world / e2e_s, "unit": "keys/s",
               "h2d_bytes_per_step": h_qkv.numel() * 4, "d2h_bytes_per_step": h_out.numel() * 4,
               "ms_per_step": e2e_s * 1e3 / K}
    if rank != 0:
        return
    pk = peaks()
    kern_avg_s = sum(kern_ms) / len(kern_ms) / 1e3
    roof = {"bound": "tensor", "achieved": 3 * useful_flop / kern_avg_s / 1e12, "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s",
            "peak_kind": f"{pk['kind']} bf16 (the f16 rate); achieved counts the 3 f16 products of each "
                         "multiply-add",
            "useful_tflops": useful_flop / kern_avg_s / 1e12}
    roof.update({"frac": roof["achieved"] / roof["peak"], "kernel": "attend_prompt_h16_kernel (full-sequence)",
                 "traffic": flash_recorded_traffic(w), "launch_ms_avg": kern_avg_s * 1e3})
    line = {
        "metric": "attended keys/s",
        "value": keys * world / (ms / 1e3 / K),
        "step": "one swa_flash call: the split-once kernel (K/V into f16 hi/lo operand blocks) and the "
                "persistent attention kernel, L2 flushed before it",
        "unit": "keys/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (f16 hi/lo tensor-core products under power-of-two block scales, f32 softmax)",
        "data": "synthetic (seeded generator, shapes of the named workload)",
        "config": flash_config(w, world),
        "roofline": roof,
        "gpu_launches": launches,
        "launches_per_step": launches / K,
        "device_errors": int(err.item()),
        "clocks": clk,
    }
    if e2e:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = flash_cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.workload in workloads.FLASH_WORKLOADS:
        w = workloads.FLASH_WORKLOADS[args.workload]
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        if args.impl == "reference":
            run_flash_reference(args, w, rank)
            return
        torch.cuda.set_device(local_rank)
        if world > 1:
            torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        try:
            run_flash_gpu(args, w, rank, world, local_rank)
        finally:
            if world > 1:
                torch.distributed.destroy_process_group()
        return
    w = workloads.WORKLOADS[args.workload]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    torch.cuda.set_device(local_rank)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_gpu(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
