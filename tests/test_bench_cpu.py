"""Host-side logic of bench.py that needs no GPU: the kernel it names for each
workload and the L2 regime it states."""
import bench
import workloads
import sliding_window_gqa_prep_gb300 as swa


def test_tensor_core_path_agrees_with_the_library_planner():
    # only the tcgen05 prompt kernel's plan adds split-once operand blocks beyond the
    # smallest workspace, so the two sizes differ exactly for the workloads that
    # bench.py attributes to that kernel
    for name, w in workloads.WORKLOADS.items():
        args = (w.B, w.t, w.nh, w.nk, w.hd, w.cap, w.ns, 0, w.far_m)
        full, least = swa.attend_workspace_size(*args), swa.attend_workspace_min(*args)
        assert full >= least > 0, name
        assert (bench.attention_path(w) == "prompt_tc") == (full > least), name


def test_l2_regime_follows_the_ring_size():
    for name, w in workloads.WORKLOADS.items():
        note = bench.workload_config(w, 1)["l2"]
        rings = w.B * w.nk * w.cap * w.hd * 8
        assert ("flushed" in note) == (rings <= 129e6), name
        assert ("larger than L2" in note) == (rings > 129e6), name
    assert "flushed" in bench.flash_config(workloads.FLASH_WORKLOADS["vision_flash"], 1)["l2"]


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) on the smallest
    workload: one JSON line with the contract's keys, its own cpu_baseline and an e2e
    block with no copies."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_decode",
                          "--steps", "1", "--warmup", "1"], cwd=root, capture_output=True, text=True,
                         timeout=600, check=True).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_decode" and d["steps"] == 1 and d["warmup"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
