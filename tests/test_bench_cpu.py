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
