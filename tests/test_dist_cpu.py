"""The multi-rank path on CPU (gloo, world size 2): sequences split across
ranks give exactly the single-process results (sequences are independent),
and the timing reduction takes the maximum over ranks. The shards are the ones
bench.py builds under torchrun (bench.rank_inputs)."""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from sliding_window_gqa_prep_gb300.dist import max_over_ranks, shard_sequences


def test_shards_cover_the_batch_once():
    for B in (1, 2, 5, 64, 127):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                seen += shard_sequences(B, r, world)
            assert seen == list(range(B))
    with pytest.raises(ValueError):
        shard_sequences(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


# per-rank shape of the multi-rank tests: 2 sequences per rank
_W = dict(B=2, t=3, nh=8, nk=2, hd=16, window=10, cap=10, ns=2, pos_mode="partial",
          pos_lo=1, pos_hi=10, seed=3)


def _oracle_out(w, inp):
    import oracle
    rope = oracle.rope_table(inp["pos0"].numpy(), w.t, w.hd)
    q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                          inp["q_scale"].numpy(), w.eps)
    a = {"meta": inp["meta"].numpy(), "q": q, "k_chunk": k, "v_chunk": v,
         "ring_k": inp["ring_k"].numpy(), "ring_v": inp["ring_v"].numpy(),
         "sink_k": inp["sink_k"].numpy(), "sink_v": inp["sink_v"].numpy(),
         "gate": inp["gate"].numpy(), "gate_scale": inp["gate_scale"].numpy()}
    return oracle.attend(a, w.score_scale, w.hpg)


def test_bench_rank_inputs_are_shards_of_one_batch():
    """Under torchrun bench.py gives rank r the sequences shard_sequences(world * B,
    r, world) of one batch; a sequence's inputs do not depend on which rank holds it."""
    import bench
    import workloads
    for name in ("spec_verify_far", "prompt_chunk"):
        w = dataclasses.replace(workloads.WORKLOADS[name], B=3, cap=64, window=64, pos_lo=1,
                                pos_hi=64)
        for world in (1, 2, 3):
            whole = workloads.make_shard_inputs(w, world * w.B, range(world * w.B))
            for r in range(world):
                mine = shard_sequences(world * w.B, r, world)
                assert len(mine) == w.B
                part = bench.rank_inputs(w, r, world)
                for k, v in part.items():
                    if k == "far":
                        for kk, vv in v.items():
                            if torch.is_tensor(vv):
                                assert torch.equal(vv, whole["far"][kk][mine]), (name, kk)
                    elif k in ("q_scale", "gate_scale"):
                        assert torch.equal(v, whole[k])
                    else:
                        assert torch.equal(v, whole[k][mine]), (name, k)


def _worker(rank, world, port, out_dir):
    import bench
    import workloads
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.custom(**_W)
        inp = bench.rank_inputs(w, rank, world)
        mine = shard_sequences(world * w.B, rank, world)
        out = _oracle_out(w, inp)
        gathered = [None] * world
        torch.distributed.all_gather_object(gathered, (mine, out))
        slowest = max_over_ranks(1.0 + rank)
        if rank == 0:
            np.save(os.path.join(out_dir, "full.npy"), np.concatenate([o for _, o in gathered]))
            np.save(os.path.join(out_dir, "order.npy"), np.concatenate([m for m, _ in gathered]))
            np.save(os.path.join(out_dir, "slowest.npy"), np.array([slowest]))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_match_one_process(tmp_path):
    import workloads
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    w = workloads.custom(**_W)
    whole = workloads.make_shard_inputs(w, world * w.B, range(world * w.B))
    ref = _oracle_out(dataclasses.replace(w, B=world * w.B), whole)
    order = np.load(tmp_path / "order.npy")
    assert order.tolist() == list(range(world * w.B))
    np.testing.assert_array_equal(np.load(tmp_path / "full.npy"), ref)
    assert np.load(tmp_path / "slowest.npy")[0] == 2.0
