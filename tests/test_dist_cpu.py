"""The multi-rank path on CPU (gloo, world size 2): sequences split across
ranks give exactly the single-process results (sequences are independent),
and the timing reduction takes the maximum over ranks."""
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


def _worker(rank, world, port, out_dir):
    import oracle
    import workloads
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.custom(B=4, t=3, nh=8, nk=2, hd=16, window=10, cap=10, ns=2,
                             pos_mode="full", pos_lo=10, pos_hi=90, seed=3)
        inp = workloads.make_inputs(w)
        mine = shard_sequences(w.B, rank, world)
        rope = oracle.rope_table(inp["pos0"].numpy()[mine], w.t, w.hd)
        q, k, v = oracle.prep(inp["yq"].numpy()[mine], inp["yk"].numpy()[mine],
                              inp["yv"].numpy()[mine], rope, inp["q_scale"].numpy(), w.eps)
        a = {"meta": inp["meta"].numpy()[mine], "q": q, "k_chunk": k, "v_chunk": v,
             "ring_k": inp["ring_k"].numpy()[mine], "ring_v": inp["ring_v"].numpy()[mine],
             "sink_k": inp["sink_k"].numpy()[mine], "sink_v": inp["sink_v"].numpy()[mine],
             "gate": inp["gate"].numpy()[mine], "gate_scale": inp["gate_scale"].numpy()}
        out = oracle.attend(a, w.score_scale, w.hpg)
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
    import oracle
    import workloads
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    w = workloads.custom(B=4, t=3, nh=8, nk=2, hd=16, window=10, cap=10, ns=2,
                         pos_mode="full", pos_lo=10, pos_hi=90, seed=3)
    inp = workloads.make_inputs(w)
    rope = oracle.rope_table(inp["pos0"].numpy(), w.t, w.hd)
    q, k, v = oracle.prep(inp["yq"].numpy(), inp["yk"].numpy(), inp["yv"].numpy(), rope,
                          inp["q_scale"].numpy(), w.eps)
    a = {"meta": inp["meta"].numpy(), "q": q, "k_chunk": k, "v_chunk": v,
         "ring_k": inp["ring_k"].numpy(), "ring_v": inp["ring_v"].numpy(),
         "sink_k": inp["sink_k"].numpy(), "sink_v": inp["sink_v"].numpy(),
         "gate": inp["gate"].numpy(), "gate_scale": inp["gate_scale"].numpy()}
    ref = oracle.attend(a, w.score_scale, w.hpg)
    order = np.load(tmp_path / "order.npy")
    assert order.tolist() == list(range(w.B))
    np.testing.assert_array_equal(np.load(tmp_path / "full.npy"), ref)
    assert np.load(tmp_path / "slowest.npy")[0] == 2.0
