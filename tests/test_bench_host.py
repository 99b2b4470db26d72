"""Host-side logic of bench.py: the max-over-ranks reduction of the replica
timing under a 2-rank gloo process group, and the algorithmic work count
used for the roofline."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import workloads as WL


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [3.5, 1.25][rank]
    out[rank] = bench.max_over_ranks(mine, world)
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(2.0, 1) == 2.0


def test_attention_work_counts_visible_pairs():
    w = WL.CONFIGS["c1"].with_(B=2, prefix=(3, 9))
    batch = WL.make_batch(w, latents=False)
    tree = O.tree_build(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
    flops, byt = bench.attn_work(w, batch.prefix_len, tree["depths"], 4)
    pairs = 0
    for b in range(w.B):
        for i in range(w.Q):
            vis = O.visible_tree_slots(tree["vis_bits"][b, i], w.Q)
            pairs += int(batch.prefix_len[b]) + int(vis.sum())
    assert flops == pairs * w.H * (4 * w.C + 2 * w.R)
    keys = int(batch.prefix_len.sum()) + w.B * w.Q
    rows = w.B * w.Q * w.H
    assert byt == keys * (w.C + w.R) * 4 + rows * (w.C + w.R) * 4 + rows * w.C * 4 + rows * 4


def test_config_names_resolve():
    assert bench.workload("c2").budget == 64
    w = bench.workload("q17_b8_l8192")
    assert (w.Q, w.B, w.prefix) == (17, 8, 8192)
    with pytest.raises(SystemExit):
        bench.workload("nope")


def test_single_sequence_oracle_step_is_that_sequences_share_of_the_batch_step():
    # the CPU baselines time one sequence at a time (own cache of its pages)
    # and extrapolate by B; each such step must do exactly what the batch
    # step does for that sequence
    w = WL.CONFIGS["c3"].with_(B=3, V=512, H=2, C=16, R=8, prefix=(40, 150))
    batch = WL.make_batch(w)
    lay = batch.layout
    whole = O.ddt_step(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V,
                       batch.q_lat, batch.q_pe, batch.kv, lay.block_table, batch.prefix_len,
                       w.scale, lay.page_size, lay.max_pages,
                       lambda t: WL.target_argmax_for(batch, t["depths"]))
    for b in range(w.B):
        one = bench.oracle_sequence(w, batch, b)()
        for k in ("tokens", "parents", "depths", "vis_bits"):
            np.testing.assert_array_equal(one["tree"][k][0], whole["tree"][k][b])
        np.testing.assert_array_equal(one["o"][0], whole["o"][b])
        for k in ("accept_idx", "accept_len", "out_tokens"):
            np.testing.assert_array_equal(one["accept"][k][0], whole["accept"][k][b])
        n = int(batch.prefix_len[b]) + w.Q
        np.testing.assert_array_equal(one["kv"][:n], whole["kv"][lay.rows_of(b, np.arange(n))])
        assert one["new_len"][0] == whole["new_len"][b]


def test_oracle_steps_extrapolate_by_batch():
    w = WL.CONFIGS["c1"].with_(B=4)
    batch = WL.make_batch(w)
    n, secs, v = bench.oracle_steps(w, batch, 0.0, 3)
    assert n == 1 and v == pytest.approx(1.0 / (4 * secs))
    n, secs, v = bench.oracle_steps(w, batch, 1e9, 5)
    assert n == 5 and v == pytest.approx(5 / (4 * secs))


def test_stress_point_accepts_a_path_off_the_rank0_chain():
    # the stress point's drafter and target (drawn with torch, here on the
    # CPU): the oracle accepts slots D+1 .. 2D, so every sequence moves D rows
    import torch
    D, K, V, B = 8, 4, 1000, 64
    logp, ids, root, target = WL.stress_inputs(B, D, K, V, torch.device("cpu"))
    tree = O.tree_build(logp.numpy(), ids.numpy(), root.numpy(), 2 * D, V)
    acc = O.tree_accept(tree["tokens"], tree["parents"], target.numpy(), D)
    assert (acc["accept_len"] == D).all()
    for b in range(B):
        assert list(tree["depths"][b][1: D + 1]) == list(range(1, D + 1))
        assert list(acc["accept_idx"][b]) == [0] + list(range(D + 1, 2 * D + 1))
        assert acc["accept_len"][b] == D
