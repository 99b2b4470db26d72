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
