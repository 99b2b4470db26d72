"""GPU tree build (ddt_tree_build through the C ABI) against the oracle,
bit for bit: tokens, parents, depths, ancestor masks, dense visibility,
first-child/next-sibling lists, node counts and status."""
import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import t, u64

pytestmark = pytest.mark.gpu


def run_both(logp, ids, root, budget, V):
    logp = np.ascontiguousarray(logp, np.float32)
    ids = np.ascontiguousarray(ids, np.int32)
    root = np.ascontiguousarray(root, np.int32)
    g = DB.ddt_tree_build(t(logp), t(ids), t(root), budget, V, with_vis=True)
    torch.cuda.synchronize()
    ref = O.tree_build(logp, ids, root, budget, V)
    return g, ref


def assert_same(g, ref):
    for k in ("tokens", "parents", "depths", "first_child", "next_sibling", "n_nodes", "status"):
        np.testing.assert_array_equal(g[k].cpu().numpy(), ref[k], err_msg=k)
    np.testing.assert_array_equal(u64(g["vis_bits"]), ref["vis_bits"])
    np.testing.assert_array_equal(g["vis"].cpu().numpy(), ref["vis"])


@pytest.mark.parametrize("cfg", ["c1", "c2", "c3", "c4"])
def test_workload_trees_bit_exact(cfg):
    w = WL.CONFIGS[cfg]
    batch = WL.make_batch(w, latents=False)
    g, ref = run_both(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
    assert_same(g, ref)


@pytest.mark.parametrize("q_len", WL.SWEEP_QLEN)
def test_sweep_qlens(q_len):
    w = WL.sweep_point(q_len, 8, 1024).with_(V=20000)
    batch = WL.make_batch(w, latents=False)
    g, ref = run_both(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
    assert_same(g, ref)


def test_tie_heavy_random_shapes():
    """Log-probs from {0, -0.5, -1, -2}: scores tie constantly, so every
    tie-break (depth, rank, parent slot) decides pops."""
    g = np.random.default_rng(123)
    for trial in range(40):
        B = int(g.integers(1, 9))
        D = int(g.integers(1, 7))
        K = int(g.integers(1, 6))
        budget = int(g.integers(0, 128))
        logp = -np.sort(g.choice([0.0, 0.5, 1.0, 2.0], (B, D, K)), axis=2)
        ids = g.integers(0, 500, (B, D, K))
        root = g.integers(0, 500, B)
        gg, ref = run_both(logp, ids, root, budget, 500)
        assert_same(gg, ref)


def test_continuous_random_shapes_and_max_budget():
    g = np.random.default_rng(7)
    for trial in range(20):
        B = int(g.integers(1, 33))
        D = int(g.integers(1, 20))
        K = int(g.integers(1, 10))
        budget = int(g.choice([1, 2, 31, 63, 64, 65, 100, 127]))
        logp = -np.sort(g.exponential(1.0, (B, D, K)), axis=2)
        ids = g.integers(0, 1 << 20, (B, D, K))
        root = g.integers(0, 1 << 20, B)
        gg, ref = run_both(logp, ids, root, budget, 1 << 20)
        assert_same(gg, ref)


def test_unsorted_and_positive_logprobs_follow_the_heap_exactly():
    """Malformed but finite drafter rows: the heap order is no longer the
    sorted order of all nodes; the kernel must still replay the heap."""
    g = np.random.default_rng(11)
    for trial in range(20):
        B, D, K = 4, int(g.integers(1, 6)), int(g.integers(1, 6))
        logp = g.normal(0, 2, (B, D, K))
        ids = g.integers(0, 100, (B, D, K))
        gg, ref = run_both(logp, ids, g.integers(0, 100, B), int(g.integers(0, 64)), 100)
        assert_same(gg, ref)


def test_padding_input_errors_and_degenerate_shapes():
    # candidate tree smaller than the budget (padding), K=1 chain, D=1 star,
    # budget 0, NaN / inf log-probs, out-of-range ids and root
    logp = np.full((6, 3, 2), -0.5, np.float32)
    ids = np.arange(36, dtype=np.int32).reshape(6, 3, 2)
    root = np.array([1, 2, 3, 4, 5, 6], np.int32)
    logp[1, 2, 1] = np.nan
    logp[2, 0, 0] = -np.inf
    ids[3, 1, 0] = 1000
    root[4] = -3
    gg, ref = run_both(logp, ids, root, 20, 1000)
    assert_same(gg, ref)
    assert ref["status"][1] & O.ST_INPUT and ref["status"][0] == O.ST_BUDGET_PAD
    for shape, budget in (((2, 9, 1), 12), ((2, 1, 9), 5), ((3, 4, 4), 0)):
        lg = -np.sort(np.random.default_rng(1).random(shape), axis=2)
        gg, ref = run_both(lg, np.random.default_rng(2).integers(0, 50, shape),
                           np.array([0] * shape[0]), budget, 50)
        assert_same(gg, ref)


def test_large_batch_stress():
    w = WL.CONFIGS["c3"].with_(V=4096, B=2048)
    g = np.random.default_rng(5)
    logp = -np.sort(g.exponential(1.0, (w.B, w.D, w.K)), axis=2)
    ids = g.integers(0, w.V, (w.B, w.D, w.K))
    gg, ref = run_both(logp, ids, g.integers(0, w.V, w.B), w.budget, w.V)
    assert_same(gg, ref)
