"""GPU greedy accept and cache compaction (through the C ABI) against the
oracle, bit for bit, including malformed trees and paths."""
import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import t

pytestmark = pytest.mark.gpu


def accept_both(tokens, parents, target, D):
    g = DB.ddt_tree_accept(t(np.asarray(tokens, np.int32)), t(np.asarray(parents, np.int32)),
                           t(np.asarray(target, np.int32)), D)
    torch.cuda.synchronize()
    ref = O.tree_accept(tokens, parents, target, D)
    for k in ("accept_idx", "accept_len", "out_tokens", "bonus", "status"):
        np.testing.assert_array_equal(g[k].cpu().numpy(), ref[k], err_msg=k)
    return ref


@pytest.mark.parametrize("cfg", ["c1", "c2", "c3", "c4"])
def test_accept_on_workload_trees(cfg):
    w = WL.CONFIGS[cfg]
    batch = WL.make_batch(w, latents=False)
    tree = O.tree_build(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
    target = WL.target_argmax_for(batch, tree["depths"])
    ref = accept_both(tree["tokens"], tree["parents"], target, w.D)
    if cfg == "c4":
        assert (ref["accept_len"] == 15).all()


def test_accept_random_and_malformed_trees():
    g = np.random.default_rng(3)
    for trial in range(30):
        B, Q = int(g.integers(1, 17)), int(g.integers(1, 129))
        D = int(g.integers(0, 20))
        tokens = g.integers(0, 4, (B, Q))
        if trial % 2:
            parents = g.integers(-1, Q, (B, Q))      # arbitrary, cycles likely
        else:
            parents = np.array([[-1] + [int(g.integers(0, c)) for c in range(1, Q)]
                                for _ in range(B)])
        target = g.integers(0, 4, (B, Q))
        accept_both(tokens, parents, target, D)


def test_accept_cycle_is_reported():
    tokens = np.array([[7, 8, 9]])
    parents = np.array([[2, 0, 1]])
    target = np.array([[8, 9, 7]])
    ref = accept_both(tokens, parents, target, 10)
    assert ref["status"][0] == O.ST_CYCLE


def compact_both(kv_np, bt, L, idx, n, page_size):
    if kv_np.dtype == np.uint16:
        kv_np = kv_np.view(np.int16)
    kv = t(kv_np)
    new_len, status = DB.ddt_cache_compact(kv, t(bt.astype(np.int32)), t(L.astype(np.int32)),
                                           t(idx.astype(np.int32)), t(n.astype(np.int32)),
                                           page_size)
    torch.cuda.synchronize()
    ref_kv, ref_len, ref_st = O.cache_compact(kv_np, bt, L, idx, n, page_size, bt.shape[1])
    np.testing.assert_array_equal(kv.cpu().numpy(), ref_kv)
    np.testing.assert_array_equal(new_len.cpu().numpy(), ref_len)
    np.testing.assert_array_equal(status.cpu().numpy(), ref_st)


@pytest.mark.parametrize("width,dt", [(576, np.uint16), (96, np.float32), (8, np.uint16)])
def test_compaction_paths_pages_and_overlaps(width, dt):
    g = np.random.default_rng(width)
    P, pages, B, D = 16, 40, 6, 7
    kv = g.integers(0, 60000, (P * pages, width)).astype(dt)
    bt = g.permutation(pages)[: B * 6].reshape(B, 6).astype(np.int32)
    L = g.integers(0, 40, B)
    idx = np.full((B, D + 1), -1)
    n = np.zeros(B, np.int64)
    for b in range(B):
        k = int(g.integers(0, D + 1))
        path = np.sort(g.choice(np.arange(1, 40), k, replace=False)) if k else []
        idx[b, 0] = 0
        idx[b, 1: k + 1] = path
        n[b] = k
    idx[0, 1:4] = [2, 3, 4]  # overlapping: slot L+1 <- L+2 <- L+3 ...
    n[0] = 3
    compact_both(kv, bt, L, idx, n, P)


def test_compaction_range_errors():
    # past capacity, a page outside the cache, a negative slot, and lists that
    # are not paths from the root (decreasing, repeated, the root itself)
    kv = np.arange(64 * 8, dtype=np.uint16).reshape(64, 8)
    bt = np.array([[0, 1], [2, 3], [1, 9], [0, 1], [0, 1], [2, 3], [1, 0], [3, 2]], np.int32)
    L = np.array([3, 28, 10, 4, 2, 5, 7, 1])
    idx = np.array([[0, 2, -1], [0, 1, 2], [0, 7, -1], [0, -4, -1], [0, 5, 3], [0, 4, 4],
                    [0, 0, 3], [0, 1, 2]])
    n = np.array([1, 2, 1, 1, 2, 2, 2, 2])
    compact_both(kv, bt, L, idx, n, 16)


@pytest.mark.parametrize("B", [3, 700])
def test_compaction_long_rows_with_overlaps_over_several_batches(B):
    # rows of 4 KB, paths whose sources are also destinations, more chunks per
    # CTA than one batch of loads holds: batches must follow increasing d
    g = np.random.default_rng(B)
    P, D, width = 8, 12, 2048
    pages_per = 4
    if B > 100:
        width = 256  # 512 B rows, eight sequences per CTA
    kv = g.integers(0, 60000, (B * pages_per * P, width)).astype(np.uint16)
    bt = g.permutation(B * pages_per).reshape(B, pages_per).astype(np.int32)
    L = g.integers(0, 6, B)
    idx = np.full((B, D + 1), -1)
    n = np.zeros(B, np.int64)
    for b in range(B):
        k = int(g.integers(0, D + 1))
        if b % 3 == 0:  # dense: every source but the last is also a destination
            path = list(range(2, k + 2))
        else:
            path = np.sort(g.choice(np.arange(1, 2 * D), k, replace=False))
        idx[b, 0] = 0
        idx[b, 1: k + 1] = path
        n[b] = k
    compact_both(kv, bt, L, idx, n, P)


def test_many_sequences_share_a_cta():
    # past two sequences per SM a CTA serves up to eight sequences (one warp
    # walks each); trees of mixed shape with and without a matching path,
    # then compaction of all of them, against the oracle bit for bit
    g = np.random.default_rng(17)
    B, Q, D = 1000, 17, 8
    parents = np.array([[-1] + [int(g.integers(0, c)) for c in range(1, Q)] for _ in range(B)])
    tokens = g.integers(0, 3, (B, Q))
    target = g.integers(0, 3, (B, Q))
    ref = accept_both(tokens, parents, target, D)
    assert ref["accept_len"].max() >= 3
    P, width = 8, 72
    pages_per = -(-(40 + Q) // P)
    kv = g.integers(0, 60000, (B * pages_per * P, width)).astype(np.uint16)
    bt = g.permutation(B * pages_per).reshape(B, pages_per).astype(np.int32)
    L = g.integers(0, 40, B)
    L[::97] = pages_per * P  # a few sequences out of range
    compact_both(kv, bt, L, np.asarray(ref["accept_idx"]), np.asarray(ref["accept_len"]), P)


def test_many_sequences_given_paths():
    # the compaction-only branch on a large batch: given accepted paths,
    # several sequences per CTA
    g = np.random.default_rng(23)
    B, D = 700, 5
    P, width = 16, 40
    pages_per = 4
    kv = g.integers(0, 60000, (B * pages_per * P, width)).astype(np.uint16)
    bt = g.permutation(B * pages_per).reshape(B, pages_per).astype(np.int32)
    L = g.integers(0, 30, B)
    n = g.integers(0, D + 1, B)
    idx = np.full((B, D + 1), -1)
    for b in range(B):
        idx[b, 0] = 0
        idx[b, 1: n[b] + 1] = np.sort(g.choice(np.arange(1, 20), n[b], replace=False))
    compact_both(kv, bt, L, idx, n, P)
