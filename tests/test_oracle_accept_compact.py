"""Pins of the oracle's greedy accept and cache compaction: perfect drafter
accepts the full depth, the pages' 8.00 tokens/step and 24-in-3 figures, the
greedy invariant, cycle safety, brute-force path enumeration, and the gather
invariants including overlapping source/destination slots."""
import numpy as np
import pytest

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import workloads as WL


def test_perfect_drafter_accepts_full_depth_on_the_deep_workload():
    w = WL.CONFIGS["c4"]
    batch = WL.make_batch(w, latents=False)
    tree = O.tree_build(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
    target = WL.target_argmax_for(batch, tree["depths"])
    acc = O.tree_accept(tree["tokens"], tree["parents"], target, w.D)
    assert (acc["accept_len"] == 15).all()
    assert (acc["accept_idx"][:, 1:] == np.arange(1, 16)).all()
    assert (acc["out_tokens"][:, :15] == batch.topk_ids[:, :, 0]).all()


def test_pages_figures_8_tokens_per_step_24_in_3_vs_24_ar_steps():
    """Oracle drafter, depth 7: every verify step commits 7 drafts + 1 bonus
    = 8.00 tokens, so 24 new tokens take 3 verify steps where greedy AR takes
    24; the committed stream equals the golden greedy stream."""
    V = 5000
    golden = O.golden_stream(64, V, seed=1)
    out, steps, per = O.decode_loop(golden, 24, D=7, K=4, budget=16, V=V, drafter_hit=1.0, seed=2)
    assert out == golden[:25]
    assert steps == 3 and per == [8, 8, 8]
    assert sum(per) / steps == 8.0
    ar_steps = len(out) - 1  # one target forward per token
    assert ar_steps == 24


@pytest.mark.parametrize("hit", [0.0, 0.4, 0.8])
def test_greedy_invariant_with_an_imperfect_drafter(hit):
    V = 3000
    golden = O.golden_stream(200, V, seed=3)
    out, steps, per = O.decode_loop(golden, 60, D=5, K=3, budget=12, V=V, drafter_hit=hit, seed=4)
    assert out == golden[:61]
    assert all(1 <= x <= 6 for x in per)
    if hit == 0.0:
        assert steps == 60


def test_cyclic_tree_stops_with_cycle_status():
    # slot 0 (root) is made the child of slot 2: 0 -> 1 -> 2 -> 0 ...
    tokens = [7, 8, 9]
    parents = [2, 0, 1]
    target = [8, 9, 7]
    r = O.accept_one(tokens, parents, target, D=10)
    assert r["status"] == O.ST_CYCLE
    assert r["accept_idx"][:3] == [0, 1, 2] and r["accept_len"] == 2
    assert r["bonus"] == 7


def test_walk_is_bounded_by_depth():
    Q = 10
    tokens = list(range(Q))
    parents = [-1] + list(range(Q - 1))  # a chain of 9 drafts
    target = [c + 1 for c in range(Q)]
    r = O.accept_one(tokens, parents, target, D=4)
    assert r["accept_len"] == 4 and r["accept_idx"] == [0, 1, 2, 3, 4]
    assert r["out_tokens"] == [1, 2, 3, 4, 5]


def _paths(parents):
    """All root-to-node paths by brute force over parent pointers."""
    out = {}
    for n in range(len(parents)):
        p, c = [], n
        while c >= 0:
            p.append(c)
            c = parents[c]
        if p[-1] == 0:
            out[n] = p[::-1]
    return out


def test_accept_equals_deepest_fully_matching_path():
    w = WL.CONFIGS["c3"].with_(V=4096)
    g = np.random.default_rng(0)
    for b in range(16):
        logp, ids = WL.drafter_topk(w, b)
        t = O.build_one(logp, ids, 3, w.budget, w.V)
        # target: usually the rank-0 child token, sometimes the rank-1 one
        target = []
        for n in range(w.Q):
            d = t["depths"][n]
            if 0 <= d < w.D:
                target.append(int(ids[d, 0 if g.random() < 0.8 else 1]))
            else:
                target.append(-5)
        r = O.accept_one(t["tokens"], t["parents"], target, w.D)
        best = [0]
        for n, path in _paths(t["parents"]).items():
            if all(t["tokens"][path[k + 1]] == target[path[k]] for k in range(len(path) - 1)):
                if len(path) > len(best):
                    best = path
        assert r["accept_idx"][: len(best)] == best
        assert r["accept_len"] == len(best) - 1
        assert r["bonus"] == target[best[-1]]


def _cache(n_rows, width, seed):
    g = np.random.default_rng(seed)
    return g.integers(0, 2 ** 16, (n_rows, width)).astype(np.uint16)


def test_compaction_moves_accepted_rows_and_nothing_else():
    P, pages = 8, 6
    kv = _cache(P * pages, 5, 0)
    bt = np.array([[4, 1, 5], [0, 2, 3]], np.int32)
    L = np.array([10, 3], np.int32)
    accept_idx = np.array([[0, 3, 5, 6, -1], [0, 1, 4, -1, -1]], np.int32)
    accept_len = np.array([3, 2], np.int32)
    new, new_len, st = O.cache_compact(kv, bt, L, accept_idx, accept_len, P, 3)
    assert list(new_len) == [14, 6] and list(st) == [0, 0]
    touched = set()
    for b in range(2):
        for d in range(1, accept_len[b] + 1):
            dst = O.slot_rows(bt[b], P, [L[b] + d])[0]
            src = O.slot_rows(bt[b], P, [L[b] + accept_idx[b, d]])[0]
            np.testing.assert_array_equal(new[dst], kv[src])
            touched.add(dst)
    for r in range(len(kv)):
        if r not in touched:
            np.testing.assert_array_equal(new[r], kv[r])


def test_compaction_reads_before_writing_when_slots_overlap():
    # path 0 -> 2 -> 3: slot L+1 <- L+2 and slot L+2 <- L+3; the first copy
    # must see the row that was at L+2 before the second copy overwrote it
    kv = np.arange(40, dtype=np.uint16).reshape(10, 4)
    bt = np.zeros((1, 1), np.int32)
    L = np.array([4], np.int32)
    new, new_len, st = O.cache_compact(kv, bt, L, np.array([[0, 2, 3]], np.int32),
                                       np.array([2], np.int32), 10, 1)
    np.testing.assert_array_equal(new[5], kv[6])
    np.testing.assert_array_equal(new[6], kv[7])
    assert new_len[0] == 7 and st[0] == 0


@pytest.mark.parametrize("bad", ["neg_idx", "past_capacity", "len_too_long", "decreasing",
                                 "repeated", "root_as_child"])
def test_compaction_range_errors_leave_sequence_untouched(bad):
    kv = _cache(16, 3, 1)
    bt = np.zeros((1, 1), np.int32)
    idx = np.array([[0, 1, 2]], np.int32)
    n = np.array([2], np.int32)
    L = np.array([5], np.int32)
    if bad == "neg_idx":
        idx[0, 2] = -1
    elif bad == "past_capacity":
        idx[0, 2] = 20
    elif bad == "len_too_long":
        n[0] = 3
    elif bad == "decreasing":  # not a path: a child pops after its parent
        idx[0, 1:] = [3, 2]
    elif bad == "repeated":
        idx[0, 1:] = [2, 2]
    else:  # slot 0 is the root, never one of its own descendants
        idx[0, 1:] = [0, 4]
    new, new_len, st = O.cache_compact(kv, bt, L, idx, n, 16, 1)
    assert st[0] == O.ST_RANGE and new_len[0] == 5
    np.testing.assert_array_equal(new, kv)


def test_qlen1_step_degenerates_to_ar():
    """budget 0: the tree is the root alone, nothing is accepted, the bonus is
    the target's argmax at the root and compaction moves nothing."""
    w = WL.CONFIGS["c1"].with_(budget=0)
    batch = WL.make_batch(w)
    res = O.ddt_step(batch.topk_logp, batch.topk_ids, batch.root_tok, 0, w.V, batch.q_lat,
                     batch.q_pe, batch.kv, batch.layout.block_table, batch.prefix_len, w.scale,
                     batch.layout.page_size, batch.layout.max_pages,
                     lambda t: WL.target_argmax_for(batch, t["depths"]))
    assert res["accept"]["accept_len"][0] == 0
    assert res["accept"]["out_tokens"][0][0] == res["target"][0][0]
    np.testing.assert_array_equal(res["kv"], batch.kv)
    assert res["new_len"][0] == batch.prefix_len[0] + 1


def test_compaction_page_outside_cache_is_a_range_error():
    kv = _cache(16, 3, 2)
    bt = np.array([[0, 7]], np.int32)  # page 7 does not exist (2 pages of 8)
    new, new_len, st = O.cache_compact(kv, bt, np.array([6], np.int32),
                                       np.array([[0, 1, 3]], np.int32), np.array([2], np.int32),
                                       8, 2)
    assert st[0] == O.ST_RANGE and new_len[0] == 6
    np.testing.assert_array_equal(new, kv)


def test_accepted_paths_increase_strictly_from_the_root():
    # the walk follows parent -> child edges and the builder numbers nodes in
    # pop order (a parent pops before its children), so every accepted path
    # is a valid compaction list: 0 = s_0 < s_1 < ... < s_len
    g = np.random.default_rng(5)
    for trial in range(40):
        w = WL.CONFIGS["c1"].with_(B=4, D=int(g.integers(1, 6)), K=int(g.integers(1, 5)),
                                   budget=int(g.integers(0, 20)), V=6)
        batch = WL.make_batch(w, latents=False)
        tree = O.tree_build(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
        target = g.integers(0, w.V, (w.B, w.Q)).astype(np.int32)
        # half the slots follow a child so that paths get long
        for b in range(w.B):
            for c in range(1, w.Q):
                p = int(tree["parents"][b][c])
                if p >= 0 and g.random() < 0.5:
                    target[b][p] = tree["tokens"][b][c]
        acc = O.tree_accept(tree["tokens"], tree["parents"], target, w.D)
        for b in range(w.B):
            n = int(acc["accept_len"][b])
            path = [int(x) for x in acc["accept_idx"][b][: n + 1]]
            assert path[0] == 0 and all(path[d] > path[d - 1] for d in range(1, n + 1))
