"""Pins of the oracle's tree build against things other than itself:
hand-worked fixtures, exhaustive enumeration of every path on tiny inputs,
structural invariants and special cases."""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import workloads as WL

HERE = os.path.dirname(os.path.abspath(__file__))


def _cases():
    with open(os.path.join(HERE, "golden", "tree_build_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_worked_fixtures(case):
    t = O.build_one(np.array(case["logp"], np.float32), np.array(case["ids"], np.int32),
                    case["root_tok"], case["budget"], case["V"])
    for k in ("tokens", "parents", "depths", "first_child", "next_sibling", "anc"):
        assert list(t[k]) == case[k], k
    assert t["n_nodes"] == case["n_nodes"]
    assert t["status"] == case["status"]


def brute_force(logp, ids, root, budget):
    """Enumerate every node of the depth-D, K-ary candidate tree, sort all of
    them by (-score, depth, rank, parent position) and keep the first
    budget+1. A node's parent position is its parent's place in the same
    sorted order, so the key of a node is compared through its parent's key
    (the parent always sorts first)."""
    D, K = logp.shape
    nodes = [((), 0.0)]  # (rank tuple, score)
    for d in range(1, D + 1):
        for tup in itertools.product(range(K), repeat=d):
            parent_score = [s for t, s in nodes if t == tup[:-1]][0]
            nodes.append((tup, parent_score + float(logp[d - 1, tup[-1]])))
    score = dict(nodes)

    def key(tup):
        if not tup:
            return (-0.0, 0, 0, ())
        return (-score[tup], len(tup), tup[-1], key(tup[:-1]))

    order = sorted(score, key=key)[: budget + 1]
    pos = {t: i for i, t in enumerate(order)}
    tokens = [root] + [int(ids[len(t) - 1, t[-1]]) for t in order[1:]]
    parents = [-1] + [pos[t[:-1]] for t in order[1:]]
    depths = [len(t) for t in order]
    return tokens, parents, depths


def _random_logp(g, D, K, mode):
    if mode == "cont":
        x = -np.sort(g.exponential(1.0, (D, K)), axis=1)
    else:  # exact binary values, many ties, zeros included
        x = -np.sort(g.choice([0.0, 0.5, 1.0, 2.0], (D, K)), axis=1)
    return np.ascontiguousarray(x[:, ::-1][:, ::-1]).astype(np.float32)


@pytest.mark.parametrize("mode", ["cont", "ties"])
@pytest.mark.parametrize("D,K", [(1, 1), (1, 4), (2, 2), (2, 3), (3, 2), (3, 3), (4, 2), (2, 4)])
def test_heap_equals_exhaustive_enumeration(mode, D, K):
    g = np.random.default_rng([D, K, 0 if mode == "cont" else 1])
    total = sum(K ** d for d in range(D + 1))
    for trial in range(6):
        logp = _random_logp(g, D, K, mode)
        assert (np.diff(logp, axis=1) <= 0).all()
        ids = g.integers(0, 1000, (D, K)).astype(np.int32)
        for budget in sorted({0, min(1, total - 1), min(2, total - 1), total // 2, total - 1}):
            t = O.build_one(logp, ids, 7, budget, 1000)
            bt, bp, bd = brute_force(logp, ids, 7, budget)
            assert t["tokens"] == bt
            assert t["parents"] == bp
            assert t["depths"] == bd
            assert t["n_nodes"] == budget + 1


def check_invariants(t, Q, ids):
    n = t["n_nodes"]
    for c in range(1, n):
        p = t["parents"][c]
        assert 0 <= p < c
        assert t["depths"][c] == t["depths"][p] + 1
        assert t["score"][c] <= t["score"][c - 1]  # pop order is best-first
    for c in range(Q):
        a = t["anc"][c]
        assert (a >> c) & 1                      # reflexive
        assert a < (1 << (c + 1))                # lower triangular
        p = t["parents"][c]
        if p >= 0:
            assert t["anc"][p] & a == t["anc"][p]  # transitive: parent's set inside
        if c < n:
            assert bin(a).count("1") == t["depths"][c] + 1
        else:
            assert a == 1 << c and t["depths"][c] == -1 and t["parents"][c] == -1
    for c in range(Q):
        kids = [x for x in range(Q) if t["parents"][x] == c]
        assert t["first_child"][c] == (kids[0] if kids else -1)
        p = t["parents"][c]
        sibs = [x for x in range(c + 1, Q) if p >= 0 and t["parents"][x] == p]
        assert t["next_sibling"][c] == (sibs[0] if sibs else -1)
    # siblings under one parent carry distinct tokens (top-k ids are distinct)
    for c in range(n):
        kids = [x for x in range(n) if t["parents"][x] == c]
        assert len({t["tokens"][x] for x in kids}) == len(kids)


@pytest.mark.parametrize("cfg", ["c1", "c2", "c3", "c4"])
def test_invariants_on_workload_drafters(cfg):
    w = WL.CONFIGS[cfg]
    if w.V > 4096:
        w = w.with_(V=4096)  # same shapes, smaller vocabulary keeps this fast
    for b in range(min(w.B, 4)):
        logp, ids = WL.drafter_topk(w, b)
        t = O.build_one(logp, ids, WL.root_token(w, b), w.budget, w.V)
        assert t["n_nodes"] == w.Q
        check_invariants(t, w.Q, ids)


def test_deep_boosted_drafter_pops_the_rank0_chain_first():
    w = WL.CONFIGS["c4"].with_(V=8192)
    logp, ids = WL.drafter_topk(w, 0)
    t = O.build_one(logp, ids, 0, w.budget, w.V)
    assert t["parents"][1:16] == list(range(15))
    assert t["depths"][1:16] == list(range(1, 16))
    assert t["tokens"][1:16] == [int(ids[d, 0]) for d in range(15)]


def test_k1_is_a_chain():
    D = 6
    logp = -np.arange(1, D + 1, dtype=np.float32).reshape(D, 1) / 3
    ids = np.arange(D, dtype=np.int32).reshape(D, 1) + 100
    t = O.build_one(logp, ids, 1, 9, 1000)
    assert t["parents"][: D + 1] == [-1] + list(range(D))
    assert t["depths"][: D + 1] == list(range(D + 1))
    assert t["n_nodes"] == D + 1 and t["status"] == O.ST_BUDGET_PAD


def test_d1_is_a_star_of_the_first_ranks():
    K = 8
    logp = np.sort(-np.random.default_rng(3).random((1, K)).astype(np.float32), axis=1)[:, ::-1]
    logp = np.ascontiguousarray(logp)
    ids = np.arange(K, dtype=np.int32).reshape(1, K) + 50
    t = O.build_one(logp, ids, 1, 5, 1000)
    assert t["parents"] == [-1] + [0] * 5
    assert t["tokens"] == [1] + [50 + r for r in range(5)]


def test_budget0_is_root_only():
    logp = np.full((3, 3), -1, np.float32)
    ids = np.zeros((3, 3), np.int32)
    t = O.build_one(logp, ids, 42, 0, 100)
    assert t["tokens"] == [42] and t["parents"] == [-1] and t["n_nodes"] == 1
    assert t["status"] == 0 and t["anc"] == [1]


@pytest.mark.parametrize("bad", ["nan", "inf", "token_hi", "token_neg", "root"])
def test_input_errors_give_root_only(bad):
    logp = np.full((2, 2), -1, np.float32)
    ids = np.array([[1, 2], [3, 4]], np.int32)
    root = 0
    if bad == "nan":
        logp[1, 1] = np.nan
    elif bad == "inf":
        logp[0, 1] = -np.inf
    elif bad == "token_hi":
        ids[1, 0] = 100
    elif bad == "token_neg":
        ids[0, 0] = -1
    else:
        root = 100
    t = O.build_one(logp, ids, root, 4, 100)
    assert t["n_nodes"] == 1
    assert t["status"] == O.ST_INPUT | O.ST_BUDGET_PAD
    assert t["parents"] == [-1] * 5


def test_batched_outputs_match_per_sequence_and_bits():
    w = WL.CONFIGS["c1"]
    batch = WL.make_batch(w, latents=False)
    out = O.tree_build(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
    t = O.build_one(batch.topk_logp[0], batch.topk_ids[0], int(batch.root_tok[0]), w.budget, w.V)
    assert list(out["tokens"][0]) == t["tokens"]
    for n in range(w.Q):
        word = int(out["vis_bits"][0, n, 0])
        assert word == t["anc"][n]
        assert [int(out["vis"][0, n, j]) for j in range(w.Q)] == \
            [(t["anc"][n] >> j) & 1 for j in range(w.Q)]


def test_two_word_masks_at_q65():
    w = WL.CONFIGS["c2"].with_(V=4096)
    logp, ids = WL.drafter_topk(w, 0)
    out = O.tree_build(logp[None], ids[None], np.array([0]), 64, w.V)
    assert out["vis_bits"].shape == (1, 65, 2)
    # node 64 is visible to itself through bit 0 of word 1
    assert int(out["vis_bits"][0, 64, 1]) & 1 == 1
    assert math.isclose(float(out["score"][0, 0]), 0.0)
