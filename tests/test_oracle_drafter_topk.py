"""Pins of the oracle's drafter top-K (log-softmax over the vocabulary, then
the K best candidates): a plain Python sort with math.fsum log-sum-exp on
small rows, tie-heavy rows, known closed forms, and the invariants the tree
builder relies on (descending log-probs, distinct ids, log-probs <= 0)."""
import math

import numpy as np
import pytest

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import workloads as WL


def plain_topk(row, K):
    vals = [float(v) for v in row]
    order = sorted(range(len(vals)), key=lambda i: (-vals[i], i))[:K]
    m = max(vals)
    lse = m + math.log(math.fsum(math.exp(v - m) for v in vals))
    return [vals[i] - lse for i in order], order


@pytest.mark.parametrize("V,K", [(1, 1), (5, 3), (64, 8), (300, 16), (1000, 4)])
def test_matches_a_plain_sort_and_fsum(V, K):
    g = np.random.default_rng(V * 31 + K)
    x = g.normal(0, 2, (6, V)).astype(np.float32)
    logp, ids = O.drafter_topk(x, K)
    for r in range(x.shape[0]):
        lp, o = plain_topk(x[r], min(K, V))
        assert ids[r].tolist()[: len(o)] == o
        np.testing.assert_allclose(logp[r][: len(o)], np.array(lp, np.float32), rtol=0, atol=1e-6)


def test_ties_go_to_the_lower_id():
    x = np.array([[1.0, 3.0, 3.0, 0.0, 3.0, 2.0, 2.0]], np.float32)
    logp, ids = O.drafter_topk(x, 5)
    assert ids[0].tolist() == [1, 2, 4, 5, 6]
    assert logp[0][0] == logp[0][1] == logp[0][2]


def test_closed_forms():
    # uniform logits: every log-prob is -log V, ids 0..K-1
    V = 4096
    logp, ids = O.drafter_topk(np.full((2, V), 0.75, np.float32), 4)
    assert ids[0].tolist() == [0, 1, 2, 3]
    np.testing.assert_allclose(logp, -math.log(V), rtol=0, atol=1e-6)
    # one logit far above the rest: log-prob ~ 0
    x = np.zeros((1, 100), np.float32)
    x[0, 42] = 60.0
    logp, ids = O.drafter_topk(x, 1)
    assert ids[0, 0] == 42 and abs(logp[0, 0]) < 1e-20 + 1e-6


def test_builder_invariants_on_workload_rows():
    w = WL.CONFIGS["c2"].with_(V=8192)
    x = WL.drafter_logits(w, 0)
    logp, ids = O.drafter_topk(x, w.K)
    assert (np.diff(logp, axis=-1) <= 0).all() and (logp <= 0).all()
    for r in range(w.D):
        assert len(set(ids[r].tolist())) == w.K
        assert (x[r][ids[r]] == np.sort(x[r])[::-1][: w.K]).all()
