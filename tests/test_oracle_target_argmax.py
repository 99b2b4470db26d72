"""Pins of the oracle's target-side argmax (the greedy token at every tree
slot): a plain Python scan on small inputs (ties, signed zeros, infinities,
NaN), and logits built so that the winner is known."""
import math

import numpy as np

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import workloads as WL


def scan_argmax(row) -> int:
    """First index of the maximum, NaN above every number, -0.0 == +0.0."""
    best, bi = None, 0
    for i, v in enumerate(row):
        v = float(v)
        if best is None:
            best, bi = v, i
            continue
        if math.isnan(best):
            continue
        if math.isnan(v) or v > best:
            best, bi = v, i
    return bi


def test_matches_a_plain_scan_on_tie_heavy_rows():
    g = np.random.default_rng(3)
    for V in (1, 2, 7, 33, 100):
        x = g.choice(np.array([-np.inf, -2.0, -0.0, 0.0, 1.5, 1.5, np.inf]), size=(20, V))
        x = x.astype(np.float32)
        got = O.target_argmax(x)
        for r in range(x.shape[0]):
            assert got[r] == scan_argmax(x[r]), (V, r, x[r])


def test_nan_is_the_largest_and_the_first_nan_wins():
    x = np.array([[1.0, np.nan, 5.0, np.nan], [np.inf, 3.0, np.nan, 0.0]], np.float32)
    assert O.target_argmax(x).tolist() == [1, 2]
    assert [scan_argmax(r) for r in x] == [1, 2]


def test_signed_zeros_tie():
    x = np.array([[-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]], np.float32)
    assert O.target_argmax(x).tolist() == [0, 0]


def test_known_winner_of_the_synthetic_target_logits():
    w = WL.CONFIGS["c2"].with_(V=4096)
    winners = np.random.default_rng(5).integers(0, w.V, w.Q)
    x = WL.target_logits(w, 0, winners)
    assert np.array_equal(O.target_argmax(x), winners.astype(np.int32))
    # and it agrees with the scan on the rows as generated (bf16-rounded)
    for r in range(0, w.Q, 16):
        assert O.target_argmax(x[r]) == scan_argmax(x[r])
