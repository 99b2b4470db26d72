"""Pins of the oracle's multi-step decode loop against what the pages state
about the native engine's generate_ddtree: with a drafter that always
proposes the right token, 8.00 tokens per verify step and 3 verify steps for
24 tokens where autoregressive decoding takes 24; and, for any drafter, the
DDTree greedy output equals the autoregressive greedy output. The
autoregressive side is a separate plain loop."""
import numpy as np
import pytest

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import workloads as WL


def case(cid, B, G, V, hit, dtype="f32"):
    golden = WL.loop_golden(cid, B, G, V)
    table = WL.loop_drafter_table(cid, golden, V, hit, dtype)
    return golden, table


def test_the_pages_oracle_drafter_numbers():
    # seven drafts + the bonus per step: 24 new tokens in 3 verify steps
    # (24 autoregressive target steps), 8.00 tokens per step
    V, D, n_new = 1024, 7, 24
    golden, table = case(1, 1, n_new + D + 1, V, hit=1.0)
    out, steps, per = O.decode_loop_table(golden[0], table[0], n_new, D=D, K=4, budget=16, V=V,
                                          max_steps=64)
    assert out == O.ar_decode(golden[0], n_new, V) == golden[0, : n_new + 1].tolist()
    assert steps == 3 and per == [8, 8, 8]
    assert sum(per) / steps == 8.0
    assert len(O.ar_decode(golden[0], n_new, V)) - 1 == 24


@pytest.mark.parametrize("hit", [0.0, 0.3, 0.7, 1.0])
@pytest.mark.parametrize("D,K,budget", [(4, 3, 8), (7, 4, 16), (6, 2, 5)])
def test_ddtree_output_equals_autoregressive_output(hit, D, K, budget):
    V, n_new = 512, 30
    golden, table = case(2, 3, n_new + D + 1, V, hit)
    for b in range(3):
        out, steps, per = O.decode_loop_table(golden[b], table[b], n_new, D, K, budget, V,
                                              max_steps=10 * n_new)
        assert out == O.ar_decode(golden[b], n_new, V)
        assert len(per) == steps and sum(per) >= n_new
        # every step commits at least the bonus and at most D drafts + bonus,
        # and never more drafts than the tree holds
        assert all(1 <= k <= min(D, budget) + 1 for k in per)
        if hit == 1.0:
            assert all(k == min(D, budget) + 1 for k in per[:-1])


def test_a_silent_drafter_still_decodes_exactly():
    # no spike anywhere: most steps commit the bonus alone
    V, n_new, D = 256, 20, 5
    golden, table = case(3, 1, n_new + D + 1, V, hit=0.0)
    out, steps, per = O.decode_loop_table(golden[0], table[0], n_new, D, 3, 8, V, max_steps=100)
    assert out == golden[0, : n_new + 1].tolist()
    assert steps <= n_new


def test_the_step_bound_stops_the_loop():
    V, D = 512, 4
    golden, table = case(4, 1, 64, V, hit=1.0)
    out, steps, per = O.decode_loop_table(golden[0], table[0], 50, D, 2, 6, V, max_steps=2)
    assert steps == 2 and per == [5, 5]
    assert out == golden[0, :11].tolist()


def test_drafter_table_puts_the_stream_token_first_on_a_hit():
    V = 300
    golden, table = case(5, 2, 12, V, hit=1.0, dtype="bf16")
    assert (table.argmax(axis=-1) == golden).all()
    assert np.array_equal(WL.round_bf16(table), table)
