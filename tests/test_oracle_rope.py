"""Pins of the oracle's rotary embedding and cache append at tree positions.

The rotation is pinned by closed forms (cos 1 and sin 1, written out as
numbers), by frequencies chosen so that every pair turns by exactly one
radian, and by the properties that make it a rotary embedding (pair norms
kept, rotations compose, dot products depend only on the position
difference). The append is pinned on a hand-worked paged example."""
import math

import numpy as np
import pytest

from oracle import ddt_oracle as O

COS1 = 0.5403023058681398
SIN1 = 0.8414709848078965


def test_position_zero_is_the_identity():
    g = np.random.default_rng(0)
    for R in (2, 8, 64):
        x = g.standard_normal((3, R))
        assert np.array_equal(O.rope_neox(x, 0, 10000.0), x)


def test_width_two_turns_by_the_position_in_radians():
    # R = 2: one pair, frequency theta**0 = 1
    assert np.allclose(O.rope_neox([1.0, 0.0], 1, 10000.0), [COS1, SIN1], rtol=0, atol=1e-15)
    assert np.allclose(O.rope_neox([0.0, 1.0], 1, 10000.0), [-SIN1, COS1], rtol=0, atol=1e-15)


def test_neox_pairs_i_with_i_plus_half():
    # R = 4, theta = 10000: frequencies [1, 10000**-0.5 = 0.01]; position 100
    # turns pair 1 = (x1, x3) by one radian and pair 0 = (x0, x2) by 100
    y = O.rope_neox([0.0, 1.0, 0.0, 0.0], 100, 10000.0)
    assert np.allclose(y, [0.0, COS1, 0.0, SIN1], rtol=0, atol=1e-14)
    y = O.rope_neox([0.0, 0.0, 0.0, 1.0], 100, 10000.0)
    assert np.allclose(y, [0.0, -SIN1, 0.0, COS1], rtol=0, atol=1e-14)
    y = O.rope_neox([1.0, 0.0, 0.0, 0.0], 1, 10000.0)
    assert np.allclose(y, [COS1, 0.0, SIN1, 0.0], rtol=0, atol=1e-15)


def test_frequency_of_pair_i_is_theta_to_minus_2i_over_R():
    # R = 8, theta = 16: frequencies 16**(-2i/8) = 2**-i, so position 2**i
    # turns pair i by exactly one radian
    R = 8
    for i in range(R // 2):
        x = np.zeros(R)
        x[i] = 1.0
        want = np.zeros(R)
        want[i], want[i + R // 2] = COS1, SIN1
        assert np.allclose(O.rope_neox(x, 2 ** i, 16.0), want, rtol=0, atol=1e-14), i


def test_rotation_properties():
    g = np.random.default_rng(1)
    R, theta = 64, 10000.0
    x = g.standard_normal((5, R))
    k = g.standard_normal((5, R))
    y = O.rope_neox(x, 37, theta)
    h = R // 2
    assert np.allclose(y[:, :h] ** 2 + y[:, h:] ** 2, x[:, :h] ** 2 + x[:, h:] ** 2, rtol=1e-13)
    # turning by a then by b is turning by a + b
    assert np.allclose(O.rope_neox(O.rope_neox(x, 11, theta), 26, theta), y, rtol=0, atol=1e-12)
    # q . k depends on the positions only through their difference
    d1 = np.sum(O.rope_neox(x, 100, theta) * O.rope_neox(k, 93, theta), axis=-1)
    d2 = np.sum(O.rope_neox(x, 4007, theta) * O.rope_neox(k, 4000, theta), axis=-1)
    assert np.allclose(d1, d2, rtol=1e-9, atol=1e-9)


def _case(prefix, block_table, depths, rows=8, page_size=2, H=2, C=3, R=4, seed=2):
    g = np.random.default_rng(seed)
    B, Q = len(prefix), len(depths[0])
    q_pe = g.standard_normal((B, Q, H, R))
    kv_new = g.standard_normal((B, Q, C + R))
    kv = g.standard_normal((rows, C + R))
    out = O.rope_append(q_pe, kv_new, kv, np.array(block_table), np.array(prefix), np.array(depths),
                        page_size, 10000.0)
    return q_pe, kv_new, kv, out


def test_append_lands_on_the_paged_slots():
    # page_size 2, pages [3, 0, 1], L = 1, Q = 3: slots 1, 2, 3 live in
    # physical rows 3*2+1 = 7, 0*2+0 = 0 and 0*2+1 = 1
    q_pe, kv_new, kv, (q_out, kv_out, st) = _case([1], [[3, 0, 1]], [[0, 1, -1]])
    assert st.tolist() == [O.ST_OK]
    want_rows = [7, 0, 1]
    untouched = [r for r in range(kv.shape[0]) if r not in want_rows]
    assert np.array_equal(kv_out[untouched], kv[untouched])
    C = 3
    for t, (r, p) in enumerate(zip(want_rows, [1, 2, 1])):  # padding slot: position L
        assert np.array_equal(kv_out[r, :C], kv_new[0, t, :C])
        assert np.allclose(kv_out[r, C:], O.rope_neox(kv_new[0, t, C:], p, 10000.0), atol=1e-15)
        for h in range(q_pe.shape[2]):
            assert np.allclose(q_out[0, t, h], O.rope_neox(q_pe[0, t, h], p, 10000.0), atol=1e-15)


def test_root_slot_keeps_its_position_L():
    # depth 0 at L: the rotation is by L, so at L = 0 the root is unchanged
    q_pe, kv_new, kv, (q_out, kv_out, st) = _case([0], [[2, 3]], [[0, 1]])
    assert np.array_equal(q_out[0, 0], q_pe[0, 0])
    assert np.array_equal(kv_out[4], kv_new[0, 0])


@pytest.mark.parametrize("prefix,table,bit", [
    ([-1], [[0, 1]], O.ST_CAPACITY),     # negative length
    ([3], [[0, 1]], O.ST_CAPACITY),      # slots 3..4 past the two pages of 2
    ([1], [[0, 9]], O.ST_RANGE),         # page 9 is outside the 8-row cache
])
def test_bad_sequences_are_left_untouched(prefix, table, bit):
    q_pe, kv_new, kv, (q_out, kv_out, st) = _case(prefix, table, [[0, 1]])
    assert st.tolist() == [bit]
    assert np.array_equal(kv_out, kv)
    assert np.isnan(q_out).all()


def test_a_bad_sequence_does_not_stop_the_others():
    _, kv_new, kv, (q_out, kv_out, st) = _case([1, 5], [[0, 1], [2, 3]], [[0, 1], [0, 1]],
                                               page_size=2)
    assert st.tolist() == [O.ST_OK, O.ST_CAPACITY]
    assert not np.isnan(q_out[0]).any() and np.isnan(q_out[1]).all()
    assert np.array_equal(kv_out[1, :3], kv_new[0, 0, :3])  # slot 1 of sequence 0
    assert math.isfinite(float(kv_out[2, 0]))
