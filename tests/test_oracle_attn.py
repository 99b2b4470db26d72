"""Pins of the oracle's verify attention: q_len = 1 equals plain decode
attention (torch's float64 SDPA), each tree node equals brute-force attention
over its prefix plus ancestor path, closed forms, layout invariance."""
import math

import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import workloads as WL


def _single(L, H, C, R, seed, budget=0, paged=False):
    g = np.random.default_rng(seed)
    Q = budget + 1
    q = g.standard_normal((1, Q, H, C + R))
    kv = g.standard_normal((L + Q, C + R))
    if paged:
        P = 4
        pages = -(-(L + Q) // P)
        perm = g.permutation(pages + 3)[:pages]
        phys = np.zeros(((pages + 3) * P, C + R))
        for s in range(L + Q):
            phys[perm[s // P] * P + s % P] = kv[s]
        return q, kv, phys, perm.reshape(1, -1).astype(np.int32), P
    return q, kv, kv, np.zeros((1, 1), np.int32), L + Q


@pytest.mark.parametrize("L", [0, 1, 7, 64, 333])
def test_qlen1_is_plain_decode_attention(L):
    H, C, R = 4, 16, 8
    q, kv, phys, bt, P = _single(L, H, C, R, seed=L)
    scale = WL.f32(1 / math.sqrt(C + R))
    vis = np.ones((1, 1, 1), np.uint64)
    o, lse = O.verify_attention(q[..., :C], q[..., C:], phys, bt, np.array([L]), vis, scale, P)
    # MQA: one latent KV head broadcast to all query heads, key dim C+R, value dim C
    qt = torch.tensor(q[0, 0], dtype=torch.float64).reshape(1, H, 1, C + R)
    kt = torch.tensor(kv, dtype=torch.float64).reshape(1, 1, L + 1, C + R).expand(1, H, L + 1, C + R)
    vt = torch.tensor(kv[:, :C], dtype=torch.float64).reshape(1, 1, L + 1, C).expand(1, H, L + 1, C)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=float(scale))
    np.testing.assert_allclose(o[0, 0], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)
    s = (q[0, 0] @ kv.T) * float(scale)
    np.testing.assert_allclose(lse[0, 0], np.log(np.exp(s).sum(1)), rtol=1e-12)


def test_every_tree_node_equals_brute_force_over_its_ancestor_path():
    w = WL.CONFIGS["c1"]
    logp, ids = WL.drafter_topk(w, 0)
    tree = O.tree_build(logp[None], ids[None], np.array([5]), w.budget, w.V)
    H, C, R, L, Q = 2, 6, 3, 5, w.Q
    g = np.random.default_rng(9)
    q = g.standard_normal((1, Q, H, C + R))
    kv = g.standard_normal((L + Q, C + R))
    scale = 0.37
    o, lse = O.verify_attention(q[..., :C], q[..., C:], kv, np.zeros((1, 1), np.int32),
                                np.array([L]), tree["vis_bits"], scale, L + Q)
    sc = float(np.float32(scale))
    for i in range(Q):
        # ancestors of i (itself included) by walking parent pointers
        path = []
        c = i
        while c >= 0:
            path.append(c)
            c = int(tree["parents"][0, c])
        slots = list(range(L)) + sorted(L + t for t in path)
        for h in range(H):
            scores = []
            for j in slots:
                acc = 0.0
                for d in range(C + R):
                    acc += float(q[0, i, h, d]) * float(kv[j, d])
                scores.append(acc * sc)
            mx = max(scores)
            ws = [math.exp(s - mx) for s in scores]
            tot = sum(ws)
            for d in range(C):
                ref = sum(wt * float(kv[j, d]) for wt, j in zip(ws, slots)) / tot
                assert abs(o[0, i, h, d] - ref) < 1e-12
            assert abs(lse[0, i, h] - (mx + math.log(tot))) < 1e-12


def test_zero_query_gives_mean_of_visible_values():
    L, H, C, R, Q = 10, 3, 8, 4, 9
    g = np.random.default_rng(1)
    kv = g.standard_normal((L + Q, C + R))
    q = np.zeros((1, Q, H, C + R))
    w = WL.CONFIGS["c1"]
    logp, ids = WL.drafter_topk(w, 0)
    tree = O.tree_build(logp[None], ids[None], np.array([5]), Q - 1, w.V)
    o, lse = O.verify_attention(q[..., :C], q[..., C:], kv, np.zeros((1, 1), np.int32),
                                np.array([L]), tree["vis_bits"], 1.0, L + Q)
    for i in range(Q):
        vis = O.visible_tree_slots(tree["vis_bits"][0, i], Q)
        rows = list(range(L)) + [L + t for t in range(Q) if vis[t]]
        np.testing.assert_allclose(o[0, i], np.broadcast_to(kv[rows, :C].mean(0), (H, C)),
                                   rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[0, i], math.log(len(rows)), rtol=1e-13)


def test_single_visible_key_returns_its_value():
    H, C, R = 2, 4, 4
    g = np.random.default_rng(2)
    kv = g.standard_normal((1, C + R))
    q = g.standard_normal((1, 1, H, C + R))
    o, lse = O.verify_attention(q[..., :C], q[..., C:], kv, np.zeros((1, 1), np.int32),
                                np.array([0]), np.ones((1, 1, 1), np.uint64), 0.5, 1)
    np.testing.assert_array_equal(o[0, 0], np.broadcast_to(kv[0, :C], (H, C)))
    np.testing.assert_allclose(lse[0, 0], (q[0, 0] @ kv[0]) * 0.5, rtol=1e-14)


def test_paged_layout_gives_the_same_numbers_as_contiguous():
    H, C, R, L = 2, 8, 4, 21
    q, kv, phys, bt, P = _single(L, H, C, R, seed=5, budget=3, paged=True)
    vis = np.array([[[1], [3], [5], [9]]], np.uint64)
    o1, l1 = O.verify_attention(q[..., :C], q[..., C:], phys, bt, np.array([L]), vis, 0.3, P)
    o2, l2 = O.verify_attention(q[..., :C], q[..., C:], kv, np.zeros((1, 1), np.int32),
                                np.array([L]), vis, 0.3, L + 4)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_scale_is_taken_as_float32():
    """The kernels receive the scale as a float32; the oracle must upcast that
    exact value, not the decimal it came from."""
    H, C, R, L = 1, 4, 2, 3
    q, kv, phys, bt, P = _single(L, H, C, R, seed=8)
    vis = np.ones((1, 1, 1), np.uint64)
    s64 = 1 / math.sqrt(3.0)
    _, lse = O.verify_attention(q[..., :C], q[..., C:], phys, bt, np.array([L]), vis, s64, P)
    s = (q[0, 0] @ kv.T) * float(np.float32(s64))
    np.testing.assert_allclose(lse[0, 0], np.log(np.exp(s).sum(1)), rtol=1e-14)


def test_capacity_and_page_range_errors_zero_the_sequence():
    H, C, R, Q = 2, 4, 4, 3
    g = np.random.default_rng(4)
    kv = g.standard_normal((32, C + R))
    q = g.standard_normal((3, Q, H, C + R))
    bt = np.array([[0, 1], [2, 3], [1, 9]], np.int32)  # page 9 is outside a 4-page cache
    L = np.array([5, 14, 7], np.int32)  # 14 + 3 > 2 pages * 8 slots; 7 + 3 reaches page 9
    vis = np.tile(np.array([1, 3, 5], np.uint64).reshape(1, Q, 1), (3, 1, 1))
    o, lse, st = O.verify_attention(q[..., :C], q[..., C:], kv, bt, L, vis, 0.5, 8,
                                    with_status=True)
    assert list(st) == [0, O.ST_CAPACITY, O.ST_RANGE]
    assert (o[1:] == 0).all() and np.isneginf(lse[1:]).all()
    assert np.isfinite(o[0]).all()
