"""Checks of the seeded input generators (shared by the oracle tests and the
CUDA path; they hold no verify-step arithmetic)."""
import numpy as np
import torch

from tree_speculative_decoding_ddt_gb300 import workloads as WL


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1e-40, 3.0e38, -3.0e38, np.inf, -np.inf], np.float32)])
    ours = WL.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(WL.bf16_bits_to_f32(ours),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_stable_topk_matches_full_sort():
    g = np.random.default_rng(1)
    for trial in range(20):
        x = g.integers(-5, 5, 200).astype(np.float64)  # many ties
        k = int(g.integers(1, 20))
        full = np.lexsort((np.arange(200), -x))[:k]
        np.testing.assert_array_equal(WL._topk_stable(x, k), full)


def test_drafter_rows_are_sorted_logprobs_with_distinct_ids():
    w = WL.CONFIGS["c3"].with_(V=8192)
    logp, ids = WL.drafter_topk(w, 3)
    assert (np.diff(logp, axis=1) <= 0).all() and (logp <= 0).all()
    for d in range(w.D):
        assert len(set(ids[d].tolist())) == w.K


def test_subsets_regenerate_identically():
    w = WL.CONFIGS["c4"].with_(V=4096)
    a = WL.cache_latents(w, 3, 9000)
    b = WL.cache_latents(w, 3, 100, first=4090)
    np.testing.assert_array_equal(a[4090:4190], b)
    l1, i1 = WL.drafter_topk(w, 5)
    l2, i2 = WL.drafter_topk(w, 5)
    np.testing.assert_array_equal(l1, l2)
    np.testing.assert_array_equal(i1, i2)


def test_paged_layout_covers_every_slot_once():
    w = WL.CONFIGS["c3"]
    lens = WL.prefix_lengths(w)
    lay = WL.cache_layout(w, lens)
    seen = set()
    for b in range(w.B):
        rows = lay.rows_of(b, np.arange(int(lens[b]) + w.Q))
        assert len(set(rows.tolist())) == len(rows)
        assert not seen & set(rows.tolist())
        seen |= set(rows.tolist())
    assert max(seen) < lay.total_rows
    assert lens.min() >= 512 and lens.max() <= 8192
