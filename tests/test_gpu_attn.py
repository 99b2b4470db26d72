"""GPU verify attention (ddt_verify_attn through the C ABI) against the
float64 oracle: fp32 path within max rel err 1e-5 per query row, bf16
tensor-core path within max abs err 2e-2; edge cases (empty prefix, ragged
key tails, paging, forced key-range splits, capacity and page errors)."""
import math

import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import latent_tensor, rel_err_rows, t, to_f64

pytestmark = pytest.mark.gpu

F32_REL = 1e-5
BF16_ABS = 2e-2


def run_case(w, batch=None, rows=None, max_len=None, check=True):
    batch = batch or WL.make_batch(w)
    tree = O.tree_build(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
    lay = batch.layout
    q_lat = latent_tensor(batch.q_lat, w.dtype)
    q_pe = latent_tensor(batch.q_pe, w.dtype)
    kv = latent_tensor(batch.kv, w.dtype)
    vis = t(tree["vis_bits"].view(np.int64))
    ml = max_len if max_len is not None else int(batch.prefix_len.max()) + w.Q
    out, lse, st = DB.ddt_verify_attn(q_lat, q_pe, kv, t(lay.block_table), t(batch.prefix_len),
                                      vis, w.scale, lay.page_size, ml)
    torch.cuda.synchronize()
    ref_o, ref_l, ref_st = O.verify_attention(batch.q_lat, batch.q_pe, batch.kv, lay.block_table,
                                              batch.prefix_len, tree["vis_bits"], w.scale,
                                              lay.page_size, rows=rows, with_status=True)
    got_o, got_l = to_f64(out), to_f64(lse)
    np.testing.assert_array_equal(st.cpu().numpy(), ref_st)
    if rows is not None:
        sel = tuple(np.array(rows).T)
        got_o, got_l, ref_o, ref_l = got_o[sel], got_l[sel], ref_o[sel], ref_l[sel]
    if check:
        assert np.isfinite(got_o).all()
        if w.dtype == "f32":
            assert rel_err_rows(got_o, ref_o) <= F32_REL
            np.testing.assert_allclose(got_l, ref_l, rtol=1e-5, atol=1e-5)
        else:
            assert np.abs(got_o - ref_o).max() <= BF16_ABS
            np.testing.assert_allclose(got_l, ref_l, rtol=0, atol=2e-2)
    return got_o, ref_o


# ------------------------------------------------------------------ fp32 path

def test_f32_tiny_workload_all_rows():
    run_case(WL.CONFIGS["c1"])


@pytest.mark.parametrize("budget", [0, 1, 8, 64, 127])
def test_f32_odd_dims_paged(budget):
    """Odd dims of the second validation model (6 heads, kv_lora 48)."""
    w = WL.CONFIGS["c1"].with_(H=6, C=48, R=16, prefix=(0, 70), B=3, page_size=16,
                               budget=budget, scale=WL.f32(1 / math.sqrt(64)))
    run_case(w)


def test_f32_k2_dims_q_len_1_is_decode():
    w = WL.CONFIGS["c2"].with_(dtype="f32", budget=0, prefix=777, V=2048)
    run_case(w)


# ------------------------------------------------------------------ bf16 path

@pytest.mark.parametrize("L", [0, 1, 63, 64, 65, 700])
@pytest.mark.parametrize("budget", [0, 8, 16, 64])
def test_bf16_ragged_prefixes(L, budget, attn_rows):
    w = WL.CONFIGS["c2"].with_(B=2, budget=budget, prefix=L, V=4096)
    run_case(w)


@pytest.mark.parametrize("H", [16, 128])
def test_bf16_other_head_counts(H, attn_rows):
    w = WL.CONFIGS["c2"].with_(B=2, H=H, budget=8, prefix=300, V=4096)
    run_case(w)


def test_bf16_paged_variable_lengths_forced_splits(attn_rows):
    w = WL.CONFIGS["c3"].with_(B=5, V=4096, prefix=(0, 1500))
    batch = WL.make_batch(w)
    run_case(w, batch)                      # the planner's own split
    run_case(w, batch, max_len=200000)      # many splits, some empty for short sequences
    run_case(w, batch, max_len=w.Q)         # no split at all


def test_bf16_max_budget_workload_all_rows(attn_rows):
    run_case(WL.CONFIGS["c2"])


def test_bf16_batched_paged_workload_sampled_rows(attn_rows):
    w = WL.CONFIGS["c3"]
    g = np.random.default_rng(0)
    rows = [(int(b), int(i)) for b, i in zip(g.integers(0, w.B, 24), g.integers(0, w.Q, 24))]
    rows += [(0, 0), (w.B - 1, w.Q - 1)]
    run_case(w, rows=rows)


def test_bf16_deep_long_workload_sampled_rows(attn_rows):
    w = WL.CONFIGS["c4"]
    rows = [(0, 0), (1, 15), (3, 40), (7, 64), (5, 7)]
    run_case(w, rows=rows)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_capacity_and_page_errors(dtype, attn_rows):
    base = WL.CONFIGS["c2"].with_(B=3, budget=8, prefix=100, V=4096, dtype=dtype,
                                  page_size=64)
    batch = WL.make_batch(base)
    lay = batch.layout
    batch.prefix_len = batch.prefix_len.copy()
    batch.prefix_len[1] = lay.max_pages * lay.page_size  # no room for the tree
    bt = lay.block_table.copy()
    bt[2, 0] = lay.total_rows // lay.page_size + 5         # page outside the cache
    lay.block_table = bt
    got, ref = run_case(base, batch, check=False)
    assert (got[1:] == 0).all() and (ref[1:] == 0).all()
    tol = F32_REL if dtype == "f32" else BF16_ABS
    if dtype == "f32":
        assert rel_err_rows(got[0], ref[0]) <= tol
    else:
        assert np.abs(got[0] - ref[0]).max() <= tol
