"""One whole verify step (ddt_step through the C ABI: build -> verify
attention -> accept + compaction) against the oracle on the workload
shapes: tree, accept and the compacted cache bit for bit, attention within
its tolerance."""
import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import latent_tensor, rel_err_rows, t, to_f64, u64

pytestmark = pytest.mark.gpu


def make_step(w, batch, target):
    lay = batch.layout
    dt = DB.DDT_BF16 if w.dtype == "bf16" else DB.DDT_F32
    max_len = int(batch.prefix_len.max()) + w.Q
    buf = DB.StepBuffers(w.B, w.D, w.K, w.budget, w.V, w.H, w.C, w.R, lay.page_size,
                         lay.max_pages, lay.total_rows, dt, w.scale, max_len, with_vis=True)
    buf.topk_logp.copy_(t(batch.topk_logp))
    buf.topk_ids.copy_(t(batch.topk_ids))
    buf.root_tok.copy_(t(batch.root_tok))
    buf.q_lat.copy_(latent_tensor(batch.q_lat, w.dtype))
    buf.q_pe.copy_(latent_tensor(batch.q_pe, w.dtype))
    buf.kv_cache.copy_(latent_tensor(batch.kv, w.dtype))
    buf.block_table.copy_(t(lay.block_table))
    buf.prefix_len.copy_(t(batch.prefix_len))
    buf.target_argmax.copy_(t(target))
    return buf


def kv_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return WL.to_bf16_bits(x).view(np.int16)
    return np.ascontiguousarray(x, np.float32).view(np.int32)


def check_step(w, rows=None, batch=None):
    batch = batch if batch is not None else WL.make_batch(w)
    lay = batch.layout
    ref = O.ddt_step(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V, batch.q_lat,
                     batch.q_pe, batch.kv, lay.block_table, batch.prefix_len, w.scale,
                     lay.page_size, lay.max_pages,
                     lambda tr: WL.target_argmax_for(batch, tr["depths"]), attn_rows=rows)
    buf = make_step(w, batch, ref["target"])
    DB.ddt_step(buf)
    torch.cuda.synchronize()
    tree = ref["tree"]
    for k in ("tokens", "parents", "depths", "first_child", "next_sibling", "n_nodes"):
        np.testing.assert_array_equal(getattr(buf, k).cpu().numpy(), tree[k], err_msg=k)
    np.testing.assert_array_equal(u64(buf.vis_bits), tree["vis_bits"])
    np.testing.assert_array_equal(buf.vis.cpu().numpy(), tree["vis"])
    acc = ref["accept"]
    for k in ("accept_idx", "accept_len", "out_tokens", "bonus"):
        np.testing.assert_array_equal(getattr(buf, k).cpu().numpy(), acc[k], err_msg=k)
    np.testing.assert_array_equal(buf.new_len.cpu().numpy(), ref["new_len"])
    np.testing.assert_array_equal(buf.status.cpu().numpy(), ref["status"])
    got_kv = buf.kv_cache.view(torch.int16 if w.dtype == "bf16" else torch.int32).cpu().numpy()
    np.testing.assert_array_equal(got_kv, kv_bits(ref["kv"], w.dtype))
    got_o = to_f64(buf.out)
    ref_o = ref["o"]
    if rows is not None:
        sel = tuple(np.array(rows).T)
        got_o, ref_o = got_o[sel], ref_o[sel]
    if w.dtype == "f32":
        assert rel_err_rows(got_o, ref_o) <= 1e-5
    else:
        assert np.abs(got_o - ref_o).max() <= 2e-2
    return ref


def test_step_tiny_f32():
    check_step(WL.CONFIGS["c1"])


def test_step_max_budget(attn_rows):
    check_step(WL.CONFIGS["c2"])


def test_step_batched_paged(attn_rows):
    g = np.random.default_rng(1)
    w = WL.CONFIGS["c3"]
    rows = [(int(b), int(i)) for b, i in zip(g.integers(0, w.B, 16), g.integers(0, w.Q, 16))]
    check_step(w, rows=rows)


def test_step_deep_long_accepts_15_and_compacts(attn_rows):
    w = WL.CONFIGS["c4"]
    ref = check_step(w, rows=[(0, 0), (2, 15), (7, 64)])
    assert (ref["accept"]["accept_len"] == 15).all()


@pytest.mark.parametrize("q_len,B,L", [(1, 8, 1024), (9, 64, 1024), (33, 1, 8192),
                                       (65, 8, 8192), (17, 1, 131072), (1, 8, 131072),
                                       (65, 64, 8192), (33, 8, 65536)])
def test_step_sweep_points(q_len, B, L, attn_rows):
    w = WL.sweep_point(q_len, B, L)
    # rows spread over sequences and over the row tiles (query positions) and
    # key ranges of the launch
    rows = sorted({(0, 0), (B - 1, q_len - 1), (B // 2, q_len // 2), (min(1, B - 1), q_len // 4),
                   (max(B - 2, 0), (3 * q_len) // 4)})
    check_step(w, rows=rows)


# ---- the bf16 step builds the tree inside the attention kernel when the
# candidate table is small; these cover that path's edges and the fallback

def test_step_bf16_large_candidate_table_runs_build_and_attention_apart(attn_rows):
    # min(D, budget) * min(K, budget) = 1600 candidates: over the fused limit
    w = WL.CONFIGS["c2"].with_(D=40, K=40, V=4096, prefix=300)
    check_step(w, rows=[(0, 0), (0, 33), (0, 64)])


def test_step_fused_build_with_invalid_drafter_input(attn_rows):
    w = WL.CONFIGS["c2"].with_(B=3, V=4096, prefix=(70, 300))
    batch = WL.make_batch(w)
    batch.topk_logp = batch.topk_logp.copy()
    batch.topk_ids = batch.topk_ids.copy()
    batch.topk_logp[1, 2, 3] = np.nan      # sequence 1: the root alone, ST_INPUT
    batch.topk_ids[2, 0, 0] = w.V + 5      # sequence 2 likewise
    ref = check_step(w, rows=[(0, 5), (1, 0), (2, 64)], batch=batch)
    assert (ref["status"][1:] & O.ST_INPUT).all() and not ref["status"][0] & O.ST_INPUT


def test_step_fused_build_when_a_sequence_cannot_be_attended(attn_rows):
    # sequence 1 has no room for the tree (capacity error): no cluster attends
    # it, yet its tree is still built and written
    w = WL.CONFIGS["c2"].with_(B=3, budget=8, prefix=100, V=4096, page_size=64)
    batch = WL.make_batch(w)
    batch.prefix_len = batch.prefix_len.copy()
    batch.prefix_len[1] = batch.layout.max_pages * batch.layout.page_size
    ref = check_step(w, rows=[(0, 0), (1, 3), (2, 8)], batch=batch)
    assert ref["status"][1] & O.ST_CAPACITY


def test_step_fused_build_short_prefixes_every_tile_holds_tree_keys(attn_rows):
    # prefixes under one key tile: every cluster waits for the tree at once
    w = WL.CONFIGS["c2"].with_(B=4, V=4096, prefix=(0, 60))
    check_step(w, rows=[(0, 0), (1, 64), (3, 17), (2, 40)])


def test_step_fused_build_budget_zero_and_one(attn_rows):
    for budget in (0, 1):
        w = WL.CONFIGS["c2"].with_(B=2, V=4096, budget=budget, prefix=(64, 200))
        check_step(w)
