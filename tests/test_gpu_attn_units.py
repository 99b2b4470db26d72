"""The 256-row verify attention with few clusters, each walking many units.

The paired-SM kernel keeps at most as many clusters as are resident at once
and each cluster takes a list of units (sequence, row tile, key range) one
after another, carrying every barrier's phase from unit to unit. At the
workload sizes most clusters hold one to nine units; here DDT_PAIR_CLUSTERS
caps a launch at one to three clusters, so that one cluster walks units of
odd and even tile counts, units with nothing to attend (empty key ranges,
capacity and page errors), split key ranges, the phantom last block, rows
that stop inside a warp, and the fused tree build, in every order the unit
list gives. Outputs are compared with the float64 oracle as in the other
attention tests.
"""
import numpy as np
import pytest

from tree_speculative_decoding_ddt_gb300 import workloads as WL
from test_gpu_attn import BF16_ABS, run_case
from test_gpu_step import check_step

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[1, 2, 3])
def few_clusters(request, monkeypatch):
    monkeypatch.setenv("DDT_VERIFY_ATTN_ROWS", "256")
    monkeypatch.setenv("DDT_PAIR_CLUSTERS", str(request.param))
    return request.param


def test_variable_lengths_paged(few_clusters):
    # 5 sequences x 5 row tiles, 1 to 13 key tiles each, lengths in any order
    w = WL.CONFIGS["c3"].with_(B=5, V=4096, prefix=(0, 1500))
    run_case(w)


def test_many_splits_some_empty(few_clusters):
    # key ranges split far past the short sequences' lengths: units with no
    # tiles sit between units with tiles
    w = WL.CONFIGS["c3"].with_(B=4, V=4096, prefix=(0, 900))
    batch = WL.make_batch(w)
    run_case(w, batch, max_len=200000)
    run_case(w, batch)


def test_capacity_and_page_errors_between_units(few_clusters):
    base = WL.CONFIGS["c2"].with_(B=4, budget=8, prefix=(100, 400), V=4096, page_size=64)
    batch = WL.make_batch(base)
    lay = batch.layout
    batch.prefix_len = batch.prefix_len.copy()
    batch.prefix_len[1] = lay.max_pages * lay.page_size  # no room for the tree
    bt = lay.block_table.copy()
    bt[2, 0] = lay.total_rows // lay.page_size + 5         # page outside the cache
    lay.block_table = bt
    got, ref = run_case(base, batch, check=False)
    assert (got[1:3] == 0).all() and (ref[1:3] == 0).all()
    for b in (0, 3):
        assert np.abs(got[b] - ref[b]).max() <= BF16_ABS


@pytest.mark.parametrize("H", [16, 48])
def test_rows_ending_inside_a_warp(H, few_clusters):
    # q_len 9: 9 * 16 = 144 and 9 * 48 = 432 rows, so a warp's 32 rows of the
    # last tile straddle the end of the sequence's rows
    w = WL.CONFIGS["c2"].with_(B=3, H=H, budget=8, prefix=(40, 500), V=4096)
    run_case(w)


@pytest.mark.parametrize("L", [0, 47, 111, 175])
def test_phantom_blocks_and_short_prefixes(L, few_clusters):
    # L + 17 keys: the last 128-key tile ends after one 64-key block for 47 and
    # 175 (a phantom second half), after two for 111; 0 is the tree alone
    w = WL.CONFIGS["c2"].with_(B=2, budget=16, prefix=L, V=4096)
    run_case(w)


def test_step_with_fused_build(few_clusters):
    # the tree of every sequence is built in the attention kernel by each unit
    # that walks tree tiles, into one of two buffers by unit parity
    w = WL.CONFIGS["c3"].with_(B=6, V=4096, prefix=(0, 1200))
    check_step(w, rows=[(0, 0), (2, 16), (3, 8), (5, 1)])


def test_step_deep_tree_fused(few_clusters):
    w = WL.CONFIGS["c2"].with_(B=3, prefix=(200, 900), V=4096)
    check_step(w, rows=[(0, 64), (1, 0), (2, 33)])
