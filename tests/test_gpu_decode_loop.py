"""GPU multi-step decode loop (ddt_loop_create / ddt_loop_launch through the C
ABI: one CUDA graph, a conditional WHILE node over whole verify steps)
against the oracle's loop, exactly: the committed tokens, the number of
verify steps and the tokens each step committed. Also the pages' numbers
(8.00 tokens per step, 24 tokens in 3 steps), DDTree == autoregressive
output, the step bound, relaunching and a sequence that runs out of cache."""
import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import latent_tensor, t

pytestmark = pytest.mark.gpu


def make(dtype, B, D, K, budget, V, H, C, R, prefix, n_new, hit, cid, max_steps,
         page_size=64, spare_pages=0):
    Q = budget + 1
    G = n_new + D + 1
    golden = WL.loop_golden(cid, B, G, V)
    table = WL.loop_drafter_table(cid, golden, V, hit, dtype)
    g = np.random.default_rng([cid, 99])

    def lat(shape):
        x = g.standard_normal(shape).astype(np.float32)
        return WL.round_bf16(x) if dtype == "bf16" else x

    prefix = np.broadcast_to(np.asarray(prefix, np.int32), (B,)).copy()
    cap = int(prefix.max()) + n_new + Q
    max_pages = -(-cap // page_size) + spare_pages
    pages = g.permutation(B * max_pages).astype(np.int32).reshape(B, max_pages)
    rows = B * max_pages * page_size
    kv = torch.zeros((rows, C + R), dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                     device="cuda")
    loop = DB.DecodeLoop(t(golden), latent_tensor(table, dtype), latent_tensor(lat((B, Q, H, C)), dtype),
                         latent_tensor(lat((B, Q, H, R)), dtype),
                         latent_tensor(lat((B, Q, C + R)), dtype), kv, t(pages), t(prefix),
                         D=D, K=K, budget=budget, n_new=n_new, max_steps=max_steps,
                         page_size=page_size, scale=0.1, max_len=cap)
    return loop, golden, table, prefix


def check_against_oracle(res, golden, table, prefix, n_new, D, K, budget, V, max_steps):
    for b in range(golden.shape[0]):
        out, steps, per = O.decode_loop_table(golden[b], table[b], n_new, D, K, budget, V,
                                              max_steps)
        n = int(res["n_committed"][b])
        assert res["status"][b] == 0, b
        assert res["committed"][b, :n].tolist() == out, b
        assert int(res["steps"][b]) == steps, b
        assert res["accepted"][b, :steps].tolist() == per, b
        assert (res["accepted"][b, steps:] == 0).all()
        assert int(res["prefix_len"][b]) == int(prefix[b]) + sum(per), b


def test_the_pages_oracle_drafter_numbers_on_the_gpu():
    # fp32 tiny shapes; seven drafts + bonus per step: 24 tokens in 3 steps
    loop, golden, table, prefix = make("f32", B=2, D=7, K=4, budget=16, V=1024, H=4, C=64, R=32,
                                       prefix=32, n_new=24, hit=1.0, cid=11, max_steps=64)
    loop.launch()
    res = loop.results()
    for b in range(2):
        assert res["committed"][b].tolist() == golden[b, :25].tolist()
        assert res["committed"][b].tolist() == O.ar_decode(golden[b], 24, 1024)
        assert int(res["steps"][b]) == 3
        assert res["accepted"][b, :3].tolist() == [8, 8, 8]
    check_against_oracle(res, golden, table, prefix, 24, 7, 4, 16, 1024, 64)
    loop.close()


@pytest.mark.parametrize("hit", [(0.5, 0.8, 1.0), (0.0, 0.3, 0.9)])
def test_k2_shapes_match_the_oracle_loop(hit):
    # bf16 K2.6 attention shapes (tcgen05 path), small vocabulary, three
    # sequences with different drafter hit rates and ragged prefixes
    V, D, K, budget, n_new = 4096, 8, 4, 16, 40
    loop, golden, table, prefix = make("bf16", B=3, D=D, K=K, budget=budget, V=V, H=64, C=512,
                                       R=64, prefix=[300, 1000, 77], n_new=n_new, hit=hit,
                                       cid=12, max_steps=100)
    loop.launch()
    res = loop.results()
    check_against_oracle(res, golden, table, prefix, n_new, D, K, budget, V, 100)
    for b in range(3):
        assert res["committed"][b].tolist() == O.ar_decode(golden[b], n_new, V)
    loop.close()


def test_max_budget_shape_with_the_full_vocabulary():
    # one sequence at D 16, K 8, budget 64 over V = 163840 (prefix 4096)
    V, D, K, budget, n_new = 163840, 16, 8, 64, 48
    loop, golden, table, prefix = make("bf16", B=1, D=D, K=K, budget=budget, V=V, H=64, C=512,
                                       R=64, prefix=4096, n_new=n_new, hit=0.8, cid=13,
                                       max_steps=64)
    loop.launch()
    res = loop.results()
    check_against_oracle(res, golden, table, prefix, n_new, D, K, budget, V, 64)
    loop.close()


def test_step_bound_and_relaunch():
    loop, golden, table, prefix = make("f32", B=2, D=4, K=2, budget=6, V=512, H=2, C=16, R=8,
                                       prefix=10, n_new=50, hit=1.0, cid=14, max_steps=2)
    loop.launch()
    first = loop.results()
    assert first["steps"].tolist() == [2, 2]
    assert first["n_committed"].tolist() == [11, 11]
    check_against_oracle(first, golden, table, prefix, 50, 4, 2, 6, 512, 2)
    loop.launch()
    again = loop.results()
    for k in first:
        np.testing.assert_array_equal(first[k], again[k])
    loop.close()


def test_a_sequence_out_of_cache_stops_alone():
    # sequence 1 starts too close to the end of its pages: its first step
    # reports DDT_ST_CAPACITY and it stops; sequence 0 decodes normally
    V, D, K, budget, n_new = 512, 4, 3, 8, 12
    loop, golden, table, prefix = make("f32", B=2, D=D, K=K, budget=budget, V=V, H=2, C=16, R=8,
                                       prefix=[5, 5], n_new=n_new, hit=1.0, cid=15,
                                       max_steps=40)
    cap_pages = loop.args.attn.max_pages
    bad = torch.tensor([5, cap_pages * 64 - 3], dtype=torch.int32, device="cuda")
    loop2 = DB.DecodeLoop(*(loop._keep[:7] + (bad,)), D=D, K=K, budget=budget, n_new=n_new,
                          max_steps=40, page_size=64, scale=0.1,
                          max_len=cap_pages * 64 + budget + 1)
    loop2.launch()
    res = loop2.results()
    assert int(res["status"][0]) == 0 and int(res["status"][1]) & DB.ST_CAPACITY
    assert int(res["steps"][1]) == 0 and int(res["n_committed"][1]) == 1
    out, steps, per = O.decode_loop_table(golden[0], table[0], n_new, D, K, budget, V, 40)
    assert res["committed"][0, : len(out)].tolist() == out and int(res["steps"][0]) == steps
    loop.close()
    loop2.close()
