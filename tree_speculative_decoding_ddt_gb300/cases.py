"""Runs library calls on a named case a given number of times and nothing
else: a short, reproducible launch sequence for a profiler.

    python -m tree_speculative_decoding_ddt_gb300.cases stress [--B 65536] [--reps 2]

``stress``: the build / accept / compaction stress case (B sequences with the
batched workload's drafter shape, D 8, K 4, budget 16, V 163840; a bf16 cache
of 576-wide rows, 16 prefix slots and one page per sequence; the accepted path
leaves the rank-0 chain at the root, so every sequence accepts 8 drafts and
moves 8 rows). Each repetition runs ddt_tree_build, then ddt_tree_accept, then
ddt_cache_compact, in that order, and the statuses are checked at the end.
"""
from __future__ import annotations

import argparse
import sys


def run_stress(B: int, reps: int) -> None:
    import torch

    from . import _binding as DB
    from . import workloads as WL
    dev = torch.device("cuda", torch.cuda.current_device())
    w = WL.CONFIGS["c3"]
    D, K, budget, V = w.D, w.K, w.budget, w.V
    logp, ids, root, target = WL.stress_inputs(B, D, K, V, dev)
    page = -(-(16 + budget + 1) // 64) * 64
    kv = torch.zeros((B * page, w.C + w.R), dtype=torch.bfloat16, device=dev)
    bt = torch.arange(B, dtype=torch.int32, device=dev).reshape(B, 1)
    L = torch.full((B,), 16, dtype=torch.int32, device=dev)
    st = torch.zeros((B,), dtype=torch.int32, device=dev)
    tree = None
    for _ in range(reps):
        tree = DB.ddt_tree_build(logp, ids, root, budget, V, out=tree)
        acc = DB.ddt_tree_accept(tree["tokens"], tree["parents"], target, D, status=st)
        DB.ddt_cache_compact(kv, bt, L, acc["accept_idx"], acc["accept_len"], page, status=st)
    torch.cuda.synchronize()
    if int((tree["status"] | st).abs().sum()) != 0 or int(acc["accept_len"].min()) != D:
        raise SystemExit("stress case: unexpected status or accept length")
    print(f"stress case: B={B}, {reps} repetitions of build, accept, compaction")


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("case", choices=["stress"])
    ap.add_argument("--B", type=int, default=65536)
    ap.add_argument("--reps", type=int, default=2)
    a = ap.parse_args(argv)
    run_stress(a.B, a.reps)
    return 0


if __name__ == "__main__":
    sys.exit(main())
