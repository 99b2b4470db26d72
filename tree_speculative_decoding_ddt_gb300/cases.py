"""Runs library calls on a named case a given number of times and nothing
else: a short, reproducible launch sequence for a profiler.

    python -m tree_speculative_decoding_ddt_gb300.cases stress [--B 65536] [--reps 2]
    python -m tree_speculative_decoding_ddt_gb300.cases attn --config c4 [--reps 2]
    python -m tree_speculative_decoding_ddt_gb300.cases step --config c2 [--reps 2]
    python -m tree_speculative_decoding_ddt_gb300.cases next --config c3 [--reps 2]

``stress``: the build / accept / compaction stress case (B sequences with the
batched workload's drafter shape, D 8, K 4, budget 16, V 163840; a bf16 cache
of 576-wide rows, 16 prefix slots and one page per sequence; the accepted path
leaves the rank-0 chain at the root, so every sequence accepts 8 drafts and
moves 8 rows). Each repetition runs ddt_tree_build, then ddt_tree_accept, then
ddt_cache_compact, in that order, and the statuses are checked at the end.

``attn`` / ``step``: the verify attention (ddt_verify_attn) or the whole step
(ddt_step) on a named workload (c1..c4, or a sweep point q<len>_b<batch>_l<prefix>)
with its seeded inputs, ``reps`` times on one stream.

``next``: the calls beside the verify step on a named workload's shapes, each
``reps`` times: ddt_target_argmax over B*Q x V logits, ddt_drafter_topk over
B*D x V logits (K of the workload), and ddt_rope_append of the workload's
q_pe and B*Q new latents into its cache at the tree's positions L + depth
(logits and latents drawn on the device from a seeded generator).
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


def _workload(name: str):
    from . import workloads as WL
    if name in WL.CONFIGS:
        return WL.CONFIGS[name]
    q, b, l = name[1:].split("_")
    return WL.sweep_point(int(q), int(b[1:]), int(l[1:]))


def run_workload(name: str, reps: int, whole_step: bool) -> None:
    import numpy as np
    import torch

    from . import _binding as DB
    from . import workloads as WL
    w = _workload(name)
    batch = WL.make_batch(w)
    lay = batch.layout
    dev = torch.device("cuda", torch.cuda.current_device())
    bf16 = w.dtype == "bf16"

    def lat(x):
        if bf16:
            bits = WL.to_bf16_bits(x).view(np.int16)
            return torch.from_numpy(np.ascontiguousarray(bits)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)

    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    max_len = int(batch.prefix_len.max()) + w.Q
    buf = DB.StepBuffers(w.B, w.D, w.K, w.budget, w.V, w.H, w.C, w.R, lay.page_size,
                         lay.max_pages, lay.total_rows, DB.DDT_BF16 if bf16 else DB.DDT_F32,
                         w.scale, max_len, device=dev)
    buf.topk_logp.copy_(torch.from_numpy(batch.topk_logp).to(dev))
    buf.topk_ids.copy_(i32(batch.topk_ids))
    buf.root_tok.copy_(i32(batch.root_tok))
    buf.q_lat.copy_(lat(batch.q_lat))
    buf.q_pe.copy_(lat(batch.q_pe))
    buf.kv_cache.copy_(lat(batch.kv))
    buf.block_table.copy_(i32(lay.block_table))
    buf.prefix_len.copy_(i32(batch.prefix_len))
    tr = DB.ddt_tree_build(buf.topk_logp, buf.topk_ids, buf.root_tok, w.budget, w.V, out={
        k: getattr(buf, k) for k in ("tokens", "parents", "depths", "first_child",
                                     "next_sibling", "vis_bits", "n_nodes", "status")})
    buf.target_argmax.copy_(i32(WL.target_argmax_for(batch, tr["depths"].cpu().numpy())))
    for _ in range(reps):
        if whole_step:
            DB.ddt_step(buf)
        else:
            DB.ddt_verify_attn(buf.q_lat, buf.q_pe, buf.kv_cache, buf.block_table,
                               buf.prefix_len, buf.vis_bits, w.scale, lay.page_size, max_len,
                               out=buf.out, lse=buf.lse, status=buf.status,
                               workspace=buf.workspace)
    torch.cuda.synchronize()
    st = buf.status.cpu().numpy()
    if (st & ~DB.ST_BUDGET_PAD).any():
        raise SystemExit(f"{name}: status reports errors: {st}")
    print(f"{'step' if whole_step else 'attn'} case: {w.name}, {reps} repetitions")


def run_next(name: str, reps: int) -> None:
    import numpy as np
    import torch

    from . import _binding as DB
    from . import workloads as WL
    w = _workload(name)
    batch = WL.make_batch(w, latents=False)
    lay = batch.layout
    dev = torch.device("cuda", torch.cuda.current_device())
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    ldt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    logits = (torch.randn((w.B * w.Q, w.V), generator=gen, device=dev) * w.logit_std).to(ldt)
    dl = (torch.randn((w.B * w.D, w.V), generator=gen, device=dev) * w.logit_std).to(ldt)
    q_pe = torch.randn((w.B, w.Q, w.H, w.R), generator=gen, device=dev).to(ldt)
    kv_new = torch.randn((w.B, w.Q, w.C + w.R), generator=gen, device=dev).to(ldt)
    kv = torch.zeros((lay.total_rows, w.C + w.R), dtype=ldt, device=dev)
    tree = DB.ddt_tree_build(torch.from_numpy(batch.topk_logp).to(dev), i32(batch.topk_ids),
                             i32(batch.root_tok), w.budget, w.V)
    bt, L = i32(lay.block_table), i32(batch.prefix_len)
    st = torch.zeros((w.B,), dtype=torch.int32, device=dev)
    am = tk = q_out = None
    for _ in range(reps):
        am = DB.ddt_target_argmax(logits, out=am)
        tk = DB.ddt_drafter_topk(dl, w.K, out=tk)
        q_out, _ = DB.ddt_rope_append(q_pe, kv_new, kv, bt, L, tree["depths"], lay.page_size,
                                      q_out=q_out, status=st)
    torch.cuda.synchronize()
    if int(st.abs().sum()) != 0:
        raise SystemExit(f"{name}: rope_append status reports errors: {st.cpu().numpy()}")
    print(f"next case: {w.name}, {reps} repetitions")


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("case", choices=["stress", "attn", "step", "next"])
    ap.add_argument("--B", type=int, default=65536)
    ap.add_argument("--config", default="c4")
    ap.add_argument("--reps", type=int, default=2)
    a = ap.parse_args(argv)
    if a.case == "stress":
        run_stress(a.B, a.reps)
    elif a.case == "next":
        run_next(a.config, a.reps)
    else:
        run_workload(a.config, a.reps, a.case == "step")
    return 0


if __name__ == "__main__":
    sys.exit(main())
