"""Times the whole verify step and the verify attention at the points of the
q_len x batch x prefix sweep on one GPU; prints one JSON line per point.

    python -m tree_speculative_decoding_ddt_gb300.sweep [--steps 20] [--points q65_b64_l8192,...]

Each point is a ``workloads.sweep_point`` (the batched workload's drafter: D 8,
K 4, V 163840, budget = q_len - 1; 64 heads, kv_lora 512, rope 64, bf16,
contiguous cache). The drafter's top-k and the synthetic target come from the
seeded generators of ``workloads``; the latents (queries and cache) are drawn
on the device from a seeded torch generator, N(0, 1) rounded to bf16, so that
the largest points (64 sequences of 131072 keys: 9.7 GB of cache) need no host
copy. A step is one ``ddt_step`` captured in a CUDA graph and replayed, L2
flushed (a 256 MiB write) before each timed replay, outside its events; the
attention is the ``ddt_verify_attn`` call timed the same way. The roofline is
the slower of the algorithmic FLOPs at the measured bf16 peak and the bytes at
the measured HBM copy bandwidth (``MEASURED_PEAKS.json``).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

import numpy as np

Q_LENS = (1, 9, 17, 33, 65)
BATCHES = (1, 8, 64)
PREFIXES = (1024, 8192, 65536, 131072)


def peaks():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = os.path.join(root, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def attn_work(w, prefix_len, depths):
    """Algorithmic FLOPs and bytes of one verify attention (every visible
    (row, key) pair: 4C + 2R FLOPs; bytes: cache rows once, Q, O, lse)."""
    flops, keys = 0, 0
    for b in range(w.B):
        L = int(prefix_len[b])
        d = np.asarray(depths[b])
        flops += int((L + np.where(d >= 0, d + 1, 1)).sum()) * w.H * (4 * w.C + 2 * w.R)
        keys += L + w.Q
    byt = (keys * (w.C + w.R) * 2 + w.B * w.Q * w.H * (w.C + w.R) * 2
           + w.B * w.Q * w.H * w.C * 2 + w.B * w.Q * w.H * 4)
    return flops, byt


def run_point(q_len: int, B: int, prefix: int, steps: int, flush) -> dict:
    import torch

    from . import _binding as DB
    from . import workloads as WL
    w = WL.sweep_point(q_len, B, prefix)
    batch = WL.make_batch(w, latents=False)
    lay = batch.layout
    dev = flush.device
    max_len = int(batch.prefix_len.max()) + w.Q
    buf = DB.StepBuffers(w.B, w.D, w.K, w.budget, w.V, w.H, w.C, w.R, lay.page_size,
                         lay.max_pages, lay.total_rows, DB.DDT_BF16, w.scale, max_len, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 * q_len + 10 * B + prefix)
    for t in (buf.q_lat, buf.q_pe):
        t.copy_(torch.randn(t.shape, generator=gen, device=dev))
    for r0 in range(0, lay.total_rows, 1 << 20):  # the cache in 1 Mi-row pieces
        r1 = min(lay.total_rows, r0 + (1 << 20))
        buf.kv_cache[r0:r1].copy_(torch.randn((r1 - r0, w.C + w.R), generator=gen, device=dev))
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    buf.topk_logp.copy_(torch.from_numpy(batch.topk_logp).to(dev))
    buf.topk_ids.copy_(i32(batch.topk_ids))
    buf.root_tok.copy_(i32(batch.root_tok))
    buf.block_table.copy_(i32(lay.block_table))
    buf.prefix_len.copy_(i32(batch.prefix_len))
    tr = DB.ddt_tree_build(buf.topk_logp, buf.topk_ids, buf.root_tok, w.budget, w.V)
    depths = tr["depths"].cpu().numpy()
    buf.target_argmax.copy_(i32(WL.target_argmax_for(batch, depths)))
    torch.cuda.synchronize()

    def step():
        DB.ddt_step(buf)

    def attn():
        DB.ddt_verify_attn(buf.q_lat, buf.q_pe, buf.kv_cache, buf.block_table, buf.prefix_len,
                           buf.vis_bits, w.scale, lay.page_size, max_len, out=buf.out,
                           lse=buf.lse, status=buf.status, workspace=buf.workspace)

    stream = torch.cuda.current_stream()
    out = {}
    for name, fn in (("step", step), ("attn", attn)):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(3):
            flush.fill_(1)
            g.replay()
        evs = []
        for _ in range(steps):
            flush.fill_(1)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            g.replay()
            e.record(stream)
            evs.append((s, e))
        torch.cuda.synchronize()
        out[name] = statistics.median(s.elapsed_time(e) for s, e in evs) / 1e3
        del g
    st = buf.status.cpu().numpy()
    if (st & ~DB.ST_BUDGET_PAD).any():
        raise SystemExit(f"q{q_len}_b{B}_l{prefix}: status reports errors: {st}")
    hbm, tf, src = peaks()
    flops, byt = attn_work(w, batch.prefix_len, depths)
    t_f, t_b = flops / (tf * 1e12), byt / (hbm * 1e9)
    bound = "tensor" if t_f >= t_b else "hbm"
    rate = flops / out["attn"] / 1e12 if bound == "tensor" else byt / out["attn"] / 1e9
    return {"point": f"q{q_len}_b{B}_l{prefix}", "q_len": q_len, "B": B, "prefix": prefix,
            "rows_per_tile": DB.ddt_verify_attn_rows_per_tile(buf.attn),
            "key_splits": DB.ddt_verify_attn_splits(buf.attn),
            "steps_per_s": 1.0 / out["step"], "step_us": out["step"] * 1e6,
            "attn_us": out["attn"] * 1e6, "bound": bound,
            "rate": rate, "rate_unit": "TFLOP/s" if bound == "tensor" else "GB/s",
            "frac": max(t_f, t_b) / out["attn"], "peak_source": src}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--points", default="", help="comma-separated q<len>_b<B>_l<prefix>")
    a = ap.parse_args(argv)
    import torch
    from . import _binding as DB
    DB.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    if a.points:
        pts = []
        for s in a.points.split(","):
            q, b, l = s[1:].split("_")
            pts.append((int(q), int(b[1:]), int(l[1:])))
    else:
        pts = [(q, b, l) for q in Q_LENS for b in BATCHES for l in PREFIXES]
    for q, b, l in pts:
        print(json.dumps(run_point(q, b, l, a.steps, flush)), flush=True)
        torch.cuda.empty_cache()
    return 0


if __name__ == "__main__":
    sys.exit(main())
