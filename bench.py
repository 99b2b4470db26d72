#!/usr/bin/env python
"""Benchmark of one DDTree verify step on GB300; prints ONE JSON line.

A step is the whole hot path through the C ABI (``ddt_step``): best-first
tree build -> tree-verify MLA-absorb attention -> greedy accept + cache
compaction, over one batch of the deep-tree long-context workload by default
(B=8, D=15, K=2, budget 64 -> q_len 65, 64 heads, kv_lora 512, rope 64,
prefix 32768, bf16; every step accepts 15 drafts and compacts them), the
largest fixed single-GPU configuration. The step is captured in a CUDA graph
and replayed; L2 is flushed (a 256 MiB write) between timed steps, outside the
per-step CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c4]
    python bench.py --impl reference ...     # the CPU oracle as the reference arm

Multi-GPU (torchrun, one process per GPU) runs independent replicas: the
path has no exchange step, so each rank verifies its own batch; ``value`` is
all ranks' steps divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DDTree verify steps/s; verify_attn TFLOP/s and % of GB300 roofline"
FLUSH_BYTES = 256 << 20


# --------------------------------------------------------------------- helpers

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c4",
                    help="c1..c4 or a sweep point q<len>_b<batch>_l<prefix>")
    ap.add_argument("--no-graph", action="store_true", help="launch each step directly")
    ap.add_argument("--cpu-seconds", type=float, default=20.0,
                    help="target CPU time of the oracle baseline sample (0 = skip it)")
    ap.add_argument("--attn-steps", type=int, default=None,
                    help="timed launches of the attention call alone (default steps/4, >= 50)")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the end-to-end host-buffer loop (default min(steps, 2000))")
    return ap.parse_args(argv)


def workload(name: str):
    from tree_speculative_decoding_ddt_gb300 import workloads as WL
    if name in WL.CONFIGS:
        return WL.CONFIGS[name]
    if name.startswith("q"):
        q, b, l = name[1:].split("_")
        return WL.sweep_point(int(q), int(b[1:]), int(l[1:]))
    raise SystemExit(f"unknown config {name}")


def describe(w) -> str:
    pre = w.prefix if not isinstance(w.prefix, tuple) else f"U[{w.prefix[0]},{w.prefix[1]}]"
    paging = f"paged {w.page_size}" if w.page_size else "contiguous"
    return (f"{w.name}: B={w.B} D={w.D} K={w.K} V={w.V} budget={w.budget} (q_len {w.Q}) "
            f"H={w.H} kv_lora={w.C} rope={w.R} prefix={pre} {paging} {w.dtype}")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the attention kernel the dispatcher picks for a workload (128-row tiles:
# k_verify_attn_bf16 in verify_attn_bf16.cu; 256-row tiles: k_verify_attn_pair
# in verify_attn_pair.cu), from ncu captures of the kernel built from the
# source whose sha256 is given; reported as null once that source changes.
MEASURED_TRAFFIC = {
    ("c2_max_budget", 256): ("verify_attn_pair.cu",
                             "6a0dd4ea256e67ff05afee0c9767985f04d128a60c7c388b21a3c8d52f9f7d62",
                             9822208 + 0),
    ("c3_batched_paged", 256): ("verify_attn_pair.cu",
                                "6a0dd4ea256e67ff05afee0c9767985f04d128a60c7c388b21a3c8d52f9f7d62",
                                450383616 + 54412800),
    ("c4_deep_long", 256): ("verify_attn_pair.cu",
                            "6a0dd4ea256e67ff05afee0c9767985f04d128a60c7c388b21a3c8d52f9f7d62",
                            458527744 + 33223168),
}


def attn_kernel_name(rows: int) -> str:
    return "k_verify_attn_pair" if rows == 256 else "k_verify_attn_bf16"


def measured_traffic(w, rows: int):
    """ncu DRAM bytes per launch of the attention kernel for workload w, or
    None when none was taken for the current kernel source."""
    import hashlib
    entry = MEASURED_TRAFFIC.get((w.name, rows))
    if entry is None:
        return None
    src = os.path.join(ROOT, "tree_speculative_decoding_ddt_gb300", "csrc", entry[0])
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    return entry[2] if digest == entry[1] else None


def attn_work(w, prefix_len, depths, dtype_bytes):
    """Algorithmic FLOPs and bytes of one verify-attention launch: every
    visible (query row, key) pair costs 2(C+R) for q.k and 2C for p.v; a
    row sees its prefix plus its ancestor path (depth+1 tree slots). Bytes:
    each cache row read once, Q read once, O written once, lse written."""
    flops = 0
    keys = 0
    for b in range(w.B):
        L = int(prefix_len[b])
        d = np.asarray(depths[b])
        n_vis = L + np.where(d >= 0, d + 1, 1)
        flops += int(n_vis.sum()) * w.H * (4 * w.C + 2 * w.R)
        keys += L + w.Q
    byt = (keys * (w.C + w.R) * dtype_bytes + w.B * w.Q * w.H * (w.C + w.R) * dtype_bytes
           + w.B * w.Q * w.H * w.C * dtype_bytes + w.B * w.Q * w.H * 4)
    return flops, byt


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 0.25 * max(x[2] for x in rows)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3][1:5])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(loaded), "power_w_max": max(r[2] for r in rows)}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of ``x`` over all ranks (identity without a process group)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------- CPU oracle arm

def oracle_sequence(w, batch, b: int):
    """The oracle's whole step (heapq build, float64 attention, accept,
    compaction) on sequence ``b`` of the batch alone, as a callable. The
    sequence's pages are gathered into a cache of its own beforehand, so the
    timed call does exactly that sequence's share of the batch's work."""
    from oracle import ddt_oracle as O
    from tree_speculative_decoding_ddt_gb300 import workloads as WL
    lay = batch.layout
    L = int(batch.prefix_len[b])
    n_pages = -(-(L + w.Q) // lay.page_size)
    kv = np.ascontiguousarray(batch.kv[lay.rows_of(b, np.arange(n_pages * lay.page_size))])
    bt = np.arange(n_pages, dtype=np.int32).reshape(1, n_pages)
    one = slice(b, b + 1)
    p = float(batch.match_p[b])

    def target(tree):
        return WL.synth_target_argmax(tree["depths"][0], batch.topk_ids[b], batch.target_u[b],
                                      batch.target_fallback[b], p)[None]

    def run():
        return O.ddt_step(batch.topk_logp[one], batch.topk_ids[one], batch.root_tok[one],
                          w.budget, w.V, batch.q_lat[one], batch.q_pe[one], kv, bt,
                          batch.prefix_len[one], w.scale, lay.page_size, n_pages, target)
    return run


def oracle_steps(w, batch, seconds: float, max_steps: int, first: int = 0):
    """Time single-sequence oracle steps (sequences first, first+1, ... cycling
    over the batch) until ``max_steps`` are done or about ``seconds`` have
    passed (at least one). Returns (sequence steps, seconds, whole-batch
    steps/s = 1 / (B x mean seconds per sequence))."""
    n, secs = 0, 0.0
    while n < max_steps:
        run = oracle_sequence(w, batch, (first + n) % w.B)
        t0 = time.perf_counter()
        run()
        secs += time.perf_counter() - t0
        n += 1
        if secs >= seconds:
            break
    return n, secs, n / (w.B * secs)


def oracle_sample_text(w, n: int, model: str) -> str:
    what = (f"{n} single-sequence oracle steps (python heapq build, numpy float64 attention, "
            f"accept, compaction) of the workload on {model}")
    if w.B == 1:
        return what
    return what + f"; whole-batch rate extrapolated as 1 / ({w.B} x mean seconds per sequence)"


def cpu_info():
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = ""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    import platform
    return cores, f"{platform.machine()} {model}".strip()


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, on the same
    workload, metric and unit as the GPU arm. Each step is one sequence of the
    batch (cycling), so a step stays a bounded sample; the whole-batch steps/s
    is extrapolated by B."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from tree_speculative_decoding_ddt_gb300 import workloads as WL
    w = workload(args.config)
    batch = WL.make_batch(w)
    # W untimed warm-up steps, cut short after 30 s of them on a slow host
    warm, t_w = 0, time.perf_counter()
    while warm < args.warmup and time.perf_counter() - t_w < 30.0:
        oracle_sequence(w, batch, warm % w.B)()
        warm += 1
    # K timed steps, cut short after 150 s so the arm ends within minutes
    n, secs, v = oracle_steps(w, batch, 150.0, max(1, args.steps), first=warm)
    cores, model = cpu_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": n, "warmup": warm, "ms_per_step": 1e3 / v,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": describe(w)},
        "cpu_baseline": {"value": v, "unit": "steps/s", "cores": cores, "kind": "oracle",
                         "sample": oracle_sample_text(w, n, model)},
        "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ GPU arm

def _event_median_s(fn, stream, flush, n: int) -> float:
    """Median device time of ``fn`` over n launches, L2 flushed before each."""
    import torch
    fn()
    ts = []
    for _ in range(max(5, min(n, 50))):
        flush.fill_(1)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        ts.append((s, e))
    torch.cuda.synchronize()
    return statistics.median([s.elapsed_time(e) for s, e in ts]) / 1e3


def time_next_rows(w, dev, stream, flush, n: int, buf=None) -> dict:
    """Event-timed launches of the steps next to the verify step on this
    workload's shapes (L2 flushed before each launch), each against the HBM
    roofline of its algorithmic bytes: the target-side argmax over
    B*Q x V logits, the drafter's top-K over B*D x V logits and (given the
    step's buffers) the rotary embedding and cache append of the tree at its
    positions L+depth."""
    import torch
    from tree_speculative_decoding_ddt_gb300 import _binding as DB
    hbm, _, src = measured_peaks()
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    ldt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    logits = (torch.randn((w.B * w.Q, w.V), generator=gen, device=dev) * w.logit_std).to(ldt)
    am = torch.empty((w.B * w.Q,), dtype=torch.int32, device=dev)
    DB.ddt_target_argmax(logits, out=am)
    ts = []
    for _ in range(max(5, min(n, 50))):
        flush.fill_(1)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        DB.ddt_target_argmax(logits, out=am)
        e.record(stream)
        ts.append((s, e))
    torch.cuda.synchronize()
    sec = statistics.median([s.elapsed_time(e) for s, e in ts]) / 1e3
    byt = logits.numel() * logits.element_size() + am.numel() * 4
    out["target_argmax"] = {"kernel": "k_target_argmax", "rows": w.B * w.Q, "V": w.V,
                            "us": sec * 1e6, "bound": "hbm", "achieved": byt / sec / 1e9,
                            "peak": hbm, "unit": "GB/s", "frac": byt / sec / 1e9 / hbm,
                            "algorithmic_bytes": byt, "peak_source": src,
                            "data": "seeded device normal logits"}
    del logits
    # the drafter's per-depth top-K over B*D x V logits
    dl = (torch.randn((w.B * w.D, w.V), generator=gen, device=dev) * w.logit_std).to(ldt)
    tk = DB.ddt_drafter_topk(dl, w.K)
    ts = []
    for _ in range(max(5, min(n, 50))):
        flush.fill_(1)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        DB.ddt_drafter_topk(dl, w.K, out=tk)
        e.record(stream)
        ts.append((s, e))
    torch.cuda.synchronize()
    sec = statistics.median([s.elapsed_time(e) for s, e in ts]) / 1e3
    byt = dl.numel() * dl.element_size() + w.B * w.D * w.K * 8
    out["drafter_topk"] = {"kernel": "k_drafter_topk", "rows": w.B * w.D, "V": w.V, "K": w.K,
                           "us": sec * 1e6, "bound": "hbm", "achieved": byt / sec / 1e9,
                           "peak": hbm, "unit": "GB/s", "frac": byt / sec / 1e9 / hbm,
                           "algorithmic_bytes": byt, "peak_source": src,
                           "data": "seeded device normal logits"}
    del dl
    if buf is not None:
        # rotary embedding + append on the step's own cache, pages and tree
        # depths (the tree the timed steps built); q turned into a separate
        # buffer, new latents drawn on the device
        ldt = buf.q_pe.dtype
        kv_new = torch.randn((w.B, w.Q, w.C + w.R), generator=gen, device=dev).to(ldt)
        q_out = torch.empty_like(buf.q_pe)
        st = torch.zeros((w.B,), dtype=torch.int32, device=dev)
        ps = buf.attn.page_size
        sec = _event_median_s(lambda: DB.ddt_rope_append(
            buf.q_pe, kv_new, buf.kv_cache, buf.block_table, buf.prefix_len, buf.depths, ps,
            q_out=q_out, status=st), stream, flush, n)
        es = buf.q_pe.element_size()
        byt = w.B * w.Q * (2 * w.H * w.R + 2 * (w.C + w.R)) * es + w.B * w.Q * 4
        out["rope_append"] = {"kernel": "k_rope_append", "slots": w.B * w.Q, "H": w.H, "R": w.R,
                              "us": sec * 1e6, "bound": "hbm", "achieved": byt / sec / 1e9,
                              "peak": hbm, "unit": "GB/s", "frac": byt / sec / 1e9 / hbm,
                              "algorithmic_bytes": byt, "peak_source": src,
                              "data": "the step's cache, pages and tree depths; seeded "
                                      "device latents"}
        if int(st.abs().sum()) != 0:
            raise SystemExit(f"rope_append status reports errors: {st.cpu().numpy()}")
        del kv_new, q_out
    return out


def _stage_rows(B, D, K, Q, C, R, elem, kv, block_table, page_size, prefix_len, topk_logp,
                topk_ids, root_tok, target, budget, V, stream, flush, n) -> dict:
    """Event-timed tree build, accept and compaction calls (L2 flushed before
    each), each with its algorithmic bytes and achieved GB/s against the
    measured HBM copy bandwidth."""
    import torch
    from tree_speculative_decoding_ddt_gb300 import _binding as DB
    hbm, _, src = measured_peaks()
    dev = topk_logp.device
    W = (Q + 63) // 64
    tree = DB.ddt_tree_build(topk_logp, topk_ids, root_tok, budget, V)
    st = torch.zeros((B,), dtype=torch.int32, device=dev)
    t_build = _event_median_s(lambda: DB.ddt_tree_build(topk_logp, topk_ids, root_tok, budget, V,
                                                        out=tree), stream, flush, n)
    acc = DB.ddt_tree_accept(tree["tokens"], tree["parents"], target, D, status=st)
    t_acc = _event_median_s(lambda: DB.ddt_tree_accept(tree["tokens"], tree["parents"], target,
                                                       D, status=st), stream, flush, n)
    t_cmp = _event_median_s(lambda: DB.ddt_cache_compact(kv, block_table, prefix_len,
                                                         acc["accept_idx"], acc["accept_len"],
                                                         page_size, status=st), stream, flush, n)
    # rows that really move: path slots not already in place
    idx = acc["accept_idx"][:, 1:]
    d = torch.arange(1, D + 1, device=dev, dtype=torch.int32)
    inside = d[None, :] <= acc["accept_len"][:, None]
    moved = int(((idx != d[None, :]) & inside).sum())
    if int(st.abs().sum()) != 0:
        raise SystemExit(f"stage timing: device status reports errors")
    out = {}
    for name, sec, byt, kern in (
            ("tree_build", t_build, B * D * K * 8 + B * Q * (12 + 8 * W + 8), "k_tree_build"),
            ("accept", t_acc, B * Q * 12 + B * (D + 1) * 8, "k_accept_compact (accept only)"),
            ("compact", t_cmp, 2 * moved * (C + R) * elem, "k_accept_compact (gather only)")):
        out[name] = {"kernel": kern, "us": sec * 1e6, "algorithmic_bytes": byt,
                     "achieved": byt / sec / 1e9, "unit": "GB/s", "peak": hbm,
                     "frac": byt / sec / 1e9 / hbm, "peak_source": src}
    out["compact"]["rows_moved"] = moved
    return out


def time_stages(w, buf, dev, stream, flush, n: int) -> dict:
    """Build, accept and compaction of this workload's step, each timed alone
    (they move kilobytes, so latency sets their time; µs is the figure)."""
    elem = buf.q_pe.element_size()
    # the compaction moves rows inside the tree slots of the step's cache,
    # which the e2e leg rewrites before every step
    return _stage_rows(w.B, w.D, w.K, w.Q, w.C, w.R, elem, buf.kv_cache, buf.block_table,
                       buf.attn.page_size, buf.prefix_len, buf.topk_logp, buf.topk_ids,
                       buf.root_tok, buf.target_argmax, w.budget, w.V, stream, flush, n)


def time_stress(dev, stream, flush, n: int, B: int = 65536) -> dict:
    """An addition to the workloads: B = 65536 sequences with the batched
    workload's drafter shape (c3: D 8, K 4, budget 16, V 163840, bf16 cache
    rows of 576), so that build, accept and compaction move megabytes and
    bandwidth becomes the meaningful figure. The accepted path leaves the
    rank-0 chain at the root (workloads.stress_inputs), so every sequence accepts 8
    drafts and compaction really moves 8 rows; the cache holds 16 prefix slots
    and the tree slots of every sequence, one page each."""
    import torch
    from tree_speculative_decoding_ddt_gb300 import workloads as WL
    w = WL.CONFIGS["c3"]
    D, K, budget, V = w.D, w.K, w.budget, w.V
    assert budget == 2 * D
    Q = budget + 1
    logp, ids, root, target = WL.stress_inputs(B, D, K, V, dev)
    page = -(-(16 + Q) // 64) * 64
    kv = torch.zeros((B * page, w.C + w.R), dtype=torch.bfloat16 if w.dtype == "bf16"
                     else torch.float32, device=dev)
    bt = torch.arange(B, dtype=torch.int32, device=dev).reshape(B, 1)
    L = torch.full((B,), 16, dtype=torch.int32, device=dev)
    out = _stage_rows(B, D, K, Q, w.C, w.R, kv.element_size(), kv, bt, page, L, logp, ids,
                      root, target, budget, V, stream, flush, n)
    out["note"] = (f"addition: B={B} sequences, drafter D={D} K={K} budget={budget}; the "
                   f"accepted path leaves the rank-0 chain at the root, {D} drafts accepted and "
                   f"{D} rows moved per sequence; seeded device inputs")
    return out


def time_decode_loop(w, dev, stream, flush, n_new: int = 256, runs: int = 5) -> dict:
    """The device decode loop (one CUDA graph, a conditional WHILE node over
    whole verify steps) on this workload's shapes: B sequences, the drafter
    hitting the stream at the workload's match rate, n_new tokens each.
    Drafter table and stream drawn on the device; the committed tokens are
    checked against the stream (DDTree == autoregressive output)."""
    import torch
    from tree_speculative_decoding_ddt_gb300 import _binding as DB
    gen = torch.Generator(device=dev)
    gen.manual_seed(4321)
    ldt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    B, Q, G = w.B, w.Q, n_new + w.D + 1
    golden = torch.randint(0, w.V - 1, (B, G), generator=gen, device=dev, dtype=torch.int32)
    table = torch.randn((B, G, w.V), generator=gen, device=dev).to(ldt)
    lo, hi = (w.match_p, w.match_p) if not isinstance(w.match_p, tuple) else w.match_p
    rate = torch.linspace(lo, hi, B, device=dev)[:, None]
    hit = torch.rand((B, G), generator=gen, device=dev) < rate
    spike = table.float().amax(dim=-1) + 8.0
    cur = table.gather(2, golden[..., None].long())[..., 0].float()
    table.scatter_(2, golden[..., None].long(), torch.where(hit, spike, cur)[..., None].to(ldt))
    lens = torch.full((B,), 4096 if not isinstance(w.prefix, int) else w.prefix,
                      dtype=torch.int32, device=dev)
    ps = 64
    cap = int(lens.max()) + n_new + Q
    pages = -(-cap // ps)
    bt = torch.arange(B * pages, dtype=torch.int32, device=dev).reshape(B, pages)
    kv = torch.randn((B * pages * ps, w.C + w.R), generator=gen, device=dev).to(ldt)
    q_lat = torch.randn((B, Q, w.H, w.C), generator=gen, device=dev).to(ldt)
    q_pe = torch.randn((B, Q, w.H, w.R), generator=gen, device=dev).to(ldt)
    kv_new = torch.randn((B, Q, w.C + w.R), generator=gen, device=dev).to(ldt)
    loop = DB.DecodeLoop(golden, table, q_lat, q_pe, kv_new, kv, bt, lens, D=w.D, K=w.K,
                         budget=w.budget, n_new=n_new, max_steps=n_new, page_size=ps,
                         scale=w.scale, max_len=cap)
    loop.launch(stream)
    torch.cuda.synchronize()
    ts = []
    for _ in range(runs):
        flush.fill_(1)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        loop.launch(stream)
        e.record(stream)
        ts.append((s, e))
    torch.cuda.synchronize()
    sec = statistics.median([s.elapsed_time(e) for s, e in ts]) / 1e3
    res = loop.results()
    ok = bool((res["committed"] == golden[:, : n_new + 1].cpu().numpy()).all())
    steps = int(res["steps"].max())
    made = int(res["accepted"].sum())
    loop.close()
    if not ok or (res["status"] != 0).any():
        raise SystemExit("decode loop: committed tokens differ from the stream")
    return {"graph": "one CUDA graph, conditional WHILE node over whole verify steps",
            "B": B, "n_new": n_new, "drafter_hit_rate": [lo, hi], "us": sec * 1e6,
            "tokens_per_s": B * n_new / sec, "verify_steps": steps,
            "tokens_per_step": made / max(int(res["steps"].sum()), 1),
            "us_per_step": sec * 1e6 / max(steps, 1), "ar_target_steps": n_new,
            "greedy_exact": ok,
            "data": "seeded device stream and drafter table; fixed synthetic projections"}


def run_ours(args):
    import torch
    from tree_speculative_decoding_ddt_gb300 import _binding as DB
    from tree_speculative_decoding_ddt_gb300 import workloads as WL

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    DB.load()

    w = workload(args.config)
    batch = WL.make_batch(w)
    lay = batch.layout
    bf16 = w.dtype == "bf16"
    dt = DB.DDT_BF16 if bf16 else DB.DDT_F32
    max_len = int(batch.prefix_len.max()) + w.Q
    buf = DB.StepBuffers(w.B, w.D, w.K, w.budget, w.V, w.H, w.C, w.R, lay.page_size,
                         lay.max_pages, lay.total_rows, dt, w.scale, max_len, device=dev)

    def dev_lat(x):
        if bf16:
            bits = WL.to_bf16_bits(x).view(np.int16)
            return torch.from_numpy(np.ascontiguousarray(bits)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)

    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    buf.topk_logp.copy_(torch.from_numpy(batch.topk_logp).to(dev))
    buf.topk_ids.copy_(i32(batch.topk_ids))
    buf.root_tok.copy_(i32(batch.root_tok))
    buf.q_lat.copy_(dev_lat(batch.q_lat))
    buf.q_pe.copy_(dev_lat(batch.q_pe))
    buf.kv_cache.copy_(dev_lat(batch.kv))
    buf.block_table.copy_(i32(lay.block_table))
    buf.prefix_len.copy_(i32(batch.prefix_len))
    # the synthetic target's argmax depends on each slot's depth: build the
    # (deterministic) tree once to read the depths
    tr = DB.ddt_tree_build(buf.topk_logp, buf.topk_ids, buf.root_tok, w.budget, w.V)
    depths = tr["depths"].cpu().numpy()
    buf.target_argmax.copy_(i32(WL.target_argmax_for(batch, depths)))
    torch.cuda.synchronize()

    split = bf16 and DB.ddt_verify_attn_splits(buf.attn) > 1
    attn_rows = DB.ddt_verify_attn_rows_per_tile(buf.attn) if bf16 else 0
    # build + attention (fused for bf16 when the candidate table is small), split merge, accept
    fused = w.dtype == "bf16" and min(w.D, w.budget) * min(w.K, w.budget) <= 1024
    launches_per_step = (2 if fused else 3) + (1 if split else 0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        DB.ddt_step(buf)

    def attn_only():
        DB.ddt_verify_attn(buf.q_lat, buf.q_pe, buf.kv_cache, buf.block_table, buf.prefix_len,
                           buf.vis_bits, w.scale, lay.page_size, max_len, out=buf.out,
                           lse=buf.lse, status=buf.status, workspace=buf.workspace)

    use_graph = not args.no_graph
    graphs = {}
    if use_graph:
        for name, fn in (("step", step), ("attn", attn_only)):
            fn()  # warm the kernels up once before capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            graphs[name] = g
    run = {k: (graphs[k].replay if use_graph else f) for k, f in
           (("step", step), ("attn", attn_only))}

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for s, e in evs:
            flush.fill_(1)
            s.record(stream)
            fn()
            e.record(stream)
        return evs

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        run["step"]()
    torch.cuda.synchronize()

    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        evs = timed(run["step"], args.steps)
        torch.cuda.synchronize()
        barrier(world)
        bracket_s = time.perf_counter() - t0
        step_ms = [s.elapsed_time(e) for s, e in evs]
        # the dominant kernel, timed the same way
        n_attn = args.attn_steps if args.attn_steps is not None else max(50, args.steps // 4)
        aevs = timed(run["attn"], n_attn)
        torch.cuda.synchronize()
        attn_ms = [s.elapsed_time(e) for s, e in aevs]
        # the next rows of the path, on this workload's shapes, timed the same way
        next_rows = time_next_rows(w, dev, stream, flush, n_attn, buf)
        next_rows["decode_loop"] = time_decode_loop(w, dev, stream, flush,
                                                    n_new=max(16, min(256, 4096 // w.B)))
        stages = time_stages(w, buf, dev, stream, flush, n_attn)
        stages["stress"] = time_stress(dev, stream, flush, n_attn)
    clocks = clk.summary()

    # end to end through the public API: host inputs in pinned memory are
    # copied in (the drafter's top-k, the queries with an unrotated rope part,
    # the tree latents with an unrotated rope part, the target argmax), the
    # tree is built, its rope parts are turned at positions L + depth and its
    # latents appended to the cache (ddt_tree_build + ddt_rope_append), the
    # step runs, and its result (accepted tokens, lengths, status) is copied
    # out, every step
    def pinned_lat(x):
        x = np.ascontiguousarray(WL.to_bf16_bits(x).view(np.int16) if bf16 else x)
        return torch.from_numpy(x).pin_memory()

    host_in = {
        "topk_logp": torch.from_numpy(batch.topk_logp).pin_memory(),
        "topk_ids": torch.from_numpy(batch.topk_ids).pin_memory(),
        "root_tok": torch.from_numpy(batch.root_tok).pin_memory(),
        "q_lat": pinned_lat(batch.q_lat),
        "target_argmax": torch.from_numpy(WL.target_argmax_for(batch, depths)).pin_memory(),
    }
    tree_rows = np.concatenate([lay.rows_of(b, np.arange(int(batch.prefix_len[b]),
                                                         int(batch.prefix_len[b]) + w.Q))
                                for b in range(w.B)])
    host_qpe = pinned_lat(batch.q_pe)
    host_tree = pinned_lat(batch.kv[tree_rows].reshape(w.B, w.Q, w.C + w.R))
    ldt = buf.q_pe.dtype
    outs = [buf.out_tokens, buf.accept_len, buf.new_len, buf.status]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + \
        host_qpe.numel() * host_qpe.element_size() + host_tree.numel() * host_tree.element_size()
    d2h = sum(t.numel() * t.element_size() for t in outs)
    rope_status = torch.zeros((w.B,), dtype=torch.int32, device=dev)

    def raw(t):  # bf16 device tensors take the host's int16 bit patterns
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t

    # Two input sets (set 0 is the step buffers' own): step i copies its
    # inputs into set i % 2 on a copy stream while step i-1 still computes.
    import types
    in_names = list(host_in.keys())
    sets = [{k: getattr(buf, k) for k in in_names + ["q_pe"]},
            {k: getattr(buf, k).clone() for k in in_names + ["q_pe"]}]
    qraw = [torch.empty_like(buf.q_pe) for _ in range(2)]
    trees = [torch.empty((w.B, w.Q, w.C + w.R), dtype=ldt, device=dev) for _ in range(2)]
    built = [DB.ddt_tree_build(sets[j]["topk_logp"], sets[j]["topk_ids"], sets[j]["root_tok"],
                               w.budget, w.V) for j in range(2)]
    a2 = DB.StepArgs.from_buffer_copy(buf.args)
    for k in in_names + ["q_pe"]:
        setattr(a2, k, sets[1][k].data_ptr())
    step_of = [buf, types.SimpleNamespace(args=a2)]
    houts = [host_out, [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]]

    def copy_body(j):
        for k, h in host_in.items():
            raw(sets[j][k]).copy_(h, non_blocking=True)
        raw(qraw[j]).copy_(host_qpe, non_blocking=True)
        raw(trees[j]).copy_(host_tree, non_blocking=True)

    def comp_body(j):
        tr = DB.ddt_tree_build(sets[j]["topk_logp"], sets[j]["topk_ids"], sets[j]["root_tok"],
                               w.budget, w.V, out=built[j])
        DB.ddt_rope_append(qraw[j], trees[j], buf.kv_cache, buf.block_table, buf.prefix_len,
                           tr["depths"], lay.page_size, q_out=sets[j]["q_pe"],
                           status=rope_status)
        DB.ddt_step(step_of[j])
        for h, t in zip(houts[j], outs):
            h.copy_(t, non_blocking=True)

    def e2e_step():
        copy_body(0)
        comp_body(0)
        torch.cuda.current_stream().synchronize()

    if use_graph:
        # Two graphs per input set: the copies (on a copy stream) and the
        # compute (build, rope + append, the step, results copied out). The
        # compute graph waits for its copy, the next copy into a set waits
        # until the step that read it is done, and the host reads every
        # step's results one step behind.
        cstream, kstream = torch.cuda.Stream(), torch.cuda.current_stream()
        g_copy, g_comp = [], []
        for j in range(2):
            copy_body(j)
            comp_body(j)
            torch.cuda.synchronize()
            gc, gk = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(gc, stream=cstream):
                copy_body(j)
            with torch.cuda.graph(gk):
                comp_body(j)
            g_copy.append(gc)
            g_comp.append(gk)
        torch.cuda.synchronize()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_free = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for j in range(2):
            ev_free[j].record(kstream)
        e2e_state = {"i": 0}

        def e2e_issue():
            i = e2e_state["i"]
            j = i % 2
            cstream.wait_event(ev_free[j])
            with torch.cuda.stream(cstream):
                g_copy[j].replay()
            ev_in[j].record(cstream)
            kstream.wait_event(ev_in[j])
            g_comp[j].replay()
            ev_free[j].record(kstream)
            ev_out[j].record(kstream)
            e2e_state["i"] = i + 1
            return j

        def e2e_run(n):
            """n steps; the host waits for (and reads) step i-1's results
            after issuing step i."""
            prev = None
            for _ in range(n):
                j = e2e_issue()
                if prev is not None:
                    ev_out[prev].synchronize()
                    _ = houts[prev][1][0].item()  # the step's accepted length
                prev = j
            ev_out[prev].synchronize()
            _ = houts[prev][1][0].item()

    n_e2e = args.e2e_steps if args.e2e_steps is not None else max(20, min(args.steps, 2000))
    if use_graph:
        e2e_run(min(3, n_e2e))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_run(n_e2e)
        e2e_s = max(time.perf_counter() - t0, 1e-9)
    else:
        for _ in range(min(3, n_e2e)):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        e2e_s = max(time.perf_counter() - t0, 1e-9)

    st = buf.status.cpu().numpy() | rope_status.cpu().numpy()
    if (st & ~DB.ST_BUDGET_PAD).any():
        raise SystemExit(f"device status reports errors: {st}")

    sum_s = sum(step_ms) / 1e3
    slowest = max_over_ranks(sum_s, world, dev)
    value = world * args.steps / slowest
    flops, byt = attn_work(w, batch.prefix_len, depths, 2 if bf16 else 4)
    attn_s = statistics.mean(attn_ms) / 1e3
    hbm, tf, src = measured_peaks()
    achieved_tf = flops / attn_s / 1e12
    achieved_gb = byt / attn_s / 1e9
    t_roof = max(flops / (tf * 1e12), byt / (hbm * 1e9))
    bound = "tensor" if flops / (tf * 1e12) >= byt / (hbm * 1e9) else "hbm"
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": 1e3 * slowest / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded numpy generators)",
        "config": {"workload": describe(w)},
        "timing": {"parallelism": f"replicas x{world}",
                   "l2": "flushed by a 256 MiB write before every timed step, outside its events",
                   "launch": "cuda_graph replay" if use_graph else "direct C-ABI calls",
                   "bracket_s_incl_flush": bracket_s},
        "roofline": {
            "kernel": "ddt_verify_attn (tcgen05 attention + split merge)" if bf16
                      else "ddt_verify_attn (fp32 SIMT)",
            "bound": bound if bf16 else "alu",
            "achieved": achieved_tf if bound == "tensor" else achieved_gb,
            "peak": tf if bound == "tensor" else hbm,
            "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
            "frac": (achieved_tf / tf) if bound == "tensor" else (achieved_gb / hbm),
            "peak_source": f"{src} (MEASURED_PEAKS.json burst)" if src == "measured" else src,
            "traffic": measured_traffic(w, attn_rows) if bf16 else None,
            "traffic_kernel": f"{attn_kernel_name(attn_rows)} (ncu, one launch)",
            "rows_per_tile": attn_rows, "key_splits": DB.ddt_verify_attn_splits(buf.attn) if bf16 else 1,
            "algorithmic_flops": flops, "algorithmic_bytes": byt,
            "attn_us": attn_s * 1e6, "roofline_us": t_roof * 1e6,
            "frac_of_roofline_time": t_roof / attn_s,
        },
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "e2e": {"value": world * max(n_e2e, 1) / max_over_ranks(e2e_s, world, dev),
                "unit": "steps/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "launch": ("per step a copy graph (pinned host -> one of two device input "
                           "sets, on a copy stream) and a compute graph (ddt_tree_build, "
                           "ddt_rope_append of q_pe and the tree latents at positions L+depth "
                           "into the cache, ddt_step, results -> pinned host); step i's copy "
                           "overlaps step i-1's compute; the host reads every step's results")
                          if use_graph else
                          "the same calls issued directly, then a host synchronize every step"},
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms)},
        "stages": stages,
        "next": next_rows,
    }
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        n, secs, v = oracle_steps(w, batch, args.cpu_seconds, 100000)
        cores, model = cpu_info()
        line["cpu_baseline"] = {"value": v, "unit": "steps/s", "cores": cores, "kind": "oracle",
                                "sample": oracle_sample_text(w, n, model)}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
