"""Seeded synthetic workloads for the DDTree verify step.

This module only *generates inputs*: the drafter's per-depth top-k candidate
lists, the query and latent tensors, the paged latent-cache layout and a
synthetic target model's argmax. None of the verify step's own arithmetic
(tree build, verify attention, greedy accept, cache compaction) lives here, so
the CUDA path and the CPU oracle can both consume these arrays without sharing
any of the method's code.

Every random draw comes from ``numpy.random.default_rng([config_id, b, stream])``
so any subset of a batch can be regenerated on its own:

=======  ==============================================
stream   what it draws
=======  ==============================================
0        drafter logits (one row of ``V`` per depth)
1        query vectors and cache latents
2        synthetic target: match draws and fallback tokens
3        batch-level draws (prefix lengths, page shuffle, match rates)
4        root token
5        target logits
6        drafter logits
7        decode loop: golden token streams
8        decode loop: drafter table (noise and hit draws)
=======  ==============================================

The workloads follow the pages' setting: Kimi K2.6 MLA dimensions
(kv_lora_rank 512, "The Milestone Commit", section "Input Knowledge
Required"), the tiny validation model's 4 heads / kv_lora 64 ("The Final
Commit", section "The Reasoning Process"), draft trees verified at
``q_len = budget + 1`` and an oracle drafter that always proposes the right
token ("The Checkpoint", section "Assumptions Made").
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

STREAM_DRAFTER = 0
STREAM_LATENT = 1
STREAM_TARGET = 2
STREAM_BATCH = 3
STREAM_ROOT = 4
STREAM_TARGET_LOGITS = 5
STREAM_DRAFTER_LOGITS = 6
STREAM_LOOP_GOLDEN = 7
STREAM_LOOP_DRAFTER = 8

#: rows of the latent cache generated per random-number call (keeps peak host
#: memory bounded and lets any row block be regenerated on its own)
LATENT_BLOCK = 4096


def f32(x: float) -> float:
    """Round a Python float to the nearest float32 value (returned as float)."""
    return float(np.float32(x))


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic verify-step workload.

    ``prefix`` is either an int (every sequence has that many cached tokens)
    or a ``(lo, hi)`` tuple (uniform integer lengths in ``[lo, hi]``).
    ``match_p`` is the probability that the synthetic target's argmax at a
    node equals that node's rank-0 child token; a ``(lo, hi)`` tuple draws
    one rate per sequence. ``page_size=None`` means one contiguous region
    per sequence.
    """

    name: str
    cid: int
    B: int
    D: int
    K: int
    V: int
    budget: int
    H: int
    C: int
    R: int
    prefix: object
    dtype: str  # "f32" or "bf16"
    scale: float
    page_size: Optional[int] = None
    match_p: object = 0.7
    boost_rank0: float = 0.0
    logit_std: float = 2.0

    @property
    def Q(self) -> int:
        return self.budget + 1

    @property
    def W(self) -> int:
        return (self.Q + 63) // 64

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _scale(qk_dim: int) -> float:
    return f32(1.0 / math.sqrt(qk_dim))


#: the five workload shapes. c1 is the tiny fp32 case, c2 the max-budget step
#: (q_len 65 at K2 dimensions), c3 the batched serving step over a paged
#: cache, c4 the deep-tree long-context step with a perfect drafter, c5 the
#: q_len / batch / prefix sweep (instantiated by :func:`sweep_point`).
CONFIGS = {
    "c1": Workload("c1_tiny_f32", 1, B=1, D=4, K=4, V=1024, budget=8, H=4, C=64, R=32,
                   prefix=32, dtype="f32", scale=_scale(96), match_p=0.7),
    "c2": Workload("c2_max_budget", 2, B=1, D=16, K=8, V=163840, budget=64, H=64, C=512,
                   R=64, prefix=4096, dtype="bf16", scale=_scale(192), match_p=0.7),
    "c3": Workload("c3_batched_paged", 3, B=64, D=8, K=4, V=163840, budget=16, H=64, C=512,
                   R=64, prefix=(512, 8192), dtype="bf16", scale=_scale(192), page_size=64,
                   match_p=(0.3, 0.9)),
    "c4": Workload("c4_deep_long", 4, B=8, D=15, K=2, V=163840, budget=64, H=64, C=512,
                   R=64, prefix=32768, dtype="bf16", scale=_scale(192), match_p=1.0,
                   boost_rank0=25.0),
}

SWEEP_QLEN = (1, 9, 17, 33, 65)
SWEEP_BATCH = (1, 8, 64)
SWEEP_PREFIX = (1024, 8192, 65536, 131072)


def sweep_point(q_len: int, batch: int, prefix: int) -> Workload:
    """One point of the q_len x batch x prefix sweep (drafter shaped like c3)."""
    return Workload(f"c5_q{q_len}_b{batch}_l{prefix}", 5, B=batch, D=8, K=4, V=163840,
                    budget=q_len - 1, H=64, C=512, R=64, prefix=prefix, dtype="bf16",
                    scale=_scale(192), match_p=0.7)


def rng(cid: int, b: int, stream: int, *extra: int) -> np.random.Generator:
    return np.random.default_rng([cid, b, stream, *extra])


# --------------------------------------------------------------------------- bf16

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (NaN kept NaN)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # no uint32 overflow for finite inputs (largest is 0xFF7FFFFF + 0x8000); NaNs are set below
    with np.errstate(over="ignore"):
        rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(to_bf16_bits(x))


# ------------------------------------------------------------------------ drafter

def _topk_stable(x: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of ``x``, ties broken by lower index,
    ordered by (value descending, index ascending)."""
    n = x.shape[0]
    k = min(k, n)
    part = np.argpartition(-x, k - 1)[:k]
    kth = x[part].min()
    above = np.flatnonzero(x > kth)
    equal = np.flatnonzero(x == kth)
    cand = np.concatenate([above, equal[: k - above.shape[0]]])
    order = np.lexsort((cand, -x[cand]))
    return cand[order]


def drafter_topk(w: Workload, b: int):
    """Per-depth top-K candidates of sequence ``b``.

    Logits are N(0, ``logit_std``) over the vocabulary (std, numpy's
    convention); ``boost_rank0`` is added to each row's largest logit (the
    near-certain drafter of the deep-tree workload). Log-probs come from a
    float64 log-softmax and are handed over as float32, rank 0 first.
    """
    g = rng(w.cid, b, STREAM_DRAFTER)
    logp = np.zeros((w.D, w.K), np.float32)
    ids = np.zeros((w.D, w.K), np.int32)
    for d in range(w.D):
        x = g.normal(0.0, w.logit_std, w.V)
        if w.boost_rank0:
            x[int(np.argmax(x))] += w.boost_rank0
        top = _topk_stable(x, w.K)
        m = x.max()
        lse = m + math.log(float(np.exp(x - m).sum()))
        logp[d] = (x[top] - lse).astype(np.float32)
        ids[d] = top.astype(np.int32)
    return logp, ids


def root_token(w: Workload, b: int) -> int:
    return int(rng(w.cid, b, STREAM_ROOT).integers(0, w.V))


# ------------------------------------------------------------------- batch draws

def prefix_lengths(w: Workload) -> np.ndarray:
    if isinstance(w.prefix, tuple):
        lo, hi = w.prefix
        return rng(w.cid, 0, STREAM_BATCH, 0).integers(lo, hi + 1, w.B).astype(np.int32)
    return np.full(w.B, int(w.prefix), np.int32)


def match_rates(w: Workload) -> np.ndarray:
    if isinstance(w.match_p, tuple):
        lo, hi = w.match_p
        return rng(w.cid, 0, STREAM_BATCH, 1).uniform(lo, hi, w.B)
    return np.full(w.B, float(w.match_p))


@dataclasses.dataclass
class CacheLayout:
    page_size: int
    max_pages: int
    block_table: np.ndarray  # int32 [B, max_pages]
    total_rows: int

    def rows_of(self, b: int, slots: np.ndarray) -> np.ndarray:
        """Physical cache rows of logical slots of sequence ``b``."""
        slots = np.asarray(slots, np.int64)
        page = self.block_table[b][slots // self.page_size].astype(np.int64)
        return page * self.page_size + slots % self.page_size


def cache_layout(w: Workload, lens: np.ndarray, extra_slots: int = 0) -> CacheLayout:
    """Paged (shuffled page ids) or contiguous layout holding ``L_b + Q`` slots
    (plus ``extra_slots``) for every sequence."""
    need = lens.astype(np.int64) + w.Q + extra_slots
    if w.page_size is None:
        cap = int(-(-int(need.max()) // 64) * 64)
        bt = np.arange(w.B, dtype=np.int32).reshape(w.B, 1)
        return CacheLayout(cap, 1, bt, w.B * cap)
    P = w.page_size
    pages = (-(-need // P)).astype(np.int64)
    max_pages = int(pages.max())
    total = int(pages.sum())
    perm = rng(w.cid, 0, STREAM_BATCH, 2).permutation(total).astype(np.int32)
    bt = np.full((w.B, max_pages), -1, np.int32)
    at = 0
    for b in range(w.B):
        bt[b, : pages[b]] = perm[at: at + pages[b]]
        at += pages[b]
    return CacheLayout(P, max_pages, bt, total * P)


# ---------------------------------------------------------------------- latents

def query_latents(w: Workload, b: int) -> np.ndarray:
    """float32 [Q, H, C+R] (bf16-representable for bf16 workloads)."""
    g = rng(w.cid, b, STREAM_LATENT, 0)
    q = g.standard_normal((w.Q, w.H, w.C + w.R), dtype=np.float32)
    return round_bf16(q) if w.dtype == "bf16" else q


def cache_latents(w: Workload, b: int, n_slots: int, first: int = 0) -> np.ndarray:
    """float32 [n_slots, C+R] latents of logical slots ``first .. first+n_slots``
    of sequence ``b``. Generated in blocks of :data:`LATENT_BLOCK` slots so any
    slot range can be regenerated without the rest."""
    out = np.empty((n_slots, w.C + w.R), np.float32)
    s = first
    while s < first + n_slots:
        blk = s // LATENT_BLOCK
        lo = blk * LATENT_BLOCK
        g = rng(w.cid, b, STREAM_LATENT, 1, blk)
        block = g.standard_normal((LATENT_BLOCK, w.C + w.R), dtype=np.float32)
        take_lo = s - lo
        take_hi = min(LATENT_BLOCK, first + n_slots - lo)
        out[s - first: s - first + (take_hi - take_lo)] = block[take_lo:take_hi]
        s = lo + take_hi
    return round_bf16(out) if w.dtype == "bf16" else out


# ----------------------------------------------------------------------- target

def target_draws(w: Workload, b: int):
    """Per-slot uniform draws and fallback tokens of the synthetic target."""
    g = rng(w.cid, b, STREAM_TARGET)
    u = g.random(w.Q)
    tok = g.integers(0, w.V, w.Q).astype(np.int32)
    return u, tok


def synth_target_argmax(depths: np.ndarray, topk_ids: np.ndarray, u: np.ndarray,
                        fallback: np.ndarray, p: float) -> np.ndarray:
    """Synthetic target model: at a tree slot of depth ``d < D`` the argmax is
    the rank-0 candidate of depth ``d+1`` (the node's rank-0 child token) when
    ``u < p``; otherwise (and at depth-``D`` or padding slots) it is the drawn
    fallback token. ``depths`` is indexed by tree slot."""
    D = topk_ids.shape[0]
    out = np.asarray(fallback, np.int32).copy()
    d = np.asarray(depths)
    ok = (d >= 0) & (d < D) & (np.asarray(u) < p)
    out[ok] = topk_ids[d[ok], 0]
    return out


def target_logits(w: Workload, b: int, winners: Optional[np.ndarray] = None) -> np.ndarray:
    """Synthetic target logits [Q, V] of sequence ``b``: N(0, ``logit_std``)
    (bf16-rounded on bf16 workloads). With ``winners`` (a token per slot) that
    token's logit is raised one unit above the slot's largest, so the slot's
    greedy token is the given one."""
    g = rng(w.cid, b, STREAM_TARGET_LOGITS)
    x = g.normal(0.0, w.logit_std, (w.Q, w.V))
    if winners is not None:
        x[np.arange(w.Q), np.asarray(winners)] = x.max(axis=1) + 1.0
    x = x.astype(np.float32)
    return round_bf16(x) if w.dtype == "bf16" else x


def drafter_logits(w: Workload, b: int) -> np.ndarray:
    """Synthetic drafter logits [D, V] of sequence ``b``: N(0, ``logit_std``)
    with ``boost_rank0`` added to each row's largest entry (bf16-rounded on
    bf16 workloads)."""
    g = rng(w.cid, b, STREAM_DRAFTER_LOGITS)
    x = g.normal(0.0, w.logit_std, (w.D, w.V))
    if w.boost_rank0:
        x[np.arange(w.D), np.argmax(x, axis=1)] += w.boost_rank0
    x = x.astype(np.float32)
    return round_bf16(x) if w.dtype == "bf16" else x


# ---------------------------------------------------------------------- batches

@dataclasses.dataclass
class Batch:
    w: Workload
    topk_logp: np.ndarray      # f32 [B, D, K]
    topk_ids: np.ndarray       # i32 [B, D, K]
    root_tok: np.ndarray       # i32 [B]
    prefix_len: np.ndarray     # i32 [B]
    layout: CacheLayout
    match_p: np.ndarray        # f64 [B]
    target_u: np.ndarray       # f64 [B, Q]
    target_fallback: np.ndarray  # i32 [B, Q]
    q: Optional[np.ndarray] = None    # f32 [B, Q, H, C+R]
    kv: Optional[np.ndarray] = None   # f32 [rows, C+R] physical layout

    @property
    def q_lat(self) -> np.ndarray:
        return np.ascontiguousarray(self.q[..., : self.w.C])

    @property
    def q_pe(self) -> np.ndarray:
        return np.ascontiguousarray(self.q[..., self.w.C:])


def make_batch(w: Workload, latents: bool = True, extra_slots: int = 0) -> Batch:
    lens = prefix_lengths(w)
    layout = cache_layout(w, lens, extra_slots)
    logp = np.zeros((w.B, w.D, w.K), np.float32)
    ids = np.zeros((w.B, w.D, w.K), np.int32)
    root = np.zeros(w.B, np.int32)
    tu = np.zeros((w.B, w.Q))
    tf = np.zeros((w.B, w.Q), np.int32)
    for b in range(w.B):
        logp[b], ids[b] = drafter_topk(w, b)
        root[b] = root_token(w, b)
        tu[b], tf[b] = target_draws(w, b)
    batch = Batch(w, logp, ids, root, lens, layout, match_rates(w), tu, tf)
    if latents:
        q = np.zeros((w.B, w.Q, w.H, w.C + w.R), np.float32)
        kv = np.zeros((layout.total_rows, w.C + w.R), np.float32)
        for b in range(w.B):
            q[b] = query_latents(w, b)
            n = int(lens[b]) + w.Q
            kv[layout.rows_of(b, np.arange(n))] = cache_latents(w, b, n)
        batch.q, batch.kv = q, kv
    return batch


def target_argmax_for(batch: Batch, depths: np.ndarray) -> np.ndarray:
    """Synthetic target argmax [B, Q] for trees whose slot depths are ``depths``."""
    w = batch.w
    out = np.zeros((w.B, w.Q), np.int32)
    for b in range(w.B):
        out[b] = synth_target_argmax(depths[b], batch.topk_ids[b], batch.target_u[b],
                                     batch.target_fallback[b], float(batch.match_p[b]))
    return out


# ------------------------------------------------------------------ decode loop

def loop_golden(cid: int, B: int, G: int, V: int) -> np.ndarray:
    """int32 [B, G]: the synthetic target's greedy token stream of every
    sequence (its continuation of any context that follows the stream).
    Tokens lie in [0, V-1): V-1 is left for the target's answer after a
    context that left the stream."""
    out = np.zeros((B, G), np.int32)
    for b in range(B):
        out[b] = rng(cid, b, STREAM_LOOP_GOLDEN).integers(0, max(V - 1, 1), G)
    return out


def loop_drafter_table(cid: int, golden: np.ndarray, V: int, hit, dtype: str,
                       spike: float = 8.0) -> np.ndarray:
    """float32 [B, G, V]: the synthetic drafter's logits for the token at
    stream position g of sequence b (row g predicts golden[b, g]). Unit
    normal noise; with probability ``hit`` (a number, or one per sequence)
    the golden token is raised ``spike`` above the row's largest noise value,
    so it is the drafter's first candidate. bf16-representable for bf16."""
    B, G = golden.shape
    hits = np.broadcast_to(np.asarray(hit, np.float64), (B,))
    out = np.empty((B, G, V), np.float32)
    for b in range(B):
        g = rng(cid, b, STREAM_LOOP_DRAFTER)
        rows = g.standard_normal((G, V), dtype=np.float32)
        if dtype == "bf16":
            rows = round_bf16(rows)
        draw = g.random(G)
        for j in range(G):
            if draw[j] < hits[b]:
                top = np.array([rows[j].max() + spike], np.float32)
                rows[j, golden[b, j]] = (round_bf16(top) if dtype == "bf16" else top)[0]
        out[b] = rows
    return out


# ------------------------------------------------------------ stress point

def stress_inputs(B: int, D: int, K: int, V: int, device, seed: int = 99):
    """Drafter and target of the build / accept / compaction stress point (B
    sequences, D depths, K >= 2 candidates, budget 2 * D), drawn with torch on
    ``device``: at depth 1 the two best candidates score -0.01 and -0.02, at
    every deeper level the best scores -0.001, all others -30 or less; the K
    candidate tokens of a depth are distinct. The tree's first D pops are then
    the rank-0 chain (slots 1..D, all above -0.02), then the rank-1 child of
    the root (slot D+1) and its rank-0 chain (slots D+2 .. 2D). The target
    picks that rank-1 child at the root and the rank-0 candidate below it, so
    every sequence accepts the D nodes of slots D+1 .. 2D and compaction
    moves D rows (slot D+d to slot d), none of them in place.
    Returns (topk_logp f32 [B,D,K], topk_ids i32 [B,D,K], root_tok i32 [B],
    target_argmax i32 [B, 2D+1])."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    Q = 2 * D + 1
    logp = -torch.rand((B, D, K), generator=gen, device=device) * 4.0 - 30.0
    logp[:, 0, 0] = -0.01
    logp[:, 0, 1] = -0.02
    logp[:, 1:, 0] = -0.001
    logp = logp.sort(dim=-1, descending=True).values.contiguous()
    base = torch.randint(0, V, (B, D, 1), generator=gen, device=device, dtype=torch.int64)
    ids = ((base + torch.arange(K, device=device)) % V).to(torch.int32).contiguous()
    root = torch.randint(0, V, (B,), generator=gen, device=device, dtype=torch.int32)
    target = torch.zeros((B, Q), dtype=torch.int32, device=device)
    target[:, 0] = ids[:, 0, 1]
    target[:, D + 1: 2 * D] = ids[:, 1:, 0]  # slot D+1+k (depth 1+k) -> its rank-0 child
    return logp, ids, root, target
