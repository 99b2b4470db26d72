"""CPU oracle of the DDTree verify step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct restatements of the four steps of one verify
step, written for checking the CUDA path and never called by it:

* :func:`tree_build`       best-first draft-tree construction (Python ``heapq``)
* :func:`verify_attention` tree-verify MLA-absorb attention in float64
* :func:`tree_accept`      greedy walk from the root, bonus token
* :func:`cache_compact`    gather of the accepted-path latents
* :func:`target_argmax`    the target's greedy token at every tree slot (the
                           input of tree_accept, one step upstream)
* :func:`drafter_topk`     the drafter's per-depth top-K log-probs (the input
                           of tree_build, one step upstream)
* :func:`rope_append`      NeoX rotary embedding of the tree's rope parts at
                           positions L+depth and the append of the tree
                           latents to the cache (just before the attention)
* :func:`decode_loop_table` the multi-step DDTree decode loop with a table
                           drafter (per-position logits) and a stream target

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module. It shares no code with the CUDA path:
it imports nothing from the package, and the status codes below are this
module's own copy of the values the C header documents.

Sources (page title, then section):

* "The Milestone Commit: Cementing a Native DDTree Inference Engine",
  "What the Message Actually Does" (commit message: GPU best-first tree
  builder, double accumulation for parity, ancestor-bitmask visibility,
  first-child/next-sibling retrieve, worker padding) and "The Reasoning Behind
  the Architecture" (how each of those works).
* same page, "Mistakes and Incorrect Assumptions": tree_accept needed a
  safety bound after cyclic random test data crashed it.
* "The Checkpoint: Committing a Working Native DDTree Engine", "The Message":
  attention via verify_attn in MLA absorb form; KV-cache scheme "process
  [verified_id, drafts] at positions L+depth, prefix = cache len,
  mask = [ones | visibility]; AR = degenerate q_len = 1; after accept gather
  accepted-path latents"; the greedy invariant DDTree == AR == golden and the
  oracle drafter's 8.00 accepted tokens per step.
* The verify-step specification this library implements fixes what the pages
  leave open: node score = sum of log-probs along the path, heap pops the
  best node and pushes its first child and its next sibling, ties break by
  lower depth then lower rank, construction stops at the token budget.

Readings of points the sources leave open:

* heap key ``(-score, depth, rank, parent_index)``; the parent index is this
  library's extension and makes the order total;
* a child's score is ``score(parent) + float(logp)`` in double precision, also
  for next siblings (never derived from the sibling's score);
* all children at depth ``d`` take their candidates from row ``d-1`` of the
  drafter's per-depth top-k (root depth 0);
* nodes are indexed in pop order (root 0), so ``parent < child``;
* slots past the last node ("worker padding"): token 0, parent -1, depth -1,
  visible to itself only, no children; status bit ``ST_BUDGET_PAD``;
* a NaN/inf log-prob or a token outside ``[0, V)`` is an input error: the tree
  is the root alone and status bit ``ST_INPUT`` is set;
* accept follows the lowest-index child whose token equals the target argmax
  at its parent, at most ``D`` hops, and stops with ``ST_CYCLE`` if it would
  revisit a node;
* compaction reads every source row before writing any destination row;
* rotary embedding: the NeoX pairing (i, i + R/2) with frequencies
  ``theta ** (-2i/R)`` and base ``theta`` a parameter (YaRN scaling is out of
  scope); a tree slot's position is ``L + depth`` and a padding slot
  (depth -1) takes position ``L``; the tree latents of slot t go to cache
  slot ``L + t`` with their rope part rotated and their latent part copied;
  a sequence whose slots ``[L, L+Q)`` leave its pages or the cache is left
  untouched with the capacity / range status bit.
"""
from __future__ import annotations

import heapq
import math

import numpy as np

# Per-sequence status bits (the library's C header documents the same values).
ST_OK = 0
ST_BUDGET_PAD = 1
ST_INPUT = 2
ST_CYCLE = 4
ST_RANGE = 8
ST_CAPACITY = 16


# =============================================================== step A: build

def build_one(logp, ids, root_tok: int, budget: int, V: int):
    """Best-first draft tree of one sequence.

    ``logp``/``ids``: [D, K] per-depth top-k (rank 0 = most likely).
    Returns a dict of Python lists of length ``budget + 1`` plus ``n_nodes``,
    ``status`` and the per-node ``score`` (float64).
    """
    logp = np.asarray(logp, np.float32)
    ids = np.asarray(ids, np.int64)
    D, K = logp.shape
    Q = budget + 1
    status = ST_OK
    ok = bool(np.isfinite(logp).all()) and bool(((ids >= 0) & (ids < V)).all()) \
        and 0 <= int(root_tok) < V

    tokens = [int(root_tok)]
    parents = [-1]
    depths = [0]
    score = [0.0]
    if not ok:
        status |= ST_INPUT
    elif budget > 0 and D > 0 and K > 0:
        # entries: (-score, depth, rank, parent index)
        heap = [(-(0.0 + float(logp[0, 0])), 1, 0, 0)]
        while len(tokens) < Q and heap:
            neg, d, r, par = heapq.heappop(heap)
            s = -neg
            n = len(tokens)
            tokens.append(int(ids[d - 1, r]))
            parents.append(par)
            depths.append(d)
            score.append(s)
            if d < D:  # first child: rank 0 one level down
                heapq.heappush(heap, (-(s + float(logp[d, 0])), d + 1, 0, n))
            if r + 1 < K:  # next sibling, scored from the parent
                heapq.heappush(heap, (-(score[par] + float(logp[d - 1, r + 1])), d, r + 1, par))

    n_nodes = len(tokens)
    if n_nodes < Q:
        status |= ST_BUDGET_PAD
    while len(tokens) < Q:
        tokens.append(0)
        parents.append(-1)
        depths.append(-1)
        score.append(-math.inf)

    # ancestor sets as Python ints: anc[n] = anc[parent] | bit n
    anc = []
    for n in range(Q):
        p = parents[n]
        anc.append((anc[p] if 0 <= p < n else 0) | (1 << n))

    first_child = [-1] * Q
    next_sibling = [-1] * Q
    for c in range(Q):
        p = parents[c]
        if p >= 0 and first_child[p] < 0:
            first_child[p] = c
    for n in range(Q):
        p = parents[n]
        if p < 0:
            continue
        for c in range(n + 1, Q):
            if parents[c] == p:
                next_sibling[n] = c
                break

    return dict(tokens=tokens, parents=parents, depths=depths, anc=anc,
                first_child=first_child, next_sibling=next_sibling,
                n_nodes=n_nodes, status=status, score=score)


def anc_to_words(anc: int, Q: int) -> list:
    W = (Q + 63) // 64
    return [(anc >> (64 * w)) & 0xFFFFFFFFFFFFFFFF for w in range(W)]


def tree_build(topk_logp, topk_ids, root_tok, budget: int, V: int):
    """Batched :func:`build_one`; returns numpy arrays shaped like the C ABI's
    outputs: tokens/parents/depths/first_child/next_sibling i32 [B, Q],
    vis_bits u64 [B, Q, W], vis u8 [B, Q, Q], n_nodes/status i32 [B]."""
    topk_logp = np.asarray(topk_logp, np.float32)
    B = topk_logp.shape[0]
    Q = budget + 1
    W = (Q + 63) // 64
    out = {k: np.zeros((B, Q), np.int32) for k in
           ("tokens", "parents", "depths", "first_child", "next_sibling")}
    out["vis_bits"] = np.zeros((B, Q, W), np.uint64)
    out["vis"] = np.zeros((B, Q, Q), np.uint8)
    out["n_nodes"] = np.zeros(B, np.int32)
    out["status"] = np.zeros(B, np.int32)
    out["score"] = np.zeros((B, Q), np.float64)
    for b in range(B):
        t = build_one(topk_logp[b], topk_ids[b], int(root_tok[b]), budget, V)
        for k in ("tokens", "parents", "depths", "first_child", "next_sibling"):
            out[k][b] = t[k]
        out["score"][b] = t["score"]
        for n in range(Q):
            out["vis_bits"][b, n] = anc_to_words(t["anc"][n], Q)
            for j in range(Q):
                out["vis"][b, n, j] = (t["anc"][n] >> j) & 1
        out["n_nodes"][b] = t["n_nodes"]
        out["status"][b] = t["status"]
    return out


# ===================================================== step B: verify attention

def visible_tree_slots(vis_bits_row, Q: int) -> np.ndarray:
    """bool [Q]: which tree slots a query row may attend to."""
    words = [int(x) for x in np.asarray(vis_bits_row, np.uint64)]
    return np.array([(words[t // 64] >> (t % 64)) & 1 for t in range(Q)], bool)


def slot_rows(block_table_row, page_size: int, slots) -> np.ndarray:
    slots = np.asarray(slots, np.int64)
    pages = np.asarray(block_table_row, np.int64)[slots // page_size]
    return pages * page_size + slots % page_size


def verify_attention(q_lat, q_pe, kv, block_table, prefix_len, vis_bits, scale: float,
                     page_size: int, rows=None, max_pages=None, with_status=False):
    """Tree-verify MLA-absorb attention in float64.

    For sequence ``b``, tree query ``i`` and head ``h``::

        s_j = (q_lat[b,i,h] . c_kv[j] + q_pe[b,i,h] . k_pe[j]) * scale
        j ranges over the prefix slots [0, L_b) (always visible) and the tree
        slots L_b + t with t visible from i; p = softmax(s); o = sum_j p_j c_kv[j]

    ``kv`` rows are ``[c_kv | k_pe]``; slot ``s`` of sequence ``b`` lives in
    physical row ``block_table[b][s // page_size] * page_size + s % page_size``.
    Inputs are upcast to float64 exactly (bf16/fp32 values). ``scale`` is the
    float32 scale the kernels receive. ``rows`` optionally restricts the work
    to a list of ``(b, i)`` pairs (other rows are left as NaN).
    A sequence with ``L < 0`` or ``L + Q > max_pages * page_size`` gets
    ``ST_CAPACITY``, one whose pages of ``[0, L + Q)`` fall outside ``kv``
    gets ``ST_RANGE``; its output is 0 and its lse -inf.
    Returns ``o`` float64 [B, Q, H, C] and ``lse`` float64 [B, Q, H] (and the
    per-sequence status when ``with_status``).
    """
    q_lat = np.asarray(q_lat)
    B, Q, H, C = q_lat.shape
    o = np.full((B, Q, H, C), np.nan)
    lse = np.full((B, Q, H), np.nan)
    sc = float(np.float32(scale))
    todo = rows if rows is not None else [(b, i) for b in range(B) for i in range(Q)]
    bt = np.asarray(block_table)
    if max_pages is None:
        max_pages = bt.shape[1]
    status = np.zeros(B, np.int32)
    n_pages_kv = len(kv) // page_size
    for b in range(B):
        L = int(prefix_len[b])
        if L < 0 or L + Q > max_pages * page_size:
            status[b] = ST_CAPACITY
        else:
            used = bt[b, : -(-(L + Q) // page_size)]
            if (used < 0).any() or (used >= n_pages_kv).any():
                status[b] = ST_RANGE
    cache = {}
    for b, i in todo:
        L = int(prefix_len[b])
        if status[b]:
            o[b, i] = 0.0
            lse[b, i] = -np.inf
            continue
        if b not in cache:
            keys = np.asarray(kv[slot_rows(block_table[b], page_size, np.arange(L + Q))],
                              np.float64)
            cache = {b: keys}
        keys = cache[b]
        qv = np.concatenate([np.asarray(q_lat[b, i], np.float64),
                             np.asarray(q_pe[b, i], np.float64)], axis=1)  # [H, C+R]
        visible = np.concatenate([np.ones(L, bool), visible_tree_slots(vis_bits[b, i], Q)])
        s = (qv @ keys.T) * sc  # [H, L+Q]
        s[:, ~visible] = -np.inf
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        o[b, i] = (p @ keys[:, :C]) / l
        lse[b, i] = (m + np.log(l))[:, 0]
    if with_status:
        return o, lse, status
    return o, lse


# ============================================================== step C: accept

def accept_one(tokens, parents, target, D: int):
    """Greedy walk of one tree: start at the root, repeatedly move to the
    lowest-index child whose token equals the target argmax at the current
    node, at most ``D`` hops; the bonus token is the target argmax where the
    walk stops. A move to a node already on the path stops the walk with
    ``ST_CYCLE``."""
    Q = len(tokens)
    path = [0]
    status = ST_OK
    cur = 0
    for _ in range(D):
        want = int(target[cur])
        nxt = -1
        for c in range(Q):
            if int(parents[c]) == cur and int(tokens[c]) == want:
                nxt = c
                break
        if nxt < 0:
            break
        if nxt in path:
            status |= ST_CYCLE
            break
        path.append(nxt)
        cur = nxt
    bonus = int(target[cur])
    n = len(path) - 1
    idx = path + [-1] * (D + 1 - len(path))
    out = [int(tokens[c]) for c in path[1:]] + [bonus] + [-1] * (D - n)
    return dict(accept_idx=idx, accept_len=n, out_tokens=out, bonus=bonus, status=status)


def tree_accept(tokens, parents, target_argmax, D: int):
    tokens = np.asarray(tokens)
    B = tokens.shape[0]
    res = dict(accept_idx=np.zeros((B, D + 1), np.int32), accept_len=np.zeros(B, np.int32),
               out_tokens=np.zeros((B, D + 1), np.int32), bonus=np.zeros(B, np.int32),
               status=np.zeros(B, np.int32))
    for b in range(B):
        r = accept_one(tokens[b], parents[b], target_argmax[b], D)
        for k in res:
            res[k][b] = r[k]
    return res


# =========================================================== step D: compaction

def cache_compact(kv, block_table, prefix_len, accept_idx, accept_len, page_size: int,
                  max_pages: int):
    """Gather of the accepted-path latents into contiguous slots.

    For ``d = 1 .. accept_len``: the row at slot ``L + accept_idx[d]`` moves
    to slot ``L + d`` (the root already sits at ``L``); every source row is
    read before any destination row is written. Returns the new cache (a
    copy), ``new_len = L + 1 + accept_len`` and per-sequence status. A
    sequence whose path or slots fall outside ``[0, max_pages * page_size)``,
    or whose pages fall outside ``kv``, is left untouched with ``ST_RANGE``.
    So is one whose list is not a path from the root: nodes are numbered in
    pop order and a parent pops before its child, so the slots of a path
    increase strictly from the root's slot 0 (``accept_idx[0]`` is the root
    and is not read).
    """
    new = np.array(kv, copy=True)
    B = len(prefix_len)
    new_len = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    cap = max_pages * page_size
    for b in range(B):
        L = int(prefix_len[b])
        n = int(accept_len[b])
        D = accept_idx.shape[1] - 1
        src_slots = [L + int(accept_idx[b][d]) for d in range(1, n + 1)] if 0 <= n <= D else None
        path = [0] + [int(accept_idx[b][d]) for d in range(1, n + 1)] if src_slots else [0]
        bad = (src_slots is None or L < 0 or L + n >= cap
               or any(int(accept_idx[b][d]) < 0 for d in range(1, n + 1))
               or any(path[d] <= path[d - 1] for d in range(1, len(path)))
               or any(s >= cap for s in src_slots))
        if not bad:
            rows_used = slot_rows(block_table[b], page_size,
                                  src_slots + [L + d for d in range(1, n + 1)]) if n else []
            bad = any(r < 0 or r >= len(kv) for r in rows_used)
        if bad:
            status[b] = ST_RANGE
            new_len[b] = L
            continue
        data = [np.array(kv[slot_rows(block_table[b], page_size, [s])[0]]) for s in src_slots]
        for d in range(1, n + 1):
            new[slot_rows(block_table[b], page_size, [L + d])[0]] = data[d - 1]
        new_len[b] = L + 1 + n
    return new, new_len, status


# ======================================================= the whole verify step

def ddt_step(topk_logp, topk_ids, root_tok, budget: int, V: int, q_lat, q_pe, kv, block_table,
             prefix_len, scale: float, page_size: int, max_pages: int, target_argmax_fn,
             attention: bool = True, attn_rows=None):
    """build -> verify attention -> accept -> compaction, in that order.

    ``target_argmax_fn(tree) -> int [B, Q]`` stands in for the target model's
    argmax at every tree slot (it needs the tree's slot order)."""
    tree = tree_build(topk_logp, topk_ids, root_tok, budget, V)
    o = lse = None
    attn_status = np.zeros(len(np.asarray(prefix_len)), np.int32)
    if attention:
        o, lse, attn_status = verify_attention(q_lat, q_pe, kv, block_table, prefix_len,
                                               tree["vis_bits"], scale, page_size,
                                               rows=attn_rows, max_pages=max_pages,
                                               with_status=True)
    target = np.asarray(target_argmax_fn(tree), np.int32)
    D = np.asarray(topk_logp).shape[1]
    acc = tree_accept(tree["tokens"], tree["parents"], target, D)
    new_kv, new_len, cst = cache_compact(kv, block_table, prefix_len, acc["accept_idx"],
                                         acc["accept_len"], page_size, max_pages)
    # a step's status is the union of its stages' statuses
    status = tree["status"] | attn_status | acc["status"] | cst
    return dict(tree=tree, o=o, lse=lse, target=target, accept=acc, kv=new_kv,
                new_len=new_len, status=status)


# ================================================ next: target-side argmax

def target_argmax(logits) -> np.ndarray:
    """The target model's greedy token at every tree slot: the index of the
    largest logit over the vocabulary (last axis). "The Checkpoint: Committing a
    Working Native DDTree Engine", "The Message": the target's argmax at each
    tree node is what tree_accept compares the drafted tokens with.

    Ties go to the lowest index; -0.0 equals +0.0; a NaN counts as larger than
    every number (the first NaN wins), as numpy's argmax treats it.
    """
    x = np.asarray(logits, dtype=np.float64)
    return np.argmax(x, axis=-1).astype(np.int32)


# ============================================ next: drafter log-softmax top-K

def drafter_topk(logits, K: int):
    """Per-depth top-K candidates of the drafter from its logits (last axis
    = vocabulary): the K largest logits, ranked by value (descending) then by
    token id (ascending), and their log-probabilities
    ``logit - log(sum(exp(logits)))``. The tree builder's input: "The
    Milestone Commit: Cementing a Native DDTree Inference Engine", "What the
    Message Actually Does" (the GPU tree builder consumes per-depth top-K
    log-probs), and the verify-step specification (node score = sum of the
    log-probs along the path).

    The ranking uses the logits exactly as given; the log-sum-exp is taken in
    float64 (shifted by the row maximum) and the log-probs are handed over as
    float32, as the builder takes them. Returns (logp f32 [..., K],
    ids int32 [..., K]).
    """
    x = np.asarray(logits, dtype=np.float64)
    lead = x.shape[:-1]
    V = x.shape[-1]
    flat = x.reshape(-1, V)
    logp = np.zeros((flat.shape[0], K), np.float32)
    ids = np.zeros((flat.shape[0], K), np.int32)
    cols = np.arange(V)
    for r in range(flat.shape[0]):
        row = flat[r]
        order = np.lexsort((cols, -row))[:K]   # value descending, id ascending
        m = row.max()
        lse = m + math.log(float(np.exp(row - m).sum()))
        ids[r] = order.astype(np.int32)
        logp[r] = (row[order] - lse).astype(np.float32)
    return logp.reshape(lead + (K,)), ids.reshape(lead + (K,))


# ================================ tree positions: rotary embedding + append

def rope_inv_freq(R: int, theta: float) -> np.ndarray:
    """Rotary frequencies of a rope part of width R (even): ``theta ** (-2i/R)``
    for i in [0, R/2), float64. "The Consolidation Point: Validating Generality
    and Wrapping the MVP", "The Journey to This Point" (NeoX-style rotary
    position embeddings in the engine's layers)."""
    i = np.arange(R // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / R)


def rope_neox(x, pos, theta: float) -> np.ndarray:
    """NeoX rotation of the last axis of ``x`` at position ``pos`` (a number,
    or an array broadcasting against ``x``'s leading axes), float64.

    The last axis holds R/2 pairs (x_i, x_{i+R/2}); pair i turns by the angle
    ``pos * theta**(-2i/R)``:
    ``y_i = x_i cos - x_{i+R/2} sin`` and ``y_{i+R/2} = x_{i+R/2} cos + x_i sin``.
    """
    x = np.asarray(x, dtype=np.float64)
    R = x.shape[-1]
    h = R // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(R, theta)
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rope_append(q_pe, kv_new, kv, block_table, prefix_len, depths, page_size: int,
                theta: float):
    """The tree's rotary embedding and cache append, one verify step.

    "The Checkpoint: Committing a Working Native DDTree Engine", "The
    Message": the tree [verified_id, drafts] is processed at positions
    L+depth with prefix = cache length (KV-cache scheme), and the engine's
    model does "cache append" of the new latents before attention (rope is one
    of its ops); "The Consolidation Point", "The Journey to This Point":
    the rotary embedding is the NeoX kind.

    Shapes: q_pe [B,Q,H,R], kv_new [B,Q,C+R] (latent part then unrotated rope
    part), kv [rows, C+R] (the paged cache, not modified), block_table
    [B, max_pages], prefix_len [B], depths [B,Q] (-1 = padding slot).
    For sequence b (L = prefix_len[b]) and slot t: position
    p = L + max(depths[b,t], 0); q_out[b,t] = rope(q_pe[b,t], p) for every
    head; cache slot L + t receives kv_new[b,t] with its last R values
    replaced by rope(them, p). A sequence with L < 0 or L + Q beyond its
    pages gets ST_CAPACITY, one whose pages leave the cache gets ST_RANGE;
    either way nothing of it is written (its q_out rows are NaN here).

    Returns (q_out float64 [B,Q,H,R], kv_out float64 copy of kv with the
    appended rows, status int32 [B]).
    """
    q_pe = np.asarray(q_pe, dtype=np.float64)
    kv_new = np.asarray(kv_new, dtype=np.float64)
    B, Q, H, R = q_pe.shape
    CR = kv_new.shape[-1]
    C = CR - R
    kv_out = np.array(kv, dtype=np.float64, copy=True)
    rows = kv_out.shape[0]
    max_pages = block_table.shape[1]
    q_out = np.full(q_pe.shape, np.nan)
    status = np.zeros(B, np.int32)
    for b in range(B):
        L = int(prefix_len[b])
        if L < 0 or L + Q > max_pages * page_size:
            status[b] |= ST_CAPACITY
            continue
        phys = slot_rows(block_table[b], page_size, np.arange(L, L + Q))
        if (phys < 0).any() or (phys >= rows).any():
            status[b] |= ST_RANGE
            continue
        for t in range(Q):
            p = L + max(int(depths[b][t]), 0)
            q_out[b, t] = rope_neox(q_pe[b, t], p, theta)
            kv_out[phys[t], :C] = kv_new[b, t, :C]
            kv_out[phys[t], C:] = rope_neox(kv_new[b, t, C:], p, theta)
    return q_out, kv_out, status


# =================================================== multi-step decode (loop)

def golden_stream(n: int, V: int, seed: int) -> list:
    """A fixed token stream standing in for the target model's greedy output."""
    g = np.random.default_rng([seed, 7])
    return [int(x) for x in g.integers(0, V, n)]


def decode_loop(golden: list, n_new: int, D: int, K: int, budget: int, V: int,
                drafter_hit: float, seed: int):
    """DDTree greedy decoding against a target whose greedy continuation is
    ``golden`` (the target's argmax after any context that matches ``golden``
    is the next golden token; after a diverged context it is a token that the
    drafter never proposes there). The drafter puts the golden token at rank 0
    of depth ``d`` with probability ``drafter_hit`` (1.0 = the pages' oracle
    drafter) and fills the other ranks with distinct wrong tokens.

    Returns the committed tokens, the number of verify steps and the accepted
    tokens per step -- the quantities behind "DDTree greedy == AR == golden",
    "avg_accept 8.00 tok/step" and "3 verify steps vs 24 AR steps".
    """
    g = np.random.default_rng([seed, 11])
    committed = [golden[0]]
    steps = 0
    per_step = []
    while len(committed) < n_new + 1:
        pos = len(committed)  # index of the next golden token
        logp = np.zeros((D, K), np.float32)
        ids = np.zeros((D, K), np.int32)
        for d in range(D):
            truth = golden[pos + d] if pos + d < len(golden) else 0
            hit = g.random() < drafter_hit
            wrong = []
            while len(wrong) < K:
                t = int(g.integers(0, V))
                if t != truth and t not in wrong:
                    wrong.append(t)
            cand = ([truth] + wrong[: K - 1]) if hit else wrong
            ids[d] = cand
            # a peaked drafter: rank 0 far ahead of the others
            logp[d] = np.array([-0.01] + [-5.0 - r for r in range(1, K)], np.float32)[:K]
        tree = build_one(logp, ids, committed[-1], budget, V)
        Q = budget + 1
        # target argmax at every slot: golden continuation if the path so far
        # matches the golden stream, otherwise a token the drafter never offers
        target = np.zeros(Q, np.int64)
        for n in range(Q):
            if tree["depths"][n] < 0:
                target[n] = V - 1
                continue
            path = []
            c = n
            while c > 0:
                path.append(tree["tokens"][c])
                c = tree["parents"][c]
            path.reverse()
            on_golden = all(path[k] == golden[pos + k] for k in range(len(path)))
            nxt = pos + len(path)
            target[n] = golden[nxt] if (on_golden and nxt < len(golden)) else V - 1
        acc = accept_one(tree["tokens"], tree["parents"], target, D)
        committed.extend(acc["out_tokens"][: acc["accept_len"] + 1])
        per_step.append(acc["accept_len"] + 1)
        steps += 1
    return committed[: n_new + 1], steps, per_step


def ar_decode(golden, n_new: int, V: int) -> list:
    """Autoregressive greedy decoding against the stream target: one target
    step per token, each committing the target's greedy token after the
    context so far (the stream's next token while the context follows the
    stream, else V-1)."""
    out = [int(golden[0])]
    on_stream = True
    while len(out) < n_new + 1:
        nxt = len(out)
        on_stream = on_stream and out[-1] == int(golden[nxt - 1])
        out.append(int(golden[nxt]) if on_stream and nxt < len(golden) else V - 1)
    return out


def decode_loop_table(golden, table, n_new: int, D: int, K: int, budget: int, V: int,
                      max_steps: int):
    """The DDTree decode loop of one sequence, as the native engine's
    generate_ddtree runs it ("The Checkpoint: Committing a Working Native DDTree
    Engine", "The Message": tree_build -> verify -> tree_accept + cache
    compaction per step, with a drafter interface; "DDTree greedy == AR ==
    golden" and the oracle drafter's 8.00 accepted tokens per step).

    Drafter: the row for depth d (1..D) is ``table[n - 1 + d]`` (row g holds
    the logits for stream position g; n = tokens committed so far), turned
    into candidates by :func:`drafter_topk`. Target: at a tree node whose
    path from the root follows the stream, the greedy token is the stream's
    next token, elsewhere V-1. Each step commits the accepted drafts and the
    bonus token; the bonus is the next step's root. Stops once ``n_new``
    tokens follow the first or after ``max_steps`` steps.

    Returns (committed tokens [<= n_new+1], steps, tokens committed by each
    step before the final truncation).
    """
    golden = [int(x) for x in golden]
    G = len(golden)
    committed = [golden[0]]
    per_step = []
    steps = 0
    while len(committed) < n_new + 1 and steps < max_steps:
        n = len(committed)
        rows = np.stack([table[min(n - 1 + d, G - 1)] for d in range(1, D + 1)])
        logp, ids = drafter_topk(rows, K)
        tree = build_one(logp, ids, committed[-1], budget, V)
        Q = budget + 1
        target = np.full(Q, V - 1, np.int64)
        for s in range(Q):
            dep = tree["depths"][s]
            if dep < 0:
                continue
            c, ok = s, True
            while c > 0:
                dc = tree["depths"][c]
                if tree["tokens"][c] != golden[min(n - 1 + dc, G - 1)]:
                    ok = False
                c = tree["parents"][c]
            if ok and n + dep < G:
                target[s] = golden[n + dep]
        acc = accept_one(tree["tokens"], tree["parents"], target, D)
        k = acc["accept_len"] + 1
        committed.extend(acc["out_tokens"][:k])
        per_step.append(k)
        steps += 1
    return committed[: n_new + 1], steps, per_step
