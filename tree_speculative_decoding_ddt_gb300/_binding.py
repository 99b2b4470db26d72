"""Thin ctypes binding of ``libddt.so`` (the C ABI in ``include/ddt.h``).

Argument marshalling only: every function takes torch CUDA tensors, checks
their dtype/shape/contiguity, passes raw pointers and the current CUDA stream
to the C entry point of the same name, and raises :class:`DdtError` on a
negative return code. All computation happens in the library's kernels;
there is no CPU fallback. If the library is not built the import of this
module's functions fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# DDT_LIB=checks selects the debug build (device bounds checks recording a
# status, see ddt_debug_checks); anything else, the release library.
LIB_PATH = os.path.join(HERE, "libddt_checks.so" if os.environ.get("DDT_LIB") == "checks"
                        else "libddt.so")

DDT_F32 = 0
DDT_BF16 = 1
DDT_MAX_Q = 128
DDT_OK, DDT_EINVAL, DDT_EUNSUPPORTED, DDT_ELAUNCH, DDT_EWORKSPACE = 0, -1, -2, -3, -4
ST_BUDGET_PAD, ST_INPUT, ST_CYCLE, ST_RANGE, ST_CAPACITY, ST_TIMEOUT, ST_CHECK = 1, 2, 4, 8, 16, 32, 64


class DdtError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with {code}: {msg}")
        self.code = code


class TreeDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("D", ctypes.c_int32), ("K", ctypes.c_int32),
                ("budget", ctypes.c_int32), ("V", ctypes.c_int32)]


class AttnDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Q", ctypes.c_int32), ("H", ctypes.c_int32),
                ("C", ctypes.c_int32), ("R", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("kv_rows", ctypes.c_int64), ("scale", ctypes.c_float),
                ("max_len", ctypes.c_int32)]


_P = ctypes.c_void_p


class StepArgs(ctypes.Structure):
    _fields_ = [("tree", TreeDims), ("attn", AttnDims)] + [
        (n, _P) for n in (
            "topk_logp", "topk_ids", "root_tok", "q_lat", "q_pe", "kv_cache", "block_table",
            "prefix_len", "target_argmax", "tokens", "parents", "depths", "vis_bits", "vis",
            "first_child", "next_sibling", "n_nodes", "out", "lse", "accept_idx", "accept_len",
            "out_tokens", "bonus", "new_len", "status", "workspace")] + [
        ("workspace_bytes", ctypes.c_size_t)]


class LoopArgs(ctypes.Structure):
    _fields_ = [("tree", TreeDims), ("attn", AttnDims), ("theta", ctypes.c_double),
                ("n_new", ctypes.c_int32), ("max_steps", ctypes.c_int32),
                ("golden_len", ctypes.c_int32)] + [
        (n, _P) for n in (
            "golden", "drafter_table", "q_lat", "q_pe", "kv_new", "kv_cache", "block_table",
            "prefix_len0", "prefix_len", "committed", "n_committed", "steps", "accepted",
            "status", "workspace")] + [("workspace_bytes", ctypes.c_size_t)]


#: every symbol the header declares, with (restype, argtypes)
SIGNATURES = {
    "ddt_tree_build": (ctypes.c_int, [ctypes.POINTER(TreeDims)] + [_P] * 13),
    "ddt_verify_attn_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(AttnDims)]),
    "ddt_verify_attn_rows_per_tile": (ctypes.c_int, [ctypes.POINTER(AttnDims)]),
    "ddt_verify_attn_splits": (ctypes.c_int, [ctypes.POINTER(AttnDims)]),
    "ddt_verify_attn": (ctypes.c_int, [ctypes.POINTER(AttnDims)] + [_P] * 10 +
                        [ctypes.c_size_t, _P]),
    "ddt_verify_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(AttnDims)] + [_P] * 10),
    "ddt_tree_accept": (ctypes.c_int, [ctypes.c_int32] * 3 + [_P] * 9),
    "ddt_cache_compact": (ctypes.c_int, [ctypes.c_int32] * 5 + [ctypes.c_int64] + [_P] * 8),
    "ddt_step_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(StepArgs)]),
    "ddt_step": (ctypes.c_int, [ctypes.POINTER(StepArgs), _P]),
    "ddt_target_argmax": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _P, _P,
                                         _P]),
    "ddt_drafter_topk": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_int, _P, _P, _P, _P]),
    "ddt_rope_append": (ctypes.c_int, [ctypes.POINTER(AttnDims), ctypes.c_double] + [_P] * 9),
    "ddt_loop_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(LoopArgs)]),
    "ddt_loop_create": (ctypes.c_int, [ctypes.POINTER(LoopArgs), ctypes.POINTER(_P)]),
    "ddt_loop_launch": (ctypes.c_int, [_P, _P]),
    "ddt_loop_destroy": (ctypes.c_int, [_P]),
    "ddt_wait_selftest": (ctypes.c_int, [_P, _P]),
    "ddt_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "ddt_last_cuda_error": (ctypes.c_int, []),
    "ddt_debug_checks": (ctypes.c_int, [_P, _P]),
    "ddt_cuda_error_name": (ctypes.c_char_p, [ctypes.c_int]),
    "ddt_abi_version": (ctypes.c_int, []),
}

_lib = None


def load(path: Optional[str] = None):
    """Load (once) and return the ctypes handle of the library."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run `python -m tree_speculative_decoding_ddt_gb300"
                          ".build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def debug_checks():
    """(built with checks, failed checks since the last call, first failing
    site) from ddt_debug_checks; reading resets the counts."""
    n, first = ctypes.c_int(0), ctypes.c_int(0)
    built = load().ddt_debug_checks(ctypes.byref(n), ctypes.byref(first))
    return bool(built), n.value, first.value


def _check(fn: str, rc: int):
    if rc != 0:
        lib = load()
        text = lib.ddt_strerror(rc).decode()
        if rc == DDT_ELAUNCH:
            err = lib.ddt_last_cuda_error()
            text += f" ({lib.ddt_cuda_error_name(err).decode()}, {err})"
        raise DdtError(fn, rc, text)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def check_attn_shapes(q_lat, q_pe, kv_cache, block_table, prefix_len, vis_bits):
    """Shape checks shared by the verify-attention wrappers, made before any
    device check or library call: the library sizes its cache views from
    (kv_rows, C + R), so a cache of any other shape would be read past its end.
    Returns (B, Q, H, C, R)."""
    if q_lat.dim() != 4:
        raise ValueError(f"q_lat must be [B, Q, H, C], got {tuple(q_lat.shape)}")
    B, Q, H, C = (int(x) for x in q_lat.shape)
    if q_pe.dim() != 4 or tuple(q_pe.shape[:3]) != (B, Q, H):
        raise ValueError(f"q_pe must be [B, Q, H, R] = [{B}, {Q}, {H}, R], "
                         f"got {tuple(q_pe.shape)}")
    R = int(q_pe.shape[3])
    if kv_cache.dim() != 2 or int(kv_cache.shape[1]) != C + R:
        raise ValueError(f"kv_cache must be [rows, C+R] = [rows, {C + R}], "
                         f"got {tuple(kv_cache.shape)}")
    if block_table.dim() != 2 or int(block_table.shape[0]) != B:
        raise ValueError(f"block_table must be [B, max_pages] with B = {B}, "
                         f"got {tuple(block_table.shape)}")
    if tuple(prefix_len.shape) != (B,):
        raise ValueError(f"prefix_len must be [{B}], got {tuple(prefix_len.shape)}")
    W = (Q + 63) // 64
    if tuple(vis_bits.shape) != (B, Q, W):
        raise ValueError(f"vis_bits must be [{B}, {Q}, {W}], got {tuple(vis_bits.shape)}")
    return B, Q, H, C, R


def ddt_tree_build(topk_logp: torch.Tensor, topk_ids: torch.Tensor, root_tok: torch.Tensor,
                   budget: int, V: int, with_vis: bool = False, out: Optional[dict] = None,
                   stream=None) -> dict:
    """A. Best-first draft tree. Returns tokens/parents/depths/first_child/
    next_sibling (int32 [B,Q]), vis_bits (int64 [B,Q,W], the uint64 words),
    vis (uint8 [B,Q,Q] or None), n_nodes and status (int32 [B])."""
    B, D, K = topk_logp.shape
    Q = budget + 1
    W = (Q + 63) // 64
    dev = topk_logp.device
    _need(topk_logp, "topk_logp", torch.float32)
    _need(topk_ids, "topk_ids", torch.int32, (B, D, K))
    _need(root_tok, "root_tok", torch.int32, (B,))
    o = out if out is not None else {}
    for k in ("tokens", "parents", "depths", "first_child", "next_sibling"):
        o.setdefault(k, torch.empty((B, Q), dtype=torch.int32, device=dev))
    o.setdefault("vis_bits", torch.empty((B, Q, W), dtype=torch.int64, device=dev))
    if with_vis:
        o.setdefault("vis", torch.empty((B, Q, Q), dtype=torch.uint8, device=dev))
    o.setdefault("n_nodes", torch.empty((B,), dtype=torch.int32, device=dev))
    o.setdefault("status", torch.empty((B,), dtype=torch.int32, device=dev))
    dims = TreeDims(B, D, K, budget, V)
    rc = load().ddt_tree_build(ctypes.byref(dims), _ptr(topk_logp), _ptr(topk_ids),
                               _ptr(root_tok), _ptr(o["tokens"]), _ptr(o["parents"]),
                               _ptr(o["depths"]), _ptr(o["vis_bits"]), _ptr(o.get("vis")),
                               _ptr(o["first_child"]), _ptr(o["next_sibling"]),
                               _ptr(o["n_nodes"]), _ptr(o["status"]), _stream(stream))
    _check("ddt_tree_build", rc)
    return o


def attn_dims(B, Q, H, C, R, page_size, max_pages, kv_rows, dtype, scale, max_len) -> AttnDims:
    return AttnDims(B, Q, H, C, R, page_size, max_pages, dtype, kv_rows, scale, max_len)


def ddt_verify_attn_workspace_size(dims: AttnDims) -> int:
    return int(load().ddt_verify_attn_workspace_size(ctypes.byref(dims)))


def ddt_verify_attn_rows_per_tile(dims: AttnDims) -> int:
    """Query rows per tile (128 or 256) of the bf16 verify attention for these
    dims on the current device; 0 for invalid or fp32 dims."""
    return int(load().ddt_verify_attn_rows_per_tile(ctypes.byref(dims)))


def ddt_verify_attn_splits(dims: AttnDims) -> int:
    """Key ranges per sequence of the bf16 verify attention for these dims on
    the current device (1 = no merge pass); 0 for invalid or fp32 dims."""
    return int(load().ddt_verify_attn_splits(ctypes.byref(dims)))


def ddt_verify_attn(q_lat, q_pe, kv_cache, block_table, prefix_len, vis_bits, scale: float,
                    page_size: int, max_len: int, out=None, lse=None, status=None,
                    workspace=None, stream=None):
    """B. Tree-verify MLA-absorb attention. ``q_lat`` [B,Q,H,C], ``q_pe``
    [B,Q,H,R], ``kv_cache`` [rows, C+R] (float32 or bfloat16), ``block_table``
    int32 [B,max_pages], ``prefix_len`` int32 [B], ``vis_bits`` int64 [B,Q,W].
    Returns (out, lse, status)."""
    B, Q, H, C, R = check_attn_shapes(q_lat, q_pe, kv_cache, block_table, prefix_len, vis_bits)
    dt = q_lat.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise TypeError("q_lat must be float32 or bfloat16")
    dtype = DDT_F32 if dt == torch.float32 else DDT_BF16
    _need(q_lat, "q_lat", dt)
    _need(q_pe, "q_pe", dt, (B, Q, H, R))
    _need(kv_cache, "kv_cache", dt)
    _need(block_table, "block_table", torch.int32)
    _need(prefix_len, "prefix_len", torch.int32, (B,))
    _need(vis_bits, "vis_bits", torch.int64, (B, Q, (Q + 63) // 64))
    dev = q_lat.device
    dims = attn_dims(B, Q, H, C, R, page_size, block_table.shape[1], kv_cache.shape[0], dtype,
                     scale, max_len)
    if out is None:
        out = torch.empty((B, Q, H, C), dtype=dt, device=dev)
    if lse is None:
        lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros((B,), dtype=torch.int32, device=dev)
    ws_bytes = ddt_verify_attn_workspace_size(dims)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    rc = load().ddt_verify_attn(ctypes.byref(dims), _ptr(q_lat), _ptr(q_pe), _ptr(kv_cache),
                                _ptr(block_table), _ptr(prefix_len), _ptr(vis_bits), _ptr(out),
                                _ptr(lse), _ptr(status), _ptr(workspace),
                                workspace.numel() if workspace is not None else 0,
                                _stream(stream))
    _check("ddt_verify_attn", rc)
    return out, lse, status


def ddt_verify_attn_noalloc(q_lat, q_pe, kv_cache, block_table, prefix_len, vis_bits,
                            scale: float, page_size: int, max_len: int, out=None, lse=None,
                            status=None, stream=None):
    """B'. :func:`ddt_verify_attn` (bf16 only) with the split-KV scratch taken
    from the library's fixed device array instead of a caller workspace, for
    callers that cannot allocate device memory. Calls that may overlap on the
    GPU share that array and must be serialised. Returns (out, lse, status)."""
    B, Q, H, C, R = check_attn_shapes(q_lat, q_pe, kv_cache, block_table, prefix_len, vis_bits)
    _need(q_lat, "q_lat", torch.bfloat16)
    _need(q_pe, "q_pe", torch.bfloat16, (B, Q, H, R))
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(prefix_len, "prefix_len", torch.int32, (B,))
    _need(vis_bits, "vis_bits", torch.int64, (B, Q, (Q + 63) // 64))
    dev = q_lat.device
    dims = attn_dims(B, Q, H, C, R, page_size, block_table.shape[1], kv_cache.shape[0], DDT_BF16,
                     scale, max_len)
    if out is None:
        out = torch.empty((B, Q, H, C), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros((B,), dtype=torch.int32, device=dev)
    rc = load().ddt_verify_attn_noalloc(ctypes.byref(dims), _ptr(q_lat), _ptr(q_pe),
                                        _ptr(kv_cache), _ptr(block_table), _ptr(prefix_len),
                                        _ptr(vis_bits), _ptr(out), _ptr(lse), _ptr(status),
                                        _stream(stream))
    _check("ddt_verify_attn_noalloc", rc)
    return out, lse, status


def ddt_wait_selftest(stream=None) -> list:
    """Runs the bounded-wait self-test (about a second); returns [status of a
    wait nothing completes, status of a completed wait, milliseconds the
    first wait lasted]."""
    out = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    _check("ddt_wait_selftest", load().ddt_wait_selftest(_ptr(out), _stream(stream)))
    return [int(x) for x in out.cpu()]


def ddt_tree_accept(tokens, parents, target_argmax, D: int, status=None, stream=None) -> dict:
    """C. Greedy accept walk; returns accept_idx/out_tokens [B,D+1],
    accept_len/bonus/status [B]."""
    B, Q = tokens.shape
    for n, t in (("tokens", tokens), ("parents", parents), ("target_argmax", target_argmax)):
        _need(t, n, torch.int32, (B, Q))
    dev = tokens.device
    o = dict(accept_idx=torch.empty((B, D + 1), dtype=torch.int32, device=dev),
             accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
             out_tokens=torch.empty((B, D + 1), dtype=torch.int32, device=dev),
             bonus=torch.empty((B,), dtype=torch.int32, device=dev),
             status=status if status is not None else torch.zeros((B,), dtype=torch.int32,
                                                                    device=dev))
    rc = load().ddt_tree_accept(B, Q, D, _ptr(tokens), _ptr(parents), _ptr(target_argmax),
                                _ptr(o["accept_idx"]), _ptr(o["accept_len"]),
                                _ptr(o["out_tokens"]), _ptr(o["bonus"]), _ptr(o["status"]),
                                _stream(stream))
    _check("ddt_tree_accept", rc)
    return o


def ddt_target_argmax(logits: torch.Tensor, out: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """Greedy token at every tree slot: int32 argmax over the last axis of
    ``logits`` (bf16 or f32, contiguous, any leading shape)."""
    if not isinstance(logits, torch.Tensor) or not logits.is_cuda:
        raise TypeError("logits must be a CUDA tensor")
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"logits must be bfloat16 or float32, got {logits.dtype}")
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    V = int(logits.shape[-1])
    lead = tuple(logits.shape[:-1])
    rows = int(logits.numel() // max(V, 1))
    if out is None:
        out = torch.empty(lead, dtype=torch.int32, device=logits.device)
    else:
        _need(out, "out", torch.int32, lead)
    dt = DDT_BF16 if logits.dtype == torch.bfloat16 else DDT_F32
    rc = load().ddt_target_argmax(rows, V, dt, _ptr(logits), _ptr(out), _stream(stream))
    _check("ddt_target_argmax", rc)
    return out


def ddt_drafter_topk(logits: torch.Tensor, K: int, out: Optional[dict] = None,
                     stream=None) -> dict:
    """Per-depth top-K of the drafter: logits (bf16 or f32, contiguous,
    [..., V]) -> topk_logp float32 [..., K] and topk_ids int32 [..., K] (the
    tree builder's inputs)."""
    if not isinstance(logits, torch.Tensor) or not logits.is_cuda:
        raise TypeError("logits must be a CUDA tensor")
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"logits must be bfloat16 or float32, got {logits.dtype}")
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    V = int(logits.shape[-1])
    lead = tuple(logits.shape[:-1])
    rows = int(logits.numel() // max(V, 1))
    dev = logits.device
    o = out if out is not None else dict(
        topk_logp=torch.empty(lead + (K,), dtype=torch.float32, device=dev),
        topk_ids=torch.empty(lead + (K,), dtype=torch.int32, device=dev))
    _need(o["topk_logp"], "topk_logp", torch.float32, lead + (K,))
    _need(o["topk_ids"], "topk_ids", torch.int32, lead + (K,))
    dt = DDT_BF16 if logits.dtype == torch.bfloat16 else DDT_F32
    rc = load().ddt_drafter_topk(rows, V, K, dt, _ptr(logits), _ptr(o["topk_logp"]),
                                 _ptr(o["topk_ids"]), _stream(stream))
    _check("ddt_drafter_topk", rc)
    return o


def ddt_rope_append(q_pe, kv_new, kv_cache, block_table, prefix_len, depths, page_size: int,
                    theta: float = 10000.0, q_out=None, status=None, stream=None):
    """Rotary embedding of the tree at positions ``prefix_len + depth`` and
    append of the tree latents to the paged cache. ``q_pe`` [B,Q,H,R] (turned
    into ``q_out``; ``q_out=q_pe`` rotates in place), ``kv_new`` [B,Q,C+R]
    (latent part, then the unrotated rope part) written to cache slots
    ``[L, L+Q)`` of ``kv_cache`` [rows, C+R]; ``depths`` int32 [B,Q] from the
    tree build. Returns (q_out, status)."""
    B, Q, H, R = q_pe.shape
    dt = q_pe.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise TypeError("q_pe must be float32 or bfloat16")
    _need(q_pe, "q_pe", dt)
    CR = int(kv_new.shape[-1])
    _need(kv_new, "kv_new", dt, (B, Q, CR))
    _need(kv_cache, "kv_cache", dt)
    if kv_cache.dim() != 2 or kv_cache.shape[1] != CR:
        raise ValueError("kv_cache must be [rows, C+R]")
    _need(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or int(block_table.shape[0]) != B:
        raise ValueError(f"block_table must be [B, max_pages] with B = {B}")
    _need(prefix_len, "prefix_len", torch.int32, (B,))
    _need(depths, "depths", torch.int32, (B, Q))
    dev = q_pe.device
    if q_out is None:
        q_out = torch.empty_like(q_pe)
    _need(q_out, "q_out", dt, (B, Q, H, R))
    if status is None:
        status = torch.zeros((B,), dtype=torch.int32, device=dev)
    dims = attn_dims(B, Q, H, CR - R, R, page_size, block_table.shape[1], kv_cache.shape[0],
                     DDT_F32 if dt == torch.float32 else DDT_BF16, 1.0, 0)
    rc = load().ddt_rope_append(ctypes.byref(dims), float(theta), _ptr(depths), _ptr(prefix_len),
                                _ptr(block_table), _ptr(q_pe), _ptr(q_out), _ptr(kv_new),
                                _ptr(kv_cache), _ptr(status), _stream(stream))
    _check("ddt_rope_append", rc)
    return q_out, status


def ddt_cache_compact(kv_cache, block_table, prefix_len, accept_idx, accept_len, page_size: int,
                      status=None, stream=None):
    """D. In-place gather of the accepted-path rows of ``kv_cache`` [rows, ...];
    returns (new_len, status)."""
    B = prefix_len.shape[0]
    D = accept_idx.shape[1] - 1
    if not kv_cache.is_cuda or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be a contiguous CUDA tensor")
    rows = kv_cache.shape[0]
    row_bytes = kv_cache[0].numel() * kv_cache.element_size() if rows else 0
    _need(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or int(block_table.shape[0]) != B:
        raise ValueError(f"block_table must be [B, max_pages] with B = {B}")
    _need(prefix_len, "prefix_len", torch.int32, (B,))
    _need(accept_idx, "accept_idx", torch.int32, (B, D + 1))
    _need(accept_len, "accept_len", torch.int32, (B,))
    dev = kv_cache.device
    new_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if status is None:
        status = torch.zeros((B,), dtype=torch.int32, device=dev)
    rc = load().ddt_cache_compact(B, D, row_bytes, page_size, block_table.shape[1], rows,
                                  _ptr(kv_cache), _ptr(block_table), _ptr(prefix_len),
                                  _ptr(accept_idx), _ptr(accept_len), _ptr(new_len),
                                  _ptr(status), _stream(stream))
    _check("ddt_cache_compact", rc)
    return new_len, status


class StepBuffers:
    """Device buffers of one verify step (inputs filled by the caller, outputs
    written by :func:`ddt_step`). Built once and reused across steps."""

    def __init__(self, B, D, K, budget, V, H, C, R, page_size, max_pages, kv_rows, dtype,
                 scale, max_len, device="cuda", with_vis=False):
        Q = budget + 1
        W = (Q + 63) // 64
        tdt = torch.float32 if dtype == DDT_F32 else torch.bfloat16
        i32 = dict(dtype=torch.int32, device=device)
        self.tree = TreeDims(B, D, K, budget, V)
        self.attn = attn_dims(B, Q, H, C, R, page_size, max_pages, kv_rows, dtype, scale, max_len)
        self.topk_logp = torch.empty((B, D, K), dtype=torch.float32, device=device)
        self.topk_ids = torch.empty((B, D, K), **i32)
        self.root_tok = torch.empty((B,), **i32)
        self.q_lat = torch.empty((B, Q, H, C), dtype=tdt, device=device)
        self.q_pe = torch.empty((B, Q, H, R), dtype=tdt, device=device)
        self.kv_cache = torch.empty((kv_rows, C + R), dtype=tdt, device=device)
        self.block_table = torch.empty((B, max_pages), **i32)
        self.prefix_len = torch.empty((B,), **i32)
        self.target_argmax = torch.empty((B, Q), **i32)
        for k in ("tokens", "parents", "depths", "first_child", "next_sibling"):
            setattr(self, k, torch.empty((B, Q), **i32))
        self.vis_bits = torch.empty((B, Q, W), dtype=torch.int64, device=device)
        self.vis = torch.empty((B, Q, Q), dtype=torch.uint8, device=device) if with_vis else None
        self.n_nodes = torch.empty((B,), **i32)
        self.out = torch.empty((B, Q, H, C), dtype=tdt, device=device)
        self.lse = torch.empty((B, Q, H), dtype=torch.float32, device=device)
        self.accept_idx = torch.empty((B, D + 1), **i32)
        self.accept_len = torch.empty((B,), **i32)
        self.out_tokens = torch.empty((B, D + 1), **i32)
        self.bonus = torch.empty((B,), **i32)
        self.new_len = torch.empty((B,), **i32)
        self.status = torch.empty((B,), **i32)
        self.args = StepArgs()
        self.args.tree = self.tree
        self.args.attn = self.attn
        ws = int(load().ddt_step_workspace_size(ctypes.byref(self.args)))
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=device)
        for name, _ in StepArgs._fields_[2:-1]:
            t = getattr(self, name)
            setattr(self.args, name, None if t is None else t.data_ptr())
        self.args.workspace_bytes = ws


def ddt_step(buf: StepBuffers, stream=None):
    """A -> B -> C+D on the current stream over the tensors of ``buf``."""
    rc = load().ddt_step(ctypes.byref(buf.args), _stream(stream))
    _check("ddt_step", rc)
    return buf


class DecodeLoop:
    """The multi-step DDTree decode loop on the device (one CUDA graph with a
    conditional WHILE node; see ``ddt_loop_create`` in the C header).

    ``golden`` int32 [B, G] and ``drafter_table`` [B, G, V] stand in for the
    target and the drafter; ``q_lat`` [B,Q,H,C], ``q_pe`` [B,Q,H,R] and
    ``kv_new`` [B,Q,C+R] are the fixed projections each step attends with;
    ``kv_cache`` [rows, C+R], ``block_table`` int32 [B, max_pages] and
    ``prefix_len0`` int32 [B] describe the cache. All CUDA tensors of one
    element type (float32 or bfloat16) except the int32 ones. Outputs live in
    device tensors read by :meth:`results`."""

    def __init__(self, golden, drafter_table, q_lat, q_pe, kv_new, kv_cache, block_table,
                 prefix_len0, D: int, K: int, budget: int, n_new: int, max_steps: int,
                 page_size: int, scale: float, max_len: int, theta: float = 10000.0):
        B, G = golden.shape
        V = int(drafter_table.shape[-1])
        Q = budget + 1
        dt = q_lat.dtype
        if dt not in (torch.float32, torch.bfloat16):
            raise TypeError("q_lat must be float32 or bfloat16")
        H, C = q_lat.shape[2], q_lat.shape[3]
        R = q_pe.shape[-1]
        _need(golden, "golden", torch.int32, (B, G))
        _need(drafter_table, "drafter_table", dt, (B, G, V))
        _need(q_lat, "q_lat", dt, (B, Q, H, C))
        _need(q_pe, "q_pe", dt, (B, Q, H, R))
        _need(kv_new, "kv_new", dt, (B, Q, C + R))
        _need(kv_cache, "kv_cache", dt)
        if kv_cache.dim() != 2 or int(kv_cache.shape[1]) != C + R:
            raise ValueError(f"kv_cache must be [rows, C+R] = [rows, {C + R}], "
                             f"got {tuple(kv_cache.shape)}")
        _need(block_table, "block_table", torch.int32)
        if block_table.dim() != 2 or int(block_table.shape[0]) != B:
            raise ValueError(f"block_table must be [B, max_pages] with B = {B}")
        _need(prefix_len0, "prefix_len0", torch.int32, (B,))
        dev = q_lat.device
        i32 = dict(dtype=torch.int32, device=dev)
        self.prefix_len = torch.empty((B,), **i32)
        self.committed = torch.empty((B, n_new + 1), **i32)
        self.n_committed = torch.empty((B,), **i32)
        self.steps = torch.empty((B,), **i32)
        self.accepted = torch.empty((B, max_steps), **i32)
        self.status = torch.empty((B,), **i32)
        self._keep = (golden, drafter_table, q_lat, q_pe, kv_new, kv_cache, block_table,
                      prefix_len0)
        a = LoopArgs()
        a.tree = TreeDims(B, D, K, budget, V)
        a.attn = attn_dims(B, Q, H, C, R, page_size, block_table.shape[1], kv_cache.shape[0],
                           DDT_F32 if dt == torch.float32 else DDT_BF16, scale, max_len)
        a.theta, a.n_new, a.max_steps, a.golden_len = float(theta), n_new, max_steps, G
        for name, tsr in (("golden", golden), ("drafter_table", drafter_table), ("q_lat", q_lat),
                          ("q_pe", q_pe), ("kv_new", kv_new), ("kv_cache", kv_cache),
                          ("block_table", block_table), ("prefix_len0", prefix_len0),
                          ("prefix_len", self.prefix_len), ("committed", self.committed),
                          ("n_committed", self.n_committed), ("steps", self.steps),
                          ("accepted", self.accepted), ("status", self.status)):
            setattr(a, name, tsr.data_ptr())
        ws = int(load().ddt_loop_workspace_size(ctypes.byref(a)))
        if ws == 0:
            raise DdtError("ddt_loop_workspace_size", -1, "invalid loop arguments")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        a.workspace, a.workspace_bytes = self.workspace.data_ptr(), ws
        self.args = a
        h = _P()
        _check("ddt_loop_create", load().ddt_loop_create(ctypes.byref(a), ctypes.byref(h)))
        self._h = h

    def launch(self, stream=None):
        """Run the whole loop on ``stream`` (asynchronously)."""
        if self._h is None:
            raise RuntimeError("loop destroyed")
        _check("ddt_loop_launch", load().ddt_loop_launch(self._h, _stream(stream)))

    def results(self) -> dict:
        """Host copies of the loop's outputs (synchronises)."""
        torch.cuda.synchronize()
        return {k: getattr(self, k).cpu().numpy() for k in
                ("committed", "n_committed", "steps", "accepted", "status", "prefix_len")}

    def close(self):
        if getattr(self, "_h", None) is not None:
            load().ddt_loop_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
