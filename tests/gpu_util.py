"""Helpers of the GPU parity tests: move seeded workloads to the device and
compare device results with the oracle's."""
import numpy as np
import torch

from tree_speculative_decoding_ddt_gb300 import workloads as WL

DEV = "cuda"


def t(x, dtype=None):
    a = np.ascontiguousarray(x)
    out = torch.from_numpy(a)
    if dtype is not None:
        out = out.to(dtype)
    return out.to(DEV)


def bf16_tensor(x_f32: np.ndarray) -> torch.Tensor:
    """float32 values that are exactly bf16 -> a bfloat16 CUDA tensor (bitwise)."""
    bits = WL.to_bf16_bits(x_f32).view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(bits)).to(DEV).view(torch.bfloat16)


def latent_tensor(x_f32: np.ndarray, dtype: str) -> torch.Tensor:
    return bf16_tensor(x_f32) if dtype == "bf16" else t(x_f32.astype(np.float32))


def u64(x) -> np.ndarray:
    return np.asarray(x.cpu().numpy() if isinstance(x, torch.Tensor) else x).view(np.uint64)


def rel_err_rows(got: np.ndarray, ref: np.ndarray) -> float:
    """max over query rows of max|got-ref| / max|ref| (rows = last axis)."""
    d = np.abs(got.astype(np.float64) - ref).max(axis=-1)
    m = np.abs(ref).max(axis=-1)
    return float((d / np.maximum(m, 1e-300)).max())


def to_f64(x: torch.Tensor) -> np.ndarray:
    return x.float().cpu().numpy().astype(np.float64)
