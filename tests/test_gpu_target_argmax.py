"""GPU target-side argmax (ddt_target_argmax through the C ABI) against the
oracle, bit for bit: workload shapes (vocab 163840), ragged vocab sizes that
take the element-by-element path, a misaligned view, and rows crafted with
ties, signed zeros, infinities and NaN."""
import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import bf16_tensor, t

pytestmark = pytest.mark.gpu


def logits_tensor(x: np.ndarray, dtype: str) -> torch.Tensor:
    return bf16_tensor(x) if dtype == "bf16" else t(np.ascontiguousarray(x, np.float32))


def check(x: np.ndarray, dtype: str):
    xv = WL.round_bf16(x) if dtype == "bf16" else x.astype(np.float32)
    got = DB.ddt_target_argmax(logits_tensor(xv, dtype))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), O.target_argmax(xv))


@pytest.mark.parametrize("cfg", ["c2", "c4"])
def test_workload_rows_with_and_without_planted_winners(cfg):
    w = WL.CONFIGS[cfg].with_(B=2)
    for b in range(w.B):
        winners = np.random.default_rng([9, b]).integers(0, w.V, w.Q)
        x = WL.target_logits(w, b, winners)
        check(x, "bf16")
        check(WL.target_logits(w, b), "bf16")


def test_batched_rows_bf16():
    w = WL.CONFIGS["c3"].with_(B=6)
    x = np.stack([WL.target_logits(w, b) for b in range(w.B)])  # [B, Q, V]
    check(x, "bf16")


def test_tiny_fp32_workload():
    w = WL.CONFIGS["c1"]
    check(np.stack([WL.target_logits(w, b) for b in range(w.B)]), "f32")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 63, 1001, 4099, 65536])
def test_ragged_vocab_sizes(dtype, V):
    g = np.random.default_rng(V)
    check(g.normal(0, 2, (37, V)), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_misaligned_rows_take_the_scalar_path(dtype):
    g = np.random.default_rng(11)
    x = g.normal(0, 2, (5 * 4096 + 1,))
    xv = WL.round_bf16(x) if dtype == "bf16" else x.astype(np.float32)
    full = logits_tensor(xv, dtype)
    view = full[1:].view(5, 4096)  # starts 2 or 4 bytes past a 16-byte boundary
    got = DB.ddt_target_argmax(view)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), O.target_argmax(xv[1:].reshape(5, 4096)))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ties_signed_zeros_infinities_nan(dtype):
    g = np.random.default_rng(4)
    vals = np.array([-np.inf, -3.0, -0.0, 0.0, 2.5, np.inf, np.nan])
    x = g.choice(vals, size=(64, 520), p=[.1, .3, .15, .15, .2, .06, .04])
    x[0] = -0.0                     # all signed zeros: index 0
    x[1, :] = -np.inf               # all -inf: index 0
    x[2, :] = 2.5
    x[2, 517] = np.inf              # a lone +inf near the end
    x[3, :] = 1.0
    x[3, 300] = np.nan              # a NaN wins
    check(x, dtype)


def test_host_argument_errors(lib):
    import ctypes
    assert lib.ddt_target_argmax(1, 8, DB.DDT_BF16, None, None, None) == -1
    buf = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.ddt_target_argmax(0, 8, DB.DDT_BF16, buf.data_ptr(), out.data_ptr(), None) == -1
    assert lib.ddt_target_argmax(1, 8, 7, buf.data_ptr(), out.data_ptr(), None) == -1
    assert lib.ddt_target_argmax(1 << 28, 8, DB.DDT_BF16, buf.data_ptr(), out.data_ptr(),
                                 None) == -2
