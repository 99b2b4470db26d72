"""GPU drafter top-K (ddt_drafter_topk through the C ABI) against the oracle:
token ids bit for bit, log-probs within 1e-5 (the fp32 online log-sum-exp
over up to 163840 logits against the oracle's float64 one). Workload shapes,
ragged and misaligned rows (element-by-element path), tie-heavy rows and
-inf entries."""
import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import bf16_tensor, t

pytestmark = pytest.mark.gpu

LOGP_ATOL = 1e-5


def dev_logits(x: np.ndarray, dtype: str) -> torch.Tensor:
    return bf16_tensor(x) if dtype == "bf16" else t(np.ascontiguousarray(x, np.float32))


def check(x: np.ndarray, K: int, dtype: str, view=None):
    xv = WL.round_bf16(x) if dtype == "bf16" else np.asarray(x, np.float32)
    got = DB.ddt_drafter_topk(view if view is not None else dev_logits(xv, dtype), K)
    torch.cuda.synchronize()
    ref_lp, ref_ids = O.drafter_topk(xv, K)
    np.testing.assert_array_equal(got["topk_ids"].cpu().numpy(), ref_ids)
    np.testing.assert_allclose(got["topk_logp"].cpu().numpy(), ref_lp, rtol=0, atol=LOGP_ATOL)


@pytest.mark.parametrize("cfg", ["c2", "c3", "c4"])
def test_workload_drafter_rows(cfg):
    w = WL.CONFIGS[cfg].with_(B=2)
    x = np.stack([WL.drafter_logits(w, b) for b in range(w.B)])  # [B, D, V]
    check(x, w.K, "bf16")


def test_tiny_fp32_workload():
    w = WL.CONFIGS["c1"]
    check(np.stack([WL.drafter_logits(w, b) for b in range(w.B)]), w.K, "f32")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V,K", [(1, 1), (7, 7), (9, 4), (63, 16), (1001, 8), (4099, 3),
                                 (65536, 16)])
def test_ragged_vocab_sizes(dtype, V, K):
    g = np.random.default_rng(V + 100 * K)
    check(g.normal(0, 2, (13, V)), K, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_misaligned_rows_take_the_scalar_path(dtype):
    g = np.random.default_rng(17)
    x = g.normal(0, 2, (6 * 2048 + 1,))
    xv = WL.round_bf16(x) if dtype == "bf16" else x.astype(np.float32)
    view = dev_logits(xv, dtype)[1:].view(6, 2048)
    check(xv[1:].reshape(6, 2048), 16, dtype, view=view)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_tie_heavy_rows_and_minus_inf(dtype):
    g = np.random.default_rng(23)
    x = g.choice(np.array([-np.inf, -1.0, 0.0, 0.5, 1.25, 2.0]), size=(40, 3000),
                 p=[.2, .3, .2, .15, .1, .05])
    x[0, :] = 0.5           # all equal: ids 0..15
    x[1, :] = -np.inf
    x[1, 2999] = 3.0        # one finite entry at the end, log-prob 0
    x[1, :16] = -1.0
    check(x, 16, dtype)


def test_host_argument_errors(lib):
    buf = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    lp = torch.zeros(16, dtype=torch.float32, device="cuda")
    ids = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = (buf.data_ptr(), lp.data_ptr(), ids.data_ptr())
    assert lib.ddt_drafter_topk(1, 64, 4, DB.DDT_BF16, None, p[1], p[2], None) == -1
    assert lib.ddt_drafter_topk(1, 64, 0, DB.DDT_BF16, *p, None) == -1
    assert lib.ddt_drafter_topk(1, 64, 17, DB.DDT_BF16, *p, None) == -2
    assert lib.ddt_drafter_topk(1, 8, 9, DB.DDT_BF16, *p, None) == -2
    assert lib.ddt_drafter_topk(1, 64, 4, 9, *p, None) == -1
