"""The allocation-free verify attention (ddt_verify_attn_noalloc).

That entry point is for callers that can pass the library their inputs and
outputs but cannot obtain device scratch memory themselves; it runs the same
bf16 kernels with the split-KV scratch taken from a fixed array the library
reserves when it is loaded. These checks call it through the C ABI and
compare it with ddt_verify_attn given a caller workspace, twice in a row (the
array keeps the previous call's contents, which must not leak into the next
result). The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import latent_tensor, t, to_f64

pytestmark = pytest.mark.gpu

BF16_ABS = 2e-2


def _inputs(w):
    batch = WL.make_batch(w)
    tree = O.tree_build(batch.topk_logp, batch.topk_ids, batch.root_tok, w.budget, w.V)
    lay = batch.layout
    args = (latent_tensor(batch.q_lat, "bf16"), latent_tensor(batch.q_pe, "bf16"),
            latent_tensor(batch.kv, "bf16"), t(lay.block_table), t(batch.prefix_len),
            t(tree["vis_bits"].view(np.int64)))
    return batch, args, lay


@pytest.mark.parametrize("cfg,mods", [
    ("c2", {}),                                   # the max-budget step: the key range is split
    ("c3", {"B": 6, "V": 4096, "prefix": (0, 3000)}),  # paged, variable lengths
])
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(cfg, mods, attn_rows):
    w = WL.CONFIGS[cfg].with_(**mods)
    batch, args, lay = _inputs(w)
    max_len = int(batch.prefix_len.max()) + w.Q
    dims = DB.attn_dims(w.B, w.Q, w.H, w.C, w.R, lay.page_size, lay.max_pages, lay.total_rows,
                        DB.DDT_BF16, w.scale, max_len)
    if cfg == "c2":
        assert DB.ddt_verify_attn_workspace_size(dims) > 0  # the scratch is really used
    ref_o, ref_l, ref_s = DB.ddt_verify_attn(*args, w.scale, lay.page_size, max_len)
    for call in range(2):
        o, l, s = DB.ddt_verify_attn_noalloc(*args, w.scale, lay.page_size, max_len)
        torch.cuda.synchronize()
        assert np.abs(to_f64(o) - to_f64(ref_o)).max() <= BF16_ABS, call
        np.testing.assert_allclose(to_f64(l), to_f64(ref_l), rtol=0, atol=BF16_ABS)
        np.testing.assert_array_equal(s.cpu().numpy(), ref_s.cpu().numpy())
    # and against the oracle for good measure
    ref, _ = O.verify_attention(batch.q_lat, batch.q_pe, batch.kv, lay.block_table,
                                batch.prefix_len, O.tree_build(batch.topk_logp, batch.topk_ids,
                                                               batch.root_tok, w.budget,
                                                               w.V)["vis_bits"],
                                w.scale, lay.page_size, rows=[(0, 0), (w.B - 1, w.Q - 1)])
    got = to_f64(o)
    for b, i in [(0, 0), (w.B - 1, w.Q - 1)]:
        assert np.abs(got[b, i] - ref[b, i]).max() <= BF16_ABS


def test_noalloc_refuses_a_request_larger_than_its_scratch():
    # Dims over a wide grid: any whose split-KV scratch would exceed the fixed
    # array are refused on the host before anything is enqueued (the buffers
    # passed are far too small for those dims, which is safe only because
    # nothing is launched). The plans keep the number of key ranges near one
    # wave of clusters, so the scratch they need may stay below the array for
    # every dims of the grid; the largest need found is then checked to fit.
    import ctypes
    small = WL.CONFIGS["c2"].with_(B=1, prefix=64, V=4096)
    _, args, _ = _inputs(small)
    lib = DB.load()
    out = torch.empty((1, 1, 1, 512), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros((64,), dtype=torch.int32, device="cuda")
    largest, refused = 0, 0
    for B in (1, 2, 8, 64):
        for Q in (1, 17, 65, 128):
            for H in (16, 64, 128):
                for L in (1 << 12, 1 << 17, 1 << 22):
                    dims = DB.attn_dims(B, Q, H, 512, 64, 64, (L + Q + 63) // 64,
                                        B * (L + Q + 64), DB.DDT_BF16, 0.07, L + Q)
                    need = DB.ddt_verify_attn_workspace_size(dims)
                    largest = max(largest, need)
                    if need > (32 << 20):
                        rc = lib.ddt_verify_attn_noalloc(
                            ctypes.byref(dims), args[0].data_ptr(), args[1].data_ptr(),
                            args[2].data_ptr(), args[3].data_ptr(), args[4].data_ptr(),
                            args[5].data_ptr(), out.data_ptr(), None, st.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
                        assert rc == -4  # DDT_EWORKSPACE
                        refused += 1
    torch.cuda.synchronize()
    assert refused > 0 or 0 < largest <= (32 << 20)
