"""GPU rotary embedding and cache append at tree positions (ddt_rope_append
through the C ABI) against the oracle: small ragged cases on both element
types and both the vector and the element-by-element paths, far positions,
the K2.6 workload shapes, and the capacity / range errors.

Tolerance, from the arithmetic the header documents: the device forms each
angle in double, reduces it modulo 2*pi and takes a float sine and cosine
(error about 2e-7), then turns the pair in fp32 (about 2.4e-7 relative to
|x_i| + |x_{i+R/2}|) and rounds once to the element type. So every rotated
value lies within 1e-6 * (|x_i| + |x_{i+R/2}|) of the exact rotation, plus
one unit in the last place of the element type for that final rounding.
Latent parts and rows the call must not touch are compared bit for bit."""
import numpy as np
import pytest
import torch

from oracle import ddt_oracle as O
from tree_speculative_decoding_ddt_gb300 import _binding as DB
from tree_speculative_decoding_ddt_gb300 import workloads as WL
from gpu_util import latent_tensor, t

pytestmark = pytest.mark.gpu

THETA = 10000.0


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Unit in the last place of |x| in the element type (normal range)."""
    mant = 7 if dtype == "bf16" else 23
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return np.exp2(e - mant)


def partner_mag(x: np.ndarray) -> np.ndarray:
    """|x_i| + |x_{i+R/2}| at every position of the last axis."""
    h = x.shape[-1] // 2
    m = np.abs(x[..., :h]) + np.abs(x[..., h:])
    return np.concatenate([m, m], axis=-1)


def assert_rotated(got: np.ndarray, exact: np.ndarray, src: np.ndarray, dtype: str, what: str):
    err = np.abs(got.astype(np.float64) - exact)
    bound = 1e-6 * partner_mag(src) + ulp(exact, dtype)
    bad = err > bound
    assert not bad.any(), (what, int(bad.sum()), float((err - bound).max()))


def to_np(x: torch.Tensor) -> np.ndarray:
    return x.float().cpu().numpy().astype(np.float64)


def gen(dtype: str, shape, g) -> np.ndarray:
    x = g.standard_normal(shape).astype(np.float32)
    return WL.round_bf16(x) if dtype == "bf16" else x


def run(dtype, prefix, table, depths, rows, H, C, R, page_size, seed=0, in_place=False,
        theta=THETA, offset=0):
    """One call on seeded inputs; returns device results and oracle results.
    ``offset`` shifts every device buffer by that many elements (breaking the
    16-byte alignment when nonzero)."""
    g = np.random.default_rng(seed)
    prefix = np.asarray(prefix, np.int32)
    table = np.asarray(table, np.int32)
    depths = np.asarray(depths, np.int32)
    B, Q = depths.shape
    q_pe = gen(dtype, (B, Q, H, R), g)
    kv_new = gen(dtype, (B, Q, C + R), g)
    kv = gen(dtype, (rows, C + R), g)

    def dev(x):
        if not offset:
            return latent_tensor(x, dtype)
        flat = np.concatenate([np.zeros(offset, np.float32), x.reshape(-1)])
        return latent_tensor(flat, dtype)[offset:].view(x.shape)

    q_d, kvn_d, kv_d = dev(q_pe), dev(kv_new), dev(kv)
    sentinel = np.full(q_pe.shape, 7.0, np.float32)
    q_out = q_d if in_place else dev(sentinel)
    st = torch.zeros(B, dtype=torch.int32, device="cuda")
    DB.ddt_rope_append(q_d, kvn_d, kv_d, t(table), t(prefix), t(depths), page_size, theta,
                       q_out=q_out, status=st)
    torch.cuda.synchronize()
    oq, okv, ost = O.rope_append(q_pe, kv_new, kv, table, prefix, depths, page_size, theta)
    # where each good sequence's slots live, to pair appended rows with sources
    dst, src = [], []
    for b in range(B):
        if ost[b] == 0:
            dst.append(O.slot_rows(table[b], page_size, np.arange(prefix[b], prefix[b] + Q)))
            src.append(kv_new[b])
    return dict(q_pe=q_pe, kv_new=kv_new, kv=kv, q_out=q_out, kv_d=kv_d, st=st.cpu().numpy(),
                oq=oq, okv=okv, ost=ost, C=C, R=R, dtype=dtype,
                dst=np.concatenate(dst) if dst else np.zeros(0, np.int64),
                src=np.concatenate(src) if src else np.zeros((0, C + R)))


def check(r, sentinel_ok=True):
    dtype, C = r["dtype"], r["C"]
    np.testing.assert_array_equal(r["st"], r["ost"])
    good = r["ost"] == 0
    got_q = to_np(r["q_out"])
    if good.any():
        assert_rotated(got_q[good], r["oq"][good], r["q_pe"][good], dtype, "q_pe")
    if (~good).any() and sentinel_ok:
        assert (got_q[~good] == 7.0).all()
    kv_got = to_np(r["kv_d"])
    kv0 = np.asarray(r["kv"], np.float64)
    untouched = np.ones(kv0.shape[0], bool)
    untouched[r["dst"]] = False
    # rows the call must leave alone: bit for bit
    np.testing.assert_array_equal(kv_got[untouched], kv0[untouched])
    np.testing.assert_array_equal(r["okv"][untouched], kv0[untouched])
    if len(r["dst"]):
        d = r["dst"]
        np.testing.assert_array_equal(kv_got[d, :C], r["okv"][d, :C])
        np.testing.assert_array_equal(kv_got[d, :C], r["src"][:, :C])
        assert_rotated(kv_got[d, C:], r["okv"][d, C:], r["src"][:, C:], dtype, "cache rope part")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("in_place", [False, True])
def test_small_ragged_cases(dtype, in_place):
    # three sequences over shuffled pages of 4 slots, ragged prefixes, Q = 9
    # with padding slots (depth -1); vector path (C, R/2 multiples of 8)
    g = np.random.default_rng(5)
    Q, ps = 9, 4
    prefix = [0, 5, 13]
    pages = g.permutation(24).astype(np.int32)
    table = pages.reshape(3, 8)
    depths = g.integers(-1, 5, (3, Q)).astype(np.int32)
    depths[:, 0] = 0
    r = run(dtype, prefix, table, depths, rows=24 * ps, H=3, C=40 if dtype == "bf16" else 36,
            R=16, page_size=ps, seed=1, in_place=in_place)
    check(r, sentinel_ok=not in_place)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("C,R,offset", [(5, 6, 0), (40, 16, 1), (0, 2, 0)])
def test_element_path(dtype, C, R, offset):
    # odd widths, a misaligned base, and a rope-only row (C = 0)
    g = np.random.default_rng(7)
    depths = g.integers(-1, 3, (2, 5)).astype(np.int32)
    r = run(dtype, [3, 0], [[1, 0, 2], [4, 5, 3]], depths, rows=18, H=2, C=C, R=R, page_size=3,
            seed=2, offset=offset)
    check(r)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_far_positions(dtype):
    # positions past 131072 with a larger base: the reduction modulo 2*pi
    # keeps the float sine and cosine accurate
    ps = 64
    prefix = [131000, 70001]
    table = np.stack([np.arange(2100, dtype=np.int32), np.arange(2100, 4200, dtype=np.int32)])
    depths = np.array([[0, 1, 2, 3, 4, 5, 6, 7, 8], [0, 1, 1, 2, 2, 3, -1, -1, -1]], np.int32)
    r = run(dtype, prefix, table, depths, rows=4200 * ps, H=2, C=8, R=64, page_size=ps, seed=3,
            theta=50000.0)
    check(r)


@pytest.mark.parametrize("cfg", ["c2", "c3", "c4"])
def test_workload_shapes(cfg):
    # the K2.6 shapes (H 64, C 512, R 64, bf16) at full batch, prefix lengths
    # and page layout; every q row and every appended cache row is checked
    w = WL.CONFIGS[cfg]
    lens = WL.prefix_lengths(w)
    lay = WL.cache_layout(w, lens)
    g = np.random.default_rng([w.cid, 77])
    depths = g.integers(-1, w.D + 1, (w.B, w.Q)).astype(np.int32)
    depths[:, 0] = 0
    q_pe = gen("bf16", (w.B, w.Q, w.H, w.R), g)
    kv_new = gen("bf16", (w.B, w.Q, w.C + w.R), g)
    kv = torch.zeros((lay.total_rows, w.C + w.R), dtype=torch.bfloat16, device="cuda")
    q_d = latent_tensor(q_pe, "bf16")
    st = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    q_out, _ = DB.ddt_rope_append(q_d, latent_tensor(kv_new, "bf16"), kv, t(lay.block_table),
                                  t(lens.astype(np.int32)), t(depths), lay.page_size, THETA,
                                  status=st)
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    pos = lens.astype(np.int64)[:, None] + np.maximum(depths, 0)
    exact_q = O.rope_neox(q_pe, pos[:, :, None], THETA)
    assert_rotated(to_np(q_out), exact_q, q_pe, "bf16", "q_pe")
    rows = np.stack([O.slot_rows(lay.block_table[b], lay.page_size,
                                 np.arange(lens[b], lens[b] + w.Q)) for b in range(w.B)])
    got = to_np(kv[torch.from_numpy(rows.reshape(-1)).cuda()]).reshape(w.B, w.Q, -1)
    np.testing.assert_array_equal(got[..., : w.C], kv_new[..., : w.C])
    exact_k = O.rope_neox(kv_new[..., w.C:], pos, THETA)
    assert_rotated(got[..., w.C:], exact_k, kv_new[..., w.C:], "bf16", "cache rope part")
    # nothing else was written
    assert int((kv != 0).any(dim=1).sum()) <= w.B * w.Q


def test_bad_sequences_are_left_untouched():
    # sequence 0 fine, 1 past its pages, 2 with a negative length, 3 on a
    # page outside the cache
    depths = np.zeros((4, 3), np.int32)
    table = [[0, 1, 2], [3, 4, 5], [6, 0, 1], [6, 99, 5]]
    r = run("bf16", [1, 4, -1, 2], table, depths, rows=14, H=2, C=8, R=8, page_size=2, seed=4)
    assert r["st"].tolist() == [0, 16, 16, 8]
    check(r)


def test_host_rejects_bad_arguments():
    g = np.random.default_rng(0)
    q = latent_tensor(gen("bf16", (1, 2, 1, 8), g), "bf16")
    kvn = latent_tensor(gen("bf16", (1, 2, 16), g), "bf16")
    kv = latent_tensor(gen("bf16", (8, 16), g), "bf16")
    bt, pl, dp = t(np.array([[0, 1]], np.int32)), t(np.array([0], np.int32)), \
        t(np.zeros((1, 2), np.int32))
    for theta in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(DB.DdtError):
            DB.ddt_rope_append(q, kvn, kv, bt, pl, dp, 4, theta)
    q7 = latent_tensor(gen("bf16", (1, 2, 1, 7), g), "bf16")
    kvn7 = latent_tensor(gen("bf16", (1, 2, 15), g), "bf16")
    kv7 = latent_tensor(gen("bf16", (8, 15), g), "bf16")
    with pytest.raises(DB.DdtError):  # odd R
        DB.ddt_rope_append(q7, kvn7, kv7, bt, pl, dp, 4)
