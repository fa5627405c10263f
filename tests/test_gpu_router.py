"""GPU parity: hard-masked softmax and the top-k kept mask (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_exact_zero, check_probs, gpu, host
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_router_workload_scaled(ro):
    r = inputs.router(0, rows=8192)
    x, mask = r["x"], r["mask"]
    p = host(ro.rowops_masked_softmax(gpu(x), gpu(mask)))
    pr = oracle.masked_softmax(x, mask)
    check_probs(p, pr, "masked softmax")
    check_exact_zero(p, mask == 0, "blocked entries")
    assert (p[r["blocked_rows"]] == 0).all()
    p32 = pr.astype(np.float32)
    kept = host(ro.rowops_topk_kept(gpu(p32), 2))
    assert np.array_equal(kept, oracle.topk_kept(p32, 2).astype(np.float32))
    kept_x = host(ro.rowops_topk_kept(gpu(x), 2))
    assert np.array_equal(kept_x, oracle.topk_kept(x, 2).astype(np.float32))


MASK_COLS = [1, 2, 3, 4, 7, 8, 16, 33, 64, 128, 255, 256, 1024, 1028, 2048, 5000, 16384, 16385]


@pytest.mark.parametrize("cols", MASK_COLS)
@pytest.mark.parametrize("misalign", [False, True])
def test_masked_shapes(ro, cols, misalign):
    r = inputs.router(cols, rows=50, cols=cols, p_allow=0.6, blocked_row_frac=0.1)
    x, mask = r["x"], r["mask"]
    mask = mask * np.uint8(1 + (np.arange(mask.size).reshape(mask.shape) % 7))  # any nonzero byte allows
    p = host(ro.rowops_masked_softmax(gpu(x, misalign), gpu(mask, misalign)))
    check_probs(p, oracle.masked_softmax(x, mask), f"masked cols={cols}")
    check_exact_zero(p, mask == 0, "blocked")


def test_masked_in_place(ro):
    r = inputs.router(2, rows=100)
    t = gpu(r["x"])
    ro.rowops_masked_softmax(t, gpu(r["mask"]), t)
    check_probs(host(t), oracle.masked_softmax(r["x"], r["mask"]), "in place")


KEPT_CASES = [(c, k) for c in (1, 2, 3, 4, 5, 8, 16, 31, 64, 100, 256, 1000, 1024, 1100, 4096)
              for k in sorted({1, min(2, c), min(3, c), min(8, c), min(9, c), max(1, c // 2),
                               max(1, c - 8), max(1, c - 1), c})]


@pytest.mark.parametrize("cols,k", KEPT_CASES)
def test_kept_exact(ro, cols, k):
    rng = np.random.default_rng(cols * 1000 + k)
    rows = 40 if cols <= 1024 else 6
    x = (rng.integers(-8, 9, (rows, cols)) / 4.0).astype(np.float32)  # many ties
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, 0.0, -0.0).astype(np.float32)
    for misalign in (False, True):
        kept = host(ro.rowops_topk_kept(gpu(x, misalign), k))
        ref = oracle.topk_kept(x, k).astype(np.float32)
        assert np.array_equal(kept, ref), (cols, k, misalign, np.argwhere(kept != ref)[:5])


@pytest.mark.parametrize("cols", [3, 8, 64, 300, 1024, 2000])
def test_kept_with_nan_and_infinities(ro, cols):
    rng = np.random.default_rng(cols)
    x = (rng.integers(-4, 5, (24, cols)) / 2.0).astype(np.float32)
    x[rng.random(x.shape) < 0.05] = np.nan
    x[rng.random(x.shape) < 0.03] = np.inf
    x[rng.random(x.shape) < 0.03] = -np.inf
    x[5] = np.nan
    for k in sorted({1, 2, min(3, cols), cols}):
        kept = host(ro.rowops_topk_kept(gpu(x), k))
        assert np.array_equal(kept, oracle.topk_kept(x, k).astype(np.float32)), (cols, k)


def _gpu_at(a: np.ndarray, offset_bytes: int) -> torch.Tensor:
    """Device copy of `a` whose data pointer is `offset_bytes` past a 256-byte boundary."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    flat = torch.empty(t.numel() + 64, dtype=t.dtype, device="cuda")
    off = offset_bytes // t.element_size()
    view = flat[off:off + t.numel()].view(t.shape)
    view.copy_(t.to("cuda"))
    assert view.data_ptr() % 256 == offset_bytes
    return view


@pytest.mark.parametrize("cols", [34, 36, 40, 62, 64, 66, 96, 100, 128, 130])
def test_kept_top2_every_alignment(ro, cols):
    # Rows on 16-byte boundaries take the float4 lane groups, the others (8- or
    # 4-byte boundaries, odd lengths) the scalar ones.  Ties, -0/+0,
    # infinities and a NaN row, at every alignment of input and output.
    rng = np.random.default_rng(cols)
    rows = 203
    x = (rng.integers(-6, 7, (rows, cols)) / 4.0).astype(np.float32)
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, 0.0, -0.0).astype(np.float32)
    x[rng.random(x.shape) < 0.02] = np.inf
    x[rng.random(x.shape) < 0.02] = -np.inf
    x[7] = -np.inf
    x[8] = 0.0
    x[9, ::3] = np.nan
    x[150] = -0.0
    for k in (1, 2):
        ref = oracle.topk_kept(x, k).astype(np.float32)
        for xo, ko in ((0, 0), (8, 0), (0, 8), (8, 8), (4, 0), (12, 4)):
            out = _gpu_at(np.zeros_like(x), ko)
            ro.rowops_topk_kept(_gpu_at(x, xo), k, out)
            assert np.array_equal(host(out), ref), (cols, k, xo, ko, np.argwhere(host(out) != ref)[:5])


def test_kept_denormals(ro):
    tiny = np.float32(1e-45)
    x = np.array([[tiny, 0.0, -tiny, -0.0, 2 * tiny, tiny]], np.float32)
    for k in range(1, 7):
        kept = host(ro.rowops_topk_kept(gpu(x), k))
        assert np.array_equal(kept, oracle.topk_kept(x, k).astype(np.float32)), k


def test_router_empty(ro):
    x = torch.empty((0, 64), device="cuda")
    m = torch.empty((0, 64), dtype=torch.uint8, device="cuda")
    assert ro.rowops_masked_softmax(x, m).shape == (0, 64)
    assert ro.rowops_topk_kept(x, 2).shape == (0, 64)


def test_kept_infinities_without_nan_rows(ro):
    rng = np.random.default_rng(77)
    for cols in (2, 3, 5, 64, 200, 1500):
        x = (rng.integers(-2, 3, (64, cols)) / 2.0).astype(np.float32)
        x[rng.random(x.shape) < 0.2] = np.inf
        x[rng.random(x.shape) < 0.2] = -np.inf
        x[3] = -np.inf
        x[4] = np.inf
        for k in sorted({1, min(2, cols), min(3, cols), max(1, cols - 1), cols}):
            kept = host(ro.rowops_topk_kept(gpu(x), k))
            assert np.array_equal(kept, oracle.topk_kept(x, k).astype(np.float32)), (cols, k)


# ------------------------------------------------------------ fused router

def test_router_fused_full_workload(ro):
    r = inputs.router(0)
    x, mask = r["x"], r["mask"]
    p, kept = ro.rowops_router_masked_topk(gpu(x), gpu(mask), r["k"])
    pr, keptr = oracle.router_masked_topk(x, mask, r["k"])
    check_probs(host(p), pr, "router p")
    check_exact_zero(host(p), mask == 0, "router blocked")
    assert np.array_equal(host(kept), keptr.astype(np.float32))
    # bit-identical to the two separate ops
    p2 = ro.rowops_masked_softmax(gpu(x), gpu(mask))
    k2 = ro.rowops_topk_kept(p2, r["k"])
    assert torch.equal(p, p2) and torch.equal(kept, k2)


@pytest.mark.parametrize("cols", [1, 3, 8, 33, 64, 256, 1024, 1100])
@pytest.mark.parametrize("misalign", [False, True])
def test_router_shapes(ro, cols, misalign):
    r = inputs.router(cols, rows=64, cols=cols, p_allow=0.7, blocked_row_frac=0.05)
    x, mask = r["x"], r["mask"]
    for k in sorted({1, min(2, cols), min(5, cols), cols}):
        p, kept = ro.rowops_router_masked_topk(gpu(x, misalign), gpu(mask, misalign), k)
        pr, keptr = oracle.router_masked_topk(x, mask, k)
        check_probs(host(p), pr, f"router p cols={cols}")
        assert np.array_equal(host(kept), keptr.astype(np.float32)), (cols, k, misalign)


# --------------------------------------------------------------- top_k_rows

def _same_bits(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32)) \
        or (np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(np.where(np.isnan(a), 0, a).view(np.uint32),
                                                                         np.where(np.isnan(b), 0, b).view(np.uint32)))


@pytest.mark.parametrize("cols", [1, 2, 5, 16, 64, 100, 256, 1024, 1500])
@pytest.mark.parametrize("misalign", [False, True])
def test_top_k_rows_exact(ro, cols, misalign):
    rng = np.random.default_rng(cols + 7)
    x = (rng.integers(-6, 7, (37, cols)) / 4.0).astype(np.float32)
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, 0.0, -0.0).astype(np.float32)
    x[rng.random(x.shape) < 0.05] = np.nan
    x[rng.random(x.shape) < 0.03] = np.inf
    x[rng.random(x.shape) < 0.03] = -np.inf
    for k in sorted({1, min(2, cols), min(7, cols), cols}):
        for largest in (True, False):
            v, i = ro.rowops_top_k_rows(gpu(x, misalign), k, largest)
            vr, ir = oracle.top_k_rows(x, k, largest)
            assert np.array_equal(host(i), ir.astype(np.float32)), (cols, k, largest)
            assert _same_bits(host(v), vr.astype(np.float32)), (cols, k, largest)


@pytest.mark.parametrize("cols", [1, 2, 3, 8, 33, 64, 100, 256, 1000])
def test_top_k_rows_top2_ties_and_signed_zeros(ro, cols):
    # k <= 2: warps whose rows hold no NaN or infinity run the tournament on
    # the (negated, for smallest) values; the others on the rank keys.  Many
    # ties and both zeros; then the same rows with a few NaN and infinite rows
    # mixed in, so warps of both kinds meet.
    rng = np.random.default_rng(cols + 101)
    x = (rng.integers(-3, 4, (203, cols)) / 2.0).astype(np.float32)
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, 0.0, -0.0).astype(np.float32)
    x[11] = -0.0
    x[12] = 0.0
    y = x.copy()
    y[40, 0] = np.nan
    y[90, -1] = np.inf
    y[150, cols // 2] = -np.inf
    for data in (x, y):
        for k in sorted({1, min(2, cols)}):
            for largest in (True, False):
                for misalign in (False, True):
                    v, i = ro.rowops_top_k_rows(gpu(data, misalign), k, largest)
                    vr, ir = oracle.top_k_rows(data, k, largest)
                    assert np.array_equal(host(i), ir.astype(np.float32)), (cols, k, largest, misalign)
                    assert _same_bits(host(v), vr.astype(np.float32)), (cols, k, largest, misalign)


def test_top_k_rows_router_logits(ro):
    r = inputs.router(1, rows=20000)
    v, i = ro.rowops_top_k_rows(gpu(r["x"]), 2, True)
    vr, ir = oracle.top_k_rows(r["x"], 2, True)
    assert np.array_equal(host(i), ir.astype(np.float32)) and np.array_equal(host(v), vr.astype(np.float32))


@pytest.mark.parametrize("rows,cols", [(3, 50304), (300, 3001)])
@pytest.mark.parametrize("misalign", [False, True])
def test_top_k_rows_long_rows(ro, rows, cols, misalign):
    # rows of more than 1024 floats: the radix select (2 <= k <= 1024) and the
    # k-pass kernel beyond; values on a coarse grid force long runs of ties
    rng = np.random.default_rng(rows + cols)
    x = (rng.normal(0, 2, (rows, cols)) * 4).round().astype(np.float32) / 4
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, 0.0, -0.0).astype(np.float32)
    x[rng.random(x.shape) < 1e-3] = np.nan
    x[rng.random(x.shape) < 1e-3] = np.inf
    x[rng.random(x.shape) < 1e-3] = -np.inf
    xg = gpu(x, misalign)
    for k in [k for k in (2, 50, 300, 1024, 1025) if k <= cols]:
        for largest in (True, False):
            v, i = ro.rowops_top_k_rows(xg, k, largest)
            vr, ir = oracle.top_k_rows(x, k, largest)
            assert np.array_equal(host(i), ir.astype(np.float32)), (cols, k, largest)
            assert _same_bits(host(v), vr.astype(np.float32)), (cols, k, largest)


@pytest.mark.parametrize("rows,cols", [(37, 1025), (5, 50304), (300, 3001), (2, 131072), (700, 4096)])
@pytest.mark.parametrize("misalign", [False, True])
def test_top_k_rows_long_rows_top2(ro, rows, cols, misalign):
    # rows of more than 1024 floats with k <= 2: one pass on the values where a
    # row holds no NaN or infinity, the rank keys again from the L2 where it
    # does; ties and both zeros (values on a coarse grid), a few NaN and
    # infinite rows among finite ones
    rng = np.random.default_rng(rows * 7 + cols)
    x = (rng.normal(0, 2, (rows, cols)) * 2).round().astype(np.float32) / 2
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, 0.0, -0.0).astype(np.float32)
    y = x.copy()
    y[0, cols // 3] = np.nan
    y[-1, -1] = np.inf
    if rows > 2:
        y[1, 5] = -np.inf
        y[1, 6] = np.nan
    for data in (x, y):
        xg = gpu(data, misalign)
        for k in (1, 2):
            for largest in (True, False):
                v, i = ro.rowops_top_k_rows(xg, k, largest)
                vr, ir = oracle.top_k_rows(data, k, largest)
                assert np.array_equal(host(i), ir.astype(np.float32)), (rows, cols, k, largest, misalign)
                assert _same_bits(host(v), vr.astype(np.float32)), (rows, cols, k, largest, misalign)


@pytest.mark.parametrize("cols", [16, 64, 100, 128, 256, 512, 1000, 1024])
@pytest.mark.parametrize("k", [3, 4, 8, 16, 32])
def test_kept_candidates(ro, cols, k):
    # 3 <= k <= group width: the candidate path (distinct values), and its
    # fallback to rounds when many entries tie (values on a 1/8 grid)
    if k >= cols:
        pytest.skip("k < cols")
    rng = np.random.default_rng(cols * 7 + k)
    xs = [rng.normal(0, 2, (300, cols)).astype(np.float32),
          (rng.integers(-32, 33, (300, cols)) / 8.0).astype(np.float32)]
    for x in xs:
        for misalign in (False, True):
            kept = host(ro.rowops_topk_kept(gpu(x, misalign), k))
            ref = oracle.topk_kept(x, k).astype(np.float32)
            assert np.array_equal(kept, ref), (cols, k, misalign, np.argwhere(kept != ref)[:5])
    r = inputs.router(cols + k, rows=300, cols=cols, p_allow=0.8, blocked_row_frac=0.02)
    p, kept = ro.rowops_router_masked_topk(gpu(r["x"]), gpu(r["mask"]), k)
    pr, kr = oracle.router_masked_topk(r["x"], r["mask"], k)
    assert np.array_equal(host(kept), kr.astype(np.float32)), (cols, k)


@pytest.mark.parametrize("cols", [16, 64, 128, 256, 1000])
@pytest.mark.parametrize("k", [3, 8, 16, 32])
def test_top_k_rows_candidates(ro, cols, k):
    # 3 <= k <= group width: the candidate path (distinct values, and values
    # with NaN, infinities and many ties that send rows to the rounds)
    if k >= cols:
        pytest.skip("k < cols")
    rng = np.random.default_rng(cols * 11 + k)
    x1 = rng.normal(0, 2, (300, cols)).astype(np.float32)
    x2 = (rng.integers(-16, 17, (300, cols)) / 4.0).astype(np.float32)
    x2[rng.random(x2.shape) < 0.02] = np.nan
    x2[rng.random(x2.shape) < 0.02] = -np.inf
    for x in (x1, x2):
        for largest in (True, False):
            for misalign in (False, True):
                v, i = ro.rowops_top_k_rows(gpu(x, misalign), k, largest)
                vr, ir = oracle.top_k_rows(x, k, largest)
                assert np.array_equal(host(i), ir.astype(np.float32)), (cols, k, largest, misalign)
                assert _same_bits(host(v), vr.astype(np.float32)), (cols, k, largest, misalign)
