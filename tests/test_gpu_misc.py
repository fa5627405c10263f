"""GPU parity: float-mask masked softmax, the softmax relevance rule
(lrp_softmax_rows) and the first-max one-hot."""
import numpy as np
import pytest

import oracle
from parity_util import check_bound, check_exact_zero, check_probs, gpu, host
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu

COLS = [1, 3, 4, 16, 33, 64, 128, 256, 257, 1024, 1028, 2048, 3000, 8192, 16384, 16385]


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("misalign", [False, True])
def test_masked_softmax_float_mask(ro, cols, misalign):
    rng = np.random.default_rng(cols)
    x = (rng.integers(-32, 33, (40, cols)) / 8.0).astype(np.float32)
    mask = rng.choice(np.array([0.0, -0.0, 1.0, 0.25, -3.0, np.nan], np.float32), size=(40, cols))
    mask[5] = 0.0
    y = host(ro.rowops_masked_softmax_fmask(gpu(x, misalign), gpu(mask, misalign)))
    check_probs(y, oracle.masked_softmax_fmask(x, mask), f"fmask cols={cols}")
    check_exact_zero(y, mask == 0, "blocked")


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("misalign", [False, True])
def test_lrp_softmax_rows(ro, cols, misalign):
    rng = np.random.default_rng(cols + 1)
    x = rng.normal(0, 1, (40, cols)).astype(np.float32)
    y = oracle.softmax_rows(rng.normal(0, 2, (40, cols))).astype(np.float32)
    r = rng.normal(0, 1, (40, cols)).astype(np.float32)
    got = host(ro.rowops_lrp_softmax_rows(gpu(x, misalign), gpu(y, misalign), gpu(r, misalign)))
    ref = oracle.lrp_softmax_rows(x, y, r)
    ax, ay, ar = (np.abs(a.astype(np.float64)) for a in (x, y, r))
    bound = 1e-5 * ax * (ar + ay * ar.sum(axis=1, keepdims=True)) + 1e-9
    check_bound(got, ref, bound, f"lrp cols={cols}")


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("misalign", [False, True])
def test_argmax_onehot(ro, cols, misalign):
    rng = np.random.default_rng(cols + 2)
    x = (rng.integers(-3, 4, (60, cols)) / 2.0).astype(np.float32)
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, 0.0, -0.0).astype(np.float32)
    x[rng.random(x.shape) < 0.03] = np.nan
    x[rng.random(x.shape) < 0.03] = np.inf
    x[7] = np.nan
    x[8] = -np.inf
    got = host(ro.rowops_argmax_onehot(gpu(x, misalign)))
    assert np.array_equal(got, oracle.argmax_onehot(x).astype(np.float32))
    assert (got.sum(axis=1) == 1).all()


def test_argmax_onehot_router_logits(ro):
    r = inputs.router(3, rows=50000)
    got = host(ro.rowops_argmax_onehot(gpu(r["x"])))
    assert np.array_equal(got, oracle.argmax_onehot(r["x"]).astype(np.float32))
