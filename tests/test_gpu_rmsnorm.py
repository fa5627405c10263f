"""GPU parity: RMSNorm forward/backward and column sums."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_bound, check_rel, gpu, host
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu


def _rms_dx_bound(g, gamma, x, rms):
    gp = np.abs(np.asarray(g, np.float64) * gamma)
    xa = np.abs(np.asarray(x, np.float64))
    r = np.asarray(rms, np.float64).reshape(-1, 1)
    return 1e-5 * (gp + xa * (gp * xa).mean(axis=1, keepdims=True) / r ** 2) / r + 1e-9


def _run(ro, n, misalign=False):
    x, gamma, dy, eps = n["x"], n["gamma"], n["dy"], n["eps"]
    out, rms = ro.rowops_rmsnorm_fwd(gpu(x, misalign), gpu(gamma, misalign), eps=eps)
    o_r, rms_r = oracle.rms_norm_forward(x, gamma, eps)
    check_rel(host(out), o_r, "rms out")
    check_bound(host(rms), rms_r, 1e-5 * np.abs(rms_r), "row_rms")
    rms32 = rms_r.astype(np.float32)
    dx, terms = ro.rowops_rmsnorm_bwd(gpu(dy, misalign), gpu(gamma, misalign), gpu(x, misalign), gpu(rms32))
    dxr, tr = oracle.rms_norm_backward(dy, gamma, x, rms32)
    check_bound(host(dx), dxr, _rms_dx_bound(dy, gamma, x, rms32), "rms dx")
    check_bound(host(terms), tr, 1e-5 * np.abs(tr) + 1e-12, "gamma_terms")
    dg = ro.rowops_column_sums(terms)
    check_bound(host(dg), oracle.column_sums(tr), 1e-4 * np.abs(tr).sum(axis=0) + 1e-9, "dgamma")


def test_rmsnorm_4096x768(ro):
    _run(ro, inputs.layernorm(0))


@pytest.mark.parametrize("cols", [1, 3, 4, 33, 128, 256, 257, 768, 1024, 1028, 2048, 3000, 4096, 8192, 16384,
                                  16385])
@pytest.mark.parametrize("misalign", [False, True])
def test_rmsnorm_shapes(ro, cols, misalign):
    _run(ro, inputs.layernorm(cols, rows=41, cols=cols), misalign)


@pytest.mark.parametrize("rows,cols", [(1, 5), (7, 768), (8, 33), (1000, 96), (100000, 64), (3, 40000)])
def test_column_sums_shapes(ro, rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    m = rng.normal(0, 1, (rows, cols)).astype(np.float32)
    bound = 1e-4 * np.abs(m.astype(np.float64)).sum(axis=0) + 1e-9
    check_bound(host(ro.rowops_column_sums(gpu(m))), oracle.column_sums(m), bound, "column sums")
    prev = rng.normal(0, 1, cols).astype(np.float32)
    got = host(ro.rowops_column_sums(gpu(m), gpu(prev), beta=0.5))
    check_bound(got, oracle.column_sums(m, prev, 0.5), bound + 1e-6 * np.abs(prev), "column sums beta")
    nan_out = gpu(np.full(cols, np.nan, np.float32))
    assert not np.isnan(host(ro.rowops_column_sums(gpu(m), nan_out, beta=0.0))).any()


def test_column_sums_zero_rows_scales_by_beta(ro):
    out = gpu(np.arange(8, dtype=np.float32))
    ro.rowops_column_sums(torch.empty((0, 8), device="cuda"), out, beta=2.0)
    assert np.array_equal(host(out), 2 * np.arange(8, dtype=np.float32))


def test_column_sums_deterministic(ro):
    m = gpu(np.random.default_rng(5).normal(0, 1, (50000, 300)).astype(np.float32))
    a = host(ro.rowops_column_sums(m))
    b = host(ro.rowops_column_sums(m))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
