"""GPU parity: logsumexp and fused softmax cross-entropy (loss, gradient,
mean loss)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_abs, check_bound, check_rel, gpu, host, softmax_bwd_bound
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu

COLS = [1, 3, 4, 7, 32, 64, 129, 256, 1000, 1024, 1028, 1536, 3001, 4096, 8192, 16384, 16385, 50304, 50305,
        131072, 140000]


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("misalign", [False, True])
def test_lse_ce_shapes(ro, cols, misalign):
    rows = 6 if cols > 4096 else 33
    c = inputs.cross_entropy(cols, rows=rows, cols=cols, outlier_frac=2e-3)
    x, t = c["logits"], c["targets"]
    lse = host(ro.rowops_logsumexp(gpu(x, misalign)))
    check_rel(lse, oracle.logsumexp_rows(x), f"lse cols={cols}")
    g, rl, ml = ro.rowops_softmax_ce(gpu(x, misalign), gpu(t), grad_scale=c["grad_scale"])
    gr, rlr, mlr = oracle.softmax_cross_entropy(x, t, c["grad_scale"])
    check_abs(host(g), gr, 2e-6 * c["grad_scale"], f"ce grad cols={cols}")
    check_rel(host(rl), rlr, f"ce row loss cols={cols}")
    check_rel(host(ml), [mlr], f"ce mean loss cols={cols}")


def test_ce_scaled_workload(ro):
    c = inputs.cross_entropy(0, rows=96, cols=50304)
    x, t = c["logits"], c["targets"]
    g, rl, ml = ro.rowops_softmax_ce(gpu(x), gpu(t), grad_scale=c["grad_scale"])
    gr, rlr, mlr = oracle.softmax_cross_entropy(x, t, c["grad_scale"])
    check_abs(host(g), gr, 2e-6 * c["grad_scale"], "ce grad 96x50304")
    check_rel(host(rl), rlr, "ce row loss")
    check_rel(host(ml), [mlr], "ce mean loss")
    check_rel(host(ro.rowops_logsumexp(gpu(x))), oracle.logsumexp_rows(x), "lse 96x50304")


def test_ce_out_of_range_targets(ro):
    c = inputs.cross_entropy(1, rows=4, cols=300)
    x = c["logits"]
    t = np.array([5, 300, -1, 299], np.int32)
    g, rl, ml = ro.rowops_softmax_ce(gpu(x), gpu(t), grad_scale=0.5)
    gr, rlr, mlr = oracle.softmax_cross_entropy(x, t, 0.5)
    rl = host(rl)
    assert not np.isnan(rl[0]) and np.isnan(rl[1]) and np.isnan(rl[2]) and not np.isnan(rl[3])
    assert np.isnan(host(ml)[0]) and np.isnan(mlr)
    check_abs(host(g), gr, 1e-6, "grad without one-hot term")


def test_lse_special_rows(ro):
    x = np.array([[-np.inf] * 8, [np.inf, 0, 0, 0, 0, 0, 0, 0], [1000] * 8, [-1000] * 8], np.float32)
    got = host(ro.rowops_logsumexp(gpu(x)))
    ref = oracle.logsumexp_rows(x)
    assert got[0] == -np.inf and got[1] == np.inf
    check_rel(got[2:], ref[2:], "lse +-1000")
    x = torch.empty((5, 0), device="cuda")
    assert (host(ro.rowops_logsumexp(x)) == -np.inf).all()


def test_ce_deterministic(ro):
    c = inputs.cross_entropy(2, rows=64, cols=50304)
    x, t = gpu(c["logits"]), gpu(c["targets"])
    a = ro.rowops_softmax_ce(x, t)
    b = ro.rowops_softmax_ce(x, t)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.parametrize("cols", [1028, 4096, 50304, 58000])
def test_long_rows_many_rows_per_cta(ro, cols):
    # more rows than SMs, so every persistent CTA walks several rows through its ring
    c = inputs.cross_entropy(cols + 1, rows=400, cols=cols, outlier_frac=1e-3)
    x, t = c["logits"], c["targets"]
    xg = gpu(x)
    check_rel(host(ro.rowops_logsumexp(xg)), oracle.logsumexp_rows(x), f"lse 400x{cols}")
    g, rl, ml = ro.rowops_softmax_ce(xg, gpu(t), grad_scale=c["grad_scale"])
    idx = np.arange(0, 400, 37)
    gr, rlr, mlr = oracle.softmax_cross_entropy(x, t, c["grad_scale"])
    check_abs(host(g)[idx], gr[idx], 2e-6 * c["grad_scale"], "ce grad")
    check_rel(host(rl), rlr, "ce row loss")
    y = host(ro.rowops_softmax_fwd(xg))
    check_abs(y[idx], oracle.softmax_rows(x[idx]), 2e-6, "softmax long rows")
    assert ro.library().rowops_pipeline_timeouts() == 0


def _exact_mean(rl):
    import math
    rl = np.asarray(rl, np.float64)
    return math.fsum(rl.tolist()) / rl.size


@pytest.mark.parametrize("rows", [1, 1000, 8192, 20001])
def test_ce_mean_of_row_losses(ro, rows):
    # the mean kernel alone: its result against the exactly rounded mean of the
    # row losses the GPU wrote (independent of the row losses' own fp32 error)
    c = inputs.cross_entropy(rows, rows=rows, cols=64)
    _, rl, ml = ro.rowops_softmax_ce(gpu(c["logits"]), gpu(c["targets"]))
    rl = host(rl)
    ref = _exact_mean(rl)
    assert abs(float(host(ml)[0]) - ref) <= 1e-12 * np.abs(rl.astype(np.float64)).mean()


def test_ce_mean_non_finite_and_fp32_overflow(ro):
    # an infinite row loss: the mean is +inf, as a double sum gives
    x = np.zeros((3, 8), np.float32)
    x[1, 2] = -np.inf
    t = np.array([0, 2, 5], np.int32)
    _, rl, ml = ro.rowops_softmax_ce(gpu(x), gpu(t))
    assert np.isinf(host(rl)[1]) and host(ml)[0] == np.inf
    assert oracle.softmax_cross_entropy(x, t, 1.0)[2] == np.inf
    # finite losses of 1e37 whose sum overflows fp32: the mean stays finite
    x = np.zeros((8192, 8), np.float32)
    x[:, 3] = -1e37
    t = np.full(8192, 3, np.int32)
    _, rl, ml = ro.rowops_softmax_ce(gpu(x), gpu(t))
    rl = host(rl)
    got = float(host(ml)[0])
    assert np.isfinite(got) and abs(got - _exact_mean(rl)) <= 1e-12 * abs(_exact_mean(rl))
    assert abs(got - oracle.softmax_cross_entropy(x, t, 1.0)[2]) <= 1e-6 * 1e37


def _at_offset(a: np.ndarray, off: int) -> torch.Tensor:
    """Device copy of `a` whose data starts `off` floats past a 256-byte boundary."""
    a = np.ascontiguousarray(a, np.float32)
    flat = torch.zeros(a.size + 8, dtype=torch.float32, device="cuda")
    view = flat[off:off + a.size].view(a.shape)
    view.copy_(torch.from_numpy(a).cuda())
    return view


@pytest.mark.parametrize("cols", [1025, 3001, 50257, 50258, 50259, 60001, 100003, 131072, 152064])
@pytest.mark.parametrize("off", [0, 1, 3])
def test_long_rows_not_on_16_byte_boundaries(ro, cols, off):
    # rows of cols % 4 != 0 (and buffers offset by `off` floats) start at every
    # position modulo 16 bytes: the long-row kernels split each row into a head,
    # a bulk-copied body and a tail; 300 rows make every CTA walk several rows
    rows = 300
    c = inputs.cross_entropy(cols + off, rows=rows, cols=cols, outlier_frac=1e-3)
    x, t = c["logits"], c["targets"]
    # targets in the first and last four columns hit the head and tail floats
    t[:8] = [0, 1, 2, 3, cols - 1, cols - 2, cols - 3, cols - 4]
    xg = _at_offset(x, off)
    idx = np.r_[0:12, 151:156, rows - 4:rows]
    check_rel(host(ro.rowops_logsumexp(xg)), oracle.logsumexp_rows(x), f"lse {rows}x{cols}+{off}")
    g = _at_offset(np.zeros_like(x), off)
    rl = torch.empty(rows, device="cuda")
    ml = torch.empty(1, dtype=torch.float64, device="cuda")
    ro.rowops_softmax_ce(xg, gpu(t), g, rl, ml, grad_scale=c["grad_scale"])
    gr, rlr, mlr = oracle.softmax_cross_entropy(x, t, c["grad_scale"])
    check_abs(host(g)[idx], gr[idx], 2e-6 * c["grad_scale"], "ce grad")
    check_rel(host(rl), rlr, "ce row loss")
    check_rel(host(ml), [mlr], "ce mean loss")
    ref = oracle.softmax_rows(x[idx])
    y = _at_offset(np.zeros_like(x), off)
    ro.rowops_softmax_fwd(xg, y)
    check_abs(host(y)[idx], ref, 2e-6, "softmax")
    ro.rowops_softmax_fwd(xg, xg)  # in place
    check_abs(host(xg)[idx], ref, 2e-6, "softmax in place")
    assert ro.library().rowops_pipeline_timeouts() == 0


@pytest.mark.parametrize("cols,off", [(1000003, 0), (1000003, 1), (2 ** 20, 0)])
def test_very_long_rows(ro, cols, off):
    # rows of a million floats: dozens of chunks per pass in the two-pass
    # kernels (each CTA of a cluster taking half a row), the streaming
    # logsumexp and the two-input softmax backward
    rows = 3
    c = inputs.cross_entropy(cols + off, rows=rows, cols=cols, outlier_frac=1e-4)
    x, t = c["logits"], c["targets"]
    t[0] = cols - 1
    xg = _at_offset(x, off)
    check_rel(host(ro.rowops_logsumexp(xg)), oracle.logsumexp_rows(x), f"lse {rows}x{cols}+{off}")
    g = _at_offset(np.zeros_like(x), off)
    rl = torch.empty(rows, device="cuda")
    ml = torch.empty(1, dtype=torch.float64, device="cuda")
    ro.rowops_softmax_ce(xg, gpu(t), g, rl, ml, grad_scale=c["grad_scale"])
    gr, rlr, mlr = oracle.softmax_cross_entropy(x, t, c["grad_scale"])
    check_abs(host(g), gr, 2e-6 * c["grad_scale"], "ce grad")
    check_rel(host(rl), rlr, "ce row loss")
    ref = oracle.softmax_rows(x)
    y = _at_offset(np.zeros_like(x), off)
    ro.rowops_softmax_fwd(xg, y)
    check_abs(host(y), ref, 2e-6, "softmax")
    y32 = ref.astype(np.float32)
    dy = np.random.default_rng(cols).normal(0, 1, x.shape).astype(np.float32)
    dx = _at_offset(np.zeros_like(x), off)
    ro.rowops_softmax_bwd(_at_offset(y32, off), _at_offset(dy, off), dx)
    check_bound(host(dx), oracle.softmax_rows_backward(y32, dy), softmax_bwd_bound(y32, dy), "softmax bwd")
    assert ro.library().rowops_pipeline_timeouts() == 0


@pytest.mark.parametrize("cols", [50304, 60001, 152064])
@pytest.mark.parametrize("offs", [(0, 1), (1, 0), (2, 3)])
def test_long_rows_output_on_another_phase(ro, cols, offs):
    # logits and gradient (or probabilities) on different 16-byte phases: the
    # bulk-copy kernels write the output rows with scalar stores
    rows = 200
    c = inputs.cross_entropy(cols + 3 * offs[0] + offs[1], rows=rows, cols=cols, outlier_frac=1e-3)
    x, t = c["logits"], c["targets"]
    xg = _at_offset(x, offs[0])
    g = _at_offset(np.zeros_like(x), offs[1])
    rl = torch.empty(rows, device="cuda")
    ml = torch.empty(1, dtype=torch.float64, device="cuda")
    ro.rowops_softmax_ce(xg, gpu(t), g, rl, ml, grad_scale=c["grad_scale"])
    gr, rlr, mlr = oracle.softmax_cross_entropy(x, t, c["grad_scale"])
    check_abs(host(g), gr, 2e-6 * c["grad_scale"], "ce grad")
    check_rel(host(rl), rlr, "ce row loss")
    check_rel(host(ml), [mlr], "ce mean loss")
    y = _at_offset(np.zeros_like(x), offs[1])
    ro.rowops_softmax_fwd(xg, y)
    check_abs(host(y), oracle.softmax_rows(x), 2e-6, "softmax")
    assert ro.library().rowops_pipeline_timeouts() == 0
