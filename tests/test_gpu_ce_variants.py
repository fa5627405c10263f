"""GPU parity: weighted-logits (soft-target) and fixed-teacher cross-entropy."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_abs, check_rel, gpu, host

pytestmark = pytest.mark.gpu

COLS = [1, 3, 4, 16, 64, 256, 1000, 1024, 1028, 8192, 50304]


def _inputs(rows, cols, seed):
    rng = np.random.default_rng(seed)
    x = (rng.normal(0, 2, (rows, cols))).astype(np.float32)
    x[rng.random(x.shape) < 1e-3] = 30.0
    w = rng.random((rows, cols)).astype(np.float32)
    w[rng.random(w.shape) < 0.5] = 0.0
    t = (rng.normal(0, 2, (rows, cols))).astype(np.float32)
    return x, w, t


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("misalign", [False, True])
def test_soft_ce(ro, cols, misalign):
    rows = 5 if cols > 4096 else 33
    x, w, _ = _inputs(rows, cols, cols)
    g, rl, ml = ro.rowops_soft_ce(gpu(x, misalign), gpu(w, misalign), grad_scale=1.0 / rows)
    gr, rlr, mlr = oracle.soft_ce(x, w, 1.0 / rows)
    wsum = np.abs(w.astype(np.float64)).sum(axis=1, keepdims=True)
    check_abs(host(g), gr, 2e-6 * (1.0 / rows) * np.maximum(1.0, wsum), f"soft ce grad cols={cols}")
    scale = np.maximum(1.0, np.abs(w.astype(np.float64)).sum(axis=1) * (np.abs(x).max(axis=1) + 10))
    check_abs(host(rl), rlr, 1e-5 * scale, f"soft ce loss cols={cols}")
    check_abs(host(ml), [mlr], 1e-5 * scale.max(), "soft ce mean")


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("misalign", [False, True])
def test_teacher_ce(ro, cols, misalign):
    rows = 5 if cols > 4096 else 33
    s, _, t = _inputs(rows, cols, cols + 1)
    sg, tg = gpu(s, misalign), gpu(t, misalign)
    g, rl, ml = ro.rowops_teacher_ce(sg, tg, grad_scale=1.0 / rows)
    gr, rlr, mlr = oracle.teacher_ce(s, t, 1.0 / rows)
    check_abs(host(g), gr, 4e-6 / rows, f"teacher grad cols={cols}")
    check_rel(host(rl), rlr, f"teacher loss cols={cols}")
    check_rel(host(ml), [mlr], "teacher mean")
    _, rl2, ml2 = ro.rowops_teacher_ce(sg, tg, with_grad=False)
    assert torch.equal(rl2, rl)


@pytest.mark.parametrize("rows,cols", [(1, 132), (151, 260), (33, 512), (4096, 768), (5000, 768), (300, 772),
                                       (153, 1020), (7000, 1024)])
def test_ce_variants_warp_rows(ro, rows, cols):
    # Rows of 129..1024 floats on 16-byte boundaries: a warp a row with the
    # second input staged in shared memory; one wave, or warps that walk
    # further rows (more than a CTA's warps per SM), ragged last CTAs.
    x, w, t = _inputs(rows, cols, rows + cols)
    g, rl, ml = ro.rowops_soft_ce(gpu(x), gpu(w), grad_scale=1.0 / rows)
    gr, rlr, mlr = oracle.soft_ce(x, w, 1.0 / rows)
    wsum = np.abs(w.astype(np.float64)).sum(axis=1, keepdims=True)
    check_abs(host(g), gr, 2e-6 * (1.0 / rows) * np.maximum(1.0, wsum), f"soft ce grad {rows}x{cols}")
    scale = np.maximum(1.0, np.abs(w.astype(np.float64)).sum(axis=1) * (np.abs(x).max(axis=1) + 10))
    check_abs(host(rl), rlr, 1e-5 * scale, f"soft ce loss {rows}x{cols}")
    g, rl, ml = ro.rowops_teacher_ce(gpu(x), gpu(t), grad_scale=1.0 / rows)
    gr, rlr, mlr = oracle.teacher_ce(x, t, 1.0 / rows)
    check_abs(host(g), gr, 4e-6 / rows, f"teacher grad {rows}x{cols}")
    check_rel(host(rl), rlr, f"teacher loss {rows}x{cols}")
    check_rel(host(ml), [mlr], "teacher mean")


def test_soft_ce_one_hot_matches_integer_targets(ro):
    rng = np.random.default_rng(9)
    x = rng.normal(0, 2, (64, 50304)).astype(np.float32)
    t = rng.integers(0, 50304, 64).astype(np.int32)
    w = np.zeros_like(x)
    w[np.arange(64), t] = 1
    g1, l1, _ = ro.rowops_soft_ce(gpu(x), gpu(w))
    g2, l2, _ = ro.rowops_softmax_ce(gpu(x), gpu(t))
    check_abs(host(g1), host(g2), 2e-6 / 64, "one-hot grad")
    check_rel(host(l1), host(l2).astype(np.float64), "one-hot loss")


@pytest.mark.parametrize("cols", [3001, 20000, 20001])
@pytest.mark.parametrize("misalign", [False, True])
def test_ce_variants_many_rows_per_cta(ro, cols, misalign):
    # more rows than SMs: each CTA of the long-row kernel walks several rows
    rows = 400
    x, w, t = _inputs(rows, cols, 7 * cols)
    g, rl, ml = ro.rowops_soft_ce(gpu(x, misalign), gpu(w, misalign), grad_scale=1.0 / rows)
    gr, rlr, mlr = oracle.soft_ce(x, w, 1.0 / rows)
    wsum = np.abs(w.astype(np.float64)).sum(axis=1, keepdims=True)
    check_abs(host(g), gr, 2e-6 * (1.0 / rows) * np.maximum(1.0, wsum), f"soft ce grad cols={cols}")
    scale = np.maximum(1.0, np.abs(w.astype(np.float64)).sum(axis=1) * (np.abs(x).max(axis=1) + 10))
    check_abs(host(rl), rlr, 1e-5 * scale, f"soft ce loss cols={cols}")
    g, rl, ml = ro.rowops_teacher_ce(gpu(x, misalign), gpu(t, misalign), grad_scale=1.0 / rows)
    gr, rlr, mlr = oracle.teacher_ce(x, t, 1.0 / rows)
    check_abs(host(g), gr, 4e-6 / rows, f"teacher grad cols={cols}")
    check_rel(host(rl), rlr, f"teacher loss cols={cols}")
    check_rel(host(ml), [mlr], "teacher mean")


def _at_offset(a: np.ndarray, off: int) -> torch.Tensor:
    """Device copy of `a` whose data starts `off` floats past a 256-byte boundary."""
    a = np.ascontiguousarray(a, np.float32)
    flat = torch.zeros(a.size + 8, dtype=torch.float32, device="cuda")
    view = flat[off:off + a.size].view(a.shape)
    view.copy_(torch.from_numpy(a).cuda())
    return view


@pytest.mark.parametrize("cols", [20000, 20001])
def test_ce_variants_inputs_on_different_16_byte_phases(ro, cols):
    # long rows whose two inputs sit on different 16-byte phases: the
    # plain-load two-pass kernel instead of the bulk copies
    rows = 200
    x, w, t = _inputs(rows, cols, 11 * cols)
    xg, wg, tg = _at_offset(x, 0), _at_offset(w, 1), _at_offset(t, 2)
    g, rl, ml = ro.rowops_soft_ce(xg, wg, grad_scale=1.0 / rows)
    gr, rlr, mlr = oracle.soft_ce(x, w, 1.0 / rows)
    wsum = np.abs(w.astype(np.float64)).sum(axis=1, keepdims=True)
    check_abs(host(g), gr, 2e-6 * (1.0 / rows) * np.maximum(1.0, wsum), f"soft ce grad cols={cols}")
    scale = np.maximum(1.0, np.abs(w.astype(np.float64)).sum(axis=1) * (np.abs(x).max(axis=1) + 10))
    check_abs(host(rl), rlr, 1e-5 * scale, f"soft ce loss cols={cols}")
    g, rl, ml = ro.rowops_teacher_ce(xg, tg, grad_scale=1.0 / rows)
    gr, rlr, mlr = oracle.teacher_ce(x, t, 1.0 / rows)
    check_abs(host(g), gr, 4e-6 / rows, f"teacher grad cols={cols}")
    check_rel(host(rl), rlr, f"teacher loss cols={cols}")
    check_rel(host(ml), [mlr], "teacher mean")
    _, rl2, _ = ro.rowops_teacher_ce(xg, tg, with_grad=False)
    assert torch.equal(rl2, rl)
