"""GPU parity: softmax_rows forward and backward against the oracle.

Covers the 256 x 128 workload in full, every row-length regime (sub-warp
groups, whole-warp registers, CTA rows, the bulk-copy pipelines, the streaming
fallback), ragged tails, misaligned (scalar-path) buffers and in-place use."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_bound, check_probs, gpu, host, softmax_bwd_bound
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu

COLS = [1, 2, 3, 4, 5, 8, 12, 16, 31, 32, 33, 64, 100, 127, 128, 129, 255, 256, 257, 768, 1000,
        1024, 1028, 1536, 2048, 3000, 4097, 8192, 12000, 16384, 16385, 50304, 140000]


def _x(rows, cols, seed):
    return inputs.softmax_pair(seed, rows=rows, cols=cols)


def test_softmax_workload_256x128(ro):
    d = inputs.softmax_pair(0)
    y = ro.rowops_softmax_fwd(gpu(d["x"]))
    check_probs(host(y), oracle.softmax_rows(d["x"]), "softmax fwd 256x128")
    y32 = oracle.softmax_rows(d["x"]).astype(np.float32)
    dx = ro.rowops_softmax_bwd(gpu(y32), gpu(d["dy"]))
    check_bound(host(dx), oracle.softmax_rows_backward(y32, d["dy"]), softmax_bwd_bound(y32, d["dy"]),
                "softmax bwd 256x128")


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("misalign", [False, True])
def test_softmax_shapes(ro, cols, misalign):
    rows = 7 if cols > 4096 else 37
    d = _x(rows, cols, cols)
    y = ro.rowops_softmax_fwd(gpu(d["x"], misalign))
    ref = oracle.softmax_rows(d["x"])
    check_probs(host(y), ref, f"softmax fwd cols={cols}")
    y32 = ref.astype(np.float32)
    dx = ro.rowops_softmax_bwd(gpu(y32, misalign), gpu(d["dy"], misalign))
    check_bound(host(dx), oracle.softmax_rows_backward(y32, d["dy"]), softmax_bwd_bound(y32, d["dy"]),
                f"softmax bwd cols={cols}")


@pytest.mark.parametrize("rows", [1, 2, 31, 33, 1000, 70001])
def test_softmax_row_counts(ro, rows):
    d = _x(rows, 64, rows)
    check_probs(host(ro.rowops_softmax_fwd(gpu(d["x"]))), oracle.softmax_rows(d["x"]), f"rows={rows}")


@pytest.mark.parametrize("cols", [128, 3000, 50304])
def test_softmax_in_place(ro, cols):
    d = _x(9, cols, 5)
    t = gpu(d["x"])
    y = ro.rowops_softmax_fwd(t, t)
    assert y.data_ptr() == t.data_ptr()
    check_probs(host(t), oracle.softmax_rows(d["x"]), "in place")


def test_softmax_extremes(ro):
    x = np.array([[1000, 1000, -1000, 0], [-1000, -1000, -1000, -1000], [88, -88, 0, 1e-30],
                  [3.4e38, 3.4e38, 0, 0]], np.float32)
    check_probs(host(ro.rowops_softmax_fwd(gpu(x))), oracle.softmax_rows(x), "extremes")


def test_softmax_empty(ro):
    import torch
    x = torch.empty((0, 128), device="cuda")
    assert ro.rowops_softmax_fwd(x).shape == (0, 128)
    x = torch.empty((5, 0), device="cuda")
    assert ro.rowops_softmax_fwd(x).shape == (5, 0)


def test_softmax_deterministic(ro):
    d = _x(512, 50304, 3)
    x = gpu(d["x"])
    a = host(ro.rowops_softmax_fwd(x))
    b = host(ro.rowops_softmax_fwd(x))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def _at_offset(a: np.ndarray, off: int) -> torch.Tensor:
    """Device copy of `a` whose data starts `off` floats past a 256-byte boundary."""
    a = np.ascontiguousarray(a, np.float32)
    flat = torch.zeros(a.size + 8, dtype=torch.float32, device="cuda")
    view = flat[off:off + a.size].view(a.shape)
    view.copy_(torch.from_numpy(a).cuda())
    return view


@pytest.mark.parametrize("rows,cols", [(400, 16388), (160, 32768), (3, 100003)])
@pytest.mark.parametrize("offs", [(0, 0, 0), (1, 1, 0), (2, 2, 3), (0, 1, 0)])
def test_softmax_bwd_long_rows(ro, rows, cols, offs):
    # rows past the block-row kernels: (y, dy) chunk pairs through the
    # bulk-copy ring, with more rows than SMs, heads and tails off 16-byte
    # boundaries, dx on another phase (scalar stores), and y and dy on
    # different phases (the streaming fallback)
    d = _x(rows, cols, rows + cols)
    y32 = oracle.softmax_rows(d["x"]).astype(np.float32)
    dx = _at_offset(np.zeros_like(y32), offs[2])
    ro.rowops_softmax_bwd(_at_offset(y32, offs[0]), _at_offset(d["dy"], offs[1]), dx)
    check_bound(host(dx), oracle.softmax_rows_backward(y32, d["dy"]), softmax_bwd_bound(y32, d["dy"]),
                f"softmax bwd {rows}x{cols} offsets {offs}")
    assert ro.library().rowops_pipeline_timeouts() == 0
