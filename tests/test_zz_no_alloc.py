"""The allocation-free LayerNorm backward (rowops_layernorm_bwd_noalloc).

It exists for callers that cannot allocate device memory at the point of the
call (a fixed device-memory budget, a host framework that owns all
allocations, code inside an allocator's out-of-memory path), so it uses a
fixed array inside the library as its workspace.  These tests call it through
the C ABI and check it against rowops_layernorm_bwd with a caller-owned
workspace: bit for bit where both run the same launch shape (the kernels are
deterministic), within the parity bounds where the array's size caps the CTA
count, and against the oracle at the benchmark's size.  A first call that
fills most of the array with other values precedes the smaller shapes, so a
read of a partial sum left by an earlier call would show.  This file sorts
last, so a run that stops at the first failure has run every other test
first."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_bound, gpu, host, ln_dx_bound, param_bound
from row_wise_softmax_warp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, dy, gamma, xh, rs, rows, cols):
    dx = torch.empty_like(dy)
    dg = torch.empty(cols, device=dy.device)
    db = torch.empty(cols, device=dy.device)
    st = lib.rowops_layernorm_bwd_noalloc(dy.data_ptr(), gamma.data_ptr(), xh.data_ptr(), rs.data_ptr(),
                                          dx.data_ptr(), dg.data_ptr(), db.data_ptr(), rows, cols,
                                          torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.rowops_status_string(st)
    return dx, dg, db


def _case(seed, rows, cols):
    n = inputs.layernorm(seed, rows=rows, cols=cols)
    _, xh, rs = oracle.layernorm_forward(n["x"], n["gamma"], n["beta"], n["eps"])
    xh32, rs32 = xh.astype(np.float32), rs.astype(np.float32)
    return n, xh32, rs32, (gpu(n["dy"]), gpu(n["gamma"]), gpu(xh32), gpu(rs32))


def _fill_array(lib):
    # 4096 x 768 writes 152 partials of 6 KB (most of the 1 MiB) with values
    # unlike those of the shapes that follow
    n, _, _, dev = _case(11, 4096, 768)
    _call_noalloc(lib, dev[0] * 3.0, *dev[1:], 4096, 768)
    torch.cuda.synchronize()


# Shapes whose launch is the same with and without the array's size limit:
# the fused kernel (aligned rows of 384..1024 floats) below its CTA cap, the
# lane-group kernel (shorter rows), the long-row kernel.
SAME_LAUNCH = [(45, 33), (300, 768), (4096, 768), (8, 16384), (3, 1000)]


@pytest.mark.parametrize("rows,cols", SAME_LAUNCH)
def test_noalloc_equals_workspace_version_twice(ro, rows, cols):
    lib = binding.library()
    _fill_array(lib)
    _, _, _, dev = _case(7, rows, cols)
    ref = ro.rowops_layernorm_bwd(*dev)  # caller-owned workspace
    for _ in range(2):  # the shared array keeps the previous call's contents
        got = _call_noalloc(lib, *dev, rows, cols)
        torch.cuda.synchronize()
        for name, u, v in zip(("dx", "dgamma", "dbeta"), got, ref):
            assert torch.equal(u, v), f"{name} differs from the workspace version at {rows}x{cols}"
    assert lib.rowops_pipeline_timeouts() == 0


@pytest.mark.parametrize("rows,cols", [(4096, 1024), (300, 1000), (20000, 900)])
def test_noalloc_capped_shapes_within_bounds(ro, rows, cols):
    # Rows of 863..1024 floats: the array holds fewer partials than one per
    # SM, so the allocation-free call runs fewer CTAs (each with more rows,
    # which can also select the other stage-1 kernel); dx and the column sums
    # then agree with the workspace version within the parity bounds.
    lib = binding.library()
    _fill_array(lib)
    n, xh32, rs32, dev = _case(8, rows, cols)
    ref = ro.rowops_layernorm_bwd(*dev)
    dxr, dgr, dbr = oracle.layernorm_backward(n["dy"], n["gamma"], xh32, rs32)
    dx_bound = ln_dx_bound(n["dy"], n["gamma"], xh32, rs32)
    for _ in range(2):
        dx, dg, db = _call_noalloc(lib, *dev, rows, cols)
        check_bound(host(dx), dxr, dx_bound, "dx vs oracle")
        check_bound(host(dx), host(ref[0]), 2 * dx_bound, "dx vs workspace version")
        check_bound(host(dg), dgr, param_bound(n["dy"], xh32), "dgamma vs oracle")
        check_bound(host(db), dbr, param_bound(n["dy"]), "dbeta vs oracle")
        check_bound(host(dg), host(ref[1]), param_bound(n["dy"], xh32), "dgamma vs workspace version")
    assert lib.rowops_pipeline_timeouts() == 0


def test_noalloc_matches_oracle_at_4096x768(ro):
    lib = binding.library()
    n, xh32, rs32, dev = _case(0, 4096, 768)
    dx, dg, db = (host(t) for t in _call_noalloc(lib, *dev, 4096, 768))
    dxr, dgr, dbr = oracle.layernorm_backward(n["dy"], n["gamma"], xh32, rs32)
    check_bound(dx, dxr, ln_dx_bound(n["dy"], n["gamma"], xh32, rs32), "dx")
    check_bound(dg, dgr, param_bound(n["dy"], xh32), "dgamma")
    check_bound(db, dbr, param_bound(n["dy"]), "dbeta")
    assert lib.rowops_pipeline_timeouts() == 0


def test_noalloc_refuses_oversize_after_the_common_checks(ro):
    lib = binding.library()
    cap = lib.rowops_layernorm_bwd_noalloc_max_bytes()
    assert cap == 1 << 20
    big = torch.empty(16, device="cuda")
    p = big.data_ptr()
    # 4096 rows of 4096 floats need more than 1 MiB of partial sums: valid,
    # separate buffers, refused by the size check before any launch
    mats = [torch.zeros(4096, 4096, device="cuda") for _ in range(3)]  # dy, xhat, dx
    vecs = [torch.zeros(4096, device="cuda") for _ in range(4)]        # gamma, inv_std, dgamma, dbeta
    ptrs = [mats[0], vecs[0], mats[1], vecs[1], mats[2], vecs[2], vecs[3]]
    assert lib.rowops_layernorm_bwd_noalloc(*(t.data_ptr() for t in ptrs), 4096, 4096, None) == 4
    del mats
    # the common checks come first: shape, NULL, alignment, overlap
    assert lib.rowops_layernorm_bwd_noalloc(None, None, None, None, None, None, None, 0, 768, None) == 0
    assert lib.rowops_layernorm_bwd_noalloc(None, None, None, None, None, None, None, 8, 0, None) == 2
    assert lib.rowops_layernorm_bwd_noalloc(None, None, None, None, None, None, None, 4096, 4096, None) == 1
    assert lib.rowops_layernorm_bwd_noalloc(p + 2, p, p, p, p, p, p, 4096, 4096, None) == 6  # ROWOPS_ERR_ALIGN
    assert lib.rowops_layernorm_bwd_noalloc(p, p + 64, p, p, p, p, p, 4096, 4096, None) == 3  # ROWOPS_ERR_ALIAS


@pytest.mark.parametrize("cols", [64, 383, 384, 768, 1000, 1024])
def test_noalloc_accepts_every_row_count_up_to_1024_columns(ro, cols):
    # The header's promise: with cols <= 1024 every row count fits the array.
    lib = binding.library()
    for rows in (1, 151, 152, 4096, 65536):
        dy = torch.zeros(rows, cols, device="cuda")
        xh = torch.zeros_like(dy)
        gamma = torch.ones(cols, device="cuda")
        rs = torch.ones(rows, device="cuda")
        dx, dg, db = _call_noalloc(lib, dy, gamma, xh, rs, rows, cols)
        torch.cuda.synchronize()
        assert not dx.any() and not dg.any() and not db.any()
    assert lib.rowops_pipeline_timeouts() == 0
