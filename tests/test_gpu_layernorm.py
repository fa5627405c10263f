"""GPU parity: LayerNorm forward (out, xhat, inv_std) and backward
(dx, dgamma, dbeta)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_bound, check_rel, gpu, host, ln_dx_bound, param_bound
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu


def _run(ro, n, misalign=False):
    x, gamma, beta, dy, eps = n["x"], n["gamma"], n["beta"], n["dy"], n["eps"]
    out, xh, rs = ro.rowops_layernorm_fwd(gpu(x, misalign), gpu(gamma, misalign), gpu(beta, misalign),
                                          eps=eps)
    o_r, xh_r, rs_r = oracle.layernorm_forward(x, gamma, beta, eps)
    check_rel(host(xh), xh_r, "xhat")
    check_rel(host(out), o_r, "out")
    check_bound(host(rs), rs_r, 1e-5 * np.abs(rs_r), "inv_std")
    xh32, rs32 = xh_r.astype(np.float32), rs_r.astype(np.float32)
    dx, dg, db = ro.rowops_layernorm_bwd(gpu(dy, misalign), gpu(gamma, misalign), gpu(xh32, misalign),
                                         gpu(rs32))
    dxr, dgr, dbr = oracle.layernorm_backward(dy, gamma, xh32, rs32)
    check_bound(host(dx), dxr, ln_dx_bound(dy, gamma, xh32, rs32), "dx")
    check_bound(host(dg), dgr, param_bound(dy, xh32), "dgamma")
    check_bound(host(db), dbr, param_bound(dy), "dbeta")


def test_layernorm_workload_4096x768(ro):
    _run(ro, inputs.layernorm(0))


@pytest.mark.parametrize("cols", [1, 2, 3, 4, 7, 16, 33, 64, 127, 128, 256, 257, 768, 1000, 1024, 1028,
                                  1536, 2049, 3000, 4096, 8192, 8193, 12000, 16384, 16388])
@pytest.mark.parametrize("misalign", [False, True])
def test_layernorm_shapes(ro, cols, misalign):
    _run(ro, inputs.layernorm(cols, rows=45, cols=cols), misalign)


@pytest.mark.parametrize("rows", [1, 7, 8, 9, 63, 64, 65, 1000, 20000, 200000])
def test_layernorm_row_counts(ro, rows):
    # covers empty CTAs and clusters, ragged last blocks and the capped partial count
    _run(ro, inputs.layernorm(rows, rows=rows, cols=256))


@pytest.mark.parametrize("rows", [1, 15, 16, 17, 151, 153, 4097, 20000])
@pytest.mark.parametrize("cols", [384, 388, 764, 1020, 1024])
def test_layernorm_bwd_row_blocks(ro, rows, cols):
    # rows of 384..1024 floats on 16-byte boundaries: blocks of rows through
    # the bulk-copy ring, with partial last slots and blocks, CTAs with fewer
    # rows than warps, and the CTA cap of the 1020- and 1024-float rows
    _run(ro, inputs.layernorm(rows * 7 + cols, rows=rows, cols=cols))


@pytest.mark.parametrize("per_sm", [2, 3, 5, 9, 13, 16])
@pytest.mark.parametrize("cols", [384, 512, 768, 1000])
def test_layernorm_bwd_column_owner_phases(ro, per_sm, cols):
    # rows of 384..1024 floats whose CTA block fits in shared memory: each row
    # set's threads take one to eight rows a phase, so the phases alternate
    # between the per-row butterfly and the reduce-scatter, and between the
    # inline sum of the warps' row sums and the once-per-row sum (sets of one
    # CTA differ by a row, so they differ there too); a ragged count leaves
    # the last CTA short
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for rows in (sms * per_sm, sms * per_sm - 77):
        _run(ro, inputs.layernorm(rows + cols, rows=rows, cols=cols))


@pytest.mark.parametrize("rows,cols", [(2000, 2048), (700, 4100), (333, 8192), (400, 16384), (300, 30001)])
@pytest.mark.parametrize("misalign", [False, True])
def test_layernorm_block_rows_many_rows_per_cta(ro, rows, cols, misalign):
    # rows of 1025..8192 floats: each CTA of the block-row backward walks
    # several rows and carries its column partials across them
    _run(ro, inputs.layernorm(rows + cols, rows=rows, cols=cols), misalign)


def test_layernorm_eps_zero_and_constant_rows(ro):
    n = inputs.layernorm(3, rows=16, cols=64, eps=0.0)
    _run(ro, n)
    x = np.full((4, 64), 2.5, np.float32)
    _, xh, rs = ro.rowops_layernorm_fwd(gpu(x), gpu(np.ones(64, np.float32)), gpu(np.zeros(64, np.float32)),
                                        eps=1e-5)
    assert (host(xh) == 0).all()
    check_bound(host(rs), np.full(4, 1 / np.sqrt(1e-5)), 1e-5 / np.sqrt(1e-5), "constant rows")


def test_layernorm_bwd_deterministic(ro):
    n = inputs.layernorm(4)
    args = [gpu(n["dy"]), gpu(n["gamma"]), gpu(n["x"]), gpu(np.ones(4096, np.float32))]
    a = ro.rowops_layernorm_bwd(*args)
    b = ro.rowops_layernorm_bwd(*args)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_layernorm_workspace_is_reusable_and_unzeroed(ro):
    n = inputs.layernorm(5, rows=300, cols=768)
    need = ro.rowops_layernorm_bwd_workspace(300, 768)
    ws = torch.full((need,), 0x7f, dtype=torch.uint8, device="cuda")  # garbage
    xh32 = oracle.layernorm_forward(n["x"], n["gamma"], n["beta"], 1e-5)[1].astype(np.float32)
    rs = np.ones(300, np.float32)
    r1 = ro.rowops_layernorm_bwd(gpu(n["dy"]), gpu(n["gamma"]), gpu(xh32), gpu(rs), workspace=ws)
    r2 = ro.rowops_layernorm_bwd(gpu(n["dy"]), gpu(n["gamma"]), gpu(xh32), gpu(rs), workspace=ws)
    for u, v in zip(r1, r2):
        assert torch.equal(u, v)
    dxr, dgr, dbr = oracle.layernorm_backward(n["dy"], n["gamma"], xh32, rs)
    check_bound(host(r1[2]), dbr, param_bound(n["dy"]), "dbeta")
