"""The allocation-free LayerNorm backward (rowops_layernorm_bwd_noalloc).

It exists for callers that cannot allocate device memory at the point of the
call (a fixed device-memory budget, a host framework that owns all
allocations, code inside an allocator's out-of-memory path), so it uses a
fixed array inside the library as its workspace.  This test calls it through
the C ABI twice in a row and checks each result against
rowops_layernorm_bwd with a caller-owned workspace, within the same bounds as
the other LayerNorm parity tests.  It lives in its own file that sorts last,
so a run that stops at the first failure has run every other test first."""
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


@pytest.mark.parametrize("rows,cols", [(4096, 768), (300, 1000), (45, 33)])
def test_noalloc_matches_workspace_version_twice(ro, rows, cols):
    lib = binding.library()
    n = inputs.layernorm(7, rows=rows, cols=cols)
    _, xh, rs = oracle.layernorm_forward(n["x"], n["gamma"], n["beta"], n["eps"])
    xh32, rs32 = xh.astype(np.float32), rs.astype(np.float32)
    dy, gamma, xh_d, rs_d = gpu(n["dy"]), gpu(n["gamma"]), gpu(xh32), gpu(rs32)
    ref = ro.rowops_layernorm_bwd(dy, gamma, xh_d, rs_d)  # caller-owned workspace
    ref = [host(t) for t in ref]
    for _ in range(2):  # the shared array keeps the previous call's contents
        dx, dg, db = (host(t) for t in _call_noalloc(lib, dy, gamma, xh_d, rs_d, rows, cols))
        check_bound(dx, ref[0], ln_dx_bound(n["dy"], n["gamma"], xh32, rs32), "dx vs workspace version")
        check_bound(dg, ref[1], param_bound(n["dy"], xh32), "dgamma vs workspace version")
        check_bound(db, ref[2], param_bound(n["dy"]), "dbeta vs workspace version")


def test_noalloc_refuses_oversize_and_keeps_common_checks(ro):
    lib = binding.library()
    cap = lib.rowops_layernorm_bwd_noalloc_max_bytes()
    assert cap == 1 << 20
    # 4096 columns x 4096 rows needs more than 1 MiB of partial sums
    assert lib.rowops_layernorm_bwd_workspace(4096, 4096) > cap
    big = torch.empty(16, device="cuda")
    p = big.data_ptr()
    assert lib.rowops_layernorm_bwd_noalloc(p, p + 64, p + 128, p + 192, p + 256, p + 320, p + 384,
                                            4096, 4096, None) == 4  # ROWOPS_ERR_WORKSPACE
    assert lib.rowops_layernorm_bwd_noalloc(None, None, None, None, None, None, None, 0, 768, None) == 0
    assert lib.rowops_layernorm_bwd_noalloc(None, None, None, None, None, None, None, 8, 768, None) == 1


def test_noalloc_fits_every_row_count_up_to_1024_columns(ro):
    # The header's promise: with cols <= 1024 the partial sums of any row
    # count fit the library's 1 MiB array (on the current device's SM count).
    lib = binding.library()
    cap = lib.rowops_layernorm_bwd_noalloc_max_bytes()
    for cols in (1, 64, 383, 384, 512, 768, 1000, 1023, 1024):
        for rows in (1, 151, 152, 4096, 65536, 10 ** 7):
            assert lib.rowops_layernorm_bwd_workspace(rows, cols) <= cap, (rows, cols)
