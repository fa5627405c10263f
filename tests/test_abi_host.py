"""The C ABI on the host: the library loads, exports what include/rowops.h
declares, and rejects bad arguments with the documented status codes before
touching the GPU.  The pointers below are never dereferenced: every call here
fails validation (or is an empty no-op), so no kernel is launched."""
import os
import re

import pytest

import __graft_entry__
from row_wise_softmax_warp_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, NULL, SHAPE, ALIAS, WORKSPACE, CUDA, ALIGN = 0, 1, 2, 3, 4, 5, 6

A = 0x7000_0000_0000  # fake, 256-byte aligned device addresses far apart
B = 0x7100_0000_0000
C = 0x7200_0000_0000
D = 0x7300_0000_0000
E = 0x7400_0000_0000
F = 0x7500_0000_0000
G = 0x7600_0000_0000
H = 0x7700_0000_0000
W = 0x7800_0000_0000


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.library()


def test_exports_every_declared_symbol(lib):
    header = open(os.path.join(ROOT, "include", "rowops.h")).read()
    declared = set(re.findall(r"\b(rowops_[a-z0-9_]+)\s*\(", header))
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(binding.SIGNATURES), declared ^ set(binding.SIGNATURES)


def test_status_strings(lib):
    for s in range(7):
        assert lib.rowops_status_string(s).startswith(b"ROWOPS")
    assert b"unknown" in lib.rowops_status_string(99)


def test_dims(lib):
    n0 = lib.rowops_kernel_launches()
    assert lib.rowops_softmax_fwd(A, B, -1, 4, None) == SHAPE
    assert lib.rowops_softmax_fwd(A, B, 4, -1, None) == SHAPE
    assert lib.rowops_softmax_fwd(A, B, 4, 1 << 31, None) == SHAPE
    assert lib.rowops_softmax_fwd(A, B, 1 << 40, 1 << 30, None) == SHAPE
    assert lib.rowops_softmax_fwd(A, B, 0, 128, None) == OK  # empty: no-op
    assert lib.rowops_softmax_fwd(None, None, 0, 128, None) == OK
    assert lib.rowops_softmax_fwd(A, B, 8, 0, None) == OK
    assert lib.rowops_softmax_bwd(A, B, C, 8, 0, None) == OK
    assert lib.rowops_masked_softmax(A, B, C, 8, 0, None) == OK
    assert lib.rowops_kernel_launches() == n0


def test_null_pointers(lib):
    assert lib.rowops_softmax_fwd(None, B, 2, 4, None) == NULL
    assert lib.rowops_softmax_bwd(A, None, C, 2, 4, None) == NULL
    assert lib.rowops_attn_softmax_fwd(A, None, 8, 8, 8, 0.5, None) == NULL
    assert lib.rowops_attn_softmax_bwd(A, B, None, 8, 8, 8, 0.5, None) == NULL
    assert lib.rowops_masked_softmax(A, None, C, 2, 4, None) == NULL
    assert lib.rowops_logsumexp(A, None, 2, 4, None) == NULL
    assert lib.rowops_softmax_ce(A, B, C, D, None, 2, 4, 0.5, None) == NULL
    assert lib.rowops_layernorm_fwd(A, B, C, D, E, None, 2, 4, 1e-5, None) == NULL
    assert lib.rowops_layernorm_bwd(A, B, C, D, E, F, None, 2, 4, W, 1 << 20, None) == NULL
    assert lib.rowops_topk_kept(None, B, 2, 4, 1, None) == NULL


def test_element_alignment(lib):
    # a float pointer that is not 4-byte aligned (or a double that is not
    # 8-byte aligned) is refused before any launch; byte masks may sit anywhere
    n0 = lib.rowops_kernel_launches()
    assert lib.rowops_softmax_fwd(A + 2, B, 2, 4, None) == ALIGN
    assert lib.rowops_softmax_fwd(A, B + 1, 2, 4, None) == ALIGN
    assert lib.rowops_softmax_bwd(A, B, C + 2, 2, 4, None) == ALIGN
    assert lib.rowops_attn_softmax_fwd(A + 2, B, 8, 8, 8, 0.5, None) == ALIGN
    assert lib.rowops_attn_softmax_bwd(A, B + 2, C, 8, 8, 8, 0.5, None) == ALIGN
    assert lib.rowops_logsumexp(A, B + 2, 2, 4, None) == ALIGN
    assert lib.rowops_softmax_ce(A, B + 2, C, D, E, 2, 4, 0.5, None) == ALIGN  # int32 targets
    assert lib.rowops_softmax_ce(A, B, C, D, E + 4, 2, 4, 0.5, None) == ALIGN  # double mean
    assert lib.rowops_layernorm_fwd(A, B, C + 2, D, E, F, 2, 4, 1e-5, None) == ALIGN
    assert lib.rowops_layernorm_bwd(A, B, C, D + 2, E, F, G, 2, 4, W, 1 << 20, None) == ALIGN
    assert lib.rowops_topk_kept(A, B + 2, 2, 4, 1, None) == ALIGN
    assert lib.rowops_masked_softmax_fmask(A, B + 2, C, 2, 4, None) == ALIGN
    assert lib.rowops_soft_ce(A, B, C, D + 2, E, 2, 4, 0.5, None) == ALIGN
    assert lib.rowops_teacher_ce(A, B, C, D, E + 4, 2, 4, 0.5, None) == ALIGN
    assert lib.rowops_masked_softmax(A + 2, B + 1, C, 2, 4, None) == ALIGN
    assert lib.rowops_kernel_launches() == n0


def test_aliasing(lib):
    n = 16 * 64 * 4
    assert lib.rowops_softmax_fwd(A, A + 64, 16, 64, None) == ALIAS       # partial overlap
    assert lib.rowops_softmax_bwd(A, B, A, 16, 64, None) == ALIAS         # dx == y
    assert lib.rowops_softmax_bwd(A, B, B + n - 4, 16, 64, None) == ALIAS  # dx tail overlaps dy
    assert lib.rowops_attn_softmax_fwd(A, A, 64, 64, 64, 0.125, None) == ALIAS
    assert lib.rowops_attn_softmax_bwd(A, B, B, 64, 64, 64, 0.125, None) == ALIAS
    assert lib.rowops_masked_softmax(A, A + 128, B, 16, 64, None) == ALIAS  # mask inside x
    assert lib.rowops_logsumexp(A, A + 8, 16, 64, None) == ALIAS
    assert lib.rowops_softmax_ce(A, B, A, D, E, 16, 64, 0.1, None) == ALIAS        # grad == logits
    assert lib.rowops_softmax_ce(A, B, C, D, D + 8, 16, 64, 0.1, None) == ALIAS    # mean in row_loss
    assert lib.rowops_layernorm_fwd(A, B, C, D, D, E, 16, 64, 1e-5, None) == ALIAS  # out == xhat
    assert lib.rowops_layernorm_bwd(A, B, C, D, A, F, G, 16, 64, W, 1 << 20, None) == ALIAS
    assert lib.rowops_layernorm_bwd(A, B, C, D, E, F, F, 16, 64, W, 1 << 20, None) == ALIAS
    assert lib.rowops_layernorm_bwd(A, B, C, D, E, F, G, 16, 64, E, 1 << 20, None) == ALIAS
    assert lib.rowops_topk_kept(A, A, 16, 64, 2, None) == ALIAS


def test_attention_shape_rules(lib):
    assert lib.rowops_attn_softmax_fwd(A, B, 64, 32, 64, 0.125, None) == SHAPE  # cols != seq_len
    assert lib.rowops_attn_softmax_fwd(A, B, 65, 64, 64, 0.125, None) == SHAPE  # rows % seq_len
    assert lib.rowops_attn_softmax_fwd(A, B, 64, 64, 0, 0.125, None) == SHAPE
    assert lib.rowops_attn_softmax_fwd(A, B, 64, 64, 64, 0.0, None) == SHAPE
    assert lib.rowops_attn_softmax_fwd(A, B, 64, 64, 64, -1.0, None) == SHAPE
    assert lib.rowops_attn_softmax_fwd(A, B, 64, 64, 64, float("inf"), None) == SHAPE
    assert lib.rowops_attn_softmax_bwd(A, B, C, 64, 64, 64, float("nan"), None) == SHAPE
    assert lib.rowops_attn_softmax_fwd(A, B, 0, 64, 64, 0.125, None) == OK


def test_scalar_rules(lib):
    assert lib.rowops_topk_kept(A, B, 4, 8, 0, None) == SHAPE
    assert lib.rowops_topk_kept(A, B, 4, 8, 9, None) == SHAPE
    assert lib.rowops_topk_kept(A, B, 4, 0, 1, None) == SHAPE
    assert lib.rowops_topk_kept(A, B, 0, 8, 8, None) == OK
    assert lib.rowops_softmax_ce(A, B, C, D, E, 4, 0, 0.25, None) == SHAPE
    assert lib.rowops_softmax_ce(A, B, C, D, E, 4, 8, float("nan"), None) == SHAPE
    assert lib.rowops_layernorm_fwd(A, B, C, D, E, F, 4, 0, 1e-5, None) == SHAPE
    assert lib.rowops_layernorm_fwd(A, B, C, D, E, F, 4, 8, -1e-5, None) == SHAPE
    assert lib.rowops_layernorm_fwd(A, B, C, D, E, F, 4, 8, float("inf"), None) == SHAPE
    assert lib.rowops_layernorm_bwd(A, B, C, D, E, F, G, 4, 0, W, 1 << 20, None) == SHAPE


def test_layernorm_workspace(lib):
    need = lib.rowops_layernorm_bwd_workspace(4096, 768)
    assert need > 0 and need % 16 == 0
    assert lib.rowops_layernorm_bwd_workspace(0, 768) == 0
    assert lib.rowops_layernorm_bwd_workspace(-1, 768) == 0
    # the partial count is capped, so the workspace grows at most linearly in cols
    big = lib.rowops_layernorm_bwd_workspace(1 << 24, 768)
    assert big <= 128 * 2 * 768 * 4
    assert lib.rowops_layernorm_bwd(A, B, C, D, E, F, G, 4096, 768, None, need, None) == WORKSPACE
    assert lib.rowops_layernorm_bwd(A, B, C, D, E, F, G, 4096, 768, W, need - 4, None) == WORKSPACE
    assert lib.rowops_layernorm_bwd(A, B, C, D, E, F, G, 4096, 768, W + 4, need, None) == WORKSPACE
    assert lib.rowops_layernorm_bwd(A, B, C, D, E, F, G, 0, 768, None, 0, None) == OK


def test_router_and_top_k_rules(lib):
    assert lib.rowops_router_masked_topk(A, B, C, D, 4, 8, 0, None) == SHAPE
    assert lib.rowops_router_masked_topk(A, B, C, D, 4, 8, 9, None) == SHAPE
    assert lib.rowops_router_masked_topk(A, B, C, C, 4, 8, 2, None) == ALIAS   # kept == p
    assert lib.rowops_router_masked_topk(A, B, A + 4, D, 4, 8, 2, None) == ALIAS  # p overlaps x partially
    assert lib.rowops_router_masked_topk(A, None, C, D, 4, 8, 2, None) == NULL
    assert lib.rowops_top_k_rows(A, B, C, 4, 8, 9, 1, None) == SHAPE
    assert lib.rowops_top_k_rows(A, B, C, 4, (1 << 24) + 4, 2, 1, None) == SHAPE
    assert lib.rowops_top_k_rows(A, B, B, 4, 8, 2, 1, None) == ALIAS
    assert lib.rowops_top_k_rows(A, None, C, 4, 8, 2, 0, None) == NULL
    assert lib.rowops_top_k_rows(A, B, C, 0, 8, 2, 0, None) == OK


def test_misc_rules(lib):
    assert lib.rowops_masked_softmax_fmask(A, A + 64, C, 4, 64, None) == ALIAS
    assert lib.rowops_masked_softmax_fmask(A, B, None, 4, 64, None) == NULL
    assert lib.rowops_lrp_softmax_rows(A, B, C, C, 4, 8, None) == ALIAS
    assert lib.rowops_lrp_softmax_rows(A, B, None, D, 4, 8, None) == NULL
    assert lib.rowops_argmax_onehot(A, A, 4, 8, None) == ALIAS
    assert lib.rowops_argmax_onehot(A, B, 4, 0, None) == OK
    assert lib.rowops_rmsnorm_fwd(A, B, C, D, 4, 8, -1.0, None) == SHAPE
    assert lib.rowops_rmsnorm_bwd(A, B, C, D, A, F, 4, 8, None) == ALIAS
    assert lib.rowops_column_sums(A, A + 16, 4, 8, 0.0, None) == ALIAS
    assert lib.rowops_column_sums(A, B, 4, 8, float("inf"), None) == SHAPE


def test_rejected_calls_launch_nothing(lib):
    n0 = lib.rowops_kernel_launches()
    lib.rowops_topk_kept(A, A, 16, 64, 2, None)
    lib.rowops_softmax_ce(A, B, C, D, E, 4, 0, 0.25, None)
    assert lib.rowops_kernel_launches() == n0


def test_header_is_plain_c(lib, tmp_path):
    # include/rowops.h compiles as strict C99 and a C program links against the
    # library and gets the documented answers (no call here reaches the GPU)
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "abi_c.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "rowops.h"
int main(void) {
    rowops_stream s = NULL;
    if (strncmp(rowops_status_string(ROWOPS_ERR_SHAPE), "ROWOPS_ERR_SHAPE", 16) != 0) return 1;
    if (rowops_softmax_fwd(NULL, NULL, -1, 4, s) != ROWOPS_ERR_SHAPE) return 2;
    if (rowops_softmax_fwd(NULL, NULL, 0, 4, s) != ROWOPS_OK) return 3;
    if (rowops_topk_kept(NULL, NULL, 4, 8, 9, s) != ROWOPS_ERR_SHAPE) return 4;
    if (rowops_layernorm_bwd_workspace(0, 768) != 0) return 5;
    puts("ok");
    return 0;
}
""")
    exe = tmp_path / "abi_c"
    libpath = binding.LIB_PATH
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"), str(src), libpath,
                           "-Wl,-rpath," + os.path.dirname(libpath), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)
