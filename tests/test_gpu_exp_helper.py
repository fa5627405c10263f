"""GPU: the exp helpers every kernel uses, tested on their own.

exp_shifted(x, m) computes exp(x - m) as 2^((x - m) * log2(e)) with the MUFU
ex2.approx instruction: the difference d = fl(x - m) is taken first, then
scaled by log2(e) and rounded (a relative error of up to 1.22 |d| * 2^-24 in
the result, counting the fp32 rounding of log2(e) itself),
then ex2.approx adds its own few ulp.  merge2 rescales two running
(max, sum of exp) pairs to their common maximum with the same helper.  These
tests run both helpers elementwise through a test-only wrapper
(tests/csrc/exp_probe.cu) over the range the kernels feed them (x - m in
[-200, 0], plus -inf) and bound the error against float64 exp of the same fp32
difference and against CUDA's expf; the measured maxima are printed (run with
-s to see them)."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
U = 2.0 ** -24  # unit roundoff of fp32
TINY = 2.0 ** -126  # smallest normal fp32; ex2.approx.ftz flushes below it


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("exp_probe") / "exp_probe.so")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "--expt-relaxed-constexpr",
           "-shared", "-Xcompiler", "-fPIC", "-o", out, os.path.join(HERE, "csrc", "exp_probe.cu")]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.probe_exp_shifted.argtypes = [P, P, P, I]
    lib.probe_expf_diff.argtypes = [P, P, P, I]
    lib.probe_merge2.argtypes = [P, P, P, P, P, P, I]
    for f in (lib.probe_exp_shifted, lib.probe_expf_diff, lib.probe_merge2):
        f.restype = I
    return lib


def _run(fn, *arrays, n_out=1):
    dev = [torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda() for a in arrays]
    outs = [torch.empty_like(dev[0]) for _ in range(n_out)]
    assert fn(*(t.data_ptr() for t in dev + outs), dev[0].numel()) == 0
    return [o.cpu().numpy() for o in outs]


def _inputs():
    rng = np.random.default_rng(0)
    n = 1 << 20
    d = -rng.uniform(0.0, 200.0, n)                      # x - m over the kernels' range
    d[: n // 4] = -rng.uniform(0.0, 1.0, n // 4)        # dense near the maximum
    m = rng.uniform(-60.0, 60.0, n).astype(np.float32)  # maxima of logit-like rows
    m[: n // 8] = rng.choice([0.0, 30.0, -30.0, 1e4, -1e4], n // 8)
    x = (m.astype(np.float64) + d).astype(np.float32)
    return x, m


def test_exp_shifted_error_bound(probe):
    x, m = _inputs()
    got = _run(probe.probe_exp_shifted, x, m)[0].astype(np.float64)
    cuda = _run(probe.probe_expf_diff, x, m)[0].astype(np.float64)
    d = x.astype(np.float32) - m.astype(np.float32)      # the fp32 difference the helper sees
    assert (d <= 0).all()
    ref = np.exp(d.astype(np.float64))
    normal = ref >= TINY
    rel = np.abs(got - ref)[normal] / ref[normal]
    # scaling by log2(e) in fp32 costs up to 1.22 |d| * 2^-24 (the rounding of
    # the product, and the fp32 constant's own 0.22 ulp); ex2.approx a few ulp
    bound = (4.0 + 1.25 * np.abs(d[normal])) * U
    assert (rel <= bound).all(), f"max rel {rel.max():.3e}, worst ratio {(rel / bound).max():.2f}"
    assert (np.abs(got - ref)[~normal] <= TINY).all()  # flushed to zero or a tiny normal
    near = normal & (d > -1.0)
    rel_near = np.abs(got - ref)[near] / ref[near]
    assert rel_near.max() <= 5 * U
    rel_cuda = np.abs(got - cuda)[normal] / ref[normal]
    assert (rel_cuda <= bound + 2 * U).all()
    print(f"\nexp_shifted: max rel err vs float64 exp of the fp32 difference: "
          f"{rel_near.max():.3e} for d in (-1, 0], {rel.max():.3e} over [-87, 0] "
          f"(worst rel/((4+1.25|d|)*2^-24) {(rel / bound).max():.2f}); vs CUDA expf {rel_cuda.max():.3e}")


def test_exp_shifted_special_values(probe):
    x = np.array([0.0, 5.0, -3.0, -np.inf, -np.inf, 1e30, -87.0, -104.0, -200.0], np.float32)
    m = np.array([0.0, 5.0, -3.0, 0.0, 7.5, 1e30, 0.0, 0.0, 0.0], np.float32)
    got = _run(probe.probe_exp_shifted, x, m)[0]
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0 and got[5] == 1.0  # x == m: exactly 1
    assert got[3] == 0.0 and got[4] == 0.0  # exp(-inf) is exactly +0
    assert got[6] > 0 and abs(got[6] - np.exp(-87.0)) <= np.exp(-87.0) * 100 * U + TINY
    assert got[7] == 0.0 and got[8] == 0.0  # below the normal range: flushed to +0
    assert not np.signbit(got[[3, 4, 7, 8]]).any()


def test_merge2_rescale(probe):
    rng = np.random.default_rng(1)
    n = 1 << 18
    m1 = rng.uniform(-50, 50, n).astype(np.float32)
    m2 = (m1 + rng.uniform(-90, 90, n)).astype(np.float32)
    m2[: n // 8] = m1[: n // 8]  # equal maxima
    s1 = rng.uniform(1.0, 5e4, n).astype(np.float32)  # each sum holds its own maximum's 1
    s2 = rng.uniform(1.0, 5e4, n).astype(np.float32)
    m1[-4:] = [-np.inf, -np.inf, 3.0, -np.inf]
    s1[-4:] = [0.0, 0.0, 2.0, 0.0]
    m2[-4:] = [1.0, -np.inf, -np.inf, -np.inf]
    s2[-4:] = [3.0, 0.0, 0.0, 0.0]
    mo, so = _run(probe.probe_merge2, m1, s1, m2, s2, n_out=2)
    mm = np.maximum(m1, m2)
    assert np.array_equal(mo, mm)
    fin = np.isfinite(mm)
    with np.errstate(invalid="ignore"):
        ref = (s1.astype(np.float64) * np.exp(m1.astype(np.float64) - mm) +
               s2.astype(np.float64) * np.exp(m2.astype(np.float64) - mm))
    rel = np.abs(so[fin] - ref[fin]) / ref[fin]
    bound = (8.0 + 1.25 * np.abs(m1 - m2)[fin]) * U
    assert (rel <= bound).all(), f"max rel {rel.max():.3e}"
    assert so[-4] == 3.0 and so[-2] == 2.0  # an empty side (max -inf, sum 0) leaves the other as it is
    assert so[-3] == 0.0 and mo[-3] == -np.inf  # both empty: unchanged
    print(f"\nmerge2: max rel err {rel.max():.3e} (worst rel/((8+1.25|m1-m2|)*2^-24) {(rel / bound).max():.2f})")
