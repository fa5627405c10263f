"""CPU oracle for the row ops (ctypes wrapper around ``rowops_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library and its
Python binding never import this package.

Every function takes numpy arrays, widens them to float64 (exact for fp32
inputs), runs the double-precision C definitions and returns float64 results.
Rows are independent, so large inputs are split into contiguous row blocks run
on a thread pool (ctypes releases the GIL); the arithmetic inside a row is the
plain sequential loop of the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rowops_oracle.c")
_LIB = os.path.join(_HERE, "librowops_oracle.so")

_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_SIGNATURES = {
    "oracle_softmax_rows": [_D, _D, _I64, _I64],
    "oracle_softmax_rows_backward": [_D, _D, _D, _I64, _I64],
    "oracle_attn_softmax_forward": [_D, _D, _I64, _I64, _I64, _I64, ctypes.c_double],
    "oracle_attn_softmax_backward": [_D, _D, _D, _I64, _I64, _I64, _I64, ctypes.c_double],
    "oracle_logsumexp_rows": [_D, _D, _I64, _I64],
    "oracle_softmax_cross_entropy": [_D, _I32, _D, _D, _I64, _I64, ctypes.c_double],
    "oracle_mean": [_D, _I64],
    "oracle_layernorm_forward": [_D, _D, _D, _D, _D, _D, _I64, _I64, ctypes.c_double],
    "oracle_layernorm_backward_input": [_D, _D, _D, _D, _D, _I64, _I64],
    "oracle_layernorm_backward_params": [_D, _D, _D, _D, _I64, _I64],
    "oracle_masked_softmax": [_D, _U8, _D, _I64, _I64],
    "oracle_topk_kept": [_D, _U8, _I64, _I64, _I64],
    "oracle_top_k_rows": [_D, _D, _D, _I64, _I64, _I64, ctypes.c_int, _U8],
    "oracle_rms_norm_forward": [_D, _D, _D, _D, _I64, _I64, ctypes.c_double],
    "oracle_rms_norm_backward": [_D, _D, _D, _D, _D, _D, _I64, _I64],
    "oracle_column_sums": [_D, _D, _I64, _I64, ctypes.c_double],
    "oracle_lrp_softmax_rows": [_D, _D, _D, _D, _I64, _I64],
    "oracle_masked_softmax_fmask": [_D, _D, _D, _I64, _I64],
    "oracle_argmax_onehot": [_D, _D, _I64, _I64],
    "oracle_soft_ce": [_D, _D, _D, _D, _I64, _I64, ctypes.c_double],
    "oracle_teacher_ce": [_D, _D, _D, _D, _I64, _I64, ctypes.c_double],
}


def bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    for name, args in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_double if name == "oracle_mean" else None
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


def swap_library(lib):
    """Make every function below call ``lib`` (a value from ``bind``); returns the
    previous one.  Used by the tests that check the pins reject planted mistakes."""
    global _lib
    prev = _load()
    _lib = lib
    return prev


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def _2d(a, cols=None) -> np.ndarray:
    a = _f64(a)
    if a.ndim == 1 and cols is not None:
        a = a.reshape(-1, cols)
    if a.ndim != 2:
        raise ValueError("expected a (rows, cols) matrix")
    return a


def _p(a, ctype=_D):
    return a.ctypes.data_as(ctype)


_THREADS = None


def threads() -> int:
    """Worker threads used for large inputs (all host cores unless ROWOPS_ORACLE_THREADS)."""
    global _THREADS
    if _THREADS is None:
        _THREADS = int(os.environ.get("ROWOPS_ORACLE_THREADS", "0")) or (os.cpu_count() or 1)
    return _THREADS


def _row_blocks(rows: int, cols: int, n_threads: int | None):
    n = n_threads or threads()
    # Keep tiny problems on the calling thread.
    if n <= 1 or rows * max(cols, 1) < (1 << 16):
        return [(0, rows)]
    n = min(n, rows)
    step = -(-rows // n)
    return [(r0, min(rows, r0 + step)) for r0 in range(0, rows, step)]


def _run(blocks, fn):
    if len(blocks) == 1:
        fn(*blocks[0])
        return
    with ThreadPoolExecutor(max_workers=len(blocks)) as ex:
        list(ex.map(lambda b: fn(*b), blocks))


def softmax_rows(x, n_threads=None) -> np.ndarray:
    lib = _load()
    x = _2d(x)
    rows, cols = x.shape
    y = np.empty_like(x)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_softmax_rows(_p(x[a:b]), _p(y[a:b]), b - a, cols))
    return y


def softmax_rows_backward(y, dy, n_threads=None) -> np.ndarray:
    lib = _load()
    y, dy = _2d(y), _2d(dy)
    rows, cols = y.shape
    dx = np.empty_like(y)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_softmax_rows_backward(_p(y[a:b]), _p(dy[a:b]), _p(dx[a:b]),
                                                       b - a, cols))
    return dx


def attn_softmax_forward(scores, seq_len: int, scale: float, row0: int = 0,
                         n_threads=None) -> np.ndarray:
    """Rows are stacked (batch*heads*seq_len) query rows; row0 = global index of the first."""
    lib = _load()
    s = _2d(scores)
    rows, cols = s.shape
    p = np.empty_like(s)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_attn_softmax_forward(_p(s[a:b]), _p(p[a:b]), b - a, cols,
                                                      seq_len, row0 + a, scale))
    return p


def attn_softmax_backward(p, dp, seq_len: int, scale: float, row0: int = 0,
                          n_threads=None) -> np.ndarray:
    lib = _load()
    p, dp = _2d(p), _2d(dp)
    rows, cols = p.shape
    ds = np.empty_like(p)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_attn_softmax_backward(_p(p[a:b]), _p(dp[a:b]), _p(ds[a:b]),
                                                       b - a, cols, seq_len, row0 + a, scale))
    return ds


def logsumexp_rows(x, n_threads=None) -> np.ndarray:
    lib = _load()
    x = _2d(x)
    rows, cols = x.shape
    out = np.empty(rows)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_logsumexp_rows(_p(x[a:b]), _p(out[a:b]), b - a, cols))
    return out


def softmax_cross_entropy(logits, targets, grad_scale: float, n_threads=None):
    """Returns (grad, row_loss, mean_loss)."""
    lib = _load()
    x = _2d(logits)
    rows, cols = x.shape
    t = np.ascontiguousarray(np.asarray(targets), dtype=np.int32).reshape(rows)
    grad = np.empty_like(x)
    row_loss = np.empty(rows)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_softmax_cross_entropy(_p(x[a:b]), _p(t[a:b], _I32), _p(grad[a:b]),
                                                       _p(row_loss[a:b]), b - a, cols, grad_scale))
    mean = lib.oracle_mean(_p(row_loss), rows) if rows else float("nan")
    return grad, row_loss, mean


def mean(v) -> float:
    lib = _load()
    v = _f64(v).reshape(-1)
    return lib.oracle_mean(_p(v), v.size)


def layernorm_forward(x, gamma, beta, eps: float, n_threads=None):
    """Returns (out, xhat, inv_std)."""
    lib = _load()
    x = _2d(x)
    rows, cols = x.shape
    gamma, beta = _f64(gamma).reshape(cols), _f64(beta).reshape(cols)
    out, xhat, inv_std = np.empty_like(x), np.empty_like(x), np.empty(rows)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_layernorm_forward(_p(x[a:b]), _p(gamma), _p(beta), _p(out[a:b]),
                                                   _p(xhat[a:b]), _p(inv_std[a:b]), b - a, cols,
                                                   eps))
    return out, xhat, inv_std


def layernorm_backward_input(g, gamma, xhat, inv_std, n_threads=None) -> np.ndarray:
    lib = _load()
    g, xhat = _2d(g), _2d(xhat)
    rows, cols = g.shape
    gamma = _f64(gamma).reshape(cols)
    inv_std = _f64(inv_std).reshape(rows)
    dx = np.empty_like(g)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_layernorm_backward_input(_p(g[a:b]), _p(gamma), _p(xhat[a:b]),
                                                          _p(inv_std[a:b]), _p(dx[a:b]), b - a,
                                                          cols))
    return dx


def layernorm_backward_params(g, xhat):
    """Returns (dgamma, dbeta): column sums in increasing row order (single thread)."""
    lib = _load()
    g, xhat = _2d(g), _2d(xhat)
    rows, cols = g.shape
    dgamma, dbeta = np.empty(cols), np.empty(cols)
    lib.oracle_layernorm_backward_params(_p(g), _p(xhat), _p(dgamma), _p(dbeta), rows, cols)
    return dgamma, dbeta


def layernorm_backward(g, gamma, xhat, inv_std, n_threads=None):
    """Returns (dx, dgamma, dbeta)."""
    dx = layernorm_backward_input(g, gamma, xhat, inv_std, n_threads)
    dgamma, dbeta = layernorm_backward_params(g, xhat)
    return dx, dgamma, dbeta


def masked_softmax(x, mask, n_threads=None) -> np.ndarray:
    lib = _load()
    x = _2d(x)
    rows, cols = x.shape
    m = np.ascontiguousarray(np.asarray(mask), dtype=np.uint8).reshape(rows, cols)
    y = np.empty_like(x)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_masked_softmax(_p(x[a:b]), _p(m[a:b], _U8), _p(y[a:b]), b - a,
                                                cols))
    return y


def topk_kept(x, k: int, n_threads=None) -> np.ndarray:
    """uint8 (rows, cols): 1 where fewer than k entries of the row beat the entry."""
    lib = _load()
    x = _2d(x)
    rows, cols = x.shape
    kept = np.empty((rows, cols), dtype=np.uint8)
    _run(_row_blocks(rows, cols * cols, n_threads),
         lambda a, b: lib.oracle_topk_kept(_p(x[a:b]), _p(kept[a:b], _U8), b - a, cols, k))
    return kept


def top_k_rows(x, k: int, largest: bool = True, n_threads=None):
    """Returns (values, indices) of shape (rows, k): the k largest (or smallest)
    entries of each row in rank order (NaN above every number, equal values
    lower column first); indices as float64 whole numbers."""
    lib = _load()
    x = _2d(x)
    rows, cols = x.shape
    values = np.empty((rows, k))
    indices = np.empty((rows, k))

    def run(a, b):
        taken = np.empty(max(cols, 1), dtype=np.uint8)
        lib.oracle_top_k_rows(_p(x[a:b]), _p(values[a:b]), _p(indices[a:b]), b - a, cols, k,
                              1 if largest else 0, _p(taken, _U8))
    _run(_row_blocks(rows, cols * max(k, 1), n_threads), run)
    return values, indices


def router_masked_topk(x, mask, k: int, n_threads=None):
    """The fused MoE router: P = masked_softmax(x, mask) and the top-k kept mask
    of P.  The kept decision is taken on P rounded to fp32, the precision in
    which the kernel stores P.  Returns (P in float64, kept as uint8)."""
    p = masked_softmax(x, mask, n_threads)
    return p, topk_kept(p.astype(np.float32), k, n_threads)


def rms_norm_forward(x, gamma, eps: float, n_threads=None):
    """Returns (out, row_rms)."""
    lib = _load()
    x = _2d(x)
    rows, cols = x.shape
    gamma = _f64(gamma).reshape(cols)
    out, rms = np.empty_like(x), np.empty(rows)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_rms_norm_forward(_p(x[a:b]), _p(gamma), _p(out[a:b]), _p(rms[a:b]), b - a,
                                                  cols, eps))
    return out, rms


def rms_norm_backward(g, gamma, x, row_rms, n_threads=None):
    """Returns (dx, gamma_terms)."""
    lib = _load()
    g, x = _2d(g), _2d(x)
    rows, cols = g.shape
    gamma = _f64(gamma).reshape(cols)
    r = _f64(row_rms).reshape(rows)
    dx, gt = np.empty_like(g), np.empty_like(g)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_rms_norm_backward(_p(g[a:b]), _p(gamma), _p(x[a:b]), _p(r[a:b]), _p(dx[a:b]),
                                                   _p(gt[a:b]), b - a, cols))
    return dx, gt


def column_sums(m, out=None, beta: float = 0.0):
    """out_j = beta * out_j + sum_i m_ij (rows in increasing order, one thread)."""
    lib = _load()
    m = _2d(m)
    rows, cols = m.shape
    o = np.zeros(cols) if out is None else _f64(out).reshape(cols).copy()
    lib.oracle_column_sums(_p(m), _p(o), rows, cols, beta)
    return o


def lrp_softmax_rows(x, y, r, n_threads=None) -> np.ndarray:
    lib = _load()
    x, y, r = _2d(x), _2d(y), _2d(r)
    rows, cols = x.shape
    out = np.empty_like(x)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_lrp_softmax_rows(_p(x[a:b]), _p(y[a:b]), _p(r[a:b]), _p(out[a:b]), b - a, cols))
    return out


def masked_softmax_fmask(x, mask, n_threads=None) -> np.ndarray:
    lib = _load()
    x, m = _2d(x), _2d(mask)
    rows, cols = x.shape
    y = np.empty_like(x)
    _run(_row_blocks(rows, cols, n_threads),
         lambda a, b: lib.oracle_masked_softmax_fmask(_p(x[a:b]), _p(m[a:b]), _p(y[a:b]), b - a, cols))
    return y


def argmax_onehot(x, n_threads=None) -> np.ndarray:
    lib = _load()
    x = _2d(x)
    rows, cols = x.shape
    out = np.empty_like(x)
    _run(_row_blocks(rows, cols * cols, n_threads),
         lambda a, b: lib.oracle_argmax_onehot(_p(x[a:b]), _p(out[a:b]), b - a, cols))
    return out


def _two_input_ce(fn_name, a, b, grad_scale, n_threads):
    lib = _load()
    a, b = _2d(a), _2d(b)
    rows, cols = a.shape
    grad, loss = np.empty_like(a), np.empty(rows)
    fn = getattr(lib, fn_name)
    _run(_row_blocks(rows, cols, n_threads),
         lambda i0, i1: fn(_p(a[i0:i1]), _p(b[i0:i1]), _p(grad[i0:i1]), _p(loss[i0:i1]), i1 - i0, cols, grad_scale))
    mean_loss = lib.oracle_mean(_p(loss), rows) if rows else float("nan")
    return grad, loss, mean_loss


def soft_ce(logits, weights, grad_scale: float, n_threads=None):
    """Weighted-logits (soft-target) cross-entropy: returns (grad, row_loss, mean_loss)."""
    return _two_input_ce("oracle_soft_ce", logits, weights, grad_scale, n_threads)


def teacher_ce(student, teacher, grad_scale: float, n_threads=None):
    """Fixed-teacher cross-entropy: returns (student grad, row_loss, mean_loss)."""
    return _two_input_ce("oracle_teacher_ce", student, teacher, grad_scale, n_threads)
