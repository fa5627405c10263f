"""Python binding of librowops (include/rowops.h): argument marshalling only.

Every function has the name of its C entry point, takes torch CUDA tensors
(fp32, contiguous, last dimension = cols, rows = numel / cols), allocates the
outputs the caller leaves as ``None`` with torch, passes raw device pointers
and the current torch stream to the C ABI and raises ``RowopsError`` on a
nonzero status.  All arithmetic happens in the library's CUDA kernels; there
is no other code path.  The library is loaded on first use and a missing build
is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librowops.so")

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float

SIGNATURES = {
    "rowops_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "rowops_kernel_launches": ([], ctypes.c_uint64),
    "rowops_pipeline_timeouts": ([], ctypes.c_uint32),
    "rowops_softmax_fwd": ([_P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_softmax_bwd": ([_P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_attn_softmax_fwd": ([_P, _P, _I64, _I64, _I64, _F, _P], ctypes.c_int),
    "rowops_attn_softmax_bwd": ([_P, _P, _P, _I64, _I64, _I64, _F, _P], ctypes.c_int),
    "rowops_masked_softmax": ([_P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_logsumexp": ([_P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_softmax_ce": ([_P, _P, _P, _P, _P, _I64, _I64, _F, _P], ctypes.c_int),
    "rowops_layernorm_fwd": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P], ctypes.c_int),
    "rowops_layernorm_bwd_workspace": ([_I64, _I64], ctypes.c_size_t),
    "rowops_layernorm_bwd": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, ctypes.c_size_t, _P],
                             ctypes.c_int),
    "rowops_topk_kept": ([_P, _P, _I64, _I64, _I64, _P], ctypes.c_int),
    "rowops_router_masked_topk": ([_P, _P, _P, _P, _I64, _I64, _I64, _P], ctypes.c_int),
    "rowops_top_k_rows": ([_P, _P, _P, _I64, _I64, _I64, ctypes.c_int, _P], ctypes.c_int),
    "rowops_rmsnorm_fwd": ([_P, _P, _P, _P, _I64, _I64, _F, _P], ctypes.c_int),
    "rowops_rmsnorm_bwd": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_column_sums": ([_P, _P, _I64, _I64, _F, _P], ctypes.c_int),
    "rowops_masked_softmax_fmask": ([_P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_lrp_softmax_rows": ([_P, _P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_argmax_onehot": ([_P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_soft_ce": ([_P, _P, _P, _P, _P, _I64, _I64, _F, _P], ctypes.c_int),
    "rowops_teacher_ce": ([_P, _P, _P, _P, _P, _I64, _I64, _F, _P], ctypes.c_int),
    "rowops_layernorm_bwd_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "rowops_layernorm_bwd_noalloc_max_bytes": ([], ctypes.c_size_t),
}


class RowopsError(RuntimeError):
    """A rowops_* entry point returned a nonzero status."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def library():
    """The loaded librowops (ctypes.CDLL) with its C signatures declared."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with row_wise_softmax_warp_gb300.build.build() "
                "(or __graft_entry__.build()); there is no fallback implementation")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _check(status: int):
    if status != 0:
        raise RowopsError(status, library().rowops_status_string(status).decode())


def _stream(t: torch.Tensor, stream):
    if stream is None:
        return torch.cuda.current_stream(t.device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _mat(t: torch.Tensor, name: str, dtype=torch.float32):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _shape(t: torch.Tensor):
    if t.dim() == 0:
        return 1, 1
    cols = int(t.shape[-1])
    return math.prod(t.shape[:-1]), cols


def _out(t, like: torch.Tensor, name: str, shape=None, dtype=torch.float32):
    if t is None:
        return torch.empty(like.shape if shape is None else shape, dtype=dtype, device=like.device)
    return _mat(t, name, dtype)


def rowops_kernel_launches() -> int:
    return int(library().rowops_kernel_launches())


def rowops_softmax_fwd(x, y=None, stream=None):
    """y = softmax(x) along the last dimension (y may be x)."""
    x = _mat(x, "x")
    y = _out(y, x, "y")
    rows, cols = _shape(x)
    _check(library().rowops_softmax_fwd(x.data_ptr(), y.data_ptr(), rows, cols, _stream(x, stream)))
    return y


def rowops_softmax_bwd(y, dy, dx=None, stream=None):
    """dx = y * (dy - sum(y * dy)) along the last dimension."""
    y, dy = _mat(y, "y"), _mat(dy, "dy")
    dx = _out(dx, y, "dx")
    rows, cols = _shape(y)
    _check(library().rowops_softmax_bwd(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), rows, cols,
                                        _stream(y, stream)))
    return dx


def rowops_attn_softmax_fwd(scores, p=None, seq_len=None, scale=1.0, stream=None):
    """Scaled causal softmax of stacked (batch*heads*seq_len, seq_len) score rows."""
    scores = _mat(scores, "scores")
    p = _out(p, scores, "p")
    rows, cols = _shape(scores)
    seq_len = cols if seq_len is None else seq_len
    _check(library().rowops_attn_softmax_fwd(scores.data_ptr(), p.data_ptr(), rows, cols, seq_len,
                                             scale, _stream(scores, stream)))
    return p


def rowops_attn_softmax_bwd(p, dp, ds=None, seq_len=None, scale=1.0, stream=None):
    """Gradient of rowops_attn_softmax_fwd with respect to the raw scores, from p."""
    p, dp = _mat(p, "p"), _mat(dp, "dp")
    ds = _out(ds, p, "ds")
    rows, cols = _shape(p)
    seq_len = cols if seq_len is None else seq_len
    _check(library().rowops_attn_softmax_bwd(p.data_ptr(), dp.data_ptr(), ds.data_ptr(), rows, cols,
                                             seq_len, scale, _stream(p, stream)))
    return ds


def rowops_masked_softmax(x, mask, y=None, stream=None):
    """Softmax over entries with mask != 0; blocked entries and empty rows are +0."""
    x = _mat(x, "x")
    mask = _mat(mask, "mask", torch.uint8)
    y = _out(y, x, "y")
    rows, cols = _shape(x)
    _check(library().rowops_masked_softmax(x.data_ptr(), mask.data_ptr(), y.data_ptr(), rows, cols,
                                           _stream(x, stream)))
    return y


def rowops_logsumexp(x, lse=None, stream=None):
    """lse = log(sum(exp(x))) along the last dimension."""
    x = _mat(x, "x")
    rows, cols = _shape(x)
    lse = _out(lse, x, "lse", shape=x.shape[:-1])
    _check(library().rowops_logsumexp(x.data_ptr(), lse.data_ptr(), rows, cols, _stream(x, stream)))
    return lse


def rowops_softmax_ce(logits, targets, grad=None, row_loss=None, mean_loss=None, grad_scale=None,
                      stream=None):
    """Returns (grad, row_loss, mean_loss); mean_loss is a one-element float64 CUDA tensor."""
    logits = _mat(logits, "logits")
    targets = _mat(targets, "targets", torch.int32)
    rows, cols = _shape(logits)
    grad = _out(grad, logits, "grad")
    row_loss = _out(row_loss, logits, "row_loss", shape=(rows,))
    mean_loss = _out(mean_loss, logits, "mean_loss", shape=(1,), dtype=torch.float64)
    if grad_scale is None:
        grad_scale = 1.0 / rows if rows else 1.0
    _check(library().rowops_softmax_ce(logits.data_ptr(), targets.data_ptr(), grad.data_ptr(),
                                       row_loss.data_ptr(), mean_loss.data_ptr(), rows, cols,
                                       grad_scale, _stream(logits, stream)))
    return grad, row_loss, mean_loss


def rowops_layernorm_fwd(x, gamma, beta, out=None, xhat=None, inv_std=None, eps=1e-5, stream=None):
    """Returns (out, xhat, inv_std)."""
    x, gamma, beta = _mat(x, "x"), _mat(gamma, "gamma"), _mat(beta, "beta")
    rows, cols = _shape(x)
    out = _out(out, x, "out")
    xhat = _out(xhat, x, "xhat")
    inv_std = _out(inv_std, x, "inv_std", shape=(rows,))
    _check(library().rowops_layernorm_fwd(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(),
                                          out.data_ptr(), xhat.data_ptr(), inv_std.data_ptr(), rows,
                                          cols, eps, _stream(x, stream)))
    return out, xhat, inv_std


def rowops_layernorm_bwd_workspace(rows: int, cols: int) -> int:
    return int(library().rowops_layernorm_bwd_workspace(rows, cols))


def rowops_layernorm_bwd(dy, gamma, xhat, inv_std, dx=None, dgamma=None, dbeta=None, workspace=None,
                         stream=None):
    """Returns (dx, dgamma, dbeta)."""
    dy, gamma, xhat = _mat(dy, "dy"), _mat(gamma, "gamma"), _mat(xhat, "xhat")
    inv_std = _mat(inv_std, "inv_std")
    rows, cols = _shape(dy)
    dx = _out(dx, dy, "dx")
    dgamma = _out(dgamma, dy, "dgamma", shape=(cols,))
    dbeta = _out(dbeta, dy, "dbeta", shape=(cols,))
    need = rowops_layernorm_bwd_workspace(rows, cols)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dy.device)
    _check(library().rowops_layernorm_bwd(dy.data_ptr(), gamma.data_ptr(), xhat.data_ptr(),
                                          inv_std.data_ptr(), dx.data_ptr(), dgamma.data_ptr(),
                                          dbeta.data_ptr(), rows, cols, workspace.data_ptr(),
                                          workspace.numel() * workspace.element_size(),
                                          _stream(dy, stream)))
    return dx, dgamma, dbeta


def rowops_topk_kept(x, k, kept=None, stream=None):
    """1.0 where fewer than k entries of the row beat the entry, else 0.0."""
    x = _mat(x, "x")
    kept = _out(kept, x, "kept")
    rows, cols = _shape(x)
    _check(library().rowops_topk_kept(x.data_ptr(), kept.data_ptr(), rows, cols, k,
                                      _stream(x, stream)))
    return kept


def rowops_router_masked_topk(x, mask, k, p=None, kept=None, stream=None):
    """Fused router: returns (p, kept) = (masked softmax of x, top-k kept mask of p)."""
    x = _mat(x, "x")
    mask = _mat(mask, "mask", torch.uint8)
    p = _out(p, x, "p")
    kept = _out(kept, x, "kept")
    rows, cols = _shape(x)
    _check(library().rowops_router_masked_topk(x.data_ptr(), mask.data_ptr(), p.data_ptr(), kept.data_ptr(),
                                               rows, cols, k, _stream(x, stream)))
    return p, kept


def rowops_top_k_rows(x, k, largest=True, values=None, indices=None, stream=None):
    """Returns (values, indices), each (rows, k): the k largest (or smallest) entries
    of every row in rank order (NaN above every number; ties by lower column)."""
    x = _mat(x, "x")
    rows, cols = _shape(x)
    values = _out(values, x, "values", shape=(*x.shape[:-1], k))
    indices = _out(indices, x, "indices", shape=(*x.shape[:-1], k))
    _check(library().rowops_top_k_rows(x.data_ptr(), values.data_ptr(), indices.data_ptr(), rows, cols, k,
                                       1 if largest else 0, _stream(x, stream)))
    return values, indices


def rowops_rmsnorm_fwd(x, gamma, out=None, row_rms=None, eps=1e-5, stream=None):
    """Returns (out, row_rms)."""
    x, gamma = _mat(x, "x"), _mat(gamma, "gamma")
    rows, cols = _shape(x)
    out = _out(out, x, "out")
    row_rms = _out(row_rms, x, "row_rms", shape=(rows,))
    _check(library().rowops_rmsnorm_fwd(x.data_ptr(), gamma.data_ptr(), out.data_ptr(), row_rms.data_ptr(),
                                        rows, cols, eps, _stream(x, stream)))
    return out, row_rms


def rowops_rmsnorm_bwd(dy, gamma, x, row_rms, dx=None, gamma_terms=None, stream=None):
    """Returns (dx, gamma_terms); gamma's gradient is rowops_column_sums(gamma_terms)."""
    dy, gamma, x, row_rms = _mat(dy, "dy"), _mat(gamma, "gamma"), _mat(x, "x"), _mat(row_rms, "row_rms")
    rows, cols = _shape(dy)
    dx = _out(dx, dy, "dx")
    gamma_terms = _out(gamma_terms, dy, "gamma_terms")
    _check(library().rowops_rmsnorm_bwd(dy.data_ptr(), gamma.data_ptr(), x.data_ptr(), row_rms.data_ptr(),
                                        dx.data_ptr(), gamma_terms.data_ptr(), rows, cols, _stream(dy, stream)))
    return dx, gamma_terms


def rowops_column_sums(m, out=None, beta=0.0, stream=None):
    """out_j = beta * out_j + sum_i m_ij (deterministic order)."""
    m = _mat(m, "in")
    rows, cols = _shape(m)
    if out is None:
        out = torch.zeros(cols, dtype=torch.float32, device=m.device)
    out = _mat(out, "out")
    _check(library().rowops_column_sums(m.data_ptr(), out.data_ptr(), rows, cols, beta, _stream(m, stream)))
    return out


def rowops_masked_softmax_fmask(x, mask, y=None, stream=None):
    """Masked softmax with an fp32 mask (allowed where mask != 0)."""
    x, mask = _mat(x, "x"), _mat(mask, "mask")
    y = _out(y, x, "y")
    rows, cols = _shape(x)
    _check(library().rowops_masked_softmax_fmask(x.data_ptr(), mask.data_ptr(), y.data_ptr(), rows, cols,
                                                 _stream(x, stream)))
    return y


def rowops_lrp_softmax_rows(x, y, r, r_in=None, stream=None):
    """r_in = x * (r - y * sum(r)) per row."""
    x, y, r = _mat(x, "x"), _mat(y, "y"), _mat(r, "r")
    r_in = _out(r_in, x, "r_in")
    rows, cols = _shape(x)
    _check(library().rowops_lrp_softmax_rows(x.data_ptr(), y.data_ptr(), r.data_ptr(), r_in.data_ptr(), rows,
                                             cols, _stream(x, stream)))
    return r_in


def rowops_argmax_onehot(x, out=None, stream=None):
    """1.0 at the first maximal coordinate of each row, 0.0 elsewhere."""
    x = _mat(x, "x")
    out = _out(out, x, "out")
    rows, cols = _shape(x)
    _check(library().rowops_argmax_onehot(x.data_ptr(), out.data_ptr(), rows, cols, _stream(x, stream)))
    return out


def _ce2(fn, x, w, grad, row_loss, mean_loss, grad_scale, stream, want_grad=True):
    x, w = _mat(x, "logits"), _mat(w, "weights")
    rows, cols = _shape(x)
    if want_grad:
        grad = _out(grad, x, "grad")
    row_loss = _out(row_loss, x, "row_loss", shape=(rows,))
    mean_loss = _out(mean_loss, x, "mean_loss", shape=(1,), dtype=torch.float64)
    if grad_scale is None:
        grad_scale = 1.0 / rows if rows else 1.0
    _check(fn(x.data_ptr(), w.data_ptr(), grad.data_ptr() if grad is not None else None, row_loss.data_ptr(),
              mean_loss.data_ptr(), rows, cols, grad_scale, _stream(x, stream)))
    return grad, row_loss, mean_loss


def rowops_soft_ce(logits, weights, grad=None, row_loss=None, mean_loss=None, grad_scale=None, stream=None):
    """Weighted-logits (soft-target) CE: returns (grad, row_loss, mean_loss)."""
    return _ce2(library().rowops_soft_ce, logits, weights, grad, row_loss, mean_loss, grad_scale, stream)


def rowops_teacher_ce(student, teacher, grad=None, row_loss=None, mean_loss=None, grad_scale=None,
                      with_grad=True, stream=None):
    """Fixed-teacher CE: returns (student grad or None, row_loss, mean_loss)."""
    return _ce2(library().rowops_teacher_ce, student, teacher, grad, row_loss, mean_loss, grad_scale, stream,
                want_grad=with_grad)


def rowops_layernorm_bwd_noalloc(dy, gamma, xhat, inv_std, dx=None, dgamma=None, dbeta=None, stream=None):
    """rowops_layernorm_bwd without a workspace argument: the library's own
    fixed device array serves as workspace (calls on one device must not
    overlap on the GPU).  Returns (dx, dgamma, dbeta)."""
    dy, gamma, xhat = _mat(dy, "dy"), _mat(gamma, "gamma"), _mat(xhat, "xhat")
    inv_std = _mat(inv_std, "inv_std")
    rows, cols = _shape(dy)
    dx = _out(dx, dy, "dx")
    dgamma = _out(dgamma, dy, "dgamma", shape=(cols,))
    dbeta = _out(dbeta, dy, "dbeta", shape=(cols,))
    _check(library().rowops_layernorm_bwd_noalloc(dy.data_ptr(), gamma.data_ptr(), xhat.data_ptr(),
                                                  inv_std.data_ptr(), dx.data_ptr(), dgamma.data_ptr(),
                                                  dbeta.data_ptr(), rows, cols, _stream(dy, stream)))
    return dx, dgamma, dbeta
