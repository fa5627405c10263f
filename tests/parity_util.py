"""Helpers for the GPU-vs-oracle parity tests: device copies (aligned and
deliberately misaligned) and the acceptance bounds, one function per output
kind.  The bounds are the stated ones where given (probabilities 2e-6 max-abs,
logsumexp/loss 1e-5 relative, dgamma/dbeta 1e-4 of the column's L1 norm, kept
mask bit-exact); the others scale with the conditioning of the computation."""
from __future__ import annotations

import numpy as np
import torch

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def gpu(a: np.ndarray, misalign: bool = False) -> torch.Tensor:
    """Device copy of `a`; with misalign the data pointer is 4 bytes past a
    256-byte boundary, which forces the scalar path."""
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    if not misalign:
        return t.to(DEV)
    flat = torch.empty(t.numel() + 16, dtype=t.dtype, device=DEV)
    off = 4 // t.element_size() if t.element_size() <= 4 else 1
    view = flat[off:off + t.numel()].view(t.shape)
    view.copy_(t.to(DEV))
    assert view.data_ptr() % 16 != 0
    return view


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def _fail(what, mask, got, ref, bound):
    idx = np.argwhere(mask)[:5]
    msg = [f"{what}: {int(mask.sum())} entries out of bounds"]
    for i in idx:
        i = tuple(i)
        msg.append(f"  at {i}: got {got[i]!r} ref {ref[i]!r} bound {np.broadcast_to(bound, got.shape)[i]!r}")
    raise AssertionError("\n".join(msg))


def check_abs(got, ref, atol, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bad = ~(np.abs(got - ref) <= atol)
    bad &= ~(np.isnan(got) & np.isnan(ref))
    if bad.any():
        _fail(what, bad, got, ref, atol)


def check_bound(got, ref, bound, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = ~(np.abs(got - ref) <= bound)
    bad &= ~(np.isnan(got) & np.isnan(ref))
    bad &= ~((got == ref) & np.isinf(ref))
    if bad.any():
        _fail(what, bad, got, ref, bound)


def check_probs(got, ref, what):
    check_abs(got, ref, 2e-6, what)


def check_rel(got, ref, what, rtol=1e-5):
    ref = np.asarray(ref, dtype=np.float64)
    check_bound(got, ref, rtol * np.maximum(1.0, np.abs(ref)), what)


def check_exact_zero(got, where, what):
    got = np.asarray(got)
    z = got[where]
    if not ((z == 0.0).all() and not np.signbit(z).any()):
        raise AssertionError(f"{what}: masked entries are not all +0.0")


def softmax_bwd_bound(y, dy, scale=1.0):
    y = np.abs(np.asarray(y, np.float64))
    dy = np.abs(np.asarray(dy, np.float64))
    s = (y * dy).sum(axis=-1, keepdims=True)
    return 1e-5 * abs(scale) * y * (dy + s) + 1e-9


def ln_dx_bound(g, gamma, xhat, inv_std):
    gp = np.abs(np.asarray(g, np.float64) * gamma)
    xh = np.abs(np.asarray(xhat, np.float64))
    r = np.asarray(inv_std, np.float64).reshape(-1, 1)
    return 1e-5 * r * (gp + gp.mean(axis=1, keepdims=True) + xh * (gp * xh).mean(axis=1, keepdims=True)) + 1e-9


def param_bound(*factors):
    prod = np.abs(np.asarray(factors[0], np.float64))
    for f in factors[1:]:
        prod = prod * np.abs(np.asarray(f, np.float64))
    return 1e-4 * prod.sum(axis=0) + 1e-9
