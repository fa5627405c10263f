"""GPU parity on seeded random shapes: every op, row lengths drawn
log-uniformly from 1 to 70000 floats (20000 for the selection ops, whose
oracle compares every pair of a row's entries), so every kernel shape and the
borders between them come up, with buffers placed 0-3 floats past a 256-byte
boundary (each buffer on its own offset), against the oracle with the bounds
of the per-op tests."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_abs, check_bound, check_probs, check_rel, host, ln_dx_bound, param_bound, \
    softmax_bwd_bound
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = 12
MAX_ELEMS = 1 << 21


def _shapes(seed, max_cols=70000, max_pairs=None):
    """Random (rows, cols, rng); max_pairs bounds rows * cols^2 for ops whose
    oracle compares every pair of entries of a row."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(CASES):
        cols = int(np.exp(rng.uniform(0, np.log(max_cols))))
        rows = min(400, MAX_ELEMS // max(cols, 1))
        if max_pairs is not None:
            rows = min(rows, max_pairs // (cols * cols))
        rows = int(rng.integers(1, max(1, rows) + 1))
        out.append((rows, cols, rng))
    return out


def _dev(a, rng, dtype=None):
    """Device copy of `a` 0-3 elements past a 256-byte boundary."""
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype))
    t = torch.from_numpy(a)
    off = int(rng.integers(0, 4))
    flat = torch.zeros(t.numel() + 8, dtype=t.dtype, device="cuda")
    view = flat[off:off + t.numel()].view(t.shape)
    view.copy_(t.cuda())
    return view


def _empty(shape, rng, dtype=torch.float32):
    off = int(rng.integers(0, 4))
    n = int(np.prod(shape))
    return torch.zeros(n + 8, dtype=dtype, device="cuda")[off:off + n].view(shape)


@pytest.mark.parametrize("seed", range(3))
def test_random_softmax_lse_ce(ro, seed):
    for rows, cols, rng in _shapes(100 + seed):
        c = inputs.cross_entropy(int(rng.integers(1 << 30)), rows=rows, cols=cols, outlier_frac=1e-3)
        x, t = c["logits"], c["targets"]
        xg = _dev(x, rng)
        y = _empty(x.shape, rng)
        ro.rowops_softmax_fwd(xg, y)
        ref = oracle.softmax_rows(x)
        check_probs(host(y), ref, f"softmax {rows}x{cols}")
        dy = rng.normal(0, 1, x.shape).astype(np.float32)
        y32 = ref.astype(np.float32)
        dx = _empty(x.shape, rng)
        ro.rowops_softmax_bwd(_dev(y32, rng), _dev(dy, rng), dx)
        check_bound(host(dx), oracle.softmax_rows_backward(y32, dy), softmax_bwd_bound(y32, dy),
                    f"softmax bwd {rows}x{cols}")
        lse = _empty((rows,), rng)
        ro.rowops_logsumexp(xg, lse)
        check_rel(host(lse), oracle.logsumexp_rows(x), f"lse {rows}x{cols}")
        g, rl = _empty(x.shape, rng), _empty((rows,), rng)
        ml = torch.zeros(1, dtype=torch.float64, device="cuda")
        ro.rowops_softmax_ce(xg, _dev(t, rng), g, rl, ml, grad_scale=c["grad_scale"])
        gr, rlr, mlr = oracle.softmax_cross_entropy(x, t, c["grad_scale"])
        check_abs(host(g), gr, 2e-6 * c["grad_scale"], f"ce grad {rows}x{cols}")
        check_rel(host(rl), rlr, f"ce row loss {rows}x{cols}")
        check_rel(host(ml), [mlr], f"ce mean {rows}x{cols}")
    assert ro.library().rowops_pipeline_timeouts() == 0


@pytest.mark.parametrize("seed", range(3))
def test_random_norms(ro, seed):
    for rows, cols, rng in _shapes(200 + seed):
        n = inputs.layernorm(int(rng.integers(1 << 30)), rows=rows, cols=cols)
        x, gamma, beta, dy, eps = n["x"], n["gamma"], n["beta"], n["dy"], n["eps"]
        out, xh, rs = _empty(x.shape, rng), _empty(x.shape, rng), _empty((rows,), rng)
        ro.rowops_layernorm_fwd(_dev(x, rng), _dev(gamma, rng), _dev(beta, rng), out, xh, rs, eps=eps)
        o_r, xh_r, rs_r = oracle.layernorm_forward(x, gamma, beta, eps)
        check_rel(host(xh), xh_r, f"xhat {rows}x{cols}")
        check_rel(host(out), o_r, f"ln out {rows}x{cols}")
        check_bound(host(rs), rs_r, 1e-5 * np.abs(rs_r), f"inv_std {rows}x{cols}")
        xh32, rs32 = xh_r.astype(np.float32), rs_r.astype(np.float32)
        dx, dg, db = ro.rowops_layernorm_bwd(_dev(dy, rng), _dev(gamma, rng), _dev(xh32, rng), _dev(rs32, rng))
        dxr, dgr, dbr = oracle.layernorm_backward(dy, gamma, xh32, rs32)
        check_bound(host(dx), dxr, ln_dx_bound(dy, gamma, xh32, rs32), f"ln dx {rows}x{cols}")
        check_bound(host(dg), dgr, param_bound(dy, xh32), f"dgamma {rows}x{cols}")
        check_bound(host(db), dbr, param_bound(dy), f"dbeta {rows}x{cols}")
        o2, rr = ro.rowops_rmsnorm_fwd(_dev(x, rng), _dev(gamma, rng), eps=eps)
        o_r2, rr_r = oracle.rms_norm_forward(x, gamma, eps)
        check_rel(host(o2), o_r2, f"rms out {rows}x{cols}")
        check_bound(host(rr), rr_r, 1e-5 * np.abs(rr_r), f"rms {rows}x{cols}")


@pytest.mark.parametrize("seed", range(3))
def test_random_masked_and_selection(ro, seed):
    for rows, cols, rng in _shapes(300 + seed, max_cols=20000, max_pairs=1 << 29):
        r = inputs.router(int(rng.integers(1 << 30)), rows=rows, cols=cols, p_allow=0.8, blocked_row_frac=0.05)
        x, m = r["x"], r["mask"]
        p = _empty(x.shape, rng)
        ro.rowops_masked_softmax(_dev(x, rng), _dev(m, rng), p)
        check_probs(host(p), oracle.masked_softmax(x, m), f"masked {rows}x{cols}")
        k = int(rng.integers(1, min(cols, 40) + 1))
        kept = _empty(x.shape, rng)
        ro.rowops_topk_kept(_dev(x, rng), k, kept)
        assert np.array_equal(host(kept), oracle.topk_kept(x, k).astype(np.float32)), (rows, cols, k)
        largest = bool(rng.integers(0, 2))
        v, i = ro.rowops_top_k_rows(_dev(x, rng), k, largest)
        vr, ir = oracle.top_k_rows(x, k, largest)
        assert np.array_equal(host(i), ir.astype(np.float32)), (rows, cols, k, largest)
        assert np.array_equal(host(v), vr.astype(np.float32)), (rows, cols, k, largest)
        oh = _empty(x.shape, rng)
        ro.rowops_argmax_onehot(_dev(x, rng), oh)
        assert np.array_equal(host(oh), oracle.argmax_onehot(x).astype(np.float32)), (rows, cols)


@pytest.mark.parametrize("seed", range(2))
def test_random_attention(ro, seed):
    rng = np.random.default_rng(400 + seed)
    for _ in range(6):
        seq = int(np.exp(rng.uniform(0, np.log(2896))))  # seq^2 <= 4 * MAX_ELEMS
        heads = int(max(1, min(3, MAX_ELEMS // (seq * seq))))
        a = inputs.attention(int(rng.integers(1 << 30)), batch=1, heads=heads, seq=seq)
        s, dp, scale = a["scores"], a["dp"], a["scale"]
        upper = np.arange(seq)[None, :] > (np.arange(s.shape[0]) % seq)[:, None]
        p = _empty(s.shape, rng)
        ro.rowops_attn_softmax_fwd(_dev(s, rng), p, seq_len=seq, scale=scale)
        ref = oracle.attn_softmax_forward(s, seq, scale)
        check_probs(host(p), ref, f"attn fwd seq={seq}")
        p32 = ref.astype(np.float32)
        ds = _empty(s.shape, rng)
        ro.rowops_attn_softmax_bwd(_dev(p32, rng), _dev(dp, rng), ds, seq_len=seq, scale=scale)
        dref = oracle.attn_softmax_backward(p32, dp, seq, scale)
        check_bound(host(ds), dref, softmax_bwd_bound(p32, np.where(upper, 0, dp), scale), f"attn bwd seq={seq}")
