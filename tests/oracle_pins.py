"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each pin is a plain function that raises AssertionError on failure.  They use
closed forms, invariants, finite differences, brute force, hand-worked cases
from the pages (tests/golden) and textbook library routines (torch float64 on
the CPU), never the oracle's own formula retyped.  ``test_oracle_pins.py`` runs
them against the oracle; ``test_oracle_mutants.py`` runs them against copies of
the oracle with planted mistakes and expects each copy to fail at least one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f(vals):
    return np.array([float(v) for v in vals], dtype=np.float64)


def _close(a, b, rtol, atol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    ok = np.isclose(a, b, rtol=rtol, atol=atol) | (np.isnan(a) & np.isnan(b))
    assert ok.all(), f"{what}: max |diff| {np.nanmax(np.abs(a - b))}"


# ----------------------------------------------------------------- softmax rows

def pin_softmax_golden():
    for c in _golden("row_op_examples.json")["softmax_rows"]["cases"]:
        y = oracle.softmax_rows(_f(c["x"])[None])
        _close(y[0], _f(c["y"]), 1e-15, 1e-15, c["why"])


def pin_softmax_rows_sum_to_one():
    x = _rng(1).normal(0, 2, (64, 129))
    y = oracle.softmax_rows(x)
    _close(y.sum(axis=1), np.ones(64), 0, 1e-14, "row sums")
    assert (y > 0).all() and (y <= 1).all()


def pin_softmax_two_columns_is_logistic():
    # softmax([a, b])_0 = 1 / (1 + exp(b - a)), the logistic function.
    ab = _rng(2).normal(0, 3, (50, 2))
    y = oracle.softmax_rows(ab)
    _close(y[:, 0], 1.0 / (1.0 + np.exp(ab[:, 1] - ab[:, 0])), 1e-14, 1e-16, "logistic")


def pin_softmax_ratios_and_shift():
    x = _rng(3).normal(0, 2, (8, 33))
    y = oracle.softmax_rows(x)
    # y_j / y_0 = exp(x_j - x_0)
    _close(y / y[:, :1], np.exp(x - x[:, :1]), 1e-13, 0, "ratios")
    _close(oracle.softmax_rows(x + 3.25), y, 1e-14, 1e-16, "shift invariance")


def pin_softmax_matches_torch():
    x = _rng(4).normal(0, 2, (16, 200))
    _close(oracle.softmax_rows(x), torch.softmax(torch.from_numpy(x), dim=1).numpy(), 1e-13,
           1e-17, "torch.softmax float64")


# -------------------------------------------------------- softmax rows backward

def pin_softmax_backward_golden():
    for c in _golden("row_op_examples.json")["softmax_rows_backward"]["cases"]:
        dx = oracle.softmax_rows_backward(_f(c["y"])[None], _f(c["dy"])[None])
        _close(dx[0], _f(c["dx"]), 0, 1e-15, c["why"])


def pin_softmax_backward_finite_differences():
    # dx must be the gradient of x -> <dy, softmax(x)>, by central differences.
    rng = _rng(5)
    x = rng.normal(0, 1, (3, 5))
    dy = rng.normal(0, 1, (3, 5))
    y = oracle.softmax_rows(x)
    dx = oracle.softmax_rows_backward(y, dy)
    h = 1e-6
    fd = np.zeros_like(x)
    for i in range(3):
        for j in range(5):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd[i, j] = (np.sum(dy * oracle.softmax_rows(xp)) - np.sum(dy * oracle.softmax_rows(xm))) / (2 * h)
    _close(dx, fd, 1e-7, 1e-9, "finite differences")


def pin_softmax_backward_invariants():
    rng = _rng(6)
    y = oracle.softmax_rows(rng.normal(0, 2, (20, 77)))
    dy = rng.normal(0, 1, (20, 77))
    dx = oracle.softmax_rows_backward(y, dy)
    _close(dx.sum(axis=1), np.zeros(20), 0, 1e-14, "rows of dx sum to 0")
    _close(oracle.softmax_rows_backward(y, np.full_like(y, 2.5)), np.zeros_like(y), 0, 1e-14,
           "constant dy")


def pin_softmax_backward_matches_torch_autograd():
    rng = _rng(7)
    x = torch.from_numpy(rng.normal(0, 2, (6, 40))).requires_grad_(True)
    dy = torch.from_numpy(rng.normal(0, 1, (6, 40)))
    y = torch.softmax(x, dim=1)
    (gx,) = torch.autograd.grad(y, x, dy)
    _close(oracle.softmax_rows_backward(y.detach().numpy(), dy.numpy()), gx.numpy(), 1e-10, 1e-15,
           "torch autograd")


# ------------------------------------------------------ causal attention softmax

def _torch_causal(s, seq_len, scale, row0=0):
    rows, cols = s.shape
    q = (np.arange(rows) + row0) % seq_len
    z = scale * torch.from_numpy(s)
    allowed = torch.from_numpy(np.arange(cols)[None, :] <= q[:, None])
    return torch.softmax(z.masked_fill(~allowed, float("-inf")), dim=1).numpy()


def pin_attn_golden():
    for c in _golden("row_op_examples.json")["attn_softmax_forward"]["cases"]:
        s = np.array([[float(v) for v in r] for r in c["scores"]])
        p = oracle.attn_softmax_forward(s, c["seq_len"], float(c["scale"]))
        if "p" in c:
            _close(p, np.array([[float(v) for v in r] for r in c["p"]]), 1e-15, 1e-16, c["why"])
        else:
            _close(p[0], _f(c["p_first_two_rows"][0]), 0, 0, c["why"])


def pin_attn_structure():
    rng = _rng(8)
    S = 37
    s = rng.normal(0, 8, (3 * S, S))
    p = oracle.attn_softmax_forward(s, S, 0.125)
    q = np.arange(3 * S) % S
    upper = np.arange(S)[None, :] > q[:, None]
    assert (p[upper] == 0.0).all() and not np.signbit(p[upper]).any(), "upper triangle exactly +0"
    _close(p.sum(axis=1), np.ones(3 * S), 0, 1e-14, "row sums")
    assert (p[q == 0, 0] == 1.0).all(), "query 0 attends only to key 0"
    # equal scores: 1/(i+1) on the visible keys
    pe = oracle.attn_softmax_forward(np.full((S, S), 1.5), S, 0.3)
    _close(pe, np.where(~upper[:S], 1.0 / (np.arange(S)[:, None] + 1.0), 0.0), 1e-14, 1e-16, "equal")


def pin_attn_last_query_is_plain_softmax():
    # With scale 1 the last query row of each head masks nothing: plain softmax.
    rng = _rng(9)
    S = 16
    s = rng.normal(0, 8, (2 * S, S))
    p = oracle.attn_softmax_forward(s, S, 1.0)
    y = oracle.softmax_rows(s[[S - 1, 2 * S - 1]])
    assert np.array_equal(p[[S - 1, 2 * S - 1]], y)


def pin_attn_matches_torch_and_scale_enters_before_exp():
    rng = _rng(10)
    S = 24
    s = rng.normal(0, 8, (4 * S, S))
    _close(oracle.attn_softmax_forward(s, S, 0.125), _torch_causal(s, S, 0.125), 1e-12, 1e-17,
           "torch masked softmax")
    # scale is applied to the scores: attn(s, c) == attn(c*s, 1)
    _close(oracle.attn_softmax_forward(s, S, 0.125), oracle.attn_softmax_forward(0.125 * s, S, 1.0),
           1e-13, 1e-17, "scale")


def pin_attn_row_offset():
    rng = _rng(11)
    S = 10
    s = rng.normal(0, 8, (5 * S, S))
    full = oracle.attn_softmax_forward(s, S, 0.2)
    part = oracle.attn_softmax_forward(s[13:31], S, 0.2, row0=13)
    assert np.array_equal(full[13:31], part)
    dp = rng.normal(0, 1, s.shape)
    fb = oracle.attn_softmax_backward(full, dp, S, 0.2)
    pb = oracle.attn_softmax_backward(full[13:31], dp[13:31], S, 0.2, row0=13)
    assert np.array_equal(fb[13:31], pb)


def pin_attn_backward_finite_differences():
    rng = _rng(12)
    S, scale = 4, 0.7
    s = rng.normal(0, 2, (2 * S, S))
    dp = rng.normal(0, 1, s.shape)
    p = oracle.attn_softmax_forward(s, S, scale)
    ds = oracle.attn_softmax_backward(p, dp, S, scale)
    h = 1e-6
    fd = np.zeros_like(s)
    for i in range(s.shape[0]):
        for j in range(S):
            sp, sm = s.copy(), s.copy()
            sp[i, j] += h
            sm[i, j] -= h
            fd[i, j] = (np.sum(dp * oracle.attn_softmax_forward(sp, S, scale))
                        - np.sum(dp * oracle.attn_softmax_forward(sm, S, scale))) / (2 * h)
    _close(ds, fd, 1e-7, 1e-9, "finite differences")
    q = np.arange(2 * S) % S
    assert (ds[np.arange(S)[None, :] > q[:, None]] == 0.0).all()


def pin_attn_backward_matches_torch_autograd():
    rng = _rng(13)
    S, scale = 12, 0.125
    s = torch.from_numpy(rng.normal(0, 8, (3 * S, S))).requires_grad_(True)
    dp = torch.from_numpy(rng.normal(0, 1, (3 * S, S)))
    q = torch.arange(3 * S) % S
    allowed = torch.arange(S)[None, :] <= q[:, None]
    p = torch.softmax((scale * s).masked_fill(~allowed, float("-inf")), dim=1)
    (gs,) = torch.autograd.grad(p, s, dp)
    _close(oracle.attn_softmax_backward(p.detach().numpy(), dp.numpy(), S, scale), gs.numpy(),
           1e-10, 1e-15, "torch autograd")


# ------------------------------------------------------------------ logsumexp

def pin_logsumexp_golden():
    for c in _golden("row_op_examples.json")["logsumexp_rows"]["cases"]:
        _close(oracle.logsumexp_rows(_f(c["x"])[None]), [float(c["lse"])], 1e-15, 0, c["why"])


def pin_logsumexp_closed_forms():
    rng = _rng(14)
    x = rng.normal(0, 2, (10, 300))
    lse = oracle.logsumexp_rows(x)
    _close(oracle.logsumexp_rows(x + 5.5), lse + 5.5, 1e-15, 0, "shift")
    assert (lse >= x.max(axis=1)).all() and (lse <= x.max(axis=1) + math.log(300)).all()
    c = np.full((3, 7), -2.25)
    _close(oracle.logsumexp_rows(c), np.full(3, -2.25 + math.log(7)), 1e-15, 0, "constant row")
    # one +30 outlier over small entries: 30 + log1p(sum exp(x - 30))
    row = rng.normal(0, 2, 500)
    row[17] = 30.0
    expect = 30.0 + math.log1p(math.fsum(np.exp(np.delete(row, 17) - 30.0)))
    _close(oracle.logsumexp_rows(row[None]), [expect], 1e-15, 0, "outlier")
    assert oracle.logsumexp_rows(np.zeros((2, 0)))[0] == -math.inf


def pin_logsumexp_matches_torch():
    x = _rng(15).normal(0, 2, (12, 1000))
    _close(oracle.logsumexp_rows(x), torch.logsumexp(torch.from_numpy(x), dim=1).numpy(), 1e-14, 0,
           "torch.logsumexp float64")


# ------------------------------------------------------- softmax cross-entropy

def pin_ce_golden():
    c = _golden("row_op_examples.json")["softmax_cross_entropy"]["cases"][0]
    g, loss, mean = oracle.softmax_cross_entropy(_f(c["logits"])[None], [c["target"]],
                                                 float(c["grad_scale"]))
    _close(loss, [float(c["loss"])], 1e-15, 0, "loss")
    _close(g[0], _f(c["grad"]), 0, 1e-15, "grad")
    _close([mean], [float(c["loss"])], 1e-15, 0, "mean")


def pin_ce_matches_torch():
    rng = _rng(16)
    R, C = 9, 300
    x = rng.normal(0, 2, (R, C))
    x[rng.integers(0, R, 5), rng.integers(0, C, 5)] = 30.0
    t = rng.integers(0, C, R).astype(np.int32)
    g, loss, mean = oracle.softmax_cross_entropy(x, t, 1.0 / R)
    xt = torch.from_numpy(x).requires_grad_(True)
    tl = torch.nn.functional.cross_entropy(xt, torch.from_numpy(t).long(), reduction="none")
    _close(loss, tl.detach().numpy(), 1e-13, 1e-15, "per-row loss")
    lm = tl.mean()
    (gx,) = torch.autograd.grad(lm, xt)
    _close([mean], [lm.item()], 1e-14, 0, "mean loss")
    _close(g, gx.numpy(), 1e-12, 1e-18, "gradient of the mean loss")


def pin_ce_identities():
    rng = _rng(17)
    R, C = 6, 50
    x = rng.normal(0, 2, (R, C))
    t = rng.integers(0, C, R).astype(np.int32)
    g, loss, mean = oracle.softmax_cross_entropy(x, t, 0.5)
    _close(loss, oracle.logsumexp_rows(x) - x[np.arange(R), t], 1e-14, 1e-15, "lse - x_t")
    _close(g.sum(axis=1), np.zeros(R), 0, 1e-15, "gradient rows sum to 0")
    onehot = np.zeros((R, C))
    onehot[np.arange(R), t] = 1
    _close(g, 0.5 * (oracle.softmax_rows(x) - onehot), 1e-14, 1e-17, "scale * (p - onehot)")
    _close([mean], [math.fsum(loss) / R], 1e-15, 0, "mean")
    # uniform logits: loss = ln C
    g2, l2, _ = oracle.softmax_cross_entropy(np.full((2, 8), 1.75), np.array([0, 7], np.int32), 1.0)
    _close(l2, [math.log(8)] * 2, 1e-15, 0, "uniform loss")
    _close(g2[1], np.r_[np.full(7, 1 / 8), [1 / 8 - 1]], 0, 1e-16, "uniform grad")


def pin_ce_finite_differences():
    rng = _rng(18)
    R, C = 3, 7
    x = rng.normal(0, 1, (R, C))
    t = rng.integers(0, C, R).astype(np.int32)
    g, _, _ = oracle.softmax_cross_entropy(x, t, 1.0 / R)
    h = 1e-6
    fd = np.zeros_like(x)
    for i in range(R):
        for j in range(C):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd[i, j] = (oracle.softmax_cross_entropy(xp, t, 1.0)[2]
                        - oracle.softmax_cross_entropy(xm, t, 1.0)[2]) / (2 * h)
    _close(g, fd, 1e-7, 1e-10, "finite differences of the mean loss")


def pin_ce_out_of_range_target():
    x = _rng(19).normal(0, 1, (3, 5))
    g, loss, mean = oracle.softmax_cross_entropy(x, np.array([1, 5, -1], np.int32), 1.0)
    assert not np.isnan(loss[0]) and np.isnan(loss[1]) and np.isnan(loss[2]) and np.isnan(mean)
    _close(g[1:], torch.softmax(torch.from_numpy(x[1:]), dim=1).numpy(), 1e-14, 0, "no one-hot term")


# ------------------------------------------------------------------ layernorm

def _ln_case(seed, R=8, C=48):
    rng = _rng(seed)
    x = rng.normal(0, 1, (R, C)) * rng.uniform(0.1, 10, (R, 1)) + rng.uniform(-5, 5, (R, 1))
    gamma = 1 + 0.1 * rng.normal(0, 1, C)
    beta = 0.1 * rng.normal(0, 1, C)
    g = rng.normal(0, 1, (R, C))
    return x, gamma, beta, g


def pin_layernorm_golden():
    c = _golden("row_op_examples.json")["layernorm_forward"]["cases"][0]
    out, xhat, r = oracle.layernorm_forward(_f(c["x"])[None], _f(c["gamma"]), _f(c["beta"]),
                                            float(c["eps"]))
    _close(xhat[0], _f(c["xhat"]), 1e-15, 0, "xhat")
    _close(out[0], _f(c["out"]), 1e-15, 0, "out")
    _close(r, [float(c["inv_std"])], 1e-15, 0, "inv_std")


def pin_layernorm_forward_invariants():
    x, gamma, beta, _ = _ln_case(20)
    for eps in (1e-5, 0.5):
        out, xhat, r = oracle.layernorm_forward(x, gamma, beta, eps)
        v = np.var(x, axis=1)  # population variance (numpy's default ddof=0)
        _close(xhat.mean(axis=1), np.zeros(len(x)), 0, 1e-14, "mean(xhat) = 0")
        _close(np.mean(xhat ** 2, axis=1), v / (v + eps), 1e-12, 0, "var(xhat) = v/(v+eps)")
        _close(r * r * (v + eps), np.ones(len(x)), 1e-13, 0, "inv_std^2 (v+eps) = 1")
        _close(out, gamma * xhat + beta, 1e-14, 1e-15, "affine")
    # with eps = 0 the normalisation forgets shift and positive scale
    _, h1, _ = oracle.layernorm_forward(x, gamma, beta, 0.0)
    _, h2, _ = oracle.layernorm_forward(3.0 * x - 7.0, gamma, beta, 0.0)
    _close(h1, h2, 1e-12, 1e-13, "affine invariance")


def pin_layernorm_forward_matches_torch():
    x, gamma, beta, _ = _ln_case(21)
    for eps in (1e-5, 0.5):
        ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (x.shape[1],), torch.from_numpy(gamma),
                                             torch.from_numpy(beta), eps).numpy()
        _close(oracle.layernorm_forward(x, gamma, beta, eps)[0], ref, 1e-12, 1e-13, "torch layer_norm")


def pin_layernorm_backward_finite_differences():
    x, gamma, beta, g = _ln_case(22, R=3, C=6)
    eps = 1e-3
    out, xhat, r = oracle.layernorm_forward(x, gamma, beta, eps)
    dx, dgamma, dbeta = oracle.layernorm_backward(g, gamma, xhat, r)
    h = 1e-6

    def loss(xx, gg, bb):
        return np.sum(g * oracle.layernorm_forward(xx, gg, bb, eps)[0])

    fdx = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fdx[i, j] = (loss(xp, gamma, beta) - loss(xm, gamma, beta)) / (2 * h)
    fdg, fdb = np.zeros_like(gamma), np.zeros_like(beta)
    for j in range(len(gamma)):
        e = np.zeros_like(gamma)
        e[j] = h
        fdg[j] = (loss(x, gamma + e, beta) - loss(x, gamma - e, beta)) / (2 * h)
        fdb[j] = (loss(x, gamma, beta + e) - loss(x, gamma, beta - e)) / (2 * h)
    _close(dx, fdx, 1e-6, 1e-8, "dX")
    _close(dgamma, fdg, 1e-7, 1e-9, "dgamma")
    _close(dbeta, fdb, 1e-7, 1e-9, "dbeta")


def pin_layernorm_backward_invariants():
    x, gamma, beta, g = _ln_case(23, R=10, C=64)
    for eps in (0.0, 1e-5):
        _, xhat, r = oracle.layernorm_forward(x, gamma, beta, eps)
        dx, dgamma, dbeta = oracle.layernorm_backward(g, gamma, xhat, r)
        _close(dx.sum(axis=1), np.zeros(len(x)), 0, 1e-12, "rows of dX sum to 0")
        v = np.var(x, axis=1)
        b = np.mean(g * gamma * xhat, axis=1)
        # sum_j dX_j xhat_j = r C b eps / (v + eps), exactly 0 when eps = 0
        _close((dx * xhat).sum(axis=1), r * x.shape[1] * b * eps / (v + eps), 1e-6, 1e-11,
               "sum dX * xhat")
        _close(dbeta, [math.fsum(col) for col in g.T], 1e-15, 1e-15, "dbeta = column sums of g")
        _close(dgamma, [math.fsum(col) for col in (g * xhat).T], 1e-14, 1e-14, "dgamma")
    # a constant upstream gradient with unit gamma gives dX = 0
    _, xhat, r = oracle.layernorm_forward(x, np.ones(64), beta, 1e-5)
    _close(oracle.layernorm_backward_input(np.full_like(x, 0.75), np.ones(64), xhat, r),
           np.zeros_like(x), 0, 1e-13, "constant g")


def pin_layernorm_backward_matches_torch_autograd():
    x, gamma, beta, g = _ln_case(24, R=7, C=96)
    eps = 1e-5
    xt = torch.from_numpy(x).requires_grad_(True)
    gt = torch.from_numpy(gamma).requires_grad_(True)
    bt = torch.from_numpy(beta).requires_grad_(True)
    y = torch.nn.functional.layer_norm(xt, (96,), gt, bt, eps)
    dxr, dgr, dbr = torch.autograd.grad(y, (xt, gt, bt), torch.from_numpy(g))
    _, xhat, r = oracle.layernorm_forward(x, gamma, beta, eps)
    dx, dgamma, dbeta = oracle.layernorm_backward(g, gamma, xhat, r)
    _close(dx, dxr.numpy(), 1e-9, 1e-12, "dX")
    _close(dgamma, dgr.numpy(), 1e-11, 1e-12, "dgamma")
    _close(dbeta, dbr.numpy(), 1e-12, 1e-12, "dbeta")


# -------------------------------------------------------------- masked softmax

def pin_masked_golden():
    for c in _golden("row_op_examples.json")["masked_softmax"]["cases"]:
        y = oracle.masked_softmax(_f(c["x"])[None], np.array([c["mask"]], np.uint8))
        _close(y[0], _f(c["y"]), 1e-15, 0, c["why"])


def pin_masked_structure():
    rng = _rng(25)
    R, C = 40, 64
    x = rng.integers(-32, 33, (R, C)) / 8.0
    mask = (rng.random((R, C)) < 0.7).astype(np.uint8)
    mask[[3, 17]] = 0
    mask[5] = 0
    mask[5, 9] = 7  # any nonzero byte allows
    y = oracle.masked_softmax(x, mask)
    assert (y[mask == 0] == 0.0).all() and not np.signbit(y[mask == 0]).any(), "blocked are +0"
    assert (y[[3, 17]] == 0.0).all(), "all-blocked rows are zero"
    assert y[5, 9] == 1.0
    live = mask.any(axis=1)
    _close(y[live].sum(axis=1), np.ones(live.sum()), 0, 1e-14, "allowed mass is 1")
    # equals softmax of the allowed sub-vector scattered back, and torch with -inf fill
    for i in np.flatnonzero(live):
        a = mask[i] != 0
        _close(y[i, a], torch.softmax(torch.from_numpy(x[i, a]), 0).numpy(), 1e-14, 1e-17, "sub-vector")
    ref = torch.softmax(torch.from_numpy(x).masked_fill(torch.from_numpy(mask == 0), float("-inf")), 1)
    _close(y[live], ref.numpy()[live], 1e-14, 1e-17, "torch -inf fill")
    assert np.array_equal(oracle.masked_softmax(x, np.ones_like(mask)), oracle.softmax_rows(x))


# ---------------------------------------------------------------- top-k kept

def pin_kept_golden():
    for c in _golden("kept_mask_examples.json")["cases"]:
        got = oracle.topk_kept(_f(c["x"])[None], c["k"])[0]
        assert got.tolist() == c["kept"], (c["x"], c["k"], got.tolist(), c["why"])


def _kept_by_sorting(row, k):
    # Stable sort by value, largest first (equal values keep index order); keep the first k.
    order = sorted(range(len(row)), key=lambda j: (-row[j], j))
    out = np.zeros(len(row), np.uint8)
    out[order[:k]] = 1
    return out


def pin_kept_brute_force_sort():
    rng = _rng(26)
    for C in (1, 2, 3, 8, 33, 64):
        x = rng.integers(-6, 7, (30, C)) / 2.0  # heavy ties
        x[x == 0] = np.where(rng.random((x == 0).sum()) < 0.5, 0.0, -0.0)  # both zeros
        for k in sorted({1, min(2, C), min(3, C), C}):
            kept = oracle.topk_kept(x, k)
            for i in range(30):
                assert np.array_equal(kept[i], _kept_by_sorting(list(x[i] + 0.0), k)), (C, k, i)
            assert (kept.sum(axis=1) == k).all()


def pin_kept_matches_torch_sort_and_argmax():
    rng = _rng(27)
    x = rng.integers(-32, 33, (50, 64)) / 8.0
    vals = torch.from_numpy(x)
    idx = torch.sort(vals, dim=1, descending=True, stable=True).indices.numpy()
    kept = oracle.topk_kept(x, 2)
    ref = np.zeros_like(kept)
    np.put_along_axis(ref, idx[:, :2], 1, axis=1)
    assert np.array_equal(kept, ref)
    one = oracle.topk_kept(x, 1)
    first = np.zeros_like(one)
    first[np.arange(50), np.argmax(x, axis=1)] = 1  # numpy argmax returns the first maximum
    assert np.array_equal(one, first)




# ------------------------------------------------------------------ top_k_rows

def pin_top_k_rows_golden():
    for c in _golden("row_op_examples.json")["top_k_rows"]["cases"]:
        v, i = oracle.top_k_rows(_f(c["x"])[None], c["k"], c["largest"])
        want_v, want_i = _f(c["values"]), _f(c["indices"])
        assert np.array_equal(i[0], want_i), (c["why"], i[0], want_i)
        same = (v[0] == want_v) | (np.isnan(v[0]) & np.isnan(want_v))
        assert same.all() and (np.signbit(v[0]) == np.signbit(want_v)).all(), c["why"]


def _top_k_by_sorting(row, k, largest):
    def rank(j):
        x = row[j]
        if np.isnan(x):
            return (0, 0.0, j) if largest else (1, 0.0, j)
        return (1, -x, j) if largest else (0, x, j)
    order = sorted(range(len(row)), key=rank)[:k]
    return np.array([row[j] for j in order]), np.array(order, dtype=np.float64)


def pin_top_k_rows_brute_force_sort():
    rng = _rng(28)
    for C in (1, 2, 5, 16, 64):
        x = rng.integers(-4, 5, (20, C)) / 2.0
        x[rng.random(x.shape) < 0.1] = np.nan
        x[rng.random(x.shape) < 0.05] = np.inf
        for k in sorted({1, min(2, C), C}):
            for largest in (True, False):
                v, i = oracle.top_k_rows(x, k, largest)
                for r in range(20):
                    wv, wi = _top_k_by_sorting(list(x[r]), k, largest)
                    assert np.array_equal(i[r], wi), (C, k, largest, r)
                    assert ((v[r] == wv) | (np.isnan(v[r]) & np.isnan(wv))).all()


def pin_top_k_rows_matches_torch_on_distinct_values():
    rng = _rng(29)
    x = rng.permutation(40 * 50).reshape(40, 50).astype(np.float64) / 7.0
    for largest in (True, False):
        v, i = oracle.top_k_rows(x, 6, largest)
        tv, ti = torch.topk(torch.from_numpy(x), 6, dim=1, largest=largest, sorted=True)
        assert np.array_equal(v, tv.numpy()) and np.array_equal(i, ti.numpy().astype(np.float64))


def pin_top_k_rows_agrees_with_kept_mask():
    # Without NaN both pages' rules rank by value, then lower column: the k
    # largest are exactly the kept entries.
    rng = _rng(30)
    x = rng.integers(-3, 4, (30, 24)) / 4.0
    for k in (1, 2, 5, 24):
        _, idx = oracle.top_k_rows(x, k, True)
        kept = oracle.topk_kept(x, k)
        for r in range(30):
            assert set(idx[r].astype(int)) == set(np.flatnonzero(kept[r]))


def pin_router_composition():
    rng = _rng(31)
    x = rng.integers(-32, 33, (64, 64)) / 8.0
    mask = (rng.random((64, 64)) < 0.8).astype(np.uint8)
    mask[7] = 0
    p, kept = oracle.router_masked_topk(x, mask, 2)
    assert (kept.sum(axis=1) == 2).all()
    assert np.array_equal(kept[7], np.r_[1, 1, np.zeros(62)].astype(np.uint8)), "all-blocked row keeps columns 0, 1"
    p32 = p.astype(np.float32)
    for r in range(64):
        assert np.array_equal(kept[r], _kept_by_sorting(list(p32[r].astype(np.float64)), 2))




# --------------------------------------------------------------------- RMSNorm

def pin_rms_norm_forward():
    x, gamma, _, _ = _ln_case(32, R=9, C=40)
    for eps in (1e-6, 0.3):
        out, rms = oracle.rms_norm_forward(x, gamma, eps)
        ms = np.mean(x * x, axis=1)
        _close(rms, np.sqrt(ms + eps), 1e-15, 0, "rms closed form")
        _close(np.mean((out / gamma) ** 2, axis=1), ms / (ms + eps), 1e-12, 0, "mean square of out/gamma")
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (40,), torch.from_numpy(gamma), eps).numpy()
        _close(out, ref, 1e-12, 1e-14, "torch rms_norm")
    o1, _ = oracle.rms_norm_forward(x, gamma, 0.0)
    o2, _ = oracle.rms_norm_forward(4.0 * x, gamma, 0.0)
    _close(o1, o2, 1e-13, 1e-14, "scale invariance at eps=0")
    out, rms = oracle.rms_norm_forward(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    _close(rms, [math.sqrt(12.5)], 1e-15, 0, "rms of (3, 4)")
    _close(out[0], [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], 1e-15, 0, "out of (3, 4)")


def pin_rms_norm_backward_finite_differences():
    x, gamma, _, g = _ln_case(33, R=3, C=6)
    eps = 1e-3
    out, rms = oracle.rms_norm_forward(x, gamma, eps)
    dx, gt = oracle.rms_norm_backward(g, gamma, x, rms)
    h = 1e-6

    def loss(xx, gg):
        return np.sum(g * oracle.rms_norm_forward(xx, gg, eps)[0])

    fdx = np.zeros_like(x)
    for i in range(3):
        for j in range(6):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fdx[i, j] = (loss(xp, gamma) - loss(xm, gamma)) / (2 * h)
    fdg = np.zeros_like(gamma)
    for j in range(6):
        e = np.zeros_like(gamma)
        e[j] = h
        fdg[j] = (loss(x, gamma + e) - loss(x, gamma - e)) / (2 * h)
    _close(dx, fdx, 1e-6, 1e-8, "dx")
    _close(oracle.column_sums(gt), fdg, 1e-7, 1e-9, "column sums of gamma_terms = dgamma")
    _close(gt, g * x / rms[:, None], 1e-15, 1e-15, "gamma_terms")


def pin_rms_norm_backward_matches_torch_autograd():
    x, gamma, _, g = _ln_case(34, R=6, C=80)
    xt = torch.from_numpy(x).requires_grad_(True)
    gt_ = torch.from_numpy(gamma).requires_grad_(True)
    y = torch.nn.functional.rms_norm(xt, (80,), gt_, 1e-5)
    dxr, dgr = torch.autograd.grad(y, (xt, gt_), torch.from_numpy(g))
    _, rms = oracle.rms_norm_forward(x, gamma, 1e-5)
    dx, terms = oracle.rms_norm_backward(g, gamma, x, rms)
    _close(dx, dxr.numpy(), 1e-9, 1e-12, "dx")
    _close(oracle.column_sums(terms), dgr.numpy(), 1e-11, 1e-12, "dgamma")
    # sum_j dx_j x_j = (1/r) s C (1 - ms/r^2) = s C eps / r^3, with s = mean(g' x)
    s = np.mean(g * gamma * x, axis=1)
    ms = np.mean(x * x, axis=1)
    _close((dx * x).sum(axis=1), s * 80 * 1e-5 / rms ** 3, 1e-6, 1e-12, "sum dx * x")


def pin_column_sums():
    rng = _rng(35)
    m = rng.normal(0, 1, (37, 11))
    _close(oracle.column_sums(m), [math.fsum(c) for c in m.T], 1e-15, 1e-15, "fsum")
    prev = rng.normal(0, 1, 11)
    _close(oracle.column_sums(m, prev, 0.5), 0.5 * prev + [math.fsum(c) for c in m.T], 1e-15, 1e-15, "beta")
    nan_prev = np.full(11, np.nan)
    assert not np.isnan(oracle.column_sums(m, nan_prev, 0.0)).any(), "beta = 0 does not read out"
    assert np.array_equal(oracle.column_sums(np.zeros((0, 4))), np.zeros(4))




# ------------------------------------------- lrp softmax, float mask, argmax

def pin_lrp_softmax_rows():
    for c in _golden("row_op_examples.json")["lrp_softmax_rows"]["cases"]:
        got = oracle.lrp_softmax_rows(_f(c["x"])[None], _f(c["y"])[None], _f(c["r"])[None])
        _close(got[0], _f(c["r_in"]), 0, 1e-15, c["why"])
    rng = _rng(36)
    x = rng.normal(0, 1, (5, 9))
    y = oracle.softmax_rows(rng.normal(0, 1, (5, 9)))
    r1, r2 = rng.normal(0, 1, (5, 9)), rng.normal(0, 1, (5, 9))
    _close(oracle.lrp_softmax_rows(x, y, 2 * r1 - 3 * r2),
           2 * oracle.lrp_softmax_rows(x, y, r1) - 3 * oracle.lrp_softmax_rows(x, y, r2), 1e-13, 1e-13, "linear in r")
    _close(oracle.lrp_softmax_rows(x, np.zeros_like(y), r1), x * r1, 1e-15, 0, "y = 0")
    onehot = np.zeros((5, 9))
    onehot[np.arange(5), [0, 3, 8, 2, 2]] = 1
    _close(oracle.lrp_softmax_rows(np.ones((5, 9)), onehot, r1), r1 - onehot * r1.sum(axis=1, keepdims=True),
           1e-14, 1e-14, "x = 1, one-hot y")


def pin_masked_softmax_float_mask():
    rng = _rng(37)
    x = rng.integers(-16, 17, (30, 20)) / 4.0
    mask = rng.choice([0.0, -0.0, 1.0, 0.25, -3.0, np.nan], size=(30, 20))
    mask[4] = 0.0
    y = oracle.masked_softmax_fmask(x, mask)
    assert np.array_equal(y, oracle.masked_softmax(x, (mask != 0).astype(np.uint8)))
    assert (y[4] == 0).all()


def pin_argmax_onehot():
    for c in _golden("row_op_examples.json")["argmax_onehot"]["cases"]:
        got = oracle.argmax_onehot(_f(c["x"])[None])
        assert np.array_equal(got[0], _f(c["out"])), c["why"]
    rng = _rng(38)
    x = rng.integers(-3, 4, (200, 17)) / 2.0
    out = oracle.argmax_onehot(x)
    ref = np.zeros_like(out)
    ref[np.arange(200), np.argmax(x, axis=1)] = 1  # numpy: the first maximum
    assert np.array_equal(out, ref)
    assert np.array_equal(out, oracle.topk_kept(x, 1).astype(np.float64)), "k = 1 kept mask without NaN"
    assert oracle.argmax_onehot(np.zeros((3, 0))).shape == (3, 0)




# ------------------------------------------------------ soft / teacher CE

def pin_soft_ce():
    rng = _rng(39)
    R, C = 7, 30
    x = rng.normal(0, 2, (R, C))
    t = rng.integers(0, C, R).astype(np.int32)
    onehot = np.zeros((R, C))
    onehot[np.arange(R), t] = 1
    g1, l1, m1 = oracle.soft_ce(x, onehot, 1 / R)
    g2, l2, m2 = oracle.softmax_cross_entropy(x, t, 1 / R)
    _close(l1, l2, 1e-13, 1e-14, "one-hot weights = integer targets")
    _close(g1, g2, 1e-13, 1e-16, "gradient")
    w = rng.random((R, C))
    w /= w.sum(axis=1, keepdims=True)
    g, loss, mean = oracle.soft_ce(x, w, 1 / R)
    xt = torch.from_numpy(x).requires_grad_(True)
    ref = torch.nn.functional.cross_entropy(xt, torch.from_numpy(w), reduction="none")
    _close(loss, ref.detach().numpy(), 1e-13, 1e-14, "torch soft-target cross_entropy")
    (gx,) = torch.autograd.grad(ref.mean(), xt)
    _close(g, gx.numpy(), 1e-12, 1e-16, "torch gradient")
    # unnormalised weights: gradient of the mean loss by finite differences
    w2 = rng.random((3, 5)) * 3
    x2 = rng.normal(0, 1, (3, 5))
    g3, _, _ = oracle.soft_ce(x2, w2, 1 / 3)
    h = 1e-6
    fd = np.zeros_like(x2)
    for i in range(3):
        for j in range(5):
            xp, xm = x2.copy(), x2.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd[i, j] = (oracle.soft_ce(xp, w2, 1.0)[2] - oracle.soft_ce(xm, w2, 1.0)[2]) / (2 * h)
    _close(g3, fd, 1e-7, 1e-10, "finite differences")
    # a zero weight on an underflowing probability contributes 0, not NaN
    _, l4, _ = oracle.soft_ce(np.array([[0.0, -2000.0]]), np.array([[1.0, 0.0]]), 1.0)
    assert np.isfinite(l4).all()


def pin_teacher_ce():
    rng = _rng(40)
    R, C = 6, 25
    s = rng.normal(0, 2, (R, C))
    t = rng.normal(0, 2, (R, C))
    q = oracle.softmax_rows(t)
    g, loss, mean = oracle.teacher_ce(s, t, 1 / R)
    gs, ls, ms = oracle.soft_ce(s, q, 1 / R)
    _close(loss, ls, 1e-13, 1e-14, "teacher CE = soft CE with softmax(t)")
    _close(g, (oracle.softmax_rows(s) - q) / R, 1e-13, 1e-17, "student gradient")
    st = torch.from_numpy(s).requires_grad_(True)
    ref = torch.nn.functional.cross_entropy(st, torch.softmax(torch.from_numpy(t), 1), reduction="none")
    _close(loss, ref.detach().numpy(), 1e-13, 1e-14, "torch")
    entropy = -(q * np.log(q)).sum(axis=1)
    assert (loss - entropy >= -1e-12).all(), "cross-entropy >= entropy (KL >= 0)"
    _close(oracle.teacher_ce(s, s, 1.0)[1], -(oracle.softmax_rows(s) * np.log(oracle.softmax_rows(s))).sum(1),
           1e-12, 1e-14, "teacher = student gives the entropy")


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
