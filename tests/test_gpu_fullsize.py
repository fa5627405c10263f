"""GPU parity at the benchmark's full sizes, through the same calls the
benchmark times.  Where the oracle cannot afford every row, it checks a seeded
sample of rows element by element (always including the first and last rows
and, for attention, the first and last query of a head) and the GPU output is
checked on every row through properties that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_abs, check_bound, check_exact_zero, check_probs, check_rel, host, \
    softmax_bwd_bound
from row_wise_softmax_warp_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample(rows, n, seed, extra=()):
    rng = np.random.default_rng(seed)
    s = set(rng.choice(rows, size=min(n, rows), replace=False).tolist())
    s.update([0, rows - 1, *extra])
    return np.array(sorted(s))


def test_attention_8x12x1024(ro):
    a = inputs.attention(0)
    s, dp, scale, S = a["scores"], a["dp"], a["scale"], a["seq_len"]
    rows = s.shape[0]
    sg = torch.from_numpy(s).cuda()
    p = ro.rowops_attn_softmax_fwd(sg, seq_len=S, scale=scale)
    idx = _sample(rows, 384, 1, extra=(S - 1, S, 2 * S - 1, rows - S))
    ref_rows = np.concatenate([oracle.attn_softmax_forward(s[i:i + 1], S, scale, row0=int(i)) for i in idx])
    check_probs(host(p[torch.from_numpy(idx).cuda()]), ref_rows, "attn fwd sampled rows")
    # every row: visible probabilities sum to 1, masked entries exactly +0
    q = torch.arange(rows, device="cuda") % S
    upper = torch.arange(S, device="cuda")[None, :] > q[:, None]
    assert bool((p.masked_select(upper) == 0).all()) and not bool(p.masked_select(upper).signbit().any())
    assert float((p.sum(dim=1, dtype=torch.float64) - 1).abs().max()) < 1e-5
    del sg
    # backward: P from the oracle (fp32), every row computed on the GPU
    p32 = np.empty_like(s)
    for r0 in range(0, rows, 8192):
        p32[r0:r0 + 8192] = oracle.attn_softmax_forward(s[r0:r0 + 8192], S, scale, row0=r0)
    ds = ro.rowops_attn_softmax_bwd(torch.from_numpy(p32).cuda(), torch.from_numpy(dp).cuda(), seq_len=S,
                                    scale=scale)
    dref = np.concatenate([oracle.attn_softmax_backward(p32[i:i + 1], dp[i:i + 1], S, scale, row0=int(i))
                           for i in idx])
    qi = idx % S
    dp_vis = np.where(np.arange(S)[None, :] <= qi[:, None], dp[idx], 0)
    check_bound(host(ds[torch.from_numpy(idx).cuda()]), dref, softmax_bwd_bound(p32[idx], dp_vis, scale),
                "attn bwd sampled rows")
    assert bool((ds.masked_select(upper) == 0).all())
    # each gradient row sums to 0 (up to fp32 rounding of scale * p * (dp - c))
    tol = 1e-5 * scale * (torch.from_numpy(p32).cuda().abs() * torch.from_numpy(dp).cuda().abs()).sum(1)
    assert bool((ds.sum(dim=1, dtype=torch.float64).abs() <= tol.double() + 1e-7).all())


def test_cross_entropy_8192x50304(ro):
    c = inputs.cross_entropy(0)
    x, t, gs = c["logits"], c["targets"], c["grad_scale"]
    rows = x.shape[0]
    xg, tg = torch.from_numpy(x).cuda(), torch.from_numpy(t).cuda()
    lse = host(ro.rowops_logsumexp(xg))
    g, rl, ml = ro.rowops_softmax_ce(xg, tg, grad_scale=gs)
    # oracle logsumexp and row losses of every row (row blocks bound host memory)
    lse_ref = np.concatenate([oracle.logsumexp_rows(x[r0:r0 + 256]) for r0 in range(0, rows, 256)])
    check_rel(lse, lse_ref, "lse every row")
    loss_ref = lse_ref - x[np.arange(rows), t].astype(np.float64)
    check_rel(host(rl), loss_ref, "row loss every row")
    check_rel(host(ml), [oracle.mean(loss_ref)], "mean loss")
    idx = _sample(rows, 48, 2)
    gr, _, _ = oracle.softmax_cross_entropy(x[idx], t[idx], gs)
    check_abs(host(g[torch.from_numpy(idx).cuda()]), gr, 2e-6 * gs, "grad sampled rows")
    # every row: the gradient sums to 0 and is -gs*(1-p_t) at the target
    assert float(g.sum(dim=1, dtype=torch.float64).abs().max()) < 1e-6 * gs * 50304 ** 0.5 + 1e-9
    assert bool((g[torch.arange(rows, device="cuda"), tg.long()] <= 0).all())


def test_router_262144x64(ro):
    r = inputs.router(0)
    x, mask = r["x"], r["mask"]
    p = host(ro.rowops_masked_softmax(torch.from_numpy(x).cuda(), torch.from_numpy(mask).cuda()))
    pr = oracle.masked_softmax(x, mask)
    check_probs(p, pr, "masked softmax every row")
    check_exact_zero(p, mask == 0, "blocked entries")
    p32 = pr.astype(np.float32)
    kept = host(ro.rowops_topk_kept(torch.from_numpy(p32).cuda(), r["k"]))
    ref = oracle.topk_kept(p32, r["k"]).astype(np.float32)
    assert np.array_equal(kept, ref)
    assert (kept.sum(axis=1) == 2).all()
