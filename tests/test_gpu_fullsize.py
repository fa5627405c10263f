"""GPU parity at the benchmark's full sizes, through the same calls the
benchmark times.  Every row of every output is compared with the oracle
element by element; the oracle runs on all host cores over blocks of rows,
so host memory stays bounded (a block's float64 reference at a time)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import check_abs, check_bound, check_exact_zero, check_probs, check_rel, host, \
    softmax_bwd_bound
from row_wise_softmax_warp_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_attention_8x12x1024(ro):
    a = inputs.attention(0)
    s, dp, scale, S = a["scores"], a["dp"], a["scale"], a["seq_len"]
    rows = s.shape[0]
    block = 8192  # rows per oracle block (8 heads of 1024 queries)
    p = ro.rowops_attn_softmax_fwd(torch.from_numpy(s).cuda(), seq_len=S, scale=scale)
    q = torch.arange(rows, device="cuda") % S
    upper = torch.arange(S, device="cuda")[None, :] > q[:, None]
    # forward, every row; the backward takes P from the oracle (fp32), never
    # from the CUDA path
    p32 = np.empty_like(s)
    for r0 in range(0, rows, block):
        ref = oracle.attn_softmax_forward(s[r0:r0 + block], S, scale, row0=r0)
        check_probs(host(p[r0:r0 + block]), ref, f"attn fwd rows {r0}..{r0 + block - 1}")
        p32[r0:r0 + block] = ref
    assert bool((p.masked_select(upper) == 0).all()) and not bool(p.masked_select(upper).signbit().any())
    del p
    ds = ro.rowops_attn_softmax_bwd(torch.from_numpy(p32).cuda(), torch.from_numpy(dp).cuda(), seq_len=S,
                                    scale=scale)
    for r0 in range(0, rows, block):
        pb, dpb = p32[r0:r0 + block], dp[r0:r0 + block]
        ref = oracle.attn_softmax_backward(pb, dpb, S, scale, row0=r0)
        qi = (np.arange(r0, r0 + pb.shape[0]) % S)[:, None]
        dp_vis = np.where(np.arange(S)[None, :] <= qi, dpb, 0)
        check_bound(host(ds[r0:r0 + block]), ref, softmax_bwd_bound(pb, dp_vis, scale),
                    f"attn bwd rows {r0}..{r0 + block - 1}")
    assert bool((ds.masked_select(upper) == 0).all()) and not bool(ds.masked_select(upper).signbit().any())


def test_cross_entropy_8192x50304(ro):
    c = inputs.cross_entropy(0)
    x, t, gs = c["logits"], c["targets"], c["grad_scale"]
    rows = x.shape[0]
    xg, tg = torch.from_numpy(x).cuda(), torch.from_numpy(t).cuda()
    lse = host(ro.rowops_logsumexp(xg))
    g, rl, ml = ro.rowops_softmax_ce(xg, tg, grad_scale=gs)
    block = 256
    lse_ref = np.empty(rows)
    loss_ref = np.empty(rows)
    for r0 in range(0, rows, block):
        gr, lr, _ = oracle.softmax_cross_entropy(x[r0:r0 + block], t[r0:r0 + block], gs)
        check_abs(host(g[r0:r0 + block]), gr, 2e-6 * gs, f"grad rows {r0}..{r0 + block - 1}")
        loss_ref[r0:r0 + block] = lr
        lse_ref[r0:r0 + block] = oracle.logsumexp_rows(x[r0:r0 + block])
    check_rel(lse, lse_ref, "lse every row")
    check_rel(host(rl), loss_ref, "row loss every row")
    check_rel(host(ml), [oracle.mean(loss_ref)], "mean loss")


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


def test_layernorm_4096x768(ro):
    n = inputs.layernorm(0)
    x, gamma, beta, dy, eps = n["x"], n["gamma"], n["beta"], n["dy"], n["eps"]
    out, xh, rs = ro.rowops_layernorm_fwd(torch.from_numpy(x).cuda(), torch.from_numpy(gamma).cuda(),
                                          torch.from_numpy(beta).cuda(), eps=eps)
    o_r, xh_r, rs_r = oracle.layernorm_forward(x, gamma, beta, eps)
    check_rel(host(xh), xh_r, "xhat every row")
    check_rel(host(out), o_r, "out every row")
    check_bound(host(rs), rs_r, 1e-5 * np.abs(rs_r), "inv_std every row")
