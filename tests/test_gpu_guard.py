"""Guard bands around every output: each output buffer sits inside a larger
allocation whose 4 KiB before and after it hold a fixed bit pattern, checked
after the call, and every input is checked to be unchanged.  A kernel that
writes one element outside its rows, or into an input, fails here (a stand-in
for a memory checker).  Shapes cover every kernel shape: lane groups, CTA
rows, the bulk-copy pipelines (one pass, two passes, two inputs), the
streaming fallbacks and the top-k select, with outputs on and off 16-byte
boundaries."""
import numpy as np
import pytest
import torch

from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PATTERN = 0x5A


class Guarded:
    """A view of `shape` inside a byte buffer filled with PATTERN, `off`
    elements past a 4 KiB (hence 256-byte aligned) boundary."""

    def __init__(self, shape, dtype=torch.float32, off=0):
        esize = torch.tensor([], dtype=dtype).element_size()
        n = int(np.prod(shape)) if len(shape) else 1
        self.lo = GUARD + off * esize
        self.hi = self.lo + n * esize
        self.raw = torch.full((self.hi + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.view = self.raw[self.lo:self.hi].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        raw = self.raw.cpu().numpy()
        bad_lo = np.nonzero(raw[:self.lo] != PATTERN)[0]
        bad_hi = np.nonzero(raw[self.hi:] != PATTERN)[0]
        assert bad_lo.size == 0, f"{what}: {bad_lo.size} bytes written before the buffer (last at -{self.lo - bad_lo[-1]})"
        assert bad_hi.size == 0, f"{what}: {bad_hi.size} bytes written after the buffer (first at +{bad_hi[0]})"


def _in(a, off=0):
    """Device input `off` elements past a 256-byte boundary, with a copy to
    check that it is left unchanged."""
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    flat = torch.zeros(t.numel() + 8, dtype=t.dtype, device="cuda")
    view = flat[off:off + t.numel()].view(t.shape)
    view.copy_(t.cuda())
    return view, view.clone()


def _unchanged(pairs, what):
    for i, (t, ref) in enumerate(pairs):
        assert torch.equal(t, ref), f"{what}: input {i} was written"


COLS = [7, 64, 768, 1025, 3001, 16385, 50257, 70001]


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("off", [0, 1])
def test_guard_softmax_family(ro, cols, off):
    rows = 3 if cols > 4096 else 9
    c = inputs.cross_entropy(cols, rows=rows, cols=cols)
    x, t = c["logits"], c["targets"]
    xg = _in(x, off)
    y = Guarded(x.shape, off=off)
    ro.rowops_softmax_fwd(xg[0], y.view)
    y.check(f"softmax y cols={cols}")
    dy = _in(np.random.default_rng(cols).normal(0, 1, x.shape).astype(np.float32), off)
    yin = _in(y.view.cpu().numpy(), off)
    dx = Guarded(x.shape, off=1 - off)
    ro.rowops_softmax_bwd(yin[0], dy[0], dx.view)
    dx.check(f"softmax dx cols={cols}")
    lse = Guarded((rows,), off=off)
    ro.rowops_logsumexp(xg[0], lse.view)
    lse.check(f"lse cols={cols}")
    tg = _in(t, off)
    g, rl, ml = Guarded(x.shape, off=off), Guarded((rows,), off=1 - off), Guarded((1,), torch.float64)
    ro.rowops_softmax_ce(xg[0], tg[0], g.view, rl.view, ml.view, grad_scale=c["grad_scale"])
    for b, n in ((g, "grad"), (rl, "row_loss"), (ml, "mean_loss")):
        b.check(f"ce {n} cols={cols}")
    w = _in(np.random.default_rng(cols + 1).random(x.shape).astype(np.float32), off)
    for f, n in ((ro.rowops_soft_ce, "soft"), (ro.rowops_teacher_ce, "teacher")):
        g2, rl2, ml2 = Guarded(x.shape, off=1 - off), Guarded((rows,)), Guarded((1,), torch.float64)
        f(xg[0], w[0], g2.view, rl2.view, ml2.view, grad_scale=1.0 / rows)
        for b, m in ((g2, "grad"), (rl2, "row_loss"), (ml2, "mean_loss")):
            b.check(f"{n} ce {m} cols={cols}")
    oh = Guarded(x.shape, off=off)
    ro.rowops_argmax_onehot(xg[0], oh.view)
    oh.check(f"argmax cols={cols}")
    rin = Guarded(x.shape, off=off)
    ro.rowops_lrp_softmax_rows(xg[0], yin[0], dy[0], rin.view)
    rin.check(f"lrp cols={cols}")
    _unchanged([xg, dy, yin, tg, w], f"softmax family cols={cols}")


@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("off", [0, 1])
def test_guard_norms(ro, cols, off):
    rows = 3 if cols > 4096 else 9
    n = inputs.layernorm(cols, rows=rows, cols=cols)
    x, gamma, beta, dy = (_in(n[k], off) for k in ("x", "gamma", "beta", "dy"))
    out, xh, rs = Guarded((rows, cols), off=off), Guarded((rows, cols), off=1 - off), Guarded((rows,), off=off)
    ro.rowops_layernorm_fwd(x[0], gamma[0], beta[0], out.view, xh.view, rs.view, eps=n["eps"])
    for b, m in ((out, "out"), (xh, "xhat"), (rs, "inv_std")):
        b.check(f"ln fwd {m} cols={cols}")
    xh_in, rs_in = _in(xh.view.cpu().numpy(), off), _in(rs.view.cpu().numpy())
    need = ro.rowops_layernorm_bwd_workspace(rows, cols)
    ws = Guarded((need,), torch.uint8)
    dx, dg, db = Guarded((rows, cols), off=off), Guarded((cols,), off=1 - off), Guarded((cols,), off=off)
    ro.rowops_layernorm_bwd(dy[0], gamma[0], xh_in[0], rs_in[0], dx.view, dg.view, db.view, workspace=ws.view)
    for b, m in ((dx, "dx"), (dg, "dgamma"), (db, "dbeta"), (ws, "workspace")):
        b.check(f"ln bwd {m} cols={cols}")
    o2, rr = Guarded((rows, cols), off=off), Guarded((rows,), off=off)
    ro.rowops_rmsnorm_fwd(x[0], gamma[0], o2.view, rr.view, eps=n["eps"])
    o2.check(f"rms out cols={cols}")
    rr.check(f"rms row_rms cols={cols}")
    rr_in = _in(rr.view.cpu().numpy())
    dx2, terms = Guarded((rows, cols), off=off), Guarded((rows, cols), off=1 - off)
    ro.rowops_rmsnorm_bwd(dy[0], gamma[0], x[0], rr_in[0], dx2.view, terms.view)
    dx2.check(f"rms dx cols={cols}")
    terms.check(f"rms terms cols={cols}")
    cs = Guarded((cols,), off=off)
    ro.rowops_column_sums(terms.view, cs.view)
    cs.check(f"column sums cols={cols}")
    _unchanged([x, gamma, beta, dy, xh_in, rs_in, rr_in], f"norms cols={cols}")


@pytest.mark.parametrize("cols", [7, 64, 256, 1025, 3001, 20000])
@pytest.mark.parametrize("off", [0, 1])
def test_guard_router_and_selection(ro, cols, off):
    rows = 5 if cols > 4096 else 17
    r = inputs.router(cols, rows=rows, cols=cols, p_allow=0.8, blocked_row_frac=0.1)
    x, m = _in(r["x"], off), _in(r["mask"], off)
    fm = _in(r["mask"].astype(np.float32), off)
    p = Guarded((rows, cols), off=off)
    ro.rowops_masked_softmax(x[0], m[0], p.view)
    p.check(f"masked cols={cols}")
    p2 = Guarded((rows, cols), off=1 - off)
    ro.rowops_masked_softmax_fmask(x[0], fm[0], p2.view)
    p2.check(f"fmask cols={cols}")
    for k in sorted({1, 2, min(5, cols), min(40, cols)}):
        kept = Guarded((rows, cols), off=off)
        ro.rowops_topk_kept(x[0], k, kept.view)
        kept.check(f"kept cols={cols} k={k}")
        pr, kr = Guarded((rows, cols), off=off), Guarded((rows, cols), off=1 - off)
        ro.rowops_router_masked_topk(x[0], m[0], k, pr.view, kr.view)
        pr.check(f"router p cols={cols} k={k}")
        kr.check(f"router kept cols={cols} k={k}")
        vals, idx = Guarded((rows, k), off=off), Guarded((rows, k), off=1 - off)
        ro.rowops_top_k_rows(x[0], k, True, vals.view, idx.view)
        vals.check(f"top_k values cols={cols} k={k}")
        idx.check(f"top_k indices cols={cols} k={k}")
    _unchanged([x, m, fm], f"router cols={cols}")


@pytest.mark.parametrize("seq", [8, 100, 1024, 2049])
@pytest.mark.parametrize("off", [0, 1])
def test_guard_attention(ro, seq, off):
    a = inputs.attention(seq, batch=1, heads=1, seq=seq)
    s, dp = _in(a["scores"], off), _in(a["dp"], off)
    p = Guarded(a["scores"].shape, off=off)
    ro.rowops_attn_softmax_fwd(s[0], p.view, seq_len=seq, scale=a["scale"])
    p.check(f"attn p seq={seq}")
    p_in = _in(p.view.cpu().numpy(), off)
    ds = Guarded(a["scores"].shape, off=1 - off)
    ro.rowops_attn_softmax_bwd(p_in[0], dp[0], ds.view, seq_len=seq, scale=a["scale"])
    ds.check(f"attn ds seq={seq}")
    _unchanged([s, dp, p_in], f"attention seq={seq}")
