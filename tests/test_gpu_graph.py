"""GPU: the row ops captured into one CUDA graph and replayed give the same
bits as the same calls made eagerly.

Every entry point only enqueues kernels on the stream it is given (no
allocation, no synchronisation), so a whole step of calls can be captured
once and replayed; this covers the group, cluster, bulk-copy pipeline
(including rows split over a cluster of CTAs) and programmatic-dependent
(two-kernel) paths."""
import numpy as np
import pytest
import torch

from parity_util import gpu
from row_wise_softmax_warp_gb300 import inputs

pytestmark = pytest.mark.gpu


class Step:
    """Inputs, outputs and the list of calls of one step (buffers fixed, so a
    graph captured from it can be replayed on new input values)."""

    def __init__(self, ro, seed):
        self.ro = ro
        d = inputs.softmax_pair(seed, rows=64, cols=128)
        self.sx, self.sdy = gpu(d["x"]), gpu(d["dy"])
        n = inputs.layernorm(seed, rows=300, cols=768)
        self.eps = n["eps"]
        self.lx, self.lg, self.lb, self.ldy = gpu(n["x"]), gpu(n["gamma"]), gpu(n["beta"]), gpu(n["dy"])
        self.lws = torch.empty(ro.rowops_layernorm_bwd_workspace(300, 768), dtype=torch.uint8, device="cuda")
        a = inputs.attention(seed, batch=1, heads=2, seq=1024)
        self.seq, self.scale = a["seq_len"], a["scale"]
        self.as_, self.adp = gpu(a["scores"]), gpu(a["dp"])
        c = inputs.cross_entropy(seed, rows=40, cols=50304)
        self.cx, self.ct, self.cgs = gpu(c["logits"]), gpu(c["targets"]), c["grad_scale"]
        r = inputs.router(seed, rows=5000, cols=64)
        self.rx, self.rm, self.k = gpu(r["x"]), gpu(r["mask"]), r["k"]
        # rows for the cluster kernels: a vocabulary row split over a cluster,
        # and the long-row softmax backward
        v = inputs.cross_entropy(seed + 7, rows=6, cols=152064)
        self.vx, self.vt, self.vgs = gpu(v["logits"]), gpu(v["targets"]), v["grad_scale"]
        w = inputs.softmax_pair(seed + 9, rows=5, cols=40000)
        self.wy, self.wdy = gpu(w["x"]).softmax(dim=1), gpu(w["dy"])
        e = torch.empty_like
        self.out = {
            "sy": e(self.sx), "sdx": e(self.sx),
            "lout": e(self.lx), "lxh": e(self.lx), "lrs": torch.empty(300, device="cuda"),
            "ldx": e(self.lx), "ldg": e(self.lg), "ldb": e(self.lg),
            "ap": e(self.as_), "ads": e(self.as_),
            "clse": torch.empty(40, device="cuda"), "cg": e(self.cx), "crl": torch.empty(40, device="cuda"),
            "cml": torch.empty(1, dtype=torch.float64, device="cuda"),
            "rp": e(self.rx), "rk": e(self.rx), "fp": e(self.rx), "fk": e(self.rx),
            "tv": torch.empty((5000, self.k), device="cuda"), "ti": torch.empty((5000, self.k), device="cuda"),
            "rms": e(self.lx), "rmsr": torch.empty(300, device="cuda"), "rmsdx": e(self.lx), "rmst": e(self.lx),
            "rmsdg": e(self.lg),
            "vg": e(self.vx), "vrl": torch.empty(6, device="cuda"),
            "vml": torch.empty(1, dtype=torch.float64, device="cuda"), "vy": e(self.vx), "wdx": e(self.wy),
        }

    def run(self):
        ro, o = self.ro, self.out
        ro.rowops_softmax_fwd(self.sx, o["sy"])
        ro.rowops_softmax_bwd(o["sy"], self.sdy, o["sdx"])
        ro.rowops_layernorm_fwd(self.lx, self.lg, self.lb, o["lout"], o["lxh"], o["lrs"], eps=self.eps)
        ro.rowops_layernorm_bwd(self.ldy, self.lg, o["lxh"], o["lrs"], o["ldx"], o["ldg"], o["ldb"],
                                workspace=self.lws)
        ro.rowops_attn_softmax_fwd(self.as_, o["ap"], seq_len=self.seq, scale=self.scale)
        ro.rowops_attn_softmax_bwd(o["ap"], self.adp, o["ads"], seq_len=self.seq, scale=self.scale)
        ro.rowops_logsumexp(self.cx, o["clse"])
        ro.rowops_softmax_ce(self.cx, self.ct, o["cg"], o["crl"], o["cml"], grad_scale=self.cgs)
        ro.rowops_masked_softmax(self.rx, self.rm, o["rp"])
        ro.rowops_topk_kept(o["rp"], self.k, o["rk"])
        ro.rowops_router_masked_topk(self.rx, self.rm, self.k, o["fp"], o["fk"])
        ro.rowops_top_k_rows(self.rx, self.k, True, o["tv"], o["ti"])
        ro.rowops_rmsnorm_fwd(self.lx, self.lg, o["rms"], o["rmsr"], eps=self.eps)
        ro.rowops_rmsnorm_bwd(self.ldy, self.lg, self.lx, o["rmsr"], o["rmsdx"], o["rmst"])
        ro.rowops_column_sums(o["rmst"], o["rmsdg"])
        ro.rowops_softmax_ce(self.vx, self.vt, o["vg"], o["vrl"], o["vml"], grad_scale=self.vgs)
        ro.rowops_softmax_fwd(self.vx, o["vy"])
        ro.rowops_softmax_bwd(self.wy, self.wdy, o["wdx"])

    def snapshot(self):
        torch.cuda.synchronize()
        return {k: v.clone() for k, v in self.out.items()}

    def poison(self):
        for v in self.out.values():
            v.fill_(float("nan"))


def _same(a, b):
    for k in a:
        x, y = a[k].cpu().numpy(), b[k].cpu().numpy()
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), k


def test_step_graph_replay_matches_eager(ro):
    step = Step(ro, 0)
    step.run()  # eager (also the first call of every kernel, outside capture)
    eager = step.snapshot()
    step.poison()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step.run()
    torch.cuda.current_stream().wait_stream(s)
    step.poison()  # capture launched nothing; the replay must write every output
    g.replay()
    _same(eager, step.snapshot())
    # New input values in the same buffers: the replay follows them.
    other = Step(ro, 1)
    for name in ("sx", "sdy", "lx", "lg", "lb", "ldy", "as_", "adp", "cx", "ct", "rx", "rm", "vx", "vt", "wy", "wdy"):
        getattr(step, name).copy_(getattr(other, name))
    other.run()
    g.replay()
    _same(other.snapshot(), step.snapshot())
