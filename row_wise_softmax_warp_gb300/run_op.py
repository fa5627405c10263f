"""Runs one row op a few times on seeded inputs of a chosen size (for profilers).

    python -m row_wise_softmax_warp_gb300.run_op --op softmax_ce --rows 1024 --cols 50304 --reps 3

Ops: softmax_fwd, softmax_bwd, attn_fwd, attn_bwd (cols = seq_len), logsumexp,
softmax_ce, layernorm_fwd, layernorm_bwd, rmsnorm_fwd, rmsnorm_bwd, masked_softmax, topk_kept,
router_masked_topk, top_k_rows, argmax_onehot, soft_ce, teacher_ce.  For rows of
more than 1024 floats, top_k_rows and argmax_onehot take logits-like rows
(top_k_rows with k from ROWOPS_TOPK, default 50); topk_kept,
router_masked_topk and top_k_rows on shorter rows take k from ROWOPS_K
(default 2).  Inputs
follow the workload distributions of ``inputs``; the L2 is flushed (512 MiB
write) before every call.  Prints the median CUDA-event time per call.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from row_wise_softmax_warp_gb300 import binding as ro  # noqa: E402
from row_wise_softmax_warp_gb300 import build, inputs  # noqa: E402


def make(op: str, rows: int, cols: int, dev):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    if op in ("softmax_fwd", "softmax_bwd"):
        d = inputs.softmax_pair(0, rows=rows, cols=cols)
        x, dy = t(d["x"]), t(d["dy"])
        y = ro.rowops_softmax_fwd(x)
        return (lambda: ro.rowops_softmax_fwd(x, y)) if op == "softmax_fwd" else \
            (lambda: ro.rowops_softmax_bwd(y, dy))
    if op in ("attn_fwd", "attn_bwd"):
        heads = max(1, rows // cols)
        a = inputs.attention(0, batch=1, heads=heads, seq=cols)
        s, dp = t(a["scores"]), t(a["dp"])
        p = ro.rowops_attn_softmax_fwd(s, seq_len=cols, scale=a["scale"])
        if op == "attn_fwd":
            return lambda: ro.rowops_attn_softmax_fwd(s, p, seq_len=cols, scale=a["scale"])
        ds = torch.empty_like(p)
        return lambda: ro.rowops_attn_softmax_bwd(p, dp, ds, seq_len=cols, scale=a["scale"])
    if op in ("logsumexp", "softmax_ce"):
        c = inputs.cross_entropy(0, rows=rows, cols=cols)
        x, tg = t(c["logits"]), t(c["targets"])
        if op == "logsumexp":
            out = torch.empty(rows, device=dev)
            return lambda: ro.rowops_logsumexp(x, out)
        g = torch.empty_like(x)
        rl = torch.empty(rows, device=dev)
        ml = torch.empty(1, dtype=torch.float64, device=dev)
        return lambda: ro.rowops_softmax_ce(x, tg, g, rl, ml, grad_scale=c["grad_scale"])
    if op in ("layernorm_fwd", "layernorm_bwd"):
        n = inputs.layernorm(0, rows=rows, cols=cols)
        x, gm, bt, dy = t(n["x"]), t(n["gamma"]), t(n["beta"]), t(n["dy"])
        out, xh, rs = ro.rowops_layernorm_fwd(x, gm, bt, eps=n["eps"])
        if op == "layernorm_fwd":
            return lambda: ro.rowops_layernorm_fwd(x, gm, bt, out, xh, rs, eps=n["eps"])
        ws = torch.empty(ro.rowops_layernorm_bwd_workspace(rows, cols), dtype=torch.uint8, device=dev)
        dx, dg, db = torch.empty_like(x), torch.empty_like(gm), torch.empty_like(gm)
        return lambda: ro.rowops_layernorm_bwd(dy, gm, xh, rs, dx, dg, db, workspace=ws)
    if op in ("rmsnorm_fwd", "rmsnorm_bwd"):
        n = inputs.layernorm(0, rows=rows, cols=cols)
        x, gm, dy = t(n["x"]), t(n["gamma"]), t(n["dy"])
        out, rr = ro.rowops_rmsnorm_fwd(x, gm, eps=n["eps"])
        if op == "rmsnorm_fwd":
            return lambda: ro.rowops_rmsnorm_fwd(x, gm, out, rr, eps=n["eps"])
        dx, terms = torch.empty_like(x), torch.empty_like(x)
        return lambda: ro.rowops_rmsnorm_bwd(dy, gm, x, rr, dx, terms)
    if op in ("masked_softmax", "topk_kept"):
        r = inputs.router(0, rows=rows, cols=cols)
        x, m = t(r["x"]), t(r["mask"])
        p = ro.rowops_masked_softmax(x, m)
        if op == "masked_softmax":
            return lambda: ro.rowops_masked_softmax(x, m, p)
        kept = torch.empty_like(p)
        return lambda: ro.rowops_topk_kept(p, int(os.environ.get("ROWOPS_K", r["k"])), kept)
    if op in ("soft_ce", "teacher_ce"):
        c = inputs.cross_entropy(0, rows=rows, cols=cols)
        c2 = inputs.cross_entropy(1, rows=rows, cols=cols)
        x, w = t(c["logits"]), t(c2["logits"])
        if op == "soft_ce":
            w = torch.softmax(w, dim=1)
        g = torch.empty_like(x)
        rl = torch.empty(rows, device=dev)
        ml = torch.empty(1, dtype=torch.float64, device=dev)
        f = ro.rowops_soft_ce if op == "soft_ce" else ro.rowops_teacher_ce
        return lambda: f(x, w, g, rl, ml, grad_scale=1.0 / rows)
    if op in ("top_k_rows", "argmax_onehot") and cols > 1024:  # vocabulary-sized rows
        x = t(inputs.cross_entropy(0, rows=rows, cols=cols)["logits"])
        if op == "top_k_rows":
            k = int(os.environ.get("ROWOPS_TOPK", "50"))
            vals = torch.empty((rows, k), device=dev)
            idx = torch.empty_like(vals)
            return lambda: ro.rowops_top_k_rows(x, k, True, vals, idx)
        oh = torch.empty_like(x)
        return lambda: ro.rowops_argmax_onehot(x, oh)
    if op in ("router_masked_topk", "top_k_rows", "argmax_onehot"):
        r = inputs.router(0, rows=rows, cols=cols)
        x, m = t(r["x"]), t(r["mask"])
        if op == "router_masked_topk":
            p, kept = torch.empty_like(x), torch.empty_like(x)
            return lambda: ro.rowops_router_masked_topk(x, m, int(os.environ.get("ROWOPS_K", r["k"])), p, kept)
        if op == "top_k_rows":
            k = int(os.environ.get("ROWOPS_K", r["k"]))
            vals = torch.empty((rows, k), device=dev)
            idx = torch.empty_like(vals)
            return lambda: ro.rowops_top_k_rows(x, k, True, vals, idx)
        oh = torch.empty_like(x)
        return lambda: ro.rowops_argmax_onehot(x, oh)
    raise SystemExit(f"unknown op {op}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", required=True)
    ap.add_argument("--rows", type=int, required=True)
    ap.add_argument("--cols", type=int, required=True)
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    build.build()
    dev = torch.device("cuda", 0)
    fn = make(args.op, args.rows, args.cols, dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    times = []
    for _ in range(args.reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    times.sort()
    print(f"{args.op} {args.rows}x{args.cols}: median {times[len(times) // 2]:.1f} us over {args.reps} calls")
    timeouts = ro.library().rowops_pipeline_timeouts()
    if timeouts:
        raise SystemExit(f"{timeouts} pipeline timeouts")


if __name__ == "__main__":
    main()
