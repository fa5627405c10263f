"""Benchmark of the row-op hot path on GB300.

One step = one call of every row op, each on its workload at full size:

  softmax_fwd / softmax_bwd   256 x 128
  layernorm_fwd / _bwd        4096 x 768 (dx, dgamma, dbeta)
  attn_softmax_fwd / _bwd     8 x 12 heads x 1024 x 1024, causal, scale 1/8
  logsumexp / softmax_ce      8192 x 50304 (mean loss + logits gradient)
  masked_softmax / topk_kept  262144 x 64, k = 2

The L2 cache is flushed (a 512 MiB write) before every op, outside its CUDA
events, so every op starts cold.  value = algorithmic bytes of all ops (the
minimum each must read and write) / summed device time, in GB/s, over all
ranks.  e2e repeats the steps through the same public calls as a training
step runs them: each step uploads its inputs from pinned host memory (each
once), keeps the intermediates on the device and reads back the mean loss,
all inside the timed region; e2e_every_buffer instead uploads every op's
inputs and reads back every output.  back_to_back times each op launched back to back (no flush, no
events between calls) while cycling through copies of its buffers that total
more than twice the L2: the per-call cost inside a training step, without the
few microseconds that an event pair around a single launch adds.
``--impl reference`` times the CPU oracle instead (see cpu_leg).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (fraction of GB300 peak) and rows/sec per row-op, fp32"
WORKLOAD = ("transformer-step row ops, full sizes: softmax fwd+bwd 256x128; LayerNorm fwd+bwd 4096x768; "
            "causal attention softmax fwd+bwd 8x12x1024x1024; logsumexp + softmax-CE 8192x50304; "
            "masked softmax + top-2 kept mask 262144x64")
FLUSH_BYTES = 512 << 20
L2_BYTES = 126 << 20  # GB300 L2 (the back-to-back sets total more than twice this)


# ---------------------------------------------------------------- workloads

def algorithmic_bytes():
    """Minimum bytes each op must read + write (fp32 = 4 bytes, mask = 1 byte)."""
    r1, c1 = 256, 128
    r2, c2 = 4096, 768
    b, h, s = 8, 12, 1024
    lower = b * h * s * (s + 1) // 2
    full = b * h * s * s
    r4, c4 = 8192, 50304
    r5, c5 = 262144, 64
    return {
        "softmax_fwd": (2 * r1 * c1 * 4, r1),
        "softmax_bwd": (3 * r1 * c1 * 4, r1),
        "layernorm_fwd": (4 * (3 * r2 * c2 + 2 * c2 + r2), r2),
        "layernorm_bwd": (4 * (3 * r2 * c2 + r2 + 3 * c2), r2),
        "attn_softmax_fwd": (4 * (lower + full), b * h * s),
        "attn_softmax_bwd": (4 * (2 * lower + full), b * h * s),
        "logsumexp": (4 * (r4 * c4 + r4), r4),
        "softmax_ce": (4 * (2 * r4 * c4 + r4) + 8, r4),
        "masked_softmax": (9 * r5 * c5, r5),
        "topk_kept": (8 * r5 * c5, r5),
    }


def next_bytes():
    """Algorithmic bytes of the ops reported beside the step."""
    r5, c5, k = 262144, 64, 2
    r2, c2 = 4096, 768
    return {
        "rmsnorm_fwd": (4 * (2 * r2 * c2 + c2 + r2), r2),         # x, gamma read; out, row_rms written
        "rmsnorm_bwd": (4 * (4 * r2 * c2 + c2 + r2), r2),         # dy, x, gamma, row_rms; dx, terms
        "column_sums": (4 * (r2 * c2 + c2), r2),                  # gamma_terms read; dgamma written
        "argmax_onehot": (8 * r5 * c5, r5),             # x read; one-hot written
        "soft_ce": (4 * (3 * r2 * c2 + r2) + 8, r2),    # logits, weights read; grad, row loss, mean
        "teacher_ce": (4 * (3 * r2 * c2 + r2) + 8, r2),  # student, teacher read; grad, row loss, mean
        "router_masked_topk": (13 * r5 * c5, r5),       # x, mask read; p, kept written
        "top_k_rows": (4 * r5 * c5 + 8 * r5 * k, r5),   # x read; values, indices written
    }


def make_inputs():
    from row_wise_softmax_warp_gb300 import inputs
    return {
        "softmax": inputs.softmax_pair(0),
        "layernorm": inputs.layernorm(0),
        "attention": inputs.attention(0),
        "ce": inputs.cross_entropy(0),
        "router": inputs.router(0),
    }


class Ops:
    """Device buffers and one closure per op (the public binding calls)."""

    def __init__(self, data, dev):
        import torch
        import row_wise_softmax_warp_gb300 as ro
        self.ro = ro
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        d = data["softmax"]
        self.sx, self.sdy = t(d["x"]), t(d["dy"])
        self.sy, self.sdx = torch.empty_like(self.sx), torch.empty_like(self.sx)
        n = data["layernorm"]
        self.eps = n["eps"]
        self.lx, self.lg, self.lb, self.ldy = t(n["x"]), t(n["gamma"]), t(n["beta"]), t(n["dy"])
        self.lout, self.lxh = torch.empty_like(self.lx), torch.empty_like(self.lx)
        self.lrs = torch.empty(self.lx.shape[0], device=dev)
        self.ldx = torch.empty_like(self.lx)
        self.ldg, self.ldb = torch.empty_like(self.lg), torch.empty_like(self.lg)
        self.lws = torch.empty(ro.rowops_layernorm_bwd_workspace(*self.lx.shape), dtype=torch.uint8, device=dev)
        a = data["attention"]
        self.seq, self.scale = a["seq_len"], a["scale"]
        self.as_, self.adp = t(a["scores"]), t(a["dp"])
        self.ap, self.ads = torch.empty_like(self.as_), torch.empty_like(self.as_)
        c = data["ce"]
        self.cx, self.ct, self.cgs = t(c["logits"]), t(c["targets"]), c["grad_scale"]
        self.clse = torch.empty(self.cx.shape[0], device=dev)
        self.cg = torch.empty_like(self.cx)
        self.crl = torch.empty(self.cx.shape[0], device=dev)
        self.cml = torch.empty(1, dtype=torch.float64, device=dev)
        r = data["router"]
        self.rx, self.rm, self.k = t(r["x"]), t(r["mask"]), r["k"]
        self.rp, self.rk = torch.empty_like(self.rx), torch.empty_like(self.rx)

    def table(self):
        ro = self.ro
        return [
            ("softmax_fwd", lambda: ro.rowops_softmax_fwd(self.sx, self.sy)),
            ("softmax_bwd", lambda: ro.rowops_softmax_bwd(self.sy, self.sdy, self.sdx)),
            ("layernorm_fwd", lambda: ro.rowops_layernorm_fwd(self.lx, self.lg, self.lb, self.lout, self.lxh,
                                                              self.lrs, eps=self.eps)),
            ("layernorm_bwd", lambda: ro.rowops_layernorm_bwd(self.ldy, self.lg, self.lxh, self.lrs, self.ldx,
                                                              self.ldg, self.ldb, workspace=self.lws)),
            ("attn_softmax_fwd", lambda: ro.rowops_attn_softmax_fwd(self.as_, self.ap, seq_len=self.seq,
                                                                    scale=self.scale)),
            ("attn_softmax_bwd", lambda: ro.rowops_attn_softmax_bwd(self.ap, self.adp, self.ads,
                                                                    seq_len=self.seq, scale=self.scale)),
            ("logsumexp", lambda: ro.rowops_logsumexp(self.cx, self.clse)),
            ("softmax_ce", lambda: ro.rowops_softmax_ce(self.cx, self.ct, self.cg, self.crl, self.cml,
                                                        grad_scale=self.cgs)),
            ("masked_softmax", lambda: ro.rowops_masked_softmax(self.rx, self.rm, self.rp)),
            ("topk_kept", lambda: ro.rowops_topk_kept(self.rp, self.k, self.rk)),
        ]

    def next_table(self):
        """Ops beyond the step (reported separately): the fused router on the
        router workload and top_k_rows (k = 2, largest) on its logits."""
        ro = self.ro
        if not hasattr(self, "fp"):
            import torch
            self.fp, self.fk = torch.empty_like(self.rx), torch.empty_like(self.rx)
            shape = (self.rx.shape[0], self.k)
            self.tv = torch.empty(shape, device=self.rx.device)
            self.ti = torch.empty(shape, device=self.rx.device)
        if not hasattr(self, "rms_out"):
            import torch
            self.rms_out, self.rms_r = torch.empty_like(self.lx), torch.empty(self.lx.shape[0], device=self.lx.device)
            self.rms_dx, self.rms_t = torch.empty_like(self.lx), torch.empty_like(self.lx)
            self.rms_dg = torch.empty_like(self.lg)
            ro.rowops_rmsnorm_fwd(self.lx, self.lg, self.rms_out, self.rms_r, eps=self.eps)
            self.ldy_soft = torch.softmax(self.ldy, dim=1)  # soft targets for the weighted-logits CE
        return [
            ("rmsnorm_fwd", lambda: ro.rowops_rmsnorm_fwd(self.lx, self.lg, self.rms_out, self.rms_r, eps=self.eps)),
            ("rmsnorm_bwd", lambda: ro.rowops_rmsnorm_bwd(self.ldy, self.lg, self.lx, self.rms_r, self.rms_dx,
                                                          self.rms_t)),
            ("column_sums", lambda: ro.rowops_column_sums(self.rms_t, self.rms_dg)),
            ("argmax_onehot", lambda: ro.rowops_argmax_onehot(self.rx, self.fk)),
            ("soft_ce", lambda: ro.rowops_soft_ce(self.lx, self.ldy_soft, self.rms_dx, self.rms_r, self.cml)),
            ("teacher_ce", lambda: ro.rowops_teacher_ce(self.lx, self.ldy, self.rms_dx, self.rms_r, self.cml)),
            ("router_masked_topk", lambda: ro.rowops_router_masked_topk(self.rx, self.rm, self.k, self.fp, self.fk)),
            ("top_k_rows", lambda: ro.rowops_top_k_rows(self.rx, self.k, True, self.tv, self.ti)),
        ]

    def next_io(self):
        """Per op beyond the step: (device inputs, device outputs) of its call."""
        return {
            "rmsnorm_fwd": ([self.lx, self.lg], [self.rms_out, self.rms_r]),
            "rmsnorm_bwd": ([self.ldy, self.lg, self.lx, self.rms_r], [self.rms_dx, self.rms_t]),
            "column_sums": ([self.rms_t], [self.rms_dg]),
            "argmax_onehot": ([self.rx], [self.fk]),
            "soft_ce": ([self.lx, self.ldy_soft], [self.rms_dx, self.rms_r, self.cml]),
            "teacher_ce": ([self.lx, self.ldy], [self.rms_dx, self.rms_r, self.cml]),
            "router_masked_topk": ([self.rx, self.rm], [self.fp, self.fk]),
            "top_k_rows": ([self.rx], [self.tv, self.ti]),
        }

    def e2e_io(self):
        """Per op: (device inputs, device outputs) that an end-to-end call moves."""
        return {
            "softmax_fwd": ([self.sx], [self.sy]),
            "softmax_bwd": ([self.sy, self.sdy], [self.sdx]),
            "layernorm_fwd": ([self.lx, self.lg, self.lb], [self.lout, self.lxh, self.lrs]),
            "layernorm_bwd": ([self.ldy, self.lg, self.lxh, self.lrs], [self.ldx, self.ldg, self.ldb]),
            "attn_softmax_fwd": ([self.as_], [self.ap]),
            "attn_softmax_bwd": ([self.ap, self.adp], [self.ads]),
            "logsumexp": ([self.cx], [self.clse]),
            "softmax_ce": ([self.cx, self.ct], [self.cg, self.crl, self.cml]),
            "masked_softmax": ([self.rx, self.rm], [self.rp]),
            "topk_kept": ([self.rp], [self.rk]),
        }


def back_to_back(ops, dev, stream, l2_bytes, calls_min=40, table="table", io_name="e2e_io"):
    """Per-call ms of each op of ops.<table>() launched back to back, as in a
    training step, with no flush and no events between the calls (the calls
    replayed as one CUDA graph).  Each op cycles through copies of its own
    buffers (ops.<io_name>()) whose total exceeds twice the L2, so every call
    still finds its inputs outside the L2.  Returns ({op: ms}, {op: sets})."""
    import copy
    import torch
    io = getattr(ops, io_name)()
    names = [n for n, _ in getattr(ops, table)()]
    per_call, sets_used = {}, {}
    for idx, name in enumerate(names):
        ins, outs = io[name]
        tensors = ins + outs
        footprint = sum(t.numel() * t.element_size() for t in tensors)
        n_sets = max(1, -(-2 * l2_bytes // footprint))
        fns = []
        for s_ in range(n_sets):
            twin = copy.copy(ops)
            if s_ > 0:  # fresh buffers for this op's arguments (inputs keep their values)
                for attr, val in vars(ops).items():
                    if any(val is t for t in ins):
                        setattr(twin, attr, val.clone())
                    elif any(val is t for t in outs):
                        setattr(twin, attr, torch.empty_like(val))
            fns.append(getattr(twin, table)()[idx][1])
        calls = max(calls_min, n_sets)
        for f in fns:  # warm-up: every set once
            f()
        torch.cuda.synchronize()
        # The calls are captured once as a CUDA graph and replayed, so that the
        # host's per-call cost (argument checks in Python, the launch itself)
        # does not starve the GPU between small kernels.
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            for i in range(calls):
                fns[i % n_sets]()
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        per_call[name] = a.elapsed_time(b) / calls
        sets_used[name] = n_sets
        del fns, graph
        torch.cuda.empty_cache()
    return per_call, sets_used


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while running (read-only queries)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.rows, self.proc, self.uuid = [], None, uuid
        self.mark = False

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((self.mark, parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        loaded = [p for m, p in self.rows if m] or [p for _, p in self.rows]
        if not loaded:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(p[1]) for p in loaded if num(p[1]) is not None]
        mx = [num(p[2]) for p in loaded if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in loaded for i in range(4) if p[5 + i].lower() == "active"})
        power = [num(p[3]) for p in loaded if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(loaded),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "dram_traffic.json")


def _traffic_records():
    if not os.path.exists(TRAFFIC_RECORD):
        return {}
    with open(TRAFFIC_RECORD) as f:
        return json.load(f)


def kernel_fingerprint(sources):
    """First 16 hex digits of the SHA-256 of the named csrc files (sorted by name)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_wise_softmax_warp_gb300", "csrc")
    for name in sorted(sources):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(op):
    """(DRAM read + write bytes per launch, the record) from the committed ncu
    record profiles/dram_traffic.json, if it was taken on the current sources
    of the op's kernel; else (None, the record or None)."""
    rec = _traffic_records().get(op)
    if not rec:
        return None, None
    if kernel_fingerprint(rec["sources"]) != rec["kernel_fingerprint"]:
        return None, rec
    return int(rec["per_launch_bytes"]), rec


def link_rates(dev, nbytes, reps=3):
    """Pinned host <-> device copy rates (GB/s) of one plain copy_ of nbytes
    (capped at 1 GiB), best of reps, CUDA events on the current stream."""
    import torch
    n = int(min(nbytes, 1 << 30))
    host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    devb = torch.empty(n, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d", devb, host), ("d2h", host, devb)):
        best = None
        for _ in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        out[name] = n / (best * 1e-3) / 1e9
    del host, devb
    return out, n


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend)
    return dist.get_rank(), dist.get_world_size(), dist


def max_over_ranks(x, dist, device):
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device):
    if dist is not None:
        import torch
        dist.barrier(device_ids=[device.index]) if device.type == "cuda" else dist.barrier()


# ----------------------------------------------------------------- GPU arm

class PinnedSlab:
    """Host buffers for the end-to-end steps as views of one pinned allocation
    (each view on a 256-byte boundary).  On GB300 a pinned buffer per input,
    from torch's caching host allocator, gave 12.2 to 18.8 ms for the same
    step on one box; views of one allocation gave 12.2 ms every time."""

    def __init__(self, tensors):
        import torch
        sizes = [(t.numel() * t.element_size() + 255) // 256 * 256 for t in tensors]
        self.buf = torch.empty(max(sum(sizes), 1), dtype=torch.uint8, pin_memory=True)
        self.off = 0

    def like(self, t, copy=False):
        nb = t.numel() * t.element_size()
        v = self.buf[self.off:self.off + nb].view(t.dtype).view(t.shape)
        self.off += (nb + 255) // 256 * 256
        if copy:
            v.copy_(t)
        return v


def e2e_every_buffer(ops, dev, stream, ke, dist):
    """End-to-end steps in which every op's inputs come from pinned host memory
    and every output goes back, per op.  Transfers run on two copy streams (one
    per direction) and compute on the launching stream, ordered by events, so
    op i's inputs travel while op i-1 computes and op i-2's outputs return.
    Returns (ms per step, H2D bytes, D2H bytes)."""
    import torch
    table = ops.table()
    io = ops.e2e_io()
    names = [n for n, _ in table]
    slab = PinnedSlab([x for n in names for x in io[n][0] + io[n][1]])
    pinned_in = {n: [slab.like(x, copy=True) for x in io[n][0]] for n in names}
    pinned_out = {n: [slab.like(x) for x in io[n][1]] for n in names}
    h2d = sum(x.numel() * x.element_size() for n in names for x in io[n][0])
    d2h = sum(x.numel() * x.element_size() for n in names for x in io[n][1])
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = {n: ev() for n in names}
    computed = {n: ev() for n in names}
    out_done = {n: ev() for n in names}
    for n in names:  # mark all as complete once, so the first step's waits pass
        computed[n].record(stream)
        out_done[n].record(stream)

    def step():
        for name, fn in table:
            with torch.cuda.stream(s_in):
                s_in.wait_event(computed[name])  # last step's op finished reading its inputs
                for dst, src in zip(io[name][0], pinned_in[name]):
                    dst.copy_(src, non_blocking=True)
                in_ready[name].record(s_in)
            stream.wait_event(in_ready[name])
            stream.wait_event(out_done[name])  # last step's outputs are home
            fn()
            computed[name].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[name])
                for dst, src in zip(pinned_out[name], io[name][1]):
                    dst.copy_(src, non_blocking=True)
                out_done[name].record(s_out)

    step()
    torch.cuda.synchronize()
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(ke):
        step()
    for n in names:
        stream.wait_event(out_done[n])
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / ke, h2d, d2h


def e2e_step_inputs(ops, dev, stream, ke, dist):
    """End-to-end steps as a training step runs them: the step's inputs come
    from pinned host memory, each uploaded once per step just before its first
    use; intermediates stay on the device (softmax y, LayerNorm xhat and
    inv_std, attention P, router P); the step's result, the mean
    cross-entropy loss, is read back.  The upload of an input for the next
    step waits until this step's last op reading it has run.  Returns
    (ms per step, H2D bytes, D2H bytes)."""
    import torch
    table = ops.table()
    names = [n for n, _ in table]
    # external inputs, by the op that first reads them, and their last reader
    first = {"softmax_fwd": [ops.sx], "softmax_bwd": [ops.sdy], "layernorm_fwd": [ops.lx, ops.lg, ops.lb],
             "layernorm_bwd": [ops.ldy], "attn_softmax_fwd": [ops.as_], "attn_softmax_bwd": [ops.adp],
             "logsumexp": [ops.cx], "softmax_ce": [ops.ct], "masked_softmax": [ops.rx, ops.rm], "topk_kept": []}
    last = {id(ops.sx): "softmax_fwd", id(ops.sdy): "softmax_bwd", id(ops.lx): "layernorm_fwd",
            id(ops.lg): "layernorm_bwd", id(ops.lb): "layernorm_fwd", id(ops.ldy): "layernorm_bwd",
            id(ops.as_): "attn_softmax_fwd", id(ops.adp): "attn_softmax_bwd", id(ops.cx): "softmax_ce",
            id(ops.ct): "softmax_ce", id(ops.rx): "masked_softmax", id(ops.rm): "masked_softmax"}
    results = {"softmax_ce": [ops.cml]}
    slab = PinnedSlab([x for n in names for x in first[n] + results.get(n, [])])
    pinned_in = {n: [slab.like(x, copy=True) for x in first[n]] for n in names}
    pinned_out = {n: [slab.like(x) for x in results.get(n, [])] for n in names}
    h2d = sum(x.numel() * x.element_size() for n in names for x in first[n])
    d2h = sum(x.numel() * x.element_size() for n in names for x in results.get(n, []))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = {n: ev() for n in names}
    computed = {n: ev() for n in names}
    out_done = {n: ev() for n in names}
    for n in names:  # mark all as complete once, so the first step's waits pass
        computed[n].record(stream)
        out_done[n].record(stream)

    def step():
        for name, fn in table:
            with torch.cuda.stream(s_in):
                for dst, src in zip(first[name], pinned_in[name]):
                    s_in.wait_event(computed[last[id(dst)]])  # last step's readers are done with it
                    dst.copy_(src, non_blocking=True)
                in_ready[name].record(s_in)
            stream.wait_event(in_ready[name])
            stream.wait_event(out_done[name])  # last step's result is home
            fn()
            computed[name].record(stream)
            if pinned_out[name]:
                with torch.cuda.stream(s_out):
                    s_out.wait_event(computed[name])
                    for dst, src in zip(pinned_out[name], results[name]):
                        dst.copy_(src, non_blocking=True)
                    out_done[name].record(s_out)

    step()
    torch.cuda.synchronize()
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(ke):
        step()
    for n in names:
        stream.wait_event(out_done[n])
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / ke, h2d, d2h


def gpu_leg(args):
    import torch
    rank, world, dist = dist_setup()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from row_wise_softmax_warp_gb300 import build
    build.build()
    import row_wise_softmax_warp_gb300 as ro
    ro.library()

    data = make_inputs()
    ops = Ops(data, dev)
    table = ops.table()
    abytes = algorithmic_bytes()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sink = torch.empty((), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        # A write larger than the L2 evicts the previous op's data (written
        # back here); a read larger than the L2 then leaves it holding only
        # clean lines, so the op's events do not include writing back the
        # flush (on GB300 up to 126 MB: logsumexp 247.5 -> 232.4 us).
        flush.zero_()
        torch.sum(clean.view(torch.int64), 0, out=sink)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()

    for _ in range(args.warmup):
        for _, fn in table:
            flush_l2()
            fn()
    torch.cuda.synchronize()

    K = args.steps
    starts = {n: [torch.cuda.Event(enable_timing=True) for _ in range(K)] for n, _ in table}
    ends = {n: [torch.cuda.Event(enable_timing=True) for _ in range(K)] for n, _ in table}
    outer0, outer1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize()
    clocks.mark = True
    launches0 = ro.rowops_kernel_launches()
    outer0.record(stream)
    for k in range(K):
        for name, fn in table:
            flush_l2()
            starts[name][k].record(stream)
            fn()
            ends[name][k].record(stream)
    outer1.record(stream)
    torch.cuda.synchronize()
    launches = ro.rowops_kernel_launches() - launches0
    barrier(dist, dev)
    per_op_ms = {n: sum(starts[n][k].elapsed_time(ends[n][k]) for k in range(K)) / K for n, _ in table}
    step_ms_local = sum(per_op_ms.values())
    wall_ms_local = outer0.elapsed_time(outer1) / K

    # The same ops after the write alone (the flush's dirty lines are then
    # written back inside each op's events), for comparison.
    kd = max(3, min(K, 20))
    dirty_ev = []
    for _ in range(kd):
        for name, fn in table:
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            dirty_ev.append((name, a, b))
    torch.cuda.synchronize()
    dirty_ms = {n: 0.0 for n, _ in table}
    for name, a, b in dirty_ev:
        dirty_ms[name] += a.elapsed_time(b) / kd
    dirty_step_ms_local = sum(dirty_ms.values())

    # ------------------------------------------- ops beyond the step
    nxt = ops.next_table()
    for _, fn in nxt:
        for _ in range(3):
            flush_l2()
            fn()
    next_ms = {}
    for name, fn in nxt:
        ts = []
        for _ in range(max(5, min(K, 20))):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        next_ms[name] = sum(a.elapsed_time(b) for a, b in ts) / len(ts)

    # ------------------------------------------- the step ops back to back
    b2b_ms, b2b_sets, next_b2b_ms = {}, {}, {}
    if not args.no_back_to_back:
        b2b_ms_local, b2b_sets = back_to_back(ops, dev, stream, L2_BYTES)
        b2b_ms = {n: max_over_ranks(b2b_ms_local[n], dist, dev) for n in b2b_ms_local}
        nb_local, _ = back_to_back(ops, dev, stream, L2_BYTES, table="next_table", io_name="next_io")
        next_b2b_ms = {n: max_over_ranks(nb_local[n], dist, dev) for n in nb_local}

    # ------------------------------------------------ the step as a CUDA graph
    # The ten calls captured once and replayed: no host work per launch and no
    # gaps between kernels.  L2 is flushed before each replay but not between
    # the ops inside it, so an op may find its predecessor's outputs in L2 (as
    # it would in a real step).  Reported beside the per-op figures.
    graph_step = None
    try:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            for _, fn in table:
                fn()
        stream.wait_stream(cap)
        for _ in range(3):
            flush_l2()
            graph.replay()
        ts = []
        for _ in range(max(5, min(K, 20))):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        graph_ms_local = sum(a.elapsed_time(b) for a, b in ts) / len(ts)
        graph_step = {"ms": max_over_ranks(graph_ms_local, dist, dev), "replays": len(ts)}
        del graph
    except RuntimeError as e:  # capture refused: report it, keep the rest of the line
        graph_step = {"unavailable": str(e).splitlines()[0][:200]}

    # ------------------------------------------------------------ e2e
    ke = max(1, args.e2e_steps if args.e2e_steps else K)
    ops2 = Ops(data, dev)
    e2e_ms_local, h2d, d2h = e2e_step_inputs(ops2, dev, stream, ke, dist)
    all_ms_local, all_h2d, all_d2h = e2e_every_buffer(ops2, dev, stream, ke, dist)
    del ops2
    torch.cuda.empty_cache()
    link, link_n = link_rates(dev, h2d)
    clocks.mark = False
    clocks.stop()

    step_ms = max_over_ranks(step_ms_local, dist, dev)
    dirty_step_ms = max_over_ranks(dirty_step_ms_local, dist, dev)
    e2e_ms = max_over_ranks(e2e_ms_local, dist, dev)
    all_ms = max_over_ranks(all_ms_local, dist, dev)
    wall_ms = max_over_ranks(wall_ms_local, dist, dev)
    per_op = {n: max_over_ranks(per_op_ms[n], dist, dev) for n, _ in table}
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peak, peak_kind = peaks()
    total_bytes = sum(b for b, _ in abytes.values())
    value = world * total_bytes / (step_ms * 1e-3) / 1e9
    breakdown = {}
    for n, _ in table:
        b, rows = abytes[n]
        gbs = b / (per_op[n] * 1e-3) / 1e9
        breakdown[n] = {"ms": round(per_op[n], 5), "GB/s": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
                        "frac_of_8TBs": round(gbs / 8000.0, 4), "rows_per_s": round(rows / (per_op[n] * 1e-3), 1),
                        "alg_bytes": b}
    top = max(per_op, key=per_op.get)
    top_gbs = abytes[top][0] / (per_op[top] * 1e-3) / 1e9
    traffic, rec = recorded_traffic(top)
    roofline = {"bound": "hbm", "kernel": top, "achieved": round(top_gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(top_gbs / peak, 4), "peak_kind": peak_kind, "traffic": traffic,
                "traffic_source": "profiles/dram_traffic.json (ncu dram__bytes_read.sum + dram__bytes_write.sum)"
                if rec else None}
    if rec and traffic is None:
        roofline["traffic_note"] = "null: the kernel's sources changed since the recorded capture"
    if rec:
        unwritten = rec["algorithmic_bytes"] - rec["per_launch_bytes"]
        if unwritten > 0:
            roofline["traffic_note"] = (
                f"the capture's DRAM writes fall {unwritten / 1e6:.0f} MB short of the algorithmic bytes: that much "
                "output is still dirty in the L2 when the isolated launch ends and is written back after its "
                "events; the back-to-back fraction pays for it")
    if top in b2b_ms:
        roofline["frac_back_to_back"] = round(abytes[top][0] / (b2b_ms[top] * 1e-3) / 1e9 / peak, 4)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64, the five workloads' distributions)",
        "config": {"workload": WORKLOAD,
                   "l2": "flushed before every op, outside the op's events: a 512 MiB device write, then a "
                         "512 MiB read, so the L2 holds only clean lines when the op starts",
                   "ms_per_step_incl_flushes": round(wall_ms, 4), "parallelism": f"replicas x{world} (rows independent)"},
        "roofline": roofline,
        "ops": breakdown,
        "gpu_launches": int(launches),
        "next_ops": {n: {"ms": round(next_ms[n], 5), "alg_bytes": next_bytes()[n][0],
                         "GB/s": round(next_bytes()[n][0] / (next_ms[n] * 1e-3) / 1e9, 1),
                         "frac_of_measured": round(next_bytes()[n][0] / (next_ms[n] * 1e-3) / 1e9 / peak, 4),
                         **({"back_to_back_ms": round(next_b2b_ms[n], 5),
                             "back_to_back_frac_of_measured":
                                 round(next_bytes()[n][0] / (next_b2b_ms[n] * 1e-3) / 1e9 / peak, 4)}
                            if n in next_b2b_ms else {})}
                     for n in next_ms},
        "e2e": {"value": round(world * total_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_ms, 3), "steps": ke,
                "note": "each step uploads the step's inputs (each once), keeps the intermediates on the "
                        "device (softmax y, LayerNorm xhat/inv_std, attention P, router P) and reads back "
                        "the mean cross-entropy loss",
                **link_share(h2d, d2h, e2e_ms, link)},
        "host_link": {"h2d_GB/s": round(link["h2d"], 1), "d2h_GB/s": round(link["d2h"], 1), "bytes": link_n,
                      "note": "one plain pinned copy_ each way (best of 3); link_ms below is the step's copies "
                              "at these rates (the longer direction: both run at once), "
                              "frac_of_link = link_ms / ms_per_step"},
        "e2e_every_buffer": {"value": round(world * total_bytes / (all_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                             "h2d_bytes_per_step": int(all_h2d), "d2h_bytes_per_step": int(all_d2h),
                             "ms_per_step": round(all_ms, 3), "steps": ke,
                             "note": "every op's inputs uploaded and every output read back, per op",
                             **link_share(all_h2d, all_d2h, all_ms, link)},
        "clocks": clocks.summary(),
        "l2_write_only_flush": {
            "ms_per_step": round(dirty_step_ms, 5),
            "GB/s": round(world * total_bytes / (dirty_step_ms * 1e-3) / 1e9, 1),
            "ops_ms": {n: round(v, 5) for n, v in dirty_ms.items()},
            "note": "the same ops after the 512 MiB write alone: each op's events then also include "
                    "writing back the dirty lines the flush left in the L2"},
    }
    if graph_step is not None and "ms" in graph_step:
        gms = graph_step["ms"]
        line["graph_step"] = {"ms": round(gms, 5), "GB/s": round(world * total_bytes / (gms * 1e-3) / 1e9, 1),
                              "replays": graph_step["replays"],
                              "note": "the ten calls as one CUDA graph; L2 flushed before each replay, "
                                      "not between the ops inside it"}
    elif graph_step is not None:
        line["graph_step"] = graph_step
    b2b_total = sum(b2b_ms.values())
    if b2b_ms:
        line["back_to_back"] = {
            "ms_per_step": round(b2b_total, 5),
            "GB/s": round(world * total_bytes / (b2b_total * 1e-3) / 1e9, 1),
            "ops": {n: {"ms": round(b2b_ms[n], 5),
                        "GB/s": round(abytes[n][0] / (b2b_ms[n] * 1e-3) / 1e9, 1),
                        "frac_of_measured": round(abytes[n][0] / (b2b_ms[n] * 1e-3) / 1e9 / peak, 4),
                        "buffer_sets": b2b_sets[n]} for n in b2b_ms},
            "note": "each op's calls replayed back to back as one CUDA graph (no flush, no events between "
                    "calls), cycling through copies of its buffers that total more than twice the L2",
        }
    if not args.no_cpu_baseline and world == 1:  # the CPU baseline belongs to the N = 1 line
        line["cpu_baseline"] = cpu_leg(data, budget_s=args.cpu_seconds)
        one = cpu_leg(data, budget_s=args.cpu_seconds / 6, n_threads=1)
        line["cpu_baseline"]["single_thread"] = {k: one[k] for k in ("value", "unit", "seconds", "sample")}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def link_share(h2d, d2h, ms, link):
    """The time a step's copies take at the measured link rates, and its share
    of the step.  The two directions run on separate copy streams at once, so
    the copies take the longer of the two."""
    link_ms = max(h2d / link["h2d"], d2h / link["d2h"]) / 1e6
    return {"link_ms": round(link_ms, 3), "frac_of_link": round(link_ms / ms, 4)}


# ----------------------------------------------------------------- CPU leg

def cpu_leg(data, budget_s=12.0, n_threads=None):
    """Times the double-precision oracle (as it stands) on all host cores (or
    `n_threads` of them), on a bounded, deterministic sample of each workload's
    rows; returns GB/s of the same algorithmic bytes per processed row."""
    import oracle
    threads = n_threads or oracle.threads()
    nt = threads
    share = budget_s / 10.0  # seconds of work per op, roughly
    results = []

    def run(name, fn, row_bytes, rows_total, probe_rows):
        # size the sample from a short probe so each op takes about `share` seconds
        t0 = time.perf_counter()
        fn(0, probe_rows)
        dt = max(time.perf_counter() - t0, 1e-6)
        n = int(min(rows_total, max(probe_rows, probe_rows * share / dt)))
        t0 = time.perf_counter()
        fn(0, n)
        dt = time.perf_counter() - t0
        results.append((name, n, row_bytes(0, n), dt))

    d = data["softmax"]
    y32 = oracle.softmax_rows(d["x"]).astype(np.float32)
    run("softmax_fwd", lambda a, b: oracle.softmax_rows(d["x"][a:b], n_threads=nt),
        lambda a, b: (b - a) * 128 * 8, 256, 256)
    run("softmax_bwd", lambda a, b: oracle.softmax_rows_backward(y32[a:b], d["dy"][a:b], n_threads=nt),
        lambda a, b: (b - a) * 128 * 12, 256, 256)
    n = data["layernorm"]
    run("layernorm_fwd",
        lambda a, b: oracle.layernorm_forward(n["x"][a:b], n["gamma"], n["beta"], n["eps"], n_threads=nt),
        lambda a, b: (b - a) * (768 * 12 + 4), 4096, 256)
    _, xh, rs = oracle.layernorm_forward(n["x"], n["gamma"], n["beta"], n["eps"])
    xh32, rs32 = xh.astype(np.float32), rs.astype(np.float32)
    run("layernorm_bwd",
        lambda a, b: oracle.layernorm_backward(n["dy"][a:b], n["gamma"], xh32[a:b], rs32[a:b], n_threads=nt),
        lambda a, b: (b - a) * (768 * 12 + 4), 4096, 256)
    at = data["attention"]
    S, sc = at["seq_len"], at["scale"]

    def attn_bytes(a, b, reads):
        q = np.arange(a, b) % S
        return int(4 * (reads * (q + 1).sum() + (b - a) * S))
    run("attn_softmax_fwd",
        lambda a, b: oracle.attn_softmax_forward(at["scores"][a:b], S, sc, row0=a, n_threads=nt),
        lambda a, b: attn_bytes(a, b, 1), at["scores"].shape[0], 1024)
    run("attn_softmax_bwd",
        lambda a, b: oracle.attn_softmax_backward(at["scores"][a:b], at["dp"][a:b], S, sc, row0=a, n_threads=nt),
        lambda a, b: attn_bytes(a, b, 2), at["scores"].shape[0], 1024)
    c = data["ce"]
    run("logsumexp", lambda a, b: oracle.logsumexp_rows(c["logits"][a:b], n_threads=nt),
        lambda a, b: (b - a) * (50304 * 4 + 4), 8192, 16)
    run("softmax_ce",
        lambda a, b: oracle.softmax_cross_entropy(c["logits"][a:b], c["targets"][a:b], 1 / 8192, n_threads=nt),
        lambda a, b: (b - a) * (50304 * 8 + 4), 8192, 16)
    r = data["router"]
    run("masked_softmax", lambda a, b: oracle.masked_softmax(r["x"][a:b], r["mask"][a:b], n_threads=nt),
        lambda a, b: (b - a) * 64 * 9, 262144, 8192)
    run("topk_kept", lambda a, b: oracle.topk_kept(r["x"][a:b], 2, n_threads=nt),
        lambda a, b: (b - a) * 64 * 8, 262144, 8192)
    tot_b = sum(x[2] for x in results)
    tot_t = sum(x[3] for x in results)
    full = {"softmax_fwd": 256, "softmax_bwd": 256, "layernorm_fwd": 4096, "layernorm_bwd": 4096,
            "attn_softmax_fwd": at["scores"].shape[0], "attn_softmax_bwd": at["scores"].shape[0],
            "logsumexp": 8192, "softmax_ce": 8192, "masked_softmax": 262144, "topk_kept": 262144}
    cores = "one host core" if threads == 1 else "all host cores" if n_threads is None else f"{threads} host cores"
    if all(k == full[n] for n, k, _, _ in results):
        sample = "the whole workload of every op (double-precision C oracle, " + cores + ")"
    else:
        sample = "; ".join(f"{n}: {k} of {full[n]} rows" for n, k, _, _ in results) + \
                 " (first rows of each workload, double-precision C oracle, " + cores + ")"
    return {"value": round(tot_b / tot_t / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": round(tot_t, 2), "sample": sample}


def reference_leg(args):
    """--impl reference: the CPU oracle as the reference arm (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    data = make_inputs()
    # Per-step sample budget, smaller for long runs so that --steps K --warmup W
    # stays within a few minutes of CPU work.
    budget = min(args.ref_step_seconds, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_leg(data, budget_s=min(1.0, budget))
    vals, secs, last = [], 0.0, None
    for _ in range(args.steps):
        last = cpu_leg(data, budget_s=budget)
        vals.append(last["value"])
        secs += last["seconds"]
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * secs / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy PCG64)",
        "config": {"workload": WORKLOAD, "sample": "bounded row sample per op, see cpu_baseline"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=0, help="end-to-end steps (default: --steps)")
    ap.add_argument("--cpu-seconds", type=float, default=30.0)
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-back-to-back", action="store_true",
                    help="skip the back-to-back figures (shorter launch lists under a profiler)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        reference_leg(args)
    else:
        gpu_leg(args)


if __name__ == "__main__":
    main()
