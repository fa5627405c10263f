"""Host-side logic of bench.py, on the CPU: algorithmic byte counts, the
max-over-ranks timing with two gloo ranks, and the reference arm's rank rule."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes():
    b = bench.algorithmic_bytes()
    assert b["softmax_fwd"][0] == 262_144 and b["softmax_bwd"][0] == 393_216
    assert b["layernorm_fwd"][0] == 37_771_264 and b["layernorm_bwd"][0] == 37_774_336
    assert b["attn_softmax_fwd"][0] == 604_176_384 and b["attn_softmax_bwd"][0] == 805_699_584
    assert b["logsumexp"][0] == 1_648_394_240 and b["softmax_ce"][0] == 3_296_755_720
    assert b["masked_softmax"][0] == 150_994_944 and b["topk_kept"][0] == 134_217_728
    # causal lower triangle: sum over 96 heads of 1024*1025/2 visible entries
    assert (b["attn_softmax_fwd"][0] - 4 * 96 * 1024 * 1024) == 4 * 96 * 1024 * 1025 // 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cpu = torch.device("cpu")
    bench.barrier(dist, cpu)
    local = 1.5 if rank == 0 else 4.25  # per-rank step times (ms)
    q.put((rank, bench.max_over_ranks(local, dist, cpu)))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 4.25, 1: 4.25}


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(3.0, None, torch.device("cpu")) == 3.0


def test_recorded_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    # The committed record is reported while the kernel's sources hash to its
    # fingerprint, and is withheld (None) once any of them changes.
    traffic, rec = bench.recorded_traffic("softmax_ce")
    assert rec is not None and set(rec["sources"]) == {"common.cuh", "pipeline.cuh", "tma_rows.cu"}
    fp_now = bench.kernel_fingerprint(rec["sources"])
    assert (traffic == rec["per_launch_bytes"]) == (fp_now == rec["kernel_fingerprint"])
    stale = dict(rec, kernel_fingerprint="0" * 16)
    p = tmp_path / "dram_traffic.json"
    p.write_text(__import__("json").dumps({"softmax_ce": stale}))
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(p))
    assert bench.recorded_traffic("softmax_ce") == (None, stale)
    assert bench.recorded_traffic("logsumexp") == (None, None)


def test_link_share():
    got = bench.link_share(2e9, 8, 20.0, {"h2d": 200.0, "d2h": 100.0})
    assert got["link_ms"] == 10.0 and got["frac_of_link"] == 0.5
    # both directions at once: the longer one
    got = bench.link_share(2e9, 1.5e9, 20.0, {"h2d": 200.0, "d2h": 100.0})
    assert got["link_ms"] == 15.0 and got["frac_of_link"] == 0.75
