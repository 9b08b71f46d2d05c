"""bench.py's host side, without a GPU.

- The reference arm (the CPU oracle, timed on the host) prints one JSON line
  with the keys of the benchmark line, for the GEMM step and for attention.
- The multi-rank helpers: with two gloo ranks on 127.0.0.1, the timing
  barrier completes, the step time is the max over ranks on every rank, and
  only rank 0 runs and prints the reference arm.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
        "e2e"}


@pytest.mark.parametrize("workload,metric", [("step", bench.METRIC), ("attn", bench.ATTN_METRIC)])
def test_reference_arm_line(workload, metric):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", workload, "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert KEYS <= set(line), KEYS - set(line)
    assert line["impl"] == "reference" and line["metric"] == metric
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = b.dist_env()
        b.barrier(w)
        m = b.max_over_ranks(1.5 + r, w)
        results[rank] = (w, r, m)
    finally:
        dist.destroy_process_group()


def test_multi_rank_helpers_gloo():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    with mp.Manager() as manager:
        results = manager.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    assert got[0] == (2, 0, 2.5) and got[1] == (2, 1, 2.5)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import argparse
    ns = argparse.Namespace(gpus=2, steps=1, warmup=3, workload="step", shape=None, split=1,
                            no_streamk=False, attn_shape=None)
    assert bench.run_reference(ns, 2, 1) == 0
    ns.workload = "attn"
    assert bench.run_reference_attention(ns, 2, 1) == 0
    assert capsys.readouterr().out == ""


def test_traffic_hash_covers_every_kernel_source():
    """Every CUDA source of the library is in the hash that keys the stored
    DRAM traffic figures, so no kernel can change without voiding them."""
    csrc = os.path.join(ROOT, "tiled_tensor_core_03_gb300", "csrc")
    sources = {f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh"))}
    assert sources == set(bench.KERNEL_SOURCES)


def test_traffic_reported_only_for_the_captured_sources(monkeypatch):
    key = next(iter(bench.TRAFFIC_CAPTURE["bytes"]))
    cur = bench.kernel_source_hash()
    monkeypatch.setitem(bench.TRAFFIC_CAPTURE, "source_hash", cur)
    value, note = bench.traffic_for(key)
    assert value == bench.TRAFFIC_CAPTURE["bytes"][key] and cur in note
    assert bench.traffic_for(("fused", 3, 5, 7))[0] is None           # shape never captured
    monkeypatch.setitem(bench.TRAFFIC_CAPTURE, "source_hash", "0" * 16)
    value, note = bench.traffic_for(key)
    assert value is None and "changed" in note
    monkeypatch.setitem(bench.TRAFFIC_CAPTURE, "source_hash", None)
    assert bench.traffic_for(key)[0] is None
