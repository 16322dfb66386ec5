"""The benchmark's one JSON line, as a user or a driver reads it.

The reference arm (the CPU oracle on a tiny sample of the 4-rank workload)
runs here on two host cores; the GPU arm runs the GPT-2-small-sized shard
(psi = 124,439,808, Nd = 8, bf16) for a few steps on a GPU.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
             "cpu_baseline"}


def _run(args, cores: int, timeout: int = 900) -> dict:
    def limit_cores():
        os.sched_setaffinity(0, set(sorted(os.sched_getaffinity(0))[:cores]))

    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args,
                         capture_output=True, text=True, timeout=timeout, cwd=ROOT,
                         preexec_fn=limit_cores)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--config", "c0", "--steps", "2", "--warmup", "3",
              "--ref-sample", "512"], cores=2)
    assert BASE_KEYS <= d.keys()
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "params/s"
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (2, 3, 1)
    assert d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("c0")
    assert d["sample_params_per_step"] == 2 * 512
    # the same config keys and values as the GPU arm prints for this workload
    assert d["config"] == _gpu_arm_config("c0", 0)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def _gpu_arm_config(key: str, rank: int, world: int = 1) -> dict:
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    import synth
    args = argparse.Namespace(config=key, psi=0, nd=0, grad_dtype=None, bucket=0, row_pad=0,
                              gathered="slot")
    return bench.bench_config(args, synth.WORKLOADS[key], rank, world)


def test_config_block_of_the_default_workload():
    c = _gpu_arm_config("c4", 0)
    # rows at a 512-element (1 KB) pitch
    assert (c["psi"], c["nd"], c["shard_params"], c["row_stride_elems"]) == \
        (7_500_000_000, 64, 117_187_500, 117_187_584)
    assert c["grad_dtype"] == "bf16" and c["bucket"] == 500_000_000
    assert c["l2"].startswith("inputs larger than L2 (18.0 GB per step)")
    assert _gpu_arm_config("c0", 0)["l2"].startswith("inputs L2-resident")


@pytest.mark.gpu
def test_gpu_arm_line():
    from zero_sharded_optimizer_02_gb300 import _abi
    d = _run(["--config", "c1", "--steps", "6", "--warmup", "3", "--e2e-steps", "1",
              "--cpu-seconds", "1", "--graph"], cores=4)
    assert BASE_KEYS | {"roofline", "gpu_launches", "clocks"} <= d.keys()
    n = 15_554_976
    assert d["config"]["shard_params"] == n and d["config"]["workload"].startswith("c1")
    assert d["value"] == pytest.approx(n / (d["ms_per_step"] * 1e-3), rel=1e-9)
    assert d["higher_is_better"] is True and d["skipped_steps"] == 0
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9)
    per_step = _abi.fused_launch_count(n, 50_000_000, 0)
    assert r["launches_per_step"] == per_step == 2
    assert r["algorithmic_bytes_per_launch"] == (2 * 8 + 26) * n / per_step
    # the read-only ceiling over the same rows is measured beside the copy peak
    assert r["read_ceiling_gbs"] > 0
    assert r["frac_of_read_ceiling"] == pytest.approx(r["achieved"] / r["read_ceiling_gbs"])
    # --graph: the same back-to-back steps timed as one CUDA graph as well
    assert r["kernel"] == "k_step_fused_ring" and r["kernel_ms_per_step_graph"] > 0
    assert r["frac_graph"] == pytest.approx(
        (2 * 8 + 26) * n / (r["kernel_ms_per_step_graph"] * 1e-3) / 1e9 / r["peak"])
    assert d["config"] == _gpu_arm_config("c1", 0)
    # the other workloads' kernel timings: every target workload but this one
    pc = d["per_config"]
    assert set(pc) == {"c0 rank 0", "c2 rank 0", "c3 rank 0", "c3 rank 1 (flat buffer slot)",
                       "c4 rank 1 (flat buffer slot)"}
    for v in pc.values():
        assert v["skipped"] is False and v["kernel_ms_per_step"] > 0
        assert v["frac"] == pytest.approx(v["achieved"] / r["peak"])
    assert pc["c3 rank 0"]["shard_params"] == 23_437_500
    assert pc["c3 rank 0"]["launches_per_step"] == 3 and "l2" in pc["c0 rank 0"]
    # the 4-rank shard runs on the short-window kernel, and being L2-resident
    # (issued slower than it runs) is also timed as one CUDA graph
    c0 = pc["c0 rank 0"]
    assert c0["kernel"] == "k_step_fused_small" and pc["c3 rank 0"]["kernel"] == "k_step_fused_ring"
    assert c0["kernel_ms_per_step_graph"] > 0
    assert c0["frac_graph"] == pytest.approx(c0["achieved_graph"] / r["peak"])
    # the timed region launches exactly one fused step per timed step
    assert d["gpu_launches"] == 6 * per_step
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 8 * n * 2 and e["d2h_bytes_per_step"] == 2 * n + 4
    # the copy engines' rate varies by box; a copy slower than the zero-copy
    # step is flagged as no bound
    assert e["link"]["frac"] > 0
    assert ("note" in e["link"]) == (e["link"]["frac"] > 1)
    assert set(e["other_forms"]) == {"fed", "sequential", "zero_copy_read_back", "copies_alone"}
    assert all(len(v) == 1 for v in e["ms_per_iteration"].values())
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 4 and cb["value"] > 0
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}


def test_reference_arm_under_torchrun_prints_one_line():
    """With two processes (as the driver launches N > 1) rank 0 alone runs
    the reference arm and prints its line; the other rank exits 0."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--config",
           "c0", "--steps", "1", "--warmup", "3", "--ref-sample", "256"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


@pytest.mark.gpu
def test_gpu_arm_two_processes():
    """The N > 1 choreography of the benchmark (barriers, max over ranks, one
    line from rank 0, whole-job value) with two processes.  One GPU is shared
    through host (gloo) collectives: each process runs its own rank's shard,
    and no kernel waits on the other process."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    env = dict(os.environ, ZERO_DIST_BACKEND="gloo")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--config", "c1", "--steps", "6",
           "--warmup", "3", "--e2e-steps", "1", "--cpu-seconds", "1"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    d = json.loads(lines[0])
    n = 15_554_976
    assert d["n_gpus"] == 2 and d["scaling"] == "weak"
    assert d["value"] == pytest.approx(2 * n / (d["ms_per_step"] * 1e-3), rel=1e-9)
    assert d["config"]["rank"] == 0 and d["skipped_steps"] == 0
    from zero_sharded_optimizer_02_gb300 import _abi
    per_step = _abi.fused_launch_count(n, 50_000_000, 0)
    assert d["gpu_launches"] == 2 * 6 * per_step     # both processes' launches
    assert d["e2e"]["value"] > 0
    assert "cpu_baseline" not in d             # the host-core baseline is timed at N = 1 only
