"""Host-side checks of bench.py (no GPU): the unmasked-pair count behind every TFLOP/s
figure, the reference arm (the fp64 oracle) end to end, and the max-over-ranks timing
reduction of the multi-process path on two gloo ranks."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("S", [1, 2, 7, 64, 130])
@pytest.mark.parametrize("causal,window", [(True, -1), (True, 0), (True, 5), (True, 129), (False, -1)])
def test_n_pairs_matches_brute_force(S, causal, window):
    brute = sum(1 for i in range(S) for j in range(S)
                if (not causal or j <= i) and (window < 0 or j >= i - window))
    assert bench.n_pairs(S, causal, window) == brute


def test_flops_counts():
    wl = bench.WORKLOADS["sweep_s8192_hkv8"]
    n = 4 * 32 * 8192 * 8193 // 2
    assert bench.flops(wl, "fwd") == n * 2 * 256
    assert bench.flops(wl, "bwd") == n * 2 * (3 * 128 + 2 * 128)
    assert abs(bench.flops(wl) / 1e12 - 7.698) < 1e-3   # the 7.698 TFLOP of the S=8192 GQA point


def test_traffic_only_for_its_workload():
    assert bench.recorded_traffic(bench.WORKLOADS["mla_b2_s4096"], "bwd_kv") is None


def test_traffic_record_is_dropped_once_its_sources_change(tmp_path, monkeypatch):
    """roofline.traffic comes from an ncu record only while the kernel sources it names
    still hash to the record's sha256; the deterministic path reads its own record."""
    import hashlib
    src = tmp_path / "kern.cu"
    src.write_text("__global__ void k() {}\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()
    rec = {"sources": ["kern.cu"], "sources_sha256": digest,
           "kernels": {"bwd_kv": {"dram_bytes_read": 300, "dram_bytes_write": 45}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "kernel_traffic.json").write_text(json.dumps(
        {"workloads": {"w": rec, "w:deterministic": dict(rec, kernels={"bwd_kv": {"dram_bytes_read": 7,
                                                                               "dram_bytes_write": 1}})}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    wl = {"name": "w"}
    assert bench.recorded_traffic(wl, "bwd_kv") == 345
    assert bench.recorded_traffic(wl, "bwd_kv", det=True) == 8
    assert bench.recorded_traffic(wl, "fwd") is None
    src.write_text("__global__ void k() { }\n")
    assert bench.recorded_traffic(wl, "bwd_kv") is None
    assert bench.recorded_traffic(wl, "bwd_kv", det=True) is None


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny_gqa_swa", "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["dtype"] == "f64"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the same config keys as the GPU arm's line, so the two lines compare the same workload
    assert d["config"] == bench.bench_config(bench.WORKLOADS["tiny_gqa_swa"], 1, False)
    assert d["higher_is_better"] is True and d["unit"] == "TFLOP/s"


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench._max_over_ranks(float(10 + rank), world, torch.device("cpu"))
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 2000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 11.0, 1: 11.0}


def test_padded_batch_workload_counts_each_entry_on_its_own_length():
    import bench
    wl = bench.WORKLOADS["varlen_gqa_b8_s4096"]
    assert len(wl["lens"]) == wl["B"] and max(wl["lens"]) <= wl["S"]
    per_pair = 2 * (wl["dqk"] + wl["dv"]) + 2 * (3 * wl["dqk"] + 2 * wl["dv"])
    want = wl["Hq"] * sum(L * (L + 1) // 2 for L in wl["lens"]) * per_pair
    assert bench.flops(wl) == want
    assert sum(bench.unit_flops(wl, b) for b in range(wl["B"])) * wl["Hq"] == want
    # a padded batch whose lengths are all S counts like the plain workload
    full = dict(wl, lens=[wl["S"]] * wl["B"])
    assert bench.flops(full) == bench.flops(dict(wl, lens=None))


def test_fp8_workloads_count_forward_flops_and_cast_bytes():
    import bench
    wl = bench.WORKLOADS["fp8_fwd_mha_b4_s2048_d64"]
    n = 4 * 8 * 2048 * 2049 // 2
    assert bench.flops(wl) == bench.flops(wl, "fwd") == n * 2 * (64 + 64)
    assert bench.flops(wl, "bwd") == 0
    elems = 4 * 2048 * 8 * 64
    assert bench.fp8_cast_bytes(wl) == 3 * (2 * elems + elems)   # bf16 in, E4M3 out, S a multiple of 16


def test_reference_arm_runs_the_fp8_oracle():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "fp8_fwd_mha_b4_s2048_d64", "--steps", "3", "--warmup", "3"], capture_output=True,
                         text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    d = json.loads([l for l in out.stdout.splitlines() if l.strip()][0])
    assert d["metric"] == bench.METRIC_FP8 and d["value"] > 0
    assert "E4M3" in d["cpu_baseline"]["sample"]
