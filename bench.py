#!/usr/bin/env python
"""Benchmark: fused attention forward + backward on GB300, in unmasked-FLOP TFLOP/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = attn_fwd + attn_bwd (every step of the hot path) over one batch of
synthetic BSHD bf16 inputs already resident in HBM.  The ``fp8_fwd_*`` workloads
time the E4M3 forward instead: one step = the per-tensor E4M3 casts of Q, K and V
(delayed scaling: the scale from the previous step's amax, this step's amax
recorded during the cast) + attn_fwd_fp8, counted in forward FLOPs.  The
``fp8_train_*`` workloads time an FP8 training step: the E4M3 casts of Q, K, V and
the E5M2 casts of dO (BSHD and transposed, delayed scaling), attn_fwd_fp8 and
attn_bwd_fp8 (dS scaled by the previous step's max |dS|), counted in forward +
backward FLOPs.  The default
workload is causal GQA at S=8192 (B=4, H_q=32, H_kv=8, d=128, vanilla softmax),
the point at which the method's target is stated.  FLOPs count only unmasked
(query, key) pairs: forward 2(d_qk + d_v) per pair, backward 2(3 d_qk + 2 d_v) per
pair.

The headline value comes from a pass with no per-kernel instrumentation; the
per-kernel split and the roofline come from a second pass of the same steps with
CUDA events around every launch.

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own copy of the
workload (independent problems, no collective on the data path: weak scaling).
``--impl reference`` times the fp64 CPU oracle on bounded samples of the same
workload instead (the only other place this script runs the oracle is the
``cpu_baseline`` leg of the default arm).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOP/s (bf16, unmasked FLOPs) and % of GB300 BF16 peak"
METRIC_FP8 = "attention fwd TFLOP/s (E4M3 Q/K/V with per-tensor scales, bf16 O; unmasked FLOPs)"
METRIC_FP8_TRAIN = ("attention fwd+bwd TFLOP/s (E4M3 Q/K/V, E5M2 dO and dS, per-tensor delayed scaling; "
                    "unmasked FLOPs)")
FP8_PER_BF16 = 2.0  # nominal dense E4M3 / bf16 tensor throughput (4.5 / 2.25 PFLOP/s)
NOMINAL_BF16_TFLOPS = 2250.0
L2_BYTES = 129 * 1024 * 1024


def _w(name, B, S, Hq, Hkv, dqk, dv, causal, window, st, scale, seed, desc, lens=None, fp8=False, bias=None,
       dropout=0.0, fp8_train=False):
    """A workload; `lens` (one length per batch entry, same for queries and keys) makes
    it a padded batch run through the varlen entry points; `fp8` makes it the E4M3
    forward, `fp8_train` the FP8 forward + backward step; `bias` = (Bb, Hb) adds a bf16
    [Bb, Hb, S, S] bias (attn_fwd_bias / attn_bwd_bias, with dbias); `dropout` = p runs
    attn_fwd_dropout / attn_bwd_dropout with the rng state DROPOUT_RNG."""
    return dict(name=name, B=B, S=S, Hq=Hq, Hkv=Hkv, dqk=dqk, dv=dv, causal=causal, window=window, st=st,
                scale=scale, seed=seed, desc=desc, lens=lens, fp8=fp8 or fp8_train, fp8_train=fp8_train, bias=bias,
                dropout=dropout)


DROPOUT_RNG = (0x5EED_2024_0001, 0)  # (seed, offset) of the dropout workloads


WORKLOADS = {
    "tiny_gqa_swa": _w("tiny_gqa_swa", 1, 128, 4, 2, 64, 64, True, 32, 0, 0.125, 0,
                       "tiny case: B=1, S=128, H_q=4, H_kv=2, d=64, causal, left window 32, vanilla, scale 1/8"),
    "gqa_swa_b4_s2048": _w("gqa_swa_b4_s2048", 4, 2048, 32, 8, 128, 128, True, 1024, 0, None, 1,
                           "BSHD GQA + SWA training shape: B=4, S=2048, H_q=32, H_kv=8, d_qk=d_v=128, causal, "
                           "left window 1024, vanilla softmax"),
    "mla_b2_s4096": _w("mla_b2_s4096", 2, 4096, 16, 16, 192, 128, True, -1, 0, 1 / math.sqrt(192), 2,
                       "MLA head dims: B=2, S=4096, H=16, d_qk=192, d_v=128, causal, scale 1/sqrt(192)"),
    "sink_obo_b2_s4096": _w("sink_obo_b2_s4096", 2, 4096, 32, 8, 64, 64, True, -1, 1, None, 3,
                            "sink attention, off-by-one: B=2, S=4096, H_q=32, H_kv=8, d=64, causal"),
    "sink_learnable_b2_s4096": _w("sink_learnable_b2_s4096", 2, 4096, 32, 8, 64, 64, True, -1, 2, None, 3,
                                  "sink attention, learnable offset [32]: B=2, S=4096, H_q=32, H_kv=8, d=64, causal"),
}
for _S in (512, 1024, 2048, 4096, 8192, 16384):
    for _H in (32, 8, 1):
        _n = f"sweep_s{_S}_hkv{_H}"
        WORKLOADS[_n] = _w(_n, 32768 // _S, _S, 32, _H, 128, 128, True, -1, 0, None, 1000 + _S + _H,
                           f"32768-token sweep: B={32768 // _S}, S={_S}, H_q=32, H_kv={_H}, d=128, causal")
# Padded batch: B=8 entries padded to S=4096, lengths spread evenly from 512 to 4096.
WORKLOADS["varlen_gqa_b8_s4096"] = _w(
    "varlen_gqa_b8_s4096", 8, 4096, 32, 8, 128, 128, True, -1, 0, None, 5,
    "padded batch: B=8 padded to S=4096, lengths 4096, 3584, ..., 512, H_q=32, H_kv=8, d=128, causal",
    lens=[4096 - 512 * i for i in range(8)])
# E4M3 forward: the pages' FP8 example shape, and the causal GQA S=8192 point.
WORKLOADS["fp8_fwd_mha_b4_s2048_d64"] = _w(
    "fp8_fwd_mha_b4_s2048_d64", 4, 2048, 8, 8, 64, 64, True, -1, 0, None, 41,
    "E4M3 forward: B=4, S=2048, H=8 (MHA), d=64, causal (the FP8 example's shape)", fp8=True)
WORKLOADS["fp8_fwd_gqa_b4_s8192_d128"] = _w(
    "fp8_fwd_gqa_b4_s8192_d128", 4, 8192, 32, 8, 128, 128, True, -1, 0, None, 42,
    "E4M3 forward: B=4, S=8192, H_q=32, H_kv=8, d=128, causal", fp8=True)
# FP8 training step (forward + backward) at the causal GQA S=8192 point.
WORKLOADS["fp8_train_gqa_b4_s8192_d128"] = _w(
    "fp8_train_gqa_b4_s8192_d128", 4, 8192, 32, 8, 128, 128, True, -1, 0, None, 43,
    "FP8 training step (E4M3 Q/K/V, E5M2 dO/dS): B=4, S=8192, H_q=32, H_kv=8, d=128, causal", fp8_train=True)
# The same step at the FP8 example's shape (MHA, d = 64).
WORKLOADS["fp8_train_mha_b4_s2048_d64"] = _w(
    "fp8_train_mha_b4_s2048_d64", 4, 2048, 8, 8, 64, 64, True, -1, 0, None, 46,
    "FP8 training step (E4M3 Q/K/V, E5M2 dO/dS): B=4, S=2048, H=8 (MHA), d=64, causal (the FP8 example's shape)",
    fp8_train=True)
# The same step at B=1: the small case its kernels are profiled on (inputs above L2, < 1 GB held).
WORKLOADS["fp8_train_gqa_b1_s8192_d128"] = _w(
    "fp8_train_gqa_b1_s8192_d128", 1, 8192, 32, 8, 128, 128, True, -1, 0, None, 44,
    "FP8 training step (E4M3 Q/K/V, E5M2 dO/dS): B=1, S=8192, H_q=32, H_kv=8, d=128, causal", fp8_train=True)
# Additive bias, one [S, S] plane per query head shared by the batch (dbias sums the batch).
WORKLOADS["bias_gqa_b2_s4096"] = _w(
    "bias_gqa_b2_s4096", 2, 4096, 32, 8, 128, 128, True, -1, 0, None, 8,
    "additive bias [1, 32, S, S] (bf16, N(0,1)) with dbias: B=2, S=4096, H_q=32, H_kv=8, d=128, causal",
    bias=(1, 32))
# Attention dropout p = 0.1 on the target point and on the GQA + SWA training shape.
WORKLOADS["dropout_gqa_b4_s8192"] = _w(
    "dropout_gqa_b4_s8192", 4, 8192, 32, 8, 128, 128, True, -1, 0, None, 1000 + 8192 + 8,
    "attention dropout p=0.1 (Philox4x32-10 decisions): B=4, S=8192, H_q=32, H_kv=8, d=128, causal", dropout=0.1)
WORKLOADS["dropout_gqa_swa_b4_s2048"] = _w(
    "dropout_gqa_swa_b4_s2048", 4, 2048, 32, 8, 128, 128, True, 1024, 0, None, 1,
    "attention dropout p=0.1 on the GQA + SWA training shape: B=4, S=2048, H_q=32, H_kv=8, d=128, causal, "
    "left window 1024", dropout=0.1)
DEFAULT = "sweep_s8192_hkv8"


def n_pairs(S, causal, window):
    """Unmasked (query, key) pairs of one (batch, head) with S_q = S_kv = S."""
    if not causal:
        return S * S
    if window < 0 or window >= S - 1:
        return S * (S + 1) // 2
    w = window
    return (w + 1) * (w + 2) // 2 + (S - w - 1) * (w + 1)


def total_pairs(wl):
    """Unmasked pairs of one query head summed over the batch (each entry over its own
    length in a padded batch)."""
    if wl.get("lens"):
        return sum(n_pairs(L, wl["causal"], wl["window"]) for L in wl["lens"])
    return wl["B"] * n_pairs(wl["S"], wl["causal"], wl["window"])


def flops(wl, part="total"):
    n = wl["Hq"] * total_pairs(wl)
    fwd = n * 2 * (wl["dqk"] + wl["dv"])
    bwd = 0 if wl.get("fp8") and not wl.get("fp8_train") else n * 2 * (3 * wl["dqk"] + 2 * wl["dv"])
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd}[part]


def kernel_flops(wl, cls, fused):
    """Algorithmic FLOPs one launch of a kernel class performs (see the design notes)."""
    n = wl["Hq"] * total_pairs(wl)
    d, e = wl["dqk"], wl["dv"]
    return {"fwd": n * 2 * (d + e),
            "bwd_kv": n * 2 * ((3 * d + 2 * e) if fused else (2 * d + 2 * e)),
            "bwd_q": n * 2 * d}.get(cls, 0)


def fp8_cast_bytes(wl):
    """Bytes the FP8 casts of one step must move, read bf16 (2 B per element) and write
    codes (1 B; transposed rows padded to 16): Q, K (BSHD) and V (transposed) for the
    forward; a training step reads Q, K, V and dO once each and writes both layouts of
    all four (dO in E5M2)."""
    B, S, Hq, Hkv, d = wl["B"], wl["S"], wl["Hq"], wl["Hkv"], wl["dqk"]
    Sp = (S + 15) // 16 * 16
    nq, nk = B * S * Hq * d, B * S * Hkv * d
    nqt, nkt = B * Hq * d * Sp, B * Hkv * d * Sp
    if not wl.get("fp8_train"):
        return 2 * (nq + 2 * nk) + nq + nk + nkt
    return 2 * (2 * nq + 2 * nk) + 2 * (nq + nqt) + 2 * (nk + nkt)


def fp8_cast_launches(wl):
    return 4 if wl.get("fp8_train") else 3


def recorded_traffic(wl, kernel, det=False):
    """DRAM bytes per launch of `kernel` from the committed ncu record of this workload
    (the deterministic backward's kernels have records of their own), or None when there
    is none or the kernel sources it names changed since."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "kernel_traffic.json")
    if not os.path.exists(p):
        return None
    key = wl["name"] + (":deterministic" if det and not wl.get("fp8") else "")
    with open(p) as f:
        rec = json.load(f).get("workloads", {}).get(key)
    if not rec or kernel not in rec.get("kernels", {}):
        return None
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec["sources_sha256"]:
        return None
    k = rec["kernels"][kernel]
    return k["dram_bytes_read"] + k["dram_bytes_write"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "MEASURED_PEAKS.json"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle samples


def oracle_units(wl):
    """(b, query head) units of the workload, in a fixed order."""
    return [(b, h) for b in range(wl["B"]) for h in range(wl["Hq"])]


def run_oracle_unit(wl, x, b, h):
    import oracle
    G = wl["Hq"] // wl["Hkv"]
    g = h // G
    if wl.get("fp8"):
        import numpy as np
        from oracle import fp8
        amax = x.setdefault("_amax", {n: np.float32(x[n].float().abs().max()) for n in ("q", "k", "v")})
        q8, _, dq = fp8.quantize(x["q"][b:b + 1, :, h:h + 1].float().numpy(), amax=amax["q"])
        k8, _, dk = fp8.quantize(x["k"][b:b + 1, :, g:g + 1].float().numpy(), amax=amax["k"])
        v8, _, dv = fp8.quantize(x["v"][b:b + 1, :, g:g + 1].float().numpy(), amax=amax["v"])
        f = fp8.attention_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=wl["causal"], window=wl["window"],
                                  softmax_type=wl["st"], scale=wl["scale"])
        if wl.get("fp8_train"):
            a_do = x.setdefault("_amax_do", np.float32(x["dout"].float().abs().max()))
            do8, _, ddo = fp8.quantize(x["dout"][b:b + 1, :, h:h + 1].float().numpy(), amax=a_do, fmt="e5m2")
            fp8.attention_bwd_fp8(q8, k8, v8, do8, dq, dk, dv, ddo, f["o"], f["lse"], 1.0, causal=wl["causal"],
                                  window=wl["window"], softmax_type=wl["st"], scale=wl["scale"])
        return
    L = wl["lens"][b] if wl.get("lens") else wl["S"]  # a padded entry computes on its own rows
    q = x["q"][b:b + 1, :L, h:h + 1].double().numpy()
    k = x["k"][b:b + 1, :L, g:g + 1].double().numpy()
    v = x["v"][b:b + 1, :L, g:g + 1].double().numpy()
    do = x["dout"][b:b + 1, :L, h:h + 1].double().numpy()
    off = x["offset"][h:h + 1].double().numpy() if wl["st"] == 2 else None
    kw = dict(causal=wl["causal"], window=wl["window"], softmax_type=wl["st"], offset=off, scale=wl["scale"])
    if wl.get("dropout"):  # the unit takes the decisions of its (b, h) in the full problem
        kw.update(dropout_p=wl["dropout"], rng_state=DROPOUT_RNG, dropout_origin=(b, h))
    if wl.get("bias"):
        Bb, Hb = wl["bias"]
        kw["bias"] = x["bias"][b if Bb > 1 else 0:(b if Bb > 1 else 0) + 1,
                               h if Hb > 1 else 0:(h if Hb > 1 else 0) + 1, :L, :L].double().numpy()
    oracle.attention_fwd(q, k, v, **kw)
    oracle.attention_bwd(q, k, v, do, **kw)


def unit_flops(wl, b=None):
    """FLOPs of one (batch, query head) unit: of entry b, or the workload's average."""
    if b is not None and wl.get("lens"):
        per = 2 * (wl["dqk"] + wl["dv"]) + (0 if wl.get("fp8") and not wl.get("fp8_train")
                                           else 2 * (3 * wl["dqk"] + 2 * wl["dv"]))
        return n_pairs(wl["lens"][b], wl["causal"], wl["window"]) * per
    return flops(wl) / (wl["B"] * wl["Hq"])


def make_cpu_inputs(wl, rank=0):
    from scaled_dot_product_tmem_gb300.inputs import Shape, make_bias, make_inputs
    shape = Shape(wl["B"], wl["S"], wl["S"], wl["Hq"], wl["Hkv"], wl["dqk"], wl["dv"])
    x = make_inputs(shape, wl["seed"] + 7919 * rank, learnable_offset=(wl["st"] == 2))
    if wl.get("bias"):
        x["bias"] = make_bias((*wl["bias"], wl["S"], wl["S"]), wl["seed"] + 1 + 7919 * rank)
    return x


def cpu_baseline(wl, x, budget_s=12.0):
    """The oracle, as it stands, on whole (batch, query head) units until ~budget_s."""
    import oracle
    units = oracle_units(wl)
    done, work, t0 = 0, 0.0, time.perf_counter()
    for b, h in units:
        run_oracle_unit(wl, x, b, h)
        done += 1
        work += unit_flops(wl, b)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": work / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{done} of {len(units)} (batch, query head) units of the workload, "
                      f"{oracle_step_desc(wl)} in fp64 "
                      f"({dt:.1f} s); TFLOP/s counts the same unmasked FLOPs as the GPU number"}


def oracle_step_desc(wl):
    if wl.get("fp8_train"):
        return "FP8 quantisation + fwd + FP8 bwd"
    return "E4M3 quantisation + fwd" if wl.get("fp8") else "fwd+bwd"


def metric_of(wl):
    if wl.get("fp8_train"):
        return METRIC_FP8_TRAIN
    return METRIC_FP8 if wl.get("fp8") else METRIC


# ----------------------------------------------------------------------------- arms


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def bench_config(wl, world, det):
    """The `config` object of the JSON line, the same for both arms."""
    fp8 = bool(wl.get("fp8"))
    return {"workload": wl["desc"], "global_batch": wl["B"] * world, "seq_len": wl["S"],
            "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU",
            **({"step": "E4M3 casts of Q, K, V and an E5M2 cast of dO, each writing BSHD and transposed "
                        "codes from one read (delayed scaling, amax recorded in the cast) + attn_fwd_fp8 + "
                        "attn_bwd_fp8 (dS scaled by the previous step's max |dS|)"} if wl.get("fp8_train") else
               {"step": "E4M3 casts of Q, K, V (delayed scaling, amax recorded in the cast) + attn_fwd_fp8"}
               if fp8 else {"bwd_path": "deterministic (query-stationary dQ)" if det else "fp32 atomic dQ"}),
            "l2": "flushed between timed steps (258 MB write outside the timed span)",
            **({"seq_lens": wl["lens"]} if wl.get("lens") else {}),
            **({"bias": f"bf16 {list(wl['bias']) + [wl['S'], wl['S']]}, dbias fp32"} if wl.get("bias") else {}),
            **({"dropout": f"p={wl['dropout']}, rng_state {list(DROPOUT_RNG)}"} if wl.get("dropout") else {})}


def uses_deterministic(wl, args):
    """The backward path bench.py runs: deterministic when asked for, or when the head
    dims have no fused dQ in the library (d_qk = 192)."""
    fused_ok = wl["dqk"] in (64, 128) and wl["dv"] in (64, 128)
    return bool(args.deterministic) or not fused_ok


def reference_arm(args, wl, world, rank):
    if rank != 0:
        return 0
    import oracle
    x = make_cpu_inputs(wl)
    units = oracle_units(wl)
    for i in range(args.warmup):
        run_oracle_unit(wl, x, *units[i % len(units)])
    t0, work = time.perf_counter(), 0.0
    for i in range(args.steps):
        u = units[(args.warmup + i) % len(units)]
        run_oracle_unit(wl, x, *u)
        work += unit_flops(wl, u[0])
    dt = time.perf_counter() - t0
    value = work / dt / 1e12
    sample = (f"each step = one (batch, query head) unit of the workload, "
              f"{oracle_step_desc(wl)} in fp64 "
              f"({unit_flops(wl) / 1e9:.2f} GFLOP)")
    line = {"metric": metric_of(wl), "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(wl, 1, uses_deterministic(wl, args)),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _step_fns_fp8(sdpa, wl, dev, x):
    """E4M3 forward step: cast Q, K (BSHD) and V (transposed) with the scales of the
    previous step's amax while recording this step's, then attn_fwd_fp8.  A training
    step (fp8_train) also casts Q^T, K^T and V (E4M3) and dO, dO^T (E5M2) the same way
    and runs attn_bwd_fp8 with dS scaled by the previous step's max |dS|."""
    import torch
    train = bool(wl.get("fp8_train"))
    B, S, Hq, Hkv, d = wl["B"], wl["S"], wl["Hq"], wl["Hkv"], wl["dqk"]
    Sp = sdpa.attn_fp8_vt_row_bytes(S)
    t = {n: x[n].to(dev) for n in (("q", "k", "v", "dout") if train else ("q", "k", "v"))}
    f32 = lambda: torch.empty(1, dtype=torch.float32, device=dev)
    amax = {n: [f32(), f32()] for n in t}          # [previous step's, this step's]
    desc = {n: f32() for n in t}
    for n in t:
        sdpa.attn_fp8_amax(t[n], amax[n][0])      # the history before the first step
    u8 = lambda *shape: torch.empty(shape, dtype=torch.uint8, device=dev)
    x8 = {"q": u8(B, S, Hq, d), "k": u8(B, S, Hkv, d), "vt": u8(B, Hkv, d, Sp)}
    # (tensor, code buffer, transposed, E5M2, BSHD buffer written by the same pass or None)
    casts = [("q", "q", False, False, None), ("k", "k", False, False, None), ("v", "vt", True, False, None)]
    if train:  # every tensor in both layouts from one read
        x8.update(qt=u8(B, Hq, d, Sp), kt=u8(B, Hkv, d, Sp), v=u8(B, S, Hkv, d), do=u8(B, S, Hq, d),
                  dot=u8(B, Hq, d, Sp))
        casts = [("q", "qt", True, False, "q"), ("k", "kt", True, False, "k"), ("v", "vt", True, False, "v"),
                 ("dout", "dot", True, True, "do")]
    o = torch.empty((B, S, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    kw = dict(causal=wl["causal"], window=wl["window"], softmax_type=wl["st"], scale=wl["scale"] or 0.0)
    outs = (o,)
    if train:
        dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
        ds_amax = [f32(), f32()]
        ds_amax[0].fill_(1.0)                      # the history before the first step
        ws = torch.empty(max(sdpa.attn_bwd_fp8_workspace_size(B, S, Hq), 256), dtype=torch.uint8, device=dev)
        outs = (o, dq, dk, dv)

    def step():
        for n, buf, tr, e5, nat in casts:
            if nat is not None:
                sdpa.attn_fp8_quantize_both(t[n], x8[nat], x8[buf], amax[n][0], desc[n], e5m2=e5,
                                            amax_out=amax[n][1])
            else:
                quant = sdpa.attn_fp8_quantize_e5m2 if e5 else sdpa.attn_fp8_quantize
                quant(t[n], x8[buf], amax[n][0], desc[n], transpose=tr, amax_out=amax[n][1])
        for n in t:
            amax[n].reverse()                      # this step's amax scales the next step
        sdpa.attn_fwd_fp8(x8["q"], x8["k"], x8["vt"], desc["q"], desc["k"], desc["v"], o, lse, **kw)
        if train:
            # the step's scales were applied above, so desc[] holds them; the amax lists were
            # swapped, so [1] is the history that scaled this step and [0] this step's record
            sdpa.attn_bwd_fp8(x8["q"], x8["k"], x8["v"], x8["do"], x8["qt"], x8["kt"], x8["dot"], desc["q"],
                              desc["k"], desc["v"], desc["dout"], o, lse, ds_amax[0], dq, dk, dv, None,
                              ds_amax_out=ds_amax[1], workspace=ws, **kw)
            ds_amax.reverse()

    return step, t, outs


def _step_fns(sdpa, wl, dev, det, x):
    import torch
    if wl.get("fp8"):
        return _step_fns_fp8(sdpa, wl, dev, x)
    B, S, Hq, Hkv, dqk, dv = wl["B"], wl["S"], wl["Hq"], wl["Hkv"], wl["dqk"], wl["dv"]
    t = {n: x[n].to(dev) for n in ("q", "k", "v", "dout")}
    off = x["offset"].to(dev) if wl["st"] == 2 else None
    o = torch.empty((B, S, Hq, dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    dq = torch.empty_like(t["q"])
    dk = torch.empty_like(t["k"])
    dvv = torch.empty_like(t["v"])
    doff = torch.empty((Hq,), dtype=torch.float32, device=dev) if wl["st"] == 2 else None
    ws = torch.empty(max(sdpa.attn_bwd_workspace_size(B, S, S, Hq, Hkv, dqk, dv, det), 256), dtype=torch.uint8,
                     device=dev)
    kw = dict(causal=wl["causal"], window=wl["window"], softmax_type=wl["st"], softmax_offset=off,
              scale=wl["scale"] or 0.0)
    if wl.get("dropout"):
        kw.update(dropout_p=wl["dropout"], rng_state=torch.tensor(list(DROPOUT_RNG), dtype=torch.int64, device=dev))
    if wl.get("lens"):
        lens = torch.tensor(wl["lens"], dtype=torch.int32, device=dev)
        kw.update(seq_lens_q=lens, seq_lens_kv=lens)
    bkw, outs = {}, (o, dq, dk, dvv)
    if wl.get("bias"):
        t["bias"] = x["bias"].to(dev)
        dbias = torch.empty(t["bias"].shape, dtype=torch.float32, device=dev)
        bkw, outs = {"dbias": dbias}, (o, dq, dk, dvv, dbias)

    def step():
        b = t.get("bias")
        sdpa.attn_fwd(t["q"], t["k"], t["v"], o, lse, bias=b, **kw)
        sdpa.attn_bwd(t["q"], t["k"], t["v"], o, t["dout"], lse, dq, dk, dvv, doff, deterministic=det,
                      workspace=ws, bias=b, **bkw, **kw)

    return step, t, outs


def measure(sdpa, wl, dev, det, x, steps, warmup, sampler=None, split_steps=10):
    """Device time of `steps` fwd+bwd steps on resident inputs (L2 flushed between
    steps), taken with per-kernel timing off; then `split_steps` more steps with CUDA
    events around every launch for the per-kernel split."""
    import torch
    step, t, outs = _step_fns(sdpa, wl, dev, det, x)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st, site = sdpa.attn_last_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st} site {site:#x} during warm-up")

    def timed_steps(n, per_kernel):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        sdpa.attn_timing_read()
        sdpa.attn_timing_enable(per_kernel)
        torch.cuda.synchronize()
        for i in range(n):
            flush.fill_(float(i))  # evict the previous step's data from L2 (outside the timed span)
            starts[i].record()
            step()
            ends[i].record()
        torch.cuda.synchronize()
        sdpa.attn_timing_enable(False)
        kt = sdpa.attn_timing_read()
        return sum(a.elapsed_time(b) for a, b in zip(starts, ends)), kt

    if sampler:
        sampler.start()
    ms, _ = timed_steps(steps, False)
    clocks = sampler.stop() if sampler else None
    _, kt = timed_steps(split_steps, True)
    st, site = sdpa.attn_last_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st} site {site:#x}")
    return ms, kt, clocks


def measure_e2e(sdpa, wl, dev, det, x, steps, warmup):
    """The same step through the C ABI from pinned HOST buffers: every step copies its
    q/k/v/dO host->device and reads O/dQ/dK/dV back device->host inside the timed span.
    Like an input pipeline, two device buffer sets alternate, the uploads run on one
    copy stream and the downloads on another, so step i+1's upload and step i-1's
    download overlap step i's kernels; events order each copy against the kernels that
    produce or consume its buffers."""
    import torch
    sets = [_step_fns(sdpa, wl, dev, det, x) for _ in range(2)]
    host_in = {n: x[n].pin_memory() for n in sets[0][1]}
    host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs] for _, _, outs in sets]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(o.numel() * o.element_size() for o in host_out[0])
    comp = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    uploaded, computed, downloaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def run(n):
        for i in range(n):
            k = i % 2
            step, t, outs = sets[k]
            with torch.cuda.stream(up):
                if started[k]:
                    up.wait_event(computed[k])      # the kernels of step i-2 read these inputs
                for nm in host_in:
                    t[nm].copy_(host_in[nm], non_blocking=True)
                uploaded[k].record(up)
            comp.wait_event(uploaded[k])
            if started[k]:
                comp.wait_event(downloaded[k])      # step i-2's outputs have left this set
            step()
            computed[k].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[k])
                for ho, o in zip(host_out[k], outs):
                    ho.copy_(o, non_blocking=True)
                downloaded[k].record(down)
            started[k] = True
        comp.wait_event(downloaded[0])
        comp.wait_event(downloaded[1])

    run(max(warmup, 2))
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    run(steps)
    b.record(comp)
    torch.cuda.synchronize()
    return a.elapsed_time(b), h2d, d2h


def _max_over_ranks(val, world, dev):
    if world == 1:
        return val
    import torch
    import torch.distributed as dist
    tt = torch.tensor([val], dtype=torch.float64, device=dev)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def ours_arm(args, wl, world, rank, local):
    import torch
    import scaled_dot_product_tmem_gb300 as sdpa
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sdpa.library()
    det = uses_deterministic(wl, args)
    fp8 = bool(wl.get("fp8"))
    x = make_cpu_inputs(wl, rank)
    ms, kt, clocks = measure(sdpa, wl, dev, det, x, args.steps, args.warmup, ClockSampler(local),
                             split_steps=min(args.steps, 10))
    total_flops = flops(wl)
    ms_max = _max_over_ranks(ms, world, dev)
    value = world * total_flops * args.steps / (ms_max / 1e3) / 1e12
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 20))
        e2e_ms, h2d, d2h = measure_e2e(sdpa, wl, dev, det, x, e2e_steps, 2)
        e2e_ms = _max_over_ranks(e2e_ms, world, dev)
        e2e = {"value": world * total_flops * e2e_steps / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "copies": "pinned host buffers; two device buffer sets, uploads and downloads on their own "
                         "streams overlapping the neighbouring steps' kernels"}
    peaks, peak_src = load_peaks()
    dom = max(kt, key=lambda k: kt[k][0])
    dms, dn = kt[dom]
    if dom == "fp8_quantize":  # a stream: bytes, against the measured copy bandwidth
        bound, unit = "hbm", "GB/s"
        achieved = fp8_cast_bytes(wl) / fp8_cast_launches(wl) / (dms / dn / 1e3) / 1e9 if dn else 0.0
        peak = float(peaks["hbm_gbs"])
        peak_desc = f"hbm_gbs from {peak_src}"
    else:
        bound, unit = "tensor", "TFLOP/s"
        dflops = kernel_flops(wl, dom, fused=not det and not wl.get("fp8_train"))
        achieved = dflops / (dms / dn / 1e3) / 1e12 if dn else 0.0
        peak = float(peaks["bf16_tflops"]) * (FP8_PER_BF16 if fp8 else 1.0)
        peak_desc = (f"bf16_tflops (burst) from {peak_src} x {FP8_PER_BF16} (nominal E4M3/bf16 ratio)"
                     if fp8 else f"bf16_tflops (burst) from {peak_src}")
    split_steps = min(args.steps, 10)   # the per-kernel pass (measure's split_steps)
    per_step = sum(v[1] for v in kt.values()) / split_steps
    launches = int(round(per_step * args.steps))  # the timed pass runs the same launches per step
    kernels = {k: {"ms_per_launch": v[0] / v[1], "launches_per_step": v[1] / split_steps,
                   "share": v[0] / sum(u[0] for u in kt.values())}
               for k, v in kt.items() if v[1]}
    line = {"metric": metric_of(wl), "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ("e4m3/e5m2" if wl.get("fp8_train") else "e4m3") if fp8 else "bf16", "data": "synthetic",
            "config": bench_config(wl, world, det),
            "pct_of_nominal_bf16_peak": 100.0 * value / world / NOMINAL_BF16_TFLOPS,
            **({"pct_of_nominal_fp8_peak": 100.0 * value / world / (FP8_PER_BF16 * NOMINAL_BF16_TFLOPS)}
               if fp8 else {}),
            "fwd_tflop": flops(wl, "fwd") / 1e12, "bwd_tflop": flops(wl, "bwd") / 1e12,
            "roofline": {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "peak_source": peak_desc,
                         "traffic": recorded_traffic(wl, dom, det), "traffic_unit": "bytes per launch (ncu DRAM read+write)"},
            "kernels": kernels,
            "kernel_split": f"a second pass of {min(args.steps, 10)} steps with CUDA events around every launch",
            "gpu_launches": launches,
            **({"e2e": e2e} if e2e else {}),
            "clocks": clocks}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, x)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--deterministic", action="store_true", help="deterministic backward (recompute dQ)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (keeps the device footprint to one step's buffers, for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, wl, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
    world, rank, local = dist_setup()
    return ours_arm(args, wl, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
