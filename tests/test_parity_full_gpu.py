"""Full-size configurations on the GPU, checked against the fp64 oracle on sampled
units.  The GPU runs each whole problem exactly as bench.py launches it; the oracle
recomputes whole (batch, kv-head group) units — every query head of the group with
its kv head, all rows — which is exact for O, LSE, dQ of those heads and for dK/dV
of that kv head (their sums never leave the unit).  d_offset sums over the batch,
so the sink case runs the oracle on the unit for every batch entry and adds them.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from parity_util import Shape, compare, gpu_run, gpu_slice, make_inputs, oracle_run, rel_l2, slice_group

pytestmark = pytest.mark.gpu

# name, shape, causal, window, softmax_type, scale, seed, sampled (b, g) units
FULL = [
    ("gqa_swa_b4_s2048", Shape(4, 2048, 2048, 32, 8, 128, 128), True, 1024, VANILLA, None, 1, [(0, 0), (3, 7)]),
    ("mla_b2_s4096", Shape(2, 4096, 4096, 16, 16, 192, 128), True, -1, VANILLA, 1 / math.sqrt(192), 2,
     [(0, 0), (1, 15)]),
    ("sweep_s512_mha", Shape(64, 512, 512, 32, 32, 128, 128), True, -1, VANILLA, None, 1000 + 512 + 32,
     [(0, 0), (63, 31)]),
    ("sweep_s512_gqa", Shape(64, 512, 512, 32, 8, 128, 128), True, -1, VANILLA, None, 1000 + 512 + 8, [(5, 3)]),
    ("sweep_s512_mqa", Shape(64, 512, 512, 32, 1, 128, 128), True, -1, VANILLA, None, 1000 + 512 + 1, [(9, 0)]),
    # S = 1024 MHA: both backward paths run persistent CTAs (tiles of 16 steps / 8 kv tiles)
    ("sweep_s1024_mha", Shape(32, 1024, 1024, 32, 32, 128, 128), True, -1, VANILLA, None, 1000 + 1024 + 32,
     [(0, 0), (31, 17)]),
    ("sweep_s2048_gqa", Shape(16, 2048, 2048, 32, 8, 128, 128), True, -1, VANILLA, None, 1000 + 2048 + 8,
     [(15, 2)]),
    # S = 4096 MHA: the deterministic path's persistent kernels at their 32-step bound
    ("sweep_s4096_mha", Shape(8, 4096, 4096, 32, 32, 128, 128), True, -1, VANILLA, None, 1000 + 4096 + 32,
     [(7, 30)]),
    ("sweep_s8192_gqa", Shape(4, 8192, 8192, 32, 8, 128, 128), True, -1, VANILLA, None, 1000 + 8192 + 8, [(1, 5)]),
    ("sweep_s16384_gqa", Shape(2, 16384, 16384, 32, 8, 128, 128), True, -1, VANILLA, None, 1000 + 16384 + 8,
     [(1, 6)]),
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
@pytest.mark.parametrize("case", FULL, ids=[c[0] for c in FULL])
def test_full_size_sampled_units(case, deterministic):
    name, shape, causal, window, st, scale, seed, units = case
    x = make_inputs(shape, seed)
    kw = dict(causal=causal, window=window, softmax_type=st, scale=scale)
    gpu = gpu_run(x, deterministic=deterministic, **kw)
    if shape.d_qk == 192 and not deterministic:
        # d_qk = 192 has no fused dQ: deterministic = 0 takes the query-stationary kernel
        # too, so both ids must give the same bits
        det = gpu_run(x, deterministic=True, **kw)
        for n in ("o", "lse", "dq", "dk", "dv"):
            assert np.array_equal(gpu[n], det[n]), f"{name}: {n} differs between the two dQ ids"
    G = shape.H_q // shape.H_kv
    for b, g in units:
        ref = oracle_run(slice_group(x, b, g, G), **kw)
        compare(gpu_slice(gpu, b, g, G), ref, f"{name} unit (b={b}, g={g})")


@pytest.mark.parametrize("deterministic", [False, True], ids=["fused_dq", "det"])
@pytest.mark.parametrize("st", [OFF_BY_ONE, LEARNABLE], ids=["off_by_one", "learnable"])
def test_sink_config_full_size(st, deterministic):
    """B=2, S=4096, H_q=32, H_kv=8, d=64, causal; learnable offset [32] N(0,1) with gradient.
    deterministic=False is the path bench.py times: the kv kernel with the fused dQ."""
    shape = Shape(2, 4096, 4096, 32, 8, 64, 64)
    x = make_inputs(shape, 3, learnable_offset=True)
    kw = dict(causal=True, window=-1, softmax_type=st, scale=None)
    gpu = gpu_run(x, deterministic=deterministic, **kw)
    G, g = 4, 6
    d_off = np.zeros(G)
    for b in range(2):
        ref = oracle_run(slice_group(x, b, g, G), **kw)
        if st == LEARNABLE:
            d_off += ref.pop("d_offset")   # one batch entry's share of the sum over b
        compare(gpu_slice(gpu, b, g, G), ref, f"sink unit (b={b}, g={g})")
    if st == LEARNABLE:
        err = rel_l2(gpu["d_offset"][g * G:(g + 1) * G], d_off)
        assert err <= 1e-2, f"d_offset relative L2 {err}"
