"""The derived d_offset bound (parity_util.d_offset_bound), checked on the CPU against
an emulated kernel.

The learnable sink's gradient d_offset_h = -sum_i p_sink_i D_i has terms of both
signs.  A fused backward only has the forward's bf16 output, so it forms
D_i = dO_i . O_i from the rounded O.  The emulation below does the kernel's
arithmetic in numpy:
  * fp32 scores and exponentials;
  * P rounded to bf16 before P.V, fp32 accumulation;
  * O = bf16(acc / l), LSE = m + ln l in fp32;
  * D from the bf16 O in fp32;
  * d_offset as an fp32 sum.
It then checks that the error against the exact fp64 oracle stays inside the bound,
for well- and badly-conditioned cases.  It also checks that the bound is not vacuous,
so that a mistake in a term would show.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import d_offset_bound, dropout_o_scale
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def emulated_kernel(x, *, causal, scale, dropout_p=0.0, rng_state=None):
    """O (bf16 values), LSE (fp32) and d_offset (fp32) the way the fused kernels form them.
    With dropout the dropped P are zeroed before P.V (the row sum keeps them) and the
    kept multiplier is applied in fp32 before O is rounded."""
    q, k, v, do = (x[n].float().numpy() for n in ("q", "k", "v", "dout"))
    off = x["offset"].float().numpy()
    B, Sq, Hq, dqk = q.shape
    _, Skv, Hkv, dv = v.shape
    G = Hq // Hkv
    scale = np.float32(scale if scale is not None else 1.0 / np.sqrt(dqk))
    o = np.zeros((B, Sq, Hq, dv), np.float32)
    lse = np.zeros((B, Hq, Sq), np.float32)
    for b in range(B):
        for h in range(Hq):
            s = (q[b, :, h, :] @ k[b, :, h // G, :].T).astype(np.float32) * scale
            if causal:
                s = np.where(np.tril(np.ones((Sq, Skv), bool)), s, -np.inf).astype(np.float32)
            c = np.float32(off[h])
            m = np.maximum(s.max(axis=1), c)
            pt = np.exp(s - m[:, None]).astype(np.float32)
            l = (pt.sum(axis=1, dtype=np.float32) + np.exp(c - m)).astype(np.float32)
            ptk, ms = pt, np.float32(1.0)
            if dropout_p > 0.0:
                ptk = np.where(oracle.dropout_keep(b, h, Sq, Skv, dropout_p, rng_state), pt, np.float32(0.0))
                ms = np.float32(dropout_o_scale(dropout_p))
            acc = (bf16(ptk) @ v[b, :, h // G, :]).astype(np.float32)
            o[b, :, h, :] = bf16(ms * acc / l[:, None])
            lse[b, h] = (m + np.log(l)).astype(np.float32)
    D = np.einsum("bshd,bshd->bhs", do, o).astype(np.float32)
    p = np.exp(off[None, :, None].astype(np.float32) - lse).astype(np.float32)
    d_off = -np.sum((p * D).astype(np.float32), axis=(0, 2), dtype=np.float32)
    return o, lse, d_off


RNG = (0x5EED_1234_ABCD, 17)
CASES = [
    # name, shape, causal, scale, dropout probability
    ("causal_gqa", Shape(1, 96, 96, 4, 2, 64, 64), True, None, 0.0),
    ("noncausal_square", Shape(2, 64, 64, 4, 2, 64, 64), False, 0.08, 0.0),
    ("noncausal_rect", Shape(2, 40, 70, 2, 2, 64, 64), False, 0.2, 0.0),
    ("noncausal_mqa", Shape(1, 50, 33, 8, 1, 128, 128), False, None, 0.0),
    ("causal_gqa_dropout", Shape(1, 96, 96, 4, 2, 64, 64), True, None, 0.1),
    ("noncausal_rect_dropout", Shape(2, 40, 70, 2, 2, 64, 64), False, 0.2, 0.5),
    ("mla_dims_dropout", Shape(1, 65, 65, 2, 2, 192, 128), True, 1 / np.sqrt(192), 0.1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_emulated_kernel_within_derived_bound(case):
    name, shape, causal, scale, p = case
    x = make_inputs(shape, 700 + CASES.index(case), learnable_offset=True)
    drop = dict(dropout_p=p, rng_state=RNG) if p > 0 else {}
    o, lse, d_off = emulated_kernel(x, causal=causal, scale=scale, **drop)
    exact, bound, on_gpu_o, kernel_bound = d_offset_bound(x, {"o": o, "lse": lse}, causal=causal, window=-1,
                                                          scale=scale, **drop)
    err = np.abs(d_off.astype(np.float64) - exact)
    assert np.all(err <= bound), f"{name}: {err} > {bound}"
    assert np.all(np.abs(d_off - on_gpu_o) <= kernel_bound), name
    # not vacuous: the bound is a small fraction of the terms' magnitudes
    f = oracle.attention_fwd(*(x[n].double().numpy() for n in ("q", "k", "v")), causal=causal,
                             softmax_type=oracle.LEARNABLE, offset=x["offset"].double().numpy(), scale=scale,
                             **drop)
    g = oracle.attention_bwd(*(x[n].double().numpy() for n in ("q", "k", "v", "dout")), causal=causal,
                             softmax_type=oracle.LEARNABLE, offset=x["offset"].double().numpy(), scale=scale,
                             **drop)
    mag = np.sum(f["psink"] * np.abs(g["D"]), axis=(0, 2))
    assert np.all(bound <= 2e-2 * mag), f"{name}: bound {bound} vs sum |p D| {mag}"


def test_bound_catches_a_dropped_rounding_of_o():
    """A planted mistake: D formed from O rounded to multiples of 1/16 instead of to bf16.
    The tolerance must reject it."""
    shape = Shape(2, 64, 64, 4, 2, 64, 64)
    x = make_inputs(shape, 701, learnable_offset=True)
    o, lse, _ = emulated_kernel(x, causal=False, scale=0.08)
    coarse = np.round(o * 16.0) / 16.0                        # a far coarser "rounding" of O
    do = x["dout"].float().numpy()
    p = np.exp(x["offset"].float().numpy()[None, :, None] - lse)
    d_bad = -np.sum(p * np.einsum("bshd,bshd->bhs", do, coarse), axis=(0, 2))
    exact, bound, _, _ = d_offset_bound(x, {"o": o, "lse": lse}, causal=False, window=-1, scale=0.08)
    assert np.any(np.abs(d_bad - exact) > bound)


def test_bound_catches_p_sink_from_the_keys_only_lse():
    """A planted mistake: p_sink taken from the LSE of the keys alone (the sink left out
    of the normaliser), i.e. p / (1 - p).  The tolerance must reject it."""
    shape = Shape(1, 96, 96, 4, 2, 64, 64)
    x = make_inputs(shape, 700, learnable_offset=True)
    o, lse, _ = emulated_kernel(x, causal=True, scale=None)
    off = x["offset"].double().numpy()[None, :, None]
    p = np.exp(off - lse.astype(np.float64))
    do = x["dout"].double().numpy()
    d_bad = -np.sum(p / (1.0 - p) * np.einsum("bshd,bshd->bhs", do, o.astype(np.float64)), axis=(0, 2))
    exact, bound, _, _ = d_offset_bound(x, {"o": o, "lse": lse}, causal=True, window=-1, scale=None)
    assert np.any(np.abs(d_bad - exact) > bound)


def test_dropout_bound_catches_d_from_the_undropped_output():
    """A planted mistake: D formed from the output without dropout (every P kept, no
    multiplier) while the exact d_offset is the dropped one.  The tolerance must reject it."""
    shape = Shape(1, 96, 96, 4, 2, 64, 64)
    x = make_inputs(shape, 704, learnable_offset=True)
    drop = dict(dropout_p=0.1, rng_state=RNG)
    o_plain, lse, _ = emulated_kernel(x, causal=True, scale=None)
    o_drop, _, _ = emulated_kernel(x, causal=True, scale=None, **drop)
    do = x["dout"].double().numpy()
    p = np.exp(x["offset"].double().numpy()[None, :, None] - lse.astype(np.float64))
    d_bad = -np.sum(p * np.einsum("bshd,bshd->bhs", do, o_plain.astype(np.float64)), axis=(0, 2))
    exact, bound, _, _ = d_offset_bound(x, {"o": o_drop, "lse": lse}, causal=True, window=-1, scale=None, **drop)
    assert np.any(np.abs(d_bad - exact) > bound)
