"""FP8 backward (E4M3 Q, K, V; E5M2 dO) on the GPU against the oracle.

Both sides get the same inputs, none of them from the CUDA path: the oracle
quantises the seeded bf16 tensors (codes and descales; the GPU's own quantisation
is pinned bit-exact separately), and the forward's O and LSE are the oracle's exact
forward of the dequantised tensors, rounded to bf16 and fp32 as the backward takes
them.  The kernel and oracle.fp8.attention_bwd_fp8 then round the same P and dS;
they may differ only where the kernel's fp32 value of 2^8 P (or s dS) lies within
its own arithmetic error of a rounding midpoint, plus fp32 accumulation and the
bf16 rounding of the outputs.  parity_util.fp8_bwd_bounds derives that tolerance
per element; the CPU tests pin it against an fp32 emulation of the kernel and show
that an unrounded backward falls outside it.
"""

import numpy as np
import pytest
import torch

from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from oracle import fp8
from parity_util import check_fp8_bwd, fp8_bwd_bounds
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs

pytestmark = pytest.mark.gpu


def _sdpa():
    import scaled_dot_product_tmem_gb300 as sdpa
    return sdpa


def _check_device():
    st, site = _sdpa().attn_last_device_error()
    assert st == 0, f"device error status {st} site {site:#x}"


def _pad_t(codes_t, S):
    """[B,H,d,S] codes -> [B,H,d,S_pad] with zeros past S (the transposed layout)."""
    Sp = _sdpa().attn_fp8_vt_row_bytes(S)
    out = np.zeros(codes_t.shape[:-1] + (Sp,), dtype=np.uint8)
    out[..., :S] = codes_t
    return out


def _oracle_inputs(x, amax=None):
    """The oracle's codes (natural and transposed) and descales of q, k, v (E4M3) and
    dout (E5M2); amax: optional per-tensor statistics (else each tensor's own)."""
    amax = amax or {}
    xf = {n: x[n].float().numpy() for n in ("q", "k", "v", "dout")}
    c = {}
    for n, fmt in (("q", "e4m3"), ("k", "e4m3"), ("v", "e4m3"), ("dout", "e5m2")):
        c[n], a, c["s_" + n] = fp8.quantize(xf[n], amax=amax.get(n), fmt=fmt)
        if n != "v":
            c[n + "_t"] = fp8.quantize(xf[n], amax=a, transpose=True, fmt=fmt)[0]
    return c


def _fwd(c, *, causal, window, softmax_type, offset, scale):
    """The exact forward of the dequantised codes: O rounded to bf16, LSE to fp32."""
    f = fp8.attention_fwd_fp8(c["q"], c["k"], c["v"], c["s_q"], c["s_k"], c["s_v"], causal=causal, window=window,
                              softmax_type=softmax_type, offset=offset, scale=scale)
    o = torch.from_numpy(f["o"]).to(torch.bfloat16)
    lse = torch.from_numpy(f["lse"]).float()
    return o, lse


def _gpu_bwd(c, o, lse, ds_amax, *, causal, window, softmax_type, offset, scale):
    sdpa = _sdpa()
    dev = torch.device("cuda")
    S_q, S_kv = c["q"].shape[1], c["k"].shape[1]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    f1 = lambda v: torch.tensor([float(v)], dtype=torch.float32, device=dev)
    q8, k8, v8, do8 = t(c["q"]), t(c["k"]), t(c["v"]), t(c["dout"])
    qt8, kt8, dot8 = t(_pad_t(c["q_t"], S_q)), t(_pad_t(c["k_t"], S_kv)), t(_pad_t(c["dout_t"], S_q))
    dq = torch.full(q8.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    dk = torch.full(k8.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    dv = torch.full(v8.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    d_off = torch.full((q8.shape[2],), float("nan"), dtype=torch.float32, device=dev)
    amax_out = torch.full((1,), 123.0, dtype=torch.float32, device=dev)
    off = None if offset is None else torch.from_numpy(np.asarray(offset, dtype=np.float32)).to(dev)
    sdpa.attn_bwd_fp8(q8, k8, v8, do8, qt8, kt8, dot8, f1(c["s_q"]), f1(c["s_k"]), f1(c["s_v"]), f1(c["s_dout"]),
                      o.to(dev), lse.to(dev), f1(ds_amax), dq, dk, dv, d_off, ds_amax_out=amax_out, causal=causal,
                      window=window, softmax_type=softmax_type, softmax_offset=off, scale=scale or 0.0)
    torch.cuda.synchronize()
    _check_device()
    res = {"dq": dq, "dk": dk, "dv": dv, "d_offset": d_off, "amax": amax_out}
    return {n: v.double().cpu().numpy() for n, v in res.items()}


CASES = [
    # name, shape, causal, window, softmax type, scale, ds statistic (x the step's own max |dS|)
    ("d64_causal_mha", Shape(2, 300, 300, 2, 2, 64, 64), True, -1, VANILLA, None, 1.0),
    ("d128_causal_gqa", Shape(1, 333, 333, 4, 2, 128, 128), True, -1, VANILLA, None, 1.0),
    ("d128_window_obo", Shape(1, 400, 400, 4, 1, 128, 128), True, 100, OFF_BY_ONE, None, 1.0),
    ("d64_learnable_window", Shape(2, 260, 260, 4, 2, 64, 64), True, 64, LEARNABLE, 0.2, 1.0),
    ("d128_noncausal_rect", Shape(1, 150, 290, 2, 1, 128, 128), False, -1, VANILLA, None, 1.0),
    ("d64_sq_gt_skv", Shape(1, 300, 170, 2, 2, 64, 64), True, -1, OFF_BY_ONE, None, 1.0),
    ("d128_keyless_rows", Shape(1, 400, 130, 2, 1, 128, 128), True, 50, VANILLA, None, 1.0),
    ("d64_one_tile", Shape(1, 128, 128, 2, 1, 64, 64), True, 32, VANILLA, 0.125, 1.0),
    # delayed scaling: a stale statistic below this step's max |dS| saturates the
    # largest dS codes; one above it leaves the top codes unused
    ("d128_stale_low_stat", Shape(1, 256, 256, 2, 2, 128, 128), True, -1, VANILLA, None, 0.25),
    ("d64_stale_high_stat", Shape(1, 200, 200, 2, 1, 64, 64), False, -1, VANILLA, None, 8.0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fp8_backward_parity(case):
    name, shape, causal, window, st, scale, stat_mul = case
    x = make_inputs(shape, 500 + len(name), learnable_offset=(st == LEARNABLE))
    offset = x["offset"].double().numpy() if st == LEARNABLE else None
    kw = dict(causal=causal, window=window, softmax_type=st, offset=offset, scale=scale)
    c = _oracle_inputs(x)
    o, lse = _fwd(c, **kw)
    codes = (c["q"], c["k"], c["v"], c["dout"], c["s_q"], c["s_k"], c["s_v"], c["s_dout"])
    on, ln = o.double().numpy(), lse.double().numpy()
    own = fp8.attention_bwd_fp8(*codes, on, ln, 1.0, round_ds=False, **kw)["amax_ds"]
    stat = np.float32(own * stat_mul)
    ref = fp8.attention_bwd_fp8(*codes, on, ln, stat, **kw)
    bnd = fp8_bwd_bounds(*codes, on, ln, stat, **kw)
    got = _gpu_bwd(c, o, lse, stat, **kw)
    ratios = check_fp8_bwd(got, ref, bnd, name)
    assert max(ratios.values()) <= 1.0
    # this call's max |dS|, before rounding
    assert abs(got["amax"][0] - ref["amax_ds"]) <= bnd["amax_ds"] + 2.0 ** -24 * ref["amax_ds"], \
        (got["amax"][0], ref["amax_ds"], bnd["amax_ds"])
    if st == LEARNABLE:
        err = np.abs(got["d_offset"] - ref["d_offset"])
        assert np.all(err <= bnd["d_offset"]), (err, bnd["d_offset"])
    else:
        assert np.all(got["d_offset"] == 0.0)


@pytest.mark.parametrize("stat", [0.0, float("inf"), float("nan")], ids=["zero", "inf", "nan"])
def test_fp8_backward_degenerate_ds_statistic(stat):
    """A dS statistic that is 0 or not finite (no history yet, or an overflowed one) scales
    dS by 1, on both sides, and the call still records this step's max |dS|."""
    shape = Shape(1, 160, 160, 2, 1, 64, 64)
    x = make_inputs(shape, 611)
    kw = dict(causal=True, window=-1, softmax_type=VANILLA, offset=None, scale=None)
    c = _oracle_inputs(x)
    o, lse = _fwd(c, **kw)
    codes = (c["q"], c["k"], c["v"], c["dout"], c["s_q"], c["s_k"], c["s_v"], c["s_dout"])
    on, ln = o.double().numpy(), lse.double().numpy()
    ref = fp8.attention_bwd_fp8(*codes, on, ln, np.float32(stat), **kw)
    bnd = fp8_bwd_bounds(*codes, on, ln, np.float32(stat), **kw)
    got = _gpu_bwd(c, o, lse, stat, **kw)
    check_fp8_bwd(got, ref, bnd, f"stat {stat}")
    assert abs(got["amax"][0] - ref["amax_ds"]) <= bnd["amax_ds"] + 2.0 ** -24 * ref["amax_ds"]


def test_fp8_backward_empty_sides():
    """No keys: dQ = 0 (every row is empty, so D = 0 and nothing flows); no queries:
    dK = dV = 0; the recorded max |dS| is 0 either way."""
    sdpa = _sdpa()
    dev = torch.device("cuda")
    one = torch.ones(1, dtype=torch.float32, device=dev)
    for S_q, S_kv in ((64, 0), (0, 64)):
        B, H, d = 2, 2, 64
        u8 = lambda S: torch.zeros((B, S, H, d), dtype=torch.uint8, device=dev)
        ut = lambda S: torch.zeros((B, H, d, sdpa.attn_fp8_vt_row_bytes(S)), dtype=torch.uint8, device=dev)
        bf = lambda S: torch.full((B, S, H, d), float("nan"), dtype=torch.bfloat16, device=dev)
        o = torch.zeros((B, S_q, H, d), dtype=torch.bfloat16, device=dev)
        lse = torch.full((B, H, S_q), float("-inf"), dtype=torch.float32, device=dev)
        dq, dk, dv = bf(S_q), bf(S_kv), bf(S_kv)
        amax_out = torch.full((1,), 5.0, dtype=torch.float32, device=dev)
        sdpa.attn_bwd_fp8(u8(S_q), u8(S_kv), u8(S_kv), u8(S_q), ut(S_q), ut(S_kv), ut(S_q), one, one, one, one, o,
                          lse, one, dq, dk, dv, None, ds_amax_out=amax_out, causal=False)
        torch.cuda.synchronize()
        _check_device()
        for t in (dq, dk, dv):
            assert t.numel() == 0 or bool((t == 0).all())
        assert amax_out.item() == 0.0


def test_fp8_backward_convenience_equals_the_entry_point():
    """sdpa_backward_fp8 (bf16 in: its own E4M3 / E5M2 casts on the GPU, natural and
    transposed) gives bitwise the results of attn_bwd_fp8 on the oracle's codes (the
    casts are bit-exact), with the same O, LSE and dS statistic."""
    sdpa = _sdpa()
    shape = Shape(1, 320, 320, 4, 2, 128, 128)
    x = make_inputs(shape, 77)
    kw = dict(causal=True, window=-1, softmax_type=VANILLA, offset=None, scale=None)
    c = _oracle_inputs(x)
    o, lse = _fwd(c, **kw)
    stat = np.float32(2.5)
    ref = _gpu_bwd(c, o, lse, stat, **kw)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    dq, dk, dv, _ = sdpa.sdpa_backward_fp8(q, k, v, o.to(dev), do, lse.to(dev),
                                           ds_amax=torch.tensor([stat], device=dev), causal=True)
    torch.cuda.synchronize()
    _check_device()
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert np.array_equal(t.double().cpu().numpy(), ref[n]), n


def test_fp8_backward_is_deterministic():
    """No atomics on dQ, dK, dV: two calls give bitwise equal results."""
    shape = Shape(2, 384, 384, 4, 1, 64, 64)
    x = make_inputs(shape, 78)
    kw = dict(causal=True, window=-1, softmax_type=VANILLA, offset=None, scale=None)
    c = _oracle_inputs(x)
    o, lse = _fwd(c, **kw)
    a = _gpu_bwd(c, o, lse, 3.0, **kw)
    b = _gpu_bwd(c, o, lse, 3.0, **kw)
    for n in ("dq", "dk", "dv", "amax"):
        assert np.array_equal(a[n], b[n]), n


# The FP8 training shapes: causal GQA at S = 8192, d = 128 (B = 4, 32 query heads, 8
# kv heads), checked on one kv-head group: every query head's dQ on sampled rows and
# the group's dK, dV on sampled keys; and the FP8 example's MHA shape, on all rows.  The checked unit gets the oracle's forward;
# every other unit gets the GPU's FP8 forward (its outputs do not reach the checked
# unit's gradients).
FULL = [
    ("fp8_gqa_b4_s8192_d128", Shape(4, 8192, 8192, 32, 8, 128, 128), 43, (1, 6),
     np.r_[0:48, 2040:2056, 5000:5016, 8160:8192], np.r_[0:32, 4096:4112, 8176:8192]),
    # the FP8 example's shape (MHA, d = 64), every row and key of one (batch, head)
    ("fp8_mha_b4_s2048_d64", Shape(4, 2048, 2048, 8, 8, 64, 64), 45, (3, 5), np.arange(2048), np.arange(2048)),
]


@pytest.mark.parametrize("case", FULL, ids=[c[0] for c in FULL])
def test_fp8_backward_full_size_sampled(case):
    name, shape, seed, (b, g), rows, keys = case
    sdpa = _sdpa()
    dev = torch.device("cuda")
    x = make_inputs(shape, seed)
    G = shape.H_q // shape.H_kv
    hs = slice(g * G, (g + 1) * G)
    # the GPU's own casts of the full tensors (bit-exact, checked on the unit below)
    xg = {n: x[n].to(dev) for n in ("q", "k", "v", "dout")}
    q8, aq, sq = sdpa.fp8_quantize(xg["q"])
    k8, ak, sk = sdpa.fp8_quantize(xg["k"])
    v8, _, sv = sdpa.fp8_quantize(xg["v"])
    do8, ado, sdo = sdpa.fp8_quantize(xg["dout"], fmt="e5m2")
    qt8, _, _ = sdpa.fp8_quantize(xg["q"], transpose=True, amax=aq)
    kt8, _, _ = sdpa.fp8_quantize(xg["k"], transpose=True, amax=ak)
    dot8, _, _ = sdpa.fp8_quantize(xg["dout"], transpose=True, amax=ado, fmt="e5m2")
    o, lse = sdpa.sdpa_forward_fp8(xg["q"], xg["k"], xg["v"], causal=True)
    # the unit (b, g) with the oracle's own casts (scales from the whole tensors' amax)
    xf = {n: x[n][b:b + 1].float().numpy() for n in ("q", "k", "v", "dout")}
    amax = {n: np.float32(x[n].float().abs().max().item()) for n in ("q", "k", "v", "dout")}
    c = {}
    c["q"], _, c["s_q"] = fp8.quantize(xf["q"][:, :, hs], amax=amax["q"])
    c["k"], _, c["s_k"] = fp8.quantize(xf["k"][:, :, g:g + 1], amax=amax["k"])
    c["v"], _, c["s_v"] = fp8.quantize(xf["v"][:, :, g:g + 1], amax=amax["v"])
    c["dout"], _, c["s_dout"] = fp8.quantize(xf["dout"][:, :, hs], amax=amax["dout"], fmt="e5m2")
    for n, t in (("q", q8[b:b + 1, :, hs]), ("k", k8[b:b + 1, :, g:g + 1]), ("v", v8[b:b + 1, :, g:g + 1]),
                 ("dout", do8[b:b + 1, :, hs])):
        assert np.array_equal(t.cpu().numpy(), c[n]), f"GPU {n} codes differ from the oracle's"
    for n, t in (("q", sq), ("k", sk), ("v", sv), ("dout", sdo)):
        assert t.item() == c["s_" + n]
    kw = dict(causal=True, window=-1, softmax_type=VANILLA, offset=None, scale=None)
    ou, lu = _fwd(c, **kw)
    o[b:b + 1, :, hs] = ou.to(dev)
    lse[b:b + 1, hs] = lu.to(dev)
    codes = (c["q"], c["k"], c["v"], c["dout"], c["s_q"], c["s_k"], c["s_v"], c["s_dout"])
    on, ln = ou.double().numpy(), lu.double().numpy()
    stat = np.float32(fp8.attention_bwd_fp8(*codes, on, ln, 1.0, q_idx=rows, round_ds=False, **kw)["amax_ds"])
    f1 = lambda v: torch.tensor([float(v)], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(xg["q"]), torch.empty_like(xg["k"]), torch.empty_like(xg["v"])
    sdpa.attn_bwd_fp8(q8, k8, v8, do8, qt8, kt8, dot8, sq, sk, sv, sdo, o, lse, f1(stat), dq, dk, dv, None,
                      causal=True)
    torch.cuda.synchronize()
    _check_device()
    ri, kj = torch.as_tensor(rows, device=dev), torch.as_tensor(keys, device=dev)
    got = {"dq": dq[b:b + 1].index_select(1, ri)[:, :, hs].double().cpu().numpy(),
           "dk": dk[b:b + 1].index_select(1, kj)[:, :, g:g + 1].double().cpu().numpy(),
           "dv": dv[b:b + 1].index_select(1, kj)[:, :, g:g + 1].double().cpu().numpy()}
    for sel, names in ((dict(q_idx=rows), ("dq",)), (dict(k_idx=keys), ("dk", "dv"))):
        ref = fp8.attention_bwd_fp8(*codes, on, ln, stat, **sel, **kw)
        bnd = fp8_bwd_bounds(*codes, on, ln, stat, **sel, **kw)
        check_fp8_bwd(got, ref, bnd, f"{name} unit (b={b}, g={g})", names=names)
