"""FP8 (E4M3) forward on the GPU against the oracle.

* Quantisation (amax, scale, codes, descale) is integer work decided by fp32
  arithmetic: bit-exact against ``oracle.fp8.quantize``, BSHD and transposed.
* The forward is compared with the oracle's exact attention of the dequantised
  tensors (the oracle quantises the same bf16 inputs itself).  The kernel rounds
  the softmax numerators to E4M3 for P.V, so O may depart from the exact value by
  the oracle's per-row ``p_rounding_bound``; on top of it the test allows bf16
  rounding of O (2^-8 |O|) and 1e-4 for the fp32 accumulation and ex2.  The LSE
  uses the unrounded numerators: max-abs <= 1e-3 as for the bf16 path.
"""

import numpy as np
import pytest
import torch

from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from oracle import fp8
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs

pytestmark = pytest.mark.gpu

TOL_LSE = 1e-3


def _sdpa():
    import scaled_dot_product_tmem_gb300 as sdpa
    return sdpa


def _check_device():
    st, site = _sdpa().attn_last_device_error()
    assert st == 0, f"device error status {st} site {site:#x}"


@pytest.mark.parametrize("shape", [(2, 200, 3, 64), (1, 77, 2, 128), (3, 128, 1, 128)])
@pytest.mark.parametrize("transpose", [False, True], ids=["bshd", "vt"])
def test_quantize_bit_exact(shape, transpose):
    sdpa = _sdpa()
    B, S, H, d = shape
    x = make_inputs(Shape(B, S, S, H, H, d, d), 11)["q"] * 3.0  # a wider range of values
    x[0, 0, 0, 0] = -7.5                                         # a known amax element
    xg = x.cuda()
    x8, amax, descale = sdpa.fp8_quantize(xg, transpose=transpose)
    torch.cuda.synchronize()
    _check_device()
    codes, a_ref, d_ref = fp8.quantize(x.float().numpy(), transpose=transpose)
    assert amax.item() == a_ref
    assert descale.item() == d_ref
    got = x8.cpu().numpy()
    if transpose:
        Sp = sdpa.attn_fp8_vt_row_bytes(S)
        assert got.shape == (B, H, d, Sp)
        assert not got[..., S:].any()                            # zero padding
        got = got[..., :S]
    assert np.array_equal(got, codes)


@pytest.mark.parametrize("transpose", [False, True], ids=["bshd", "vt"])
def test_quantize_with_a_given_amax_and_saturation(transpose):
    """A caller's amax (an amax history's max) sets the scale; values above it
    saturate to +-448 instead of overflowing; amax_out records the tensor's own amax
    in the same pass."""
    sdpa = _sdpa()
    x = make_inputs(Shape(2, 100, 100, 3, 3, 64, 64), 12)["k"]
    a = torch.tensor([0.5], dtype=torch.float32, device="cuda")  # below the true amax
    rec = torch.full((1,), 123.0, dtype=torch.float32, device="cuda")  # overwritten
    x8, _, descale = sdpa.fp8_quantize(x.cuda(), amax=a, amax_out=rec, transpose=transpose)
    torch.cuda.synchronize()
    _check_device()
    codes, _, d_ref = fp8.quantize(x.float().numpy(), amax=np.float32(0.5), transpose=transpose)
    assert descale.item() == d_ref
    got = x8.cpu().numpy()
    assert np.array_equal(got[..., :100] if transpose else got, codes)
    assert (np.abs(fp8.e4m3_decode(codes)) == 448.0).sum() > 10
    assert rec.item() == float(np.abs(x.float().numpy()).max())


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("shape", [(2, 200, 3, 64), (1, 77, 2, 128)])
def test_quantize_both_layouts_in_one_pass(shape, fmt):
    """attn_fp8_quantize_both writes the BSHD and the transposed codes from one read: both
    equal the oracle's casts, with the same descale and the tensor's amax recorded."""
    sdpa = _sdpa()
    B, S, H, d = shape
    x = make_inputs(Shape(B, S, S, H, H, d, d), 13)["q"] * 2.0
    rec = torch.full((1,), 7.0, dtype=torch.float32, device="cuda")
    x8, x8t, amax, descale = sdpa.fp8_quantize_both(x.cuda(), fmt=fmt, amax_out=rec)
    torch.cuda.synchronize()
    _check_device()
    xf = x.float().numpy()
    codes, a_ref, d_ref = fp8.quantize(xf, fmt=fmt)
    codes_t, _, _ = fp8.quantize(xf, fmt=fmt, transpose=True)
    assert amax.item() == a_ref and descale.item() == d_ref
    assert rec.item() == float(np.abs(xf).max())
    assert np.array_equal(x8.cpu().numpy(), codes)
    got_t = x8t.cpu().numpy()
    assert not got_t[..., S:].any()
    assert np.array_equal(got_t[..., :S], codes_t)


def _oracle_fp8(x, *, causal, window, softmax_type, scale, rows=None):
    """The oracle's own quantisation of the bf16 inputs, then the exact forward of the
    dequantised tensors and the P-rounding bound."""
    xf = {n: x[n].float().numpy() for n in ("q", "k", "v")}
    q8, _, dq = fp8.quantize(xf["q"])
    k8, _, dk = fp8.quantize(xf["k"])
    v8, _, dv = fp8.quantize(xf["v"])
    off = x["offset"].double().numpy() if softmax_type == LEARNABLE else None
    kw = dict(causal=causal, window=window, softmax_type=softmax_type, offset=off, scale=scale)
    ref = fp8.attention_fwd_fp8(q8, k8, v8, dq, dk, dv, **kw)
    bound = fp8.p_rounding_bound(fp8.dequantize(q8, dq), fp8.dequantize(k8, dk), fp8.dequantize(v8, dv),
                                 ref["lse"], causal=causal, window=window, scale=scale,
                                 softmax_type=softmax_type, offset=off, rows=rows)
    return ref, bound


def _gpu_fp8(x, *, causal, window, softmax_type, scale):
    sdpa = _sdpa()
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    off = x["offset"].cuda() if softmax_type == LEARNABLE else None
    o, lse = sdpa.sdpa_forward_fp8(q, k, v, causal=causal, window=window, softmax_type=softmax_type,
                                   softmax_offset=off, scale=scale or 0.0)
    torch.cuda.synchronize()
    _check_device()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _compare(o, lse, ref, bound, what, rows=None):
    ro, rl = ref["o"], ref["lse"]
    if rows is not None:
        ro, rl, o, lse = ro[:, rows], rl[:, :, rows], o[:, rows], lse[:, :, rows]
    # bound [B,H,S] -> per element of O [B,S,H,d]
    tol = np.transpose(bound, (0, 2, 1))[..., None] + 2.0 ** -8 * np.abs(ro) + 1e-4
    err = np.abs(o - ro)
    assert np.all(err <= tol), f"{what}: O off by {float((err - tol).max()):.3g} beyond the bound"
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse)), f"{what}: LSE finiteness differs"
    if fin.any():
        e = float(np.abs(lse[fin] - rl[fin]).max())
        assert e <= TOL_LSE, f"{what}: LSE max-abs {e}"
    return float(err.max()), float((err / tol).max())


CASES = [
    # name, shape, causal, window, softmax type, scale
    ("d64_causal_mha", Shape(2, 300, 300, 2, 2, 64, 64), True, -1, VANILLA, None),
    ("d128_causal_gqa", Shape(1, 333, 333, 4, 2, 128, 128), True, -1, VANILLA, None),
    ("d128_window_obo", Shape(1, 400, 400, 4, 1, 128, 128), True, 100, OFF_BY_ONE, None),
    ("d64_learnable_window", Shape(2, 260, 260, 4, 2, 64, 64), True, 64, LEARNABLE, 0.2),
    ("d128_noncausal_rect", Shape(1, 150, 290, 2, 1, 128, 128), False, -1, VANILLA, None),
    ("d64_sq_gt_skv", Shape(1, 300, 170, 2, 2, 64, 64), True, -1, OFF_BY_ONE, None),
    ("d128_keyless_rows", Shape(1, 400, 130, 2, 1, 128, 128), True, 50, VANILLA, None),
    ("d64_one_tile", Shape(1, 128, 128, 2, 1, 64, 64), True, 32, VANILLA, 0.125),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fp8_forward_parity(case):
    name, shape, causal, window, st, scale = case
    x = make_inputs(shape, 300 + len(name), with_dout=False, learnable_offset=(st == LEARNABLE))
    kw = dict(causal=causal, window=window, softmax_type=st, scale=scale)
    o, lse = _gpu_fp8(x, **kw)
    ref, bound = _oracle_fp8(x, **kw)
    _compare(o, lse, ref, bound, name)


def test_fp8_forward_against_the_bf16_path():
    """The pages compare the FP8 output with the bf16 output by the largest absolute
    difference: both paths against the same exact reference stay within their own
    tolerances, and FP8 is the coarser of the two."""
    sdpa = _sdpa()
    shape = Shape(1, 512, 512, 4, 4, 64, 64)
    x = make_inputs(shape, 21, with_dout=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o8, _ = sdpa.sdpa_forward_fp8(q, k, v, causal=True)
    o16, _ = sdpa.sdpa_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    diff = float((o8.float() - o16.float()).abs().max())
    assert 0 < diff < 0.25, diff


# The FP8 benchmark shapes: the pages' FP8 example (B=4, S=2048, 8 heads, d=64,
# causal) checked on every row of two heads, and causal GQA at S=8192, d=128 checked
# on sampled rows of one kv-head group.
FULL = [
    ("fp8_mha_b4_s2048_d64", Shape(4, 2048, 2048, 8, 8, 64, 64), 41, [(0, 0), (3, 7)], None),
    ("fp8_gqa_b4_s8192_d128", Shape(4, 8192, 8192, 32, 8, 128, 128), 42, [(2, 5)],
     np.r_[0:64, 1000:1040, 4090:4110, 8100:8192]),
]


@pytest.mark.parametrize("case", FULL, ids=[c[0] for c in FULL])
def test_fp8_forward_full_size_sampled(case):
    name, shape, seed, units, rows = case
    x = make_inputs(shape, seed, with_dout=False)
    o, lse = _gpu_fp8(x, causal=True, window=-1, softmax_type=VANILLA, scale=None)
    G = shape.H_q // shape.H_kv
    # the per-tensor scales come from the whole tensors' amax; the codes of a slice
    # are then the slice's own elementwise conversion
    xf = {n: x[n].float().numpy() for n in ("q", "k", "v")}
    amax = {n: np.float32(np.abs(xf[n]).max()) for n in xf}
    for b, g in units:
        hs = slice(g * G, (g + 1) * G)
        q8, _, dq = fp8.quantize(xf["q"][b:b + 1, :, hs], amax=amax["q"])
        k8, _, dk = fp8.quantize(xf["k"][b:b + 1, :, g:g + 1], amax=amax["k"])
        v8, _, dv = fp8.quantize(xf["v"][b:b + 1, :, g:g + 1], amax=amax["v"])
        ref = fp8.attention_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=True)
        bound = fp8.p_rounding_bound(fp8.dequantize(q8, dq), fp8.dequantize(k8, dk), fp8.dequantize(v8, dv),
                                     ref["lse"], causal=True, rows=rows)
        ob, lb = o[b:b + 1, :, hs], lse[b:b + 1, hs]
        if rows is not None:
            ref = {"o": ref["o"][:, rows], "lse": ref["lse"][:, :, rows]}
            ob, lb = ob[:, rows], lb[:, :, rows]
        _compare(ob, lb, ref, bound, f"{name} unit (b={b}, g={g})")
