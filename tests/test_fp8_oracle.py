"""Pins of the FP8 (E4M3) oracle: the codec against the format's closed forms, a
brute-force nearest search and torch's own E4M3 cast; per-tensor quantisation
against its defining properties; the P-rounding bound against an emulation of a
kernel that rounds its softmax numerators."""
import numpy as np
import pytest
import torch

import oracle
from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from oracle import fp8


def test_e4m3_decode_closed_forms():
    d = fp8.e4m3_decode
    assert d(0x7E) == 448.0                      # S.1111.110: largest finite
    assert d(0x01) == 2.0 ** -9                  # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9              # largest subnormal
    assert d(0x08) == 2.0 ** -6                  # smallest normal
    assert d(0x38) == 1.0                        # exponent field 7 = bias
    assert d(0xB8) == -1.0
    assert d(0x39) == 1.125 and d(0x3F) == 1.875
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    codes = np.arange(256, dtype=np.uint8)
    vals = d(codes)
    fin = np.isfinite(vals)
    assert fin.sum() == 254 and len(np.unique(vals[fin])) == 253  # +0 and -0 coincide
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0)               # increasing with the code


def test_e4m3_encode_round_trip_and_ties():
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.e4m3_decode(codes)
    fin = np.isfinite(vals)
    assert np.array_equal(fp8.e4m3_encode(vals[fin]), codes[fin])
    e = fp8.e4m3_encode
    assert e(1.0625) == 0x38                      # tie 1 | 1.125 -> even code 0x38
    assert e(1.1875) == 0x3A                      # tie 1.125 | 1.25 -> even code 0x3A
    assert e(2.0 ** -10) == 0x00                  # tie 0 | 2^-9 -> 0
    assert e(3 * 2.0 ** -10) == 0x02              # tie 2^-9 | 2^-8 -> even code 0x02
    assert e(1000.0) == 0x7E and e(-1e9) == 0xFE and e(464.0) == 0x7E  # satfinite
    assert e(-1e-12) == 0x80                      # sign kept when rounding to zero
    assert e(np.nan) == 0x7F


def test_e4m3_encode_matches_brute_force_nearest():
    rng = np.random.default_rng(0)
    codes = np.arange(0x7F)
    pos = fp8.e4m3_decode(codes.astype(np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    x = np.concatenate([rng.uniform(0, 460, 4000), np.exp(rng.uniform(-14, 6, 4000)), mids,
                        mids * (1 + 1e-12), mids * (1 - 1e-12)])
    x = np.concatenate([x, -x])
    got = fp8.e4m3_encode(x)
    a = np.minimum(np.abs(x), 448.0)
    dist = np.abs(a[:, None] - pos[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = np.where(dist == best, codes[None, :], 1000)
    # among equidistant codes the even one; otherwise the unique nearest
    even = np.where((cand % 2 == 0) & (cand < 1000), cand, 1000).min(axis=1)
    want = np.where((dist == best).sum(axis=1) > 1, even, cand.min(axis=1))
    want = want | np.where(np.signbit(x), 0x80, 0)
    assert np.array_equal(got, want.astype(np.uint8))


def test_e4m3_encode_matches_torch_cast_in_range():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 30, 20000), rng.uniform(-448, 448, 20000),
                        np.exp(rng.uniform(-16, 6, 5000))]).astype(np.float32)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), t)


def test_quantize_per_tensor_amax_scaling():
    x = torch.randn(2, 64, 3, 32, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    xf = x.float().numpy()
    codes, amax, descale = fp8.quantize(xf)
    assert amax == np.float32(np.abs(xf).max())
    scale = np.float32(448.0) / amax
    assert descale == np.float32(1.0) / scale
    # the amax element lands on +-448; every value within half an E4M3 step
    assert np.max(np.abs(fp8.e4m3_decode(codes))) == 448.0
    deq = fp8.dequantize(codes, descale)
    rel = np.abs(deq - xf) / np.maximum(np.abs(xf), 2.0 ** -6 * amax / 448.0)
    assert np.all(rel <= 2.0 ** -4 * (1 + 1e-6))
    # transposed layout [B,H,d,S] holds the same codes
    ct, _, _ = fp8.quantize(xf, transpose=True)
    assert np.array_equal(ct, codes.transpose(0, 2, 3, 1))
    # a zero tensor: scale 1, codes 0
    z, za, zd = fp8.quantize(np.zeros((1, 4, 1, 8), np.float32))
    assert za == 0 and zd == 1 and not z.any()


def test_fp8_forward_of_representable_inputs_is_the_plain_forward():
    """Inputs that are E4M3 values times a power of two survive quantisation
    exactly, so the FP8 oracle must equal the plain oracle on them bit for bit."""
    rng = np.random.default_rng(4)
    shape = (1, 40, 2, 16)
    mk = lambda: fp8.e4m3_decode(rng.integers(0, 0x7F, shape, dtype=np.uint8) | np.where(
        rng.random(shape) < 0.5, 0x80, 0).astype(np.uint8)) * 2.0 ** -5
    q, k, v = mk(), mk(), mk()
    for t in (q, k, v):
        t.flat[0] = 448.0 * 2.0 ** -5             # pins amax: scale = 2^5 exactly
    q8, _, dq = fp8.quantize(q)
    k8, _, dk = fp8.quantize(k)
    v8, _, dv = fp8.quantize(v)
    assert dq == dk == dv == np.float32(2.0 ** -5)
    a = fp8.attention_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=True, window=7)
    b = oracle.attention_fwd(q, k, v, causal=True, window=7)
    assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["lse"], b["lse"])


@pytest.mark.parametrize("st", [VANILLA, OFF_BY_ONE, LEARNABLE])
def test_p_rounding_bound_covers_an_emulated_kernel(st):
    """Round p_j = exp(s_j - m') to E4M3 for stale maxima m' anywhere in
    [M - 8 ln 2, M] (the lazy rescale's range), keep the denominator exact, and
    check every output element against the bound."""
    rng = np.random.default_rng(10 + st)
    B, S, H, d = 1, 150, 2, 32
    q = rng.normal(0, 1.5, (B, S, H, d))
    k = rng.normal(0, 1.5, (B, S, H, d))
    v = rng.normal(0, 1, (B, S, H, d))
    off = rng.normal(0, 1, H)
    kw = dict(causal=True, window=60, softmax_type=st, offset=off if st == LEARNABLE else None)
    ref = oracle.attention_fwd(q, k, v, **kw)
    bound = fp8.p_rounding_bound(q, k, v, ref["lse"], causal=True, window=60, softmax_type=st,
                                 offset=off)
    sc = 1 / np.sqrt(d)
    worst = 0.0
    for h in range(H):
        s = sc * q[0, :, h] @ k[0, :, h].T
        i, j = np.arange(S)[:, None], np.arange(S)[None, :]
        vis = (j <= i) & (j >= i - 60)
        s = np.where(vis, s, -np.inf)
        c = {VANILLA: -np.inf, OFF_BY_ONE: 0.0, LEARNABLE: off[h]}[st]
        M = np.maximum(s.max(axis=1), c)
        for delta in (0.0, 2.5, 8 * np.log(2) * 0.999):
            mp = (M - delta)[:, None]
            p = np.where(vis, np.exp(s - mp), 0.0)
            l = p.sum(axis=1) + np.exp(c - mp[:, 0])
            pr = fp8.e4m3_decode(fp8.e4m3_encode(p))
            o = (pr @ v[0, :, h]) / l[:, None]
            err = np.abs(o - ref["o"][0, :, h]).max(axis=1)
            assert np.all(err <= bound[0, h] * (1 + 1e-9) + 1e-12)
            worst = max(worst, float((err / bound[0, h]).max()))
    assert worst > 0.3             # and it is tight: some element reaches 30 % of it
