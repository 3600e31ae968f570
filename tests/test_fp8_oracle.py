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


# ----------------------------------------------------------------------------- E5M2 and the FP8 backward

def test_e5m2_decode_closed_forms_and_torch():
    d = fp8.e5m2_decode
    assert d(0x7B) == 57344.0                    # S.11110.11: largest finite
    assert d(0x01) == 2.0 ** -16                 # smallest subnormal
    assert d(0x04) == 2.0 ** -14                 # smallest normal
    assert d(0x3C) == 1.0 and d(0xBC) == -1.0    # exponent field 15 = bias
    assert d(0x3D) == 1.25 and d(0x3F) == 1.75
    assert d(0x7C) == np.inf and d(0xFC) == -np.inf
    assert np.isnan(d(0x7D)) and np.isnan(d(0x7F))
    codes = np.arange(256, dtype=np.uint8)
    ours = d(codes)
    theirs = torch.tensor(codes).view(torch.float8_e5m2).double().numpy()
    same = (ours == theirs) | (np.isnan(ours) & np.isnan(theirs))
    assert same.all()


def test_e5m2_encode_round_trip_ties_saturation_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.e5m2_decode(codes)
    fin = np.isfinite(vals)
    assert np.array_equal(fp8.e5m2_encode(vals[fin]), codes[fin])
    e = fp8.e5m2_encode
    assert e(1.125) == 0x3C                       # tie 1 | 1.25 -> even code 0x3C
    assert e(1.375) == 0x3E                       # tie 1.25 | 1.5 -> even code 0x3E
    assert e(70000.0) == 0x7B and e(-1e30) == 0xFB and e(np.inf) == 0x7B   # satfinite
    assert e(np.nan) == 0x7F
    x = np.random.default_rng(5).normal(0, 100, 20000) * np.exp2(np.random.default_rng(6).integers(-20, 8, 20000))
    x = x[np.abs(x) <= 57344.0]
    theirs = torch.tensor(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(e(x), theirs)


def test_e5m2_quantize_properties():
    x = np.random.default_rng(7).normal(size=(2, 40, 3, 64)).astype(np.float32)
    codes, amax, descale = fp8.quantize(x, fmt="e5m2")
    assert amax == np.float32(np.abs(x).max())
    back = fp8.dequantize(codes, descale, "e5m2")
    assert np.abs(back).max() == pytest.approx(amax, rel=2 ** -3)
    rel = np.abs(back - x) / np.maximum(np.abs(x), 2.0 ** -14 * float(descale))
    assert rel.max() <= 2.0 ** -3 + 1e-6          # half an E5M2 step (2 mantissa bits)
    t, _, _ = fp8.quantize(x, fmt="e5m2", transpose=True)
    assert np.array_equal(t, codes.transpose(0, 2, 3, 1))


def _fp8_bwd_case(seed, causal=True, window=-1, st=VANILLA, Sq=37, Skv=37, Hq=4, Hkv=2, d=16):
    rng = np.random.default_rng(seed)
    bf = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    q, k, v, do = (bf(rng.normal(size=s)) for s in ((2, Sq, Hq, d), (2, Skv, Hkv, d), (2, Skv, Hkv, d), (2, Sq, Hq, d)))
    off = rng.normal(size=Hq)
    q8, _, dq_ = fp8.quantize(q)
    k8, _, dk_ = fp8.quantize(k)
    v8, _, dv_ = fp8.quantize(v)
    do8, _, ddo = fp8.quantize(do, fmt="e5m2")
    kw = dict(causal=causal, window=window, softmax_type=st, offset=off if st == LEARNABLE else None, scale=0.3)
    deq = dict(q=fp8.dequantize(q8, dq_), k=fp8.dequantize(k8, dk_), v=fp8.dequantize(v8, dv_),
               do=fp8.dequantize(do8, ddo, "e5m2"))
    f = oracle.attention_fwd(deq["q"], deq["k"], deq["v"], **kw)
    return (q8, k8, v8, do8, dq_, dk_, dv_, ddo), deq, f, kw


@pytest.mark.parametrize("st,causal,window", [(VANILLA, True, -1), (LEARNABLE, True, 5), (OFF_BY_ONE, False, -1)])
def test_fp8_backward_without_roundings_is_the_exact_backward(st, causal, window):
    """With both roundings off, the FP8 backward's steps are the backward of the
    dequantised inputs: the C oracle's, computed on its own."""
    codes, deq, f, kw = _fp8_bwd_case(11, causal, window, st)
    got = fp8.attention_bwd_fp8(*codes, f["o"], f["lse"], 1.0, round_p=False, round_ds=False, **kw)
    ref = oracle.attention_bwd(deq["q"], deq["k"], deq["v"], deq["do"], **kw)
    for n in ("dq", "dk", "dv", "d_offset"):
        np.testing.assert_allclose(got[n], ref[n], rtol=0, atol=1e-10, err_msg=n)


def test_fp8_backward_roundings_match_torchs_casts():
    """The two roundings written with torch's own float8 casts: P as E4M3(256 P) / 256
    in dV, dS as E5M2(s dS) / s in dK and dQ."""
    codes, deq, f, kw = _fp8_bwd_case(13, True, -1, VANILLA)
    stat = 4.0  # covers this step's max |dS| (3.64), so nothing saturates (torch's cast would give inf)
    got = fp8.attention_bwd_fp8(*codes, f["o"], f["lse"], stat, **kw)
    s = float(np.float32(57344.0) / np.float32(stat))
    q, k, v, do = (torch.tensor(deq[n]) for n in ("q", "k", "v", "do"))
    o = torch.tensor(f["o"])
    B, Sq, Hq, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    mask = torch.tril(torch.ones(Sq, Skv, dtype=torch.bool))
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            S = 0.3 * q[b, :, h] @ k[b, :, g].T
            P = torch.where(mask, torch.exp(S - torch.tensor(f["lse"][b, h])[:, None]), torch.zeros(()))
            Pr = (P * 256).to(torch.float8_e4m3fn).double() / 256
            dP = do[b, :, h] @ v[b, :, g].T
            D = (do[b, :, h] * o[b, :, h]).sum(1)
            dS = P * (dP - D[:, None])
            dSr = (dS * s).to(torch.float8_e5m2).double() / s
            dv[b, :, g] += Pr.T @ do[b, :, h]
            dk[b, :, g] += 0.3 * dSr.T @ q[b, :, h]
            dq[b, :, h] = 0.3 * dSr @ k[b, :, g]
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got[n], t.numpy(), rtol=0, atol=1e-12, err_msg=n)
    assert got["amax_ds"] < stat


def test_fp8_backward_roundings_move_the_gradients_by_their_size():
    """The roundings are real but bounded: E4M3 P (3 bits) and E5M2 dS (2 bits) move
    the gradients by at most a few per cent in relative L2, and not at all when off."""
    codes, deq, f, kw = _fp8_bwd_case(17)
    exact = fp8.attention_bwd_fp8(*codes, f["o"], f["lse"], 1.0, round_p=False, round_ds=False, **kw)
    amax = exact["amax_ds"]
    r = fp8.attention_bwd_fp8(*codes, f["o"], f["lse"], amax, **kw)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 1e-4 < rel(r["dv"], exact["dv"]) < 2 ** -5
    for n in ("dq", "dk"):
        assert 1e-3 < rel(r[n], exact[n]) < 2 ** -3


@pytest.mark.parametrize("causal,window", [(True, -1), (True, 40), (False, -1)])
def test_fp8_backward_sampled_positions_match_the_full_result(causal, window):
    """q_idx / k_idx only restrict which rows and keys are summed, at their absolute
    positions: with all keys the dq rows, with all rows the dk / dv rows equal the
    full result's."""
    codes, deq, f, kw = _fp8_bwd_case(19, causal, window)
    kw.pop("offset"), kw.pop("softmax_type")
    full = fp8.attention_bwd_fp8(*codes, f["o"], f["lse"], 2.0, **kw)
    Sq, Skv = codes[0].shape[1], codes[1].shape[1]
    rows = np.array([0, 3, Sq // 2, Sq - 1])
    keys = np.array([1, Skv // 3, Skv - 2])
    a = fp8.attention_bwd_fp8(*codes, f["o"], f["lse"], 2.0, q_idx=rows, **kw)
    b = fp8.attention_bwd_fp8(*codes, f["o"], f["lse"], 2.0, k_idx=keys, **kw)
    np.testing.assert_array_equal(a["dq"], full["dq"][:, rows])
    np.testing.assert_allclose(b["dk"], full["dk"][:, keys], rtol=0, atol=1e-13)
    np.testing.assert_allclose(b["dv"], full["dv"][:, keys], rtol=0, atol=1e-13)


def _emulate_fp8_bwd_kernel(codes, o, lse, ds_amax, causal, window, scale):
    """The FP8 backward in the kernel's fp32 arithmetic: S and dP as fp32 sums of the
    codes' products; per row l' = -LSE log2(e) + 8 and D' = -D s / 2^8 (D = fp32 sum of
    dO8 O times descale); 2^8 P = 2^(S sl2 + l') and s dS = 2^8 P (dP dsc' + D') with
    dsc' = descale_do descale_v s / 2^8, each rounded to fp32; the two roundings of those
    fp32 values; the output sums scaled by the descales and rounded to bf16."""
    f32 = np.float32
    q8, k8, v8, do8, dsq, dsk, dsv, dsdo = codes
    q, k, v = (fp8.e4m3_decode(c).astype(f32) for c in (q8, k8, v8))
    do = fp8.e5m2_decode(do8).astype(f32)
    B, Sq, Hq, d = q.shape
    Skv, G = k.shape[1], Hq // k.shape[2]
    sc = f32(scale)
    log2e = f32(1.4426950408889634)
    sl2 = f32(f32(f32(sc * log2e) * f32(dsq)) * f32(dsk))
    s_ds = fp8.scale_from_amax(ds_amax, "e5m2")
    s8 = f32(s_ds / f32(256))
    dsc = f32(f32(f32(dsdo) * f32(dsv)) * s8)
    i, j = np.arange(Sq)[:, None], np.arange(Skv)[None, :]
    vis = np.ones((Sq, Skv), dtype=bool)
    if causal:
        vis &= j <= i
    if window >= 0:
        vis &= j >= i - window
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            lp = (-np.asarray(lse[b, h], dtype=f32) * log2e + f32(8)).astype(f32)[:, None]
            P8 = np.exp2(((q[b, :, h] @ k[b, :, g].T).astype(f32) * sl2 + lp).astype(f32)).astype(f32)
            P8 = np.where(vis, P8, f32(0))
            Pt = fp8.e4m3_decode(fp8.e4m3_encode(P8))
            D = (np.sum(do[b, :, h] * np.asarray(o[b, :, h], dtype=f32), axis=1, dtype=f32) * f32(dsdo)).astype(f32)
            Dp = (D * -s8).astype(f32)
            t = ((do[b, :, h] @ v[b, :, g].T).astype(f32) * dsc + Dp[:, None]).astype(f32)
            St = fp8.e5m2_decode(fp8.e5m2_encode((P8 * t).astype(f32)))
            dv[b, :, g] += (Pt.T @ do[b, :, h]) * float(dsdo) / 256
            dk[b, :, g] += (St.T @ q[b, :, h]) * float(sc * dsq / s_ds)
            dq[b, :, h] = (St @ k[b, :, g]) * float(sc * dsk / s_ds)
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16).double().numpy()
    return {"dq": bf(dq), "dk": bf(dk), "dv": bf(dv)}


@pytest.mark.parametrize("causal,window,seed", [(True, -1, 23), (True, 6, 29), (False, -1, 31)])
def test_fp8_backward_bound_covers_the_kernel_arithmetic_and_catches_missing_roundings(causal, window, seed):
    """The GPU tests' per-element FP8 backward tolerance (parity_util.fp8_bwd_bounds):
    an fp32 emulation of the kernel's arithmetic stays inside it, while the backward
    without either rounding leaves it on a large share of the elements."""
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    import parity_util as pu
    codes, deq, f, kw = _fp8_bwd_case(seed, causal, window)
    o = torch.from_numpy(f["o"]).to(torch.bfloat16).double().numpy()
    lse = f["lse"].astype(np.float32).astype(np.float64)
    kw = dict(causal=causal, window=window, scale=0.3)
    amax = np.float32(fp8.attention_bwd_fp8(*codes, o, lse, 1.0, **kw)["amax_ds"])
    ref = fp8.attention_bwd_fp8(*codes, o, lse, amax, **kw)
    bnd = pu.fp8_bwd_bounds(*codes, o, lse, amax, softmax_type=VANILLA, offset=None, **kw)
    ratios = pu.check_fp8_bwd(_emulate_fp8_bwd_kernel(codes, o, lse, amax, causal, window, 0.3), ref, bnd, "emu")
    assert max(ratios.values()) < 1.0
    assert bnd["flips"] < 0.1
    for variant in (dict(round_p=False), dict(round_ds=False)):
        wrong = fp8.attention_bwd_fp8(*codes, o, lse, amax, **variant, **kw)
        names = ("dv",) if "round_p" in variant else ("dq", "dk")
        for n in names:
            t = bnd["t_" + n]
            beyond = np.abs(wrong[n] - ref[n]) > t + pu.BF16_U * (np.abs(ref[n]) + t)
            assert beyond.mean() > 0.2, (variant, n, beyond.mean())
