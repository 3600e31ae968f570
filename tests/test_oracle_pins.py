"""Pins for the fp64 oracle: facts the pages and the mathematics fix, checked
without trusting the oracle's own formulas.

Each test names the passage it follows.  Together they are chosen so that a
plausible slip in the oracle (a dropped sink term, +e instead of +1, a wrong GQA
head index, an off-by-one window edge, a transposed operand, a wrong gradient
sign or a missing scale) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inp(shape, seed, learnable=False):
    t = make_inputs(shape, seed, learnable_offset=learnable)
    return {k: x.double().numpy() for k, x in t.items()}


def _visible_counts(Sq, Skv, causal, window):
    n = np.zeros(Sq, dtype=np.int64)
    for i in range(Sq):
        for j in range(Skv):
            if causal and j > i:
                continue
            if window >= 0 and j < i - window:
                continue
            n[i] += 1
    return n


# ---------------------------------------------------------------------------
# Worked examples, derived by hand (tests/golden/worked_examples.json)
# ---------------------------------------------------------------------------

def test_golden_worked_examples():
    """Hand-derived 2x2 cases of the four steps of "How attention works" in the
    cuDNN/TransformerEngine codelab, with the sink denominators of the sink
    attention PR (+1 for off-by-one, +exp(alpha) for learnable)."""
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    assert cases
    for c in cases:
        q = np.array(c["q"], dtype=np.float64)
        k = np.array(c["k"], dtype=np.float64)
        v = np.array(c["v"], dtype=np.float64)
        off = np.array(c["offset"], dtype=np.float64) if c.get("offset") is not None else None
        st = {"vanilla": VANILLA, "off_by_one": OFF_BY_ONE, "learnable": LEARNABLE}[c["softmax_type"]]
        f = oracle.attention_fwd(q, k, v, causal=c["causal"], window=c["window"], softmax_type=st,
                                 offset=off, scale=c["scale"])
        np.testing.assert_allclose(f["o"], np.array(c["expect_o"]), rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(f["lse"], np.array(c["expect_lse"]), rtol=0, atol=1e-14, err_msg=c["name"])
        if "dout" in c:
            dout = np.array(c["dout"], dtype=np.float64)
            g = oracle.attention_bwd(q, k, v, dout, causal=c["causal"], window=c["window"],
                                     softmax_type=st, offset=off, scale=c["scale"])
            np.testing.assert_allclose(g["d_offset"], np.array(c["expect_d_offset"]), rtol=0,
                                       atol=1e-14, err_msg=c["name"])


# ---------------------------------------------------------------------------
# P1 row sums (codelab: "softmax converts scores to attention weights that sum
# to 1"; the sink types leave the sink's share out of the visible weights)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("st", [VANILLA, OFF_BY_ONE, LEARNABLE])
def test_row_sums(st):
    s = Shape(1, 37, 37, 4, 2, 16, 8)
    x = _inp(s, 11, learnable=True)
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=9, softmax_type=st,
                             offset=x["offset"] if st == LEARNABLE else None, scale=0.3)
    if st == VANILLA:
        np.testing.assert_allclose(f["rowsum"], 1.0, atol=1e-13)
        assert np.all(f["psink"] == 0)
    else:
        assert np.all(f["psink"] > 0)
        np.testing.assert_allclose(f["rowsum"] + f["psink"], 1.0, atol=1e-13)


# ---------------------------------------------------------------------------
# P2 GQA == MHA with K/V heads repeated (TE page section 1: the baseline repeats
# K/V heads; codelab step 9: MHA/GQA/MQA share the output shape)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("Hkv", [1, 2])
def test_gqa_equals_repeated_mha(Hkv):
    Hq = 4
    G = Hq // Hkv
    s = Shape(2, 19, 23, Hq, Hkv, 8, 12)
    x = _inp(s, 3, learnable=True)
    kr = np.repeat(x["k"], G, axis=2)
    vr = np.repeat(x["v"], G, axis=2)
    for st in (VANILLA, LEARNABLE):
        off = x["offset"] if st == LEARNABLE else None
        a = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=False, softmax_type=st, offset=off)
        b = oracle.attention_fwd(x["q"], kr, vr, causal=False, softmax_type=st, offset=off)
        np.testing.assert_allclose(a["o"], b["o"], atol=1e-13)
        np.testing.assert_allclose(a["lse"], b["lse"], atol=1e-13)
        ga = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=False, softmax_type=st, offset=off)
        gb = oracle.attention_bwd(x["q"], kr, vr, x["dout"], causal=False, softmax_type=st, offset=off)
        np.testing.assert_allclose(ga["dq"], gb["dq"], atol=1e-12)
        dk_sum = gb["dk"].reshape(2, 23, Hkv, G, 8).sum(axis=3)
        dv_sum = gb["dv"].reshape(2, 23, Hkv, G, 12).sum(axis=3)
        np.testing.assert_allclose(ga["dk"], dk_sum, atol=1e-12)
        np.testing.assert_allclose(ga["dv"], dv_sum, atol=1e-12)
        np.testing.assert_allclose(ga["d_offset"], gb["d_offset"], atol=1e-12)


# ---------------------------------------------------------------------------
# P3 window edge cases (TE page: causal sliding window; reading: i-w <= j <= i)
# ---------------------------------------------------------------------------

def test_window_large_equals_causal_and_zero_is_identity():
    s = Shape(1, 33, 33, 2, 1, 8, 8)
    x = _inp(s, 5)
    c = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=-1)
    for w in (32, 33, 1000):
        ww = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=w)
        np.testing.assert_array_equal(ww["o"], c["o"])
        np.testing.assert_array_equal(ww["lse"], c["lse"])
    # window 31 must differ from causal on the last row only (it drops key 0 there)
    w31 = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=31)
    np.testing.assert_array_equal(w31["o"][:, :32], c["o"][:, :32])
    assert np.abs(w31["o"][:, 32] - c["o"][:, 32]).max() > 1e-6
    # window 0: every query sees only itself, so O_i = v_i exactly (vanilla)
    z = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=0)
    np.testing.assert_allclose(z["o"], np.repeat(x["v"], 2, axis=2), atol=1e-15)


# ---------------------------------------------------------------------------
# P4 closed forms: with Q = 0 every visible score is 0, so the weights are
# uniform over the visible keys and the sink contributes exp(c) (c = 0 for
# off-by-one, c = alpha_h for learnable).  This is where "+1" and "+e" differ by
# far more than any tolerance (the off-by-one review thread of the sink PR).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("st", [VANILLA, OFF_BY_ONE, LEARNABLE])
@pytest.mark.parametrize("window", [-1, 5])
def test_zero_query_closed_form(st, window):
    s = Shape(2, 17, 17, 3, 3, 8, 6)
    x = _inp(s, 7, learnable=True)
    q0 = np.zeros_like(x["q"])
    off = x["offset"] if st == LEARNABLE else None
    f = oracle.attention_fwd(q0, x["k"], x["v"], causal=True, window=window, softmax_type=st, offset=off)
    n = _visible_counts(17, 17, True, window)
    for b in range(2):
        for h in range(3):
            sink = {VANILLA: 0.0, OFF_BY_ONE: 1.0, LEARNABLE: math.exp(off[h]) if off is not None else 0}[st]
            for i in range(17):
                lo = 0 if window < 0 else max(0, i - window)
                vsum = x["v"][b, lo:i + 1, h].sum(axis=0)
                np.testing.assert_allclose(f["o"][b, i, h], vsum / (n[i] + sink), atol=1e-14)
                np.testing.assert_allclose(f["lse"][b, h, i], math.log(n[i] + sink), atol=1e-14)


def test_causal_row0_closed_forms():
    """Row 0 of a causal mask sees only key 0 (codelab step 7)."""
    s = Shape(1, 9, 9, 2, 2, 8, 8)
    x = _inp(s, 9)
    sc = 0.5
    van = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, scale=sc)
    np.testing.assert_allclose(van["o"][:, 0], x["v"][:, 0], atol=1e-15)
    obo = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, scale=sc, softmax_type=OFF_BY_ONE)
    for h in range(2):
        s00 = sc * float(x["q"][0, 0, h] @ x["k"][0, 0, h])
        sig = 1.0 / (1.0 + math.exp(-s00))
        np.testing.assert_allclose(obo["o"][0, 0, h], x["v"][0, 0, h] * sig, atol=1e-14)
        np.testing.assert_allclose(obo["lse"][0, h, 0], math.log1p(math.exp(s00)), atol=1e-14)


# ---------------------------------------------------------------------------
# P5 cross-type identities (sink PR: off-by-one is the learnable form with a
# zero logit; a very negative learnable logit removes the sink)
# ---------------------------------------------------------------------------

def test_cross_type_identities():
    s = Shape(1, 21, 21, 4, 2, 8, 8)
    x = _inp(s, 13)
    kw = dict(causal=True, window=7, scale=0.4)
    obo = oracle.attention_fwd(x["q"], x["k"], x["v"], softmax_type=OFF_BY_ONE, **kw)
    l0 = oracle.attention_fwd(x["q"], x["k"], x["v"], softmax_type=LEARNABLE, offset=np.zeros(4), **kw)
    np.testing.assert_allclose(l0["o"], obo["o"], atol=1e-15)
    np.testing.assert_allclose(l0["lse"], obo["lse"], atol=1e-15)
    van = oracle.attention_fwd(x["q"], x["k"], x["v"], **kw)
    lm = oracle.attention_fwd(x["q"], x["k"], x["v"], softmax_type=LEARNABLE, offset=np.full(4, -1e4), **kw)
    np.testing.assert_allclose(lm["o"], van["o"], atol=1e-15)
    np.testing.assert_allclose(lm["lse"], van["lse"], atol=1e-15)
    gobo = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], softmax_type=OFF_BY_ONE, **kw)
    gl0 = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], softmax_type=LEARNABLE,
                               offset=np.zeros(4), **kw)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(gl0[key], gobo[key], atol=1e-14)
    assert np.all(gobo["d_offset"] == 0)   # no parameter, no gradient
    assert np.abs(gl0["d_offset"]).max() > 1e-6


# ---------------------------------------------------------------------------
# P6 causal last row equals the unmasked last row (codelab step 7)
# ---------------------------------------------------------------------------

def test_causal_last_row_matches_full():
    s = Shape(2, 15, 15, 2, 1, 8, 8)
    x = _inp(s, 17)
    c = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True)
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=False)
    np.testing.assert_allclose(c["o"][:, -1], f["o"][:, -1], atol=1e-15)
    assert np.abs(c["o"][:, 0] - f["o"][:, 0]).max() > 1e-3


# ---------------------------------------------------------------------------
# P7 special case reducing to a library routine: torch's scaled_dot_product_attention
# in fp64 on the CPU (math backend), with an explicit boolean->additive mask,
# K/V heads repeated for GQA, and the sink written as one appended key whose k
# and v are zero (score 0 -> off-by-one) plus alpha_h added on that column
# (learnable).  Gradients, d_offset included, come from torch autograd.
# ---------------------------------------------------------------------------

def _torch_reference(x, causal, window, st, scale, lens_q=None, lens_kv=None):
    q = torch.tensor(x["q"]).permute(0, 2, 1, 3).requires_grad_(True)   # B,Hq,Sq,d
    k = torch.tensor(x["k"]).permute(0, 2, 1, 3).requires_grad_(True)
    v = torch.tensor(x["v"]).permute(0, 2, 1, 3).requires_grad_(True)
    B, Hq, Sq, dqk = q.shape
    Hkv, Skv, dv = k.shape[1], k.shape[2], v.shape[3]
    G = Hq // Hkv
    kk = k.repeat_interleave(G, dim=1)
    vv = v.repeat_interleave(G, dim=1)
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Skv)[None, :]
    allowed = torch.ones(Sq, Skv, dtype=torch.bool)
    if causal:
        allowed &= j <= i
    if window >= 0:
        allowed &= j >= i - window
    allowed = allowed.expand(B, Sq, Skv).clone()
    if lens_q is not None:
        # padded batch: keys past Lkv are masked; a padded query row keeps key 0 only
        # (its output is not compared and its dO is zero, so it adds no gradient)
        for b in range(B):
            allowed[b, :, lens_kv[b]:] = False
            allowed[b, lens_q[b]:, :] = False
            allowed[b, lens_q[b]:, 0] = True
    mask = torch.zeros(B, Sq, Skv, dtype=torch.float64).masked_fill(~allowed, float("-inf"))
    mask = mask[:, None].expand(B, Hq, Sq, Skv)
    off = None
    if st != VANILLA:
        kk = torch.cat([kk, torch.zeros(B, Hq, 1, dqk, dtype=torch.float64)], dim=2)
        vv = torch.cat([vv, torch.zeros(B, Hq, 1, dv, dtype=torch.float64)], dim=2)
        if st == LEARNABLE:
            off = torch.tensor(x["offset"]).requires_grad_(True)
            col = off[None, :, None, None].expand(B, Hq, Sq, 1)
        else:
            col = torch.zeros(B, Hq, Sq, 1, dtype=torch.float64)
        mask = torch.cat([mask, col], dim=3)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=scale)
    do = torch.tensor(x["dout"]).permute(0, 2, 1, 3).clone()
    if lens_q is not None:
        for b in range(B):
            do[b, :, lens_q[b]:] = 0
    (o * do).sum().backward()
    res = {"o": o.detach().permute(0, 2, 1, 3).numpy(),
           "dq": q.grad.permute(0, 2, 1, 3).numpy(),
           "dk": k.grad.permute(0, 2, 1, 3).numpy(),
           "dv": v.grad.permute(0, 2, 1, 3).numpy()}
    if off is not None:
        res["d_offset"] = off.grad.numpy()
    return res


@pytest.mark.parametrize("st", [VANILLA, OFF_BY_ONE, LEARNABLE])
@pytest.mark.parametrize("causal,window,Sq,Skv", [(True, -1, 29, 29), (True, 6, 29, 29),
                                                  (False, -1, 13, 31), (True, 4, 24, 40)])
def test_matches_torch_sdpa_fp64(st, causal, window, Sq, Skv):
    s = Shape(2, Sq, Skv, 4, 2, 16, 8)
    x = _inp(s, 23, learnable=True)
    scale = 0.37
    off = x["offset"] if st == LEARNABLE else None
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=causal, window=window, softmax_type=st,
                             offset=off, scale=scale)
    g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=causal, window=window,
                             softmax_type=st, offset=off, scale=scale)
    ref = _torch_reference(x, causal, window, st, scale)
    np.testing.assert_allclose(f["o"], ref["o"], atol=1e-12)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(g[key], ref[key], atol=1e-11)
    if st == LEARNABLE:
        np.testing.assert_allclose(g["d_offset"], ref["d_offset"], atol=1e-11)


def test_default_scale_is_inverse_sqrt_dqk():
    """MLA dims: the default scale uses the Q/K head dim (TE page section 4)."""
    s = Shape(1, 8, 8, 1, 1, 12, 4)
    x = _inp(s, 29)
    a = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True)
    b = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, scale=1 / math.sqrt(12))
    np.testing.assert_array_equal(a["o"], b["o"])
    c = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, scale=1 / math.sqrt(4))
    assert np.abs(a["o"] - c["o"]).max() > 1e-6


# ---------------------------------------------------------------------------
# P8 gradients by brute force: central differences of L = sum(dO * O) (and of
# LSE-free quantities) on tiny inputs, for dq, dk, dv and d_offset.
# ---------------------------------------------------------------------------

def _loss(x, key, val, **kw):
    y = dict(x)
    y[key] = val
    f = oracle.attention_fwd(y["q"], y["k"], y["v"], offset=y.get("offset"), **kw)
    return float((f["o"] * y["dout"]).sum())


@pytest.mark.parametrize("st,causal,window", [(VANILLA, True, 2), (OFF_BY_ONE, True, -1),
                                              (LEARNABLE, True, 3), (LEARNABLE, False, -1)])
def test_central_differences(st, causal, window):
    s = Shape(2, 6, 6, 4, 2, 3, 2)
    x = _inp(s, 31, learnable=True)
    kw = dict(causal=causal, window=window, softmax_type=st, scale=0.7)
    off = x["offset"] if st == LEARNABLE else None
    g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], offset=off, **kw)
    if st != LEARNABLE:
        x = {k: v for k, v in x.items() if k != "offset"}
    eps = 1e-6
    targets = [("q", "dq"), ("k", "dk"), ("v", "dv")] + ([("offset", "d_offset")] if st == LEARNABLE else [])
    for key, gkey in targets:
        base = x[key]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            p = base.copy(); p[idx] += eps
            m = base.copy(); m[idx] -= eps
            num[idx] = (_loss(x, key, p, **kw) - _loss(x, key, m, **kw)) / (2 * eps)
        np.testing.assert_allclose(g[gkey], num, atol=2e-8, rtol=1e-6, err_msg=f"{gkey} st={st}")


def test_D_is_rowdot_of_dout_and_o():
    s = Shape(1, 11, 11, 2, 1, 8, 8)
    x = _inp(s, 37, learnable=True)
    kw = dict(causal=True, window=4, softmax_type=LEARNABLE, offset=x["offset"])
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], **kw)
    g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **kw)
    D = np.einsum("bshd,bshd->bhs", x["dout"], f["o"])
    np.testing.assert_allclose(g["D"], D, atol=1e-13)
    # d_offset_h = -sum_{b,i} p_sink D  (derived from the learnable denominator)
    np.testing.assert_allclose(g["d_offset"], -(f["psink"] * D).sum(axis=(0, 2)), atol=1e-13)


# ---------------------------------------------------------------------------
# Edge cases of the definition: empty inputs and rows with no visible key
# ---------------------------------------------------------------------------

def test_empty_and_keyless_rows():
    s = Shape(1, 0, 5, 2, 1, 4, 4)
    x = _inp(s, 41)
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True)
    assert f["o"].shape == (1, 0, 2, 4)
    # window applied with causal on S_q > S_kv: rows i > S_kv - 1 + w see no key
    s = Shape(1, 8, 3, 1, 1, 4, 4)
    x = _inp(s, 43, learnable=True)
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=1)
    assert np.all(f["o"][0, 4:] == 0) and np.all(np.isneginf(f["lse"][0, 0, 4:]))
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=1, softmax_type=LEARNABLE,
                             offset=x["offset"])
    np.testing.assert_allclose(f["lse"][0, 0, 4:], x["offset"][0], atol=0)
    np.testing.assert_allclose(f["psink"][0, 0, 4:], 1.0, atol=0)


# ---------------------------------------------------------------------------
# Padded batches (per-entry lengths): the oracle runs each entry on its valid
# rows alone; torch gets the full padded tensors with the padding masked instead.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("st", [VANILLA, OFF_BY_ONE, LEARNABLE])
@pytest.mark.parametrize("causal,window", [(True, -1), (True, 5), (False, -1)])
def test_varlen_matches_torch_sdpa_fp64(st, causal, window):
    s = Shape(4, 21, 26, 4, 2, 16, 8)
    x = _inp(s, 31, learnable=True)
    lq, lkv = [21, 9, 1, 14], [26, 12, 7, 3]
    scale = 0.29
    off = x["offset"] if st == LEARNABLE else None
    kw = dict(seq_lens_q=lq, seq_lens_kv=lkv, causal=causal, window=window, softmax_type=st, offset=off,
              scale=scale)
    f = oracle.attention_fwd_varlen(x["q"], x["k"], x["v"], **kw)
    g = oracle.attention_bwd_varlen(x["q"], x["k"], x["v"], x["dout"], **kw)
    ref = _torch_reference(x, causal, window, st, scale, lq, lkv)
    for b in range(4):
        # valid rows that see at least one key (with causal top-left, rows >= Lkv see keys < Lkv)
        np.testing.assert_allclose(f["o"][b, :lq[b]], ref["o"][b, :lq[b]], atol=1e-12)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(g[key], ref[key], atol=1e-11)
    if st == LEARNABLE:
        np.testing.assert_allclose(g["d_offset"], ref["d_offset"], atol=1e-11)


def test_varlen_padding_and_full_lengths():
    s = Shape(3, 12, 10, 2, 1, 8, 8)
    x = _inp(s, 37, learnable=True)
    # full lengths reproduce the plain oracle exactly
    kw = dict(causal=True, window=4, softmax_type=LEARNABLE, offset=x["offset"])
    f0 = oracle.attention_fwd(x["q"], x["k"], x["v"], **kw)
    f1 = oracle.attention_fwd_varlen(x["q"], x["k"], x["v"], seq_lens_q=[12, 12, 12], seq_lens_kv=[10, 10, 10], **kw)
    g0 = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **kw)
    g1 = oracle.attention_bwd_varlen(x["q"], x["k"], x["v"], x["dout"], seq_lens_q=None, seq_lens_kv=[10] * 3, **kw)
    for key in ("o", "lse"):
        assert np.array_equal(f0[key], f1[key])
    for key in ("dq", "dk", "dv", "d_offset"):
        assert np.array_equal(g0[key], g1[key])
    # padded rows: O = 0 and LSE = the sink logit; padded keys and rows get no gradient;
    # an entry with no key (Lkv = 0) is all padding; lengths past S are clamped
    lq, lkv = [5, 12, 30], [0, 4, 10]
    for st in (VANILLA, OFF_BY_ONE, LEARNABLE):
        kw = dict(seq_lens_q=lq, seq_lens_kv=lkv, causal=True, softmax_type=st, offset=x["offset"])
        f = oracle.attention_fwd_varlen(x["q"], x["k"], x["v"], **kw)
        g = oracle.attention_bwd_varlen(x["q"], x["k"], x["v"], x["dout"], **kw)
        c = {VANILLA: -np.inf, OFF_BY_ONE: 0.0, LEARNABLE: None}[st]
        for b, (a, kk) in enumerate(zip([5, 12, 12], [0, 4, 10])):
            assert np.all(f["o"][b, a:] == 0) and np.all(g["dq"][b, a:] == 0)
            assert np.all(g["dk"][b, kk:] == 0) and np.all(g["dv"][b, kk:] == 0)
            for h in range(2):
                want = x["offset"][h] if st == LEARNABLE else c
                assert np.all(f["lse"][b, h, a:] == want)
        assert np.all(f["o"][0] == 0) and np.all(g["dq"][0] == 0)
        # a valid entry is the plain oracle on its own rows
        r = oracle.attention_fwd(x["q"][1:2, :12], x["k"][1:2, :4], x["v"][1:2, :4], causal=True, softmax_type=st,
                                 offset=x["offset"])
        assert np.array_equal(f["o"][1], r["o"][0])
