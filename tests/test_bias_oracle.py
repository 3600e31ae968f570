"""Pins of the oracle's additive bias (and dbias): torch's fp64 math SDPA with the bias
as a float mask and autograd for every gradient (dbias = the mask's gradient, summed
over broadcast dims by torch itself), finite differences on a tiny case, and the
special cases bias = 0 and bias = -inf outside the causal triangle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import LEARNABLE, OFF_BY_ONE, VANILLA


def _inputs(B, Sq, Skv, Hq, Hkv, d, seed, st, bias_shape):
    rng = np.random.default_rng(seed)
    x = {"q": rng.normal(size=(B, Sq, Hq, d)), "k": rng.normal(size=(B, Skv, Hkv, d)),
         "v": rng.normal(size=(B, Skv, Hkv, d)), "dout": rng.normal(size=(B, Sq, Hq, d)),
         "offset": rng.normal(size=(Hq,)), "bias": rng.normal(0, 2.0, size=bias_shape)}
    return x


def _torch(x, causal, window, st, scale):
    q = torch.tensor(x["q"]).permute(0, 2, 1, 3).requires_grad_(True)
    k = torch.tensor(x["k"]).permute(0, 2, 1, 3).requires_grad_(True)
    v = torch.tensor(x["v"]).permute(0, 2, 1, 3).requires_grad_(True)
    bias = torch.tensor(x["bias"]).requires_grad_(True)
    B, Hq, Sq, d = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    i, j = torch.arange(Sq)[:, None], torch.arange(Skv)[None, :]
    allowed = torch.ones(Sq, Skv, dtype=torch.bool)
    if causal:
        allowed &= j <= i
    if window >= 0:
        allowed &= j >= i - window
    mask = bias.expand(B, Hq, Sq, Skv) + torch.zeros(Sq, Skv, dtype=torch.float64).masked_fill(
        ~allowed, float("-inf"))
    if st != VANILLA:  # the sink as one more key with a zero value vector
        kk = torch.cat([kk, torch.zeros(B, Hq, 1, d, dtype=torch.float64)], dim=2)
        vv = torch.cat([vv, torch.zeros(B, Hq, 1, d, dtype=torch.float64)], dim=2)
        c = torch.tensor(x["offset"]) if st == LEARNABLE else torch.zeros(Hq, dtype=torch.float64)
        mask = torch.cat([mask, c[None, :, None, None].expand(B, Hq, Sq, 1)], dim=3)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=scale)
    (o * torch.tensor(x["dout"]).permute(0, 2, 1, 3)).sum().backward()
    return {"o": o.detach().permute(0, 2, 1, 3).numpy(), "dq": q.grad.permute(0, 2, 1, 3).numpy(),
            "dk": k.grad.permute(0, 2, 1, 3).numpy(), "dv": v.grad.permute(0, 2, 1, 3).numpy(),
            "dbias": bias.grad.numpy()}


CASES = [
    # B, Sq, Skv, Hq, Hkv, d, causal, window, softmax type, bias shape (Bb, Hb)
    (2, 9, 9, 4, 2, 8, True, -1, VANILLA, (1, 4)),
    (2, 9, 9, 4, 2, 8, True, 3, OFF_BY_ONE, (2, 1)),
    (1, 7, 11, 2, 1, 8, False, -1, LEARNABLE, (1, 1)),
    (2, 12, 12, 2, 2, 4, True, 5, VANILLA, (2, 2)),
]


@pytest.mark.parametrize("case", CASES)
def test_bias_matches_torch_sdpa_with_autograd(case):
    B, Sq, Skv, Hq, Hkv, d, causal, window, st, (Bb, Hb) = case
    x = _inputs(B, Sq, Skv, Hq, Hkv, d, 7, st, (Bb, Hb, Sq, Skv))
    scale = 0.4
    kw = dict(causal=causal, window=window, softmax_type=st, scale=scale, bias=x["bias"],
              offset=x["offset"] if st == LEARNABLE else None)
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], **kw)
    g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **kw)
    t = _torch(x, causal, window, st, scale)
    np.testing.assert_allclose(f["o"], t["o"], rtol=0, atol=1e-12)
    for n in ("dq", "dk", "dv", "dbias"):
        np.testing.assert_allclose(g[n], t[n], rtol=0, atol=1e-11, err_msg=n)
    assert g["dbias"].shape == (Bb, Hb, Sq, Skv)


def test_dbias_by_finite_differences():
    B, S, H, d = 1, 5, 2, 4
    x = _inputs(B, S, S, H, H, d, 3, OFF_BY_ONE, (1, H, S, S))
    kw = dict(causal=True, window=-1, softmax_type=OFF_BY_ONE, scale=0.5)

    def loss(bias):
        return float((oracle.attention_fwd(x["q"], x["k"], x["v"], bias=bias, **kw)["o"] * x["dout"]).sum())

    g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], bias=x["bias"], **kw)["dbias"]
    eps = 1e-6
    for h, i, j in [(0, 0, 0), (1, 3, 1), (0, 4, 4), (1, 2, 2), (0, 1, 3)]:
        bp, bm = x["bias"].copy(), x["bias"].copy()
        bp[0, h, i, j] += eps
        bm[0, h, i, j] -= eps
        num = (loss(bp) - loss(bm)) / (2 * eps)
        assert abs(num - g[0, h, i, j]) < 1e-7, (h, i, j, num, g[0, h, i, j])
    assert g[0, 1, 1, 3] == 0.0  # a masked pair (j > i) has no gradient


def test_zero_bias_and_minus_inf_bias_special_cases():
    B, S, Hq, Hkv, d = 2, 10, 4, 2, 8
    x = _inputs(B, S, S, Hq, Hkv, d, 5, VANILLA, (1, 1, S, S))
    plain = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=4)
    zero = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=4, bias=np.zeros((1, 1, S, S)))
    assert np.array_equal(plain["o"], zero["o"]) and np.array_equal(plain["lse"], zero["lse"])
    # -inf above the diagonal on a non-causal call equals the causal call
    tri = np.where(np.arange(S)[None, :] > np.arange(S)[:, None], -np.inf, 0.0)[None, None]
    a = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=False, bias=tri)
    b = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True)
    np.testing.assert_allclose(a["o"], b["o"], rtol=0, atol=1e-14)
    ga = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=False, bias=tri)
    gb = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=True)
    for n in ("dq", "dk", "dv"):
        np.testing.assert_allclose(ga[n], gb[n], rtol=0, atol=1e-13)
    assert np.all(ga["dbias"][0, 0][np.isinf(tri[0, 0])] == 0)
    # a bias constant along each row shifts every logit of the row alike: O unchanged,
    # LSE shifted by the constant, and (vanilla) each row of dbias sums to zero
    rowc = np.broadcast_to(np.arange(S, dtype=np.float64)[:, None], (S, S))[None, None]
    r = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=True, window=4, bias=rowc)
    np.testing.assert_allclose(r["o"], plain["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["lse"], plain["lse"] + np.arange(S)[None, None], rtol=0, atol=1e-12)
    gr = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=True, window=4, bias=rowc)
    np.testing.assert_allclose(gr["dbias"].sum(axis=3), 0.0, atol=1e-12)


@pytest.mark.parametrize("st,causal,window,bias_bh", [(VANILLA, True, -1, (1, 4)), (LEARNABLE, True, 3, (2, 1)),
                                                      (OFF_BY_ONE, False, -1, (2, 4))])
def test_bias_with_padded_batches_matches_torch(st, causal, window, bias_bh):
    """A padded batch with a bias: each entry uses the top-left [Lq, Lkv] corner of its
    bias planes.  Torch gets the full padded tensors with the padding masked, the bias
    in the additive mask, and dO = 0 on padded rows (a padded row keeps key 0 so that
    its softmax is defined; it adds nothing); dbias comes from autograd and is zero
    outside each entry's corner."""
    B, S, Hq, Hkv, d = 2, 10, 4, 2, 8
    lq, lkv = [7, 10], [10, 6] if not causal else [7, 10]
    x = _inputs(B, S, S, Hq, Hkv, d, 11, st, (*bias_bh, S, S))
    for b in range(B):
        x["dout"][b, lq[b]:] = 0.0
    kw = dict(causal=causal, window=window, softmax_type=st, scale=0.4, bias=x["bias"],
              offset=x["offset"] if st == LEARNABLE else None, seq_lens_q=lq, seq_lens_kv=lkv)
    f = oracle.attention_fwd_varlen(x["q"], x["k"], x["v"], **kw)
    g = oracle.attention_bwd_varlen(x["q"], x["k"], x["v"], x["dout"], **kw)
    # torch: the padding as -inf in the additive mask, through a bias of the padded shape
    pad = np.zeros((B, 1, S, S))
    for b in range(B):
        pad[b, :, :, lkv[b]:] = -np.inf
        pad[b, :, lq[b]:, :] = -np.inf
        pad[b, :, lq[b]:, 0] = 0.0
    bias_t = torch.tensor(x["bias"]).requires_grad_(True)
    q = torch.tensor(x["q"]).permute(0, 2, 1, 3).requires_grad_(True)
    k = torch.tensor(x["k"]).permute(0, 2, 1, 3).requires_grad_(True)
    v = torch.tensor(x["v"]).permute(0, 2, 1, 3).requires_grad_(True)
    G = Hq // Hkv
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    i, j = torch.arange(S)[:, None], torch.arange(S)[None, :]
    allowed = torch.ones(S, S, dtype=torch.bool)
    if causal:
        allowed &= j <= i
    if window >= 0:
        allowed &= j >= i - window
    mask = (bias_t.expand(B, Hq, S, S) + torch.tensor(pad)
            + torch.zeros(S, S, dtype=torch.float64).masked_fill(~allowed, float("-inf")))
    for b in range(B):  # a padded row keeps key 0 whatever the causal mask says
        mask = mask.clone()
        mask[b, :, lq[b]:, 0] = bias_t.expand(B, Hq, S, S)[b, :, lq[b]:, 0]
    if st != VANILLA:
        kk = torch.cat([kk, torch.zeros(B, Hq, 1, d, dtype=torch.float64)], dim=2)
        vv = torch.cat([vv, torch.zeros(B, Hq, 1, d, dtype=torch.float64)], dim=2)
        c = torch.tensor(x["offset"]) if st == LEARNABLE else torch.zeros(Hq, dtype=torch.float64)
        mask = torch.cat([mask, c[None, :, None, None].expand(B, Hq, S, 1)], dim=3)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=0.4)
    (o * torch.tensor(x["dout"]).permute(0, 2, 1, 3)).sum().backward()
    o = o.detach().permute(0, 2, 1, 3).numpy()
    for b in range(B):
        np.testing.assert_allclose(f["o"][b, :lq[b]], o[b, :lq[b]], rtol=0, atol=1e-12)
        assert np.all(f["o"][b, lq[b]:] == 0)
    np.testing.assert_allclose(g["dq"], q.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g["dk"], k.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g["dv"], v.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g["dbias"], bias_t.grad.numpy(), rtol=0, atol=1e-11)
    assert g["dbias"].shape == x["bias"].shape
