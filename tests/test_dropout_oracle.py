"""Pins for the oracle's attention dropout.

"JAX: Single-GPU Attention with TransformerEngine", section "Other attention knobs",
offers `attention_dropout`.  The sequence diagrams of "[JAX] Add support for sink
attention in JAX #2225" show the fused forward returning an rng_state that the fused
backward takes.  The oracle reads this as a counter-based generator,
Philox4x64-10 (Salmon et al., SC'11).  The generator is keyed by rng_state =
(seed, offset), and its 16-bit fields decide each (query, key) pair.  These tests
pin the oracle against things it does not compute itself:
  * the generator against numpy's Philox bit generator, a library implementation of
    the same published algorithm;
  * the keep rate against binomial bounds;
  * p = 0 against the plain oracle;
  * the dropped forward and backward against torch autograd in fp64 on the same keep
    decisions (torch's softmax and matmul, not the oracle's loops);
  * the gradients against central differences on tiny inputs (the decisions are fixed
    by the seed, so the function is smooth).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs

U64 = 2 ** 64 - 1


def _inp(shape, seed):
    return {k: x.double().numpy() for k, x in make_inputs(shape, seed, learnable_offset=True).items()}


@pytest.mark.parametrize("counter,key", [
    ((1, 0, 0, 0), (0, 0)),
    ((7, 3, 2, 1), (12345, 678)),
    ((2 ** 40 + 5, 2 ** 63, U64, 17), (U64, 2 ** 62 + 11)),
    ((123456789, 987654321, 31, 4), (0x243F6A8885A308D3, 0x13198A2E03707344)),
])
def test_philox_matches_numpy_bit_generator(counter, key):
    """numpy's Philox increments its counter before each block, so the block numpy
    produces from counter c - 1 is the Philox of c (c0 >= 1 here: no carry)."""
    start = np.array([counter[0] - 1, *counter[1:]], dtype=np.uint64)
    ref = np.random.Philox(counter=start, key=np.array(key, dtype=np.uint64)).random_raw(4)
    np.testing.assert_array_equal(oracle.philox4x64_10(counter, key), ref.astype(np.uint64))


def test_threshold_rule():
    assert oracle.dropout_threshold(0.0) == 0
    assert oracle.dropout_threshold(0.5) == 32768
    assert oracle.dropout_threshold(0.1) == 6554          # 6553.6 rounds up
    assert oracle.dropout_threshold(1.0 - 2 ** -17 - 2 ** -30) == 65535
    for bad in (-0.1, 1.0, 1.0 - 2 ** -18):
        with pytest.raises(ValueError):
            oracle.dropout_threshold(bad)


@pytest.mark.parametrize("p", [0.1, 0.5])
def test_keep_rate_within_binomial_bounds(p):
    n_rows, n_cols = 512, 512
    keep = np.concatenate([oracle.dropout_keep(b, h, n_rows, n_cols, p, (2024, 7)).ravel()
                           for b in range(2) for h in range(3)])
    q = 1.0 - oracle.dropout_threshold(p) / 65536.0
    n = keep.size
    assert abs(keep.mean() - q) <= 5.0 * np.sqrt(q * (1 - q) / n)
    # neighbouring pairs (same generator call) are not correlated
    a = oracle.dropout_keep(0, 0, n_rows, n_cols, p, (2024, 7)).astype(np.float64)
    for da, db in ((0, 1), (1, 0), (1, 1), (0, 4)):
        x, y = a[:n_rows - da, :n_cols - db].ravel(), a[da:, db:].ravel()
        assert abs(np.corrcoef(x, y)[0, 1]) <= 5.0 / np.sqrt(x.size)


def test_seed_offset_batch_and_head_change_the_decisions():
    base = oracle.dropout_keep(0, 0, 64, 64, 0.5, (1, 2))
    for other in (oracle.dropout_keep(0, 0, 64, 64, 0.5, (2, 2)), oracle.dropout_keep(0, 0, 64, 64, 0.5, (1, 3)),
                  oracle.dropout_keep(1, 0, 64, 64, 0.5, (1, 2)), oracle.dropout_keep(0, 1, 64, 64, 0.5, (1, 2))):
        assert 0.4 < np.mean(base != other) < 0.6
    np.testing.assert_array_equal(base, oracle.dropout_keep(0, 0, 64, 64, 0.5, (1, 2)))


@pytest.mark.parametrize("st", [VANILLA, LEARNABLE])
def test_zero_probability_is_the_plain_oracle(st):
    s = Shape(1, 40, 40, 2, 1, 16, 16)
    x = _inp(s, 3)
    kw = dict(causal=True, window=10, softmax_type=st, offset=x["offset"], scale=0.3)
    a = oracle.attention_fwd(x["q"], x["k"], x["v"], **kw)
    b = oracle.attention_fwd(x["q"], x["k"], x["v"], dropout_p=0.0, rng_state=(5, 6), **kw)
    np.testing.assert_array_equal(a["o"], b["o"])
    ga = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **kw)
    gb = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], dropout_p=0.0, rng_state=(5, 6), **kw)
    for key in ("dq", "dk", "dv", "d_offset"):
        np.testing.assert_array_equal(ga[key], gb[key])


def _torch_dropout_reference(x, causal, window, st, scale, p, rng):
    """Attention with torch's fp64 softmax and matmul, the sink as an extra logit
    column, and the oracle's keep decisions applied to the probabilities."""
    q = torch.tensor(x["q"]).permute(0, 2, 1, 3).requires_grad_(True)
    k = torch.tensor(x["k"]).permute(0, 2, 1, 3).requires_grad_(True)
    v = torch.tensor(x["v"]).permute(0, 2, 1, 3).requires_grad_(True)
    B, Hq, Sq, _ = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    s = scale * q @ k.repeat_interleave(G, dim=1).transpose(-1, -2)
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Skv)[None, :]
    allowed = torch.ones(Sq, Skv, dtype=torch.bool)
    if causal:
        allowed &= j <= i
    if window >= 0:
        allowed &= j >= i - window
    s = s.masked_fill(~allowed, float("-inf"))
    off = None
    if st != VANILLA:
        if st == LEARNABLE:
            off = torch.tensor(x["offset"]).requires_grad_(True)
            col = off[None, :, None, None].expand(B, Hq, Sq, 1)
        else:
            col = torch.zeros(B, Hq, Sq, 1, dtype=torch.float64)
        s = torch.cat([s, col], dim=3)
    P = torch.softmax(s, dim=3)[..., :Skv]
    t = oracle.dropout_threshold(p)
    keep = np.stack([np.stack([oracle.dropout_keep(b, h, Sq, Skv, p, rng) for h in range(Hq)]) for b in range(B)])
    M = torch.tensor(keep, dtype=torch.float64) * (65536.0 / (65536.0 - t))
    o = (P * M) @ v.repeat_interleave(G, dim=1)
    (o * torch.tensor(x["dout"]).permute(0, 2, 1, 3)).sum().backward()
    res = {"o": o.detach().permute(0, 2, 1, 3).numpy(), "dq": q.grad.permute(0, 2, 1, 3).numpy(),
           "dk": k.grad.permute(0, 2, 1, 3).numpy(), "dv": v.grad.permute(0, 2, 1, 3).numpy()}
    if off is not None:
        res["d_offset"] = off.grad.numpy()
    return res


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("st,causal,window,Sq,Skv", [(VANILLA, True, -1, 29, 29), (OFF_BY_ONE, True, 6, 29, 29),
                                                     (LEARNABLE, False, -1, 13, 31), (LEARNABLE, True, 4, 24, 40)])
def test_dropout_matches_torch_autograd_fp64(p, st, causal, window, Sq, Skv):
    s = Shape(2, Sq, Skv, 4, 2, 16, 8)
    x = _inp(s, 41)
    rng = (0x5EED, 3)
    off = x["offset"] if st == LEARNABLE else None
    kw = dict(causal=causal, window=window, softmax_type=st, offset=off, scale=0.37, dropout_p=p, rng_state=rng)
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], **kw)
    g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **kw)
    ref = _torch_dropout_reference(x, causal, window, st, 0.37, p, rng)
    np.testing.assert_allclose(f["o"], ref["o"], atol=1e-12)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(g[key], ref[key], atol=1e-11)
    if st == LEARNABLE:
        np.testing.assert_allclose(g["d_offset"], ref["d_offset"], atol=1e-11)
    # the undropped statistics: LSE is the softmax's, whatever is dropped
    plain = oracle.attention_fwd(x["q"], x["k"], x["v"], **dict(kw, dropout_p=0.0))
    np.testing.assert_array_equal(f["lse"], plain["lse"])


def test_dropout_central_differences():
    s = Shape(1, 6, 6, 2, 1, 3, 2)
    x = _inp(s, 43)
    kw = dict(causal=True, window=-1, softmax_type=LEARNABLE, scale=0.7, dropout_p=0.5, rng_state=(9, 1))
    g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], offset=x["offset"], **kw)

    def loss(key, val):
        y = dict(x)
        y[key] = val
        f = oracle.attention_fwd(y["q"], y["k"], y["v"], offset=y["offset"], **kw)
        return float((f["o"] * y["dout"]).sum())

    eps = 1e-6
    for key, gkey in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("offset", "d_offset")):
        base = x[key]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            pp = base.copy(); pp[idx] += eps
            mm = base.copy(); mm[idx] -= eps
            num[idx] = (loss(key, pp) - loss(key, mm)) / (2 * eps)
        np.testing.assert_allclose(g[gkey], num, atol=2e-8, rtol=1e-6, err_msg=gkey)


def test_dropout_origin_takes_the_decisions_of_the_bigger_problem():
    """A slice (batch entry 1, query heads 2..3 with kv head 1) computed on its own with
    dropout_origin = (1, 2) equals that slice of the whole problem."""
    s = Shape(2, 20, 20, 4, 2, 8, 8)
    x = _inp(s, 45)
    kw = dict(causal=True, softmax_type=VANILLA, scale=0.5, dropout_p=0.5, rng_state=(3, 4))
    f = oracle.attention_fwd(x["q"], x["k"], x["v"], **kw)
    g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], **kw)
    sl = lambda a, hs: a[1:2, :, hs].copy()
    fu = oracle.attention_fwd(sl(x["q"], slice(2, 4)), sl(x["k"], slice(1, 2)), sl(x["v"], slice(1, 2)),
                              dropout_origin=(1, 2), **kw)
    gu = oracle.attention_bwd(sl(x["q"], slice(2, 4)), sl(x["k"], slice(1, 2)), sl(x["v"], slice(1, 2)),
                              sl(x["dout"], slice(2, 4)), dropout_origin=(1, 2), **kw)
    np.testing.assert_array_equal(fu["o"], f["o"][1:2, :, 2:4])
    np.testing.assert_array_equal(gu["dq"], g["dq"][1:2, :, 2:4])
    np.testing.assert_allclose(gu["dk"], g["dk"][1:2, :, 1:2], atol=1e-14)
