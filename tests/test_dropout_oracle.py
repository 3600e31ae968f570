"""Pins for the oracle's attention dropout.

"JAX: Single-GPU Attention with TransformerEngine", section "Other attention knobs",
offers `attention_dropout`.  The sequence diagrams of "[JAX] Add support for sink
attention in JAX #2225" show the fused forward returning an rng_state that the fused
backward takes.  The oracle reads this as a counter-based generator,
Philox4x32-10 (Salmon et al., SC'11).  The generator is keyed by the seed of
rng_state = (seed, offset), and its 16-bit fields decide each (query, key) pair.
These tests pin the oracle against things it does not compute itself:
  * the generator against the known-answer vectors published with the Random123
    library (the SC'11 paper's reference implementation), and against Triton's
    `tl.philox`, a library implementation of the same algorithm, run by Triton's CPU
    interpreter;
  * the keep rate against binomial bounds;
  * p = 0 against the plain oracle;
  * the dropped forward and backward against torch autograd in fp64 on the same keep
    decisions (torch's softmax and matmul, not the oracle's loops);
  * the gradients against central differences on tiny inputs (the decisions are fixed
    by the seed, so the function is smooth).
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs

U32 = 2 ** 32 - 1


def _inp(shape, seed):
    return {k: x.double().numpy() for k, x in make_inputs(shape, seed, learnable_offset=True).items()}


# Philox4x32-10 known-answer vectors of the Random123 distribution (counter, key, output)
KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((U32, U32, U32, U32), (U32, U32), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("counter,key,expected", KAT)
def test_philox_known_answers(counter, key, expected):
    np.testing.assert_array_equal(oracle.philox4x32_10(counter, key), np.array(expected, dtype=np.uint32))


_TRITON_PHILOX = """
import json, sys
import torch, triton, triton.language as tl

@triton.jit
def philox_kernel(seed_ptr, ctr_ptr, out_ptr, N: tl.constexpr):
    n = tl.arange(0, N)
    seed = tl.load(seed_ptr + n)
    a, b, c, d = tl.philox(seed, tl.load(ctr_ptr + 4 * n), tl.load(ctr_ptr + 4 * n + 1),
                           tl.load(ctr_ptr + 4 * n + 2), tl.load(ctr_ptr + 4 * n + 3), 10)
    tl.store(out_ptr + 4 * n, a)
    tl.store(out_ptr + 4 * n + 1, b)
    tl.store(out_ptr + 4 * n + 2, c)
    tl.store(out_ptr + 4 * n + 3, d)

args = json.loads(sys.stdin.read())
n = len(args["seeds"])
out = torch.zeros(4 * n, dtype=torch.int32)
philox_kernel[(1,)](torch.tensor(args["seeds"], dtype=torch.int64), torch.tensor(args["ctr"], dtype=torch.int32),
                    out, N=n)
print(json.dumps(out.tolist()))
"""


def test_philox_matches_triton_library_generator():
    """Triton's tl.philox(seed, c0, c1, c2, c3) is Philox4x32-10 with the key (low,
    high) 32 bits of a 64-bit seed.  Its CPU interpreter (TRITON_INTERPRET=1, set
    before Triton is imported, so in a child process) runs it without a GPU."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(20240607)
    n = 16
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64)
    ctr[0] = (5, 0, 0, 0)
    ctr[1] = (U32, 17, 2 ** 31, 123456789)
    key = rng.integers(0, 2 ** 32, size=(n, 2), dtype=np.uint64)
    key[0] = (0, 0)
    key[1] = (U32, U32)
    # signed carriers of the same bits: the seed as int64, the counters as int32 (32-bit
    # counters select the 4 x 32-bit generator in tl.philox)
    seeds = [int(np.uint64(k0) | (np.uint64(k1) << np.uint64(32))) - (2 ** 64 if k1 >= 2 ** 31 else 0)
             for k0, k1 in key]
    ctr32 = [int(x) - (2 ** 32 if x >= 2 ** 31 else 0) for x in ctr.ravel()]
    env = dict(os.environ, TRITON_INTERPRET="1")
    res = subprocess.run([sys.executable, "-c", _TRITON_PHILOX], input=json.dumps({"seeds": seeds,
                         "ctr": ctr32}), capture_output=True, text=True, env=env,
                         timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    ref = np.array(json.loads(res.stdout.strip().splitlines()[-1]), dtype=np.int64).reshape(n, 4) & U32
    for m in range(n):
        np.testing.assert_array_equal(oracle.philox4x32_10(ctr[m], key[m]).astype(np.int64), ref[m])


def test_decisions_follow_the_stated_counter_layout():
    """Pair (b, h, i, j) reads the 16-bit field j % 2 of word i % 4 of the call with
    counter (j / 2, i / 4, 65536 b + h, offset mod 2^32) under the key (seed low, high)."""
    seed, off, b, h, t = 0x0123456789ABCDEF, 2 ** 32 + 9, 3, 65535, 30000
    keep = oracle.dropout_keep(b, h, 9, 7, t / 65536.0, (seed, off))
    for i in range(9):
        for j in range(7):
            w = oracle.philox4x32_10((j // 2, i // 4, 65536 * b + h, off & U32), (seed & U32, seed >> 32))
            assert keep[i, j] == (((int(w[i % 4]) >> (16 * (j % 2))) & 0xFFFF) >= t)
    # the offset counts modulo 2^32; batch entries and heads are below 65536
    np.testing.assert_array_equal(keep, oracle.dropout_keep(b, h, 9, 7, t / 65536.0, (seed, off + 2 ** 33)))
    for bad in ((65536, 0), (0, 65536)):
        with pytest.raises(ValueError):
            oracle.dropout_keep(*bad, 4, 4, 0.5, (1, 2))


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
