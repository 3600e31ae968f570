"""Pins of the sampled-position oracle (oracle/sampled.py) against the full oracle.

The full oracle is pinned on its own (worked examples, closed forms, torch fp64
autograd, finite differences).  The sampled form evaluates the same definitions one
row at a time and gathers each key's gradient from the rows that see it, so on every
small problem it must agree with the full score-matrix computation at every row and
key, to fp64 rounding.  The cases move each part a mistake could hide in: the causal
bound, the left window on both sides, non-square problems with key-less rows, the
grouped-query head map and the three softmax types."""
import numpy as np
import pytest

import oracle
from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from oracle.sampled import attention_sampled

CASES = [
    # B, S_q, S_kv, H_q, H_kv, d_qk, d_v, causal, window, softmax type, scale
    (2, 90, 90, 4, 2, 16, 8, True, -1, VANILLA, None),
    (2, 90, 90, 4, 2, 16, 8, True, 20, OFF_BY_ONE, 0.4),
    (1, 50, 77, 6, 2, 8, 12, False, 10, LEARNABLE, None),
    (1, 60, 20, 2, 1, 8, 8, True, 5, VANILLA, None),      # rows past 24 see no key
    (1, 60, 20, 2, 1, 8, 8, True, 5, LEARNABLE, 0.7),     # the same rows keep the sink
    (1, 33, 33, 4, 1, 16, 16, False, -1, OFF_BY_ONE, None),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_sampled_matches_full_oracle(case):
    B, Sq, Skv, Hq, Hkv, dqk, dv, causal, window, st, scale = case
    rng = np.random.default_rng(1234 + len(CASES) * Sq + Skv)
    q = rng.standard_normal((B, Sq, Hq, dqk))
    k = rng.standard_normal((B, Skv, Hkv, dqk))
    v = rng.standard_normal((B, Skv, Hkv, dv))
    do = rng.standard_normal((B, Sq, Hq, dv))
    off = rng.standard_normal(Hq) if st == LEARNABLE else None
    kw = dict(causal=causal, window=window, softmax_type=st, offset=off, scale=scale)
    f = oracle.attention_fwd(q, k, v, **kw)
    g = oracle.attention_bwd(q, k, v, do, **kw)
    for b in range(B):
        s = attention_sampled(q, k, v, do, b=b, rows=range(Sq), keys=range(Skv), **kw)
        lse_full = f["lse"][b].T              # [Sq, Hq]
        fin = np.isfinite(lse_full)
        assert np.array_equal(fin, np.isfinite(s["lse"]))
        assert np.all(s["lse"][~fin] == lse_full[~fin])
        np.testing.assert_allclose(s["lse"][fin], lse_full[fin], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(s["o"], f["o"][b], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s["dq"], g["dq"][b], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s["dk"], g["dk"][b], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s["dv"], g["dv"][b], rtol=1e-10, atol=1e-12)


def test_sampled_subsets_equal_the_full_sampling():
    """Sampling a few rows and keys gives the same values as sampling all of them (the
    per-row cache and the key gathering do not depend on what else is sampled)."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 64, 4, 8))
    k = rng.standard_normal((1, 64, 2, 8))
    v = rng.standard_normal((1, 64, 2, 8))
    do = rng.standard_normal((1, 64, 4, 8))
    kw = dict(causal=True, window=9, softmax_type=OFF_BY_ONE)
    full = attention_sampled(q, k, v, do, rows=range(64), keys=range(64), **kw)
    rows, keys = [0, 9, 10, 63], [0, 31, 54, 63]
    part = attention_sampled(q, k, v, do, rows=rows, keys=keys, **kw)
    for n in ("o", "lse", "dq"):
        np.testing.assert_array_equal(part[n], full[n][rows])
    for n in ("dk", "dv"):
        np.testing.assert_array_equal(part[n], full[n][keys])
