"""Sequences of 131,072 tokens on the GPU, checked against the oracle at sampled rows
and keys (oracle/sampled.py evaluates the oracle's definitions there exactly; the full
score matrix would not fit).

The kernels' row and key offsets then reach the top of the sequence, and the tiles
near it are the ones the sampled positions fall in.  Query rows are sampled at tile
boundaries and across the sequence.  Keys are sampled where the rows that see them are
few: the last keys of a causal sequence, and anywhere under a sliding window.  A padded
batch has its entry checked as the problem of its own length, and its padding rows and
keys against their fixed values.  Both backward paths run, each against the same
tolerances as the other parity tests."""
import numpy as np
import pytest
import torch

from oracle import OFF_BY_ONE, VANILLA
from oracle.sampled import attention_sampled
from parity_util import TOL_GRAD, TOL_LSE, TOL_O, Shape, make_inputs, rel_l2

pytestmark = pytest.mark.gpu

S = 131072
L1 = 40001  # the second entry's length in the padded batch
CASES = [
    # name, shape, causal, window, softmax type, seed, sampled rows, sampled keys,
    # per-entry lengths (None: full length), the batch entry sampled
    ("gqa_d128_causal", Shape(1, S, S, 8, 2, 128, 128), True, -1, VANILLA, 71,
     [0, 1, 127, 128, 129, 4095, 65535, 65536, 100000, S - 129, S - 1],
     [S - 1, S - 2, S - 64, S - 128, S - 129], None, 0),
    ("mqa_d64_window1024_obo", Shape(1, S, S, 8, 1, 64, 64), True, 1024, OFF_BY_ONE, 72,
     [0, 1000, 1024, 1025, 65536, 130000, S - 1],
     [0, 500, 65536, 130000, S - 1], None, 0),
    # a padded batch: entry 1 holds L1 of S/2 rows; its sampled positions end at L1 - 1
    ("padded_gqa_d128_causal", Shape(2, S // 2, S // 2, 8, 2, 128, 128), True, -1, VANILLA, 73,
     [0, 128, 20000, L1 - 129, L1 - 1], [L1 - 1, L1 - 2, L1 - 64, L1 - 129], [S // 2, L1], 1),
]
# padding rows and keys of the padded entry: no key is seen (O = 0, LSE = -inf) and
# no query sees them (dK = dV = 0)
PAD_ROWS, PAD_KEYS = [L1, L1 + 1, S // 2 - 1], [L1, S // 2 - 1]


def _gpu(x, rows, keys, *, causal, window, softmax_type, deterministic, lens=None, b=0):
    import scaled_dot_product_tmem_gb300 as sdpa
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    kw = dict(causal=causal, window=window, softmax_type=softmax_type)
    if lens is not None:
        lt = torch.tensor(lens, dtype=torch.int32, device=dev)
        kw.update(seq_lens_q=lt, seq_lens_kv=lt)
    o, lse = sdpa.sdpa_forward(q, k, v, **kw)
    dq, dk, dv, _ = sdpa.sdpa_backward(q, k, v, o, do, lse, deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    st, site = sdpa.attn_last_device_error()
    assert st == 0, f"device error status {st} site {site:#x}"
    r = torch.tensor(rows, device=dev)
    c = torch.tensor(keys, device=dev)
    return {"o": o[b, r].float().cpu().numpy(), "lse": lse[b][:, r].T.float().cpu().numpy(),
            "dq": dq[b, r].float().cpu().numpy(), "dk": dk[b, c].float().cpu().numpy(),
            "dv": dv[b, c].float().cpu().numpy()}


@pytest.fixture(scope="module")
def oracle_values():
    """Inputs and the oracle's values per case, computed once for both backward paths."""
    out = {}
    for name, shape, causal, window, st, seed, rows, keys, lens, b in CASES:
        x = make_inputs(shape, seed)
        # a padded entry is the problem of its own length (rows and keys past it excluded)
        n = lens[b] if lens is not None else shape.S_q
        xn = {t_: x[t_][b:b + 1, :n].float().numpy() for t_ in ("q", "k", "v", "dout")}
        ref = attention_sampled(xn["q"], xn["k"], xn["v"], xn["dout"], rows=rows, keys=keys, causal=causal,
                                window=window, softmax_type=st)
        out[name] = (x, ref)
    return out


@pytest.mark.parametrize("deterministic", [False, True], ids=["fused_dq", "det"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_long_sequence_sampled(case, deterministic, oracle_values):
    name, shape, causal, window, st, seed, rows, keys, lens, b = case
    x, ref = oracle_values[name]
    gpu = _gpu(x, rows, keys, causal=causal, window=window, softmax_type=st, deterministic=deterministic,
               lens=lens, b=b)
    err_o = float(np.abs(gpu["o"] - ref["o"]).max())
    assert err_o <= TOL_O, f"{name}: O max-abs {err_o}"
    assert np.all(np.isfinite(ref["lse"]))
    err_lse = float(np.abs(gpu["lse"] - ref["lse"]).max())
    assert err_lse <= TOL_LSE, f"{name}: LSE max-abs {err_lse}"
    for n in ("dq", "dk", "dv"):
        e = float(rel_l2(gpu[n], ref[n]))
        assert e <= TOL_GRAD, f"{name}: {n} relative L2 {e}"
    if lens is not None:
        pad = _gpu(x, PAD_ROWS, PAD_KEYS, causal=causal, window=window, softmax_type=st,
                   deterministic=deterministic, lens=lens, b=b)
        assert np.all(pad["o"] == 0) and np.all(np.isneginf(pad["lse"])) and np.all(pad["dq"] == 0)
        assert np.all(pad["dk"] == 0) and np.all(pad["dv"] == 0)
