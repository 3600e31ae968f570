"""Padded batches on the GPU (attn_fwd_varlen / attn_bwd_varlen through the C ABI)
against the fp64 oracle on the same seeded inputs: every entry computes on its own
first Lq[b] queries and Lkv[b] keys, padded query rows give O = 0 and LSE = the sink
logit, and padding gets exactly zero gradients.  ("JAX: Single-GPU Attention with
TransformerEngine", section 1: the sequence descriptor carries each sequence's
length and its padding.)"""
import numpy as np
import pytest
import torch

from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from parity_util import Shape, compare, gpu_run, make_inputs, oracle_run

pytestmark = pytest.mark.gpu

# name, shape, causal, window, softmax_type, lens_q, lens_kv
CASES = [
    ("gqa_d128_mixed", Shape(4, 300, 300, 8, 2, 128, 128), True, -1, VANILLA, [300, 177, 64, 1], [300, 177, 64, 1]),
    ("gqa_d128_q_ne_kv_window_learnable", Shape(4, 300, 333, 8, 2, 128, 128), True, 50, LEARNABLE,
     [300, 129, 200, 31], [333, 250, 17, 128]),
    ("mqa_d64_offbyone_empty_entries", Shape(5, 257, 257, 4, 1, 64, 64), True, -1, OFF_BY_ONE,
     [257, 0, 100, 150, 64], [257, 90, 0, 150, 200]),
    ("mla_d192_128", Shape(3, 200, 200, 4, 4, 192, 128), True, -1, VANILLA, [200, 70, 129], [200, 70, 129]),
    ("noncausal_d128_d64", Shape(3, 190, 260, 4, 2, 128, 64), False, -1, VANILLA, [190, 5, 133], [260, 77, 1]),
    ("lengths_clamped", Shape(2, 140, 140, 2, 1, 64, 64), True, 20, LEARNABLE, [1000, -3], [140, 999]),
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_varlen_parity(case, deterministic):
    name, shape, causal, window, st, lq, lkv = case
    x = make_inputs(shape, 7, learnable_offset=True)
    kw = dict(causal=causal, window=window, softmax_type=st, scale=None)
    gpu = gpu_run(x, deterministic=deterministic, lens_q=lq, lens_kv=lkv, **kw)
    ref = oracle_run(x, lens_q=lq, lens_kv=lkv, **kw)
    compare(gpu, ref, name)
    # padding is exact: O, dQ on padded rows and dK, dV on padded keys are zero
    for b in range(shape.B):
        a = min(max(lq[b], 0), shape.S_q)
        kk = min(max(lkv[b], 0), shape.S_kv)
        assert np.all(gpu["o"][b, a:] == 0) and np.all(gpu["dq"][b, a:] == 0), f"{name}: padded rows of entry {b}"
        assert np.all(gpu["dk"][b, kk:] == 0) and np.all(gpu["dv"][b, kk:] == 0), f"{name}: padded keys of entry {b}"


def test_varlen_full_lengths_equal_plain_call():
    """Length arrays that say 'full length' reproduce attn_fwd / the deterministic
    attn_bwd bit for bit."""
    shape = Shape(3, 250, 250, 8, 2, 128, 128)
    x = make_inputs(shape, 9, learnable_offset=True)
    kw = dict(causal=True, window=70, softmax_type=LEARNABLE, scale=None, deterministic=True)
    a = gpu_run(x, **kw)
    b = gpu_run(x, lens_q=[250] * 3, lens_kv=[250] * 3, **kw)
    for n in ("o", "lse", "dq", "dk", "dv", "d_offset"):
        assert np.array_equal(a[n], b[n]), n


def test_varlen_full_size_sampled_entries():
    """A length mix at the training shape (B=8, S=2048, GQA 32/8, d=128, causal): the
    GPU runs the whole padded batch; the oracle recomputes two whole entries."""
    shape = Shape(8, 2048, 2048, 32, 8, 128, 128)
    x = make_inputs(shape, 11)
    gen = torch.Generator().manual_seed(12)
    lens = torch.randint(1, 2049, (8,), generator=gen).tolist()
    lens[0] = 2048
    kw = dict(causal=True, window=-1, softmax_type=VANILLA, scale=None)
    gpu = gpu_run(x, deterministic=False, lens_q=lens, lens_kv=lens, **kw)
    for b in (0, 5):
        L = lens[b]
        xb = {n: t[b:b + 1] for n, t in x.items() if n != "offset"}
        # the oracle on the entry's own rows: one head group at a time keeps it fast
        for g in (0, 7):
            sl = {"q": xb["q"][:, :L, 4 * g:4 * g + 4].contiguous(), "k": xb["k"][:, :L, g:g + 1].contiguous(),
                  "v": xb["v"][:, :L, g:g + 1].contiguous(), "dout": xb["dout"][:, :L, 4 * g:4 * g + 4].contiguous()}
            ref = oracle_run(sl, **kw)
            got = {"o": gpu["o"][b:b + 1, :L, 4 * g:4 * g + 4], "lse": gpu["lse"][b:b + 1, 4 * g:4 * g + 4, :L],
                   "dq": gpu["dq"][b:b + 1, :L, 4 * g:4 * g + 4], "dk": gpu["dk"][b:b + 1, :L, g:g + 1],
                   "dv": gpu["dv"][b:b + 1, :L, g:g + 1]}
            compare(got, ref, f"entry {b} (L={L}) group {g}")
        assert np.all(gpu["o"][b, L:] == 0) and np.all(gpu["dk"][b, L:] == 0)
