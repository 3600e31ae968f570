"""Attention dropout on the GPU (attn_fwd_dropout / attn_bwd_dropout) against the fp64
oracle, which regenerates the same keep decisions from the same rng_state.

Two kinds of check:
  * the keep decisions themselves, bit for bit.  Inputs are constructed so that an
    output exposes the decisions of the kernel that made it:
      - forward: Q = 0, V one-hot over the keys, so O_id = P M_id with a uniform P;
      - kv backward: dO one-hot over the rows, so dV_jd = P M_dj;
      - the dS of the dQ kernels: K one-hot, V = dO = e_0, so dQ_id has the sign of
        M_id - mean_j M_ij.
    All three are compared with oracle.dropout_keep, and the keep rate is held to
    binomial bounds;
  * parity of O, LSE, dQ, dK, dV and d_offset with the oracle at the stated tolerances
    (the O bound times the kept-value multiplier 1/(1 - p), see dropout_o_scale),
    for p in {0.1, 0.5}, on both dQ paths, the sink types, GQA, windows, MLA dims and
    ragged sizes, and that a fixed rng_state is bitwise reproducible.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import LEARNABLE, OFF_BY_ONE, VANILLA
from parity_util import check_d_offset_bound, compare, dropout_o_scale, rel_l2
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs

pytestmark = pytest.mark.gpu

RNG = (0x5EED_1234_ABCD, 17)


def _sdpa():
    import scaled_dot_product_tmem_gb300 as sdpa
    return sdpa


def _rng(dev, rng=RNG):
    return torch.tensor(list(rng), dtype=torch.int64, device=dev)


def _gpu(x, *, causal, window, st, scale, p, det, rng=RNG):
    sdpa = _sdpa()
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = x["offset"].to(dev) if st == LEARNABLE else None
    kw = dict(causal=causal, window=window, softmax_type=st, softmax_offset=off, scale=scale or 0.0,
              dropout_p=p, rng_state=_rng(dev, rng))
    o, lse = sdpa.sdpa_forward(q, k, v, **kw)
    dq, dk, dv, d_off = sdpa.sdpa_backward(q, k, v, o, do, lse, deterministic=det, **kw)
    torch.cuda.synchronize()
    status, site = sdpa.attn_last_device_error()
    assert status == 0, f"device error {status} site {site:#x}"
    out = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    if d_off is not None:
        out["d_offset"] = d_off
    return {n: t.float().cpu().numpy() for n, t in out.items()}


def _ref(x, *, causal, window, st, scale, p, rng=RNG, origin=(0, 0)):
    xd = {n: t.double().numpy() for n, t in x.items()}
    kw = dict(causal=causal, window=window, softmax_type=st, offset=xd["offset"] if st == LEARNABLE else None,
              scale=scale, dropout_p=p, rng_state=rng, dropout_origin=origin)
    f = oracle.attention_fwd(xd["q"], xd["k"], xd["v"], **kw)
    g = oracle.attention_bwd(xd["q"], xd["k"], xd["v"], xd["dout"], **kw)
    out = {"o": f["o"], "lse": f["lse"], "dq": g["dq"], "dk": g["dk"], "dv": g["dv"]}
    if st == LEARNABLE:
        out["d_offset"] = g["d_offset"]
    return out


def _keep_ref(B, H, Sq, Skv, p, rng=RNG):
    return np.stack([np.stack([oracle.dropout_keep(b, h, Sq, Skv, p, rng) for h in range(H)]) for b in range(B)])


def _binomial_ok(keep, p):
    q = 1.0 - oracle.dropout_threshold(p) / 65536.0
    n = keep.size
    return abs(keep.mean() - q) <= 5.0 * np.sqrt(q * (1.0 - q) / n)


@pytest.mark.parametrize("p", [0.1, 0.5])
def test_forward_keep_decisions_are_the_oracles(p):
    """Q = 0, V one-hot over 128 keys: O_id = M_id / 128, so O > 0 iff (i, d) is kept."""
    sdpa = _sdpa()
    dev = torch.device("cuda")
    B, Sq, Skv, H = 2, 1000, 128, 3
    q = torch.zeros((B, Sq, H, 128), dtype=torch.bfloat16, device=dev)
    k = torch.randn((B, Skv, H, 128), device=dev).to(torch.bfloat16)
    v = torch.eye(128, dtype=torch.bfloat16, device=dev)[None, :, None, :].expand(B, Skv, H, 128).contiguous()
    o, lse = sdpa.sdpa_forward(q, k, v, causal=False, dropout_p=p, rng_state=_rng(dev))
    torch.cuda.synchronize()
    keep = (o.float() > 0).permute(0, 2, 1, 3).cpu().numpy()        # [B, H, Sq, Skv]
    ref = _keep_ref(B, H, Sq, Skv, p)
    assert np.array_equal(keep, ref), f"{np.sum(keep != ref)} decisions differ"
    assert _binomial_ok(keep, p)
    scale = 65536.0 / (65536.0 - oracle.dropout_threshold(p)) / Skv
    np.testing.assert_allclose(o.float().cpu().numpy()[o.float().cpu().numpy() > 0], scale, rtol=2 ** -8)


@pytest.mark.parametrize("det", [True, False], ids=["det", "fused_dq"])
def test_kv_backward_keep_decisions_are_the_oracles(det):
    """Q = 0, dO one-hot over 128 query rows: dV_jd = M_dj / S_kv (MHA, so no head sum)."""
    sdpa = _sdpa()
    dev = torch.device("cuda")
    p = 0.3
    B, Sq, Skv, H = 2, 128, 700, 2
    q = torch.zeros((B, Sq, H, 128), dtype=torch.bfloat16, device=dev)
    k = torch.randn((B, Skv, H, 128), device=dev).to(torch.bfloat16)
    v = torch.randn((B, Skv, H, 128), device=dev).to(torch.bfloat16)
    do = torch.eye(128, dtype=torch.bfloat16, device=dev)[None, :, None, :].expand(B, Sq, H, 128).contiguous()
    kw = dict(causal=False, dropout_p=p, rng_state=_rng(dev))
    o, lse = sdpa.sdpa_forward(q, k, v, **kw)
    dq, dk, dv, _ = sdpa.sdpa_backward(q, k, v, o, do, lse, deterministic=det, **kw)
    torch.cuda.synchronize()
    keep = (dv.float() > 0).permute(0, 2, 3, 1).cpu().numpy()       # [B, H, d = query row, key]
    ref = _keep_ref(B, H, Sq, Skv, p)
    assert np.array_equal(keep, ref), f"{np.sum(keep != ref)} decisions differ"
    assert _binomial_ok(keep, p)


@pytest.mark.parametrize("det", [True, False], ids=["det", "fused_dq"])
def test_dq_keep_decisions_are_the_oracles(det):
    """Q = 0, K one-hot over 128 keys, V = dO = e_0: dS_ij = (M_ij - mean_j M_ij) / S_kv
    and dQ_id = scale dS_id, positive iff (i, d) is kept."""
    sdpa = _sdpa()
    dev = torch.device("cuda")
    p = 0.5
    B, Sq, Skv, H = 1, 900, 128, 2
    e0 = torch.zeros(128, dtype=torch.bfloat16, device=dev)
    e0[0] = 1
    q = torch.zeros((B, Sq, H, 128), dtype=torch.bfloat16, device=dev)
    k = torch.eye(128, dtype=torch.bfloat16, device=dev)[None, :, None, :].expand(B, Skv, H, 128).contiguous()
    v = e0.expand(B, Skv, H, 128).contiguous()
    do = e0.expand(B, Sq, H, 128).contiguous()
    kw = dict(causal=False, dropout_p=p, rng_state=_rng(dev))
    o, lse = sdpa.sdpa_forward(q, k, v, **kw)
    dq, dk, dv, _ = sdpa.sdpa_backward(q, k, v, o, do, lse, deterministic=det, **kw)
    torch.cuda.synchronize()
    keep = (dq.float() > 0).permute(0, 2, 1, 3).cpu().numpy()       # [B, H, Sq, key]
    ref = _keep_ref(B, H, Sq, Skv, p)
    full = ref.all(axis=3) | (~ref).all(axis=3)                      # rows with no sign to read
    assert not full.any()
    assert np.array_equal(keep, ref), f"{np.sum(keep != ref)} decisions differ"


CASES = [
    # name, shape, causal, window, softmax type, scale
    ("gqa_ragged", Shape(2, 300, 300, 4, 2, 128, 128), True, -1, VANILLA, None),
    ("d64_window_obo", Shape(1, 333, 333, 4, 1, 64, 64), True, 100, OFF_BY_ONE, None),
    ("d64_learnable", Shape(2, 200, 200, 4, 2, 64, 64), True, -1, LEARNABLE, None),
    ("noncausal_rect", Shape(1, 150, 290, 2, 1, 128, 128), False, -1, VANILLA, 0.3),
    ("mqa_multi_tile", Shape(1, 700, 700, 8, 1, 128, 128), True, 300, VANILLA, 0.09),
]


@pytest.mark.parametrize("det", [True, False], ids=["det", "fused_dq"])
@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_dropout_parity(case, p, det):
    name, shape, causal, window, st, scale = case
    x = make_inputs(shape, 900 + CASES.index(case), learnable_offset=True)
    kw = dict(causal=causal, window=window, st=st, scale=scale, p=p)
    _check(x, _gpu(x, det=det, **kw), _ref(x, **kw), f"{name} p={p}", kw)


def _check(x, gpu, ref, what, kw):
    """compare() at the dropout O bound.  The learnable sink's d_offset is held to the
    derived bound (parity_util.d_offset_bound, with the same dropout), as for the other
    cases whose d_offset terms cancel."""
    if "d_offset" in ref:
        ref = {n: a for n, a in ref.items() if n != "d_offset"}
        check_d_offset_bound(x, gpu, what, causal=kw["causal"], window=kw["window"], scale=kw["scale"],
                             dropout_p=kw["p"], rng_state=RNG)
    compare({n: a for n, a in gpu.items() if n != "d_offset"}, ref, what, o_scale=dropout_o_scale(kw["p"]))


@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout_parity_mla(p):
    """MLA head dims (192 / 128, scale 1/sqrt(192)): the query-stationary dQ path."""
    shape = Shape(1, 257, 257, 2, 2, 192, 128)
    x = make_inputs(shape, 950, learnable_offset=True)
    kw = dict(causal=True, window=-1, st=LEARNABLE, scale=1 / np.sqrt(192), p=p)
    _check(x, _gpu(x, det=True, **kw), _ref(x, **kw), f"mla p={p}", kw)


def test_fixed_rng_state_is_reproducible_and_offset_changes_the_result():
    shape = Shape(2, 260, 260, 4, 2, 128, 128)
    x = make_inputs(shape, 960, learnable_offset=True)
    kw = dict(causal=True, window=-1, st=LEARNABLE, scale=None, p=0.2, det=True)
    a = _gpu(x, **kw)
    b = _gpu(x, **kw)
    for n in a:
        assert np.array_equal(a[n], b[n]), n
    c = _gpu(x, rng=(RNG[0], RNG[1] + 1), **kw)
    assert rel_l2(c["o"], a["o"]) > 0.05
    np.testing.assert_array_equal(c["lse"], a["lse"])  # the softmax statistics do not depend on the drops


def test_zero_probability_runs_the_plain_kernels():
    """attn_fwd_dropout with p = 0 (t = 0) through the C ABI equals attn_fwd bit for bit."""
    import ctypes
    sdpa = _sdpa()
    lib = sdpa.library()
    shape = Shape(1, 200, 200, 4, 2, 128, 128)
    x = make_inputs(shape, 970)
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o0, l0 = sdpa.sdpa_forward(q, k, v)
    o1, l1 = torch.empty_like(o0), torch.empty_like(l0)
    rng = _rng(dev)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.attn_fwd_dropout(ptr(q), ptr(k), ptr(v), ptr(o1), ptr(l1), 1, 200, 200, 4, 2, 128, 128,
                              ctypes.c_float(0.0), 1, -1, 0, None, ctypes.c_float(0.0), ptr(rng),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_dropout_full_size_sampled():
    """The GQA + SWA training shape (B=4, S=2048, H_q=32, H_kv=8, d=128, causal, window
    1024) with p = 0.1, on the fused dQ path bench.py times: the oracle runs whole
    (batch, kv-group) units."""
    from parity_util import gpu_slice, slice_group
    shape = Shape(4, 2048, 2048, 32, 8, 128, 128)
    x = make_inputs(shape, 11)
    kw = dict(causal=True, window=1024, st=VANILLA, scale=None, p=0.1)
    gpu = _gpu(x, det=False, **kw)
    G = 4
    for b, g in ((0, 0), (3, 7)):
        # a unit takes the decisions of its own (b, h) in the full problem
        ref = _ref(slice_group(x, b, g, G), origin=(b, g * G), **kw)
        compare(gpu_slice(gpu, b, g, G), ref, f"dropout unit (b={b}, g={g})", o_scale=dropout_o_scale(kw["p"]))
