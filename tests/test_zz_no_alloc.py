"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory
(runtimes that freeze their memory footprint at start-up and forbid allocation on
the launch path, or C callers without a device allocator).  It keeps its scratch in
a fixed array inside the library.

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It calls the entry point through the C
ABI three times in a row with different shapes, so each later call runs on an array
that still holds the previous call's contents, and checks:
  * against attn_bwd with deterministic != 0: bitwise equal where attn_bwd also walks
    every query head of a kv group in one CTA (no head split: the same arithmetic on the
    same inputs), within the gradient tolerance where attn_bwd splits the heads (its
    partial dK/dV slices add in another fp32 order).  On grids of many short tiles
    attn_bwd runs persistent CTAs that take their tiles from a counter, and this entry
    point (no counter in its scratch) one CTA per tile: the bitwise comparison then also
    checks the persistent kernels' tile hand-over;
  * against the fp64 oracle on the first shape, with the tolerances of every other
    parity test.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity_util import TOL_GRAD, Shape, compare, make_inputs, oracle_run, rel_l2

pytestmark = pytest.mark.gpu

OK, WORKSPACE = 0, 6
NUM_SMS = 152  # attn_bwd splits a group's query heads when its kv grid has < 3 CTAs per SM


def _splits(shape):
    """Whether attn_bwd splits the query heads of a kv group for this shape."""
    ctas = -(-shape.S_kv // 128) * shape.H_kv * shape.B
    return ctas < 3 * NUM_SMS and shape.H_q // shape.H_kv > 1


def _run_both(sdpa, lib, shape, seed, st, window):
    dev = torch.device("cuda")
    x = make_inputs(shape, seed, learnable_offset=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    off = x["offset"].to(dev) if st == sdpa.LEARNABLE else None
    kw = dict(causal=True, window=window, softmax_type=st, softmax_offset=off)
    o, lse = sdpa.sdpa_forward(q, k, v, **kw)
    ref = sdpa.sdpa_backward(q, k, v, o, do, lse, deterministic=True, **kw)

    dq, dk, dv = torch.full_like(q, 3.0), torch.full_like(k, 3.0), torch.full_like(v, 3.0)
    d_off = torch.full((shape.H_q,), 3.0, device=dev) if off is not None else None
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    B, S_q, H_q, d_qk = q.shape
    _, S_kv, H_kv, d_v = v.shape
    rc = lib.attn_bwd_noalloc(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv), p(d_off), B, S_q, S_kv,
                              H_q, H_kv, d_qk, d_v, ctypes.c_float(0.0), 1, window, st, p(off),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == OK, lib.attn_bwd_noalloc_message().decode()
    torch.cuda.synchronize()
    status, site = sdpa.attn_last_device_error()
    assert status == 0, f"device error {status} at site {site:#x}"
    got = [dq, dk, dv] + ([d_off] if d_off is not None else [])
    want = [ref[0], ref[1], ref[2]] + ([ref[3]] if d_off is not None else [])
    names = ("dq", "dk", "dv", "d_offset")
    if _splits(shape):
        for name, g, w in zip(names, got, want):
            err = rel_l2(g.float().cpu().numpy(), w.float().cpu().numpy())
            assert err <= TOL_GRAD, f"{name}: relative L2 {err} vs attn_bwd"
    else:
        for name, g, w in zip(names, got, want):
            assert torch.equal(g, w), f"{name}: not bitwise equal to attn_bwd (deterministic)"
    res = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    if d_off is not None:
        res["d_offset"] = d_off
    return x, {n: t.float().cpu().numpy() for n, t in res.items()}


def test_no_alloc_backward_three_calls_in_a_row():
    import scaled_dot_product_tmem_gb300 as sdpa
    lib = sdpa.library()
    # first call: learnable sink, GQA (attn_bwd splits the group's heads), ragged, window
    shape = Shape(2, 300, 300, 8, 2, 128, 128)
    assert _splits(shape)
    x, gpu = _run_both(sdpa, lib, shape, 201, sdpa.LEARNABLE, 100)
    compare(gpu, oracle_run(x, causal=True, window=100, softmax_type=sdpa.LEARNABLE, scale=None), "noalloc vs oracle")
    # second call right after, other shape (MHA: no split): bitwise equal to attn_bwd
    shape = Shape(1, 200, 200, 4, 4, 64, 64)
    assert not _splits(shape)
    _run_both(sdpa, lib, shape, 202, sdpa.VANILLA, -1)
    # third call: GQA with 512 kv CTAs (no split), off-by-one sink: bitwise equal to attn_bwd
    # (whose dQ kernel runs persistent CTAs here)
    shape = Shape(16, 512, 512, 16, 8, 64, 64)
    assert not _splits(shape)
    _run_both(sdpa, lib, shape, 203, sdpa.OFF_BY_ONE, -1)
    # fourth call: MHA d = 128 at S = 512, where attn_bwd's kv and dQ kernels both run
    # persistent CTAs and the last kv tile of each sequence is a single step
    shape = Shape(16, 512, 512, 16, 16, 128, 128)
    assert not _splits(shape)
    _run_both(sdpa, lib, shape, 204, sdpa.VANILLA, -1)


def test_persistent_deterministic_backward_repeats_bitwise():
    """Two deterministic backward calls on a grid of many one- and two-step tiles, where
    the kv and dQ kernels hand tiles out through a counter, give the same bits."""
    import scaled_dot_product_tmem_gb300 as sdpa
    dev = torch.device("cuda")
    x = make_inputs(Shape(32, 384, 384, 16, 16, 128, 128), 205)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = sdpa.sdpa_forward(q, k, v, causal=True)
    a = sdpa.sdpa_backward(q, k, v, o, do, lse, causal=True, deterministic=True)
    b = sdpa.sdpa_backward(q, k, v, o, do, lse, causal=True, deterministic=True)
    torch.cuda.synchronize()
    for ta, tb in zip(a[:3], b[:3]):
        assert torch.equal(ta, tb)


def test_no_alloc_rejects_problems_beyond_its_array():
    import scaled_dot_product_tmem_gb300 as sdpa
    lib = sdpa.library()
    cap = lib.attn_bwd_noalloc_max_scratch_bytes()
    assert cap == 8 << 20
    fake = ctypes.c_void_p(0x10000)
    # B * H_q * S_pad = 8 * 32 * 8192 rows needs 16 MiB > 8 MiB: rejected before any launch
    rc = lib.attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, None, 8, 8192, 8192, 32, 8,
                              128, 128, ctypes.c_float(0.0), 1, -1, 0, None, None)
    assert rc == WORKSPACE
    assert "scratch" in lib.attn_bwd_noalloc_message().decode()
