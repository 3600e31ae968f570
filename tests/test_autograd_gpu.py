"""The autograd wrapper `attention()` on the GPU: forward and backward through
torch.autograd give the same bits as calling the entry points directly (the kernels
themselves are held to the oracle by the parity tests), for the plain path, the
learnable sink, padded batches, a bias with its gradient and attention dropout."""

import pytest
import torch

from oracle import LEARNABLE
from scaled_dot_product_tmem_gb300.inputs import Shape, make_bias, make_inputs

pytestmark = pytest.mark.gpu


def _sdpa():
    import scaled_dot_product_tmem_gb300 as sdpa
    return sdpa


def _leaf(t):
    return t.cuda().requires_grad_(True)


def _check_device():
    st, site = _sdpa().attn_last_device_error()
    assert st == 0, f"device error status {st} site {site:#x}"


def _run_both(x, fwd_kw, bias=None, bias_grad=True):
    """attention() + backward, and the direct forward/backward, on the same inputs."""
    sdpa = _sdpa()
    q, k, v = (_leaf(x[n]) for n in ("q", "k", "v"))
    off = _leaf(x["offset"]) if "offset" in x else None
    b = None
    if bias is not None:
        b = bias.cuda()
        if bias_grad:
            b.requires_grad_(True)
    do = x["dout"].cuda()
    o = sdpa.attention(q, k, v, off, bias=b, **fwd_kw)
    o.backward(do)
    torch.cuda.synchronize()
    _check_device()
    kw = dict(fwd_kw)
    det = kw.pop("deterministic", True)
    qd, kd, vd = (x[n].cuda() for n in ("q", "k", "v"))
    offd = x["offset"].cuda() if "offset" in x else None
    od, lse = sdpa.sdpa_forward(qd, kd, vd, softmax_offset=offd, bias=None if bias is None else bias.cuda(), **kw)
    res = sdpa.sdpa_backward(qd, kd, vd, od, do, lse, softmax_offset=offd, deterministic=det,
                             bias=None if bias is None else bias.cuda(), **kw)
    torch.cuda.synchronize()
    _check_device()
    got = {"o": o.detach(), "dq": q.grad, "dk": k.grad, "dv": v.grad}
    ref = {"o": od, "dq": res[0], "dk": res[1], "dv": res[2]}
    if off is not None:
        got["d_offset"], ref["d_offset"] = off.grad, res[3]
    if bias is not None and bias_grad:
        got["dbias"], ref["dbias"] = b.grad, res[4].to(b.dtype)
    if bias is not None and not bias_grad:
        assert b.grad is None
    return got, ref


def _equal(got, ref):
    for n in ref:
        assert got[n] is not None, f"{n}: no gradient"
        assert got[n].dtype == ref[n].dtype and got[n].shape == ref[n].shape, n
        assert torch.equal(got[n], ref[n]), f"{n} differs from the direct call"


def test_autograd_plain_and_learnable_sink():
    shape = Shape(2, 200, 200, 4, 2, 128, 128)
    x = make_inputs(shape, 901)
    _equal(*_run_both(x, dict(causal=True, window=64)))
    x = make_inputs(shape, 902, learnable_offset=True)
    _equal(*_run_both(x, dict(causal=True, softmax_type=LEARNABLE)))


def test_autograd_padded_batch():
    shape = Shape(3, 256, 256, 4, 2, 64, 64)
    x = make_inputs(shape, 903)
    lens = torch.tensor([256, 130, 7], dtype=torch.int32, device="cuda")
    _equal(*_run_both(x, dict(causal=True, seq_lens_q=lens, seq_lens_kv=lens)))


@pytest.mark.parametrize("bias_grad", [True, False], ids=["dbias", "no_dbias"])
def test_autograd_bias(bias_grad):
    """A per-(b, h) bias: each dbias element has one contribution, so the deterministic
    path is allowed and the bits are reproducible."""
    shape = Shape(2, 192, 192, 4, 2, 128, 128)
    x = make_inputs(shape, 904)
    bias = make_bias((2, 4, 192, 192), 905)
    _equal(*_run_both(x, dict(causal=False), bias=bias, bias_grad=bias_grad))


def test_autograd_dropout_same_rng_state():
    shape = Shape(2, 256, 256, 4, 2, 128, 128)
    x = make_inputs(shape, 906)
    rng = torch.tensor([0x5EED, 3], dtype=torch.int64, device="cuda")
    _equal(*_run_both(x, dict(causal=True, dropout_p=0.1, rng_state=rng)))


def test_autograd_dropout_fresh_rng_state_is_used_by_both_passes():
    """With no rng_state the wrapper draws one and hands the same one to both passes:
    the step runs clean and its dV differs from the undropped one."""
    sdpa = _sdpa()
    x = make_inputs(Shape(1, 128, 128, 2, 2, 64, 64), 907)
    q, k, v = (_leaf(x[n]) for n in ("q", "k", "v"))
    o = sdpa.attention(q, k, v, causal=True, dropout_p=0.5)
    o.backward(x["dout"].cuda())
    torch.cuda.synchronize()
    _check_device()
    q2, k2, v2 = (_leaf(x[n]) for n in ("q", "k", "v"))
    sdpa.attention(q2, k2, v2, causal=True).backward(x["dout"].cuda())
    assert torch.isfinite(v.grad.float()).all() and v.grad.abs().sum() > 0
    assert not torch.equal(v.grad, v2.grad)
