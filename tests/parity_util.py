"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and the fp64 oracle on the same seeded bf16 inputs, and compare with the
tolerances the target states (O max-abs <= 2e-2, LSE max-abs <= 1e-3, dQ/dK/dV/
d_offset relative L2 <= 1e-2)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from scaled_dot_product_tmem_gb300.inputs import Shape, make_inputs

TOL_O = 2e-2
TOL_LSE = 1e-3
TOL_GRAD = 1e-2


def gpu_run(x, *, causal, window, softmax_type, scale, deterministic=True, bwd=True, lens_q=None, lens_kv=None):
    import scaled_dot_product_tmem_gb300 as sdpa
    dev = torch.device("cuda")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    off = x["offset"].to(dev) if softmax_type == oracle.LEARNABLE else None
    kw = dict(causal=causal, window=window, softmax_type=softmax_type, softmax_offset=off, scale=scale)
    if lens_q is not None or lens_kv is not None:
        kw["seq_lens_q"] = None if lens_q is None else torch.tensor(lens_q, dtype=torch.int32, device=dev)
        kw["seq_lens_kv"] = None if lens_kv is None else torch.tensor(lens_kv, dtype=torch.int32, device=dev)
    o, lse = sdpa.sdpa_forward(q, k, v, **kw)
    res = {"o": o, "lse": lse}
    if bwd:
        do = x["dout"].to(dev)
        dq, dk, dv, d_off = sdpa.sdpa_backward(q, k, v, o, do, lse, deterministic=deterministic, **kw)
        res.update(dq=dq, dk=dk, dv=dv)
        if d_off is not None:
            res["d_offset"] = d_off
    torch.cuda.synchronize()
    st, site = sdpa.attn_last_device_error()
    assert st == 0, f"device error status {st} site {site:#x}"
    return {n: t.float().cpu().numpy() for n, t in res.items()}


def oracle_run(x, *, causal, window, softmax_type, scale, bwd=True, lens_q=None, lens_kv=None):
    xd = {n: t.double().numpy() for n, t in x.items()}
    off = xd.get("offset") if softmax_type == oracle.LEARNABLE else None
    kw = dict(causal=causal, window=window, softmax_type=softmax_type, offset=off, scale=scale)
    varlen = lens_q is not None or lens_kv is not None
    fwd, bwd_fn = (oracle.attention_fwd_varlen, oracle.attention_bwd_varlen) if varlen else \
        (oracle.attention_fwd, oracle.attention_bwd)
    if varlen:
        kw.update(seq_lens_q=lens_q, seq_lens_kv=lens_kv)
    f = fwd(xd["q"], xd["k"], xd["v"], **kw)
    res = {"o": f["o"], "lse": f["lse"]}
    if bwd:
        g = bwd_fn(xd["q"], xd["k"], xd["v"], xd["dout"], **kw)
        res.update(dq=g["dq"], dk=g["dk"], dv=g["dv"])
        if softmax_type == oracle.LEARNABLE:
            res["d_offset"] = g["d_offset"]
    return res


def rel_l2(a, ref):
    den = np.linalg.norm(ref)
    num = np.linalg.norm(a - ref)
    return num / den if den > 0 else num


def compare(gpu, ref, what=""):
    """Assert every tolerance; return a dict of the measured errors."""
    errs = {}
    assert gpu["o"].shape == ref["o"].shape
    errs["o"] = float(np.abs(gpu["o"] - ref["o"]).max()) if ref["o"].size else 0.0
    assert errs["o"] <= TOL_O, f"{what}: O max-abs {errs['o']}"
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(fin, np.isfinite(gpu["lse"])), f"{what}: LSE finiteness differs"
    assert np.all(gpu["lse"][~fin] == ref["lse"][~fin]), f"{what}: infinite LSE differs"
    errs["lse"] = float(np.abs(gpu["lse"][fin] - ref["lse"][fin]).max()) if fin.any() else 0.0
    assert errs["lse"] <= TOL_LSE, f"{what}: LSE max-abs {errs['lse']}"
    for n in ("dq", "dk", "dv", "d_offset"):
        if n in ref:
            assert gpu[n].shape == ref[n].shape, f"{what}: {n} shape"
            errs[n] = float(rel_l2(gpu[n], ref[n]))
            assert errs[n] <= TOL_GRAD, f"{what}: {n} relative L2 {errs[n]}"
    return errs


def slice_group(x, b, g, G):
    """The inputs of one (batch b, kv head g) unit: query heads g*G..g*G+G-1 with kv head g."""
    out = {}
    out["q"] = x["q"][b:b + 1, :, g * G:(g + 1) * G].contiguous()
    out["k"] = x["k"][b:b + 1, :, g:g + 1].contiguous()
    out["v"] = x["v"][b:b + 1, :, g:g + 1].contiguous()
    if "dout" in x:
        out["dout"] = x["dout"][b:b + 1, :, g * G:(g + 1) * G].contiguous()
    if "offset" in x:
        out["offset"] = x["offset"][g * G:(g + 1) * G].contiguous()
    return out


def gpu_slice(res, b, g, G):
    """The same unit cut out of full GPU results."""
    out = {"o": res["o"][b:b + 1, :, g * G:(g + 1) * G], "lse": res["lse"][b:b + 1, g * G:(g + 1) * G]}
    if "dq" in res:
        out["dq"] = res["dq"][b:b + 1, :, g * G:(g + 1) * G]
        out["dk"] = res["dk"][b:b + 1, :, g:g + 1]
        out["dv"] = res["dv"][b:b + 1, :, g:g + 1]
    return out


__all__ = ["Shape", "make_inputs", "gpu_run", "oracle_run", "compare", "slice_group", "gpu_slice", "rel_l2"]
