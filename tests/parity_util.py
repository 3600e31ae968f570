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


def compare(gpu, ref, what="", o_scale=1.0):
    """Assert every tolerance; return a dict of the measured errors.  o_scale multiplies
    the O bound: under attention dropout O is 1/(1 - p) times a sum of the same kind as
    the plain path's O (kept probabilities times values), so its bf16 errors scale by
    that factor (see dropout_o_scale)."""
    errs = {}
    assert gpu["o"].shape == ref["o"].shape
    errs["o"] = float(np.abs(gpu["o"] - ref["o"]).max()) if ref["o"].size else 0.0
    assert errs["o"] <= TOL_O * o_scale, f"{what}: O max-abs {errs['o']} (bound {TOL_O * o_scale})"
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


def dropout_o_scale(p):
    """The O bound's factor under dropout probability p: the kept-value multiplier
    65536 / (65536 - t), t = floor(65536 p + 1/2).  O_i = s sum_j P_ij keep_ij v_j: the sum
    is a sub-convex combination of value rows, as the plain O is, and the kernel applies
    s in fp32 before the one bf16 rounding of O, so every error term of O is s times the
    plain path's.  The relative-L2 gradient bounds are scale-free and LSE is the undropped
    one, so neither changes."""
    t = int(np.floor(p * 65536.0 + 0.5))
    return 65536.0 / (65536.0 - t)


BF16_U = 2.0 ** -8  # unit roundoff of bf16 (8 significant bits)


def d_offset_bound(x, gpu, *, causal, window, scale, bias=None, sigmas=6.0, dropout_p=0.0, rng_state=None,
                   dropout_origin=(0, 0)):
    """Tolerance for the learnable sink's d_offset, from the rounding the design imposes.

    d_offset_h = -sum_{b,i} p_i D_i, with p_i = exp(o_h - LSE_i) and D_i = dO_i . O_i.
    The terms have both signs, and the sum can be a small fraction of sum |p_i D_i|.
    A fused backward has only the forward's stored bf16 output O^, so it forms
    D^_i = dO_i . O^_i.  O^ carries two roundings to bf16 (unit roundoff u = 2^-8):
    P is rounded before P.V, and O is rounded on output.  Each rounding moves its value
    by at most u|value|; with the absolute error spread over +-half an ulp, its variance
    is at most u^2 value^2 / 3.  Rounding errors of different elements are independent,
    and dO is independent of them.  So, to first order,
      Var(O^_id - O_id) <= u^2/3 (O_id^2 + sum_j P_ij^2 v_jd^2),
      Var(D^_i - D_i)   = sum_d dO_id^2 Var(O^_id - O_id),
      Var(d^_h - d_h)   = sum_{b,i} p_i^2 Var(D^_i - D_i).
    The tolerance is `sigmas` standard deviations of that, plus three deterministic
    terms, none of which comes from rounding O:
      * r sum p |D^|, where r = e^e_LSE - 1 and e_LSE is the measured LSE error
        (p^ is within r of p, relative);
      * the fp32 dot of D^ over d_v terms: d_v 2^-24 sum_i p_i sum_d |dO_id O^_id|;
      * the fp32 sum of n = B*S_q terms per head, one thread per 256th of them then
        a 256-wide tree: (n/256 + 16) 2^-24 sum p |D^|.
    sum_j P_ij^2 v_jd^2 comes from the oracle: its forward with every logit doubled
    (scale, offset and bias times 2) on v^2 gives sum_j P'_ij v_jd^2, with
    P'_ij = P_ij^2 e^{2 LSE_i - LSE'_i}.

    With attention dropout (dropout_p, rng_state, dropout_origin as the oracle takes
    them) O_i = s sum_j P_ij M_ij v_j, M the keep decisions and s = 1/(1 - p) the kept
    multiplier.  The kernel rounds the kept P to bf16 and applies s in fp32 before the
    output rounding, so the P term becomes s^2 sum_j P_ij^2 M_ij v_jd^2.  The doubled-logit
    forward with the same decisions returns s sum_j P'_ij M_ij v_jd^2, one factor s short.
    D, p_sink and the exact d_offset come from the oracle with the same dropout.

    `gpu` holds the kernel's stored O ("o") and LSE ("lse").  Returns
      (exact d_offset, tolerance, the formula in fp64 on the stored O, kernel tolerance).
    The kernel tolerance is the deterministic part alone.  The last two isolate the
    kernel's own arithmetic from the rounding of O.
    """
    xd = {n: t.double().numpy() for n, t in x.items()}
    sc = oracle.default_scale(xd["q"].shape[-1]) if scale is None else float(scale)
    kw = dict(causal=causal, window=window, softmax_type=oracle.LEARNABLE, offset=xd["offset"], scale=sc)
    drop_s = 1.0
    if dropout_p > 0.0:
        kw.update(dropout_p=dropout_p, rng_state=rng_state, dropout_origin=dropout_origin)
        drop_s = dropout_o_scale(dropout_p)
    kw2 = dict(kw, offset=2.0 * xd["offset"], scale=2.0 * sc)
    if bias is not None:
        kw["bias"] = bias
        kw2["bias"] = 2.0 * bias
    f = oracle.attention_fwd(xd["q"], xd["k"], xd["v"], **kw)
    g = oracle.attention_bwd(xd["q"], xd["k"], xd["v"], xd["dout"], **kw)
    f2 = oracle.attention_fwd(xd["q"], xd["k"], xd["v"] ** 2, **kw2)
    with np.errstate(invalid="ignore"):
        w = np.exp(f2["lse"] - 2.0 * f["lse"])                       # [B, H_q, S_q]
    w = np.where(np.isfinite(w), w, 0.0)
    p2v2 = drop_s * f2["o"] * np.transpose(w, (0, 2, 1))[..., None]  # (s^2) sum_j P_ij^2 (M_ij) v_jd^2
    var_o = BF16_U ** 2 / 3.0 * (f["o"] ** 2 + p2v2)
    dO = xd["dout"]
    var_d = np.einsum("bshd,bshd->bhs", dO ** 2, var_o)
    p = f["psink"]
    sigma = np.sqrt(np.sum(p ** 2 * var_d, axis=(0, 2)))
    o_gpu = np.asarray(gpu["o"], dtype=np.float64)
    D_gpu = np.einsum("bshd,bshd->bhs", dO, o_gpu)
    fin = np.isfinite(f["lse"])
    e_lse = float(np.abs(np.asarray(gpu["lse"], np.float64)[fin] - f["lse"][fin]).max()) if fin.any() else 0.0
    r = np.expm1(e_lse)
    n = p.shape[0] * p.shape[2]
    summation = (n / 256 + 16) * 2.0 ** -24 * np.sum(p * np.abs(D_gpu), axis=(0, 2))
    dot = dO.shape[-1] * 2.0 ** -24 * np.einsum("bshd,bshd->bhs", np.abs(dO), np.abs(o_gpu))
    kernel_tol = np.sum(p * (r * np.abs(D_gpu) + dot), axis=(0, 2)) + summation
    on_gpu_o = -np.sum(p * D_gpu, axis=(0, 2))
    return g["d_offset"], sigmas * sigma + kernel_tol, on_gpu_o, kernel_tol


def check_d_offset_bound(x, gpu, what, **kw):
    """Assert the derived per-head d_offset tolerance (d_offset_bound).  Also assert
    that the kernel's reduction reproduces the fp64 formula on its own stored O within
    the deterministic part.  Returns (relative L2 error vs exact, relative L2 error vs
    the formula on the GPU's O)."""
    exact, tol, on_gpu_o, kernel_tol = d_offset_bound(x, gpu, **kw)
    got = np.asarray(gpu["d_offset"], dtype=np.float64)
    err = np.abs(got - exact)
    assert np.all(err <= tol), f"{what}: d_offset error {err} above the derived tolerance {tol}"
    kern = np.abs(got - on_gpu_o)
    assert np.all(kern <= kernel_tol), \
        f"{what}: d_offset differs from the formula on its own O by {kern} (tolerance {kernel_tol})"
    return float(rel_l2(got, exact)), float(rel_l2(got, on_gpu_o))


# Accumulation allowance of a tensor-core product of 8-bit operands over n terms: each
# K = 32 block summed with at least 14 significant bits (an assumed floor: the
# hardware's internal accumulation width is not documented), the blocks added in fp32.
def fp8_acc_rel(n):
    return 2.0 ** -13 + np.ceil(n / 32.0) * 2.0 ** -24


def fp8_bwd_bounds(q8, k8, v8, do8, descale_q, descale_k, descale_v, descale_do, o, lse, ds_amax, *, causal,
                   window, softmax_type, offset, scale, q_idx=None, k_idx=None):
    """Per-element tolerances of the FP8 backward against oracle.fp8.attention_bwd_fp8
    (with its roundings on), derived from the kernel's arithmetic.

    Both sides round the same two matrices, P~ = E4M3(2^8 P) / 2^8 and
    dS~ = E5M2(s dS) / s, and agree exactly wherever the kernel's fp32 value of 2^8 P
    (or s dS) rounds to the same code as the exact one.  The kernel's value lies in
    [x - e, x + e] around the exact x, with e from its error model below; rounding is
    monotone, so its code lies between the codes of x - e and x + e, and the rounded
    value may move by at most the larger of their distances from round(x) (zero where
    both ends round alike).  Error model (fp32 unit roundoff 2^-24):
      S     = scale q.k:  fp8_acc_rel(d) scale sum_d |q k| + 2^-22 |S|  (descale product)
      exponent (natural units): e_S + 2^-23 (|S| + |LSE| + 8) (the kernel adds log2 of
            the code scale 2^8 inside it), then ex2: 2^-21 relative, so
            e_P = P (e_exp + 2^-21) 1.01;
      dP    = dO.v:  fp8_acc_rel(d) sum_d |dO v| + 2^-22 |dP|;
      D     = dO.O in fp32 over d terms:  d 2^-24 sum_d |dO O| + 2^-23 |D|;
      dS    = P (dP - D):  |dP - D| e_P + P (e_dP + e_D) + 2^-23 |dS|.
    The outputs are sums of the rounded matrices with fp32 tensor-core accumulation
    over n terms (n = the rows, or keys, of every head summed), then one bf16 rounding
    (u = 2^-8):
      dV_jd: t = sum_i gapP_ij |dO_id| + fp8_acc_rel(n) sum_i P~_ij |dO_id|,
      dK_jd: t = scale (sum_i gapS_ij |q_id| + fp8_acc_rel(n) sum_i |dS~_ij q_id|),
      dQ_id: t = scale (sum_j gapS_ij |k_jd| + fp8_acc_rel(n) sum_j |dS~_ij k_jd|),
      tolerance = t + 2^-8 (|exact| + t).
    amax: max |dS| moves by at most max e_dS.  d_offset_h = -sum_i w_i D_i with
    w = exp(c - LSE) taken by ex2 in fp32: sum_i w_i (e_D + (2^-21 + 2^-23 (|c| +
    |LSE|)) |D|) + (n / 256 + 16) 2^-24 sum |w D| (a 256-wide fixed-order sum).

    q_idx / k_idx as in attention_bwd_fp8.  Returns a dict of tolerances shaped like
    its outputs (dq, dk, dv, d_offset) and amax_ds, plus "flips": the fraction of
    (P, dS) elements whose code may differ."""
    from oracle import fp8
    q = fp8.dequantize(q8, descale_q)
    k = fp8.dequantize(k8, descale_k)
    v = fp8.dequantize(v8, descale_v)
    do = fp8.dequantize(do8, descale_do, "e5m2")
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = v.shape
    G = Hq // Hkv
    qi = np.arange(Sq) if q_idx is None else np.asarray(q_idx)
    kj = np.arange(Skv) if k_idx is None else np.asarray(k_idx)
    q, do, o, lse = q[:, qi], do[:, qi], o[:, qi], lse[:, :, qi]
    k, v = k[:, kj], v[:, kj]
    sc = (1.0 / np.sqrt(d)) if scale is None else float(scale)
    s_ds = np.float64(fp8.scale_from_amax(ds_amax, "e5m2"))
    vis = np.ones((len(qi), len(kj)), dtype=bool)
    if causal:
        vis &= kj[None, :] <= qi[:, None]
    if window >= 0:
        vis &= kj[None, :] >= qi[:, None] - window
    acc_d = fp8_acc_rel(d)
    acc_kv = fp8_acc_rel(len(qi) * G)      # dK, dV: every row of the group
    acc_q = fp8_acc_rel(len(kj))           # dQ: every key
    r4 = lambda x: fp8.e4m3_decode(fp8.e4m3_encode(x))
    r5 = lambda x: fp8.e5m2_decode(fp8.e5m2_encode(x))
    t_dq, t_dk, t_dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    t_doff = np.zeros(Hq)
    amax_tol = 0.0
    flips, total = 0, 0
    for b in range(B):
        for h in range(Hq):
            g = h // G
            L = lse[b, h][:, None]
            ok = np.isfinite(L)
            Lf = np.where(ok, L, 0.0)
            S = sc * q[b, :, h, :] @ k[b, :, g, :].T
            Sabs = sc * np.abs(q[b, :, h, :]) @ np.abs(k[b, :, g, :]).T
            m = vis & ok
            P = np.where(m, np.exp(np.where(m, S, 0.0) - Lf), 0.0)
            e_exp = acc_d * Sabs + 2.0 ** -22 * np.abs(S) + 2.0 ** -23 * (np.abs(S) + np.abs(Lf) + 8.0)
            e_P = np.where(m, P * (e_exp + 2.0 ** -21) * 1.01, 0.0)
            x = P * fp8.P_SCALE
            ex = e_P * fp8.P_SCALE
            Pr = r4(x)
            gapP = np.maximum(np.abs(r4(x + ex) - Pr), np.abs(r4(np.maximum(x - ex, 0.0)) - Pr)) / fp8.P_SCALE
            dP = do[b, :, h, :] @ v[b, :, g, :].T
            dPabs = np.abs(do[b, :, h, :]) @ np.abs(v[b, :, g, :]).T
            D = np.sum(do[b, :, h, :] * o[b, :, h, :], axis=1)
            Dabs = np.sum(np.abs(do[b, :, h, :] * o[b, :, h, :]), axis=1)
            e_D = d * 2.0 ** -24 * Dabs + 2.0 ** -23 * np.abs(D)
            e_dP = acc_d * dPabs + 2.0 ** -22 * np.abs(dP)
            dS = P * (dP - D[:, None])
            e_dS = np.where(m, np.abs(dP - D[:, None]) * e_P + P * (e_dP + e_D[:, None]) + 2.0 ** -23 * np.abs(dS),
                            0.0)
            amax_tol = max(amax_tol, float(e_dS.max()) if e_dS.size else 0.0)
            y = dS * s_ds
            ey = e_dS * s_ds + 2.0 ** -24 * np.abs(y)
            Sr = r5(y)
            gapS = np.maximum(np.abs(r5(y + ey) - Sr), np.abs(r5(y - ey) - Sr)) / s_ds
            Pt = Pr / fp8.P_SCALE
            dSt = Sr / s_ds
            flips += int(np.count_nonzero(gapP) + np.count_nonzero(gapS))
            total += 2 * int(m.sum())
            ado, aq, ak = np.abs(do[b, :, h, :]), np.abs(q[b, :, h, :]), np.abs(k[b, :, g, :])
            t_dv[b, :, g, :] += gapP.T @ ado + acc_kv * (Pt.T @ ado)
            t_dk[b, :, g, :] += sc * (gapS.T @ aq + acc_kv * (np.abs(dSt).T @ aq))
            t_dq[b, :, h, :] = sc * (gapS @ ak + acc_q * (np.abs(dSt) @ ak))
            if softmax_type == 2:
                c = float(np.asarray(offset).reshape(-1)[h])
                w = np.where(ok[:, 0], np.exp(c - Lf[:, 0]), 0.0)
                n = B * len(qi)
                t_doff[h] += float(np.sum(w * (e_D + (2.0 ** -21 + 2.0 ** -23 * (abs(c) + np.abs(Lf[:, 0])))
                                               * np.abs(D))) + (n / 256 + 16) * 2.0 ** -24 * np.sum(np.abs(w * D)))
    return {"t_dq": t_dq, "t_dk": t_dk, "t_dv": t_dv, "d_offset": t_doff, "amax_ds": amax_tol,
            "flips": flips / max(total, 1)}


def check_fp8_bwd(got, ref, bounds, what, names=("dq", "dk", "dv")):
    """Assert |got - exact| <= t + 2^-8 (|exact| + t) per element (fp8_bwd_bounds);
    return the largest ratio of error to tolerance per output."""
    ratios = {}
    for n in names:
        g = np.asarray(got[n], dtype=np.float64)
        r = ref[n]
        t = bounds["t_" + n]
        tol = t + BF16_U * (np.abs(r) + t)
        err = np.abs(g - r)
        bad = err > tol
        assert not bad.any(), (f"{what}: {n} off at {int(bad.sum())} elements, worst {float((err - tol).max()):.3g} "
                               f"beyond the bound (first at {np.argwhere(bad)[0].tolist()})")
        ratios[n] = float((err / np.maximum(tol, 1e-30)).max()) if err.size else 0.0
    return ratios


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


__all__ = ["Shape", "make_inputs", "gpu_run", "oracle_run", "compare", "slice_group", "gpu_slice", "rel_l2",
           "d_offset_bound", "check_d_offset_bound", "fp8_acc_rel",
           "fp8_bwd_bounds", "check_fp8_bwd"]
