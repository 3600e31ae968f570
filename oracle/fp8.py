"""FP8 attention: the E4M3 and E5M2 codecs, per-tensor quantisation, the E4M3
forward, and the backward of the hybrid recipe (E4M3 inputs, E5M2 gradients).

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle``): the tests, ``smoke()`` and
``bench.py``'s CPU baseline may call it; the product package never imports it.

Source: "Speed up attention on GPU with cuDNN and TransformerEngine", step 10
("Benchmark NVIDIA TransformerEngine and FP8", section "Inspect the FP8 path"):
the forward runs in E4M3 (4 exponent and 3 mantissa bits) with per-tensor scaling
factors derived from the absolute maximum (DelayedScaling, margin 0, ``max`` over
the amax history); the output stays bf16 and is compared with the bf16 path by
its largest absolute difference.

Readings (the pages name the format and the recipe, not the arithmetic):
  * E4M3 is the OCP 8-bit float with exponent bias 7, no infinities, largest
    finite value 448 (S.1111.110) and NaN at S.1111.111; conversion rounds to
    nearest, ties to even, and saturates to +-448 (``satfinite``).
  * Per-tensor scaling with margin 0: scale = 448 / amax, x8 = E4M3(x * scale),
    descale = 1 / scale, all in fp32.  A history of length 1 (the tensor's own
    amax) is the plainest instance; a caller with a longer history passes the
    history's max as ``amax``.
  * The forward computes attention of the dequantised tensors
    (decode(x8) * descale) exactly; that is what ``attention_fwd_fp8`` returns.
    A kernel that also rounds the softmax numerators P to E4M3 before P.V departs
    from it by at most ``p_rounding_bound`` per row.

Backward (same step 10: the hybrid recipe keeps E4M3 for the forward's tensors and
E5M2, 5 exponent and 2 mantissa bits, for the gradients).  Readings:
  * E5M2 is the OCP 8-bit float with exponent bias 15, infinities at S.11111.00,
    NaN above them, largest finite value 57344 (S.11110.11).  Casts round to nearest
    even and saturate finite values to +-57344 (``satfinite``).  Per-tensor scaling
    is as for E4M3 with 57344 in place of 448.
  * The backward takes Q, K, V as the forward's E4M3 codes and dO as E5M2 codes,
    each with its descale, plus the forward's bf16 O and fp32 LSE.  It computes
    (``attention_bwd_fp8``), in this order:
      1. the probabilities P_ij = exp(scale q_i.k_j - LSE_i) of the dequantised
         inputs;
      2. P rounded for the dV product as E4M3(P * 2^8) / 2^8 (a fixed power-of-two
         scale: P <= 1, so the codes stay below 448 and small P keep 3 bits);
      3. dP_ij = dO_i.v_j and D_i = dO_i.O_i with the dequantised dO;
      4. dS_ij = P_ij (dP_ij - D_i) from the unrounded P;
      5. dS rounded for the dK and dQ products as E5M2(dS * s) / s, with s the
         per-tensor scale of the dS statistic passed in (delayed scaling: a
         previous step's amax); the step's max |dS| is returned for the next one;
      6. dV_j = sum_i P~_ij dO_i, dK_j = scale sum_i dS~_ij q_i and
         dQ_i = scale sum_j dS~_ij k_j (the GQA sums over the group), and the
         learnable offset's gradient -sum p_sink D as in the bf16 backward.
"""
from __future__ import annotations

import numpy as np

from . import VANILLA, attention_fwd

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 byte (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# the 127 non-negative finite values, increasing with the code 0x00 .. 0x7E
_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(x) -> np.ndarray:
    """E4M3 byte of each value: round to nearest, ties to the even code, saturate
    to +-448; the sign is kept (a negative value that rounds to 0 gives 0x80);
    NaN gives 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(_POS, a, side="left"), 0, 0x7E)  # first value >= a
    lo = np.clip(hi - 1, 0, 0x7E)
    below, above = _POS[lo], _POS[hi]
    mid = (below + above) / 2.0
    pick_lo = (a < mid) | ((a == mid) & (lo % 2 == 0))
    code = np.where(a >= _POS[hi], hi, np.where(pick_lo, lo, hi))
    code = np.where(a >= E4M3_MAX, 0x7E, code)  # saturate (and exact 448)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


E5M2_MAX = 57344.0


def e5m2_decode(codes) -> np.ndarray:
    """float64 value of each E5M2 byte (+-inf for S.11111.00, NaN above)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 2) & 0x1F
    m = c & 0x3
    mag = np.where(e == 0, m / 4.0 * 2.0 ** -14, (1.0 + m / 4.0) * np.exp2(e - 15.0))
    mag = np.where(e == 31, np.where(m == 0, np.inf, np.nan), mag)
    return sign * mag


# the 124 non-negative finite values, increasing with the code 0x00 .. 0x7B
_POS5 = e5m2_decode(np.arange(0x7C, dtype=np.uint8))


def e5m2_encode(x) -> np.ndarray:
    """E5M2 byte of each value: round to nearest, ties to the even code, saturate
    finite values (and infinities) to +-57344; the sign is kept; NaN gives 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(_POS5, a, side="left"), 0, 0x7B)
    lo = np.clip(hi - 1, 0, 0x7B)
    below, above = _POS5[lo], _POS5[hi]
    mid = (below + above) / 2.0
    pick_lo = (a < mid) | ((a == mid) & (lo % 2 == 0))
    code = np.where(a >= _POS5[hi], hi, np.where(pick_lo, lo, hi))
    code = np.where(a >= E5M2_MAX, 0x7B, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def _codec(fmt):
    return (e4m3_encode, e4m3_decode, E4M3_MAX) if fmt == "e4m3" else (e5m2_encode, e5m2_decode, E5M2_MAX)


def scale_from_amax(amax, fmt="e4m3") -> np.float32:
    """fp32 scale max_finite / amax (margin 0); 1 when amax is 0 or not finite."""
    a = np.float32(amax)
    if not np.isfinite(a) or a <= 0:
        return np.float32(1.0)
    return np.float32(np.float32(_codec(fmt)[2]) / a)


def quantize(x, amax=None, transpose=False, fmt="e4m3"):
    """Per-tensor quantisation of a bf16-valued BSHD tensor [B,S,H,d] to E4M3 (or
    E5M2 with fmt="e5m2").

    amax: the scaling statistic (default: max |x| of this tensor).  Returns
    (codes uint8, amax fp32, descale fp32): codes = encode(fp32(x) * scale) with the
    product rounded to fp32 first, descale = fp32(1 / scale).  transpose=True gives
    the codes as [B,H,d,S] (the sequence innermost), the layout in which a product
    that sums over the sequence reads the tensor as a K-major operand.
    """
    enc = _codec(fmt)[0]
    xf = np.asarray(x, dtype=np.float32)
    a = np.float32(np.max(np.abs(xf))) if amax is None else np.float32(amax)
    scale = scale_from_amax(a, fmt)
    codes = enc((xf * scale).astype(np.float32))
    descale = np.float32(np.float32(1.0) / scale)
    if transpose:
        codes = np.ascontiguousarray(codes.transpose(0, 2, 3, 1))
    return codes, a, descale


def dequantize(codes, descale, fmt="e4m3") -> np.ndarray:
    """float64 tensor the codes stand for: decode(codes) * descale."""
    return _codec(fmt)[1](codes) * np.float64(np.float32(descale))


def attention_fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, *, causal=True, window=-1,
                      softmax_type=VANILLA, offset=None, scale=None):
    """Attention forward of the dequantised BSHD tensors (v8 in BSHD, not transposed).

    Same outputs as ``attention_fwd`` (o, lse, psink, rowsum), in fp64."""
    q = dequantize(q8, descale_q)
    k = dequantize(k8, descale_k)
    v = dequantize(v8, descale_v)
    return attention_fwd(q, k, v, causal=causal, window=window, softmax_type=softmax_type,
                         offset=offset, scale=scale)


def p_rounding_bound(q, k, v, lse, *, causal=True, window=-1, scale=None, softmax_type=VANILLA,
                     offset=None, rows=None):
    """Per-row bound [B,Hq,Sq] on |O_rounded - O| when the softmax numerators are
    rounded to E4M3 before the P.V product while the denominator keeps them exact.

    A kernel holds p_j = exp(s_j - m') for a running max m' that never exceeds
    M = max(max_j s_j, sink logit), and divides by l' = exp(lse - m') >= exp(lse - M).
    Rounding p_j to E4M3 moves it by at most 2^-4 p_j (normal range, 3 mantissa bits)
    plus min(2^-10, p_j) (half the subnormal spacing 2^-9, or p_j itself when it
    rounds to 0).  Divided by l', per output element that is at most
        2^-4 * sum_j P_j |v_j| + sum_j min(2^-10 * exp(M - lse), P_j) |v_j|
    with P_j = exp(s_j - lse) the exact probabilities of the visible keys.  The
    bound is returned per row as the max over the head dim; ``rows`` (query indices)
    restricts it to those rows, in that order.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, Hq, dqk = q.shape
    _, Skv, Hkv, dv = v.shape
    G = Hq // Hkv
    sc = (1.0 / np.sqrt(dqk)) if scale is None else float(scale)
    rows = np.arange(Sq) if rows is None else np.asarray(rows)
    q = q[:, rows]
    lse = np.asarray(lse)[:, :, rows]
    i = rows[:, None]  # query i sees keys j <= i (causal), j >= i - window
    j = np.arange(Skv)[None, :]
    vis = np.ones((len(rows), Skv), dtype=bool)
    if causal:
        vis &= j <= i
    if window >= 0:
        vis &= j >= i - window
    out = np.zeros((B, Hq, len(rows)))
    for b in range(B):
        for h in range(Hq):
            s = np.where(vis, sc * q[b, :, h, :] @ k[b, :, h // G, :].T, -np.inf)
            M = np.max(s, axis=1, keepdims=True)
            if softmax_type == 1:
                M = np.maximum(M, 0.0)
            elif softmax_type == 2:
                M = np.maximum(M, float(np.asarray(offset).reshape(-1)[h]))
            L = lse[b, h][:, None]
            ok = np.isfinite(L) & np.isfinite(M)
            Lf, Mf = np.where(ok, L, 0.0), np.where(ok, M, 0.0)
            P = np.where(vis & ok, np.exp(s - Lf), 0.0)
            floor = 2.0 ** -10 * np.exp(Mf - Lf)
            av = np.abs(v[b, :, h // G, :])
            out[b, h] = np.max(2.0 ** -4 * (P @ av) + np.minimum(floor, P) @ av, axis=1)
    return out


P_SCALE = 256.0  # the fixed power-of-two scale of P in the FP8 backward's dV product


def attention_bwd_fp8(q8, k8, v8, do8, descale_q, descale_k, descale_v, descale_do, o, lse, ds_amax, *,
                      causal=True, window=-1, softmax_type=VANILLA, offset=None, scale=None,
                      round_p=True, round_ds=True, q_idx=None, k_idx=None):
    """The FP8 backward's steps (module docstring) on BSHD codes: q8, k8, v8 E4M3, do8
    E5M2, all in BSHD; o the forward's output (bf16 values), lse [B,Hq,Sq] its LSE;
    ds_amax the dS scaling statistic (s = 57344 / ds_amax).  round_p / round_ds
    switch the two roundings off (then this is the exact backward of the dequantised
    inputs, with D from the given O).  Returns a dict of float64 dq, dk, dv,
    d_offset [Hq] and amax_ds = max |dS| (fp64).

    q_idx / k_idx (sorted absolute positions, default all) restrict the sums to those
    query rows and keys, the masks still taken at the absolute positions: dq is then
    [B, len(q_idx), Hq, d] summed over the keys k_idx, dk and dv [B, len(k_idx), Hkv, d]
    summed over the rows q_idx, d_offset and amax_ds over the rows q_idx.  With
    k_idx = all keys the dq rows are exact, with q_idx = all rows the dk, dv rows are."""
    q = dequantize(q8, descale_q)
    k = dequantize(k8, descale_k)
    v = dequantize(v8, descale_v)
    do = dequantize(do8, descale_do, "e5m2")
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    B, Sq, Hq, dqk = q.shape
    _, Skv, Hkv, dv = v.shape
    G = Hq // Hkv
    qi = np.arange(Sq) if q_idx is None else np.asarray(q_idx)
    kj = np.arange(Skv) if k_idx is None else np.asarray(k_idx)
    q, do, o, lse = q[:, qi], do[:, qi], o[:, qi], lse[:, :, qi]
    k, v = k[:, kj], v[:, kj]
    sc = (1.0 / np.sqrt(dqk)) if scale is None else float(scale)
    s_ds = np.float64(scale_from_amax(ds_amax, "e5m2"))
    i = qi[:, None]
    j = kj[None, :]
    vis = np.ones((len(qi), len(kj)), dtype=bool)
    if causal:
        vis &= j <= i
    if window >= 0:
        vis &= j >= i - window
    dq, dk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    doff = np.zeros(Hq)
    amax = 0.0
    for b in range(B):
        for h in range(Hq):
            g = h // G
            L = lse[b, h][:, None]
            ok = np.isfinite(L)
            S = sc * q[b, :, h, :] @ k[b, :, g, :].T                         # step 1
            P = np.where(vis & ok, np.exp(np.where(vis, S, 0.0) - np.where(ok, L, 0.0)), 0.0)
            Pr = e4m3_decode(e4m3_encode(P * P_SCALE)) / P_SCALE if round_p else P   # step 2
            dP = do[b, :, h, :] @ v[b, :, g, :].T                            # step 3
            D = np.sum(do[b, :, h, :] * o[b, :, h, :], axis=1)
            dS = P * (dP - D[:, None])                                       # step 4
            amax = max(amax, float(np.max(np.abs(dS))) if dS.size else 0.0)
            dSr = e5m2_decode(e5m2_encode(dS * s_ds)) / s_ds if round_ds else dS   # step 5
            dvv[b, :, g, :] += Pr.T @ do[b, :, h, :]                         # step 6
            dk[b, :, g, :] += sc * dSr.T @ q[b, :, h, :]
            dq[b, :, h, :] = sc * dSr @ k[b, :, g, :]
            if softmax_type == 2:
                c = float(np.asarray(offset).reshape(-1)[h])
                doff[h] -= float(np.sum(np.where(ok[:, 0], np.exp(c - np.where(ok, L, 0.0)[:, 0]), 0.0) * D))
    return {"dq": dq, "dk": dk, "dv": dvv, "d_offset": doff, "amax_ds": amax}
