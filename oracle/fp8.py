"""FP8 (E4M3) forward: codec, per-tensor quantisation and the attention it feeds.

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


def scale_from_amax(amax) -> np.float32:
    """fp32 scale 448 / amax (margin 0); 1 when amax is 0 or not finite."""
    a = np.float32(amax)
    if not np.isfinite(a) or a <= 0:
        return np.float32(1.0)
    return np.float32(np.float32(E4M3_MAX) / a)


def quantize(x, amax=None, transpose=False):
    """Per-tensor E4M3 quantisation of a bf16-valued BSHD tensor [B,S,H,d].

    amax: the scaling statistic (default: max |x| of this tensor).  Returns
    (codes uint8, amax fp32, descale fp32): codes = E4M3(fp32(x) * scale) with the
    product rounded to fp32 first, descale = fp32(1 / scale).  transpose=True gives
    the codes as [B,H,d,S] (keys innermost), the layout the P.V product reads V in.
    """
    xf = np.asarray(x, dtype=np.float32)
    a = np.float32(np.max(np.abs(xf))) if amax is None else np.float32(amax)
    scale = scale_from_amax(a)
    codes = e4m3_encode((xf * scale).astype(np.float32))
    descale = np.float32(np.float32(1.0) / scale)
    if transpose:
        codes = np.ascontiguousarray(codes.transpose(0, 2, 3, 1))
    return codes, a, descale


def dequantize(codes, descale) -> np.ndarray:
    """float64 tensor the codes stand for: decode(codes) * descale."""
    return e4m3_decode(codes) * np.float64(np.float32(descale))


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
