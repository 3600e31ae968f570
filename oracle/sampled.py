"""Exact attention values at sampled positions of long sequences, in fp64 numpy.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the tests may call it; the
product package never imports it.  It shares no code with the CUDA path.

The full oracle (``oracle.c``) materialises the ``S_q x S_kv`` score matrix of one
(batch, head) at a time, which a sequence of 131,072 tokens cannot hold (137 GB in
fp64).  Every quantity it returns is nevertheless a function of a few rows or columns
of that matrix:

  * O_i, LSE_i and dQ_i depend only on query row i and the keys row i sees;
  * dK_j and dV_j depend only on the rows that see key j, through each such row's
    own LSE_i and D_i = dO_i . O_i.

This module evaluates the oracle's definitions at chosen rows and keys, one row at a
time, with no blocking or reordering beyond that:

  * scores s_ij = scale q_i . k_j on the visible keys ("Speed up attention on GPU with
    cuDNN and TransformerEngine", section "How attention works");
  * key j is visible to query i iff j <= i when causal (same codelab, step 7, "Add
    causal masking") and j >= i - w with a left window w >= 0 ("JAX: Single-GPU
    Attention with TransformerEngine", sections 1-2); the kv head of query head h is
    h // (H_q / H_kv) (same page, section 4, grouped-query attention);
  * the sink softmax types ("[JAX] Add support for sink attention in JAX #2225",
    Greptile summaries): the denominator gains exp(c) with c = 0 (off-by-one) or
    c = offset_h (learnable); vanilla has none;
  * P_ij = exp(s_ij - LSE_i), LSE_i = ln(exp(c) + sum_j exp(s_ij)), O_i = sum_j P_ij v_j;
  * the backward of that forward: dP_ij = dO_i . v_j, D_i = dO_i . O_i,
    dS_ij = P_ij (dP_ij - D_i), dQ_i = scale sum_j dS_ij k_j,
    dK_j = scale sum_{h in group} sum_i dS_ij q_i, dV_j = sum_{h in group} sum_i P_ij dO_i.
"""
from __future__ import annotations

import numpy as np

VANILLA, OFF_BY_ONE, LEARNABLE = 0, 1, 2


def _visible_keys(i: int, S_kv: int, causal: bool, window: int):
    """Inclusive bounds [lo, hi] of the keys query row i sees (empty when lo > hi)."""
    lo = max(0, i - window) if window >= 0 else 0
    hi = min(i, S_kv - 1) if causal else S_kv - 1
    return lo, hi


def _rows_seeing(j: int, S_q: int, causal: bool, window: int):
    """Inclusive bounds [lo, hi] of the query rows that see key j."""
    lo = j if causal else 0
    hi = min(S_q - 1, j + window) if window >= 0 else S_q - 1
    return lo, hi


def _sink(softmax_type: int, offset, h: int) -> float:
    if softmax_type == OFF_BY_ONE:
        return 0.0
    if softmax_type == LEARNABLE:
        return float(offset[h])
    return -np.inf


def _row(q, kh, vh, dout, b, h, i, scale, causal, window, c):
    """Every per-row quantity of query row i, head h: o, lse, and over the visible key
    range [lo, hi] the probabilities P and dS; plus dq.  kh, vh: the keys and values of
    h's kv head in batch entry b, [S_kv, d] in fp64."""
    S_kv = kh.shape[0]
    lo, hi = _visible_keys(i, S_kv, causal, window)
    K = kh[lo:hi + 1] if hi >= lo else kh[:0]
    V = vh[lo:hi + 1] if hi >= lo else vh[:0]
    dqk, dv_ = K.shape[1], V.shape[1]
    qi = np.asarray(q[b, i, h], dtype=np.float64)
    doi = np.asarray(dout[b, i, h], dtype=np.float64)
    s = scale * (K @ qi)
    m = max(float(s.max()) if s.size else -np.inf, c)
    if m == -np.inf:  # no visible key and no sink: an empty row
        return {"o": np.zeros(dv_), "lse": -np.inf, "lo": lo, "P": np.zeros(s.size), "dS": np.zeros(s.size),
                "dq": np.zeros(dqk)}
    e = np.exp(s - m)
    z = e.sum() + (np.exp(c - m) if c > -np.inf else 0.0)
    P = e / z
    o = P @ V
    dP = V @ doi
    D = float(doi @ o)
    dS = P * (dP - D)
    return {"o": o, "lse": m + np.log(z), "lo": lo, "P": P, "dS": dS, "dq": scale * (dS @ K)}


def attention_sampled(q, k, v, dout, *, b=0, rows=(), keys=(), causal=True, window=-1,
                      softmax_type=VANILLA, offset=None, scale=None):
    """Forward and backward values of batch entry b at sampled positions.

    q [B,S_q,H_q,d_qk], k [B,S_kv,H_kv,d_qk], v [B,S_kv,H_kv,d_v], dout [B,S_q,H_q,d_v]:
    numpy arrays of any float dtype, read a slice at a time and computed in fp64.
    rows: query indices; keys: key indices.
    Returns a dict of float64 arrays:
      o [len(rows), H_q, d_v], lse [len(rows), H_q], dq [len(rows), H_q, d_qk],
      dk [len(keys), H_kv, d_qk], dv [len(keys), H_kv, d_v] (summed over the query
      heads of each kv head's group).
    The cost of a key is the number of rows that see it times their visible keys, so
    causal keys are cheap near the end of the sequence and windowed keys anywhere.
    """
    B, S_q, H_q, dqk = q.shape
    _, S_kv, H_kv, dv_ = v.shape
    G = H_q // H_kv
    scale = 1.0 / np.sqrt(dqk) if scale is None else float(scale)
    rows, keys = list(rows), list(keys)
    cache, heads = {}, {}

    def kv(hk):  # one kv head's K and V of entry b in fp64, converted once
        if hk not in heads:
            heads[hk] = (np.ascontiguousarray(k[b, :, hk], dtype=np.float64),
                         np.ascontiguousarray(v[b, :, hk], dtype=np.float64))
        return heads[hk]

    def row(h, i):
        if (h, i) not in cache:
            kh, vh = kv(h // G)
            cache[(h, i)] = _row(q, kh, vh, dout, b, h, i, scale, causal, window, _sink(softmax_type, offset, h))
        return cache[(h, i)]

    out = {"o": np.zeros((len(rows), H_q, dv_)), "lse": np.zeros((len(rows), H_q)),
           "dq": np.zeros((len(rows), H_q, dqk)), "dk": np.zeros((len(keys), H_kv, dqk)),
           "dv": np.zeros((len(keys), H_kv, dv_))}
    for n, i in enumerate(rows):
        for h in range(H_q):
            r = row(h, i)
            out["o"][n, h] = r["o"]
            out["lse"][n, h] = r["lse"]
            out["dq"][n, h] = r["dq"]
    for n, j in enumerate(keys):
        lo, hi = _rows_seeing(j, S_q, causal, window)
        for h in range(H_q):
            hk = h // G
            for i in range(lo, hi + 1):
                r = row(h, i)
                t = j - r["lo"]
                if t < 0 or t >= r["P"].size:  # key j is outside row i's range
                    continue
                out["dk"][n, hk] += scale * r["dS"][t] * np.asarray(q[b, i, h], dtype=np.float64)
                out["dv"][n, hk] += r["P"][t] * np.asarray(dout[b, i, h], dtype=np.float64)
    return out
