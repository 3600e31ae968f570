"""fp64 CPU oracle for fused BSHD attention (forward + backward).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may call this module; the product package never
imports it.  It shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain loops over a fully materialised
score matrix, one (batch, head) at a time).  This module only compiles it with
gcc on first use and marshals numpy arrays through ctypes.

Definitions followed (see ``oracle.c`` for the full statement):
  * "Speed up attention on GPU with cuDNN and TransformerEngine", section "How
    attention works" and steps 4 and 7 (naive attention, causal masking);
  * "JAX: Single-GPU Attention with TransformerEngine", sections 1, 4 and
    "Other attention knobs" (GQA, sliding window, MLA head dims, scale_factor,
    sink softmax types);
  * "[JAX] Add support for sink attention in JAX #2225", Greptile summaries and
    the review thread on the off-by-one offset (vanilla / off-by-one / learnable).

``oracle.fp8`` adds the E4M3 codec, per-tensor quantisation and the FP8 forward
(codelab step 10, "Inspect the FP8 path") in numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

VANILLA, OFF_BY_ONE, LEARNABLE = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_oracle.so (gcc, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        i, d = ctypes.c_int, ctypes.c_double
        u64 = ctypes.c_uint64
        lib.oracle_fwd.argtypes = [dp, dp, dp, i, i, i, i, i, i, i, d, i, i, i, dp, dp, i, i, i, u64, u64, i, i,
                                   dp, dp, dp, dp]
        lib.oracle_fwd.restype = ctypes.c_int
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i, i, d, i, i, i, dp, dp, i, i, i, u64, u64, i, i,
                                   dp, dp, dp, dp, dp, dp]
        lib.oracle_bwd.restype = ctypes.c_int
        u32p = ctypes.POINTER(ctypes.c_uint32)
        lib.oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_dropout_keep.argtypes = [i, i, i, i, i, u64, u64, ctypes.POINTER(ctypes.c_ubyte)]
        lib.oracle_dropout_keep.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_scale(d_qk: int) -> float:
    """1/sqrt(d_qk): the codelab's 1/sqrt(d_k) (the Q/K head dim under MLA dims)."""
    return 1.0 / np.sqrt(d_qk)


def dropout_threshold(p: float) -> int:
    """The drop threshold t of probability p: pairs whose 16-bit uniform is below t are
    dropped, so p is realised as t / 65536 (t = floor(p * 65536 + 1/2))."""
    p = float(p)
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    t = int(np.floor(p * 65536.0 + 0.5))
    if t > 65535:
        raise ValueError("dropout probability rounds to 1")
    return t


def philox4x32_10(counter, key):
    """Philox4x32-10 of one 4 x 32-bit counter under a 2 x 32-bit key (four uint32 words)."""
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in counter])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    out = (ctypes.c_uint32 * 4)()
    _load().oracle_philox4x32_10(c, k, out)
    return np.array(list(out), dtype=np.uint32)


def dropout_keep(b, h, Sq, Skv, p, rng_state):
    """Keep decisions [Sq, Skv] (bool) of batch b, query head h for drop probability p
    and rng_state = (seed, offset)."""
    keep = np.zeros((Sq, Skv), dtype=np.uint8)
    rc = _load().oracle_dropout_keep(int(b), int(h), int(Sq), int(Skv), dropout_threshold(p),
                                     int(rng_state[0]), int(rng_state[1]),
                                     keep.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)))
    if rc != 0:
        raise ValueError("oracle_dropout_keep rejected its arguments")
    return keep.astype(bool)


def _drop_args(dropout_p, rng_state):
    t = dropout_threshold(dropout_p)
    seed, off = (0, 0) if rng_state is None else (int(rng_state[0]), int(rng_state[1]))
    return t, seed, off


def _bias_args(bias, B, Hq, Sq, Skv):
    if bias is None:
        return None, 1, 1
    bias = _f64(bias)
    Bb, Hb = bias.shape[0], bias.shape[1]
    assert bias.shape == (Bb, Hb, Sq, Skv) and Bb in (1, B) and Hb in (1, Hq), bias.shape
    return bias, Bb, Hb


def attention_fwd(q, k, v, *, causal=True, window=-1, softmax_type=VANILLA,
                  offset=None, scale=None, bias=None, dropout_p=0.0, rng_state=None, dropout_origin=(0, 0)):
    """O, LSE, p_sink, rowsum for BSHD q [B,Sq,Hq,dqk], k [B,Skv,Hkv,dqk], v [B,Skv,Hkv,dv].

    bias: optional [Bb,Hb,Sq,Skv] (Bb in {1,B}, Hb in {1,Hq}) added to the scaled scores.
    dropout_p, rng_state = (seed, offset): attention dropout (see oracle.c); rowsum,
    LSE and p_sink are those of the undropped probabilities.  dropout_origin = (b0, h0):
    the arrays are batch entries b0.. and query heads h0.. of a bigger problem, whose
    decisions they take.
    Returns a dict of float64 arrays: o [B,Sq,Hq,dv]; lse, psink, rowsum [B,Hq,Sq].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, dqk = q.shape
    _, Skv, Hkv, dv = v.shape
    assert k.shape == (B, Skv, Hkv, dqk)
    scale = default_scale(dqk) if scale is None else float(scale)
    off = _f64(offset).reshape(-1) if offset is not None else None
    bias, Bb, Hb = _bias_args(bias, B, Hq, Sq, Skv)
    o = np.zeros((B, Sq, Hq, dv))
    lse = np.zeros((B, Hq, Sq))
    psink = np.zeros((B, Hq, Sq))
    rowsum = np.zeros((B, Hq, Sq))
    t, seed, roff = _drop_args(dropout_p, rng_state)
    rc = _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, Hq, Hkv, dqk, dv,
                            scale, int(bool(causal)), int(window), int(softmax_type),
                            _ptr(off), _ptr(bias), Bb, Hb, t, seed, roff,
                            int(dropout_origin[0]), int(dropout_origin[1]),
                            _ptr(o), _ptr(lse), _ptr(psink), _ptr(rowsum))
    if rc != 0:
        raise ValueError("oracle_fwd rejected its arguments")
    return {"o": o, "lse": lse, "psink": psink, "rowsum": rowsum}


def attention_bwd(q, k, v, dout, *, causal=True, window=-1, softmax_type=VANILLA,
                  offset=None, scale=None, bias=None, dropout_p=0.0, rng_state=None, dropout_origin=(0, 0)):
    """dq, dk, dv, d_offset [Hq], D [B,Hq,Sq] (= dO.O) and, with a bias, dbias (its
    shape) for the same arguments as fwd."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Sq, Hq, dqk = q.shape
    _, Skv, Hkv, dv = v.shape
    assert dout.shape == (B, Sq, Hq, dv)
    scale = default_scale(dqk) if scale is None else float(scale)
    off = _f64(offset).reshape(-1) if offset is not None else None
    bias, Bb, Hb = _bias_args(bias, B, Hq, Sq, Skv)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    doff = np.zeros(Hq)
    D = np.zeros((B, Hq, Sq))
    dbias = np.zeros_like(bias) if bias is not None else None
    t, seed, roff = _drop_args(dropout_p, rng_state)
    rc = _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, Sq, Skv, Hq, Hkv,
                            dqk, dv, scale, int(bool(causal)), int(window),
                            int(softmax_type), _ptr(off), _ptr(bias), Bb, Hb, t, seed, roff,
                            int(dropout_origin[0]), int(dropout_origin[1]),
                            _ptr(dq), _ptr(dk), _ptr(dvv), _ptr(doff), _ptr(D), _ptr(dbias))
    if rc != 0:
        raise ValueError("oracle_bwd rejected its arguments")
    out = {"dq": dq, "dk": dk, "dv": dvv, "d_offset": doff, "D": D}
    if dbias is not None:
        out["dbias"] = dbias
    return out


# ----------------------------------------------------------------------------- padded batches
def _lens(seq_lens, B: int, S: int):
    """Per-entry lengths clamped to [0, S]; None means every entry is full length."""
    if seq_lens is None:
        return [S] * B
    lens = np.asarray(seq_lens).reshape(-1)
    assert lens.shape == (B,), "one length per batch entry"
    return [int(min(max(int(x), 0), S)) for x in lens]


def _sink_logit(softmax_type, off, h):
    if softmax_type == OFF_BY_ONE:
        return 0.0
    if softmax_type == LEARNABLE:
        return float(off[h])
    return -np.inf


def _entry_bias(bias, b, lq, lkv):
    """The bias planes entry b of a padded batch sees, cropped to its own rows and keys."""
    if bias is None:
        return None
    bias = np.asarray(bias)
    return bias[(b if bias.shape[0] > 1 else 0):][:1, :, :lq, :lkv]


def attention_fwd_varlen(q, k, v, *, seq_lens_q=None, seq_lens_kv=None, causal=True, window=-1,
                         softmax_type=VANILLA, offset=None, scale=None, bias=None):
    """Padded batch: entry b holds its Lq[b] queries and Lkv[b] keys at the front of
    its rows.  Its result is attention_fwd on those rows alone; a padded query row
    sees no key, so O = 0, LSE = the sink logit c (-inf for vanilla), p_sink = 1
    with a sink (0 without) and rowsum = 0.  Lengths are clamped to [0, S].
    bias: optional [Bb, Hb, S_q, S_kv] over the padded shape; an entry uses the top-left
    [Lq, Lkv] corner of its planes.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Hq, dqk = q.shape
    _, Skv, Hkv, dv = v.shape
    Lq, Lkv = _lens(seq_lens_q, B, Sq), _lens(seq_lens_kv, B, Skv)
    off = _f64(offset).reshape(-1) if offset is not None else None
    o = np.zeros((B, Sq, Hq, dv))
    lse = np.empty((B, Hq, Sq))
    psink = np.empty((B, Hq, Sq))
    rowsum = np.zeros((B, Hq, Sq))
    for h in range(Hq):  # padded rows first; valid rows are overwritten below
        c = _sink_logit(softmax_type, off, h)
        lse[:, h, :] = c
        psink[:, h, :] = 0.0 if softmax_type == VANILLA else 1.0
    for b in range(B):
        if Lq[b] == 0 or Lkv[b] == 0:
            continue  # every row of the entry sees no key
        r = attention_fwd(q[b:b + 1, :Lq[b]], k[b:b + 1, :Lkv[b]], v[b:b + 1, :Lkv[b]], causal=causal,
                          window=window, softmax_type=softmax_type, offset=offset, scale=scale,
                          bias=_entry_bias(bias, b, Lq[b], Lkv[b]))
        o[b, :Lq[b]] = r["o"][0]
        lse[b, :, :Lq[b]] = r["lse"][0]
        psink[b, :, :Lq[b]] = r["psink"][0]
        rowsum[b, :, :Lq[b]] = r["rowsum"][0]
    return {"o": o, "lse": lse, "psink": psink, "rowsum": rowsum}


def attention_bwd_varlen(q, k, v, dout, *, seq_lens_q=None, seq_lens_kv=None, causal=True, window=-1,
                         softmax_type=VANILLA, offset=None, scale=None, bias=None):
    """Gradients for attention_fwd_varlen: padded query rows and padded keys get zero
    gradients (dO of a padded row is ignored), and d_offset sums the valid rows of
    every entry.  With a bias, also dbias (the bias's shape): each entry's dS added into
    the corner of its planes, zero elsewhere."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Sq, Hq, dqk = q.shape
    _, Skv, Hkv, dv = v.shape
    Lq, Lkv = _lens(seq_lens_q, B, Sq), _lens(seq_lens_kv, B, Skv)
    dq, dk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    doff = np.zeros(Hq)
    D = np.zeros((B, Hq, Sq))
    dbias = None if bias is None else np.zeros(np.asarray(bias).shape)
    for b in range(B):
        if Lq[b] == 0 or Lkv[b] == 0:
            continue  # O = 0 on every row of the entry: nothing flows back
        r = attention_bwd(q[b:b + 1, :Lq[b]], k[b:b + 1, :Lkv[b]], v[b:b + 1, :Lkv[b]], dout[b:b + 1, :Lq[b]],
                          causal=causal, window=window, softmax_type=softmax_type, offset=offset, scale=scale,
                          bias=_entry_bias(bias, b, Lq[b], Lkv[b]))
        dq[b, :Lq[b]] = r["dq"][0]
        dk[b, :Lkv[b]] = r["dk"][0]
        dvv[b, :Lkv[b]] = r["dv"][0]
        D[b, :, :Lq[b]] = r["D"][0]
        doff += r["d_offset"]
        if dbias is not None:
            dbias[(b if dbias.shape[0] > 1 else 0), :, :Lq[b], :Lkv[b]] += r["dbias"][0]
    out = {"dq": dq, "dk": dk, "dv": dvv, "d_offset": doff, "D": D}
    if dbias is not None:
        out["dbias"] = dbias
    return out
