"""GB300 (sm_103a) fused scaled-dot-product attention, forward and backward.

A thin Python binding over the C ABI of ``libsdpa_tmem.so`` (declared in
``include/sdpa_tmem.h``): the functions below carry the same names and only
marshal torch tensors into device pointers and the current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; there is no other
path.  Importing this package does not load the library; the first call does,
and it raises if the library has not been built.

    from scaled_dot_product_tmem_gb300 import sdpa_forward, sdpa_backward
    o, lse = sdpa_forward(q, k, v, causal=True, window=1024)
    dq, dk, dv, d_off = sdpa_backward(q, k, v, o, dout, lse, causal=True, window=1024)

Tensors are BSHD bf16 on the GPU: q [B,S_q,H_q,d_qk], k [B,S_kv,H_kv,d_qk],
v [B,S_kv,H_kv,d_v]; lse fp32 [B,H_q,S_q]; softmax_offset fp32 [H_q].
"""
from __future__ import annotations

import ctypes
import os

import torch

VANILLA, OFF_BY_ONE, LEARNABLE = 0, 1, 2
SOFTMAX_TYPES = {"vanilla": VANILLA, "off_by_one": OFF_BY_ONE, "learnable": LEARNABLE}
ATTN_OK = 0

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdpa_tmem.so")
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = attn_last_error_message()
        super().__init__(f"{what}: {attn_status_string(status)} (status {status})" + (f" [{detail}]" if detail else ""))


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m scaled_dot_product_tmem_gb300.build`"
                           " (or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp, vp]
    lib.attn_fwd.restype = i
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
    lib.attn_bwd_workspace_size.restype = sz
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp, i, vp, sz,
                             vp]
    lib.attn_bwd.restype = i
    lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp, vp, vp, vp]
    lib.attn_fwd_varlen.restype = i
    lib.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp, vp,
                                    vp, i, vp, sz, vp]
    lib.attn_bwd_varlen.restype = i
    lib.attn_status_string.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_last_error_message.argtypes = []
    lib.attn_last_error_message.restype = ctypes.c_char_p
    lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp,
                                     vp]
    lib.attn_bwd_noalloc.restype = i
    lib.attn_bwd_noalloc_max_scratch_bytes.argtypes = []
    lib.attn_bwd_noalloc_max_scratch_bytes.restype = sz
    lib.attn_bwd_noalloc_message.argtypes = []
    lib.attn_bwd_noalloc_message.restype = ctypes.c_char_p
    lib.attn_timing_enable.argtypes = [i]
    lib.attn_timing_enable.restype = i
    lib.attn_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int), i]
    lib.attn_timing_read.restype = i
    lib.attn_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.attn_last_device_error.restype = i
    lib.attn_selftest_wait_timeout.argtypes = [i, vp]
    lib.attn_selftest_wait_timeout.restype = i
    lib.attn_fwd_bias.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i, i, i, vp, vp]
    lib.attn_fwd_bias.restype = i
    lib.attn_bwd_bias.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, vp, i, i, i, i, i, i, i, f, i, i,
                                  i, vp, i, vp, sz, vp]
    lib.attn_bwd_bias.restype = i
    lib.attn_fp8_amax.argtypes = [vp, sz, vp, vp]
    lib.attn_fp8_amax.restype = i
    lib.attn_fp8_quantize.argtypes = [vp, vp, i, i, i, i, i, vp, vp, vp, vp]
    lib.attn_fp8_quantize.restype = i
    lib.attn_fp8_vt_row_bytes.argtypes = [i]
    lib.attn_fp8_vt_row_bytes.restype = i
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i, vp, vp]
    lib.attn_fwd_fp8.restype = i
    lib.attn_fwd_varlen_bias.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i, i, i, vp, vp, vp,
                                         vp]
    lib.attn_fwd_varlen_bias.restype = i
    lib.attn_bwd_varlen_bias.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, vp, i, i, i, i, i, i, i, f,
                                         i, i, i, vp, vp, vp, i, vp, sz, vp]
    lib.attn_bwd_varlen_bias.restype = i
    lib.attn_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp, f, vp, vp]
    lib.attn_fwd_dropout.restype = i
    lib.attn_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp, f,
                                     vp, i, vp, sz, vp]
    lib.attn_bwd_dropout.restype = i
    lib.attn_fp8_quantize_e5m2.argtypes = [vp, vp, i, i, i, i, i, vp, vp, vp, vp]
    lib.attn_fp8_quantize_e5m2.restype = i
    lib.attn_fp8_quantize_both.argtypes = [vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp]
    lib.attn_fp8_quantize_both.restype = i
    lib.attn_bwd_fp8_workspace_size.argtypes = [i, i, i]
    lib.attn_bwd_fp8_workspace_size.restype = sz
    lib.attn_bwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i,
                                 i, i, i, f, i, i, i, vp, vp, sz, vp]
    lib.attn_bwd_fp8.restype = i
    _lib = lib
    return lib


def library():
    """The loaded ctypes library (loads it on first use)."""
    return _load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, ndim):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _stype(softmax_type):
    return SOFTMAX_TYPES[softmax_type] if isinstance(softmax_type, str) else int(softmax_type)


# ----------------------------------------------------------------------------- C ABI, same names


def attn_status_string(status: int) -> str:
    return _load().attn_status_string(int(status)).decode()


def attn_last_error_message() -> str:
    return _load().attn_last_error_message().decode()


def attn_last_device_error(stream=None):
    """Synchronise the stream; return (status, site) of the device error word and clear it."""
    site = ctypes.c_int(0)
    st = _load().attn_last_device_error(_stream(stream), ctypes.byref(site))
    return st, site.value


def attn_selftest_wait_timeout(site: int, stream=None) -> None:
    """Enqueue the failure-path self-test (a bounded wait that runs out; no fault)."""
    st = _load().attn_selftest_wait_timeout(int(site), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_selftest_wait_timeout")


def _check_lens(t, name, B):
    if t is not None:
        _check(t, name, torch.int32, 1)
        if t.shape[0] != B:
            raise ValueError(f"{name}: one length per batch entry ({B}), got {t.shape[0]}")


def _check_bias(bias, B, H_q, S_q, S_kv):
    _check(bias, "bias", torch.bfloat16, 4)
    Bb, Hb = bias.shape[0], bias.shape[1]
    if tuple(bias.shape[2:]) != (S_q, S_kv) or Bb not in (1, B) or Hb not in (1, H_q):
        raise ValueError(f"bias must be [1 or {B}, 1 or {H_q}, {S_q}, {S_kv}], got {tuple(bias.shape)}")
    return Bb, Hb


def _check_rng(rng_state):
    """rng_state: a CUDA int64 (or uint64) tensor of two values, seed then offset."""
    if rng_state is None:
        raise ValueError("dropout needs rng_state: a CUDA int64 tensor [seed, offset]")
    if rng_state.dtype not in (torch.int64, getattr(torch, "uint64", torch.int64)):
        raise TypeError(f"rng_state must be int64 or uint64, got {rng_state.dtype}")
    if tuple(rng_state.shape) != (2,) or not rng_state.is_contiguous() or not rng_state.is_cuda:
        raise ValueError("rng_state must be a contiguous CUDA tensor of shape [2] (seed, offset)")


def attn_fwd(q, k, v, o, lse, *, causal=True, window=-1, softmax_type=VANILLA, softmax_offset=None, scale=0.0,
             seq_lens_q=None, seq_lens_kv=None, bias=None, dropout_p=0.0, rng_state=None, stream=None):
    """Forward into preallocated o [B,S_q,H_q,d_v] bf16 and lse [B,H_q,S_q] fp32.

    seq_lens_q / seq_lens_kv: optional int32 [B] device tensors for a padded batch
    (attn_fwd_varlen); None means full length.
    bias: optional bf16 [1 or B, 1 or H_q, S_q, S_kv] added to the scaled scores
    (attn_fwd_bias).
    dropout_p, rng_state: attention dropout (attn_fwd_dropout); rng_state is a CUDA
    int64 tensor [seed, offset], to be passed to the backward of the same step too.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _check(t, n, torch.bfloat16, 4)
    _check(lse, "lse", torch.float32, 3)
    if softmax_offset is not None:
        _check(softmax_offset, "softmax_offset", torch.float32, 1)
    B, S_q, H_q, d_qk = q.shape
    _, S_kv, H_kv, d_v = v.shape
    _check_lens(seq_lens_q, "seq_lens_q", B)
    _check_lens(seq_lens_kv, "seq_lens_kv", B)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, S_q, S_kv, H_q, H_kv, d_qk, d_v, float(scale or 0.0),
            int(bool(causal)), int(window), _stype(softmax_type), _ptr(softmax_offset))
    if dropout_p:
        if bias is not None or seq_lens_q is not None or seq_lens_kv is not None:
            raise ValueError("dropout with a bias or padded batches is not supported")
        _check_rng(rng_state)
        st = _load().attn_fwd_dropout(*args, float(dropout_p), _ptr(rng_state), _stream(stream))
    elif bias is not None:
        Bb, Hb = _check_bias(bias, B, H_q, S_q, S_kv)
        if seq_lens_q is None and seq_lens_kv is None:
            st = _load().attn_fwd_bias(*args[:5], _ptr(bias), Bb, Hb, *args[5:], _stream(stream))
        else:
            st = _load().attn_fwd_varlen_bias(*args[:5], _ptr(bias), Bb, Hb, *args[5:], _ptr(seq_lens_q),
                                              _ptr(seq_lens_kv), _stream(stream))
    elif seq_lens_q is None and seq_lens_kv is None:
        st = _load().attn_fwd(*args, _stream(stream))
    else:
        st = _load().attn_fwd_varlen(*args, _ptr(seq_lens_q), _ptr(seq_lens_kv), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")


def attn_bwd_workspace_size(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, deterministic=True) -> int:
    return int(_load().attn_bwd_workspace_size(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, int(bool(deterministic))))


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, d_offset=None, *, causal=True, window=-1, softmax_type=VANILLA,
             softmax_offset=None, scale=0.0, deterministic=True, workspace=None, seq_lens_q=None, seq_lens_kv=None,
             bias=None, dbias=None, dropout_p=0.0, rng_state=None, stream=None):
    """Backward into preallocated dq, dk, dv (bf16) and d_offset (fp32 [H_q], learnable).

    seq_lens_q / seq_lens_kv as for attn_fwd (attn_bwd_varlen).  bias as for attn_fwd,
    with dbias an optional preallocated fp32 tensor of the bias's shape
    (attn_bwd_bias).  dropout_p / rng_state as for attn_fwd (attn_bwd_dropout; the
    forward's values).
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, torch.bfloat16, 4)
    _check(lse, "lse", torch.float32, 3)
    B, S_q, H_q, d_qk = q.shape
    _, S_kv, H_kv, d_v = v.shape
    _check_lens(seq_lens_q, "seq_lens_q", B)
    _check_lens(seq_lens_kv, "seq_lens_kv", B)
    need = attn_bwd_workspace_size(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, deterministic)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(d_offset),
            B, S_q, S_kv, H_q, H_kv, d_qk, d_v, float(scale or 0.0), int(bool(causal)), int(window),
            _stype(softmax_type), _ptr(softmax_offset))
    tail = (int(bool(deterministic)), _ptr(workspace), workspace.numel(), _stream(stream))
    if dropout_p:
        if bias is not None or seq_lens_q is not None or seq_lens_kv is not None:
            raise ValueError("dropout with a bias or padded batches is not supported")
        _check_rng(rng_state)
        st = _load().attn_bwd_dropout(*args, float(dropout_p), _ptr(rng_state), *tail)
    elif bias is not None:
        Bb, Hb = _check_bias(bias, B, H_q, S_q, S_kv)
        if dbias is not None:
            _check(dbias, "dbias", torch.float32, 4)
            if dbias.shape != bias.shape:
                raise ValueError("dbias must have the bias's shape")
        if seq_lens_q is None and seq_lens_kv is None:
            st = _load().attn_bwd_bias(*args[:10], _ptr(bias), Bb, Hb, _ptr(dbias), *args[10:], *tail)
        else:
            st = _load().attn_bwd_varlen_bias(*args[:10], _ptr(bias), Bb, Hb, _ptr(dbias), *args[10:],
                                              _ptr(seq_lens_q), _ptr(seq_lens_kv), *tail)
    elif seq_lens_q is None and seq_lens_kv is None:
        st = _load().attn_bwd(*args, *tail)
    else:
        st = _load().attn_bwd_varlen(*args, _ptr(seq_lens_q), _ptr(seq_lens_kv), *tail)
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")


def attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, d_offset=None, *, causal=True, window=-1,
                     softmax_type=VANILLA, softmax_offset=None, scale=0.0, stream=None):
    """attn_bwd without a workspace: for callers that must not allocate device memory.

    The library keeps the scratch in a fixed built-in array (see
    attn_bwd_noalloc_max_scratch_bytes); this function allocates nothing either.
    Always the deterministic backward.  Calls that overlap on the GPU race on the
    shared array; the first call on a device must come before any stream capture.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, torch.bfloat16, 4)
    _check(lse, "lse", torch.float32, 3)
    B, S_q, H_q, d_qk = q.shape
    _, S_kv, H_kv, d_v = v.shape
    st = _load().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(d_offset), B, S_q, S_kv, H_q, H_kv, d_qk, d_v, float(scale or 0.0),
                                  int(bool(causal)), int(window), _stype(softmax_type), _ptr(softmax_offset),
                                  _stream(stream))
    if st != ATTN_OK:
        msg = _load().attn_bwd_noalloc_message().decode()
        raise AttnError(st, "attn_bwd_noalloc" + (f" ({msg})" if msg else ""))


def attn_bwd_noalloc_max_scratch_bytes() -> int:
    return int(_load().attn_bwd_noalloc_max_scratch_bytes())


def attn_bwd_noalloc_message() -> str:
    return _load().attn_bwd_noalloc_message().decode()


def attn_fwd_varlen(q, k, v, o, lse, seq_lens_q, seq_lens_kv, **kw):
    """attn_fwd on a padded batch: int32 [B] device tensors of query / key lengths."""
    attn_fwd(q, k, v, o, lse, seq_lens_q=seq_lens_q, seq_lens_kv=seq_lens_kv, **kw)


def attn_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, d_offset, seq_lens_q, seq_lens_kv, **kw):
    """attn_bwd on a padded batch (lengths as for attn_fwd_varlen)."""
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, d_offset, seq_lens_q=seq_lens_q, seq_lens_kv=seq_lens_kv, **kw)


def attn_fwd_varlen_bias(q, k, v, o, lse, bias, seq_lens_q, seq_lens_kv, **kw):
    """attn_fwd with an additive bias on a padded batch (entry b uses the top-left
    [Lq[b], Lkv[b]] corner of its bias planes)."""
    attn_fwd(q, k, v, o, lse, bias=bias, seq_lens_q=seq_lens_q, seq_lens_kv=seq_lens_kv, **kw)


def attn_bwd_varlen_bias(q, k, v, o, dout, lse, dq, dk, dv, d_offset, bias, dbias, seq_lens_q, seq_lens_kv, **kw):
    """attn_bwd with an additive bias on a padded batch; dbias is zero outside each
    entry's corner."""
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, d_offset, bias=bias, dbias=dbias, seq_lens_q=seq_lens_q,
             seq_lens_kv=seq_lens_kv, **kw)


def attn_fwd_dropout(q, k, v, o, lse, dropout_p, rng_state, **kw):
    """attn_fwd with attention dropout: probability dropout_p, rng_state a CUDA int64
    tensor [seed, offset]."""
    attn_fwd(q, k, v, o, lse, dropout_p=dropout_p, rng_state=rng_state, **kw)


def attn_bwd_dropout(q, k, v, o, dout, lse, dq, dk, dv, d_offset, dropout_p, rng_state, **kw):
    """attn_bwd of a forward with attention dropout (the forward's dropout_p and rng_state)."""
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, d_offset, dropout_p=dropout_p, rng_state=rng_state, **kw)


def attn_fwd_bias(q, k, v, o, lse, bias, **kw):
    """attn_fwd with an additive bf16 bias [1 or B, 1 or H_q, S_q, S_kv]."""
    attn_fwd(q, k, v, o, lse, bias=bias, **kw)


def attn_bwd_bias(q, k, v, o, dout, lse, dq, dk, dv, d_offset, bias, dbias, **kw):
    """attn_bwd with an additive bias; dbias: fp32 tensor of the bias's shape, or None."""
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, d_offset, bias=bias, dbias=dbias, **kw)


KERNEL_CLASSES = ("fwd", "bwd_preprocess", "bwd_kv", "bwd_q", "bwd_dq_convert", "fp8_quantize")


def attn_timing_enable(on: bool = True) -> None:
    _load().attn_timing_enable(int(bool(on)))


def attn_timing_read():
    """{class: (milliseconds, kernel launches)} accumulated since the last read."""
    n = len(KERNEL_CLASSES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    st = _load().attn_timing_read(ms, cnt, n)
    if st != ATTN_OK:
        raise AttnError(st, "attn_timing_read")
    return {name: (ms[k], cnt[k]) for k, name in enumerate(KERNEL_CLASSES)}


# ----------------------------------------------------------------------------- FP8 (E4M3) forward


def attn_fp8_vt_row_bytes(S: int) -> int:
    return int(_load().attn_fp8_vt_row_bytes(int(S)))


def attn_fp8_amax(x, amax, *, stream=None):
    """amax (fp32 [1], device) = max |x| over the bf16 tensor x."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or not x.is_cuda:
        raise TypeError("x must be a contiguous bf16 CUDA tensor")
    _check(amax, "amax", torch.float32, 1)
    st = _load().attn_fp8_amax(_ptr(x), x.numel(), _ptr(amax), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fp8_amax")


def _fp8_quantize(name, x, x8, amax, descale, transpose, amax_out, stream):
    _check(x, "x", torch.bfloat16, 4)
    _check(x8, "x8", torch.uint8, 4)
    _check(amax, "amax", torch.float32, 1)
    _check(descale, "descale", torch.float32, 1)
    B, S, H, d = x.shape
    want = (B, H, d, attn_fp8_vt_row_bytes(S)) if transpose else (B, S, H, d)
    if tuple(x8.shape) != want:
        raise ValueError(f"x8 must have shape {want}, got {tuple(x8.shape)}")
    if amax_out is not None:
        _check(amax_out, "amax_out", torch.float32, 1)
    st = getattr(_load(), name)(_ptr(x), _ptr(x8), B, S, H, d, int(bool(transpose)), _ptr(amax), _ptr(descale),
                                _ptr(amax_out), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, name)


def attn_fp8_quantize(x, x8, amax, descale, *, transpose=False, amax_out=None, stream=None):
    """x8 (uint8 E4M3) = E4M3(x * 448 / amax); descale (fp32 [1]) = amax / 448 as 1 / scale.

    x bf16 BSHD [B,S,H,d]; x8 the same shape, or [B,H,d,S_pad] with transpose=True.
    amax_out (fp32 [1], optional): records max |x| during the same pass."""
    _fp8_quantize("attn_fp8_quantize", x, x8, amax, descale, transpose, amax_out, stream)


def attn_fp8_quantize_e5m2(x, x8, amax, descale, *, transpose=False, amax_out=None, stream=None):
    """attn_fp8_quantize with E5M2 codes: x8 = E5M2(x * 57344 / amax)."""
    _fp8_quantize("attn_fp8_quantize_e5m2", x, x8, amax, descale, transpose, amax_out, stream)


def attn_fp8_quantize_both(x, x8, x8t, amax, descale, *, e5m2=False, amax_out=None, stream=None):
    """One read of x, both layouts: x8 BSHD [B,S,H,d] and x8t [B,H,d,S_pad] (uint8), E4M3 or
    (e5m2=True) E5M2, with the same codes as the two separate casts."""
    _check(x, "x", torch.bfloat16, 4)
    _check(x8, "x8", torch.uint8, 4)
    _check(x8t, "x8t", torch.uint8, 4)
    _check(amax, "amax", torch.float32, 1)
    _check(descale, "descale", torch.float32, 1)
    B, S, H, d = x.shape
    if tuple(x8.shape) != (B, S, H, d):
        raise ValueError(f"x8 must have shape {(B, S, H, d)}, got {tuple(x8.shape)}")
    want = (B, H, d, attn_fp8_vt_row_bytes(S))
    if tuple(x8t.shape) != want:
        raise ValueError(f"x8t must have shape {want}, got {tuple(x8t.shape)}")
    if amax_out is not None:
        _check(amax_out, "amax_out", torch.float32, 1)
    st = _load().attn_fp8_quantize_both(_ptr(x), _ptr(x8), _ptr(x8t), B, S, H, d, int(bool(e5m2)), _ptr(amax),
                                        _ptr(descale), _ptr(amax_out), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fp8_quantize_both")


def fp8_quantize_both(x, *, amax=None, amax_out=None, fmt="e4m3", stream=None):
    """fp8_quantize in both layouts from one read: returns (x8, x8t, amax, descale)."""
    if fmt not in ("e4m3", "e5m2"):
        raise ValueError(f"fmt must be 'e4m3' or 'e5m2', got {fmt!r}")
    B, S, H, d = x.shape
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
        attn_fp8_amax(x, amax, stream=stream)
    x8 = torch.empty((B, S, H, d), dtype=torch.uint8, device=x.device)
    x8t = torch.empty((B, H, d, attn_fp8_vt_row_bytes(S)), dtype=torch.uint8, device=x.device)
    descale = torch.empty(1, dtype=torch.float32, device=x.device)
    attn_fp8_quantize_both(x, x8, x8t, amax, descale, e5m2=(fmt == "e5m2"), amax_out=amax_out, stream=stream)
    return x8, x8t, amax, descale


def attn_fwd_fp8(q8, k8, vt8, descale_q, descale_k, descale_v, o, lse, *, causal=True, window=-1,
                 softmax_type=VANILLA, softmax_offset=None, scale=0.0, stream=None):
    """E4M3 forward into preallocated o [B,S_q,H_q,d] bf16 and lse [B,H_q,S_q] fp32.

    q8 [B,S_q,H_q,d], k8 [B,S_kv,H_kv,d] uint8 E4M3 BSHD; vt8 [B,H_kv,d,S_pad] from
    attn_fp8_quantize(transpose=True); descale_* fp32 [1] device tensors."""
    for t, n in ((q8, "q8"), (k8, "k8"), (vt8, "vt8")):
        _check(t, n, torch.uint8, 4)
    for t, n in ((descale_q, "descale_q"), (descale_k, "descale_k"), (descale_v, "descale_v")):
        _check(t, n, torch.float32, 1)
    _check(o, "o", torch.bfloat16, 4)
    _check(lse, "lse", torch.float32, 3)
    if softmax_offset is not None:
        _check(softmax_offset, "softmax_offset", torch.float32, 1)
    B, S_q, H_q, d = q8.shape
    _, S_kv, H_kv, _ = k8.shape
    if tuple(vt8.shape) != (B, H_kv, d, attn_fp8_vt_row_bytes(S_kv)):
        raise ValueError(f"vt8 must have shape {(B, H_kv, d, attn_fp8_vt_row_bytes(S_kv))}, got {tuple(vt8.shape)}")
    st = _load().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(descale_q), _ptr(descale_k), _ptr(descale_v),
                              _ptr(o), _ptr(lse), B, S_q, S_kv, H_q, H_kv, d, float(scale or 0.0),
                              int(bool(causal)), int(window), _stype(softmax_type), _ptr(softmax_offset),
                              _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8")


def fp8_quantize(x, *, transpose=False, amax=None, amax_out=None, fmt="e4m3", stream=None):
    """Per-tensor E4M3 (fmt="e5m2": E5M2) quantisation of a bf16 BSHD tensor: returns
    (x8, amax, descale).

    amax: an fp32 [1] device tensor holding the scaling statistic (for example the
    max of an amax history); None computes this tensor's own amax first (a second
    pass).  amax_out: optional fp32 [1] device tensor that records this tensor's
    amax during the cast (delayed scaling)."""
    if fmt not in ("e4m3", "e5m2"):
        raise ValueError(f"fmt must be 'e4m3' or 'e5m2', got {fmt!r}")
    B, S, H, d = x.shape
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
        attn_fp8_amax(x, amax, stream=stream)
    shape = (B, H, d, attn_fp8_vt_row_bytes(S)) if transpose else (B, S, H, d)
    x8 = torch.empty(shape, dtype=torch.uint8, device=x.device)
    descale = torch.empty(1, dtype=torch.float32, device=x.device)
    quant = attn_fp8_quantize_e5m2 if fmt == "e5m2" else attn_fp8_quantize
    quant(x, x8, amax, descale, transpose=transpose, amax_out=amax_out, stream=stream)
    return x8, amax, descale


def sdpa_forward_fp8(q, k, v, *, causal=True, window=-1, softmax_type=VANILLA, softmax_offset=None, scale=0.0,
                     stream=None):
    """bf16 in, bf16 out through the E4M3 forward: quantise Q, K (BSHD) and V
    (transposed) with their own amax, then run attn_fwd_fp8.  Returns (o, lse)."""
    q8, _, dq = fp8_quantize(q, stream=stream)
    k8, _, dk = fp8_quantize(k, stream=stream)
    vt8, _, dv = fp8_quantize(v, transpose=True, stream=stream)
    B, S_q, H_q, d = q.shape
    o = torch.empty((B, S_q, H_q, d), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H_q, S_q), dtype=torch.float32, device=q.device)
    attn_fwd_fp8(q8, k8, vt8, dq, dk, dv, o, lse, causal=causal, window=window, softmax_type=softmax_type,
                 softmax_offset=softmax_offset, scale=scale, stream=stream)
    return o, lse


def attn_bwd_fp8_workspace_size(B, S_q, H_q) -> int:
    return int(_load().attn_bwd_fp8_workspace_size(int(B), int(S_q), int(H_q)))


def attn_bwd_fp8(q8, k8, v8, do8, qt8, kt8, dot8, descale_q, descale_k, descale_v, descale_do, o, lse, ds_amax,
                 dq, dk, dv, d_offset=None, *, ds_amax_out=None, causal=True, window=-1, softmax_type=VANILLA,
                 softmax_offset=None, scale=0.0, workspace=None, stream=None):
    """FP8 backward into preallocated bf16 dq, dk, dv (BSHD) and d_offset (fp32 [H_q],
    learnable sinks).  q8, k8, v8 uint8 E4M3 BSHD; do8 uint8 E5M2 BSHD; qt8, dot8
    [B,H_q,d,S_pad(S_q)] and kt8 [B,H_kv,d,S_pad(S_kv)] the same codes transposed;
    o, lse the forward's outputs; descale_*, ds_amax (s = 57344 / ds_amax for dS) and
    ds_amax_out (receives max |dS|) fp32 [1] device tensors."""
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8"), (do8, "do8"), (qt8, "qt8"), (kt8, "kt8"), (dot8, "dot8")):
        _check(t, n, torch.uint8, 4)
    for t, n in ((descale_q, "descale_q"), (descale_k, "descale_k"), (descale_v, "descale_v"),
                 (descale_do, "descale_do"), (ds_amax, "ds_amax")):
        _check(t, n, torch.float32, 1)
    if ds_amax_out is not None:
        _check(ds_amax_out, "ds_amax_out", torch.float32, 1)
    for t, n in ((o, "o"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, torch.bfloat16, 4)
    _check(lse, "lse", torch.float32, 3)
    if softmax_offset is not None:
        _check(softmax_offset, "softmax_offset", torch.float32, 1)
    if d_offset is not None:
        _check(d_offset, "d_offset", torch.float32, 1)
    B, S_q, H_q, d = q8.shape
    _, S_kv, H_kv, _ = k8.shape
    want = {"qt8": (B, H_q, d, attn_fp8_vt_row_bytes(S_q)), "dot8": (B, H_q, d, attn_fp8_vt_row_bytes(S_q)),
            "kt8": (B, H_kv, d, attn_fp8_vt_row_bytes(S_kv))}
    for t, n in ((qt8, "qt8"), (dot8, "dot8"), (kt8, "kt8")):
        if tuple(t.shape) != want[n]:
            raise ValueError(f"{n} must have shape {want[n]}, got {tuple(t.shape)}")
    for t, n, shp in ((v8, "v8", k8.shape), (do8, "do8", q8.shape), (o, "o", q8.shape), (dq, "dq", q8.shape),
                      (dk, "dk", k8.shape), (dv, "dv", k8.shape)):
        if tuple(t.shape) != tuple(shp):
            raise ValueError(f"{n} must have shape {tuple(shp)}, got {tuple(t.shape)}")
    need = attn_bwd_fp8_workspace_size(B, S_q, H_q)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q8.device)
    st = _load().attn_bwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(do8), _ptr(qt8), _ptr(kt8), _ptr(dot8),
                              _ptr(descale_q), _ptr(descale_k), _ptr(descale_v), _ptr(descale_do), _ptr(o), _ptr(lse),
                              _ptr(ds_amax), _ptr(ds_amax_out), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(d_offset), B, S_q,
                              S_kv, H_q, H_kv, d, float(scale or 0.0), int(bool(causal)), int(window),
                              _stype(softmax_type), _ptr(softmax_offset), _ptr(workspace), workspace.numel(),
                              _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_fp8")


def sdpa_backward_fp8(q, k, v, o, dout, lse, *, ds_amax=None, ds_amax_out=None, causal=True, window=-1,
                      softmax_type=VANILLA, softmax_offset=None, scale=0.0, stream=None):
    """bf16 in, bf16 out through the FP8 backward: quantise Q, K, V (E4M3) and dO (E5M2)
    with their own amax, natural and transposed, then run attn_bwd_fp8.  ds_amax: the
    dS scaling statistic (fp32 [1] device tensor, e.g. the max of an amax history);
    None runs the backward twice, the first time only to record this step's max |dS|.
    Returns (dq, dk, dv, d_offset)."""
    q8, qt8, _, sq = fp8_quantize_both(q, stream=stream)
    k8, kt8, _, sk = fp8_quantize_both(k, stream=stream)
    v8, _, sv = fp8_quantize(v, stream=stream)
    do8, dot8, _, sdo = fp8_quantize_both(dout, fmt="e5m2", stream=stream)
    B, S_q, H_q, d = q.shape
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    d_offset = torch.empty(H_q, dtype=torch.float32, device=q.device)
    kw = dict(causal=causal, window=window, softmax_type=softmax_type, softmax_offset=softmax_offset, scale=scale,
              stream=stream)
    if ds_amax is None:
        ds_amax = torch.empty(1, dtype=torch.float32, device=q.device)
        first = torch.ones(1, dtype=torch.float32, device=q.device)
        attn_bwd_fp8(q8, k8, v8, do8, qt8, kt8, dot8, sq, sk, sv, sdo, o, lse, first, dq, dk, dv, d_offset,
                     ds_amax_out=ds_amax, **kw)
    attn_bwd_fp8(q8, k8, v8, do8, qt8, kt8, dot8, sq, sk, sv, sdo, o, lse, ds_amax, dq, dk, dv, d_offset,
                 ds_amax_out=ds_amax_out, **kw)
    return dq, dk, dv, d_offset


# ----------------------------------------------------------------------------- conveniences


def sdpa_forward(q, k, v, *, causal=True, window=-1, softmax_type=VANILLA, softmax_offset=None, scale=0.0,
                 seq_lens_q=None, seq_lens_kv=None, bias=None, dropout_p=0.0, rng_state=None, stream=None):
    """Allocate O and LSE, run attn_fwd, return (o, lse)."""
    B, S_q, H_q, _ = q.shape
    d_v = v.shape[3]
    o = torch.empty((B, S_q, H_q, d_v), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H_q, S_q), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, v, o, lse, causal=causal, window=window, softmax_type=softmax_type,
             softmax_offset=softmax_offset, scale=scale, seq_lens_q=seq_lens_q, seq_lens_kv=seq_lens_kv,
             bias=bias, dropout_p=dropout_p, rng_state=rng_state, stream=stream)
    return o, lse


def sdpa_backward(q, k, v, o, dout, lse, *, causal=True, window=-1, softmax_type=VANILLA, softmax_offset=None,
                  scale=0.0, deterministic=True, workspace=None, seq_lens_q=None, seq_lens_kv=None, bias=None,
                  dropout_p=0.0, rng_state=None, stream=None):
    """Allocate dQ, dK, dV (and d_offset for the learnable sink), run attn_bwd, return them;
    with a bias, also dbias (fp32, the bias's shape) as a fifth output."""
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    st = _stype(softmax_type)
    d_off = torch.empty((q.shape[2],), dtype=torch.float32, device=q.device) if st == LEARNABLE else None
    dbias = torch.empty(bias.shape, dtype=torch.float32, device=q.device) if bias is not None else None
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, d_off, causal=causal, window=window, softmax_type=st,
             softmax_offset=softmax_offset, scale=scale, deterministic=deterministic, workspace=workspace,
             seq_lens_q=seq_lens_q, seq_lens_kv=seq_lens_kv, bias=bias, dbias=dbias, dropout_p=dropout_p,
             rng_state=rng_state, stream=stream)
    return (dq, dk, dv, d_off) if bias is None else (dq, dk, dv, d_off, dbias)


class SDPAFunction(torch.autograd.Function):
    """autograd wrapper: forward and backward both run in the library's kernels (the
    plain, padded-batch, bias and dropout entry points, chosen by the arguments)."""

    @staticmethod
    def forward(ctx, q, k, v, softmax_offset, bias, causal, window, softmax_type, scale, deterministic,
                seq_lens_q, seq_lens_kv, dropout_p, rng_state):
        kw = dict(causal=causal, window=window, softmax_type=softmax_type, scale=scale, seq_lens_q=seq_lens_q,
                  seq_lens_kv=seq_lens_kv, dropout_p=dropout_p, rng_state=rng_state)
        o, lse = sdpa_forward(q, k, v, softmax_offset=softmax_offset, bias=bias, **kw)
        ctx.save_for_backward(q, k, v, o, lse, softmax_offset, bias)
        ctx.kw = dict(kw, deterministic=deterministic)
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse, off, bias = ctx.saved_tensors
        res = sdpa_backward(q, k, v, o, dout.contiguous(), lse, softmax_offset=off, bias=bias, **ctx.kw)
        dq, dk, dv, d_off = res[:4]
        dbias = None
        if bias is not None and ctx.needs_input_grad[4]:
            dbias = res[4] if bias.dtype == torch.float32 else res[4].to(bias.dtype)  # autograd wants bias's dtype
        return dq, dk, dv, d_off, dbias, None, None, None, None, None, None, None, None, None


def new_rng_state(device=None):
    """A fresh dropout rng_state: a CUDA int64 [seed, offset] with a seed drawn from
    torch's default generator and offset 0."""
    seed = int(torch.randint(0, 2 ** 62, (1,)).item())
    return torch.tensor([seed, 0], dtype=torch.int64, device=device or "cuda")


def attention(q, k, v, softmax_offset=None, *, causal=True, window=-1, softmax_type=VANILLA, scale=0.0,
              deterministic=True, bias=None, seq_lens_q=None, seq_lens_kv=None, dropout_p=0.0, rng_state=None):
    """Differentiable fused attention. q, k, v, the learnable offset and the bias receive
    gradients. seq_lens_q / seq_lens_kv (int32 [B] on the device) make it a padded batch;
    dropout_p > 0 applies attention dropout with rng_state (a fresh one when None; the
    backward regenerates the same decisions from it)."""
    if dropout_p and rng_state is None:
        rng_state = new_rng_state(q.device)
    return SDPAFunction.apply(q, k, v, softmax_offset, bias, causal, window, softmax_type, scale, deterministic,
                              seq_lens_q, seq_lens_kv, dropout_p, rng_state)
