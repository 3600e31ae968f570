"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports every
function include/sdpa_tmem.h declares, and rejects bad arguments with the documented
status codes before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa_tmem.h")


@pytest.fixture(scope="module")
def lib():
    from scaled_dot_product_tmem_gb300 import build
    build.build()
    import scaled_dot_product_tmem_gb300 as sdpa
    return sdpa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_status_string", "attn_last_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} is declared in sdpa_tmem.h but not exported"


def test_status_strings(lib):
    import scaled_dot_product_tmem_gb300 as sdpa
    for st in range(7):
        assert sdpa.attn_status_string(st) not in ("", "unknown status")
    assert sdpa.attn_status_string(99) == "unknown status"


OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA, TIMEOUT, WORKSPACE = range(7)
P = ctypes.c_void_p(0x10000)   # a fake, 16-byte aligned "device" address (never dereferenced)
MIS = ctypes.c_void_p(0x10008)


def fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, Sq=64, Skv=64, Hq=4, Hkv=2, dqk=128, dv=128, scale=0.0,
        causal=1, window=-1, st=0, off=None):
    return lib.attn_fwd(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, dqk, dv, ctypes.c_float(scale), causal, window, st,
                        off, None)


def test_fwd_argument_validation(lib):
    assert fwd(lib, Hq=3, Hkv=2) == INVALID
    assert fwd(lib, Hkv=0) == INVALID
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, st=3) == INVALID
    assert fwd(lib, st=2, off=None) == INVALID          # learnable needs the offset
    assert fwd(lib, dqk=96) == UNSUPPORTED
    assert fwd(lib, dv=192) == UNSUPPORTED
    assert fwd(lib, causal=0, window=8) == UNSUPPORTED  # window only with causal
    assert fwd(lib, B=70000) == UNSUPPORTED
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, q=MIS) == MISALIGNED
    assert fwd(lib, o=MIS) == MISALIGNED
    assert fwd(lib, B=0) == OK                          # empty: nothing to launch
    assert fwd(lib, Sq=0) == OK


def test_bwd_workspace_and_validation(lib):
    import scaled_dot_product_tmem_gb300 as sdpa
    det = sdpa.attn_bwd_workspace_size(4, 2048, 2048, 32, 8, 128, 128, True)
    atom = sdpa.attn_bwd_workspace_size(4, 2048, 2048, 32, 8, 128, 128, False)
    rows = 4 * 32 * 2048
    assert det == 2 * rows * 4 + 256                    # lse2 + D (fp32), tile counters
    assert atom == det + 4 * 2048 * 32 * 128 * 4        # + fp32 dQ accumulator
    # B=1, S=100, H_kv=2: 2 kv CTAs, so the 2 query heads of each group go to 2 CTAs
    # and the workspace adds 2 fp32 partial slices of dK and dV
    part = 2 * 1 * 100 * 2 * 64 * 4
    assert sdpa.attn_bwd_workspace_size(1, 100, 100, 4, 2, 64, 64, True) == 2 * 4 * 128 * 4 + 2 * part + 256
    # MQA at 32,768 tokens: 256 kv CTAs (under 3 per SM) -> 4 splits, 1024 CTAs
    mqa = sdpa.attn_bwd_workspace_size(4, 8192, 8192, 32, 1, 128, 128, True)
    assert mqa == 2 * 4 * 32 * 8192 * 4 + 2 * 4 * (4 * 8192 * 1 * 128 * 4) + 256
    # GQA B=4 S=2048 H_kv=8: 512 CTAs, no split (checked above: det has no partials)
    # MHA has no head loop to split
    assert sdpa.attn_bwd_workspace_size(1, 100, 100, 4, 4, 64, 64, True) == 2 * 4 * 128 * 4 + 256
    assert sdpa.attn_bwd_workspace_size(1, 100, 100, 4, 3, 64, 64, True) == 0

    def bwd(ws=P, ws_bytes=1 << 30, q=P, Hq=4, Hkv=2, st=0, doff=None, off=None, window=-1, causal=1):
        return lib.attn_bwd(q, P, P, P, P, P, P, P, P, doff, 1, 64, 64, Hq, Hkv, 128, 128, ctypes.c_float(0.0),
                            causal, window, st, off, 1, ws, ctypes.c_size_t(ws_bytes), None)

    assert bwd(Hq=5) == INVALID
    assert bwd(st=2, off=P, doff=None) == INVALID       # learnable needs d_offset
    assert bwd(causal=0, window=3) == UNSUPPORTED
    assert bwd(q=MIS) == MISALIGNED
    assert bwd(ws=None) == WORKSPACE
    assert bwd(ws_bytes=16) == WORKSPACE
    assert bwd(ws=ctypes.c_void_p(0x10010)) == WORKSPACE  # needs 256-byte alignment


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import scaled_dot_product_tmem_gb300 as sdpa
    monkeypatch.setattr(sdpa, "_lib", None)
    monkeypatch.setattr(sdpa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        sdpa.library()


def test_fp8_argument_validation(lib):
    assert lib.attn_fp8_vt_row_bytes(1) == 16 and lib.attn_fp8_vt_row_bytes(16) == 16
    assert lib.attn_fp8_vt_row_bytes(2049) == 2064 and lib.attn_fp8_vt_row_bytes(0) == 0

    def f8(q=P, k=P, vt=P, dq=P, dk=P, dv=P, o=P, lse=P, B=1, Sq=64, Skv=64, Hq=4, Hkv=2, d=128, causal=1,
           window=-1, st=0, off=None):
        return lib.attn_fwd_fp8(q, k, vt, dq, dk, dv, o, lse, B, Sq, Skv, Hq, Hkv, d, ctypes.c_float(0.0), causal,
                                window, st, off, None)

    assert f8(d=96) == UNSUPPORTED                      # E4M3 head dims: 64 and 128
    assert f8(d=192) == UNSUPPORTED
    assert f8(Hq=3) == INVALID
    assert f8(dq=None) == INVALID                       # descales are required
    assert f8(vt=MIS) == MISALIGNED
    assert f8(dv=ctypes.c_void_p(0x10002)) == MISALIGNED
    assert f8(B=0) == OK and f8(Sq=0) == OK             # nothing to launch

    def qz(x=P, x8=P, B=1, S=64, H=2, d=128, t=0, amax=P, desc=P, aout=None):
        return lib.attn_fp8_quantize(x, x8, B, S, H, d, t, amax, desc, aout, None)

    assert qz(d=96, t=1) == UNSUPPORTED                 # the transposed form: d = 64 or 128
    assert qz(d=12) == INVALID                          # rows of whole 16-byte chunks
    assert qz(amax=None) == INVALID
    assert qz(x8=MIS) == MISALIGNED
    assert qz(B=0) == OK
    assert qz(aout=P) == INVALID                        # amax_out may not alias amax
    assert qz(aout=ctypes.c_void_p(0x10022)) == MISALIGNED
    assert lib.attn_fp8_amax(P, ctypes.c_size_t(8), None, None) == INVALID
    assert lib.attn_fp8_amax(MIS, ctypes.c_size_t(8), P, None) == MISALIGNED


def test_bias_argument_validation(lib):
    def fb(bias=P, Bb=1, Hb=4, B=2, Hq=4, Hkv=2, d=128, dv=None):
        return lib.attn_fwd_bias(P, P, P, P, P, bias, Bb, Hb, B, 64, 64, Hq, Hkv, d, d if dv is None else dv,
                                 ctypes.c_float(0.0), 1, -1, 0, None, None)

    assert fb(bias=None) == INVALID
    assert fb(Bb=3) == INVALID and fb(Hb=2) == INVALID   # broadcast dims are 1 or the full size
    assert fb(d=128, dv=64) == UNSUPPORTED               # bias kernels: (64, 64), (128, 128), (192, 128)
    assert fb(d=192, dv=64) == UNSUPPORTED
    assert fb(bias=MIS) == MISALIGNED
    assert fb(B=0, Bb=1) == OK

    def bb(Bb=1, Hb=4, dbias=P, det=1, bias=P):
        return lib.attn_bwd_bias(P, P, P, P, P, P, P, P, P, None, bias, Bb, Hb, dbias, 2, 64, 64, 4, 2, 128, 128,
                                 ctypes.c_float(0.0), 1, -1, 0, None, det, P, ctypes.c_size_t(1 << 30), None)

    assert bb() == UNSUPPORTED                           # broadcast dbias is summed with atomics
    assert bb(Bb=2, Hb=4, dbias=ctypes.c_void_p(0x10002)) == MISALIGNED
    assert bb(bias=None) == INVALID


def test_binding_has_every_boundary_name():
    """The Python binding exposes each C-ABI function under the same name."""
    import scaled_dot_product_tmem_gb300 as sdpa
    for n in declared_functions():
        assert callable(getattr(sdpa, n, None)), f"{n} has no binding of the same name"


def test_dropout_argument_validation(lib):
    """attn_fwd_dropout / attn_bwd_dropout reject a probability outside [0, 1) (or one
    that rounds to t = 65536), a missing rng_state and a misaligned one, before any
    device work."""
    f = ctypes.c_float
    MIS4 = ctypes.c_void_p(0x10004)

    def fwd_d(p, rng):
        return lib.attn_fwd_dropout(P, P, P, P, P, 1, 64, 64, 4, 2, 128, 128, f(0.0), 1, -1, 0, None, f(p), rng, None)

    def bwd_d(p, rng):
        return lib.attn_bwd_dropout(P, P, P, P, P, P, P, P, P, None, 1, 64, 64, 4, 2, 128, 128, f(0.0), 1, -1, 0,
                                    None, f(p), rng, 1, P, 1 << 20, None)

    for call in (fwd_d, bwd_d):
        assert call(-0.1, P) == INVALID
        assert call(1.0, P) == INVALID
        assert call(float("nan"), P) == INVALID
        assert call(1.0 - 2.0 ** -18, P) == INVALID   # rounds to t = 65536: everything dropped
        assert call(0.1, None) == INVALID             # a drop probability needs the rng state
        assert call(0.1, MIS4) == MISALIGNED


def test_fp8_backward_argument_validation(lib):
    """attn_bwd_fp8 and attn_fp8_quantize_e5m2 reject bad arguments before any device
    work; the workspace is two fp32 rows per (b, h) of S_q rounded up to 128."""
    lib.attn_bwd_fp8_workspace_size.restype = ctypes.c_size_t
    assert lib.attn_bwd_fp8_workspace_size(2, 100, 4) == 2 * 2 * 4 * 128 * 4
    assert lib.attn_bwd_fp8_workspace_size(1, 1, 1) == 2 * 512
    assert lib.attn_bwd_fp8_workspace_size(-1, 1, 1) == 0

    def b8(q=P, dsq=P, dsa=P, dsout=None, doff=None, B=1, Sq=64, Skv=64, Hq=4, Hkv=2, d=128, st=0, off=None,
           ws=P, wsb=1 << 20):
        return lib.attn_bwd_fp8(q, P, P, P, P, P, P, dsq, P, P, P, P, P, dsa, dsout, P, P, P, doff, B, Sq, Skv, Hq,
                                Hkv, d, ctypes.c_float(0.0), 1, -1, st, off, ws, ctypes.c_size_t(wsb), None)

    assert b8(d=96) == UNSUPPORTED and b8(d=192) == UNSUPPORTED   # d = 64 or 128
    assert b8(Hq=3) == INVALID
    assert b8(dsq=None) == INVALID                      # descales are required
    assert b8(dsa=None) == INVALID                      # so is the dS scaling statistic
    assert b8(dsout=P) == INVALID                       # ds_amax_out may not alias ds_amax
    assert b8(dsout=ctypes.c_void_p(0x10022)) == MISALIGNED
    assert b8(st=2, off=P, doff=None) == INVALID        # learnable sinks need d_offset
    assert b8(q=MIS) == MISALIGNED
    assert b8(q=None) == INVALID
    assert b8(B=0) == OK                                # nothing to launch

    def qz(x=P, x8=P, B=1, S=64, H=2, d=128, t=0, amax=P, desc=P, aout=None):
        return lib.attn_fp8_quantize_e5m2(x, x8, B, S, H, d, t, amax, desc, aout, None)

    assert qz(d=96, t=1) == UNSUPPORTED
    assert qz(d=12) == INVALID
    assert qz(desc=None) == INVALID
    assert qz(x=MIS) == MISALIGNED
    assert qz(B=0) == OK


def test_fp8_quantize_both_argument_validation(lib):
    """attn_fp8_quantize_both needs two distinct outputs and the transposed layout's head
    dims (64 or 128)."""
    Q = ctypes.c_void_p(0x20000)

    def qb(x=P, x8=P, x8t=Q, B=1, S=64, H=2, d=128, e5=0, amax=P, desc=ctypes.c_void_p(0x30000)):
        return lib.attn_fp8_quantize_both(x, x8, x8t, B, S, H, d, e5, amax, desc, None, None)

    assert qb(x8t=P) == INVALID                         # the two layouts may not share a buffer
    assert qb(x8=None) == INVALID
    assert qb(d=96) == UNSUPPORTED
    assert qb(x8=MIS) == MISALIGNED
    assert qb(B=0) == OK
