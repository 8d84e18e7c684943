"""CPU oracle for FP8 / BF16 causal prefill attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never does; the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over rows); this
module compiles it on demand with gcc and marshals numpy arrays.  Function
docstrings name the passage each definition follows:

* [ART-MTP] "Zyphra ZYFA: FP8 FlashAttention for AMD MI355X, Up to 1.76x Faster"
* [ART-EN]  "Breaking the FP8 Attention Bottleneck on AMD MI355X: How Zyphra
  ZYFA Unleashes Performance"

Every function here is pinned by ``tests/test_oracle_*.py`` against values
fixed by the articles, closed forms, library routines or brute force.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

#: default half-width of the rounding-ambiguity band, relative to
#: 8*lambda*sum_d|q_d k_d| (code units).  An fp32 accumulation of a 128- or
#: 192-term dot product is accurate to far better than this; the margin also
#: covers accumulators that keep fewer bits than binary32.
DEFAULT_KAPPA = 2.0 ** -14


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared",
           "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        u8 = ctypes.c_void_p
        i64p = ctypes.c_void_p
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint]
        lib.oracle_bf16_decode.restype = ctypes.c_double
        lib.oracle_bf16_decode.argtypes = [ctypes.c_uint]
        lib.oracle_e4m3_round.restype = ctypes.c_double
        lib.oracle_e4m3_round.argtypes = [ctypes.c_double]
        lib.oracle_bf16_round.restype = ctypes.c_double
        lib.oracle_bf16_round.argtypes = [ctypes.c_double]
        lib.oracle_leanp_code.restype = ctypes.c_int
        lib.oracle_leanp_code.argtypes = [ctypes.c_double]
        shape = [ctypes.c_int] * 6
        lib.oracle_ref_fp64.argtypes = [u8, u8, u8, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_double, *shape, ctypes.c_double, i64p,
                                        ctypes.c_int64, dp]
        lib.oracle_ref_fp64_bf16.argtypes = [u8, u8, u8, *shape, ctypes.c_double, i64p,
                                             ctypes.c_int64, dp]
        lib.oracle_emul_leanp.argtypes = [u8, u8, u8, ctypes.c_double, ctypes.c_double,
                                          ctypes.c_double, *shape, ctypes.c_double, i64p,
                                          ctypes.c_int64, ctypes.c_double, dp, dp]
        lib.oracle_emul_exact_fp8.argtypes = lib.oracle_emul_leanp.argtypes
        dp = ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        lib.oracle_ref_fp64_ex.argtypes = [vp, vp, vp, ctypes.c_int, dp, dp, dp, ctypes.c_int,
                                           ctypes.c_int, *shape, ctypes.c_double, i64p,
                                           ctypes.c_int64, dp, dp]
        lib.oracle_emul_leanp_ex.argtypes = [vp, vp, vp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                             *shape, ctypes.c_double, i64p, ctypes.c_int64,
                                             ctypes.c_double, dp, dp, dp]
        lib.oracle_emul_exact_ex.argtypes = [vp, vp, vp, ctypes.c_int, dp, dp, dp, ctypes.c_int,
                                             ctypes.c_int, *shape, ctypes.c_double, i64p,
                                             ctypes.c_int64, ctypes.c_double, dp, dp, dp]
        lib.oracle_emul_variant_e.argtypes = [vp, vp, vp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                              *shape, ctypes.c_double, i64p, ctypes.c_int64,
                                              ctypes.c_double, dp, dp, dp]
        lib.oracle_emul_leanp_a3.argtypes = lib.oracle_emul_variant_e.argtypes
        for fn in ("oracle_ref_fp64_ex", "oracle_emul_leanp_ex", "oracle_emul_exact_ex",
                   "oracle_emul_variant_e", "oracle_emul_leanp_a3"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.oracle_quantize_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.POINTER(ctypes.c_float)]
        lib.oracle_quantize_e4m3.restype = ctypes.c_int
        lib.oracle_emul_bf16.argtypes = [u8, u8, u8, *shape, ctypes.c_double, i64p,
                                         ctypes.c_int64, dp]
        for f in ("oracle_ref_fp64", "oracle_ref_fp64_bf16", "oracle_emul_leanp",
                  "oracle_emul_exact_fp8", "oracle_emul_bf16"):
            getattr(lib, f).restype = ctypes.c_int
        lib.oracle_leanp_C.restype = ctypes.c_int
        lib.oracle_leanp_T.restype = ctypes.c_int
        _lib = lib
        return lib


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Decode OCP E4M3 codes (uint8) to fp64, from the format's definition."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.oracle_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def bf16_decode(bits) -> np.ndarray:
    """Decode bfloat16 bit patterns (uint16) to fp64."""
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.vectorize(lambda x: lib.oracle_bf16_decode(int(x)), otypes=[np.float64])(b)


def e4m3_round(x) -> np.ndarray:
    """Round fp64 values to e4m3 (nearest, ties to even, saturating at 448)."""
    lib = _load()
    return np.vectorize(lambda t: lib.oracle_e4m3_round(float(t)), otypes=[np.float64])(
        np.asarray(x, dtype=np.float64))


def bf16_round(x) -> np.ndarray:
    """Round fp64 values to bfloat16 (nearest, ties to even)."""
    lib = _load()
    return np.vectorize(lambda t: lib.oracle_bf16_round(float(t)), otypes=[np.float64])(
        np.asarray(x, dtype=np.float64))


def leanp_code(x) -> np.ndarray:
    """Lean-P code of a code-unit argument: clamp(floor(x), 0, 126)."""
    lib = _load()
    return np.vectorize(lambda t: lib.oracle_leanp_code(float(t)), otypes=[np.int64])(
        np.asarray(x, dtype=np.float64))


def leanp_constants() -> tuple[int, int]:
    """(T, C): Lean-P headroom exponent and the e4m3 code of 2^T."""
    lib = _load()
    return lib.oracle_leanp_T(), lib.oracle_leanp_C()


# --------------------------------------------------------------------------
# attention definitions
# --------------------------------------------------------------------------

def _shape(q, k, v):
    B, S, Hq, Dqk = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    Bv, Sv, Hv, Dv = v.shape
    if (Bk, Sk, Dk) != (B, S, Dqk) or (Bv, Sv, Hv) != (B, S, Hkv) or Hq % Hkv:
        raise ValueError("inconsistent q/k/v shapes")
    return B, Hq, Hkv, S, Dqk, Dv


def _rows(rows, shape):
    B, Hq, Hkv, S, Dqk, Dv = shape
    if rows is None:
        return None, B * S * Hq
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    return r, r.shape[0]


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _finish(out, rows, shape):
    B, Hq, Hkv, S, Dqk, Dv = shape
    return out.reshape(B, S, Hq, Dv) if rows is None else out


def _scale(scale, Dqk):
    return 1.0 / math.sqrt(Dqk) if scale is None else float(scale)


def ref_fp64(q, k, v, dq, dk, dv, scale=None, rows=None):
    """fp64 causal attention on the dequantized e4m3 inputs.

    softmax(scale * (dq*Q)(dk*K)^T, causal) (dv*V), the quantity whose RMS error
    the article [ART-MTP] reports in "How accurate is ZYFA's FP8 attention?".
    ``q`` [B,S,Hq,Dqk], ``k`` [B,S,Hkv,Dqk], ``v`` [B,S,Hkv,Dv] are uint8 e4m3
    codes.  ``rows`` is an optional (n,3) array of (b, h, i); the result is then
    (n, Dv), else [B,S,Hq,Dv].
    """
    lib = _load()
    q, k, v = (np.ascontiguousarray(a, dtype=np.uint8) for a in (q, k, v))
    shape = _shape(q, k, v)
    r, n = _rows(rows, shape)
    out = np.empty((n, shape[5]), dtype=np.float64)
    rc = lib.oracle_ref_fp64(_ptr(q), _ptr(k), _ptr(v), float(dq), float(dk), float(dv), *shape,
                             _scale(scale, shape[4]), None if r is None else _ptr(r), n, _dptr(out))
    if rc:
        raise ValueError("oracle_ref_fp64: bad arguments")
    return _finish(out, r, shape)


def ref_fp64_bf16(q, k, v, scale=None, rows=None):
    """fp64 causal attention on bf16 inputs (``q``/``k``/``v`` are uint16 bits)."""
    lib = _load()
    q, k, v = (np.ascontiguousarray(a, dtype=np.uint16) for a in (q, k, v))
    shape = _shape(q, k, v)
    r, n = _rows(rows, shape)
    out = np.empty((n, shape[5]), dtype=np.float64)
    rc = lib.oracle_ref_fp64_bf16(_ptr(q), _ptr(k), _ptr(v), *shape, _scale(scale, shape[4]),
                                  None if r is None else _ptr(r), n, _dptr(out))
    if rc:
        raise ValueError("oracle_ref_fp64_bf16: bad arguments")
    return _finish(out, r, shape)


def emul_leanp(q, k, v, dq, dk, dv, scale=None, rows=None, kappa=DEFAULT_KAPPA):
    """Scalar emulation of the Lean-P / per-block scale / rounded row sum scheme.

    Follows [ART-MTP] "Lean P: one multiply-add instead of an exponential" and
    "Per-block scaling and a rounded row sum" (definition in oracle.c).
    Returns ``(out, amb)``: the fp64 output and, per row, the normalised weight
    mass that an fp32 evaluation may move across a rounding decision (0 when
    no decision is within the band ``kappa``).
    """
    lib = _load()
    q, k, v = (np.ascontiguousarray(a, dtype=np.uint8) for a in (q, k, v))
    shape = _shape(q, k, v)
    r, n = _rows(rows, shape)
    out = np.empty((n, shape[5]), dtype=np.float64)
    amb = np.empty((n,), dtype=np.float64)
    rc = lib.oracle_emul_leanp(_ptr(q), _ptr(k), _ptr(v), float(dq), float(dk), float(dv), *shape,
                               _scale(scale, shape[4]), None if r is None else _ptr(r), n,
                               float(kappa), _dptr(out), _dptr(amb))
    if rc:
        raise ValueError("oracle_emul_leanp: bad arguments")
    if r is None:
        return _finish(out, r, shape), amb.reshape(shape[0], shape[3], shape[1])
    return out, amb


def emul_exact_fp8(q, k, v, dq, dk, dv, scale=None, rows=None, kappa=DEFAULT_KAPPA):
    """Exact-softmax FP8 ablation: exact exp, e4m3-rounded P, unrounded row sum.

    The "hardware exponential" approach of [ART-MTP] "How does ZYFA compare
    with other attention kernels?", run with a running max per 128-key tile.
    Returns ``(out, amb)`` like :func:`emul_leanp`.
    """
    lib = _load()
    q, k, v = (np.ascontiguousarray(a, dtype=np.uint8) for a in (q, k, v))
    shape = _shape(q, k, v)
    r, n = _rows(rows, shape)
    out = np.empty((n, shape[5]), dtype=np.float64)
    amb = np.empty((n,), dtype=np.float64)
    rc = lib.oracle_emul_exact_fp8(_ptr(q), _ptr(k), _ptr(v), float(dq), float(dk), float(dv),
                                   *shape, _scale(scale, shape[4]), None if r is None else _ptr(r),
                                   n, float(kappa), _dptr(out), _dptr(amb))
    if rc:
        raise ValueError("oracle_emul_exact_fp8: bad arguments")
    if r is None:
        return _finish(out, r, shape), amb.reshape(shape[0], shape[3], shape[1])
    return out, amb


def emul_bf16(q, k, v, scale=None, rows=None):
    """Exact-softmax BF16 path: exact exp, bf16-rounded P, unrounded row sum."""
    lib = _load()
    q, k, v = (np.ascontiguousarray(a, dtype=np.uint16) for a in (q, k, v))
    shape = _shape(q, k, v)
    r, n = _rows(rows, shape)
    out = np.empty((n, shape[5]), dtype=np.float64)
    rc = lib.oracle_emul_bf16(_ptr(q), _ptr(k), _ptr(v), *shape, _scale(scale, shape[4]),
                              None if r is None else _ptr(r), n, _dptr(out))
    if rc:
        raise ValueError("oracle_emul_bf16: bad arguments")
    return _finish(out, r, shape)


def quantize_e4m3(x, rotate: bool):
    """Per-tensor e4m3 quantisation of Q or K, optionally after the Hadamard
    rotation of every head vector (definition in oracle.c; [ART-MTP] "How
    accurate is ZYFA's FP8 attention?").  ``x`` is float32, or uint16 bf16
    bits, with the head dimension last (128 or 192).  Returns ``(codes,
    descale)``: uint8 codes of x's shape and the fp32 descale."""
    lib = _load()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        is_f32 = 1
    elif x.dtype == np.uint16:
        is_f32 = 0
    else:
        raise TypeError("x must be float32 or uint16 bf16 bits")
    D = x.shape[-1]
    n_vec = x.size // D
    codes = np.empty(x.shape, dtype=np.uint8)
    ds = ctypes.c_float()
    rc = lib.oracle_quantize_e4m3(x.ctypes.data_as(ctypes.c_void_p), is_f32, n_vec, D, int(bool(rotate)),
                                  codes.ctypes.data_as(ctypes.c_void_p), ctypes.byref(ds))
    if rc:
        raise ValueError("oracle_quantize_e4m3: bad arguments")
    return codes, float(ds.value)


def _descales(dq, dk, dv, B, Hkv):
    """One value each, or [B, Hkv] arrays (per batch and kv head)."""
    arrs = [np.ascontiguousarray(np.asarray(d, dtype=np.float64).reshape(-1)) for d in (dq, dk, dv)]
    sizes = {a.size for a in arrs}
    if sizes == {1}:
        return arrs, 0
    if sizes == {B * Hkv}:
        return arrs, 1
    raise ValueError("descales must be scalars or [B, Hkv] arrays")


def attention(path, q, k, v, dq=1.0, dk=1.0, dv=1.0, scale=None, rows=None, causal=True,
              kappa=DEFAULT_KAPPA):
    """All definitions with every option (non-causal, per-(batch, kv head)
    descales) and the per-row log-sum-exp.  ``path`` is "ref" (fp64 on e4m3
    codes), "ref_bf16", "leanp", "exact_fp8", "bf16" or "variant_e" (the
    diagnostic: Lean-P's blocks and rounded sum with exact, RNE-rounded
    weights, the GPU's ATTN_VARIANT_BLOCK_EXACT).  Returns ``(out, amb,
    lse)``: out [B,S,Hq,Dv] or (n, Dv) for ``rows``; amb per row (None for the
    reference and BF16 paths); lse per row, natural log of the row sum (the
    unnormalised weights of that path), shaped [B,Hq,S] or (n,)."""
    lib = _load()
    bf16 = path in ("ref_bf16", "bf16")
    dt = np.uint16 if bf16 else np.uint8
    q, k, v = (np.ascontiguousarray(a, dtype=dt) for a in (q, k, v))
    shape = _shape(q, k, v)
    B, Hq, Hkv = shape[0], shape[1], shape[2]
    (aq, ak, av), per = _descales(dq, dk, dv, B, Hkv)
    r, n = _rows(rows, shape)
    out = np.empty((n, shape[5]), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    amb = None if path in ("ref", "ref_bf16", "bf16") else np.empty((n,), dtype=np.float64)
    rp = None if r is None else _ptr(r)
    args = (_dptr(aq), _dptr(ak), _dptr(av), per, int(bool(causal)), *shape,
            _scale(scale, shape[4]), rp, n)
    if path in ("ref", "ref_bf16"):
        rc = lib.oracle_ref_fp64_ex(_ptr(q), _ptr(k), _ptr(v), int(bf16), *args, _dptr(out), _dptr(lse))
    elif path == "leanp":
        rc = lib.oracle_emul_leanp_ex(_ptr(q), _ptr(k), _ptr(v), *args, float(kappa), _dptr(out),
                                      _dptr(amb), _dptr(lse))
    elif path == "leanp_a3":
        rc = lib.oracle_emul_leanp_a3(_ptr(q), _ptr(k), _ptr(v), *args, float(kappa), _dptr(out),
                                      _dptr(amb), _dptr(lse))
    elif path == "variant_e":
        rc = lib.oracle_emul_variant_e(_ptr(q), _ptr(k), _ptr(v), *args, float(kappa), _dptr(out),
                                       _dptr(amb), _dptr(lse))
    elif path in ("exact_fp8", "bf16"):
        rc = lib.oracle_emul_exact_ex(_ptr(q), _ptr(k), _ptr(v), int(bf16), *args, float(kappa),
                                      _dptr(out), None if amb is None else _dptr(amb), _dptr(lse))
    else:
        raise ValueError(path)
    if rc:
        raise ValueError(f"oracle {path}: bad arguments")
    if r is None:
        out = out.reshape(B, shape[3], Hq, shape[5])
        lse = lse.reshape(B, shape[3], Hq).transpose(0, 2, 1).copy()
        if amb is not None:
            amb = amb.reshape(B, shape[3], Hq)
    return out, amb, lse
