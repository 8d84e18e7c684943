"""GB300-native FP8 / BF16 causal prefill FlashAttention.

A thin binding over the C ABI of ``libfp8attn.so`` (``include/fp8attn.h``).
It only marshals torch tensors into pointers, sizes and the current CUDA
stream: every step of the computation runs in the library's sm_103a kernels.
If the library has not been built the calls raise; there is no CPU path.

Entry points (same names as the C ABI):

* ``attn_fwd_fp8(q, k, v, descale_q, descale_k, descale_v)`` -- Lean-P
* ``attn_fwd_fp8_exact(...)`` -- exact-softmax FP8 ablation
* ``attn_fwd_bf16(q, k, v)`` -- exact-softmax BF16
* ``attn_fwd_ex(variant, ...)`` -- fp32 output, explicit scale, status word
* ``attn_fwd_full(variant, ...)`` -- plus non-causal, per-(batch, kv head)
  descales, LSE, and the split schedule for problems with few work items
  (its workspace comes from torch's caching allocator on the call's stream)

Tensors are [B, S, H, D] contiguous CUDA tensors: uint8 / float8_e4m3fn codes
for FP8 (descales are one-element float32 CUDA tensors), bfloat16 for BF16.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import numpy as np
import torch

from . import _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ARCH = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5

ATTN_VARIANT_LEANP = 0
ATTN_VARIANT_EXACT_FP8 = 1
ATTN_VARIANT_BF16 = 2
ATTN_VARIANT_BLOCK_EXACT = 3  # diagnostic: Lean-P block scale + rounded sum, exact e4m3-rounded p
ATTN_VARIANT_LEANP_A3 = 4  # Lean-P with the code grid anchored at the running row maximum
ATTN_OUT_BF16 = 0
ATTN_OUT_F32 = 1
ATTN_FLAG_TEST_STALL_LOADS = 1
ATTN_FLAG_DESCALE_PER_BKV = 2
ATTN_FLAG_TEST_CHUNK_UNITS = 4
ATTN_IN_BF16 = 0
ATTN_IN_F32 = 1

HEADER = os.path.join(_build.ROOT, "include", "fp8attn.h")
LIBRARY_PATH = _build.SO

_lib = None
_lib_tl = None
_TIMELINE = os.environ.get("FP8ATTN_TIMELINE") == "1"
_lock = threading.Lock()


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def build(force: bool = False, timeline: bool = False) -> str:
    """Compile libfp8attn.so in-tree (nvcc, sm_103a); ``timeline`` builds the
    debug library libfp8attn_timeline.so instead."""
    return _build.build(force=force, timeline=timeline)


def _open(path):
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fp8_args = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.attn_fwd_fp8.argtypes = fp8_args
    lib.attn_fwd_fp8_exact.argtypes = fp8_args
    lib.attn_fwd_bf16.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.attn_fwd_ex.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i,
                                vp, vp]
    lib.attn_quantize_fp8.argtypes = [vp, i, vp, vp, i, i, i, i, i, vp]
    lib.attn_fwd_full.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, f,
                                  i, vp, vp, sz, vp]
    lib.attn_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i, ctypes.POINTER(sz)]
    lib.attn_split_plan.argtypes = [i, i, i, i, i, i, i, i, i, i, ctypes.POINTER(i),
                                    ctypes.POINTER(i), ctypes.POINTER(sz)]
    lib.attn_debug_timeline.argtypes = [vp, i, i]
    for name in ("attn_fwd_fp8", "attn_fwd_fp8_exact", "attn_fwd_bf16", "attn_fwd_ex",
                 "attn_quantize_fp8", "attn_fwd_full", "attn_launches_per_call",
                 "attn_api_version", "attn_debug_timeline", "attn_workspace_size",
                 "attn_split_plan"):
        getattr(lib, name).restype = ctypes.c_int
    lib.attn_status_string.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    return lib


def load_library():
    """Load libfp8attn.so; raise if it has not been built.  With the
    environment variable FP8ATTN_TIMELINE=1 (read when the package is
    imported) every call goes to the debug library with the role timeline
    instead (see debug_timeline)."""
    global _lib
    if _lib is not None:
        return _lib
    if _TIMELINE:
        return load_timeline_library()
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIBRARY_PATH):
            raise RuntimeError(
                f"{LIBRARY_PATH} is missing: build it with fp8_causal_prefill_flash_gb300.build()")
        _lib = _open(LIBRARY_PATH)
        return _lib


def load_timeline_library():
    """Build (if needed) and load the debug library whose kernels record the
    clock64 role timeline; its entry points are called through ctypes like
    the release library's (the Python functions here use the release one)."""
    global _lib_tl
    with _lock:
        if _lib_tl is None:
            _lib_tl = _open(_build.build(timeline=True))
        return _lib_tl


def debug_timeline(lib, reset: bool = True) -> np.ndarray:
    """The role timeline of the last call made through ``lib`` (the debug
    library): uint64 clock64 stamps [6, 64, 8], layout as in fp8attn.h."""
    buf = np.zeros((6, 64, 8), dtype=np.uint64)
    st = lib.attn_debug_timeline(buf.ctypes.data, buf.size, int(bool(reset)))
    _raise(st, "attn_debug_timeline")
    return buf


def declared_functions() -> list[str]:
    """Names of the functions include/fp8attn.h declares."""
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(attn_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else t.data_ptr()


# torch's raw current-stream query (no Stream object); the public API otherwise
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(t=None):
    """The current CUDA stream as a plain integer handle.  The library launches
    on the current device, so t (the call's first tensor) must live there."""
    dev = torch.cuda.current_device()
    if t is not None and t.get_device() != dev:
        raise ValueError(f"tensors are on cuda:{t.get_device()} but the current device is "
                         f"cuda:{dev}; call inside torch.cuda.device({t.get_device()})")
    if _raw_stream is not None:
        return _raw_stream(dev)
    return torch.cuda.current_stream().cuda_stream


def _check_qkv(q, k, v, fp8: bool):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, S, H, D] tensor")
        if fp8 and t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError(f"{name} must hold e4m3 codes (uint8 or float8_e4m3fn)")
        if not fp8 and t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
    B, S, Hq, Dqk = q.shape
    _, _, Hkv, _ = k.shape
    Dv = v.shape[3]
    return B, Hq, Hkv, S, Dqk, Dv


def _check_descale(name, t):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 or t.numel() < 1:
        raise TypeError(f"{name} must be a float32 CUDA tensor with one element")


def _out(out, q, Dv, dtype):
    B, S, Hq, _ = q.shape
    if out is None:
        return torch.empty((B, S, Hq, Dv), dtype=dtype, device=q.device)
    if out.shape != (B, S, Hq, Dv) or out.dtype != dtype or not out.is_contiguous():
        raise ValueError("out has the wrong shape, dtype or layout")
    return out


def _raise(status, what):
    if status != ATTN_OK:
        raise AttnError(status, what)


def attn_fwd_fp8(q, k, v, descale_q, descale_k, descale_v, out=None, causal=True):
    """Lean-P FP8 causal prefill attention; returns bf16 [B, S, Hq, Dv]."""
    lib = load_library()
    B, Hq, Hkv, S, Dqk, Dv = _check_qkv(q, k, v, True)
    for n, t in (("descale_q", descale_q), ("descale_k", descale_k), ("descale_v", descale_v)):
        _check_descale(n, t)
    out = _out(out, q, Dv, torch.bfloat16)
    st = lib.attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(descale_q), _ptr(descale_k),
                          _ptr(descale_v), _ptr(out), B, Hq, Hkv, S, Dqk, Dv, int(bool(causal)),
                          _stream_handle(q))
    _raise(st, "attn_fwd_fp8")
    return out


def attn_fwd_fp8_exact(q, k, v, descale_q, descale_k, descale_v, out=None, causal=True):
    """Exact-softmax FP8 ablation; returns bf16 [B, S, Hq, Dv]."""
    lib = load_library()
    B, Hq, Hkv, S, Dqk, Dv = _check_qkv(q, k, v, True)
    for n, t in (("descale_q", descale_q), ("descale_k", descale_k), ("descale_v", descale_v)):
        _check_descale(n, t)
    out = _out(out, q, Dv, torch.bfloat16)
    st = lib.attn_fwd_fp8_exact(_ptr(q), _ptr(k), _ptr(v), _ptr(descale_q), _ptr(descale_k),
                                _ptr(descale_v), _ptr(out), B, Hq, Hkv, S, Dqk, Dv,
                                int(bool(causal)), _stream_handle(q))
    _raise(st, "attn_fwd_fp8_exact")
    return out


def attn_fwd_bf16(q, k, v, out=None, causal=True):
    """Exact-softmax BF16 causal prefill attention; returns bf16 [B, S, Hq, Dv]."""
    lib = load_library()
    B, Hq, Hkv, S, Dqk, Dv = _check_qkv(q, k, v, False)
    out = _out(out, q, Dv, torch.bfloat16)
    st = lib.attn_fwd_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, S, Dqk, Dv,
                           int(bool(causal)), _stream_handle(q))
    _raise(st, "attn_fwd_bf16")
    return out


def attn_fwd_ex(variant, q, k, v, descale_q=None, descale_k=None, descale_v=None, out=None,
                out_dtype=ATTN_OUT_F32, softmax_scale=0.0, flags=0, dev_status=None,
                causal=True, raise_on_error=True):
    """Extended call: any variant, fp32 or bf16 output, explicit softmax scale,
    test flags and an optional int32 CUDA status tensor (zeroed by the caller)."""
    lib = load_library()
    fp8 = variant != ATTN_VARIANT_BF16
    B, Hq, Hkv, S, Dqk, Dv = _check_qkv(q, k, v, fp8)
    if fp8:
        for n, t in (("descale_q", descale_q), ("descale_k", descale_k), ("descale_v", descale_v)):
            _check_descale(n, t)
    dtype = torch.float32 if out_dtype == ATTN_OUT_F32 else torch.bfloat16
    out = _out(out, q, Dv, dtype)
    st = lib.attn_fwd_ex(int(variant), _ptr(q), _ptr(k), _ptr(v), _ptr(descale_q),
                         _ptr(descale_k), _ptr(descale_v), _ptr(out), int(out_dtype), B, Hq, Hkv,
                         S, Dqk, Dv, int(bool(causal)), float(softmax_scale), int(flags),
                         _ptr(dev_status), _stream_handle(q))
    if raise_on_error:
        _raise(st, "attn_fwd_ex")
        return out
    return out, st


def attn_quantize_fp8(x, hadamard=False, codes=None, descale=None):
    """Per-tensor e4m3 quantisation of Q or K (``attn_quantize_fp8`` of the C
    ABI), optionally after the Hadamard rotation of every head vector; rotate
    Q and K alike.  ``x`` is a CUDA bf16 or fp32 tensor [B, S, H, D], D in
    {128, 192}.  Returns ``(codes, descale)``: uint8 e4m3 codes of x's shape and
    a one-element fp32 tensor, ready for :func:`attn_fwd_fp8`."""
    lib = load_library()
    if not x.is_cuda or x.dim() != 4 or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor [B, S, H, D]")
    if x.dtype == torch.bfloat16:
        in_dtype = ATTN_IN_BF16
    elif x.dtype == torch.float32:
        in_dtype = ATTN_IN_F32
    else:
        raise ValueError("x must be bfloat16 or float32")
    B, S, H, D = x.shape
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if descale is None:
        descale = torch.empty(1, dtype=torch.float32, device=x.device)
    if codes.shape != x.shape or codes.dtype != torch.uint8 or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 tensor of x's shape")
    if descale.dtype != torch.float32 or descale.numel() != 1:
        raise ValueError("descale must be a one-element float32 tensor")
    st = lib.attn_quantize_fp8(_ptr(x), in_dtype, _ptr(codes), _ptr(descale), B, S, H, D,
                               int(bool(hadamard)), _stream_handle(x))
    _raise(st, "attn_quantize_fp8")
    return codes, descale


def workspace_size(variant, B, Hq, Hkv, S, Dqk, Dv, causal=True, flags=0) -> int:
    """Bytes of workspace ``attn_fwd_full`` uses on the current device for
    these arguments (``attn_workspace_size`` of the C ABI): 0 unless the
    problem has too few work items to fill the SMs and the variant splits
    (Lean-P, block-exact and BF16)."""
    n = ctypes.c_size_t(0)
    st = load_library().attn_workspace_size(int(variant), B, Hq, Hkv, S, Dqk, Dv,
                                            int(bool(causal)), int(flags), ctypes.byref(n))
    _raise(st, "attn_workspace_size")
    return int(n.value)


def split_plan(variant, B, Hq, Hkv, S, Dqk, Dv, causal, sms, flags=0):
    """The split schedule ``attn_fwd_full`` would choose on a GPU with ``sms``
    SMs (``attn_split_plan`` of the C ABI; host only, no device needed):
    ``(split_qb, ns, bytes)``, ``(0, 1, 0)`` when the problem runs whole
    items."""
    qb, ns, n = ctypes.c_int(0), ctypes.c_int(1), ctypes.c_size_t(0)
    st = load_library().attn_split_plan(int(variant), B, Hq, Hkv, S, Dqk, Dv, int(bool(causal)),
                                        int(flags), int(sms), ctypes.byref(qb), ctypes.byref(ns),
                                        ctypes.byref(n))
    _raise(st, "attn_split_plan")
    return qb.value, ns.value, n.value


def attn_fwd_full(variant, q, k, v, descale_q=None, descale_k=None, descale_v=None, out=None,
                  out_dtype=ATTN_OUT_BF16, causal=True, softmax_scale=None, return_lse=False,
                  dev_status=None, flags=0, split=True, workspace=None):
    """The general entry point (``attn_fwd_full`` of the C ABI).  Descales are
    one-element tensors or [B, Hkv] tensors (one per batch and kv head).
    With ``split`` (the default) a problem with too few work items to fill
    the SMs splits its longest items along the keys; the workspace this needs
    is ``workspace`` (a uint8 CUDA tensor of at least ``workspace_size``
    bytes, used by one call at a time) or, by default, a new tensor from
    torch's caching allocator, which keeps it for this call's stream until the
    call's work is done.  ``split=False`` runs every item whole.
    Returns ``out``, or ``(out, lse)`` with lse fp32 [B, Hq, S] (natural log of
    the row's own unnormalised weights)."""
    lib = load_library()
    fp8 = variant != ATTN_VARIANT_BF16
    B, Hq, Hkv, S, Dqk, Dv = _check_qkv(q, k, v, fp8)
    if fp8:
        sizes = {int(t.numel()) for t in (descale_q, descale_k, descale_v)}
        if sizes == {B * Hkv} and B * Hkv != 1:
            flags |= ATTN_FLAG_DESCALE_PER_BKV
        elif sizes != {1}:
            raise ValueError("descales must be one-element or [B, Hkv] float32 tensors")
        for name, t in (("descale_q", descale_q), ("descale_k", descale_k), ("descale_v", descale_v)):
            if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    dtype = torch.float32 if out_dtype == ATTN_OUT_F32 else torch.bfloat16
    out = _out(out, q, Dv, dtype)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device) if return_lse else None
    stream = _stream_handle(q)
    ws, ws_bytes = None, 0
    if split:
        need = workspace_size(variant, B, Hq, Hkv, S, Dqk, Dv, causal, flags)
        if need:
            if workspace is None:
                workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            elif (not workspace.is_cuda or workspace.dtype != torch.uint8 or
                  workspace.numel() < need or not workspace.is_contiguous()):
                raise ValueError(f"workspace must be a contiguous uint8 CUDA tensor of at least "
                                 f"{need} bytes")
            ws, ws_bytes = workspace, int(workspace.numel())
    st = lib.attn_fwd_full(variant, _ptr(q), _ptr(k), _ptr(v), _ptr(descale_q), _ptr(descale_k),
                           _ptr(descale_v), _ptr(out), out_dtype, _ptr(lse), B, Hq, Hkv, S, Dqk,
                           Dv, int(bool(causal)), float(softmax_scale or 0.0), flags,
                           _ptr(dev_status), _ptr(ws), ws_bytes, stream)
    _raise(st, "attn_fwd_full")
    return (out, lse) if return_lse else out


def host_descale(name, x):
    """A descale given as a host number: it must be finite and greater than
    zero (the library's contract; device descales cannot be checked without
    a synchronisation).  Returns it as a float."""
    try:
        f = float(x)
    except (TypeError, ValueError):
        raise TypeError(f"{name} must be a number or a float32 CUDA tensor") from None
    if not (f > 0.0 and f != float("inf")):
        raise ValueError(f"{name} must be finite and greater than zero, got {x!r}")
    return f


def flash_attn_fp8_func(q, k, v, q_descale=None, k_descale=None, v_descale=None,
                        softmax_scale=None, causal=True, return_softmax_lse=False, exact=False):
    """flash_attn_func-style call on e4m3 inputs (uint8 codes, BSHD): the
    Lean-P path, or the exact-softmax ablation with ``exact=True``.
    Descales default to 1; each may be a one-element or [B, Hkv] float32 CUDA
    tensor, or a host number (checked: finite and greater than zero)."""
    def dev(name, x):
        if x is None:
            x = 1.0
        if isinstance(x, torch.Tensor):
            return x
        return torch.tensor([host_descale(name, x)], dtype=torch.float32, device=q.device)
    return attn_fwd_full(ATTN_VARIANT_EXACT_FP8 if exact else ATTN_VARIANT_LEANP, q, k, v,
                         dev("q_descale", q_descale), dev("k_descale", k_descale),
                         dev("v_descale", v_descale), causal=causal, softmax_scale=softmax_scale,
                         return_lse=return_softmax_lse)


def flash_attn_fp8_from_bf16(q, k, v, hadamard=True, softmax_scale=None, causal=True,
                             return_softmax_lse=False):
    """Lean-P attention on bf16 (or fp32) activations: Q and K are quantised
    per tensor to e4m3, after the Hadamard rotation when ``hadamard`` is set
    (it leaves Q K^T unchanged and spreads outlier channels, "Zyphra ZYFA: FP8
    FlashAttention for AMD MI355X", "How accurate is ZYFA's FP8 attention?"),
    V is quantised as it is, and the three codes and descales go to the
    Lean-P kernel.  Four library calls on the current stream; the codes are
    new tensors."""
    cq, dq = attn_quantize_fp8(q, hadamard=hadamard)
    ck, dk = attn_quantize_fp8(k, hadamard=hadamard)
    cv, dv = attn_quantize_fp8(v, hadamard=False)
    return flash_attn_fp8_func(cq, ck, cv, dq, dk, dv, softmax_scale=softmax_scale, causal=causal,
                               return_softmax_lse=return_softmax_lse)


def flash_attn_bf16_func(q, k, v, softmax_scale=None, causal=True, return_softmax_lse=False):
    """flash_attn_func-style call on bf16 inputs (exact softmax)."""
    return attn_fwd_full(ATTN_VARIANT_BF16, q, k, v, causal=causal, softmax_scale=softmax_scale,
                         return_lse=return_softmax_lse)
