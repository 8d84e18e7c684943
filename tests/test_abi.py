"""CPU checks of the C-ABI boundary: the library builds for sm_103a, loads,
exports every function include/fp8attn.h declares, and rejects bad arguments
before touching any device (so these run without a GPU)."""
import ctypes

import pytest

import fp8_causal_prefill_flash_gb300 as fa


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load_library()


def test_header_declares_the_entry_points():
    names = fa.declared_functions()
    for n in ("attn_fwd_fp8", "attn_fwd_fp8_exact", "attn_fwd_bf16", "attn_fwd_ex",
              "attn_quantize_fp8", "attn_fwd_full", "attn_status_string",
              "attn_launches_per_call", "attn_api_version", "attn_debug_timeline",
              "attn_workspace_size", "attn_split_plan"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in fa.declared_functions():
        assert hasattr(lib, n), n
    assert lib.attn_api_version() == 9
    assert lib.attn_launches_per_call() == 1


def test_status_strings(lib):
    for st in range(6):
        assert fa.status_string(st)
    assert fa.status_string(99) == "unknown status"


P = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
MIS = ctypes.c_void_p(0x10001)    # misaligned


def call_ex(lib, variant=0, q=P, k=P, v=P, dq=P, dk=P, dv=P, out=P, out_dtype=0, B=1, Hq=2,
            Hkv=2, S=128, Dqk=128, Dv=128, causal=1, scale=0.0, flags=0, status=None):
    return lib.attn_fwd_ex(variant, q, k, v, dq, dk, dv, out, out_dtype, B, Hq, Hkv, S, Dqk, Dv,
                           causal, scale, flags, status, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), fa.ATTN_ERR_INVALID_ARG),
    (dict(out=None), fa.ATTN_ERR_INVALID_ARG),
    (dict(dq=None), fa.ATTN_ERR_INVALID_ARG),
    (dict(k=MIS), fa.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), fa.ATTN_ERR_INVALID_ARG),
    (dict(S=0), fa.ATTN_ERR_INVALID_ARG),
    (dict(B=0), fa.ATTN_ERR_INVALID_ARG),
    (dict(variant=7), fa.ATTN_ERR_INVALID_ARG),
    (dict(variant=5), fa.ATTN_ERR_INVALID_ARG),
    (dict(variant=3, dq=None), fa.ATTN_ERR_INVALID_ARG),       # block-exact is an FP8 path
    (dict(variant=4, dk=None), fa.ATTN_ERR_INVALID_ARG),       # so is the running-max anchor
    (dict(variant=4, Dqk=64), fa.ATTN_ERR_UNSUPPORTED),
    (dict(variant=3, Dv=64), fa.ATTN_ERR_UNSUPPORTED),
    (dict(out_dtype=3), fa.ATTN_ERR_INVALID_ARG),
    (dict(flags=1), fa.ATTN_ERR_INVALID_ARG),          # stall test hook needs a status word
    (dict(scale=float("nan")), fa.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), fa.ATTN_ERR_INVALID_ARG),
    (dict(flags=8), fa.ATTN_ERR_INVALID_ARG),          # unknown flag
    (dict(flags=16), fa.ATTN_ERR_INVALID_ARG),         # unknown flag
    (dict(Dqk=64), fa.ATTN_ERR_UNSUPPORTED),
    (dict(Dv=64), fa.ATTN_ERR_UNSUPPORTED),
    (dict(variant=2, Dqk=192), fa.ATTN_ERR_UNSUPPORTED),
])
def test_bad_arguments_are_rejected_before_launch(lib, kw, want):
    assert call_ex(lib, **kw) == want


def test_bf16_needs_no_descales(lib):
    # descales may be NULL on the BF16 path; with Dqk = 192 the call stops at
    # the (host-side) support check, before any device work
    assert call_ex(lib, variant=2, dq=None, dk=None, dv=None, causal=0, Dqk=192) == \
        fa.ATTN_ERR_UNSUPPORTED


def test_product_entry_points_check_arguments(lib):
    assert lib.attn_fwd_fp8(None, P, P, P, P, P, P, 1, 2, 2, 128, 128, 128, 1, None) == \
        fa.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_fp8_exact(P, P, P, P, P, P, P, 1, 2, 2, 128, 128, 64, 0, None) == \
        fa.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd_bf16(P, P, P, P, 1, 2, 2, 128, 192, 128, 1, None) == \
        fa.ATTN_ERR_UNSUPPORTED


def test_quantize_argument_errors(lib):
    """Host-side validation of attn_quantize_fp8 runs before any device access."""
    vp = ctypes.c_void_p
    q = lib.attn_quantize_fp8
    assert q(None, 0, P, P, 1, 1, 1, 128, 0, None) == fa.ATTN_ERR_INVALID_ARG   # null x
    assert q(P, 2, P, P, 1, 1, 1, 128, 0, None) == fa.ATTN_ERR_INVALID_ARG      # dtype
    assert q(P, 0, P, P, 0, 1, 1, 128, 0, None) == fa.ATTN_ERR_INVALID_ARG      # B = 0
    assert q(P, 0, P, P, 1, 1, 1, 128, 2, None) == fa.ATTN_ERR_INVALID_ARG      # hadamard
    assert q(P, 0, P, P, 1, 1, 1, 64, 0, None) == fa.ATTN_ERR_UNSUPPORTED       # D
    assert q(MIS, 0, P, P, 1, 1, 1, 128, 0, None) == fa.ATTN_ERR_INVALID_ARG    # x alignment
    assert q(vp(0x10008), 0, P, P, 1, 1, 1, 128, 0, None) == fa.ATTN_ERR_INVALID_ARG  # x needs 16 B
    assert q(P, 0, vp(0x10004), P, 1, 1, 1, 128, 0, None) == fa.ATTN_ERR_INVALID_ARG  # codes 16 B
    assert q(P, 0, MIS, P, 1, 1, 1, 128, 0, None) == fa.ATTN_ERR_INVALID_ARG    # codes alignment


def test_full_entry_point_checks_arguments(lib):
    """attn_fwd_full validates the LSE pointer and the descale flag like the rest."""
    f = lib.attn_fwd_full
    args = lambda **kw: [kw.get("variant", 0), P, P, P, P, P, P, P, 0, kw.get("lse", None), 1, 2, 2,
                         128, 128, kw.get("Dv", 128), kw.get("causal", 1), 0.0, kw.get("flags", 0),
                         None, kw.get("ws", None), kw.get("ws_bytes", 0), None]
    assert f(*args(lse=MIS)) == fa.ATTN_ERR_INVALID_ARG                  # misaligned lse
    assert f(*args(flags=8)) == fa.ATTN_ERR_INVALID_ARG                  # unknown flag
    assert f(*args(causal=-1)) == fa.ATTN_ERR_INVALID_ARG
    assert f(*args(Dv=64, flags=fa.ATTN_FLAG_DESCALE_PER_BKV)) == fa.ATTN_ERR_UNSUPPORTED
    # the workspace must be 256-byte aligned (checked before the device)
    assert f(*args(ws=ctypes.c_void_p(0x10010), ws_bytes=1 << 20)) == fa.ATTN_ERR_INVALID_ARG


def test_workspace_size_query(lib):
    """attn_workspace_size: argument errors, and 0 (no split, no device
    needed) for the variants that never split (the running-maximum anchor and
    the exact-FP8 ablation) and for problems whose K and V are large enough
    for the chunked order."""
    n = ctypes.c_size_t(123)
    q = lambda *a, **kw: lib.attn_workspace_size(*a, ctypes.byref(n))
    assert lib.attn_workspace_size(0, 1, 2, 2, 128, 128, 128, 1, 0, None) == fa.ATTN_ERR_INVALID_ARG
    assert q(0, 1, 3, 2, 128, 128, 128, 1, 0) == fa.ATTN_ERR_INVALID_ARG and n.value == 0  # Hq % Hkv
    assert q(9, 1, 2, 2, 128, 128, 128, 1, 0) == fa.ATTN_ERR_INVALID_ARG                 # variant
    assert q(0, 1, 2, 2, 128, 128, 128, 2, 0) == fa.ATTN_ERR_INVALID_ARG                 # causal
    for variant in (fa.ATTN_VARIANT_EXACT_FP8, fa.ATTN_VARIANT_LEANP_A3):
        n.value = 123
        assert q(variant, 1, 8, 8, 4096, 128, 128, 1, 0) == fa.ATTN_OK and n.value == 0
    n.value = 123
    assert q(0, 1, 8, 8, 4096, 128, 128, 1, fa.ATTN_FLAG_TEST_CHUNK_UNITS) == fa.ATTN_OK
    assert n.value == 0
    n.value = 123
    assert q(0, 1, 32, 32, 65536, 128, 128, 1, 0) == fa.ATTN_OK and n.value == 0      # chunked
    n.value = 123
    assert q(fa.ATTN_VARIANT_BF16, 1, 16, 16, 65536, 128, 128, 1, 0) == fa.ATTN_OK  # bf16 K, V:
    assert n.value == 0                                                   # 2 bytes each


def test_release_library_has_no_timeline(lib):
    """The release build answers the debug timeline call with UNSUPPORTED
    before touching any device."""
    import numpy as np
    buf = np.zeros(16, dtype=np.uint64)
    assert lib.attn_debug_timeline(buf.ctypes.data, buf.size, 1) == fa.ATTN_ERR_UNSUPPORTED


def test_host_descales_must_be_finite_and_positive():
    """The binding checks descales it is given as host numbers (the library's
    contract: finite and greater than zero); device descales cannot be read
    without a synchronisation and are the caller's responsibility."""
    assert fa.host_descale("q_descale", 0.0125) == 0.0125
    assert fa.host_descale("q_descale", 3) == 3.0
    for bad in (0.0, -0.5, float("inf"), float("-inf"), float("nan")):
        with pytest.raises(ValueError):
            fa.host_descale("k_descale", bad)
    with pytest.raises(TypeError):
        fa.host_descale("v_descale", "one")
