"""The C ABI library, on the CPU: it builds, loads, exports every entry point
include/attn.h declares, and rejects bad arguments before touching a device.
None of these calls launches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    import attention_fwd_bwd_gb300 as attn
    return attn.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("attn_fwd", "attn_fwd_residual", "attn_bwd", "attn_bwd_workspace_size",
              "attn_status_string", "attn_bwd_preprocess", "attn_bwd_main"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), f"libattn.so does not export {n}"


def test_status_strings(L):
    for code in range(7):
        assert L.attn_status_string(code) != b"unknown status"
    assert L.attn_status_string(99) == b"unknown status"


FAKE = 0x10000  # aligned, never dereferenced: validation fails before any use


def _fwd(L, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, S=128, D=64, causal=1, scale=0.125):
    return L.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, S, D, causal, scale, None)


def test_fwd_argument_validation(L):
    assert _fwd(L, D=96) == 2                 # unsupported head dim
    assert _fwd(L, D=256) == 2
    assert _fwd(L, Hq=3, Hkv=2) == 1          # Hq not a multiple of Hkv
    assert _fwd(L, Hkv=0) == 1
    assert _fwd(L, Hq=0) == 1
    assert _fwd(L, B=-1) == 1
    assert _fwd(L, S=-5) == 1
    assert _fwd(L, S=(1 << 24) + 1) == 2
    assert _fwd(L, scale=float("nan")) == 1
    assert _fwd(L, scale=float("inf")) == 1
    assert _fwd(L, q=None) == 1               # null pointer
    assert _fwd(L, lse=None) == 1
    assert _fwd(L, o=FAKE + 8) == 1           # not 16-byte aligned
    assert _fwd(L, B=0, q=None, k=None, v=None, o=None, lse=None) == 0   # empty: no-op
    assert _fwd(L, S=0, q=None, k=None, v=None, o=None, lse=None) == 0


def test_window_argument_validation(L):
    fwd = lambda window, causal=1, B=1: L.attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, None, FAKE, B, 2, 1, 128, 64,
                                                     causal, window, 0.125, None)
    assert fwd(-1) == 1                       # negative window
    assert fwd(4, causal=0) == 1              # a window needs causal
    assert fwd(-1, B=0) == 1                  # checked with the sizes, before the empty no-op
    assert fwd(4, B=0) == 0                   # empty: no-op
    bwd = lambda window, causal=1: L.attn_bwd_ex(*([FAKE] * 9 + [None]), 1, 2, 1, 128, 64, causal, window,
                                                 0.125, FAKE * 16, 1 << 30, None)
    assert bwd(-3) == 1
    assert bwd(128, causal=0) == 1
    main = lambda window, causal=1: L.attn_bwd_main_ex(*([FAKE] * 7), 1, 2, 1, 128, 64, causal, window,
                                                       0.125, FAKE * 16, 1 << 30, None)
    assert main(-3) == 1
    assert main(128, causal=0) == 1


def test_sparse_argument_validation(L):
    def fwd(B=1, T=4, H=128, P=10, K=8, DK=128, DV=64, scale=0.1, ptrs=None):
        p = ptrs if ptrs is not None else [FAKE] * 5 + [None, FAKE]
        return L.attn_sparse_fwd(*p, B, T, H, P, K, DK, DV, scale, None)
    assert fwd(H=0) == 1
    assert fwd(H=129) == 1                    # one token's heads fill at most one 128-row tile
    assert fwd(K=6) == 1                      # K a multiple of 4
    assert fwd(K=0) == 1
    assert fwd(P=0) == 1
    assert fwd(T=-1) == 1
    assert fwd(DK=96) == 2
    assert fwd(DV=256) == 2
    assert fwd(scale=float("nan")) == 1
    assert fwd(B=0, ptrs=[None] * 7) == 0     # empty: no-op
    assert fwd(ptrs=[FAKE, FAKE, FAKE, None, FAKE, None, FAKE]) == 1   # null idx
    assert fwd(ptrs=[FAKE, FAKE, FAKE, FAKE + 4, FAKE, None, FAKE]) == 1  # misaligned idx


def test_sparse_bwd_argument_validation(L):
    def bwd(B=1, T=4, H=128, P=10, K=8, DK=128, DV=64, ws=FAKE * 16, wsb=1 << 30, ptrs=None):
        p = ptrs if ptrs is not None else [FAKE] * 5 + [None] + [FAKE] * 5
        return L.attn_sparse_bwd(*p, B, T, H, P, K, DK, DV, 0.1, ws, wsb, None)
    assert bwd(H=200) == 1
    assert bwd(K=5) == 1
    assert bwd(DK=32) == 2
    assert bwd(ws=None) == 5                  # workspace missing
    assert bwd(ws=FAKE * 16 + 16) == 5        # not 256-byte aligned
    assert bwd(wsb=16) == 5                   # too small
    assert bwd(B=0, ptrs=[None] * 11) == 0
    assert L.attn_sparse_bwd_workspace_size(1, 4, 128) == 256 + 2 * 2048
    assert L.attn_sparse_bwd_workspace_size(1, 4, 0) == 0


def test_bwd_argument_validation(L):
    def bwd(ws=FAKE * 16, wsb=1 << 30, B=1, S=128, D=64, ptrs=None, Hq=2, Hkv=1):
        p = ptrs if ptrs is not None else [FAKE] * 9 + [None]
        return L.attn_bwd(*p, B, Hq, Hkv, S, D, 1, 0.125, ws, wsb, None)

    need = L.attn_bwd_workspace_size(1, 2, 1, 128, 64)
    assert need > 0
    assert bwd(ws=None) == 5
    assert bwd(ws=FAKE * 16 + 16) == 5        # workspace must be 256-byte aligned
    assert bwd(wsb=need - 1) == 5
    assert bwd(D=80) == 2
    assert bwd(Hq=4, Hkv=3) == 1
    assert bwd(ptrs=[FAKE] * 8 + [None, None]) == 1          # dv missing
    assert bwd(ptrs=[FAKE] * 5 + [FAKE + 4] + [FAKE] * 3 + [None]) == 1
    assert bwd(ptrs=[FAKE] * 9 + [FAKE + 8]) == 1            # misaligned o_lo
    assert bwd(B=0, ptrs=[None] * 10, ws=None, wsb=0) == 0


def test_workspace_size_formula(L):
    # status word block + two fp32 row vectors (log2-scaled LSE and Dvec), with
    # the sequence padded to a multiple of 128 and each part 256-byte aligned.
    def expect(B, Hq, S, D):
        al = lambda x: (x + 255) // 256 * 256
        rows = B * Hq * ((S + 127) // 128 * 128)
        return 256 + 2 * al(rows * 4)
    for args in ((1, 1, 128, 64), (2, 32, 4096, 128), (1, 3, 300, 128), (1, 64, 8192, 128)):
        B, Hq, S, D = args
        assert L.attn_bwd_workspace_size(B, Hq, 1, S, D) == expect(B, Hq, S, D)
    assert L.attn_bwd_workspace_size(1, 2, 1, 128, 96) == 0
    assert L.attn_bwd_workspace_size(0, 2, 1, 128, 64) == 0


def test_fwd_residual_requires_o_lo(L):
    assert L.attn_fwd_residual(FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, 2, 1, 128, 64, 1, 0.125, None) == 1
    assert L.attn_fwd_residual(FAKE, FAKE, FAKE, FAKE, FAKE + 4, FAKE, 1, 2, 1, 128, 64, 1, 0.125, None) == 1
    assert L.attn_fwd_residual(None, None, None, None, None, None, 0, 2, 1, 128, 64, 1, 0.125, None) == 0


def test_binding_fails_loudly_without_library(monkeypatch):
    import attention_fwd_bwd_gb300 as attn
    monkeypatch.setattr(attn, "_lib", None)
    monkeypatch.setattr(attn, "LIB_PATH", "/nonexistent/libattn.so")
    with pytest.raises(ImportError):
        attn.lib()


def test_build_hash_covers_every_source_and_header():
    from attention_fwd_bwd_gb300 import _build as B
    present = sorted(f for f in os.listdir(B.CSRC) if f.endswith((".cu", ".cuh")))
    assert sorted(B.SOURCES + B.HEADERS) == present


def test_binding_covers_every_entry_point():
    import attention_fwd_bwd_gb300 as attn
    for n in _declared():
        assert n in attn.__all__ and callable(getattr(attn, n)), f"no Python binding for {n}"


def test_bounds_checked_build_compiles_and_exports_the_same_symbols():
    """The bounds-checked build (-DATTN_DEBUG_BOUNDS) compiles for sm_103a and
    exports every declared entry point; its argument checks are the same."""
    from attention_fwd_bwd_gb300._build import build
    path = build(debug=True)
    D = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(D, n), f"libattn_debug.so does not export {n}"
    D.attn_fwd.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_void_p]
    assert D.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 1, 128, 96, 1, 0.125, None) == 2
    assert D.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 3, 2, 128, 64, 1, 0.125, None) == 1
