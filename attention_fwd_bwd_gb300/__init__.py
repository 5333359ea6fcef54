"""GB300 (sm_103a) fused attention forward and backward.

A thin ctypes binding over libattn.so, whose C ABI is declared in
include/attn.h. Each function here only marshals arguments: it checks the
torch tensors' dtype, device and layout, reads the sizes off their shapes and
passes raw device pointers and the current CUDA stream to the library of the
same name. All compute runs in the library's CUDA kernels; there is no other
code path. If libattn.so is missing the first call raises.

Layout: q, o, o_lo, dO are [B, S, Hq, D] bf16; k, v are [B, S, Hkv, D] bf16;
dq is [B, S, Hq, D] fp32; dk, dv are [B, S, Hkv, D] fp32; lse is [B, Hq, S]
fp32; all contiguous on one CUDA device.
"""
import ctypes
import os

__all__ = [
    "AttnError",
    "lib",
    "attn_fwd",
    "attn_fwd_residual",
    "attn_fwd_ex",
    "attn_bwd",
    "attn_bwd_ex",
    "attn_bwd_main_ex",
    "attn_bwd_preprocess",
    "attn_bwd_main",
    "attn_bwd_dvec",
    "attn_bwd_noalloc",
    "attn_sparse_fwd",
    "attn_sparse_bwd",
    "attn_sparse_bwd_workspace_size",
    "attn_bwd_workspace_size",
    "attn_check_status",
    "attn_set_wait_timeout_ns",
    "attn_set_fault_injection",
    "attn_status_string",
    "use_debug_library",
    "STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libattn.so")
# The bounds-checked build (index checks that report ATTN_ERR_BOUNDS), for tests.
LIB_DEBUG_PATH = os.path.join(_HERE, "_lib", "libattn_debug.so")

STATUS = {
    0: "ATTN_OK",
    1: "ATTN_ERR_INVALID_ARG",
    2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_CUDA",
    4: "ATTN_ERR_TIMEOUT",
    5: "ATTN_ERR_WORKSPACE",
    6: "ATTN_ERR_BOUNDS",
}

_lib = None
_lib_debug = None
_use_debug = False


def use_debug_library(flag=True):
    """Route every call of this module to the bounds-checked build
    libattn_debug.so (flag True) or back to libattn.so."""
    global _use_debug
    _use_debug = bool(flag)


class AttnError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({attn_status_string(code)})")


def lib():
    """The loaded libattn.so (or, after use_debug_library(True),
    libattn_debug.so) with argument types set (raises if it is missing)."""
    global _lib, _lib_debug
    if _use_debug and _lib_debug is not None:
        return _lib_debug
    if not _use_debug and _lib is not None:
        return _lib
    path = LIB_DEBUG_PATH if _use_debug else LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{os.path.basename(path)} not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "or `python attention_fwd_bwd_gb300/_build.py`"
            + (" (debug=True for the bounds-checked build)" if _use_debug else ""))
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    L.attn_fwd.restype = i
    L.attn_fwd_residual.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    L.attn_fwd_residual.restype = i
    L.attn_bwd_workspace_size.argtypes = [i, i, i, i, i]
    L.attn_bwd_workspace_size.restype = sz
    L.attn_bwd.argtypes = [vp] * 10 + [i] * 6 + [f, vp, sz, vp]
    L.attn_bwd.restype = i
    L.attn_bwd_preprocess.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp, sz, vp]
    L.attn_bwd_preprocess.restype = i
    L.attn_bwd_main.argtypes = [vp] * 7 + [i] * 6 + [f, vp, sz, vp]
    L.attn_bwd_main.restype = i
    L.attn_bwd_dvec.argtypes = [vp] * 4 + [i] * 7 + [f, vp, sz, vp]
    L.attn_bwd_dvec.restype = i
    L.attn_fwd_ex.argtypes = [vp] * 6 + [i] * 7 + [f, vp]
    L.attn_fwd_ex.restype = i
    L.attn_bwd_ex.argtypes = [vp] * 10 + [i] * 7 + [f, vp, sz, vp]
    L.attn_bwd_ex.restype = i
    L.attn_bwd_main_ex.argtypes = [vp] * 7 + [i] * 7 + [f, vp, sz, vp]
    L.attn_bwd_main_ex.restype = i
    L.attn_bwd_noalloc.argtypes = [vp] * 10 + [i] * 6 + [f, vp]
    L.attn_bwd_noalloc.restype = i
    L.attn_sparse_fwd.argtypes = [vp] * 7 + [i] * 7 + [f, vp]
    L.attn_sparse_fwd.restype = i
    L.attn_sparse_bwd_workspace_size.argtypes = [i, i, i]
    L.attn_sparse_bwd_workspace_size.restype = sz
    L.attn_sparse_bwd.argtypes = [vp] * 11 + [i] * 7 + [f, vp, sz, vp]
    L.attn_sparse_bwd.restype = i
    L.attn_status_string.argtypes = [i]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_check_status.argtypes = [vp]
    L.attn_check_status.restype = i
    L.attn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.attn_set_wait_timeout_ns.restype = None
    L.attn_set_fault_injection.argtypes = [i]
    L.attn_set_fault_injection.restype = None
    if _use_debug:
        _lib_debug = L
    else:
        _lib = L
    return L


def attn_status_string(code):
    return lib().attn_status_string(int(code)).decode()


def _check(fn, code):
    if code != 0:
        raise AttnError(fn, code)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _sizes(q, k):
    import torch
    for t in (q, k):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v, o, o_lo, dO must be contiguous 4-D bf16 CUDA tensors [B,S,H,D]")
    B, S, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if (Bk, Sk, Dk) != (B, S, D):
        raise ValueError(f"k shape {tuple(k.shape)} does not match q shape {tuple(q.shape)}")
    return B, Hq, Hkv, S, D


def _like(t, ref, what, dtype=None):
    dtype = ref.dtype if dtype is None else dtype
    if t.shape != ref.shape or t.dtype != dtype or not t.is_contiguous() or t.device != ref.device:
        raise ValueError(f"{what} must be a contiguous {dtype} tensor of shape {tuple(ref.shape)}")


def _lse_ok(lse, B, Hq, S, dev):
    import torch
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, S) or not lse.is_contiguous() or lse.device != dev:
        raise ValueError(f"lse must be a contiguous fp32 tensor of shape {(B, Hq, S)}")


def _opt(t):
    return None if t is None else _ptr(t)


def attn_fwd(q, k, v, o, lse, causal, scale, stream=None):
    """o, lse <- attention(q, k, v); see attn_fwd in include/attn.h."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    _like(v, k, "v")
    _like(o, q, "o")
    _lse_ok(lse, B, Hq, S, q.device)
    _check("attn_fwd", lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, S, D,
                                      int(bool(causal)), float(scale), _stream(stream)))


def attn_fwd_residual(q, k, v, o, o_lo, lse, causal, scale, stream=None):
    """o, o_lo, lse <- attention(q, k, v); see attn_fwd_residual in include/attn.h."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    _like(v, k, "v")
    _like(o, q, "o")
    _like(o_lo, q, "o_lo")
    _lse_ok(lse, B, Hq, S, q.device)
    _check("attn_fwd_residual", lib().attn_fwd_residual(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_lo), _ptr(lse),
                                                        B, Hq, Hkv, S, D, int(bool(causal)), float(scale),
                                                        _stream(stream)))


def attn_fwd_ex(q, k, v, o, lse, causal, window, scale, o_lo=None, stream=None):
    """Forward with a sliding window (window > 0: query i sees keys i-window+1..i,
    needs causal); with o_lo it is the residual forward. See attn_fwd_ex in
    include/attn.h."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    _like(v, k, "v")
    _like(o, q, "o")
    if o_lo is not None:
        _like(o_lo, q, "o_lo")
    _lse_ok(lse, B, Hq, S, q.device)
    _check("attn_fwd_ex", lib().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _opt(o_lo), _ptr(lse),
                                            B, Hq, Hkv, S, D, int(bool(causal)), int(window), float(scale),
                                            _stream(stream)))


def _sparse_sizes(q, kp, vp, idx):
    import torch
    for t in (q, kp, vp):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, kp, vp, o, o_lo, dO must be contiguous bf16 CUDA tensors")
    if q.dim() != 4 or kp.dim() != 3 or vp.dim() != 3:
        raise ValueError("q is [B,T,H,DK], kp [B,P,DK], vp [B,P,DV]")
    B, T, H, DK = q.shape
    if kp.shape[0] != B or kp.shape[2] != DK or tuple(vp.shape[:2]) != tuple(kp.shape[:2]):
        raise ValueError(f"kp {tuple(kp.shape)} / vp {tuple(vp.shape)} do not match q {tuple(q.shape)}")
    if (idx.dtype != torch.int32 or not idx.is_contiguous() or idx.dim() != 3
            or tuple(idx.shape[:2]) != (B, T) or idx.device != q.device):
        raise ValueError("idx must be a contiguous int32 tensor [B, T, K] on q's device")
    return B, T, H, kp.shape[1], idx.shape[2], DK, vp.shape[2]


def attn_sparse_fwd(q, kp, vp, idx, o, lse, scale, o_lo=None, stream=None):
    """o (and o_lo), lse <- sparse top-k gather attention; see attn_sparse_fwd
    in include/attn.h."""
    import torch
    B, T, H, P, K, DK, DV = _sparse_sizes(q, kp, vp, idx)
    ref = torch.empty((B, T, H, DV), dtype=torch.bfloat16, device="meta")
    for t, what in ((o, "o"), (o_lo, "o_lo")):
        if t is not None and (tuple(t.shape) != tuple(ref.shape) or t.dtype != torch.bfloat16
                              or not t.is_contiguous() or t.device != q.device):
            raise ValueError(f"{what} must be a contiguous bf16 tensor of shape {tuple(ref.shape)}")
    _lse_ok(lse, B, H, T, q.device)
    _check("attn_sparse_fwd", lib().attn_sparse_fwd(_ptr(q), _ptr(kp), _ptr(vp), _ptr(idx), _ptr(o), _opt(o_lo),
                                                    _ptr(lse), B, T, H, P, K, DK, DV, float(scale),
                                                    _stream(stream)))


def attn_sparse_bwd_workspace_size(B, T, H):
    return int(lib().attn_sparse_bwd_workspace_size(B, T, H))


def attn_sparse_bwd(q, kp, vp, idx, o, dO, lse, dq, dkp, dvp, scale, workspace, o_lo=None, stream=None):
    """dq, dkp, dvp <- gradient of sparse top-k gather attention; see
    attn_sparse_bwd in include/attn.h."""
    import torch
    B, T, H, P, K, DK, DV = _sparse_sizes(q, kp, vp, idx)
    for t, what, shape, dt in ((o, "o", (B, T, H, DV), torch.bfloat16), (dO, "dO", (B, T, H, DV), torch.bfloat16),
                               (o_lo, "o_lo", (B, T, H, DV), torch.bfloat16),
                               (dq, "dq", (B, T, H, DK), torch.float32), (dkp, "dkp", (B, P, DK), torch.float32),
                               (dvp, "dvp", (B, P, DV), torch.float32)):
        if t is not None and (tuple(t.shape) != shape or t.dtype != dt or not t.is_contiguous()
                              or t.device != q.device):
            raise ValueError(f"{what} must be a contiguous {dt} tensor of shape {shape}")
    _lse_ok(lse, B, H, T, q.device)
    ws, wsb = _ws(workspace)
    _check("attn_sparse_bwd", lib().attn_sparse_bwd(_ptr(q), _ptr(kp), _ptr(vp), _ptr(idx), _ptr(o), _opt(o_lo),
                                                    _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dkp), _ptr(dvp),
                                                    B, T, H, P, K, DK, DV, float(scale), ws, wsb,
                                                    _stream(stream)))


def attn_bwd_workspace_size(B, Hq, Hkv, S, D):
    return int(lib().attn_bwd_workspace_size(B, Hq, Hkv, S, D))


def _ws(workspace):
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def _grads_ok(q, k, dq, dk, dv):
    import torch
    _like(dq, q, "dq", torch.float32)
    _like(dk, k, "dk", torch.float32)
    _like(dv, k, "dv", torch.float32)


def attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, causal, scale, workspace, o_lo=None, stream=None):
    """dq, dk, dv (fp32) <- gradients of sum(dO * o); see attn_bwd in include/attn.h."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    for t, ref, n in ((v, k, "v"), (o, q, "o"), (dO, q, "dO")):
        _like(t, ref, n)
    if o_lo is not None:
        _like(o_lo, q, "o_lo")
    _grads_ok(q, k, dq, dk, dv)
    _lse_ok(lse, B, Hq, S, q.device)
    wp, wb = _ws(workspace)
    _check("attn_bwd", lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                                      _ptr(dk), _ptr(dv), _opt(o_lo), B, Hq, Hkv, S, D, int(bool(causal)),
                                      float(scale), wp, wb, _stream(stream)))


def attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv, causal, window, scale, workspace, o_lo=None, stream=None):
    """attn_bwd with a sliding window; see attn_bwd_ex in include/attn.h."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    for t, ref, n in ((v, k, "v"), (o, q, "o"), (dO, q, "dO")):
        _like(t, ref, n)
    if o_lo is not None:
        _like(o_lo, q, "o_lo")
    _grads_ok(q, k, dq, dk, dv)
    _lse_ok(lse, B, Hq, S, q.device)
    wp, wb = _ws(workspace)
    _check("attn_bwd_ex", lib().attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                                            _ptr(dk), _ptr(dv), _opt(o_lo), B, Hq, Hkv, S, D, int(bool(causal)),
                                            int(window), float(scale), wp, wb, _stream(stream)))


def attn_bwd_preprocess(q, k, o, dO, lse, dq, workspace, o_lo=None, stream=None):
    """Stage 1 of attn_bwd (q and k only supply the sizes)."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    wp, wb = _ws(workspace)
    _check("attn_bwd_preprocess", lib().attn_bwd_preprocess(_ptr(o), _opt(o_lo), _ptr(dO), _ptr(lse), _ptr(dq),
                                                            B, Hq, Hkv, S, D, wp, wb, _stream(stream)))


def attn_bwd_dvec(q, k, v, dO, causal, scale, workspace, window=0, stream=None):
    """Optional stage between attn_bwd_preprocess and attn_bwd_main: Dvec =
    sum_j P_ij dP_ij from q, k, v, dO and the LSE rows in the workspace."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    wp, wb = _ws(workspace)
    _check("attn_bwd_dvec", lib().attn_bwd_dvec(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), B, Hq, Hkv, S, D,
                                                int(bool(causal)), int(window), float(scale), wp, wb,
                                                _stream(stream)))


def attn_bwd_main(q, k, v, dO, dq, dk, dv, causal, scale, workspace, stream=None):
    """Stage 2 of attn_bwd."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    wp, wb = _ws(workspace)
    _check("attn_bwd_main", lib().attn_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk),
                                                _ptr(dv), B, Hq, Hkv, S, D, int(bool(causal)), float(scale),
                                                wp, wb, _stream(stream)))


def attn_bwd_main_ex(q, k, v, dO, dq, dk, dv, causal, window, scale, workspace, stream=None):
    """Stage 2 of attn_bwd_ex."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    wp, wb = _ws(workspace)
    _check("attn_bwd_main_ex", lib().attn_bwd_main_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk),
                                                      _ptr(dv), B, Hq, Hkv, S, D, int(bool(causal)), int(window),
                                                      float(scale), wp, wb, _stream(stream)))


def attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, causal, scale, o_lo=None, stream=None):
    """attn_bwd without a workspace, for callers that cannot allocate device
    memory: it uses the library's built-in 16 MiB scratch array (see
    attn_bwd_noalloc in include/attn.h)."""
    B, Hq, Hkv, S, D = _sizes(q, k)
    for t, ref, n in ((v, k, "v"), (o, q, "o"), (dO, q, "dO")):
        _like(t, ref, n)
    if o_lo is not None:
        _like(o_lo, q, "o_lo")
    _grads_ok(q, k, dq, dk, dv)
    _lse_ok(lse, B, Hq, S, q.device)
    _check("attn_bwd_noalloc", lib().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                                                      _ptr(dq), _ptr(dk), _ptr(dv), _opt(o_lo), B, Hq, Hkv, S, D,
                                                      int(bool(causal)), float(scale), _stream(stream)))


def attn_check_status(workspace=None):
    """Synchronises and returns the device status code (0 = ok, 4 = a wait timed out)."""
    return int(lib().attn_check_status(None if workspace is None else ctypes.c_void_p(workspace.data_ptr())))


def attn_set_wait_timeout_ns(ns):
    lib().attn_set_wait_timeout_ns(int(ns))


def attn_set_fault_injection(mask):
    """Testing hook: bit 0 stalls the forward's MMA warp, bit 1 the backward's."""
    lib().attn_set_fault_injection(int(mask))
