"""attn_bwd_noalloc, the backward for callers that cannot allocate device
memory (a plugin that only receives the tensors of one call, or a path where
a device-synchronising cudaMalloc is not allowed), checked on the GPU against
the workspace-taking attn_bwd through the C ABI.

This file sorts last so that a run stopping at its first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import attention_fwd_bwd_gb300 as attn
from attention_fwd_bwd_gb300.inputs import make_inputs
from tests.helpers import TOL_GRAD_REL_RMS

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_matches_workspace_backward_twice():
    L = attn.lib()
    dev = torch.device("cuda", 0)
    B, Hq, Hkv, S, D, causal = 1, 4, 2, 384, 128, True
    scale = D ** -0.5
    q, k, v, do = (t.to(dev) for t in make_inputs(B, Hq, Hkv, S, D, seed=99))
    o, o_lo = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    assert L.attn_fwd_residual(_p(q), _p(k), _p(v), _p(o), _p(o_lo), _p(lse), B, Hq, Hkv, S, D,
                               int(causal), scale, None) == 0
    f32 = dict(dtype=torch.float32, device=dev)
    ref = [torch.empty(q.shape, **f32), torch.empty(k.shape, **f32), torch.empty(k.shape, **f32)]
    ws = torch.empty(L.attn_bwd_workspace_size(B, Hq, Hkv, S, D), dtype=torch.uint8, device=dev)
    assert L.attn_bwd(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), *(_p(t) for t in ref), _p(o_lo),
                      B, Hq, Hkv, S, D, int(causal), scale, _p(ws), ws.numel(), None) == 0
    torch.cuda.synchronize()
    for call in range(2):
        got = [torch.full(q.shape, float("nan"), **f32), torch.full(k.shape, float("nan"), **f32),
               torch.full(k.shape, float("nan"), **f32)]
        assert L.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), *(_p(t) for t in got),
                                  _p(o_lo), B, Hq, Hkv, S, D, int(causal), scale, None) == 0
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            rms = float(r.double().pow(2).mean().sqrt())
            err = float((g.double() - r.double()).abs().max())
            assert err <= TOL_GRAD_REL_RMS * rms, f"call {call}: {name} error {err:.3e} vs rms {rms:.3e}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = attn.lib()
    # B*Hq*S_pad = 4 * 64 * 8192 rows need 2 * 8 MiB + 256 bytes of scratch > 16 MiB.
    fake = ctypes.c_void_p(0x10000)
    st = L.attn_bwd_noalloc(*([fake] * 9), None, 4, 64, 8, 8192, 128, 1, 0.088, None)
    assert st == 5  # ATTN_ERR_WORKSPACE, nothing launched


def test_noalloc_reports_a_timeout_through_check_status():
    """A bounded wait that runs out inside attn_bwd_noalloc is reported by
    attn_check_status(NULL), which reads the status word in the library's
    scratch array once a call on the device has looked the array up. The
    stall comes from the testing hook (the backward's MMA warp issues
    nothing) with a 2 ms wait limit: no fault, trap or unbounded wait."""
    L = attn.lib()
    dev = torch.device("cuda", 0)
    B, Hq, Hkv, S, D = 1, 2, 1, 256, 64
    scale = D ** -0.5
    q, k, v, do = (t.to(dev) for t in make_inputs(B, Hq, Hkv, S, D, seed=3))
    o, o_lo = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty(q.shape, **f32), torch.empty(k.shape, **f32), torch.empty(k.shape, **f32)
    assert L.attn_fwd_residual(_p(q), _p(k), _p(v), _p(o), _p(o_lo), _p(lse), B, Hq, Hkv, S, D, 1,
                               scale, None) == 0
    assert attn.attn_check_status(None) == 0
    attn.attn_set_wait_timeout_ns(2_000_000)
    try:
        attn.attn_set_fault_injection(2)
        assert L.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                                  _p(o_lo), B, Hq, Hkv, S, D, 1, scale, None) == 0
        assert attn.attn_check_status(None) == 4  # ATTN_ERR_TIMEOUT
        assert attn.attn_check_status(None) == 0  # reading cleared it
    finally:
        attn.attn_set_fault_injection(0)
        attn.attn_set_wait_timeout_ns(0)
    assert L.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                              _p(o_lo), B, Hq, Hkv, S, D, 1, scale, None) == 0
    assert attn.attn_check_status(None) == 0
