"""Failure detection on the GPU without a GPU fault.

A testing hook makes the MMA warp of the forward (or backward) kernel issue
nothing; the other warps' bounded pipeline waits then run out after a short
time limit, the kernel stops early and reports ATTN_ERR_TIMEOUT through its
status word. No fault, trap or unbounded wait is involved. The test then
checks that the same process still computes correct results.
"""
import numpy as np
import pytest
import torch

import attention_fwd_bwd_gb300 as attn
from attention_fwd_bwd_gb300.inputs import make_inputs
from oracle import attn_ref_fwd
from tests.helpers import assert_close_fwd, gpu_fwd_bwd, np64

pytestmark = pytest.mark.gpu

TIMEOUT_STATUS = 4


def _buffers(B, Hq, Hkv, S, D, seed):
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in make_inputs(B, Hq, Hkv, S, D, seed))
    o, o_lo = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty(q.shape, **f32), torch.empty(k.shape, **f32), torch.empty(k.shape, **f32)
    ws = torch.empty(attn.attn_bwd_workspace_size(B, Hq, Hkv, S, D), dtype=torch.uint8, device=dev)
    return q, k, v, do, o, o_lo, lse, dq, dk, dv, ws


@pytest.mark.parametrize("D", [128, 64])
def test_stalled_pipeline_times_out_and_context_survives(D):
    # D = 64 takes the forward with one MMA warp per query tile and the
    # backward whose P/dS warps read dQ^T themselves.
    B, Hq, Hkv, S = 1, 4, 2, 512
    q, k, v, do, o, o_lo, lse, dq, dk, dv, ws = _buffers(B, Hq, Hkv, S, D, seed=5)
    scale = D ** -0.5
    assert attn.attn_check_status(None) == 0
    attn.attn_set_wait_timeout_ns(2_000_000)  # 2 ms
    try:
        attn.attn_set_fault_injection(1)
        attn.attn_fwd_residual(q, k, v, o, o_lo, lse, True, scale)
        assert attn.attn_check_status(None) == TIMEOUT_STATUS
        attn.attn_set_fault_injection(2)
        attn.attn_fwd_residual(q, k, v, o, o_lo, lse, True, scale)
        attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, True, scale, ws, o_lo=o_lo)
        assert attn.attn_check_status(ws) == TIMEOUT_STATUS
        assert attn.attn_check_status(ws) == 0  # reading clears the word
        # Without o_lo the backward also runs the Dvec pass; its MMA warp
        # takes the same hook.
        attn.attn_bwd_preprocess(q, k, o, do, lse, dq, ws)
        attn.attn_bwd_dvec(q, k, v, do, True, scale, ws)
        assert attn.attn_check_status(ws) == TIMEOUT_STATUS
        attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, True, scale, ws)
        assert attn.attn_check_status(ws) == TIMEOUT_STATUS
        # A timeout stays recorded until it is read: a later call on the same
        # workspace does not erase it.
        attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, True, scale, ws, o_lo=o_lo)
        attn.attn_set_fault_injection(0)
        attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, True, scale, ws, o_lo=o_lo)
        assert attn.attn_check_status(ws) == TIMEOUT_STATUS
        assert attn.attn_check_status(ws) == 0
    finally:
        attn.attn_set_fault_injection(0)
        attn.attn_set_wait_timeout_ns(0)
    # The context is intact: a normal run afterwards is correct.
    qc, kc, vc, doc = make_inputs(B, Hq, Hkv, S, D, seed=5)
    got = gpu_fwd_bwd(qc, kc, vc, doc, True, scale)
    o_ref, lse_ref = attn_ref_fwd(np64(qc), np64(kc), np64(vc), True, scale)
    assert_close_fwd(got["o"], got["lse"], o_ref, lse_ref, "after injected timeout")
