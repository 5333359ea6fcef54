"""Shared helpers of the GPU tests: run the CUDA path through the C ABI and
compare its results with the oracle under the stated tolerances."""
import numpy as np
import torch

import attention_fwd_bwd_gb300 as attn

# Tolerances: O max-abs <= 2e-2, LSE max-abs <= 1e-3, and each of dQ, dK, dV
# max-abs <= 5e-2 * rms of the oracle's gradient.
TOL_O = 2e-2
TOL_LSE = 1e-3
TOL_GRAD_REL_RMS = 5e-2


def gpu_fwd_bwd(q, k, v, do, causal, scale, with_bwd=True, window=0, residual=True):
    """Run attn_fwd_residual (and attn_bwd with the residual) on cuda:0 for
    bf16 CPU tensors; returns a dict of CPU tensors (o, lse, dq, dk, dv).
    With window > 0 the sliding-window forms (attn_fwd_ex, attn_bwd_ex) run.
    With residual=False the plain calls run instead: attn_fwd (o and lse only)
    and attn_bwd with o_lo = None (or their window forms without o_lo)."""
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev).contiguous() for t in (q, k, v, do))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    o = torch.empty_like(qd)
    o_lo = torch.empty_like(qd) if residual else None
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    if window:
        attn.attn_fwd_ex(qd, kd, vd, o, lse, causal, window, scale, o_lo=o_lo)
    elif residual:
        attn.attn_fwd_residual(qd, kd, vd, o, o_lo, lse, causal, scale)
    else:
        attn.attn_fwd(qd, kd, vd, o, lse, causal, scale)
    out = {"o": o, "lse": lse}
    ws = None
    if with_bwd:
        ws = torch.empty(max(256, attn.attn_bwd_workspace_size(B, Hq, Hkv, S, D)), dtype=torch.uint8, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        dq = torch.empty(qd.shape, **f32)
        dk, dv = torch.empty(kd.shape, **f32), torch.empty(vd.shape, **f32)
        if window:
            attn.attn_bwd_ex(qd, kd, vd, o, dod, lse, dq, dk, dv, causal, window, scale, ws, o_lo=o_lo)
        else:
            attn.attn_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, causal, scale, ws, o_lo=o_lo)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    st = attn.attn_check_status(ws)
    assert st == 0, f"device status {st}"
    return {n: t.cpu() for n, t in out.items()}


def np64(t):
    return t.to(torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, dtype=np.float64)


def assert_close_fwd(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    eo = np.max(np.abs(np64(o_gpu) - o_ref)) if o_ref.size else 0.0
    el = np.max(np.abs(np64(lse_gpu) - lse_ref)) if lse_ref.size else 0.0
    assert eo <= TOL_O, f"{what} O max-abs error {eo:.3e} > {TOL_O}"
    assert el <= TOL_LSE, f"{what} LSE max-abs error {el:.3e} > {TOL_LSE}"
    return eo, el


# When the exact gradient is identically zero (a row or tile with a single
# visible key has dS = 0), a bound relative to its rms is zero too; the GPU's
# fp32 rounding of dP - Dvec is then held to this absolute floor instead.
ZERO_GRAD_FLOOR = 1e-5


def assert_close_grad(g_gpu, g_ref, name, what=""):
    rms = float(np.sqrt(np.mean(g_ref ** 2))) if g_ref.size else 0.0
    err = float(np.max(np.abs(np64(g_gpu) - g_ref))) if g_ref.size else 0.0
    bound = TOL_GRAD_REL_RMS * rms if rms > 0 else ZERO_GRAD_FLOOR
    assert err <= bound, (
        f"{what} {name} max-abs error {err:.3e} > {TOL_GRAD_REL_RMS} * rms {rms:.3e}")
    return err, rms
