"""GPU parity of sliding-window causal attention (query i sees keys
i-W+1..i) through attn_fwd_ex / attn_bwd_ex, against the fp64 oracle.

Windows smaller than, equal to and larger than a 128-key tile, windows that
are not multiples of the tile, a one-key window, and windows at least as long
as the sequence (which must equal plain causal attention) are compared element
by element on every output. One full-size workload (Llama-3-8B shape, window
128) is checked on sampled rows and keys.
"""
import numpy as np
import pytest
import torch

from attention_fwd_bwd_gb300.inputs import make_inputs
from oracle import attn_ref_bwd, attn_ref_fwd, attn_ref_keys_dkdv, attn_ref_rows_dq, attn_ref_rows_fwd
from tests.helpers import assert_close_fwd, assert_close_grad, gpu_fwd_bwd, np64

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, S, D, window
    (1, 2, 1, 300, 128, 128),
    (2, 4, 2, 256, 64, 64),
    (1, 2, 2, 200, 128, 1),
    (1, 2, 1, 640, 128, 200),
    (1, 3, 3, 129, 64, 77),
    (1, 4, 1, 512, 128, 257),
    (1, 2, 1, 256, 128, 1000),
    (1, 8, 2, 1024, 128, 384),
]


# residual=False: attn_fwd_ex without o_lo, then attn_bwd_ex without o_lo,
# whose Dvec comes from the windowed Dvec pass.
@pytest.mark.parametrize("residual", [True, False], ids=["residual", "plain"])
@pytest.mark.parametrize("B,Hq,Hkv,S,D,W", CASES)
def test_window_elementwise(B, Hq, Hkv, S, D, W, residual):
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=500 + S + W)
    got = gpu_fwd_bwd(q, k, v, do, True, scale, window=W, residual=residual)
    o_ref, lse_ref = attn_ref_fwd(np64(q), np64(k), np64(v), True, scale, window=W)
    dq_ref, dk_ref, dv_ref = attn_ref_bwd(np64(q), np64(k), np64(v), np64(do), True, scale, window=W)
    what = f"B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} window={W} residual={residual}"
    assert_close_fwd(got["o"], got["lse"], o_ref, lse_ref, what)
    assert_close_grad(got["dq"], dq_ref, "dQ", what)
    assert_close_grad(got["dk"], dk_ref, "dK", what)
    assert_close_grad(got["dv"], dv_ref, "dV", what)


def test_window_of_sequence_length_is_plain_causal():
    B, Hq, Hkv, S, D = 1, 2, 1, 384, 128
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=77)
    a = gpu_fwd_bwd(q, k, v, do, True, 0.088, window=S)
    b = gpu_fwd_bwd(q, k, v, do, True, 0.088)
    for n in ("o", "lse", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n
    assert torch.allclose(a["dq"], b["dq"], rtol=0, atol=1e-6)


def test_window_full_size_sampled():
    # Llama-3-8B shape with a 128-key window, at full size.
    B, Hq, Hkv, S, D, W = 2, 32, 8, 4096, 128, 128
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=4242)
    got = gpu_fwd_bwd(q, k, v, do, True, scale, window=W)
    qf, kf, vf, df = (t.float().numpy() for t in (q, k, v, do))
    rng = np.random.default_rng(4242)
    rows = [(int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(S))) for _ in range(48)]
    rows[0], rows[1] = (0, 0, 0), (B - 1, Hq - 1, S - 1)
    o_ref, lse_ref = attn_ref_rows_fwd(qf, kf, vf, True, scale, rows, window=W)
    dq_ref = attn_ref_rows_dq(qf, kf, vf, df, True, scale, rows, window=W)
    o_g = np.stack([np64(got["o"][b, i, h]) for b, h, i in rows])
    l_g = np.array([float(got["lse"][b, h, i]) for b, h, i in rows])
    dq_g = np.stack([np64(got["dq"][b, i, h]) for b, h, i in rows])
    assert_close_fwd(o_g, l_g, o_ref, lse_ref, "window full size")
    assert_close_grad(dq_g, dq_ref, "dQ rows", "window full size")
    b, g = 1, 5
    keys = sorted({0, 127, 128, 2000, 4095} | {int(x) for x in rng.integers(S, size=11)})
    dk_ref, dv_ref = attn_ref_keys_dkdv(qf, kf, vf, df, True, scale, b, g, keys, window=W)
    assert_close_grad(np64(got["dk"][b, keys, g]), dk_ref, "dK keys", "window full size")
    assert_close_grad(np64(got["dv"][b, keys, g]), dv_ref, "dV keys", "window full size")
