"""The bounds-checked build (libattn_debug.so, compiled with
-DATTN_DEBUG_BOUNDS) on the GPU: the dense kernels check their computed
indices (K/V tile and query-tile coordinates, ring stages, workspace rows,
dq reduction coordinates, dK/dV and LSE rows) and report ATTN_ERR_BOUNDS,
skipping the access, when one is out of range. On valid inputs no check may
fire, and the results must still match the fp64 oracle. This stands in for a
memory checker, which is not available here.
"""
import numpy as np
import pytest

import attention_fwd_bwd_gb300 as attn
from attention_fwd_bwd_gb300.inputs import make_inputs
from oracle import attn_ref_bwd, attn_ref_fwd
from tests.helpers import assert_close_fwd, assert_close_grad, gpu_fwd_bwd, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_library():
    from attention_fwd_bwd_gb300._build import build
    build(debug=True)
    attn.use_debug_library(True)
    try:
        yield
    finally:
        attn.use_debug_library(False)


CASES = [
    # B, Hq, Hkv, S, D, causal, window, residual
    (1, 2, 1, 300, 128, True, 0, True),     # ragged tail, GQA
    (2, 4, 2, 256, 64, True, 0, False),     # plain pair: the Dvec pass
    (1, 2, 2, 77, 128, False, 0, True),     # shorter than a tile, non-causal
    (1, 4, 1, 512, 128, True, 200, True),   # sliding window
    (1, 3, 3, 129, 64, True, 77, False),    # window, ragged, plain pair
    (1, 8, 2, 640, 128, True, 0, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,window,residual", CASES)
def test_bounds_checked_build_is_clean_and_correct(debug_library, B, Hq, Hkv, S, D, causal, window,
                                                   residual):
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, Hq, Hkv, S, D, seed=900 + S + D)
    # gpu_fwd_bwd asserts that attn_check_status reports ATTN_OK (no check fired).
    got = gpu_fwd_bwd(q, k, v, do, causal, scale, window=window, residual=residual)
    o_ref, lse_ref = attn_ref_fwd(np64(q), np64(k), np64(v), causal, scale, window=window)
    dq_ref, dk_ref, dv_ref = attn_ref_bwd(np64(q), np64(k), np64(v), np64(do), causal, scale,
                                          window=window)
    what = f"debug build B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal} W={window} residual={residual}"
    assert_close_fwd(got["o"], got["lse"], o_ref, lse_ref, what)
    assert_close_grad(got["dq"], dq_ref, "dQ", what)
    assert_close_grad(got["dk"], dk_ref, "dK", what)
    assert_close_grad(got["dv"], dv_ref, "dV", what)
