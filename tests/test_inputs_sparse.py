"""The sparse top-k list generator follows its stated recipe (CPU only): the
window part, visibility of the compressed rows, list lengths, order and
distinct entries; the workload shapes match Table 7's cr4 rows."""
import torch

from attention_fwd_bwd_gb300.inputs import SPARSE_BY_NAME, make_sparse_index, make_sparse_inputs


def test_sparse_index_recipe():
    T, W, topk, ratio = 600, 16, 40, 4
    idx = make_sparse_index(T, W, topk, ratio, torch.Generator().manual_seed(5))
    assert idx.shape == (T, W + topk) and idx.dtype == torch.int32
    for t in range(T):
        win = idx[t, :W].tolist()
        assert win == [x if x >= 0 else -1 for x in range(t - W + 1, t + 1)]
        comp = [x for x in idx[t, W:].tolist()]
        filled = [x for x in comp if x >= 0]
        assert comp[:len(filled)] == filled          # filled entries first, -1 after
        assert all(x == -1 for x in comp[len(filled):])
        n_vis = (t + 1) // ratio
        assert len(filled) == min(topk, n_vis)
        assert filled == sorted(set(filled))          # ascending and distinct
        for x in filled:
            c = x - T
            assert 0 <= c and (c + 1) * ratio <= t + 1  # a compressed row whose tokens end by t
        if n_vis <= topk:
            assert filled == [T + c for c in range(n_vis)]


def test_sparse_index_picks_vary():
    T, W, topk, ratio = 2048, 8, 16, 4
    idx = make_sparse_index(T, W, topk, ratio, torch.Generator().manual_seed(1))
    late = idx[T - 64:, W:]
    assert len({tuple(r) for r in late.tolist()}) > 60  # random subsets differ between tokens


def test_sparse_workload_shapes():
    pro, flash = SPARSE_BY_NAME["csa_pro_cr4_t16384"], SPARSE_BY_NAME["csa_flash_cr4_t8192"]
    assert (pro.H, pro.K, pro.window, pro.topk, pro.ratio) == (128, 1152, 128, 1024, 4)
    assert (flash.H, flash.K, flash.window, flash.topk, flash.ratio) == (64, 640, 128, 512, 4)
    assert pro.P == pro.T + pro.T // 4
    w = SPARSE_BY_NAME["csa_small_t512"]
    q, kp, vp, do, idx = make_sparse_inputs(w)
    assert q.shape == (w.B, w.T, w.H, w.DK) and kp.shape == (w.B, w.P, w.DK) and vp.shape == (w.B, w.P, w.DV)
    assert do.shape == (w.B, w.T, w.H, w.DV) and idx.shape == (w.B, w.T, w.K)
    assert int(idx.max()) < w.P and int(idx.min()) >= -1
    q2 = make_sparse_inputs(w)[0]
    assert torch.equal(q, q2)  # seeded
