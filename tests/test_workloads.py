"""Shape and structure checks of the seeded workloads (no GPU)."""
import math

import torch

import workloads as W


def test_tiny_and_uniform_shapes():
    w = W.make_workload(1)
    assert (w.B, w.H, w.D, w.T, w.NT, w.max_kv) == (1, 2, 64, 64, 4, 2)
    assert (w.block_sizes == 64).all() and (w.q2k_num == 2).all()
    assert abs(w.scale - 1 / 8) < 1e-15 and not w.want_lse
    for b, h, t in zip(*torch.nonzero(w.q2k_num >= 0, as_tuple=True)):
        sel = w.q2k_idx[b, h, t].tolist()
        assert len(set(sel)) == 2 and all(0 <= j < 4 for j in sel)
    assert W.effective_flops(w) == 4 * 64 * 64 * 64 * 2 * 4 * 2


def test_ragged_structure():
    w = W.make_workload(3)
    assert (w.B, w.H, w.D, w.T, w.NT) == (2, 8, 64, 64, 63)
    assert int(w.block_sizes.min()) >= 1 and int(w.block_sizes.max()) <= 64
    frac_empty = float((w.q2k_num == 0).float().mean())
    assert 0.05 < frac_empty < 0.2
    assert int(w.q2k_num.max()) <= round(0.5 * 63)
    # padding rows hold NaN / +Inf / -Inf, valid rows are finite
    Sp = w.Sp
    pos = torch.arange(Sp) % 64
    valid = pos < w.block_sizes[torch.arange(Sp) // 64]
    for x in (w.q, w.k, w.v):
        assert torch.isfinite(x[:, :, valid].float()).all()
        assert not torch.isfinite(x[:, :, ~valid].float()).any()
    assert w.notes["scaled_k_elements"] > 0


def test_video_topk_geometry():
    w = W.make_workload(4)
    assert w.NT == 336 and w.S == 32760 and int(w.block_sizes.sum()) == 32760
    assert set(w.block_sizes.tolist()) <= {8, 16, 32, 64, 128}
    assert int((w.block_sizes == 128).sum()) == 210
    assert (w.q2k_num == 42).all()
    for b, h, t in [(0, 0, 0), (0, 11, 335), (0, 5, 100)]:
        assert len(set(w.q2k_idx[b, h, t].tolist())) == 42


def test_dense_limit_shape():
    w = W.make_workload(5)
    assert (w.B, w.H, w.D, w.T, w.NT, w.S) == (1, 6, 128, 128, 244, 31200)
    assert int(w.block_sizes[-1]) == 96 and (w.block_sizes[:-1] == 128).all()
    assert (w.q2k_num == 244).all() and w.want_lse
    assert W.effective_flops(w) == 4 * 31200 ** 2 * 128 * 6


def test_seeded_determinism():
    a, b = W.make_workload(3), W.make_workload(3)
    assert torch.equal(a.q2k_idx, b.q2k_idx)
    assert a.q.view(torch.int16).equal(b.q.view(torch.int16))
