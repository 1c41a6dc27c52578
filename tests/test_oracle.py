"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a
hand-worked example with closed-form values, dense softmax attention from a
library routine, a brute-force masked softmax over an explicit mask matrix,
exact special cases, and the invariants the FastVideo kernel page states for
the block-sparse forward (hao-ai-lab/FastVideo commit 8503617,
fastvideo-kernel/python: empty selections give 0, NaN/Inf padding never reaches
the output, a NaN softmax sum gives a NaN row).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float64), dtype=torch.float32).to(torch.bfloat16)


def _to_f(x):
    return {"nan": math.nan, "inf": math.inf, "-inf": -math.inf}.get(x, x) if isinstance(x, str) else x


def _closed(expr):
    return float(eval(expr, {"__builtins__": {}}, {"e": math.e, "log": math.log, "inf": math.inf}))


def _random_problem(seed, B=1, H=2, NT=4, T=8, D=8, full=False, empty_frac=0.2, pad="naninf"):
    g = torch.Generator().manual_seed(seed)
    if full:
        bs = torch.full((NT,), T, dtype=torch.int32)
    else:
        bs = torch.randint(0, T + 1, (NT,), generator=g).to(torch.int32)
        bs[0] = T
    counts = torch.randint(0, NT + 1, (B, H, NT), generator=g).to(torch.int32)
    counts[torch.rand((B, H, NT), generator=g) < empty_frac] = 0
    idx = W.random_selection(g, B, H, NT, counts, NT)
    q, k, v = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(3))
    if not full and pad:
        q, k, v = (W.pad_tile_major(x, bs, T, pad) for x in (q, k, v))
    return q, k, v, idx, counts, bs


def _bruteforce(q, k, v, idx, counts, bs, T, scale):
    """Dense masked softmax over an explicit 0/1 mask matrix (FP64 numpy):
    M[row, col] = 1 iff row is a valid query row, col is a valid key row, and
    col's tile is in row's tile selection.  Fully masked rows give 0 and
    lse = -inf.  Scores of masked pairs are never formed, so NaN padding does
    not enter."""
    from scipy.special import logsumexp
    B, H, Sp, D = q.shape
    NT = Sp // T
    qf, kf, vf = (x.double().numpy() for x in (q, k, v))
    tile = np.arange(Sp) // T
    pos = np.arange(Sp) % T
    valid = pos < bs.numpy()[tile]
    out = np.zeros((B, H, Sp, D))
    lse = np.full((B, H, Sp), -np.inf)
    for b in range(B):
        for h in range(H):
            sel = np.zeros((NT, NT), dtype=bool)
            for t in range(NT):
                for i in range(int(counts[b, h, t])):
                    sel[t, int(idx[b, h, t, i])] = True
            M = sel[tile][:, tile] & valid[:, None] & valid[None, :]
            for r in range(Sp):
                cols = np.nonzero(M[r])[0]
                if cols.size == 0:
                    continue
                s = scale * (kf[b, h, cols] @ qf[b, h, r])
                w = np.exp(s - s.max())
                out[b, h, r] = (w @ vf[b, h, cols]) / w.sum()
                lse[b, h, r] = logsumexp(s)
    return out, lse


def _oracle_full(oracle_mod, q, k, v, idx, counts, bs, T, scale):
    B, H, Sp, D = q.shape
    out, lse = oracle_mod.block_sparse_attention(q, k, v, idx, counts, bs, T, scale, nthreads=2)
    return out.reshape(B, H, Sp, D), lse.reshape(B, H, Sp)


def test_golden_hand_worked(oracle_mod):
    with open(os.path.join(GOLDEN, "hand_worked_2x2.json")) as f:
        G = json.load(f)
    conv = lambda a: _bf16(np.vectorize(_to_f, otypes=[float])(np.array(a, dtype=object)))
    q, k, v = conv(G["q"]), conv(G["k"]), conv(G["v"])
    out, lse = _oracle_full(oracle_mod, q, k, v, torch.tensor(G["q2k_idx"], dtype=torch.int32),
                            torch.tensor(G["q2k_num"], dtype=torch.int32),
                            torch.tensor(G["block_sizes"], dtype=torch.int32), G["T"], G["scale"])
    exp_out = np.vectorize(_closed)(np.array(G["expected_out"], dtype=object)).astype(float)
    exp_lse = np.vectorize(_closed)(np.array(G["expected_lse"], dtype=object)).astype(float)
    np.testing.assert_allclose(out, exp_out, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(exp_lse))
    fin = np.isfinite(exp_lse)
    np.testing.assert_allclose(lse[fin], exp_lse[fin], rtol=0, atol=1e-14)
    # padding and empty rows are exactly +0.0
    zero_rows = (exp_out == 0).all(-1)
    assert not np.signbit(out[zero_rows]).any()


@pytest.mark.parametrize("seed", [0, 1])
def test_dense_equals_sdpa(oracle_mod, seed):
    """Every tile selected and full: the oracle is dense softmax attention
    (torch's scaled_dot_product_attention in float64 on the CPU)."""
    B, H, NT, T, D = 1, 2, 4, 8, 16
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(3))
    bs = torch.full((NT,), T, dtype=torch.int32)
    counts = torch.full((B, H, NT), NT, dtype=torch.int32)
    idx = torch.stack([torch.randperm(NT, generator=g) for _ in range(B * H * NT)]).view(B, H, NT, NT).int()
    scale = 1.0 / math.sqrt(D)
    out, lse = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, T, scale)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double(), scale=scale)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)
    ref_lse = torch.logsumexp(scale * q.double() @ k.double().transpose(-1, -2), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed,T,D,NT", [(0, 4, 4, 3), (1, 8, 8, 4), (2, 8, 4, 5), (3, 4, 8, 6)])
def test_bruteforce_masked(oracle_mod, seed, T, D, NT):
    q, k, v, idx, counts, bs = _random_problem(seed, B=2, H=2, NT=NT, T=T, D=D)
    scale = 0.7
    out, lse = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, T, scale)
    ref, ref_lse = _bruteforce(q, k, v, idx, counts, bs, T, scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)


def test_empty_selection_is_exact_zero(oracle_mod):
    q, k, v, idx, counts, bs = _random_problem(5, NT=4, T=8, D=8)
    counts[:] = 0
    out, lse = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, 8, 0.5)
    assert (out == 0).all() and not np.signbit(out).any()
    assert np.isneginf(lse).all()


def test_permutation_invariance(oracle_mod):
    q, k, v, idx, counts, bs = _random_problem(6, NT=6, T=8, D=8, empty_frac=0.0)
    out, lse = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, 8, 0.4)
    g = torch.Generator().manual_seed(99)
    idx2 = idx.clone()
    for b, h, t in np.ndindex(*counts.shape):
        c = int(counts[b, h, t])
        idx2[b, h, t, :c] = idx[b, h, t, :c][torch.randperm(c, generator=g)]
    out2, lse2 = _oracle_full(oracle_mod, q, k, v, idx2, counts, bs, 8, 0.4)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)


def test_padding_values_never_reach_output(oracle_mod):
    q, k, v, idx, counts, bs = _random_problem(7, NT=5, T=8, D=8, pad="zero")
    a = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, 8, 0.5)
    qn, kn, vn = (W.pad_tile_major(x, bs, 8, "naninf") for x in (q, k, v))
    b = _oracle_full(oracle_mod, qn, kn, vn, idx, counts, bs, 8, 0.5)
    assert a[0].tobytes() == b[0].tobytes() and a[1].tobytes() == b[1].tobytes()


def test_single_key_gives_its_value(oracle_mod):
    """A key list holding one valid key: softmax of one element is 1, so the
    output row is that key's value row exactly and lse is its score."""
    q, k, v, idx, counts, bs = _random_problem(8, NT=3, T=4, D=8, full=True)
    bs[2] = 1
    counts[:] = 1
    idx[:] = -1
    idx[..., 0] = 2
    out, lse = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, 4, 0.3)
    vrow = v[:, :, 8, :].double().numpy()
    for r in range(12):
        if r >= 8 and r % 4 >= 1:
            continue
        np.testing.assert_array_equal(out[:, :, r, :], vrow)
        s = 0.3 * (q[:, :, r, :].double() * k[:, :, 8, :].double()).sum(-1).numpy()
        np.testing.assert_allclose(lse[:, :, r], s, rtol=0, atol=1e-13)


def test_equal_scores_give_mean_of_values(oracle_mod):
    """All valid K rows zero: every score is 0, so each output row is the plain
    mean of the valid V rows of its selected tiles."""
    q, k, v, idx, counts, bs = _random_problem(9, NT=4, T=8, D=8, empty_frac=0.0)
    k = torch.zeros_like(k)
    out, lse = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, 8, 1.0)
    vf = v.double().numpy()
    for b, h, t in np.ndindex(*counts.shape):
        rows = [j * 8 + c for j in idx[b, h, t, :int(counts[b, h, t])].tolist() for c in range(int(bs[j]))]
        for r in range(int(bs[t])):
            if not rows:
                assert (out[b, h, t * 8 + r] == 0).all()
                continue
            np.testing.assert_allclose(out[b, h, t * 8 + r], vf[b, h, rows].mean(0), rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[b, h, t * 8 + r], math.log(len(rows)), rtol=0, atol=1e-13)


def test_nan_score_gives_nan_row(oracle_mod):
    """A NaN inside a valid K row makes that key's score NaN for every query
    row that selects its tile: the softmax sum is NaN, so the whole output row
    is NaN; rows that do not select the tile are unaffected."""
    q, k, v, idx, counts, bs = _random_problem(10, NT=4, T=8, D=8, full=True, empty_frac=0.0)
    ref = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, 8, 0.5)
    k[0, 0, 8 + 3, 5] = float("nan")         # tile 1, row 3 of head (0, 0)
    out, lse = _oracle_full(oracle_mod, q, k, v, idx, counts, bs, 8, 0.5)
    for t in range(4):
        sel = idx[0, 0, t, :int(counts[0, 0, t])].tolist()
        rows = slice(t * 8, t * 8 + 8)
        if 1 in sel:
            assert np.isnan(out[0, 0, rows]).all() and np.isnan(lse[0, 0, rows]).all()
        else:
            np.testing.assert_array_equal(out[0, 0, rows], ref[0][0, 0, rows])
    np.testing.assert_array_equal(out[0, 1], ref[0][0, 1])


def test_rejects_bad_selection(oracle_mod):
    q, k, v, idx, counts, bs = _random_problem(11, NT=4, T=4, D=4, empty_frac=0.0)
    counts[0, 0, 0] = 2
    bad = idx.clone()
    bad[0, 0, 0, :2] = torch.tensor([1, 1])
    with pytest.raises(ValueError):
        oracle_mod.block_sparse_attention(q, k, v, bad, counts, bs, 4, 1.0)
    bad[0, 0, 0, :2] = torch.tensor([0, 4])
    with pytest.raises(ValueError):
        oracle_mod.block_sparse_attention(q, k, v, bad, counts, bs, 4, 1.0)


def test_unit_subset_matches_full(oracle_mod):
    q, k, v, idx, counts, bs = _random_problem(12, B=2, H=2, NT=5, T=8, D=8)
    full, full_lse = oracle_mod.block_sparse_attention(q, k, v, idx, counts, bs, 8, 0.5, nthreads=3)
    units = [19, 0, 7, 7]
    sub, sub_lse = oracle_mod.block_sparse_attention(q, k, v, idx, counts, bs, 8, 0.5, units=units)
    np.testing.assert_array_equal(sub, full[units])
    np.testing.assert_array_equal(sub_lse, full_lse[units])


def test_layout_matches_index_gather(oracle_mod):
    """The layout oracle against numpy fancy indexing on the video-cube
    geometry (every token lands in exactly one row; padding rows are +0)."""
    r2t, bs, _, _ = W.video_cube_tiling((5, 6, 9), (2, 2, 4), 16)
    NT, T = int(bs.numel()), 16
    S = 5 * 6 * 9
    toks = r2t[r2t >= 0].numpy()
    assert sorted(toks.tolist()) == list(range(S))
    g = torch.Generator().manual_seed(3)
    x = torch.randn((2, S, 3, 8), generator=g).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.tile_layout(x, r2t, NT, T)
    m = r2t.numpy().astype(np.int64)
    ref = bits[:, np.clip(m, 0, None), :, :].transpose(0, 2, 1, 3).copy()
    ref[:, :, m < 0, :] = 0
    np.testing.assert_array_equal(got, ref)
    for t in range(NT):
        assert (r2t[t * T: t * T + int(bs[t])] >= 0).all() and (r2t[t * T + int(bs[t]): (t + 1) * T] == -1).all()
