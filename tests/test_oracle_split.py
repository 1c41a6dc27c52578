"""The split tail's combine, on the oracle (no GPU).

When the last wave of work items leaves SMs idle, the forward cuts a
128-row unit's selected key tiles into ranges by tile index (range p of np:
[floor(p NT / np), floor((p+1) NT / np)), bounds rounded down to even, the
last ending at NT), computes each range on its own, and merges the ranges
(the flash-decoding split-K combine).  Attention over a union of disjoint key
sets is the LSE-weighted mix of the attention over each set:
    LSE = log sum_r exp(LSE_r),   O = sum_r exp(LSE_r - LSE) O_r,
which is the kernel's merge of (unnormalised O_r, row maximum m_r, row sum
l_r) written with LSE_r = ln(l_r) + m_r ln 2.  Here the FP64 oracle is run
once on each range's selections and once on the whole selections, and the
combine of the former must give the latter, including rows whose ranges are
all empty (+0, LSE -inf), ranges with no selected tile, and a NaN in a valid
key (a NaN row on both sides).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W


def _ranges(NT, parts):
    """The forward's key-tile ranges for `parts` cuts of NT kernel tiles."""
    out = []
    for p in range(parts):
        lo = (p * NT // parts) & ~1
        hi = NT if p + 1 == parts else ((p + 1) * NT // parts) & ~1
        out.append((lo, hi))
    return out


def _restrict(idx, num, lo, hi):
    """Each row's selections inside [lo, hi), compacted to the front."""
    B, H, NT, K = idx.shape
    ri = torch.full_like(idx, -1)
    rn = torch.zeros_like(num)
    for b in range(B):
        for h in range(H):
            for t in range(NT):
                sel = [int(j) for j in idx[b, h, t, :int(num[b, h, t])] if lo <= int(j) < hi]
                rn[b, h, t] = len(sel)
                if sel:
                    ri[b, h, t, :len(sel)] = torch.tensor(sel, dtype=idx.dtype)
    return ri, rn


@pytest.mark.parametrize("parts", [2, 3, 8])
def test_key_range_combine_matches_whole(oracle_mod, parts):
    B, H, NT, T, D = 1, 2, 11, 128, 64
    g = torch.Generator().manual_seed(40 + parts)
    bs = torch.randint(1, T + 1, (NT,), generator=g).int()
    bs[3] = 0                                            # an empty tile
    counts = torch.randint(0, 5, (B, H, NT), generator=g).int()
    counts[0, 0, 0] = 0                                  # a row with no selection
    idx = W.random_selection(g, B, H, NT, counts, 5)
    q, k, v = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(3))
    k[0, 1, 7 * T + 2, 5] = float("nan")                 # a NaN in a valid key of tile 7, head 1
    if bs[7] < 3:
        bs[7] = 3
    if 7 not in idx[0, 1, 5, :int(counts[0, 1, 5])].tolist():   # query tile 5 of head 1 selects tile 7
        counts[0, 1, 5] = max(int(counts[0, 1, 5]), 1)
        idx[0, 1, 5, 0] = 7
    q, k, v = (W.pad_tile_major(x, bs, T, "naninf") for x in (q, k, v))
    scale = 1.0 / math.sqrt(D)
    ref, ref_lse = oracle_mod.block_sparse_attention(q, k, v, idx, counts, bs, T, scale)

    rng = _ranges(NT, parts)
    assert rng[0][0] == 0 and rng[-1][1] == NT
    assert all(a[1] == b[0] for a, b in zip(rng, rng[1:])), "ranges tile [0, NT)"
    outs, lses = [], []
    for lo, hi in rng:
        ri, rn = _restrict(idx, counts, lo, hi)
        o, l = oracle_mod.block_sparse_attention(q, k, v, ri, rn, bs, T, scale)
        outs.append(o)
        lses.append(l)
    L = np.stack(lses)                                   # [parts, units, T]
    with np.errstate(invalid="ignore", divide="ignore"):
        M = np.max(np.where(np.isnan(L), -np.inf, L), axis=0)
        lse = M + np.log(np.sum(np.exp(L - np.where(np.isfinite(M), M, 0.0)), axis=0))
        lse = np.where(np.isneginf(M), -np.inf, lse)
        lse = np.where(np.isnan(L).any(axis=0), np.nan, lse)
        w = np.exp(L - np.where(np.isfinite(lse), lse, 0.0)[None])
        w = np.where(np.isneginf(L), 0.0, w)
        out = np.einsum("put,putd->utd", w, np.stack(outs))
    out = np.where(np.isneginf(lse)[..., None], 0.0, out)

    ref_nan = np.isnan(ref).any(-1)
    assert ref_nan.any(), "the NaN key must reach some rows"
    np.testing.assert_array_equal(np.isnan(out).any(-1), ref_nan)
    np.testing.assert_array_equal(np.isnan(lse), np.isnan(ref_lse))
    ok = ~ref_nan
    np.testing.assert_allclose(out[ok], ref[ok], rtol=1e-12, atol=1e-12)
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    assert np.isneginf(ref_lse).any() and (ref[np.isneginf(ref_lse)] == 0).all()
