"""Pins for the oracle's output un-tiling with the gate (no GPU).

The un-tiling is the step after the block-sparse forward in the tiled layer
path the FastVideo kernel page describes (fused tile_to_bhsd commit: Q, K, V
and the gate go into a tile buffer).  Pinned against: the oracle layout (the
un-tiling without a gate is its exact inverse on every token), torch's own
float32 product and bfloat16 rounding for the gated case, and the isolation of
padding rows.
"""
import numpy as np
import torch

import workloads as W


def _bits(x):
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_inverse_of_the_layout(oracle_mod):
    # linear ragged tiling and the video cube tiling: untile(layout(x)) == x
    g = torch.Generator().manual_seed(3)
    for r2t, bs, S, T in (W.linear_row_map(300, 64) + (300, 64),
                          W.video_cube_tiling((5, 6, 9), (2, 3, 4), 32)[:2] + (5 * 6 * 9, 32)):
        NT = int(bs.numel())
        x = torch.randn((2, S, 3, 16), generator=g).to(torch.bfloat16)
        tiled = oracle_mod.tile_layout(x, r2t, NT, T)
        back = oracle_mod.untile(tiled, None, r2t, S, T)
        assert np.array_equal(back, _bits(x))


def test_gate_is_one_rounded_product(oracle_mod):
    g = torch.Generator().manual_seed(4)
    r2t, bs = W.linear_row_map(200, 64)
    NT, S, T = int(bs.numel()), 200, 64
    o = torch.randn((1, 2, NT * T, 32), generator=g).to(torch.bfloat16)
    gate = (torch.rand((1, S, 2, 32), generator=g) * 4 - 2).to(torch.bfloat16)
    gate[0, :3, 0, :4] = torch.tensor([float("inf"), float("nan"), 0.0, -0.0])
    got = oracle_mod.untile(o, gate, r2t, S, T)
    # library reference: gather the rows with torch indexing, multiply in
    # float32 (exact for bf16 inputs), round with torch's bfloat16 cast
    valid = r2t >= 0
    rows = torch.nonzero(valid).flatten()
    toks = r2t[valid].long()
    ref = torch.zeros((1, S, 2, 32), dtype=torch.bfloat16)
    ref[0, toks] = (o[0, :, rows, :].permute(1, 0, 2).float() * gate[0, toks].float()).to(torch.bfloat16)
    r = _bits(ref)
    gf = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float()
    nan = torch.isnan(gf)
    assert torch.equal(nan, torch.isnan(ref.float()))
    assert np.array_equal(got[~nan.numpy()], r[~nan.numpy()])


def test_padding_rows_are_never_read(oracle_mod):
    g = torch.Generator().manual_seed(5)
    r2t, bs = W.linear_row_map(150, 64)
    NT, S, T = int(bs.numel()), 150, 64
    o = torch.randn((1, 1, NT * T, 16), generator=g).to(torch.bfloat16)
    a = oracle_mod.untile(W.pad_tile_major(o, bs, T, "zero"), None, r2t, S, T)
    b = oracle_mod.untile(W.pad_tile_major(o, bs, T, "naninf"), None, r2t, S, T)
    assert np.array_equal(a, b)
