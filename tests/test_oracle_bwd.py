"""Pins for the oracle's block-sparse backward (no GPU).

The gradients are those of the forward on the FastVideo kernel page (the
Attn-QAT SM100 commit names the backward pass).  Pinned against torch autograd
in float64 on a dense attention with an explicit 0/1 mask (a library routine),
against a directional finite difference of the oracle's own forward (a
mathematical identity, independent of autograd), and against the isolation
of NaN/Inf padding and of keys no row selects.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W


def _case(seed, B=1, H=2, NT=4, T=8, D=8, pad="naninf"):
    g = torch.Generator().manual_seed(seed)
    bs = torch.randint(0, T + 1, (NT,), generator=g).to(torch.int32)
    bs[0] = T
    counts = torch.randint(0, NT + 1, (B, H, NT), generator=g).to(torch.int32)
    idx = W.random_selection(g, B, H, NT, counts, NT)
    q, k, v, do = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(4))
    if pad:
        q, k, v, do = (W.pad_tile_major(x, bs, T, pad) for x in (q, k, v, do))
    return q, k, v, do, idx, counts, bs


def _mask(idx, counts, bs, T):
    B, H, NT, _ = idx.shape
    Sp = NT * T
    tile = np.arange(Sp) // T
    valid = (np.arange(Sp) % T) < bs.numpy()[tile]
    M = np.zeros((B, H, Sp, Sp), dtype=bool)
    for b in range(B):
        for h in range(H):
            sel = np.zeros((NT, NT), dtype=bool)
            for t in range(NT):
                for i in range(int(counts[b, h, t])):
                    sel[t, int(idx[b, h, t, i])] = True
            M[b, h] = sel[tile][:, tile] & valid[:, None] & valid[None, :]
    return torch.from_numpy(M)


@pytest.mark.parametrize("seed,T,D,NT", [(0, 8, 8, 4), (1, 4, 16, 5), (2, 16, 8, 3)])
def test_matches_torch_autograd(oracle_mod, seed, T, D, NT):
    q, k, v, do, idx, counts, bs = _case(seed, NT=NT, T=T, D=D)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = oracle_mod.block_sparse_attention_bwd(q, k, v, do, idx, counts, bs, T, scale, nthreads=2)
    M = _mask(idx, counts, bs, T)
    # autograd reference on the padding-free values (padding rows zeroed; they
    # are masked out of every score, so their values do not matter)
    zq, zk, zv, zd = (W.pad_tile_major(x, bs, T, "zero").double() for x in (q, k, v, do))
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (zq, zk, zv))
    s = scale * qq @ kk.transpose(-1, -2)
    s = s.masked_fill(~M, float("-inf"))
    has = M.any(-1, keepdim=True)
    p = torch.where(has, torch.softmax(torch.where(has, s, torch.zeros_like(s)), -1), torch.zeros_like(s))
    p = torch.where(M, p, torch.zeros_like(p))
    out = p @ vv
    out.backward(zd)
    for got, ref, name in ((dq, qq.grad, "dq"), (dk, kk.grad, "dk"), (dv, vv.grad, "dv")):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-9, atol=1e-11, err_msg=name)


def test_directional_finite_difference(oracle_mod):
    # L(q, k, v) = sum(dout * out(q, k, v)); for a direction u in q (and in k,
    # v), (L(x + eps u) - L(x - eps u)) / (2 eps) = <grad, u> up to O(eps^2).
    # Inputs are bf16, so the direction only touches entries whose perturbed
    # values stay exactly representable.
    q, k, v, do, idx, counts, bs = _case(7, NT=3, T=8, D=8, pad=None)
    T, scale = 8, 1.0 / math.sqrt(8)
    dq, dk, dv = oracle_mod.block_sparse_attention_bwd(q, k, v, do, idx, counts, bs, T, scale, nthreads=1)
    dof = do.double().numpy()

    def loss(q_, k_, v_):
        out, _ = oracle_mod.block_sparse_attention(q_, k_, v_, idx, counts, bs, T, scale, nthreads=1)
        B, H, Sp, D = q_.shape
        return float((out.reshape(B, H, Sp, D) * dof).sum())

    g = torch.Generator().manual_seed(9)
    eps = 2.0 ** -6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        base = [q, k, v][which].float()
        # entries in [0.5, 1): bf16 spacing there is 2^-8, so x +- eps stays exact
        cand = torch.nonzero(((base.abs() >= 0.5) & (base.abs() < 1.0)).view(-1)).flatten()
        pick = cand[torch.randperm(cand.numel(), generator=g)[:6]]
        u = torch.zeros_like(base)
        u.view(-1)[pick] = 1.0
        plus, minus = base + eps * u, base - eps * u
        assert torch.equal(plus.to(torch.bfloat16).float(), plus)
        assert torch.equal(minus.to(torch.bfloat16).float(), minus)
        args_p, args_m = [q, k, v], [q, k, v]
        args_p[which], args_m[which] = plus.to(torch.bfloat16), minus.to(torch.bfloat16)
        fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        an = float((grad * u.double().numpy()).sum())
        assert abs(an) > 1e-3, "the direction must carry gradient"
        assert abs(fd - an) <= 2e-3 * max(1.0, abs(an)), (which, fd, an)


def test_padding_and_unselected_keys(oracle_mod):
    q, k, v, do, idx, counts, bs = _case(3, NT=5, T=8, D=8)
    scale = 0.3
    a = oracle_mod.block_sparse_attention_bwd(q, k, v, do, idx, counts, bs, 8, scale, nthreads=2)
    z = [W.pad_tile_major(x, bs, 8, "zero") for x in (q, k, v, do)]
    b = oracle_mod.block_sparse_attention_bwd(*z, idx, counts, bs, 8, scale, nthreads=2)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)               # padding never read
        assert np.isfinite(x).all()
    # keys that no query tile selects get zero dk, dv; padding rows are zero
    B, H, NT = counts.shape
    for bb in range(B):
        for h in range(H):
            chosen = set()
            for t in range(NT):
                chosen |= set(idx[bb, h, t, :int(counts[bb, h, t])].tolist())
            for j in range(NT):
                rows = slice(j * 8, (j + 1) * 8)
                if j not in chosen:
                    assert (a[1][bb, h, rows] == 0).all() and (a[2][bb, h, rows] == 0).all()
                assert (a[0][bb, h, j * 8 + int(bs[j]):(j + 1) * 8] == 0).all()
