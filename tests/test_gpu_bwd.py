"""GPU parity of the block-sparse backward (through the C ABI) against the
FP64 oracle backward.

The GPU backward takes the GPU forward's bf16 output and LSE, forms P and dS
in bf16 for the tensor cores and accumulates in fp32; the oracle recomputes
everything in FP64.  The bar follows from that arithmetic.  With u = 2^-8,
the unit roundoff of bf16 (round to nearest), every term of a gradient sum
(p dout for dV, scale ds q for dK, scale ds k for dQ) reaches the GPU sum
through at most three roundings of relative size u: P or dS rounded to
bf16, the forward's LSE (l sums bf16-rounded P, so lse is off by up to
ln(1 + u), i.e. p by a factor within 1 +- u), and the bf16 output of the
gradient itself.  dS also carries the error of delta = rowsum(dout * out)
taken from the bf16-rounded out, at most u * sum_d |dout_d out_d| per row.
fp32 accumulation adds only O(2^-24) per term.  So element by element

    |gpu - ref| <= 3u * A,

where A is the same sum over the absolute values of its terms (with the
delta error added to |ds|), computed here in float64 from the same inputs.
The tensor-level relative RMS error is one such rounding on average, u/sqrt(3)
= 2.26e-3 for independent errors; the bar is u (3.9e-3).  Padding rows and
keys no row selects must be exactly +0.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

U = 2.0 ** -8      # bf16 unit roundoff (round to nearest)
REL_RMS = U        # tensor-level relative RMS error
ELEM = 3 * U       # per element, times the sum of the absolute values of the terms


@pytest.fixture(scope="module")
def vsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_gathered_gb300 as V
    assert V.vsa_check_device_status() == 0
    return V


def _case(seed, B, H, NT, D, T=128, full=False, pad="naninf", empty_frac=0.1):
    g = torch.Generator().manual_seed(seed)
    bs = torch.full((NT,), T, dtype=torch.int32) if full else torch.randint(1, T + 1, (NT,), generator=g).int()
    if not full:
        bs[torch.rand(NT, generator=g) < 0.1] = 0
        bs[NT // 2] = T
    counts = torch.full((B, H, NT), NT, dtype=torch.int32) if full else \
        torch.randint(0, NT + 1, (B, H, NT), generator=g).int()
    if not full:
        counts[torch.rand((B, H, NT), generator=g) < empty_frac] = 0
    idx = W.random_selection(g, B, H, NT, counts, NT)
    q, k, v, do = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(4))
    if not full and pad:
        q, k, v, do = (W.pad_tile_major(x, bs, T, pad) for x in (q, k, v, do))
    return q, k, v, do, idx, counts, bs


def _structural_zero_tiles(idx, counts, bs):
    """[B, H, NT] masks of the tiles whose gradient rows are 0 by the selection
    alone: query tiles with no non-empty key tile (dq), and key tiles that no
    non-empty query tile selects (dk, dv).  Rows whose reference is 0 only by
    cancellation (one key: dout.v = delta) are held to the tolerance instead."""
    B, H, NT, _ = idx.shape
    n = bs.numpy()
    q_zero = np.ones((B, H, NT), dtype=bool)
    k_zero = np.ones((B, H, NT), dtype=bool)
    for b in range(B):
        for h in range(H):
            for t in range(NT):
                for j in idx[b, h, t, :int(counts[b, h, t])].tolist():
                    if n[j] > 0 and n[t] > 0:
                        q_zero[b, h, t] = False
                        k_zero[b, h, j] = False
    return q_zero, k_zero


def _abs_term_sums(q, k, v, do, idx, counts, bs, T, scale):
    """float64 sums of the absolute values of the terms of dq, dk and dv (the
    A of the element-wise bar), from a dense attention with an explicit
    selection mask; padding rows are excluded."""
    B, H, Sp, D = q.shape
    n = bs.numpy()
    rows = np.arange(Sp)
    valid = (rows % T) < n[rows // T]
    f = lambda x: np.where(valid[None, None, :, None], x.float().numpy().astype(np.float64), 0.0)
    qd, kd, vd, dod = f(q), f(k), f(v), f(do)
    A_dq, A_dk, A_dv = np.zeros_like(qd), np.zeros_like(qd), np.zeros_like(qd)
    for b in range(B):
        for h in range(H):
            sel = np.zeros((Sp // T, Sp // T), dtype=bool)
            for t in range(Sp // T):
                sel[t, idx[b, h, t, :int(counts[b, h, t])].numpy()] = True
            mask = sel[rows[:, None] // T, rows[None, :] // T] & valid[:, None] & valid[None, :]
            s = np.where(mask, scale * qd[b, h] @ kd[b, h].T, -np.inf)
            mrow = s.max(1, keepdims=True)
            mrow[~np.isfinite(mrow)] = 0.0
            e = np.where(mask, np.exp(s - mrow), 0.0)
            lrow = e.sum(1, keepdims=True)
            p = np.where(lrow > 0, e / np.where(lrow > 0, lrow, 1.0), 0.0)
            out = p @ vd[b, h]
            dp = dod[b, h] @ vd[b, h].T
            delta = (p * dp).sum(1, keepdims=True)
            ds = np.abs(p * (dp - delta)) + p * U * (np.abs(dod[b, h]) * np.abs(out)).sum(1, keepdims=True)
            A_dv[b, h] = p.T @ np.abs(dod[b, h])
            A_dk[b, h] = scale * ds.T @ np.abs(qd[b, h])
            A_dq[b, h] = scale * ds @ np.abs(kd[b, h])
    return A_dq, A_dk, A_dv


def _check(name, got, ref, bs, T, zero_tiles, A):
    g = got.float().cpu().numpy().astype(np.float64)
    B, H, Sp, D = g.shape
    valid = (np.arange(Sp) % T) < bs.numpy()[np.arange(Sp) // T]
    assert (got[:, :, ~torch.from_numpy(valid)].view(torch.int16) == 0).all(), f"{name}: padding rows not +0"
    gv, rv, av = g[:, :, valid], ref[:, :, valid], A[:, :, valid]
    zero_rows = np.repeat(zero_tiles, T, axis=2)[:, :, valid]
    assert (rv[zero_rows] == 0).all(), f"{name}: oracle rows not 0 where the selection makes them 0"
    assert (gv[zero_rows] == 0).all(), f"{name}: rows that must be 0 are not"
    err = np.abs(gv - rv)
    rel = float(np.linalg.norm(gv - rv) / max(np.linalg.norm(rv), 1e-30))
    ratio = float((err / np.maximum(av, 1e-30)).max())  # of the element-wise bar, in units of A
    print(f"[bwd] {name}: rel rms {rel:.3e} (bar {REL_RMS:.2e}), max |err| / A {ratio:.3e} (bar {ELEM:.2e}), "
          f"max abs {float(err.max()):.3e}")
    assert rel <= REL_RMS, f"{name}: rel rms {rel:.3e}"
    bad = err > ELEM * av + 1e-7
    assert not bad.any(), f"{name}: {int(bad.sum())} elements beyond 3u * A (worst ratio {ratio:.3e})"


@pytest.mark.parametrize("B,H,NT,D,full,T", [
    (1, 2, 3, 128, True, 128), (2, 2, 5, 64, False, 128), (1, 3, 6, 128, False, 128),
    # 64-token tiles: two per kernel tile with a block mask; odd counts leave a half-empty last one
    (1, 2, 7, 64, False, 64), (2, 2, 9, 128, False, 64), (1, 2, 4, 64, True, 64),
    # 256-token tiles: two kernel tiles each
    (1, 2, 3, 128, False, 256), (1, 1, 2, 64, True, 256),
])
def test_bwd_matches_oracle(vsa, oracle_mod, B, H, NT, D, full, T):
    q, k, v, do, idx, counts, bs = _case(50 + NT + D + T, B, H, NT, D, T=T, full=full)
    dev = "cuda"
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    idd, cd, bsd = idx.to(dev), counts.to(dev), bs.to(dev)
    out, lse = vsa.block_sparse_attention(qd, kd, vd, idd, cd, bsd, T, want_lse=True)
    dq, dk, dv = vsa.block_sparse_attention_bwd(qd, kd, vd, out, dod, lse, idd, cd, bsd, T)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    r = vsa.vsa_last_route()
    assert r["kernel"] == vsa.VSA_KERNEL_BWD and r["tile"] == T and r["head_dim"] == D
    rq, rk, rv = oracle_mod.block_sparse_attention_bwd(q, k, v, do, idx, counts, bs, T, 1.0 / math.sqrt(D))
    label = f"B{B}H{H}NT{NT}D{D}T{T}{'dense' if full else 'ragged'}"
    q_zero, k_zero = _structural_zero_tiles(idx, counts, bs)
    A_dq, A_dk, A_dv = _abs_term_sums(q, k, v, do, idx, counts, bs, T, 1.0 / math.sqrt(D))
    _check(label + " dq", dq, rq, bs, T, q_zero, A_dq)
    _check(label + " dk", dk, rk, bs, T, k_zero, A_dk)
    _check(label + " dv", dv, rv, bs, T, k_zero, A_dv)


@pytest.mark.parametrize("T", [64, 128])
def test_bwd_deterministic(vsa, T):
    q, k, v, do, idx, counts, bs = _case(77, 1, 2, 6, 128, T=T)
    dev = "cuda"
    args = [x.to(dev) for x in (q, k, v)]
    idd, cd, bsd = idx.to(dev), counts.to(dev), bs.to(dev)
    out, lse = vsa.block_sparse_attention(*args, idd, cd, bsd, T, want_lse=True)
    a = vsa.block_sparse_attention_bwd(*args, out, do.to(dev), lse, idd, cd, bsd, T)
    b = vsa.block_sparse_attention_bwd(*args, out, do.to(dev), lse, idd, cd, bsd, T)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_bwd_odd_64_tiles_leave_next_head_alone(vsa):
    """With an odd count of 64-token tiles the last kernel tile of a head
    reaches 64 rows into the next head's rows; they must stay untouched."""
    B, H, NT, D, T = 1, 3, 5, 64, 64
    q, k, v, do, idx, counts, bs = _case(91, B, H, NT, D, T=T, full=True)
    dev = "cuda"
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    idd, cd, bsd = idx.to(dev), counts.to(dev), bs.to(dev)
    out, lse = vsa.block_sparse_attention(qd, kd, vd, idd, cd, bsd, T, want_lse=True)
    dq, dk, dv = vsa.block_sparse_attention_bwd(qd, kd, vd, out, dod, lse, idd, cd, bsd, T)
    # per-head results must not depend on the other heads: run each head alone
    for h in range(H):
        sl = slice(h, h + 1)
        o1, l1 = vsa.block_sparse_attention(qd[:, sl].contiguous(), kd[:, sl].contiguous(), vd[:, sl].contiguous(),
                                            idd[:, sl].contiguous(), cd[:, sl].contiguous(), bsd, T, want_lse=True)
        g1 = vsa.block_sparse_attention_bwd(qd[:, sl].contiguous(), kd[:, sl].contiguous(), vd[:, sl].contiguous(),
                                            o1, dod[:, sl].contiguous(), l1, idd[:, sl].contiguous(),
                                            cd[:, sl].contiguous(), bsd, T)
        for full_g, one in zip((dq, dk, dv), g1):
            assert torch.equal(full_g[:, sl].view(torch.int16), one.view(torch.int16)), f"head {h}"


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_t64_pair_isolation(vsa, oracle_mod, D):
    """64-token tiles share 128-row kernel tiles in pairs.  NaN in a VALID row
    of Q, K or dO reaches exactly the gradients the definition sends it to:
    query tile t selects key tiles t and t + 3 (of 6), so no key tile serves
    both tiles of a pair, and the partner's gradients (where a zero weight
    times NaN would otherwise be NaN) must stay finite and match the oracle.
    Every element's NaN-ness must match the oracle's."""
    B, H, NT, T = 1, 2, 6, 64
    g = torch.Generator().manual_seed(4100 + D)
    bs = torch.full((NT,), T, dtype=torch.int32)
    idx = torch.empty((B, H, NT, 2), dtype=torch.int32)
    for t in range(NT):
        idx[:, :, t, 0] = t
        idx[:, :, t, 1] = (t + NT // 2) % NT
    counts = torch.full((B, H, NT), 2, dtype=torch.int32)
    q, k, v, do = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(4))
    nan = float("nan")
    q[0, 0, 0 * 64 + 5, 3] = nan     # head 0: a query row of tile 0 (its dK reaches key tiles 1 and 2)
    k[0, 1, 2 * 64 + 7, 9] = nan     # head 1: a key row of tile 2 (its dQ reaches query tile 3)
    do[0, 1, 4 * 64 + 3, 1] = nan    # head 1: a dout row of tile 4 (its dV reaches key tiles 0 and 5)
    dev = "cuda"
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    idd, cd, bsd = idx.to(dev), counts.to(dev), bs.to(dev)
    out, lse = vsa.block_sparse_attention(qd, kd, vd, idd, cd, bsd, T, want_lse=True)
    dq, dk, dv = vsa.block_sparse_attention_bwd(qd, kd, vd, out, dod, lse, idd, cd, bsd, T)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    refs = oracle_mod.block_sparse_attention_bwd(q, k, v, do, idx, counts, bs, T, 1.0 / math.sqrt(D))
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        gv = got.float().cpu().numpy().astype(np.float64)
        rn = np.isnan(ref)
        assert rn.any() and not rn.all(), name
        np.testing.assert_array_equal(np.isnan(gv), rn, err_msg=f"D{D} {name}: NaN elements differ")
        assert np.isfinite(gv[~rn]).all(), f"D{D} {name}: Inf where the oracle is finite"
        err = gv[~rn] - ref[~rn]
        rel = float(np.linalg.norm(err) / max(np.linalg.norm(ref[~rn]), 1e-30))
        mx = float(np.abs(err).max())
        print(f"[bwd] pairs D{D} {name}: {int(rn.sum())} NaN matched, rel rms {rel:.3e}, max abs {mx:.3e}")
        assert rel <= REL_RMS, f"D{D} {name}: rel rms {rel:.3e}"
    # the partners named above are finite: dK of key tiles 1, 2 (head 0),
    # dQ of query tile 3 and dV of key tile 0 (head 1; key tile 5's dV is NaN
    # by the definition, since query tiles 2 and 5 meet the NaN key)
    for h, tens, tiles in ((0, dk, (1, 2)), (1, dq, (3,)), (1, dv, (0,))):
        for t in tiles:
            assert torch.isfinite(tens[0, h, t * 64:(t + 1) * 64].float()).all(), (h, t)
