"""GPU parity of the block-sparse backward (through the C ABI) against the
FP64 oracle backward.

The GPU backward takes the GPU forward's bf16 output and LSE, forms P and dS
in bf16 for the tensor cores and accumulates in fp32; the oracle recomputes
everything in FP64.  The bar per gradient tensor: relative RMS error over the
valid rows <= 1e-2 and max abs error <= 5e-2 * max |reference| (bf16 P and dS
carry 2^-9 relative rounding into sums over up to thousands of keys);
padding rows and keys no row selects must be exactly +0.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

REL_RMS = 1e-2
MAX_REL = 5e-2


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


def _check(name, got, ref, bs, T):
    g = got.float().cpu().numpy().astype(np.float64)
    B, H, Sp, D = g.shape
    valid = (np.arange(Sp) % T) < bs.numpy()[np.arange(Sp) // T]
    assert (got[:, :, ~torch.from_numpy(valid)].view(torch.int16) == 0).all(), f"{name}: padding rows not +0"
    gv, rv = g[:, :, valid], ref[:, :, valid]
    zero_ref = (rv == 0).all(-1)
    assert (gv[zero_ref] == 0).all(), f"{name}: rows that must be 0 are not"
    err = gv - rv
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(rv), 1e-30))
    mx = float(np.abs(err).max())
    scale = float(np.abs(rv).max())
    print(f"[bwd] {name}: rel rms {rel:.3e}, max abs {mx:.3e} (max |ref| {scale:.3e})")
    assert rel <= REL_RMS and mx <= MAX_REL * max(scale, 1e-30), f"{name}: rel rms {rel:.3e}, max abs {mx:.3e}"


@pytest.mark.parametrize("B,H,NT,D,full", [(1, 2, 3, 128, True), (2, 2, 5, 64, False), (1, 3, 6, 128, False)])
def test_bwd_matches_oracle(vsa, oracle_mod, B, H, NT, D, full):
    T = 128
    q, k, v, do, idx, counts, bs = _case(50 + NT + D, B, H, NT, D, full=full)
    dev = "cuda"
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    idd, cd, bsd = idx.to(dev), counts.to(dev), bs.to(dev)
    out, lse = vsa.block_sparse_attention(qd, kd, vd, idd, cd, bsd, T, want_lse=True)
    dq, dk, dv = vsa.block_sparse_attention_bwd(qd, kd, vd, out, dod, lse, idd, cd, bsd, T)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    r = vsa.vsa_last_route()
    assert r["kernel"] == vsa.VSA_KERNEL_BWD and r["tile"] == 128 and r["head_dim"] == D
    rq, rk, rv = oracle_mod.block_sparse_attention_bwd(q, k, v, do, idx, counts, bs, T, 1.0 / math.sqrt(D))
    label = f"B{B}H{H}NT{NT}D{D}{'dense' if full else 'ragged'}"
    _check(label + " dq", dq, rq, bs, T)
    _check(label + " dk", dk, rk, bs, T)
    _check(label + " dv", dv, rv, bs, T)


def test_bwd_deterministic(vsa):
    q, k, v, do, idx, counts, bs = _case(77, 1, 2, 6, 128)
    dev = "cuda"
    args = [x.to(dev) for x in (q, k, v)]
    idd, cd, bsd = idx.to(dev), counts.to(dev), bs.to(dev)
    out, lse = vsa.block_sparse_attention(*args, idd, cd, bsd, 128, want_lse=True)
    a = vsa.block_sparse_attention_bwd(*args, out, do.to(dev), lse, idd, cd, bsd, 128)
    b = vsa.block_sparse_attention_bwd(*args, out, do.to(dev), lse, idd, cd, bsd, 128)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
