"""GPU parity of the coarse key-tile selection (through the C ABI) against the
oracle's selection.

The kept set is an integer result decided by floating point.  The library and
the oracle take that decision with the same fp32 arithmetic (means summed over
rows in order and divided once; scores summed over d in order of fused
multiply-adds), so the selection must match exactly: same
q2k_num, same tiles in the same ascending order, -1 after.  Output buffers are
pre-filled with a sentinel so that unwritten entries show up.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests import _parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_gathered_gb300 as V
    assert V.vsa_check_device_status() == 0
    return V


def _gpu_select(vsa, q, k, bs, T, topk):
    dev = "cuda"
    qd, kd, bsd = q.to(dev).contiguous(), k.to(dev).contiguous(), bs.to(dev).contiguous()
    B, H, Sp, D = q.shape
    NT = Sp // T
    dims = vsa.make_dims(B, H, NT, T, D, topk)
    ws = torch.empty(vsa.vsa_coarse_select_workspace_size(dims), dtype=torch.uint8, device=dev)
    idx = torch.full((B, H, NT, topk), -7, dtype=torch.int32, device=dev)
    num = torch.full((B, H, NT), -7, dtype=torch.int32, device=dev)
    vsa.vsa_coarse_select(qd, kd, bsd, topk, idx, num, dims, ws)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    r = vsa.vsa_last_route()
    assert r["kernel"] == vsa.VSA_KERNEL_SELECT and r["tile"] == T and r["head_dim"] == D
    return idx.cpu().numpy(), num.cpu().numpy()


def _compare(vsa, oracle_mod, q, k, bs, T, topk, label):
    gi, gn = _gpu_select(vsa, q, k, bs, T, topk)
    oi, on, _ = oracle_mod.coarse_select(q, k, bs, T, topk, want_scores=False)
    assert np.array_equal(gn, on), f"{label}: q2k_num differs at {np.argwhere(gn != on)[:5].tolist()}"
    assert np.array_equal(gi, oi), f"{label}: q2k_idx differs at {np.argwhere(gi != oi)[:5].tolist()}"
    print(f"[select] {label}: {gn.size} query tiles, {int(gn.sum())} kept, exact")
    return gi, gn


@pytest.mark.parametrize("B,H,NT,T,D,topk", [
    (1, 2, 4, 64, 64, 2),        # tiny, like the first workload
    (2, 3, 37, 64, 64, 9),       # odd tile count, ragged sizes
    (1, 4, 70, 128, 128, 12),    # more than two 32-tile chunks of key means
    (1, 2, 9, 128, 64, 20),      # topk above the tile count
    (2, 2, 33, 64, 128, 0),      # topk = 0
    (1, 2, 9, 256, 128, 4),      # 256-token tiles
])
def test_select_matches_oracle(vsa, oracle_mod, B, H, NT, T, D, topk):
    g = torch.Generator().manual_seed(100 + NT + topk)
    bs = torch.randint(1, T + 1, (NT,), generator=g).to(torch.int32)
    bs[torch.rand((NT,), generator=g) < 0.1] = 0  # some empty tiles
    off = torch.randn((B, H, NT, 1, D), generator=g) * 0.5
    q = (torch.randn((B, H, NT, T, D), generator=g) + off).reshape(B, H, NT * T, D).to(torch.bfloat16)
    k = (torch.randn((B, H, NT, T, D), generator=g) + off).reshape(B, H, NT * T, D).to(torch.bfloat16)
    q, k = (W.pad_tile_major(x, bs, T, "naninf") for x in (q, k))
    _compare(vsa, oracle_mod, q, k, bs, T, topk, f"B{B}H{H}NT{NT}T{T}D{D}k{topk}")


def test_select_ties_and_equal_scores(vsa, oracle_mod):
    # identical key tiles: every score of a row is equal, so the smallest
    # indices are kept; -0 and +0 scores count as equal
    B, H, NT, T, D, topk = 1, 2, 40, 64, 64, 7
    bs = torch.full((NT,), T, dtype=torch.int32)
    g = torch.Generator().manual_seed(9)
    q = torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, 1, T, D), generator=g).expand(B, H, NT, T, D).reshape(B, H, NT * T, D)
    k = k.contiguous().to(torch.bfloat16)
    k[:, 1] = 0  # head 1: all scores are +0 or -0
    gi, gn = _compare(vsa, oracle_mod, q, k, bs, T, topk, "ties")
    assert (gi[..., :topk] == np.arange(topk)).all()


def test_select_video_workload(vsa, oracle_mod):
    # the video-grid workload at full size: 12 heads, 336 ragged cube tiles,
    # top 42 per query tile, after the GPU tile layout
    w = W.make_workload(4)
    dev = "cuda"
    r2t = w.row_to_token.to(dev)
    gq, gk, _ = vsa.tile_layout(w.q_tok.to(dev), w.k_tok.to(dev), None, r2t, w.NT, w.T)
    k_top = int(w.notes["topk"])
    gi, gn = _compare(vsa, oracle_mod, gq.cpu(), gk.cpu(), w.block_sizes, w.T, k_top, "video 21x30x52 top42")
    assert (gn == k_top).all()


def test_select_feeds_attention(vsa, oracle_mod):
    # the GPU selection goes straight into the GPU forward; parity of the
    # result against the oracle forward on the oracle's own selection
    B, H, NT, T, D, topk = 1, 3, 24, 128, 128, 6
    g = torch.Generator().manual_seed(21)
    bs = torch.randint(1, T + 1, (NT,), generator=g).to(torch.int32)
    q, k, v = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(3))
    q, k, v = (W.pad_tile_major(x, bs, T, "naninf") for x in (q, k, v))
    dev = "cuda"
    idx, num = vsa.coarse_select(q.to(dev), k.to(dev), bs.to(dev), T, topk)
    out = torch.full((B, H, NT * T, D), float("nan"), dtype=torch.bfloat16, device=dev)
    out, lse = vsa.block_sparse_attention(q.to(dev), k.to(dev), v.to(dev), idx, num, bs.to(dev), T,
                                          want_lse=True, out=out)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    oi, on, _ = oracle_mod.coarse_select(q, k, bs, T, topk, want_scores=False)
    assert np.array_equal(idx.cpu().numpy(), oi) and np.array_equal(num.cpu().numpy(), on)
    units = list(range(B * H * NT))
    ref, ref_lse = oracle_mod.block_sparse_attention(q, k, v, torch.from_numpy(oi), torch.from_numpy(on), bs, T,
                                                     1.0 / D ** 0.5, units=units)
    PT.assert_parity(PT.gather_gpu_units(out, units, NT, T), ref, bs.numpy(), units, NT, T,
                     PT.gather_gpu_lse(lse, units, NT, T), ref_lse, label="select->attention")
