"""GPU parity of the output un-tiling with the gate, through the C ABI,
against the oracle (bit for bit; NaN compared as NaN)."""
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


def _bits(x):
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _same(got, ref, label):
    gf = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float()
    rf = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float()
    nan = torch.isnan(rf)
    assert torch.equal(torch.isnan(gf), nan), f"{label}: NaN pattern differs"
    m = ~nan.numpy()
    assert np.array_equal(got[m], ref[m]), f"{label}: {int((got[m] != ref[m]).sum())} elements differ"


@pytest.mark.parametrize("tiling", ["video", "linear"])
def test_untile_inverts_layout_and_applies_gate(vsa, oracle_mod, tiling):
    g = torch.Generator().manual_seed(31)
    if tiling == "video":
        r2t, bs, _, _ = W.video_cube_tiling((21, 30, 52), (4, 4, 8), 128)
        S, T, B, H, D = 21 * 30 * 52, 128, 1, 3, 128
    else:
        S, T, B, H, D = 5000, 64, 2, 4, 64
        r2t, bs = W.linear_row_map(S, T)
    NT = int(bs.numel())
    dev = "cuda"
    x = torch.randn((B, S, H, D), generator=g).to(torch.bfloat16)
    gate = (torch.rand((B, S, H, D), generator=g) * 4 - 2).to(torch.bfloat16)
    gate.view(-1)[:4] = torch.tensor([float("inf"), float("nan"), 0.0, -0.0])
    r2t_d = r2t.to(dev)
    (xt,) = [t for t in vsa.tile_layout(x.to(dev), None, None, r2t_d, NT, T) if t is not None]
    # no gate: the exact inverse of the layout
    back = vsa.untile(xt, r2t_d, S, T)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    assert vsa.vsa_last_route()["kernel"] == vsa.VSA_KERNEL_UNTILE
    assert np.array_equal(_bits(back), _bits(x))
    # with the gate: one rounded product per element, as the oracle computes it
    o = torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16)
    o = W.pad_tile_major(o, bs, T, "naninf")
    got = vsa.untile(o.to(dev), r2t_d, S, T, gate_tok=gate.to(dev))
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    _same(_bits(got), oracle_mod.untile(o, gate, r2t, S, T), f"{tiling} gated")
    print(f"[untile] {tiling}: B{B} H{H} S{S} D{D}, exact")


def test_untile_bad_map_is_flagged(vsa):
    dev = "cuda"
    S, T, NT, H, D = 100, 64, 2, 2, 64
    r2t, _ = W.linear_row_map(S, T)
    r2t[5] = S + 7  # out of range: skipped and flagged
    o = torch.randn((1, H, NT * T, D), device=dev).to(torch.bfloat16)
    out = torch.zeros((1, S, H, D), dtype=torch.bfloat16, device=dev)
    vsa.vsa_untile(o, None, out, r2t.to(dev), 1, S, H, D, NT, T)
    assert vsa.vsa_check_device_status() == vsa.VSA_ERR_INDEX
    assert vsa.vsa_check_device_status() == vsa.VSA_OK  # read and cleared


def test_layout_select_attention_untile_pipeline(vsa, oracle_mod):
    # the whole tiled layer path on a small video grid: token-major q/k/v ->
    # tile layout -> coarse top-k selection -> block-sparse forward ->
    # un-tiling with the gate, against the oracle chain (bf16 output of the
    # oracle forward, then the oracle un-tiling)
    g = torch.Generator().manual_seed(41)
    r2t, bs, _, _ = W.video_cube_tiling((6, 8, 16), (2, 4, 8), 64)
    S, T, B, H, D, topk = 6 * 8 * 16, 64, 1, 2, 64, 5
    NT = int(bs.numel())
    dev = "cuda"
    q, k, v, gate = (torch.randn((B, S, H, D), generator=g).to(torch.bfloat16) for _ in range(4))
    r2t_d = r2t.to(dev)
    qt, kt, vt = vsa.tile_layout(q.to(dev), k.to(dev), v.to(dev), r2t_d, NT, T)
    idx, num = vsa.coarse_select(qt, kt, bs.to(dev), T, topk)
    out_t = vsa.block_sparse_attention(qt, kt, vt, idx, num, bs.to(dev), T)
    out = vsa.untile(out_t, r2t_d, S, T, gate_tok=gate.to(dev))
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    refs = [oracle_mod.tile_layout(x, r2t, NT, T) for x in (q, k, v)]
    oi, on, _ = oracle_mod.coarse_select(refs[0], refs[1], bs, T, topk, want_scores=False)
    assert np.array_equal(idx.cpu().numpy(), oi) and np.array_equal(num.cpu().numpy(), on)
    units = list(range(B * H * NT))
    ref, _ = oracle_mod.block_sparse_attention(refs[0], refs[1], refs[2], oi, on, bs, T, 1.0 / D ** 0.5,
                                               units=units, want_lse=False)
    PT.assert_parity(PT.gather_gpu_units(out_t, units, NT, T), ref, bs.numpy(), units, NT, T, label="pipeline fwd")
    # un-tile the GPU forward output with the oracle and compare bit for bit
    _same(_bits(out), oracle_mod.untile(out_t.cpu(), gate, r2t, S, T), "pipeline untile")
