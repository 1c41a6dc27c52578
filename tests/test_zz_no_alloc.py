"""The no-allocation forward entry point.

vsa_block_sparse_fwd_noalloc serves callers that cannot call cudaMalloc --
host callbacks, plug-ins whose device memory belongs to a host framework, code
that must keep a fixed footprint -- by using a scratch array the library owns
instead of a caller-provided workspace.  These tests check, through the C ABI,
that it gives the same results as vsa_block_sparse_fwd on two calls in a row
(the scratch keeps the previous call's contents, which must not matter), and
that problems too large for the fixed scratch are refused before any launch.

This file is named so that pytest collects it last.
"""
import ctypes
import math

import pytest
import torch

import workloads as W

MAX_ABS = 2e-2
REL_RMS = 5e-3


@pytest.fixture(scope="module")
def vsa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_gathered_gb300 as V
    return V


def test_oversized_problem_is_refused_before_launch(vsa):
    # 2048 heads x 8192 tiles of 64 tokens -> 4.2M work items, far beyond the
    # 1 MiB scratch; the check happens before any device call, so the fake
    # pointers below are never touched.
    d = vsa.make_dims(1, 2048, 8192, 64, 64, 4)
    assert vsa.vsa_block_sparse_workspace_size_min(d) > vsa.VSA_NOALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p
    fake = P(0x100000)
    st = vsa.library().vsa_block_sparse_fwd_noalloc(fake, fake, fake, fake, fake, fake, fake, None,
                                                    ctypes.byref(d), None)
    assert st == vsa.VSA_ERR_LIMITS
    # invalid dims give the main entry point's error
    bad = vsa.make_dims(1, 2, 4, 32, 64, 2)
    st = vsa.library().vsa_block_sparse_fwd_noalloc(fake, fake, fake, fake, fake, fake, fake, None,
                                                    ctypes.byref(bad), None)
    assert st == vsa.VSA_ERR_ARG


def test_noalloc_limit_at_boundary(vsa):
    """The scratch of a problem is its least forward workspace: a 256-byte
    header plus 4 bytes per work item and per possible split entry (256 of
    them): exactly 1 MiB holds 261,824 work items; one more is refused before
    anything reaches the device.  (The split tail's partial results do not
    fit: a last wave then runs its one-unit entries whole.)"""
    fit = vsa.make_dims(1, 64, 8182, 128, 64, 1)      # 64 heads x 4091 items = 261,824
    over = vsa.make_dims(1, 75, 6982, 128, 64, 1)     # 75 heads x 3491 items = 261,825
    assert vsa.vsa_block_sparse_workspace_size_min(fit) == vsa.VSA_NOALLOC_SCRATCH_BYTES
    assert vsa.vsa_block_sparse_workspace_size_min(over) == vsa.VSA_NOALLOC_SCRATCH_BYTES + 4
    assert (vsa.VSA_NOALLOC_SCRATCH_BYTES - 256) // 4 - 256 == 261824
    fake = ctypes.c_void_p(0x100000)
    st = vsa.library().vsa_block_sparse_fwd_noalloc(fake, fake, fake, fake, fake, fake, fake, None,
                                                    ctypes.byref(over), None)
    assert st == vsa.VSA_ERR_LIMITS


def _compare(got, ref, label):
    g, r = got.float(), ref.float()
    gn, rn = torch.isnan(g), torch.isnan(r)
    assert torch.equal(gn, rn), f"{label}: NaN pattern differs"
    zero = (r == 0).all(-1)
    assert (got[zero].view(torch.int16) == 0).all(), f"{label}: zero rows differ"
    fin = ~rn
    diff = (g - r)[fin].double()
    mx = float(diff.abs().max()) if diff.numel() else 0.0
    rel = float(diff.norm() / max(float(r[fin].double().norm()), 1e-30)) if diff.numel() else 0.0
    assert mx <= MAX_ABS and rel <= REL_RMS, f"{label}: max abs {mx:.3e}, rel rms {rel:.3e}"


def _case(seed, B, H, NT, T, D):
    g = torch.Generator().manual_seed(seed)
    bs = torch.randint(1, T + 1, (NT,), generator=g).int()
    counts = torch.randint(0, NT + 1, (B, H, NT), generator=g).int()
    idx = W.random_selection(g, B, H, NT, counts, NT)
    q, k, v = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(3))
    q, k, v = (W.pad_tile_major(x, bs, T, "naninf") for x in (q, k, v))
    return q, k, v, idx, counts, bs


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [("ragged", 3), ("t128", (2, 3, 7, 128, 128)), ("t64d128", (1, 4, 9, 64, 128))])
def test_no_alloc_matches_workspace_entry(vsa, cfg):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda"
    name, spec = cfg
    if spec == 3:
        w = W.make_workload(3)
        q, k, v, idx, num, bs, T, scale = w.q, w.k, w.v, w.q2k_idx, w.q2k_num, w.block_sizes, w.T, w.scale
    else:
        B, H, NT, T, D = spec
        q, k, v, idx, num, bs = _case(11 + NT, B, H, NT, T, D)
        scale = 1.0 / math.sqrt(D)
    q, k, v, idx, num, bs = (x.to(dev).contiguous() for x in (q, k, v, idx, num, bs))
    B, H, Sp, D = q.shape
    dims = vsa.make_dims(B, H, Sp // T, T, D, idx.shape[-1], scale)

    ref_out, ref_lse = vsa.block_sparse_attention(q, k, v, idx, num, bs, T, scale=scale, want_lse=True)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == vsa.VSA_OK

    outs = [torch.full_like(q, float("nan")) for _ in range(2)]
    lses = [torch.full((B, H, Sp), float("nan"), dtype=torch.float32, device=dev) for _ in range(2)]
    for call in range(2):
        out, lse = outs[call], lses[call]
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        vsa.vsa_block_sparse_fwd_noalloc(q, k, v, idx, num, bs, out, lse, dims)
        torch.cuda.synchronize()
        # the second call (the first may load the library's device code) must
        # leave the device's free memory exactly as it was
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before, f"{name}: device memory changed"
        assert vsa.vsa_check_device_status() == vsa.VSA_OK
        _compare(out, ref_out, f"{name} call {call} out")
        assert torch.equal(torch.isneginf(lse), torch.isneginf(ref_lse))
        fin = torch.isfinite(ref_lse)
        assert float((lse[fin] - ref_lse[fin]).abs().max()) <= 2e-3
