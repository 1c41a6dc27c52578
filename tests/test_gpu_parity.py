"""GPU parity: the CUDA path (through the C ABI) against the FP64 CPU oracle.

Every case draws seeded inputs from ``workloads``, runs the library's kernels
on the GPU, and compares with ``oracle`` on the same inputs (see
``tests/_parity.py`` for the bar).  Output buffers are pre-filled with NaN so
that any row the kernel fails to write shows up (the NaN-filled allocator of
the sm_121a test list on the FastVideo kernel page).
"""
import dataclasses
import math

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


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _to_tile_major(w, vsa, oracle_mod):
    """Returns GPU tile-major q, k, v and the oracle's tile-major bit arrays.
    Token-major workloads go through the GPU layout kernel, which must match
    the oracle's layout bit for bit."""
    dev = "cuda"
    if w.token_major:
        r2t = w.row_to_token.to(dev)
        gq, gk, gv = vsa.tile_layout(w.q_tok.to(dev), w.k_tok.to(dev), w.v_tok.to(dev), r2t, w.NT, w.T)
        refs = [oracle_mod.tile_layout(x, w.row_to_token, w.NT, w.T) for x in (w.q_tok, w.k_tok, w.v_tok)]
        for g, r in zip((gq, gk, gv), refs):
            assert np.array_equal(_bits(g), r), "layout kernel differs from the oracle layout"
        return (gq, gk, gv), refs
    return tuple(x.to(dev) for x in (w.q, w.k, w.v)), [_bits(x) for x in (w.q, w.k, w.v)]


def _run(vsa, q, k, v, w, scale=None):
    dev = q.device
    out = torch.full_like(q, float("nan"))
    res = vsa.block_sparse_attention(q, k, v, w.q2k_idx.to(dev), w.q2k_num.to(dev), w.block_sizes.to(dev),
                                     w.T, scale=w.scale if scale is None else scale, want_lse=True, out=out)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    return res


def _check_steps(vsa, w):
    """The route's step counts: full key tiles unmasked, partly filled ones masked."""
    got = vsa.vsa_last_step_counts()
    want = PT.expected_step_counts(w.q2k_idx, w.q2k_num, w.block_sizes, w.T)
    assert got == want, f"(tail, full) steps {got}, expected {want}"
    return got


def _check(w, gpu_out, gpu_lse, refs, oracle_mod, units, label):
    ref, ref_lse = oracle_mod.block_sparse_attention(refs[0], refs[1], refs[2], w.q2k_idx, w.q2k_num,
                                                     w.block_sizes, w.T, w.scale, units=units)
    g = PT.gather_gpu_units(gpu_out, units, w.NT, w.T)
    gl = PT.gather_gpu_lse(gpu_lse, units, w.NT, w.T)
    PT.assert_parity(g, ref, w.block_sizes.numpy(), units, w.NT, w.T, gl, ref_lse, label=label)


def test_tiny_full(vsa, oracle_mod):
    w = W.make_workload(1)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    units = list(range(w.B * w.H * w.NT))
    _check(w, out, lse, refs, oracle_mod, units, "tiny")
    assert _check_steps(vsa, w) == (0, 2 * 4 * 2)
    r = vsa.vsa_last_route()
    assert r["kernel"] == vsa.VSA_KERNEL_ATTN_TCGEN05 and (r["tile"], r["head_dim"]) == (64, 64)
    assert r["work_items"] == 2 and r["grid"] == 2


def test_ragged_nan_padding_full(vsa, oracle_mod):
    w = W.make_workload(3)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    units = list(range(w.B * w.H * w.NT))
    _check(w, out, lse, refs, oracle_mod, units, "ragged")
    _check_steps(vsa, w)
    # empty selections give exactly +0 and -inf
    empty = (w.q2k_num == 0).nonzero().tolist()
    assert empty
    for b, h, t in empty[:20]:
        rows = out[b, h, t * 64:(t + 1) * 64]
        assert (rows.view(torch.int16) == 0).all()
        assert torch.isneginf(lse[b, h, t * 64:(t + 1) * 64]).all()


def test_uniform_full(vsa, oracle_mod):
    """Full size, every one of the 1536 query tiles against the oracle."""
    w = W.make_workload(2)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    _check(w, out, lse, refs, oracle_mod, list(range(w.B * w.H * w.NT)), "uniform")
    assert torch.isfinite(out.float()).all()


def test_video_topk_full(vsa, oracle_mod):
    """Full size, every one of the 4032 query tiles (ragged cubes) against the oracle."""
    w = W.make_workload(4)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    _check(w, out, lse, refs, oracle_mod, list(range(w.B * w.H * w.NT)), "video")
    tail, full = _check_steps(vsa, w)
    assert tail > 0 and full > 0


def test_dense_limit_sampled(vsa, oracle_mod):
    """Full size, in the bench's launch configuration (layout + attention, LSE
    on): 160 of the 1464 query tiles (11 %) against the oracle, the tail tile
    of every head among them, and properties over the whole output."""
    w = W.make_workload(5)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    last = w.NT - 1
    must = [h * w.NT + last for h in range(w.H)] + [0]
    units = PT.sample_units(w.B, w.H, w.NT, 160, seed=5, must=must)
    _check(w, out, lse, refs, oracle_mod, units, "dense")
    # properties over the whole output: valid rows finite, padding rows +0
    assert torch.isfinite(out[:, :, :31200].float()).all()
    assert (out[:, :, 31200:].view(torch.int16) == 0).all()
    assert torch.isneginf(lse[:, :, 31200:]).all() and torch.isfinite(lse[:, :, :31200]).all()
    # one masked step per query tile (the 96-token tail key tile), 243 full ones
    assert _check_steps(vsa, w) == (6 * 244, 6 * 244 * 243)
    r = vsa.vsa_last_route()
    assert r["kernel"] == vsa.VSA_KERNEL_ATTN_TCGEN05 and (r["tile"], r["head_dim"]) == (128, 128)
    assert r["work_items"] == 6 * 122
    assert r["grid"] == min(6 * 122, torch.cuda.get_device_properties(0).multi_processor_count)


@pytest.mark.parametrize("D", [128, 64])
def test_dense_t64_sampled(vsa, oracle_mod, D):
    """The dense workload at 64-token tiles, full size, in the bench's launch
    configuration: the dense form (key-tile pairs).  96 of the 2928 query
    tiles against the oracle, the 32-token tail tile of every head among
    them, and properties over the whole output."""
    w = W.make_workload(5, tile=64, head_dim=D)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    r = vsa.vsa_last_route()
    assert (r["tile"], r["head_dim"], r["layout"]) == (64, D, vsa.VSA_LAYOUT_PAIRED)
    last = w.NT - 1
    must = [h * w.NT + last for h in range(w.H)] + [0, 1]
    units = PT.sample_units(w.B, w.H, w.NT, 96, seed=7 + D, must=must)
    _check(w, out, lse, refs, oracle_mod, units, f"dense T64 D{D}")
    assert torch.isfinite(out[:, :, :31200].float()).all()
    assert (out[:, :, 31200:].view(torch.int16) == 0).all()
    # one masked step per query tile (the 32-token tail key tile), 487 full ones
    assert _check_steps(vsa, w) == (6 * 488, 6 * 488 * 487)


def _random_case(seed, B, H, NT, T, D, pad="naninf", empty_frac=0.15, full=False, max_kv=None):
    g = torch.Generator().manual_seed(seed)
    max_kv = NT if max_kv is None else max_kv
    bs = torch.full((NT,), T, dtype=torch.int32) if full else torch.randint(1, T + 1, (NT,), generator=g).int()
    if not full:
        bs[torch.rand(NT, generator=g) < 0.1] = 0           # a few empty tiles
        bs[NT // 2] = T
    counts = torch.randint(0, max_kv + 1, (B, H, NT), generator=g).int()
    counts[torch.rand((B, H, NT), generator=g) < empty_frac] = 0
    idx = W.random_selection(g, B, H, NT, counts, max_kv)
    q, k, v = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(3))
    if not full:
        q, k, v = (W.pad_tile_major(x, bs, T, pad) for x in (q, k, v))
    return W.Workload("random", B, H, D, T, NT, bs, idx, counts, 1.0 / math.sqrt(D), True, q=q, k=k, v=v)


@pytest.mark.parametrize("T,D,NT,narrow", [(64, 64, 9, False), (64, 128, 7, False), (128, 64, 5, False),
                                           (128, 128, 5, False), (64, 64, 1, False), (128, 128, 3, False),
                                           (256, 64, 5, False), (256, 128, 3, False), (256, 128, 1, False),
                                           (64, 64, 9, True), (64, 128, 8, True), (128, 128, 5, True)])
def test_variants_ragged(vsa, oracle_mod, T, D, NT, narrow):
    """Random selections on ragged tiles with NaN/Inf padding, every element
    against the oracle.  Rows of q2k_idx hold every key tile (the dense form:
    key-tile pairs at 64-token tiles, the paired MMA issue at 128) unless
    `narrow` (one slot short: the split, per-tile form)."""
    w = _random_case(100 + T + D + NT + (7 if narrow else 0), 2, 3, NT, T, D, max_kv=NT - 1 if narrow else None)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    # 256-token tiles always share one selection per unit pair (the dense form at D = 128)
    dense_form = (T == 256 and D == 128) or (not narrow and (T == 64 or (T == 128 and D == 128)))
    assert vsa.vsa_last_route()["layout"] == (vsa.VSA_LAYOUT_PAIRED if dense_form else vsa.VSA_LAYOUT_SPLIT)
    _check(w, out, lse, refs, oracle_mod, list(range(w.B * w.H * w.NT)), f"T{T}D{D}NT{NT}{' narrow' if narrow else ''}")
    _check_steps(vsa, w)


def _rescale_events(q, k, w):
    """Rows (over valid query rows) whose running maximum, taken over the
    selected key tiles in ascending order, grows by more than 2^8 after the
    first tile: the rows that take the softmax's lazy rescale of O.  Plain
    float64 over the valid keys of each tile."""
    B, H, Sp, D = q.shape
    T, NT = w.T, w.NT
    bs = w.block_sizes.numpy()
    c = w.scale / math.log(2.0)
    qd, kd = q.double().numpy(), k.double().numpy()
    events = []
    for b in range(B):
        for h in range(H):
            for t in range(NT):
                n = int(w.q2k_num[b, h, t])
                if bs[t] == 0 or n == 0:
                    continue
                qt = qd[b, h, t * T:t * T + bs[t]]
                m = np.full(qt.shape[0], -np.inf)
                ev = np.zeros(qt.shape[0], dtype=int)
                for j in sorted(int(x) for x in w.q2k_idx[b, h, t, :n]):
                    if bs[j] == 0:
                        continue
                    mx = (qt @ kd[b, h, j * T:j * T + bs[j]].T).max(axis=1) * c
                    ev += (np.isfinite(m) & (mx > m + 8.0)).astype(int)
                    m = np.maximum(m, mx)
                events.append(ev)
    return np.concatenate(events)


@pytest.mark.parametrize("T,D,narrow", [(128, 128, True), (128, 128, False), (128, 64, True),
                                        (64, 128, True), (64, 128, False), (64, 64, True)])
def test_growing_max_rescales_o(vsa, oracle_mod, T, D, narrow):
    """Scores that climb from key tile to key tile, at a rate drawn per query
    row (some rows climb fast, so their running maximum grows by more than
    2^8 several times and the softmax rescales O; some climb slowly and never
    rescale; some fall, so the first tile keeps the maximum), on ragged tiles
    with NaN/Inf padding.  Every element against the oracle, in the sparse
    (split) and dense (paired issue, key-tile pairs) forms."""
    NT = 8 if T == 128 else 12
    B, H, Sp = 1, 4, NT * T
    w = _random_case(500 + T + D + int(narrow), B, H, NT, T, D, max_kv=NT - 1 if narrow else None)
    g = torch.Generator().manual_seed(900 + T + D)
    # per query row: half climb fast, a quarter stay flat, a quarter fall
    kind = torch.rand((B, H, Sp, 1), generator=g)
    mag = torch.rand((B, H, Sp, 1), generator=g)
    rate = torch.where(kind < 0.5, 4.0 + 4.0 * mag, torch.where(kind < 0.75, 2.0 * mag - 1.0, -4.0 - 4.0 * mag))
    step = 8.0 if T == 128 else 6.0                                  # per key tile
    ramp = (torch.arange(NT).repeat_interleave(T).float() * step)[None, None, :, None]
    q = 0.5 * torch.randn((B, H, Sp, D), generator=g)
    k = 0.5 * torch.randn((B, H, Sp, D), generator=g)
    q[..., :1] += rate
    k[..., :1] += ramp
    q, k = (W.pad_tile_major(x.to(torch.bfloat16), w.block_sizes, T, "naninf") for x in (q, k))
    w = dataclasses.replace(w, q=q, k=k)
    ev = _rescale_events(q, k, w)
    assert (ev >= 1).mean() > 0.2 and (ev >= 2).sum() > 50 and (ev == 0).mean() > 0.2, "the input must rescale O"
    (qg, kg, vg), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, qg, kg, vg, w)
    dense_form = not narrow and (T == 64 or D == 128)
    assert vsa.vsa_last_route()["layout"] == (vsa.VSA_LAYOUT_PAIRED if dense_form else vsa.VSA_LAYOUT_SPLIT)
    _check(w, out, lse, refs, oracle_mod, list(range(w.B * w.H * w.NT)),
           f"rescale T{T}D{D}{' narrow' if narrow else ''}")


def test_many_waves(vsa, oracle_mod):
    """More work items than SMs: every CTA takes several items."""
    w = _random_case(7, 4, 48, 6, 128, 64, full=True)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    assert vsa.vsa_last_route()["work_items"] == 4 * 48 * 3
    units = PT.sample_units(w.B, w.H, w.NT, 64, seed=8)
    _check(w, out, lse, refs, oracle_mod, units, "waves")


@pytest.mark.parametrize("T", [64, 128, 256])
@pytest.mark.parametrize("form", ["sparse", "dense"])
def test_split_last_wave(vsa, oracle_mod, T, form):
    """One work item per SM plus a few: the last wave's items run as one-unit
    entries, and each CTA writes only its unit's rows.  With 128-token kernel
    tiles each unit is also cut into key-tile ranges on separate CTAs: every
    range leaves its partial O, row maximum and row sum in the workspace and
    the last one merges them (ranges with no selected key tile included, as
    the sparse case's three-tile rows leave most ranges empty).  Both forms:
    short rows of q2k_idx (sparse) and rows that hold every key tile at
    D = 128 (dense: the paired MMA issue at 128- and 256-token tiles, key-tile
    pairs at 64)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_items = sms + 5
    NT = n_items * 256 // T
    if form == "sparse":
        w = _random_case(300 + T, 1, 1, NT, T, 64, max_kv=3)
    else:
        w = _random_case(310 + T, 1, 1, NT, T, 128)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    r = vsa.vsa_last_route()
    assert r["work_items"] == n_items
    assert r["layout"] == (vsa.VSA_LAYOUT_PAIRED if form == "dense" else vsa.VSA_LAYOUT_SPLIT)
    # 128-token kernel tiles: each one-unit entry is cut into key-tile ranges
    # (as many as keep the 2 x 5 units' ranges within the grid, at most 8)
    assert r["tail_parts"] == (1 if T == 64 else min(8, min(sms, 256) // 10))
    _check(w, out, lse, refs, oracle_mod, list(range(w.B * w.H * w.NT)), f"split T{T} {form}")
    _check_steps(vsa, w)   # split items count each (query tile, key tile) step once
    # bit-identical across runs, although which items are split may differ
    # (items of equal length take their places in any order)
    again, _ = _run(vsa, q, k, v, w)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    # the least workspace has no room for the ranges' partial results: the
    # one-unit entries then run whole, against the same oracle
    dims = vsa.make_dims(w.B, w.H, w.NT, w.T, w.D, w.q2k_idx.shape[-1], w.scale)
    ws = torch.empty(vsa.vsa_block_sparse_workspace_size_min(dims), dtype=torch.uint8, device="cuda")
    whole = torch.full_like(q, float("nan"))
    whole_lse = torch.full(lse.shape, float("nan"), dtype=torch.float32, device="cuda")
    vsa.vsa_block_sparse_fwd(q, k, v, w.q2k_idx.cuda(), w.q2k_num.cuda(), w.block_sizes.cuda(), whole, whole_lse,
                             dims, ws)
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    assert vsa.vsa_last_route()["tail_parts"] == 1
    _check(w, whole, whole_lse, refs, oracle_mod, list(range(w.B * w.H * w.NT)), f"split T{T} {form} whole units")


@pytest.mark.parametrize("T", [64, 128])
def test_tiles_beyond_shared_memory_bitmaps(vsa, oracle_mod, T):
    """8200 tiles, just above the 8192 whose selection bitmaps fit in shared
    memory: the kernel keeps them in the workspace instead (the hardening
    commit's limit is 2^22 tiles).  Selections reach tiles on both sides of
    8192; 640 query tiles are compared with the oracle, among them every
    query tile that selects a tile past 8191 in one head."""
    NT = 8200
    w = _random_case(4242 + T, 1, 2, NT, T, 64, max_kv=4, empty_frac=0.05)
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    high = [t for t in range(NT)
            if (w.q2k_idx[0, 0, t, :int(w.q2k_num[0, 0, t])] >= 8192).any()][:300]
    assert high
    units = PT.sample_units(w.B, w.H, w.NT, 640, seed=T, must=high + [NT - 1, 2 * NT - 1, 8191, 8192 + NT])
    _check(w, out, lse, refs, oracle_mod, units, f"8200 tiles T{T}")
    _check_steps(vsa, w)
    assert vsa.vsa_last_route()["work_items"] == 2 * (NT * T // 256)


def test_all_empty_and_zero_max_kv(vsa):
    dev = "cuda"
    B, H, NT, T, D = 1, 2, 4, 128, 128
    q = torch.randn((B, H, NT * T, D), device=dev).to(torch.bfloat16)
    bs = torch.full((NT,), T, dtype=torch.int32, device=dev)
    for max_kv in (3, 0):
        idx = torch.zeros((B, H, NT, max_kv), dtype=torch.int32, device=dev)
        num = torch.zeros((B, H, NT), dtype=torch.int32, device=dev)
        out = torch.full_like(q, float("nan"))
        out, lse = vsa.block_sparse_attention(q, q, q, idx, num, bs, T, want_lse=True, out=out)
        torch.cuda.synchronize()
        assert (out.view(torch.int16) == 0).all() and torch.isneginf(lse).all()
    assert vsa.vsa_check_device_status() == 0


def test_nan_in_valid_key_gives_nan_rows(vsa, oracle_mod):
    w = _random_case(21, 1, 2, 5, 64, 64, full=True, empty_frac=0.0)
    w.k = w.k.clone()
    w.k[0, 1, 2 * 64 + 5, 7] = float("nan")   # tile 2 of head 1
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    _check(w, out, lse, refs, oracle_mod, list(range(10)), "nan-key")
    sel = [2 in w.q2k_idx[0, 1, t, :int(w.q2k_num[0, 1, t])].tolist() for t in range(5)]
    assert any(sel)
    for t in range(5):
        assert bool(torch.isnan(out[0, 1, t * 64:(t + 1) * 64].float()).all()) == sel[t]


def _pair_case(seed, D, NT=6, ragged=False):
    """64-token tiles whose pairs (2i, 2i+1) select disjoint key tiles: query
    tile t selects key tiles t and (t + NT/2) mod NT, so every key tile serves
    exactly one tile of one pair and two pairs in all."""
    T, B, H = 64, 1, 2
    g = torch.Generator().manual_seed(seed)
    bs = torch.full((NT,), T, dtype=torch.int32)
    if ragged:
        bs = torch.randint(24, T + 1, (NT,), generator=g).int()
    idx = torch.empty((B, H, NT, 2), dtype=torch.int32)
    for t in range(NT):
        idx[:, :, t, 0] = t
        idx[:, :, t, 1] = (t + NT // 2) % NT
    num = torch.full((B, H, NT), 2, dtype=torch.int32)
    q, k, v = (torch.randn((B, H, NT * T, D), generator=g).to(torch.bfloat16) for _ in range(3))
    if ragged:
        q, k, v = (W.pad_tile_major(x, bs, T, "naninf") for x in (q, k, v))
    return W.Workload("pairs", B, H, D, T, NT, bs, idx, num, 1.0 / math.sqrt(D), True, q=q, k=k, v=v)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("where", ["v", "k"])
@pytest.mark.parametrize("ragged", [False, True])
@pytest.mark.parametrize("form", ["tile", "pair"])
def test_t64_pair_isolation(vsa, oracle_mod, D, where, ragged, form):
    """Two 64-token query tiles share one 128-lane accumulator.  A NaN, +Inf or
    -Inf in a VALID row of a key tile that only one tile of the pair selects
    must reach only that tile's rows, as in the definition (each query tile
    attends to its own list); the partner tile's rows stay finite and match
    the oracle, and every non-finite element matches the oracle's exactly.
    Both 64-token forms run: one ring entry per key tile, and (rows of
    q2k_idx padded to every key tile: the dense form) one per pair of key
    tiles, where the two query tiles of a unit select different tiles of one
    pair (query tile 0 key tile 0, query tile 1 key tile 1)."""
    w = _pair_case(900 + D + (1 if ragged else 0), D, ragged=ragged)
    if form == "pair":
        wide = torch.full((w.B, w.H, w.NT, w.NT), -1, dtype=torch.int32)
        wide[..., : w.max_kv] = w.q2k_idx
        w = dataclasses.replace(w, q2k_idx=wide)
    x = (w.v if where == "v" else w.k).clone()
    # key tiles 0 and 3 are selected by query tiles 0 and 3 only, whose pair
    # partners (1 and 2) select neither; head 0 gets infinities only (a NaN in
    # K makes whole rows NaN and would hide them), head 1 NaN and +Inf
    inf, nan = float("inf"), float("nan")
    plant = {0: ((0, 9, 3, inf), (3, 20, D - 3, -inf), (0, 21, 8, -inf)),
             1: ((0, 5, 7, nan), (3, 2, 11, inf), (3, 17, 0, nan))}
    for h, cells in plant.items():
        for j, r, c, val in cells:
            assert r < int(w.block_sizes[j])
            x[0, h, j * 64 + r, c] = val
    if where == "v":
        w.v = x
    else:
        w.k = x
    (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
    out, lse = _run(vsa, q, k, v, w)
    assert vsa.vsa_last_route()["layout"] == (vsa.VSA_LAYOUT_PAIRED if form == "pair" else vsa.VSA_LAYOUT_SPLIT)
    units = list(range(w.B * w.H * w.NT))
    ref, ref_lse = oracle_mod.block_sparse_attention(refs[0], refs[1], refs[2], w.q2k_idx, w.q2k_num,
                                                     w.block_sizes, w.T, w.scale, units=units)
    g = PT.gather_gpu_units(out, units, w.NT, w.T)
    gl = PT.gather_gpu_lse(lse, units, w.NT, w.T)
    PT.assert_parity_elementwise(g, ref, w.block_sizes.numpy(), units, w.NT, w.T, gl, ref_lse,
                                 label=f"pairs {where} D{D}{' ragged' if ragged else ''} {form}")
    # the pair partners of the tiles that meet the planted values stay finite
    for h in range(2):
        for t in (1, 2, 4, 5):
            assert torch.isfinite(out[0, h, t * 64:t * 64 + int(w.block_sizes[t])].float()).all(), (h, t)
    assert not np.isfinite(g).all()


def test_deterministic(vsa, oracle_mod):
    w = W.make_workload(3)
    (q, k, v), _ = _to_tile_major(w, vsa, oracle_mod)
    a, la = _run(vsa, q, k, v, w)
    b, lb = _run(vsa, q, k, v, w)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(la.view(torch.int32), lb.view(torch.int32))


def test_issue_layouts_agree_bitwise(vsa, oracle_mod):
    """The split and paired MMA-issue layouts run the same products in the same
    order per accumulator, so they give bit-identical results.  The layout
    follows the row length of q2k_idx: the same selections, with rows padded
    to every key tile, switch a sparse case from split to paired."""
    for T, D, NT in ((128, 128, 9), (128, 128, 4)):
        w = _random_case(500 + T + NT, 2, 3, NT, T, D, max_kv=max(1, NT // 3))
        (q, k, v), refs = _to_tile_major(w, vsa, oracle_mod)
        a, la = _run(vsa, q, k, v, w)
        assert vsa.vsa_last_route()["layout"] == vsa.VSA_LAYOUT_SPLIT
        wide = torch.full((w.B, w.H, w.NT, w.NT), -1, dtype=torch.int32)
        wide[..., : w.max_kv] = w.q2k_idx
        w_wide = dataclasses.replace(w, q2k_idx=wide)
        b, lb = _run(vsa, q, k, v, w_wide)
        assert vsa.vsa_last_route()["layout"] == vsa.VSA_LAYOUT_PAIRED
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"T{T}: layouts differ"
        assert torch.equal(la.view(torch.int32), lb.view(torch.int32))
        _check(w, a, la, refs, oracle_mod, list(range(w.B * w.H * w.NT)), f"layouts T{T}")


def test_bad_indices_are_flagged_not_faulted(vsa):
    dev = "cuda"
    B, H, NT, T, D = 1, 1, 4, 64, 64
    q = torch.randn((B, H, NT * T, D), device=dev).to(torch.bfloat16)
    bs = torch.full((NT,), T, dtype=torch.int32, device=dev)
    num = torch.full((B, H, NT), 2, dtype=torch.int32, device=dev)
    idx = torch.tensor([[[[0, 1], [1, 1], [2, 9], [3, -4]]]], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    d = vsa.make_dims(B, H, NT, T, D, 2)
    vsa.vsa_validate_indices(idx, num, bs, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == vsa.VSA_ERR_INDEX
    vsa.block_sparse_attention(q, q, q, idx, num, bs, T)
    assert vsa.vsa_check_device_status() == vsa.VSA_ERR_INDEX
    assert vsa.vsa_check_device_status() == 0          # the word is cleared by reading
    ok = torch.tensor([[[[0, 1], [1, 2], [2, 3], [3, 0]]]], dtype=torch.int32, device=dev)
    vsa.vsa_validate_indices(ok, num, bs, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_layout_partial_and_bad_map(vsa, oracle_mod):
    dev = "cuda"
    r2t, bs, _, _ = W.video_cube_tiling((5, 6, 9), (2, 2, 4), 16)
    S, NT = 5 * 6 * 9, int(bs.numel())
    x = torch.randn((2, S, 3, 64)).to(torch.bfloat16)
    (got, _, _) = vsa.tile_layout(x.to(dev), None, None, r2t.to(dev), NT, 16)
    assert np.array_equal(_bits(got), oracle_mod.tile_layout(x, r2t, NT, 16))
    assert vsa.vsa_check_device_status() == 0
    bad = r2t.clone()
    bad[3] = S + 5
    vsa.tile_layout(x.to(dev), None, None, bad.to(dev), NT, 16)
    assert vsa.vsa_check_device_status() == vsa.VSA_ERR_INDEX
