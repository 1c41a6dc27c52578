"""Seeded synthetic inputs for the block-sparse attention forward pass.

This module only draws inputs: random tensors, tile geometries, and key-tile
selections.  It holds none of the attention arithmetic, so both the CPU oracle
(``oracle/``) and the CUDA path are fed from here without sharing any of the
method's code.

The five workloads follow the shapes and value distributions used for the
block-sparse forward on the FastVideo kernel page (hao-ai-lab/FastVideo commit
8503617, fastvideo-kernel/python):

* the tile sizes 64 and 128 and the ``q2k_idx`` / ``q2k_num`` /
  ``variable_block_sizes`` arguments come from the commit that adds the sm_121a
  tile-128 forward;
* ragged blocks, empty selections, odd block counts and NaN/Inf padding come
  from the test lists of that commit and of the sm_121a hardening commit;
* the 64-token video-tile layout comes from the fused ``tile_to_bhsd`` commit;
* the 6-head, 31200-token dense case comes from the Attn-QAT SM100 commit.

Where the page is silent (value distributions, the video cube order, the
top-k ranking), the generators below state the reading they implement.

Tensor conventions (shared with the library and the oracle):

* tile-major Q/K/V/O: bf16 ``[B, H, NT*T, D]`` (row ``t*T + r`` is token ``r`` of
  tile ``t``); rows ``r >= block_sizes[t]`` are padding;
* token-major Q/K/V: bf16 ``[B, S, H, D]``;
* ``row_to_token``: int32 ``[NT*T]``, the token feeding each tile-major row,
  ``-1`` for a padding row;
* ``q2k_idx``: int32 ``[B, H, NT, max_kv]`` (entries past ``q2k_num`` are -1);
* ``q2k_num``: int32 ``[B, H, NT]``; ``block_sizes``: int32 ``[NT]``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

__all__ = ["Workload", "make_workload", "WORKLOAD_NAMES", "SEED_BASE",
           "linear_row_map", "video_cube_tiling", "random_selection",
           "effective_flops", "padded_flops", "pad_tile_major"]

SEED_BASE = 1234

WORKLOAD_NAMES = {
    1: "tiny_b1h2d64_t64x4",
    2: "uniform_b1h12d128_t128x128_k32",
    3: "ragged_b2h8d64_t64x63_nanpad",
    4: "video_topk_b1h12d128_21x30x52_cube4x4x8_top42",
    5: "dense_b1h6d128_s31200_t128x244_lse",
}


@dataclass
class Workload:
    """One seeded problem instance.

    Exactly one of (token-major inputs + ``row_to_token``) or (tile-major
    inputs) is set.
    """

    name: str
    B: int
    H: int
    D: int
    T: int
    NT: int
    block_sizes: torch.Tensor          # int32 [NT]
    q2k_idx: torch.Tensor              # int32 [B, H, NT, max_kv]
    q2k_num: torch.Tensor              # int32 [B, H, NT]
    scale: float
    want_lse: bool
    S: int = 0                         # tokens per sequence (token-major form)
    q_tok: Optional[torch.Tensor] = None   # bf16 [B, S, H, D]
    k_tok: Optional[torch.Tensor] = None
    v_tok: Optional[torch.Tensor] = None
    row_to_token: Optional[torch.Tensor] = None  # int32 [NT*T]
    q: Optional[torch.Tensor] = None   # bf16 [B, H, NT*T, D]
    k: Optional[torch.Tensor] = None
    v: Optional[torch.Tensor] = None
    notes: dict = field(default_factory=dict)

    @property
    def Sp(self) -> int:
        return self.NT * self.T

    @property
    def max_kv(self) -> int:
        return int(self.q2k_idx.shape[-1])

    @property
    def token_major(self) -> bool:
        return self.q_tok is not None


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def linear_row_map(S: int, T: int) -> tuple[torch.Tensor, torch.Tensor]:
    """1-D tiling of ``S`` tokens into ``ceil(S/T)`` tiles; only the last tile is
    partial.  Returns ``(row_to_token [NT*T], block_sizes [NT])``."""
    NT = (S + T - 1) // T
    rows = torch.arange(NT * T, dtype=torch.int64)
    r2t = torch.where(rows < S, rows, torch.full_like(rows, -1)).to(torch.int32)
    bs = torch.full((NT,), T, dtype=torch.int32)
    bs[-1] = S - (NT - 1) * T
    return r2t, bs


def video_cube_tiling(grid=(21, 30, 52), cube=(4, 4, 8), T=128):
    """Cut a (T, H, W) token grid into cubes; cubes in t-major, then h, then w
    order; tokens inside a cube in (t, h, w) raster order.  Token ids are the
    raster index ``(t*GH + h)*GW + w``.

    Returns ``(row_to_token [NT*T], block_sizes [NT], cube_of_token [S],
    n_cubes_per_axis)``."""
    GT, GH, GW = grid
    CT, CH, CW = cube
    assert CT * CH * CW <= T
    nct, nch, ncw = (GT + CT - 1) // CT, (GH + CH - 1) // CH, (GW + CW - 1) // CW
    NT = nct * nch * ncw
    r2t = torch.full((NT * T,), -1, dtype=torch.int32)
    bs = torch.zeros((NT,), dtype=torch.int32)
    cube_of = torch.empty((GT * GH * GW,), dtype=torch.int64)
    tile = 0
    for ct in range(nct):
        t0, t1 = ct * CT, min(GT, ct * CT + CT)
        for ch in range(nch):
            h0, h1 = ch * CH, min(GH, ch * CH + CH)
            for cw in range(ncw):
                w0, w1 = cw * CW, min(GW, cw * CW + CW)
                tt, hh, ww = torch.meshgrid(torch.arange(t0, t1), torch.arange(h0, h1),
                                            torch.arange(w0, w1), indexing="ij")
                tok = ((tt * GH + hh) * GW + ww).reshape(-1)
                n = tok.numel()
                r2t[tile * T: tile * T + n] = tok.to(torch.int32)
                bs[tile] = n
                cube_of[tok] = tile
                tile += 1
    return r2t, bs, cube_of, (nct, nch, ncw)


def random_selection(g: torch.Generator, B: int, H: int, NT: int, counts: torch.Tensor,
                     max_kv: int) -> torch.Tensor:
    """For each (b, h, t), ``counts[b,h,t]`` distinct key tiles drawn uniformly
    without replacement (order as drawn); unused slots are -1."""
    idx = torch.full((B, H, NT, max_kv), -1, dtype=torch.int32)
    for b in range(B):
        for h in range(H):
            for t in range(NT):
                c = int(counts[b, h, t])
                if c:
                    idx[b, h, t, :c] = torch.randperm(NT, generator=g)[:c].to(torch.int32)
    return idx


def effective_flops(w: Workload) -> int:
    """Valid-token FLOPs: 4*D*sum over selected (b,h,t,j) of n_t*n_j (QK^T and PV,
    2 flops per multiply-add each)."""
    bs = w.block_sizes.to(torch.int64)
    num = w.q2k_num.to(torch.int64)
    idx = w.q2k_idx.to(torch.int64)
    live = torch.arange(w.max_kv).view(1, 1, 1, -1) < num.unsqueeze(-1)
    nj = torch.where(live, bs[idx.clamp(min=0)], torch.zeros_like(idx))
    per_tile = nj.sum(-1) * bs.view(1, 1, -1)
    return int(4 * w.D * per_tile.sum())


def padded_flops(w: Workload) -> int:
    """Padded-tile FLOPs: 4*D*T*T per selected (query tile, key tile) pair."""
    return int(4 * w.D * w.T * w.T * w.q2k_num.to(torch.int64).sum())


def pad_tile_major(x: torch.Tensor, block_sizes: torch.Tensor, T: int, fill: str) -> torch.Tensor:
    """Overwrite the padding rows of a tile-major tensor with ``fill``:
    ``"zero"``, or ``"naninf"`` (rows cycle through NaN, +Inf, -Inf)."""
    B, H, Sp, D = x.shape
    out = x.clone()
    NT = Sp // T
    for t in range(NT):
        n = int(block_sizes[t])
        for r in range(n, T):
            row = t * T + r
            if fill == "zero":
                out[:, :, row, :] = 0
            else:
                out[:, :, row, :] = (float("nan"), float("inf"), float("-inf"))[row % 3]
    return out


def _bf16_normal(g: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def _tiny(seed: int) -> Workload:
    g = _gen(seed)
    B, H, D, T, NT = 1, 2, 64, 64, 4
    S = NT * T
    r2t, bs = linear_row_map(S, T)
    q, k, v = (_bf16_normal(g, (B, S, H, D)) for _ in range(3))
    counts = torch.full((B, H, NT), 2, dtype=torch.int32)
    idx = random_selection(g, B, H, NT, counts, 2)
    return Workload(WORKLOAD_NAMES[1], B, H, D, T, NT, bs, idx, counts, 1.0 / math.sqrt(64),
                    False, S=S, q_tok=q, k_tok=k, v_tok=v, row_to_token=r2t)


def _uniform(seed: int) -> Workload:
    g = _gen(seed)
    B, H, D, T, NT = 1, 12, 128, 128, 128
    S = NT * T
    r2t, bs = linear_row_map(S, T)
    q, k, v = (_bf16_normal(g, (B, S, H, D)) for _ in range(3))
    counts = torch.full((B, H, NT), 32, dtype=torch.int32)
    idx = random_selection(g, B, H, NT, counts, 32)
    return Workload(WORKLOAD_NAMES[2], B, H, D, T, NT, bs, idx, counts, 1.0 / math.sqrt(D),
                    False, S=S, q_tok=q, k_tok=k, v_tok=v, row_to_token=r2t)


def _ragged(seed: int) -> Workload:
    """Tile-major inputs built directly, so the NaN/Inf padding reaches the
    attention kernel unchanged."""
    g = _gen(seed)
    B, H, D, T, NT = 2, 8, 64, 64, 63
    Sp = NT * T
    bs = torch.randint(1, T + 1, (NT,), generator=g, dtype=torch.int64).to(torch.int32)
    empty = torch.rand((B, H, NT), generator=g) < 0.10
    density = torch.rand((B, H, NT), generator=g) * 0.5
    counts = torch.round(density * NT).to(torch.int32)
    counts[empty] = 0
    max_kv = max(1, int(counts.max()))
    idx = random_selection(g, B, H, NT, counts, max_kv)
    q, k, v = (_bf16_normal(g, (B, H, Sp, D)) for _ in range(3))
    # 1% of the valid K elements scaled by 1e3 (in fp32, then rounded to bf16).
    big = torch.rand((B, H, Sp, D), generator=g) < 0.01
    kf = k.float()
    kf = torch.where(big, kf * 1e3, kf)
    k = kf.to(torch.bfloat16)
    q, k, v = (pad_tile_major(x, bs, T, "naninf") for x in (q, k, v))
    return Workload(WORKLOAD_NAMES[3], B, H, D, T, NT, bs, idx, counts, 1.0 / math.sqrt(D),
                    True, q=q, k=k, v=v, notes={"scaled_k_elements": int(big.sum())})


def _smooth_cube_offset(g: torch.Generator, B: int, H: int, ncubes, D: int, std: float) -> torch.Tensor:
    """i.i.d. N(0,1) per (b, h, cube, d), box-averaged over the 3x3x3 cube
    neighbourhood (clamped at the borders), rescaled to standard deviation
    ``std``.  Returns ``[B, H, n_cubes, D]`` fp32 in cube order."""
    nct, nch, ncw = ncubes
    z = torch.randn((B, H, nct, nch, ncw, D), generator=g, dtype=torch.float32)
    acc = torch.zeros_like(z)
    cnt = torch.zeros((nct, nch, ncw), dtype=torch.float32)
    for dt in (-1, 0, 1):
        for dh in (-1, 0, 1):
            for dw in (-1, 0, 1):
                ts = slice(max(0, dt), nct + min(0, dt))
                td = slice(max(0, -dt), nct + min(0, -dt))
                hs = slice(max(0, dh), nch + min(0, dh))
                hd = slice(max(0, -dh), nch + min(0, -dh))
                ws = slice(max(0, dw), ncw + min(0, dw))
                wd = slice(max(0, -dw), ncw + min(0, -dw))
                acc[:, :, td, hd, wd, :] += z[:, :, ts, hs, ws, :]
                cnt[td, hd, wd] += 1
    sm = acc / cnt.view(1, 1, nct, nch, ncw, 1)
    sm = sm * (std / sm.std())
    return sm.reshape(B, H, nct * nch * ncw, D)


def _video_topk(seed: int) -> Workload:
    g = _gen(seed)
    B, H, D, T = 1, 12, 128, 128
    r2t, bs, cube_of, ncubes = video_cube_tiling((21, 30, 52), (4, 4, 8), T)
    NT = int(bs.numel())
    S = 21 * 30 * 52
    toks = []
    for _ in range(3):
        base = torch.randn((B, S, H, D), generator=g, dtype=torch.float32)
        off = _smooth_cube_offset(g, B, H, ncubes, D, 0.5)        # [B, H, NT, D]
        base = base + off[:, :, cube_of, :].permute(0, 2, 1, 3)   # -> [B, S, H, D]
        toks.append(base.to(torch.bfloat16))
    q, k, v = toks
    topk = int(math.ceil(0.125 * NT))
    # Selection: fp32 mean over the valid tokens of each tile, fp32 dot product of
    # the pooled query and key, top-k per query tile with ties to the lower index.
    tok_of_tile = [r2t[t * T: t * T + int(bs[t])].to(torch.int64) for t in range(NT)]
    qm = torch.stack([q[:, tt, :, :].float().mean(dim=1) for tt in tok_of_tile], dim=2)  # [B,H,NT,D]
    km = torch.stack([k[:, tt, :, :].float().mean(dim=1) for tt in tok_of_tile], dim=2)
    score = torch.matmul(qm, km.transpose(-1, -2))                       # [B,H,NT,NT] fp32
    order = torch.sort(-score, dim=-1, stable=True).indices[..., :topk]
    idx = order.to(torch.int32).contiguous()
    counts = torch.full((B, H, NT), topk, dtype=torch.int32)
    return Workload(WORKLOAD_NAMES[4], B, H, D, T, NT, bs, idx, counts, 1.0 / math.sqrt(D),
                    False, S=S, q_tok=q, k_tok=k, v_tok=v, row_to_token=r2t,
                    notes={"topk": topk})


def _dense(seed: int, S: int = 31200, H: int = 6, T: int = 128, D: int = 128) -> Workload:
    g = _gen(seed)
    B = 1
    r2t, bs = linear_row_map(S, T)
    NT = int(bs.numel())
    q, k, v = (_bf16_normal(g, (B, S, H, D)) for _ in range(3))
    counts = torch.full((B, H, NT), NT, dtype=torch.int32)
    idx = torch.arange(NT, dtype=torch.int32).view(1, 1, 1, NT).expand(B, H, NT, NT).contiguous()
    name = WORKLOAD_NAMES[5] if (T, D) == (128, 128) else f"dense_b1h6d{D}_s31200_t{T}x{NT}_lse"
    return Workload(name, B, H, D, T, NT, bs, idx, counts, 1.0 / math.sqrt(D),
                    True, S=S, q_tok=q, k_tok=k, v_tok=v, row_to_token=r2t)


def make_workload(cfg: int, seed: Optional[int] = None, tile: Optional[int] = None,
                  head_dim: Optional[int] = None) -> Workload:
    """Build workload ``cfg`` (1..5) with seed ``SEED_BASE + cfg`` by default.
    ``tile`` (64 or 256) and ``head_dim`` (64) re-shape the dense-limit
    workload (5): the same 6 heads x 31200 tokens, every key tile selected."""
    seed = SEED_BASE + cfg if seed is None else seed
    if (tile is not None and tile != 128) or (head_dim is not None and head_dim != 128):
        if cfg != 5:
            raise ValueError("only the dense-limit workload takes another tile size or head_dim")
        return _dense(seed, T=tile or 128, D=head_dim or 128)
    return {1: _tiny, 2: _uniform, 3: _ragged, 4: _video_topk, 5: _dense}[cfg](seed)
