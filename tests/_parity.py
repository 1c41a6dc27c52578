"""Comparison helpers for GPU-vs-oracle parity tests.

The bar (block-sparse forward, BF16 in / FP32 accumulate): over valid,
non-NaN query rows, max |gpu - ref| <= 2e-2 and ||gpu - ref||_2 / ||ref||_2 <=
5e-3 with the FP64 oracle rounded to FP32; rows the oracle gives as exact zero
(empty selections, padding) must be bitwise +0.0; NaN rows must be NaN in every
element on both sides; padding rows of the output must be +0.0.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 2e-2
REL_RMS = 5e-3
# LSE = m + log(l) with l the sum of the bf16-rounded P that P V uses (so the
# output weights P / l are exactly normalised).  One bf16 rounding is at most
# 2^-8 relative, so when one key dominates a row log(l) is off by up to
# ln(1 + 2^-8) = 3.9e-3.  The scores are accumulated in FP32 over D products,
# so their error grows with the score's size (about D * 2^-24 * sum|q_d k_d|):
# the bound is an absolute part plus a part relative to |lse|.
LSE_ABS = 4e-3
LSE_REL = 8e-6

RESULTS = []  # (label, max_abs, rel_rms, lse_max_abs) of every passing comparison


def unit_rows(units, NT, T):
    """(bh, t) pairs of flat unit ids."""
    return [(u // NT, u % NT) for u in units]


def gather_gpu_units(out: torch.Tensor, units, NT, T):
    """GPU tile-major output -> [n_units, T, D] float32 numpy (exact widening)."""
    B, H, Sp, D = out.shape
    flat = out.reshape(B * H, Sp, D)
    tiles = torch.stack([flat[bh, t * T:(t + 1) * T] for bh, t in unit_rows(units, NT, T)])
    return tiles.float().cpu().numpy()


def gather_gpu_lse(lse: torch.Tensor, units, NT, T):
    B, H, Sp = lse.shape
    flat = lse.reshape(B * H, Sp)
    return torch.stack([flat[bh, t * T:(t + 1) * T] for bh, t in unit_rows(units, NT, T)]).cpu().numpy()


def assert_parity(gpu: np.ndarray, ref: np.ndarray, block_sizes, units, NT, T, gpu_lse=None, ref_lse=None,
                  label=""):
    """gpu [n, T, D] float32; ref [n, T, D] float64 from the oracle."""
    bs = np.asarray(block_sizes)
    ref32 = ref.astype(np.float32)
    n = gpu.shape[0]
    valid = np.zeros((n, T), dtype=bool)
    for i, (_, t) in enumerate(unit_rows(units, NT, T)):
        valid[i, :int(bs[t])] = True
    # padding rows: +0 exactly
    pad = gpu[~valid]
    assert (pad.view(np.uint32) == 0).all(), f"{label}: padding rows not +0"
    ref_nan = np.isnan(ref32).all(-1)
    gpu_nan = np.isnan(gpu).all(-1)
    assert (np.isnan(ref32).any(-1) == ref_nan).all()
    np.testing.assert_array_equal(gpu_nan[valid], ref_nan[valid], err_msg=f"{label}: NaN rows differ")
    assert not (np.isnan(gpu).any(-1) & ~gpu_nan)[valid].any(), f"{label}: partial NaN row"
    zero_rows = (ref32 == 0).all(-1) & valid
    assert (gpu[zero_rows].view(np.uint32) == 0).all(), f"{label}: empty rows not +0"
    live = valid & ~ref_nan
    g, r = gpu[live].astype(np.float64), ref32[live].astype(np.float64)
    if g.size:
        err = np.abs(g - r)
        mx = float(err.max())
        rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
        assert mx <= MAX_ABS and rel <= REL_RMS, f"{label}: max abs {mx:.3e}, rel rms {rel:.3e}"
    if gpu_lse is not None:
        rl = ref_lse.astype(np.float32)
        assert np.isneginf(gpu_lse[~valid]).all(), f"{label}: padding lse not -inf"
        np.testing.assert_array_equal(np.isneginf(gpu_lse[valid]), np.isneginf(rl[valid]))
        np.testing.assert_array_equal(np.isnan(gpu_lse[valid]), np.isnan(rl[valid]))
        fin = valid & np.isfinite(rl)
        if fin.any():
            diff = np.abs(gpu_lse[fin].astype(np.float64) - rl[fin])
            bound = LSE_ABS + LSE_REL * np.abs(rl[fin].astype(np.float64))
            d = float(diff.max())
            assert (diff <= bound).all(), f"{label}: lse max abs {d:.3e} (bound {float(bound.max()):.3e})"
    if g.size:
        RESULTS.append((label, mx, rel, d if gpu_lse is not None and fin.any() else None))
        print(f"[parity] {label}: max abs {mx:.3e}, rel rms {rel:.3e}"
              + (f", lse max abs {d:.3e}" if gpu_lse is not None and fin.any() else ""))


def sample_units(B, H, NT, n, seed, must=()):
    """Seeded sample of flat unit ids, always including `must` (e.g. tails)."""
    rng = np.random.default_rng(seed)
    total = B * H * NT
    picked = set(int(u) for u in must if 0 <= u < total)
    while len(picked) < min(n, total):
        picked.add(int(rng.integers(total)))
    return sorted(picked)


def assert_parity_elementwise(gpu: np.ndarray, ref: np.ndarray, block_sizes, units, NT, T, gpu_lse=None,
                              ref_lse=None, label=""):
    """Element-by-element comparison for inputs that carry NaN or +-Inf in
    valid rows: every element the oracle (rounded to FP32) gives as NaN, +Inf
    or -Inf must be exactly that on the GPU, and the finite elements meet the
    same bar as ``assert_parity`` (max abs and relative RMS over them).  A
    non-finite value in a valid V row reaches only some columns of the rows
    that select it, so rows are not required to be all-NaN here."""
    bs = np.asarray(block_sizes)
    ref32 = ref.astype(np.float32)
    n = gpu.shape[0]
    valid = np.zeros((n, T), dtype=bool)
    for i, (_, t) in enumerate(unit_rows(units, NT, T)):
        valid[i, :int(bs[t])] = True
    assert (gpu[~valid].view(np.uint32) == 0).all(), f"{label}: padding rows not +0"
    g, r = gpu[valid], ref32[valid]
    for name, f in (("NaN", np.isnan), ("+Inf", np.isposinf), ("-Inf", np.isneginf)):
        bad = f(g) != f(r)
        assert not bad.any(), f"{label}: {int(bad.sum())} elements differ in being {name}"
    fin = np.isfinite(r)
    err = np.abs(g[fin].astype(np.float64) - r[fin])
    mx = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(r[fin].astype(np.float64)), 1e-30))
    assert mx <= MAX_ABS and rel <= REL_RMS, f"{label}: max abs {mx:.3e}, rel rms {rel:.3e}"
    if gpu_lse is not None:
        gl, rl = gpu_lse[valid], ref_lse.astype(np.float32)[valid]
        for name, f in (("NaN", np.isnan), ("+Inf", np.isposinf), ("-Inf", np.isneginf)):
            assert (f(gl) == f(rl)).all(), f"{label}: lse differs in being {name}"
        lf = np.isfinite(rl)
        diff = np.abs(gl[lf].astype(np.float64) - rl[lf])
        assert (diff <= LSE_ABS + LSE_REL * np.abs(rl[lf].astype(np.float64))).all(), f"{label}: lse"
    print(f"[parity] {label}: {int((~fin).sum())} non-finite elements matched, "
          f"finite max abs {mx:.3e}, rel rms {rel:.3e}")


def expected_step_counts(q2k_idx, q2k_num, block_sizes, T):
    """(tail, full) key-tile steps the attention kernel reports for a valid
    selection, counted on the host: one step per (query kernel tile, selected
    key kernel tile with a valid key); tail when the key tile is partly filled.
    Kernel tiles are the caller's tiles, or the 128-token halves of 256-token
    tiles (both halves of a query tile run, each against every key half)."""
    idx = np.asarray(q2k_idx).reshape(-1, np.asarray(q2k_idx).shape[-1]) if np.asarray(q2k_idx).size else None
    num = np.asarray(q2k_num).reshape(-1)
    bs = np.asarray(block_sizes).astype(np.int64)
    if T == 256:
        halves = np.stack([np.clip(bs, 0, 128), np.clip(bs - 128, 0, 128)], axis=1)  # [NT, 2]
        per_key_tail = ((halves > 0) & (halves < 128)).sum(1)
        per_key_full = (halves == 128).sum(1)
        q_mult = 2
    else:
        per_key_tail = ((bs > 0) & (bs < T)).astype(np.int64)
        per_key_full = (bs == T).astype(np.int64)
        q_mult = 1
    tail = full = 0
    for row in range(num.shape[0]):
        n = int(num[row])
        if n == 0:
            continue
        sel = idx[row, :n]
        tail += int(per_key_tail[sel].sum())
        full += int(per_key_full[sel].sum())
    return q_mult * tail, q_mult * full
