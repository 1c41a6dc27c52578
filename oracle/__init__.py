"""CPU oracle for the block-sparse attention forward pass (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never loads it and it
loads nothing of the GPU library: the two share no code.  The arithmetic lives
in ``vsa_oracle.c`` (plain C, FP64, threads over query tiles); this module only
builds that file with gcc and marshals numpy arrays into it.

Every function here states the definition it follows in ``vsa_oracle.c``:
FastVideo commit 8503617 (fastvideo-kernel/python), the commits that add and
harden the sm_121a tile-128 block-sparse forward, the fused ``tile_to_bhsd``
layout commit, and the Attn-QAT SM100 commit (softmax statistics).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lib = None

ERRORS = {-1: "bad argument", -7: "bad key-tile selection (range or duplicate)", -8: "out of memory"}


def build(force: bool = False) -> str:
    """Compile ``vsa_oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, no fused
    multiply-add, no fast-math) and return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
                               "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_block_sparse_fwd.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64,
                                                P, i64, P, P, i32]
        lib.oracle_block_sparse_fwd.restype = i32
        lib.oracle_tile_layout.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32]
        lib.oracle_tile_layout.restype = i32
        lib.oracle_coarse_select.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P, P, P]
        lib.oracle_coarse_select.restype = i32
        lib.oracle_untile.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32]
        lib.oracle_untile.restype = i32
        lib.oracle_block_sparse_bwd.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, P, P, P, i32]
        lib.oracle_block_sparse_bwd.restype = i32
        _lib = lib
    return _lib


def _bf16_bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 bit array (numpy) -> contiguous uint16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def block_sparse_attention(q, k, v, q2k_idx, q2k_num, block_sizes, T: int, scale: float,
                           units: Optional[Sequence[int]] = None, want_lse: bool = True,
                           nthreads: Optional[int] = None):
    """FP64 block-sparse attention forward for tile-major bf16 ``q, k, v``
    ``[B, H, NT*T, D]``.

    ``units`` lists flat query-tile ids ``(b*H + h)*NT + t`` (default: all).
    Returns ``(out [n_units, T, D] float64, lse [n_units, T] float64 or None)``.
    """
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    B, H, Sp, D = qb.shape
    assert kb.shape == qb.shape and vb.shape == qb.shape and Sp % T == 0
    NT = Sp // T
    idx, num, bs = _i32(q2k_idx), _i32(q2k_num), _i32(block_sizes)
    assert num.shape == (B, H, NT) and idx.shape[:3] == (B, H, NT) and bs.shape == (NT,)
    max_kv = int(idx.shape[3])
    if units is None:
        units = np.arange(B * H * NT, dtype=np.int64)
    u = np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    out = np.zeros((len(u), T, D), dtype=np.float64)
    lse = np.zeros((len(u), T), dtype=np.float64) if want_lse else None
    rc = _load().oracle_block_sparse_fwd(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(idx), _ptr(num), _ptr(bs), B, H, NT, T, D, max_kv,
        float(scale), _ptr(u), len(u), _ptr(out), _ptr(lse) if lse is not None else None,
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_block_sparse_fwd: {ERRORS.get(rc, rc)}")
    return out, lse


def block_sparse_attention_bwd(q, k, v, dout, q2k_idx, q2k_num, block_sizes, T: int, scale: float,
                               nthreads: Optional[int] = None):
    """FP64 gradients (dq, dk, dv) of the block-sparse forward for tile-major
    bf16 ``q, k, v`` and upstream gradient ``dout`` ``[B, H, NT*T, D]``; each is a
    float64 array of the same shape (see ``oracle_block_sparse_bwd``)."""
    qb, kb, vb, db = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v), _bf16_bits(dout)
    B, H, Sp, D = qb.shape
    NT = Sp // T
    idx, num, bs = _i32(q2k_idx), _i32(q2k_num), _i32(block_sizes)
    max_kv = int(idx.shape[3])
    dq, dk, dv = (np.empty((B, H, Sp, D), dtype=np.float64) for _ in range(3))
    rc = _load().oracle_block_sparse_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), _ptr(idx), _ptr(num), _ptr(bs),
                                         B, H, NT, T, D, max_kv, float(scale), _ptr(dq), _ptr(dk), _ptr(dv),
                                         int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_block_sparse_bwd: {ERRORS.get(rc, rc)}")
    return dq, dk, dv


def tile_layout(x_tok, row_to_token, NT: int, T: int) -> np.ndarray:
    """Token-major bf16 ``[B, S, H, D]`` -> tile-major bf16 bits ``[B, H, NT*T, D]``
    (uint16); rows mapped to -1 are written as +0."""
    src = _bf16_bits(x_tok)
    B, S, H, D = src.shape
    r2t = _i32(row_to_token)
    assert r2t.shape == (NT * T,)
    dst = np.empty((B, H, NT * T, D), dtype=np.uint16)
    rc = _load().oracle_tile_layout(_ptr(src), _ptr(r2t), _ptr(dst), B, S, H, D, NT, T)
    if rc != 0:
        raise ValueError(f"oracle_tile_layout: {ERRORS.get(rc, rc)}")
    return dst


def coarse_select(q, k, block_sizes, T: int, topk: int, want_scores: bool = True):
    """Coarse key-tile selection (see ``oracle_coarse_select`` in vsa_oracle.c):
    tile means of the valid rows, tile-level q.k scores, the ``topk`` best key
    tiles per query tile (ties to the smaller index), all in fp32 with sums in
    index order.  ``q, k``: tile-major bf16 ``[B, H, NT*T, D]``.

    Returns ``(q2k_idx [B,H,NT,topk] int32 ascending, -1 padded;
    q2k_num [B,H,NT] int32; scores [B,H,NT,NT] float32 or None)``.
    """
    qb, kb = _bf16_bits(q), _bf16_bits(k)
    B, H, Sp, D = qb.shape
    assert kb.shape == qb.shape and Sp % T == 0
    NT = Sp // T
    bs = _i32(block_sizes)
    assert bs.shape == (NT,)
    idx = np.empty((B, H, NT, topk), dtype=np.int32)
    num = np.empty((B, H, NT), dtype=np.int32)
    sc = np.empty((B, H, NT, NT), dtype=np.float32) if want_scores else None
    rc = _load().oracle_coarse_select(_ptr(qb), _ptr(kb), _ptr(bs), B, H, NT, T, D, int(topk), _ptr(idx),
                                      _ptr(num), _ptr(sc) if sc is not None else None)
    if rc != 0:
        raise ValueError(f"oracle_coarse_select: {ERRORS.get(rc, rc)}")
    return idx, num, sc


def untile(o_tile, gate_tok, row_to_token, S: int, T: int, out=None) -> np.ndarray:
    """Tile-major bf16 ``o_tile [B, H, NT*T, D]`` -> token-major bf16 bits
    ``[B, S, H, D]``, times ``gate_tok`` (bf16 ``[B, S, H, D]``) when given, one
    round-to-nearest-even per element (see ``oracle_untile``).  Tokens no row
    maps to keep the values of ``out`` (zeros by default)."""
    ob = _bf16_bits(o_tile)
    B, H, Sp, D = ob.shape
    NT = Sp // T
    gb = _bf16_bits(gate_tok) if gate_tok is not None else None
    r2t = _i32(row_to_token)
    assert r2t.shape == (Sp,)
    dst = np.zeros((B, S, H, D), dtype=np.uint16) if out is None else np.ascontiguousarray(out, dtype=np.uint16)
    rc = _load().oracle_untile(_ptr(ob), _ptr(gb) if gb is not None else None, _ptr(r2t), _ptr(dst), B, S, H, D,
                               NT, T)
    if rc != 0:
        raise ValueError(f"oracle_untile: {ERRORS.get(rc, rc)}")
    return dst


def bits_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
