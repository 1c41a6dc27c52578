"""GB300 (sm_103a) block-sparse attention forward: Python binding.

A thin ``ctypes`` layer over the C ABI in ``include/vsa.h`` (library
``_build/libvsa.so``).  It only marshals arguments -- tensor pointers, sizes,
the current CUDA stream -- every step of the computation runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  There
is no CPU fallback: if the library is missing, importing the binding raises.

The functions named ``vsa_*`` mirror the C entry points one to one.  The
helpers ``block_sparse_attention`` and ``tile_layout`` allocate outputs and
the workspace with torch and call them.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libvsa.so")

VSA_OK, VSA_ERR_ARG, VSA_ERR_ALIGN, VSA_ERR_LIMITS, VSA_ERR_ARCH = 0, -1, -2, -3, -4
VSA_ERR_CUDA, VSA_ERR_TIMEOUT, VSA_ERR_INDEX, VSA_ERR_WORKSPACE = -5, -6, -7, -8
VSA_KERNEL_NONE, VSA_KERNEL_ATTN_TCGEN05, VSA_KERNEL_LAYOUT, VSA_KERNEL_VALIDATE = 0, 1, 2, 3
VSA_KERNEL_SELECT, VSA_KERNEL_UNTILE, VSA_KERNEL_BWD = 4, 5, 6
VSA_LAYOUT_SPLIT, VSA_LAYOUT_PAIRED = 0, 1  # vsa_route.layout: MMA-issue layout of the attention kernel
VSA_MAX_BATCH_HEADS, VSA_MAX_TILES, VSA_MAX_TILES_BWD, VSA_SMEM_BITMAP_TILES = 65535, (1 << 22) - 1, 8192, 8192


class VsaDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("num_tiles", ctypes.c_int32),
                ("tile", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("max_kv", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class VsaRoute(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("tile", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("block", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("work_items", ctypes.c_int64), ("sort_bins", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("layout", ctypes.c_int32), ("tail_parts", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class VsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {vsa_status_string(status)} ({status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libvsa.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                           "or python block_sparse_attention_gathered_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    dims_p = ctypes.POINTER(VsaDims)
    sig = {
        "vsa_block_sparse_workspace_size": ([dims_p], sz),
        "vsa_block_sparse_workspace_size_min": ([dims_p], sz),
        "vsa_block_sparse_fwd": ([P, P, P, P, P, P, P, P, dims_p, P, sz, P], i32),
        "vsa_block_sparse_fwd_noalloc": ([P, P, P, P, P, P, P, P, dims_p, P], i32),
        "vsa_tile_layout": ([P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P], i32),
        "vsa_validate_indices": ([P, P, P, dims_p, P, P], i32),
        "vsa_untile": ([P, P, P, P, i32, i32, i32, i32, i32, i32, P], i32),
        "vsa_block_sparse_bwd_workspace_size": ([dims_p], sz),
        "vsa_block_sparse_bwd": ([P] * 12 + [dims_p, P, sz, P], i32),
        "vsa_coarse_select_workspace_size": ([dims_p], sz),
        "vsa_coarse_select": ([P, P, P, i32, P, P, dims_p, P, sz, P], i32),
        "vsa_check_device_status": ([P], i32),
        "vsa_wait_probe": ([i32, ctypes.c_uint32, P], i32),
        "vsa_last_route": ([ctypes.POINTER(VsaRoute)], i32),
        "vsa_last_step_counts": ([ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)], i32),
        "vsa_status_string": ([i32], ctypes.c_char_p),
        "vsa_version": ([], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    return lib


_lib = _load()
EXPORTED = ("vsa_block_sparse_workspace_size", "vsa_block_sparse_workspace_size_min", "vsa_block_sparse_fwd", "vsa_block_sparse_fwd_noalloc",
            "vsa_block_sparse_bwd_workspace_size", "vsa_block_sparse_bwd", "vsa_tile_layout", "vsa_untile",
            "vsa_coarse_select_workspace_size", "vsa_coarse_select", "vsa_validate_indices",
            "vsa_check_device_status", "vsa_wait_probe", "vsa_last_route", "vsa_last_step_counts",
            "vsa_status_string", "vsa_version")


def library() -> ctypes.CDLL:
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_dims(B, H, num_tiles, tile, head_dim, max_kv, scale=None) -> VsaDims:
    return VsaDims(int(B), int(H), int(num_tiles), int(tile), int(head_dim), int(max_kv),
                   float(scale) if scale is not None else 0.0)


def vsa_status_string(status: int) -> str:
    return _lib.vsa_status_string(int(status)).decode()


def vsa_version() -> int:
    return int(_lib.vsa_version())


def vsa_wait_probe(arrive: bool, limit_us: int, stream=None) -> int:
    """Launches the bounded-wait probe; returns the launch status (the
    timeout, if any, shows in ``vsa_check_device_status``)."""
    return int(_lib.vsa_wait_probe(1 if arrive else 0, int(limit_us), _stream(stream)))


def vsa_block_sparse_workspace_size(dims: VsaDims) -> int:
    return int(_lib.vsa_block_sparse_workspace_size(ctypes.byref(dims)))


def vsa_block_sparse_workspace_size_min(dims: VsaDims) -> int:
    return int(_lib.vsa_block_sparse_workspace_size_min(ctypes.byref(dims)))


def vsa_block_sparse_fwd(q, k, v, q2k_idx, q2k_num, block_sizes, out, lse, dims: VsaDims,
                         workspace: torch.Tensor, stream=None) -> None:
    """Calls the C entry point on device tensors; raises VsaError on a status."""
    st = _lib.vsa_block_sparse_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(q2k_idx), _ptr(q2k_num),
                                   _ptr(block_sizes), _ptr(out), _ptr(lse), ctypes.byref(dims),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream))
    if st != VSA_OK:
        raise VsaError(st, "vsa_block_sparse_fwd")


VSA_NOALLOC_SCRATCH_BYTES = 1 << 20


def vsa_block_sparse_fwd_noalloc(q, k, v, q2k_idx, q2k_num, block_sizes, out, lse, dims: VsaDims,
                                 stream=None) -> None:
    """The forward pass without a workspace, for callers that cannot allocate
    device memory: the library's own fixed scratch array (1 MiB per GPU) is
    used instead.  Calls on one device must not overlap on the GPU."""
    st = _lib.vsa_block_sparse_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(q2k_idx), _ptr(q2k_num),
                                           _ptr(block_sizes), _ptr(out), _ptr(lse), ctypes.byref(dims),
                                           _stream(stream))
    if st != VSA_OK:
        raise VsaError(st, "vsa_block_sparse_fwd_noalloc")


def vsa_tile_layout(q_tok, k_tok, v_tok, q_tile, k_tile, v_tile, row_to_token, B, S, H, D,
                    num_tiles, tile, stream=None) -> None:
    st = _lib.vsa_tile_layout(_ptr(q_tok), _ptr(k_tok), _ptr(v_tok), _ptr(q_tile), _ptr(k_tile),
                              _ptr(v_tile), _ptr(row_to_token), int(B), int(S), int(H), int(D),
                              int(num_tiles), int(tile), _stream(stream))
    if st != VSA_OK:
        raise VsaError(st, "vsa_tile_layout")


def vsa_block_sparse_bwd_workspace_size(dims: VsaDims) -> int:
    return int(_lib.vsa_block_sparse_bwd_workspace_size(ctypes.byref(dims)))


def vsa_block_sparse_bwd(q, k, v, out, dout, lse, q2k_idx, q2k_num, block_sizes, dq, dk, dv, dims: VsaDims,
                         workspace: torch.Tensor, stream=None) -> None:
    st = _lib.vsa_block_sparse_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(q2k_idx),
                                   _ptr(q2k_num), _ptr(block_sizes), _ptr(dq), _ptr(dk), _ptr(dv),
                                   ctypes.byref(dims), _ptr(workspace),
                                   workspace.numel() * workspace.element_size() if workspace is not None else 0,
                                   _stream(stream))
    if st != VSA_OK:
        raise VsaError(st, "vsa_block_sparse_bwd")


def vsa_untile(o_tile, gate_tok, out_tok, row_to_token, B, S, H, D, num_tiles, tile, stream=None) -> None:
    st = _lib.vsa_untile(_ptr(o_tile), _ptr(gate_tok), _ptr(out_tok), _ptr(row_to_token), int(B), int(S), int(H),
                         int(D), int(num_tiles), int(tile), _stream(stream))
    if st != VSA_OK:
        raise VsaError(st, "vsa_untile")


def vsa_coarse_select_workspace_size(dims: VsaDims) -> int:
    return int(_lib.vsa_coarse_select_workspace_size(ctypes.byref(dims)))


def vsa_coarse_select(q, k, block_sizes, topk: int, q2k_idx, q2k_num, dims: VsaDims, workspace: torch.Tensor,
                      stream=None) -> None:
    st = _lib.vsa_coarse_select(_ptr(q), _ptr(k), _ptr(block_sizes), int(topk), _ptr(q2k_idx), _ptr(q2k_num),
                                ctypes.byref(dims), _ptr(workspace),
                                workspace.numel() * workspace.element_size() if workspace is not None else 0,
                                _stream(stream))
    if st != VSA_OK:
        raise VsaError(st, "vsa_coarse_select")


def vsa_validate_indices(q2k_idx, q2k_num, block_sizes, dims: VsaDims, dev_status: torch.Tensor,
                         stream=None) -> None:
    st = _lib.vsa_validate_indices(_ptr(q2k_idx), _ptr(q2k_num), _ptr(block_sizes),
                                   ctypes.byref(dims), _ptr(dev_status), _stream(stream))
    if st != VSA_OK:
        raise VsaError(st, "vsa_validate_indices")


def vsa_check_device_status(stream=None) -> int:
    return int(_lib.vsa_check_device_status(_stream(stream)))


def vsa_last_route() -> dict:
    r = VsaRoute()
    st = _lib.vsa_last_route(ctypes.byref(r))
    if st != VSA_OK:
        raise VsaError(st, "vsa_last_route")
    return r.as_dict()


def vsa_last_step_counts() -> tuple:
    """(tail_steps, full_steps) of the last forward call on the current device
    (waits for the device)."""
    tail, full = ctypes.c_int64(0), ctypes.c_int64(0)
    st = _lib.vsa_last_step_counts(ctypes.byref(tail), ctypes.byref(full))
    if st != VSA_OK:
        raise VsaError(st, "vsa_last_step_counts")
    return int(tail.value), int(full.value)


# ------------------------------------------------------------------ helpers
def _check_bf16_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("expected contiguous bf16 CUDA tensors")


def block_sparse_attention(q, k, v, q2k_idx, q2k_num, block_sizes, tile: int,
                           scale: Optional[float] = None, want_lse: bool = False,
                           out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                           stream=None):
    """Block-sparse attention forward on tile-major bf16 ``[B, H, NT*tile, D]``.

    Returns ``out`` (bf16, same shape) or ``(out, lse)`` with ``lse`` fp32
    ``[B, H, NT*tile]`` when ``want_lse``."""
    _check_bf16_cuda(q, k, v)
    B, H, Sp, D = q.shape
    if Sp % tile:
        raise ValueError("sequence length is not a multiple of the tile")
    NT = Sp // tile
    q2k_idx = q2k_idx.contiguous()
    dims = make_dims(B, H, NT, tile, D, q2k_idx.shape[-1], scale)
    if out is None:
        out = torch.empty_like(q)
    lse = torch.empty((B, H, Sp), dtype=torch.float32, device=q.device) if want_lse else None
    need = vsa_block_sparse_workspace_size(dims)
    if need == 0:
        raise VsaError(VSA_ERR_ARG if B * H <= VSA_MAX_BATCH_HEADS and NT <= VSA_MAX_TILES
                       else VSA_ERR_LIMITS, "vsa_block_sparse_workspace_size")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    vsa_block_sparse_fwd(q, k, v, q2k_idx, q2k_num.contiguous(), block_sizes.contiguous(), out, lse,
                         dims, workspace, stream)
    return (out, lse) if want_lse else out


def block_sparse_attention_bwd(q, k, v, out, dout, lse, q2k_idx, q2k_num, block_sizes, tile: int,
                               scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None,
                               stream=None):
    """Gradients ``(dq, dk, dv)`` (bf16, tile-major like ``q``) of the forward
    that produced ``out`` and ``lse``."""
    _check_bf16_cuda(q, k, v, out, dout)
    B, H, Sp, D = q.shape
    NT = Sp // tile
    q2k_idx = q2k_idx.contiguous()
    dims = make_dims(B, H, NT, tile, D, q2k_idx.shape[-1], scale)
    need = vsa_block_sparse_bwd_workspace_size(dims)
    if need == 0:
        raise VsaError(VSA_ERR_ARG, "vsa_block_sparse_bwd_workspace_size")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    vsa_block_sparse_bwd(q, k, v, out, dout, lse.contiguous(), q2k_idx, q2k_num.contiguous(),
                         block_sizes.contiguous(), dq, dk, dv, dims, workspace, stream)
    return dq, dk, dv


def coarse_select(q, k, block_sizes, tile: int, topk: int, workspace: Optional[torch.Tensor] = None,
                  stream=None):
    """Coarse key-tile selection on tile-major bf16 ``q, k`` ``[B, H, NT*tile, D]``:
    returns ``(q2k_idx [B, H, NT, topk] int32, q2k_num [B, H, NT] int32)``,
    ready for ``block_sparse_attention`` with ``max_kv = topk``."""
    _check_bf16_cuda(q, k)
    B, H, Sp, D = q.shape
    if Sp % tile:
        raise ValueError("sequence length is not a multiple of the tile")
    NT = Sp // tile
    dims = make_dims(B, H, NT, tile, D, topk)
    need = vsa_coarse_select_workspace_size(dims)
    if need == 0:
        raise VsaError(VSA_ERR_ARG, "vsa_coarse_select_workspace_size")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    idx = torch.empty((B, H, NT, topk), dtype=torch.int32, device=q.device)
    num = torch.empty((B, H, NT), dtype=torch.int32, device=q.device)
    vsa_coarse_select(q, k, block_sizes.contiguous(), topk, idx, num, dims, workspace, stream)
    return idx, num


def untile(o_tile, row_to_token, num_tokens: int, tile: int, gate_tok=None, out=None, stream=None):
    """Tile-major bf16 ``o_tile [B, H, NT*tile, D]`` -> token-major ``[B, S, H, D]``
    (times ``gate_tok`` when given)."""
    _check_bf16_cuda(o_tile, gate_tok)
    B, H, Sp, D = o_tile.shape
    if out is None:
        out = torch.zeros((B, num_tokens, H, D), dtype=torch.bfloat16, device=o_tile.device)
    vsa_untile(o_tile, gate_tok, out, row_to_token.contiguous(), B, num_tokens, H, D, Sp // tile, tile, stream)
    return out


def tile_layout(q_tok, k_tok, v_tok, row_to_token, num_tiles: int, tile: int, stream=None):
    """Token-major bf16 ``[B, S, H, D]`` (any of the three may be None) ->
    tile-major ``[B, H, num_tiles*tile, D]``; padding rows are +0."""
    src = [t for t in (q_tok, k_tok, v_tok)]
    ref = next(t for t in src if t is not None)
    _check_bf16_cuda(*src)
    B, S, H, D = ref.shape
    dst = [None if t is None else torch.empty((B, H, num_tiles * tile, D), dtype=torch.bfloat16,
                                              device=ref.device) for t in src]
    vsa_tile_layout(src[0], src[1], src[2], dst[0], dst[1], dst[2], row_to_token.contiguous(),
                    B, S, H, D, num_tiles, tile, stream)
    return tuple(dst)
