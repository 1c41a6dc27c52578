"""Host-side checks of the C-ABI library (no GPU needed).

The library must load, export every entry point declared in include/vsa.h,
and reject bad arguments and over-limit sizes with a status code before it
touches the device (the sm_121a hardening commit on the FastVideo kernel page:
limits are checked before launch; errors are reported, never silently
accepted).  Pointers below are fake but never dereferenced: every call fails
its host-side checks first.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def vsa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_gathered_gb300 as V
    return V


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "vsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vsa_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(vsa):
    declared = _declared_symbols()
    assert len(declared) >= 8
    lib = ctypes.CDLL(vsa.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(vsa.EXPORTED)
    assert vsa.vsa_version() == 1002


def test_status_strings(vsa):
    for code in range(0, -9, -1):
        s = vsa.vsa_status_string(code)
        assert s and s != "unknown status"
    assert vsa.vsa_status_string(-99) == "unknown status"


FAKE = 0x100000  # 16-byte aligned, never dereferenced


def _fwd(vsa, dims, q=FAKE, k=FAKE, v=FAKE, idx=FAKE, num=FAKE, bs=FAKE, out=FAKE, lse=None,
         ws=FAKE, ws_bytes=1 << 30):
    P = ctypes.c_void_p
    return vsa.library().vsa_block_sparse_fwd(P(q), P(k), P(v), P(idx), P(num), P(bs), P(out),
                                               P(lse) if lse else None, ctypes.byref(dims), P(ws),
                                               ws_bytes, None)


def test_argument_errors(vsa):
    ok = vsa.make_dims(1, 2, 4, 64, 64, 2)
    assert _fwd(vsa, vsa.make_dims(1, 2, 4, 32, 64, 2)) == vsa.VSA_ERR_ARG          # tile
    assert _fwd(vsa, vsa.make_dims(1, 2, 4, 64, 96, 2)) == vsa.VSA_ERR_ARG          # head_dim
    assert _fwd(vsa, vsa.make_dims(0, 2, 4, 64, 64, 2)) == vsa.VSA_ERR_ARG          # batch
    assert _fwd(vsa, vsa.make_dims(1, 2, 0, 64, 64, 2)) == vsa.VSA_ERR_ARG          # tiles
    assert _fwd(vsa, vsa.make_dims(1, 2, 4, 64, 64, -1)) == vsa.VSA_ERR_ARG         # max_kv
    assert _fwd(vsa, vsa.make_dims(1, 2, 4, 64, 64, 2, float("nan"))) == vsa.VSA_ERR_ARG
    assert _fwd(vsa, ok, q=0) == vsa.VSA_ERR_ARG
    assert _fwd(vsa, ok, out=0) == vsa.VSA_ERR_ARG
    assert _fwd(vsa, ok, num=0) == vsa.VSA_ERR_ARG
    assert _fwd(vsa, ok, q=FAKE + 8) == vsa.VSA_ERR_ALIGN
    assert _fwd(vsa, ok, out=FAKE + 2) == vsa.VSA_ERR_ALIGN
    assert _fwd(vsa, ok, lse=FAKE + 2) == vsa.VSA_ERR_ALIGN
    assert _fwd(vsa, ok, ws=0) == vsa.VSA_ERR_WORKSPACE
    assert _fwd(vsa, ok, ws_bytes=16) == vsa.VSA_ERR_WORKSPACE


def test_launch_limits(vsa):
    # batch * heads <= 65535
    assert _fwd(vsa, vsa.make_dims(256, 256, 4, 64, 64, 2)) == vsa.VSA_ERR_LIMITS
    assert vsa.vsa_block_sparse_workspace_size(vsa.make_dims(256, 256, 4, 64, 64, 2)) == 0
    # kernel tiles < 2^22 (the hardening commit's MaxTiles)
    assert vsa.VSA_MAX_TILES == (1 << 22) - 1
    assert vsa.vsa_block_sparse_workspace_size(vsa.make_dims(1, 1, (1 << 22) - 1, 64, 64, 2)) > 0
    assert vsa.vsa_block_sparse_workspace_size(vsa.make_dims(1, 1, 1 << 22, 64, 64, 2)) == 0
    assert _fwd(vsa, vsa.make_dims(1, 1, 1 << 22, 64, 64, 2)) == vsa.VSA_ERR_LIMITS
    # rows < 2^31
    assert _fwd(vsa, vsa.make_dims(16, 4096, 8192, 128, 64, 2)) == vsa.VSA_ERR_LIMITS
    assert _fwd(vsa, vsa.make_dims(65535, 1, 257, 128, 128, 1)) == vsa.VSA_ERR_LIMITS


def test_tile_256_limits(vsa):
    # 256-token tiles run as two 128-token halves, and the limit counts halves
    half = (1 << 21) - 1   # 2 * half = 2^22 - 2 kernel tiles
    assert vsa.vsa_block_sparse_workspace_size(vsa.make_dims(1, 2, half, 256, 128, 2)) > 0
    assert vsa.vsa_block_sparse_workspace_size(vsa.make_dims(1, 2, half + 1, 256, 128, 2)) == 0
    assert _fwd(vsa, vsa.make_dims(1, 2, half + 1, 256, 128, 2)) == vsa.VSA_ERR_LIMITS
    assert _fwd(vsa, vsa.make_dims(1, 2, 4, 512, 128, 2)) == vsa.VSA_ERR_ARG
    # the backward and the coarse selection keep 8192 kernel tiles
    assert vsa.vsa_block_sparse_bwd_workspace_size(vsa.make_dims(1, 2, 4096, 256, 128, 2)) > 0
    assert vsa.vsa_block_sparse_bwd_workspace_size(vsa.make_dims(1, 2, 4097, 256, 128, 2)) == 0
    assert vsa.vsa_block_sparse_bwd_workspace_size(vsa.make_dims(1, 1, 8192, 64, 64, 2)) > 0
    assert vsa.vsa_block_sparse_bwd_workspace_size(vsa.make_dims(1, 1, 8193, 64, 64, 2)) == 0
    assert vsa.vsa_coarse_select_workspace_size(vsa.make_dims(1, 1, 8193, 64, 64, 2)) == 0


def _with_tail(base, items, D):
    """The full forward workspace: beyond 128 work items, the split tail's
    region after the base (256-byte aligned): 256 work-item slots, 256 pieces
    of 128 (row maximum, row sum) pairs, 256 pieces of 128 fp32 O rows."""
    if items <= 128:
        return base
    return (base + 255) // 256 * 256 + 256 * 4 + 256 * 128 * 8 + 256 * 128 * D * 4


def test_bitmap_workspace_beyond_shared_memory(vsa):
    # up to 8192 kernel tiles the selection bitmaps live in shared memory and
    # the workspace is the header plus the order list; beyond, each CTA (at
    # most 1024, at most one per work item) gets 2 x 5 bitmaps in the workspace
    # (two buffers of the four slot bitmaps and the partial-tile bitmap)
    small = vsa.make_dims(1, 1, 8192, 64, 64, 2)
    items = 8192 * 64 // 256
    assert vsa.vsa_block_sparse_workspace_size_min(small) == 256 + 4 * (items + 256)
    assert vsa.vsa_block_sparse_workspace_size(small) == _with_tail(256 + 4 * (items + 256), items, 64)
    big = vsa.make_dims(1, 1, 8200, 64, 64, 2)
    items = 8200 * 64 // 256
    order = 256 + 4 * (items + 256)
    words = (8200 + 31) // 32
    base = ((order + 255) // 256) * 256 + 1024 * 2 * 5 * words * 4
    assert vsa.vsa_block_sparse_workspace_size_min(big) == base
    assert vsa.vsa_block_sparse_workspace_size(big) == _with_tail(base, items, 64)
    few = vsa.make_dims(1, 1, 8200, 256, 64, 2)  # 16400 kernel tiles, 8200 work items
    words = (16400 + 31) // 32
    order = 256 + 4 * (8200 + 256)
    base = ((order + 255) // 256) * 256 + 1024 * 2 * 5 * words * 4
    assert vsa.vsa_block_sparse_workspace_size_min(few) == base
    assert vsa.vsa_block_sparse_workspace_size(few) == _with_tail(base, 8200, 64)
    # one 256-row work item per 256-token tile
    assert vsa.vsa_block_sparse_workspace_size(vsa.make_dims(2, 3, 10, 256, 64, 4)) == 256 + 4 * (6 * 10 + 256)


def test_workspace_size(vsa):
    # header (256 bytes) + one int32 per 256-query-row work item, + 256 for
    # the entries of a partial last wave split into one-unit entries; beyond
    # 128 work items, the split tail's partial results
    d = vsa.make_dims(1, 6, 244, 128, 128, 244)
    assert vsa.vsa_block_sparse_workspace_size_min(d) == 256 + 4 * (6 * 122 + 256)
    assert vsa.vsa_block_sparse_workspace_size(d) == _with_tail(256 + 4 * (6 * 122 + 256), 6 * 122, 128)
    assert vsa.vsa_block_sparse_workspace_size(d) - vsa.vsa_block_sparse_workspace_size_min(d) < 18 << 20
    d = vsa.make_dims(2, 8, 63, 64, 64, 31)
    assert vsa.vsa_block_sparse_workspace_size(d) == _with_tail(256 + 4 * (16 * 16 + 256), 16 * 16, 64)
    d = vsa.make_dims(1, 2, 10, 128, 64, 4)   # 10 work items: no split tail region
    assert vsa.vsa_block_sparse_workspace_size(d) == 256 + 4 * (10 + 256)
    assert vsa.vsa_block_sparse_workspace_size_min(d) == vsa.vsa_block_sparse_workspace_size(d)
    assert vsa.vsa_block_sparse_workspace_size_min(vsa.make_dims(256, 256, 4, 64, 64, 2)) == 0


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("B,H,NT,T,D,max_kv", [(1, 6, 244, 128, 128, 244), (2, 8, 63, 64, 64, 32),
                                              (1, 2, 3, 256, 128, 3), (1, 1, 1, 64, 64, 0)])
def test_bwd_workspace_size(vsa, B, H, NT, T, D, max_kv):
    """The backward workspace: -delta and -lse*log2(e) per row of whole 128-row
    kernel tiles, partner counts and lists, transposed offsets and lists."""
    d = vsa.make_dims(B, H, NT, T, D, max_kv)
    BH = B * H
    NTk = (NT + 1) // 2 if T == 64 else (NT if T == 128 else 2 * NT)
    maxlen = max(1, min(NTk, (1 if T == 128 else 2) * max(max_kv, 1)))
    Spk = NTk * 128
    lists = 4 * BH * NTk * maxlen
    want = (256 + 2 * _align256(4 * BH * Spk) + _align256(4 * BH * NTk) + _align256(lists)
            + _align256(4 * BH * (NTk + 1)) + _align256(lists))
    assert vsa.vsa_block_sparse_bwd_workspace_size(d) == want


def test_bwd_workspace_size_invalid(vsa):
    assert vsa.vsa_block_sparse_bwd_workspace_size(vsa.make_dims(1, 1, 4, 96, 64, 2)) == 0    # tile
    assert vsa.vsa_block_sparse_bwd_workspace_size(vsa.make_dims(1, 1, 4, 128, 96, 2)) == 0   # head_dim
    assert vsa.vsa_block_sparse_bwd_workspace_size(vsa.make_dims(256, 256, 4, 64, 64, 2)) == 0  # B*H


def test_layout_argument_errors(vsa):
    P = ctypes.c_void_p
    L = vsa.library().vsa_tile_layout
    f = lambda *a: L(*[P(x) if x else None for x in a[:7]], *a[7:], None)
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 8, 2, 64, 1, 8) == vsa.VSA_ERR_ARG       # map
    assert f(FAKE, 0, 0, FAKE, FAKE, 0, FAKE, 1, 8, 2, 64, 1, 8) == vsa.VSA_ERR_ARG            # pair
    assert f(0, 0, 0, 0, 0, 0, FAKE, 1, 8, 2, 64, 1, 8) == vsa.VSA_ERR_ARG                     # none
    assert f(FAKE, 0, 0, FAKE, 0, 0, FAKE, 1, 8, 2, 60, 1, 8) == vsa.VSA_ERR_ARG               # D%8
    assert f(FAKE + 4, 0, 0, FAKE, 0, 0, FAKE, 1, 8, 2, 64, 1, 8) == vsa.VSA_ERR_ALIGN


def test_validate_argument_errors(vsa):
    P = ctypes.c_void_p
    d = vsa.make_dims(1, 2, 4, 64, 64, 2)
    V = vsa.library().vsa_validate_indices
    assert V(P(FAKE), P(FAKE), P(FAKE), ctypes.byref(d), None, None) == vsa.VSA_ERR_ARG
    assert V(P(FAKE), P(FAKE + 2), P(FAKE), ctypes.byref(d), P(FAKE), None) == vsa.VSA_ERR_ALIGN


def test_untile_argument_errors(vsa):
    P = ctypes.c_void_p
    U = vsa.library().vsa_untile
    f = lambda o, g, out, m, *a: U(P(o) if o else None, P(g) if g else None, P(out) if out else None,
                                   P(m) if m else None, *a, None)
    assert f(0, 0, FAKE, FAKE, 1, 8, 2, 64, 1, 8) == vsa.VSA_ERR_ARG            # no input
    assert f(FAKE, 0, FAKE, 0, 1, 8, 2, 64, 1, 8) == vsa.VSA_ERR_ARG            # no map
    assert f(FAKE, 0, FAKE, FAKE, 1, 8, 2, 60, 1, 8) == vsa.VSA_ERR_ARG         # D % 8
    assert f(FAKE, FAKE + 8, FAKE, FAKE, 1, 8, 2, 64, 1, 8) == vsa.VSA_ERR_ALIGN  # gate
    assert f(FAKE, 0, FAKE + 4, FAKE, 1, 8, 2, 64, 1, 8) == vsa.VSA_ERR_ALIGN   # output
    assert f(FAKE, 0, FAKE, FAKE, 256, 8, 256, 64, 1, 8) == vsa.VSA_ERR_LIMITS  # batch * heads


def test_coarse_select_argument_errors(vsa):
    P = ctypes.c_void_p
    d = vsa.make_dims(1, 2, 4, 64, 64, 0)
    S = vsa.library().vsa_coarse_select
    need = vsa.vsa_coarse_select_workspace_size(d)
    assert need == 2 * 1 * 2 * 4 * 64 * 4  # fp32 tile means of q and k

    def f(q=FAKE, k=FAKE, bs=FAKE, topk=2, idx=FAKE, num=FAKE, dims=d, ws=FAKE, ws_bytes=need):
        return S(P(q) if q else None, P(k) if k else None, P(bs) if bs else None, topk,
                 P(idx) if idx else None, P(num) if num else None, ctypes.byref(dims),
                 P(ws) if ws else None, ws_bytes, None)

    assert f(q=0) == vsa.VSA_ERR_ARG
    assert f(num=0) == vsa.VSA_ERR_ARG
    assert f(topk=-1) == vsa.VSA_ERR_ARG
    assert f(idx=0) == vsa.VSA_ERR_ARG                    # topk > 0 needs q2k_idx
    assert f(topk=8193) == vsa.VSA_ERR_LIMITS
    assert f(dims=vsa.make_dims(1, 2, 4, 48, 64, 0)) == vsa.VSA_ERR_ARG
    assert f(k=FAKE + 8) == vsa.VSA_ERR_ALIGN
    assert f(idx=FAKE + 2) == vsa.VSA_ERR_ALIGN
    assert f(ws=0) == vsa.VSA_ERR_WORKSPACE
    assert f(ws_bytes=need - 1) == vsa.VSA_ERR_WORKSPACE
    assert vsa.vsa_coarse_select_workspace_size(vsa.make_dims(256, 256, 4, 64, 64, 0)) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_is_an_error_not_a_launch(vsa):
    st = _fwd(vsa, vsa.make_dims(1, 2, 4, 64, 64, 2))
    assert st in (vsa.VSA_ERR_CUDA, vsa.VSA_ERR_ARCH)
    assert vsa.vsa_check_device_status(0) in (vsa.VSA_ERR_CUDA, vsa.VSA_ERR_ARCH)


def test_wait_probe_argument_errors(vsa):
    # limit checked before any device work (no GPU here)
    assert vsa.library().vsa_wait_probe(0, 0, None) == vsa.VSA_ERR_ARG
    assert vsa.library().vsa_wait_probe(0, 2000001, None) == vsa.VSA_ERR_ARG
    assert vsa.library().vsa_wait_probe(0, 1000, None) in (vsa.VSA_ERR_CUDA, vsa.VSA_ERR_ARCH)


def test_binding_structs_match_the_header(vsa, tmp_path):
    """The ctypes mirrors of vsa_dims and vsa_route have the C structs' size
    and field offsets (a C program built against include/vsa.h reports them),
    so a field added on one side only is caught without a GPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"vsa_dims": vsa.VsaDims, "vsa_route": vsa.VsaRoute}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "vsa.h"', 'int main(void) {']
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ['  return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)
