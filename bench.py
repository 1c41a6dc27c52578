"""Benchmark: block-sparse attention forward on one GB300 per rank.

One step = the whole hot path on one batch of synthetic input: the fused tile
layout of token-major Q/K/V, the on-device work ordering, and the tcgen05
attention kernel with LSE.  Default workload: the dense-limit case of the
FastVideo kernel page's Attn-QAT SM100 commit -- 6 heads, 31200 tokens (244
tiles of 128, last tile 96), head_dim 128, every query tile selecting every key
tile, bf16, LSE on.

Prints ONE JSON line (rank 0).  ``value`` is effective TFLOPS on selected tiles
(4*D*sum n_t*n_j over the selected tile pairs, valid tokens only) over the
device-timed step; ``e2e`` repeats the measurement through the C ABI from
pinned host buffers with the host<->device copies inside the timed region.
After the headline step (and outside it) the default run also times the
backward pass of the same workload (``bwd``) and, each on its own, the other
workloads (``workloads``: the tiny, uniform, ragged 64-token and video top-k
cases, and the dense case re-tiled with 64-token tiles at head_dim 128 and 64
and with 256-token tiles), each with its attention roofline and, for
token-major inputs, its layout roofline.
With ``--impl reference`` the CPU oracle is timed instead, on a bounded sample
of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "effective BF16 TFLOPS on selected tiles"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per attention launch from one ncu capture of
# dram__bytes_read.sum + dram__bytes_write.sum, keyed by workload and by the
# hash of the attention kernel code the capture was taken with
# (_attn_source_hash); a changed kernel reports null until it is captured again.
ATTN_TRAFFIC = {
    ("dense_b1h6d128_s31200_t128x244_lse", "bed0972dfe06b682"): 254.28e6,  # 220.6 MB read + 33.7 MB written
    ("uniform_b1h12d128_t128x128_k32", "bed0972dfe06b682"): 207.98e6,      # 173.5 MB read + 34.5 MB written
    # (both captured at 89a00684306c1328; the one later change compiles the split
    # tail's range code out of the 64-token kernels only)
}

# Workloads timed after the headline step in the default run (attention, and
# the tile layout where the inputs are token-major): (label, cfg, tile, head_dim).
EXTRA_WORKLOADS = (
    ("tiny", 1, None, None),
    ("uniform", 2, None, None),
    ("ragged_t64", 3, None, None),
    ("video_topk", 4, None, None),
    ("dense_t64_d128", 5, 64, None),
    ("dense_t64_d64", 5, 64, 64),
    ("dense_t256", 5, 256, None),
)


def _rank_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), d.get("hbm_gbs", FALLBACK_HBM_GBS), "measured"
    return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


def _attn_source_hash():
    """SHA-256 (first 16 hex digits) of the attention kernel's code: the source
    with `//` comments, trailing blanks and empty lines removed, so that a
    comment edit keeps the key of a capture taken with the same code."""
    with open(os.path.join(ROOT, "block_sparse_attention_gathered_gb300", "csrc", "vsa_attn.cu")) as f:
        lines = (line.split("//", 1)[0].rstrip() for line in f)
        code = "\n".join(line for line in lines if line)
    return hashlib.sha256(code.encode()).hexdigest()[:16]


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.start = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # start timing only once the sampler is producing lines
            t0 = time.monotonic()
            while not self.lines and self.proc.poll() is None and time.monotonic() - t0 < 5.0:
                time.sleep(0.01)
            self.start = len(self.lines)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[self.start:]:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _cpu_sample_units(w, budget_s: float, nthreads: int):
    """Pick a bounded, seeded sample of query tiles for the oracle, sized from a
    one-tile probe to take about ``budget_s`` on ``nthreads`` host threads."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(1234)
    total = w.B * w.H * w.NT
    refs = [oracle.tile_layout(x, w.row_to_token, w.NT, w.T) for x in (w.q_tok, w.k_tok, w.v_tok)] \
        if w.token_major else [x for x in (w.q, w.k, w.v)]
    t0 = time.perf_counter()
    oracle.block_sparse_attention(refs[0], refs[1], refs[2], w.q2k_idx, w.q2k_num, w.block_sizes, w.T,
                                  w.scale, units=[0], nthreads=1)
    one = max(time.perf_counter() - t0, 1e-3)
    n = int(max(1, min(total, budget_s * nthreads / one)))
    n = max(n - n % nthreads, min(total, nthreads))
    units = sorted(rng.choice(total, size=min(n, total), replace=False).tolist())
    return refs, units


def _unit_flops(w, units):
    bs = w.block_sizes.tolist()
    D = w.D
    tot = 0
    for u in units:
        b, h, t = u // (w.H * w.NT), (u // w.NT) % w.H, u % w.NT
        sel = w.q2k_idx[b, h, t, :int(w.q2k_num[b, h, t])].tolist()
        tot += 4 * D * bs[t] * sum(bs[j] for j in sel)
    return tot


def cpu_oracle_run(w, budget_s: float):
    import oracle
    nthreads = oracle.default_threads()
    refs, units = _cpu_sample_units(w, budget_s, nthreads)
    t0 = time.perf_counter()
    oracle.block_sparse_attention(refs[0], refs[1], refs[2], w.q2k_idx, w.q2k_num, w.block_sizes, w.T, w.scale,
                                  units=units, want_lse=w.want_lse, nthreads=nthreads)
    dt = time.perf_counter() - t0
    fl = _unit_flops(w, units)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{len(units)} of {w.B * w.H * w.NT} query tiles of {w.name} (seeded), "
                      f"{fl:.3e} effective flops in {dt:.1f} s, FP64"}


def run_reference(args, cfg):
    rank, world, _ = _rank_env()
    if rank != 0:
        return
    w = W.make_workload(cfg, tile=args.tile, head_dim=args.head_dim)
    import oracle
    oracle.build()
    nthreads = oracle.default_threads()
    # each step times the oracle on a sample sized so that the whole run stays
    # within a few minutes
    refs, units = _cpu_sample_units(w, min(4.0, 150.0 / max(1, args.steps + args.warmup)), nthreads)
    fl = _unit_flops(w, units)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.block_sparse_attention(refs[0], refs[1], refs[2], w.q2k_idx, w.q2k_num, w.block_sizes, w.T,
                                      w.scale, units=units, want_lse=w.want_lse, nthreads=nthreads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    val = fl / (ms / 1e3) / 1e12
    sample = f"{len(units)} of {w.B * w.H * w.NT} query tiles of {w.name} per step (seeded), FP64"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def config_dict(w, eff=None) -> dict:
    """The ``config`` object of a bench line: the same keys for both arms."""
    if eff is None:
        eff = W.effective_flops(w)
    return {"workload": w.name, "B": w.B, "H": w.H, "S": w.S or w.Sp, "head_dim": w.D, "tile": w.T,
            "num_tiles": w.NT, "density": round(density(w), 4), "lse": w.want_lse, "effective_flops": eff,
            "padded_flops": W.padded_flops(w), "l2": "flushed (256 MB write) between steps",
            "step": ("tile layout (q,k,v) + " if w.token_major else "") + "work ordering + tcgen05 attention"}


def density(w) -> float:
    """Fraction of (query tile, key tile) pairs selected."""
    return float(w.q2k_num.sum()) / float(w.B * w.H * w.NT * w.NT)


def layout_bytes(w) -> int:
    """Algorithmic bytes of one tile-layout launch: every token's q/k/v head
    vectors read once, every tile-major row (padding included) written once,
    plus the 4-byte row map."""
    return 3 * 2 * w.B * w.H * w.D * (w.S + w.Sp) + 4 * w.Sp


def selected_flops(q2k_idx, q2k_num, block_sizes, D: int) -> int:
    """4*D*sum over selected (b,h,t,j) of n_t*n_j for a selection given as tensors."""
    bs = block_sizes.to(torch.int64)
    B, H, NT, K = q2k_idx.shape
    live = torch.arange(K)[None, None, None, :] < q2k_num[..., None].to(torch.int64)
    nj = torch.where(live, bs[q2k_idx.clamp(min=0).to(torch.int64)], torch.zeros((), dtype=torch.int64))
    return int(4 * D * (nj.sum(-1) * bs[None, None, :]).sum())


def pooled_bytes(w) -> int:
    """Bytes the tile pooling reads: every valid row of q and k once."""
    return 2 * w.B * w.H * int(w.block_sizes.sum()) * w.D * 2


def max_over_ranks(x: float, device) -> float:
    """The largest value of ``x`` over all ranks (``x`` itself on one rank)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(eff_flops_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job effective TFLOP/s: every rank runs one full problem (weak
    scaling, independent replicas), timed by the slowest rank."""
    return world * eff_flops_per_rank / (ms_max / 1e3) / 1e12


def time_workload(vsa, w, dev, steps: int, warmup: int, flush) -> dict:
    """Times one workload on its own: the tile layout (token-major inputs only)
    and the forward call (work ordering + attention), each with CUDA events on
    the launching stream, L2 flushed before every step.  Returns its roofline
    entry for the bench line."""
    B, H, D, T, NT, S, Sp = w.B, w.H, w.D, w.T, w.NT, w.S, w.Sp
    stream = torch.cuda.current_stream()
    idx, num, bs = w.q2k_idx.to(dev), w.q2k_num.to(dev), w.block_sizes.to(dev)
    if w.token_major:
        src = [x.to(dev) for x in (w.q_tok, w.k_tok, w.v_tok)]
        r2t = w.row_to_token.to(dev)
        tiles = [torch.empty((B, H, Sp, D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    else:
        tiles = [x.to(dev) for x in (w.q, w.k, w.v)]
    out = torch.empty((B, H, Sp, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, Sp), dtype=torch.float32, device=dev) if w.want_lse else None
    dims = vsa.make_dims(B, H, NT, T, D, idx.shape[-1], w.scale)
    ws = torch.empty(vsa.vsa_block_sparse_workspace_size(dims), dtype=torch.uint8, device=dev)

    def one():
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        if w.token_major:
            vsa.vsa_tile_layout(src[0], src[1], src[2], tiles[0], tiles[1], tiles[2], r2t, B, S, H, D, NT, T,
                                stream)
        e[1].record(stream)
        vsa.vsa_block_sparse_fwd(tiles[0], tiles[1], tiles[2], idx, num, bs, out, lse, dims, ws, stream)
        e[2].record(stream)
        return e

    for _ in range(max(warmup, 3)):
        one()
    torch.cuda.synchronize()
    marks = []
    for _ in range(steps):
        flush.zero_()
        marks.append(one())
    torch.cuda.synchronize()
    if vsa.vsa_check_device_status() != 0:
        raise RuntimeError(f"device status error on {w.name}")
    route = vsa.vsa_last_route()
    tail, full = vsa.vsa_last_step_counts()
    peak, hbm, _ = _peaks()
    eff = W.effective_flops(w)
    attn = sum(m[1].elapsed_time(m[2]) for m in marks) / steps
    ach = eff / (attn / 1e3) / 1e12
    entry = {"workload": w.name, "attn_ms": attn, "effective_flops": eff, "padded_flops": W.padded_flops(w),
             "achieved": ach, "unit": UNIT, "frac": ach / peak, "density": round(density(w), 4),
             "layout": "paired" if route["layout"] == vsa.VSA_LAYOUT_PAIRED else "split",
             "kernel": f"attn_fwd_kernel<{min(T, 128)},{D}>", "grid": route["grid"],
             "work_items": route["work_items"], "stages": route["stages"],
             "steps_tail_full": [tail, full], "timed_calls": steps}
    if w.token_major:
        lay = sum(m[0].elapsed_time(m[1]) for m in marks) / steps
        gbs = layout_bytes(w) / (lay / 1e3) / 1e9
        entry["layout_ms"] = lay
        entry["layout_roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                    "frac": gbs / hbm, "bytes": layout_bytes(w)}
    return entry


def run_ours(args, cfg):
    import block_sparse_attention_gathered_gb300 as vsa

    rank, world, local = _rank_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.make_workload(cfg, tile=args.tile, head_dim=args.head_dim)
    token = w.token_major
    eff = W.effective_flops(w)
    B, H, D, T, NT, S = w.B, w.H, w.D, w.T, w.NT, w.S
    Sp = w.Sp

    if token:
        q_tok, k_tok, v_tok = (x.to(dev) for x in (w.q_tok, w.k_tok, w.v_tok))
        r2t = w.row_to_token.to(dev)
        tiles = [torch.empty((B, H, Sp, D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    else:
        # tile-major inputs (the ragged workload's NaN/Inf padding must reach
        # the kernel as it is): no layout step
        tiles = [x.to(dev) for x in (w.q, w.k, w.v)]
    idx, num, bs = w.q2k_idx.to(dev), w.q2k_num.to(dev), w.block_sizes.to(dev)
    out = torch.empty((B, H, Sp, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, Sp), dtype=torch.float32, device=dev) if w.want_lse else None
    select = bool(args.select)
    if select:
        # the step also selects the key tiles on the GPU (coarse stage), and
        # the attention runs on that selection
        topk = int(w.notes["topk"])
        sel_dims = vsa.make_dims(B, H, NT, T, D, topk)
        sel_ws = torch.empty(vsa.vsa_coarse_select_workspace_size(sel_dims), dtype=torch.uint8, device=dev)
        idx = torch.empty((B, H, NT, topk), dtype=torch.int32, device=dev)
        num = torch.empty((B, H, NT), dtype=torch.int32, device=dev)
    untile = bool(args.untile)
    if untile:
        # the step ends with the un-tiling of the output, times a gate
        gate = (torch.rand((B, S, H, D), generator=torch.Generator().manual_seed(W.SEED_BASE + 100)) * 2
                ).to(torch.bfloat16).to(dev)
        out_tok = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    dims = vsa.make_dims(B, H, NT, T, D, idx.shape[-1], w.scale)
    ws = torch.empty(vsa.vsa_block_sparse_workspace_size(dims), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > 129 MB L2
    stream = torch.cuda.current_stream()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def step():
        """One pass of the hot path; returns events before the step, after the
        layout, after the selection (the same event when there is none), after
        the attention call and after the un-tiling (recorded on the launching
        stream)."""
        l0, a1 = ev(), ev()
        l0.record(stream)
        l1 = l0
        if token:
            vsa.vsa_tile_layout(q_tok, k_tok, v_tok, tiles[0], tiles[1], tiles[2], r2t, B, S, H, D, NT, T, stream)
            l1 = ev()
            l1.record(stream)
        s1 = l1
        if select:
            vsa.vsa_coarse_select(tiles[0], tiles[1], bs, topk, idx, num, sel_dims, sel_ws, stream)
            s1 = ev()
            s1.record(stream)
        vsa.vsa_block_sparse_fwd(tiles[0], tiles[1], tiles[2], idx, num, bs, out, lse, dims, ws, stream)
        a1.record(stream)
        u1 = a1
        if untile:
            vsa.vsa_untile(out, gate, out_tok, r2t, B, S, H, D, NT, T, stream)
            u1 = ev()
            u1.record(stream)
        return l0, l1, s1, a1, u1

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step()
    barrier()
    if vsa.vsa_check_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    if select:  # effective FLOPs of the selection the GPU made
        eff = selected_flops(idx.cpu(), num.cpu(), w.block_sizes, D)

    # ---------------------------------------------------------------- device-timed steps
    marks = []
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        for _ in range(args.steps):
            flush.zero_()  # L2 flush, outside the timed events
            marks.append(step())
        barrier()
    step_ms = [m[0].elapsed_time(m[4]) for m in marks]
    untile_ms = [m[3].elapsed_time(m[4]) for m in marks] if untile else None
    layout_ms = [m[0].elapsed_time(m[1]) for m in marks] if token else None
    select_ms = [m[1].elapsed_time(m[2]) for m in marks] if select else None
    attn_ms = [m[2].elapsed_time(m[3]) for m in marks]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), dev)
    if vsa.vsa_check_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    route = vsa.vsa_last_route()
    steps_tail_full = list(vsa.vsa_last_step_counts())

    # ---------------------------------------------------------------- backward (outside the step)
    bwd_line = None
    if args.bwd and w.want_lse:
        dout = torch.randn((B, H, Sp, D), generator=torch.Generator().manual_seed(W.SEED_BASE + 200)).to(
            torch.bfloat16).to(dev)
        grads = [torch.empty_like(out) for _ in range(3)]
        bdims = vsa.make_dims(B, H, NT, T, D, idx.shape[-1], w.scale)
        bws = torch.empty(vsa.vsa_block_sparse_bwd_workspace_size(bdims), dtype=torch.uint8, device=dev)

        def bwd_step():
            vsa.vsa_block_sparse_bwd(tiles[0], tiles[1], tiles[2], out, dout, lse, idx, num, bs, grads[0],
                                     grads[1], grads[2], bdims, bws, stream)

        step()
        for _ in range(max(args.warmup, 3)):
            bwd_step()
        barrier()
        b_marks = []
        for _ in range(max(3, args.steps // 5)):
            flush.zero_()
            b0, b1 = ev(), ev()
            b0.record(stream)
            bwd_step()
            b1.record(stream)
            b_marks.append((b0, b1))
        barrier()
        if vsa.vsa_check_device_status() != 0:
            raise RuntimeError("device status error in the backward")
        b_ms = sum(a.elapsed_time(b) for a, b in b_marks) / len(b_marks)
        b_flops = 2.5 * eff  # dV, dP, dS-weighted dQ and dK, plus S: 5 products of the forward's 2
        bwd_line = {"ms": b_ms, "effective_flops": b_flops, "achieved": b_flops / (b_ms / 1e3) / 1e12,
                    "unit": "TFLOP/s", "frac": b_flops / (b_ms / 1e3) / 1e12 / _peaks()[0],
                    "timed_calls": len(b_marks), "kernels": "delta, pairs, k2q transpose, dK/dV, dQ (tcgen05)"}

    # ---------------------------------------------------------------- end to end from host buffers
    if token:
        hq, hk, hv = (x.pin_memory() for x in (w.q_tok, w.k_tok, w.v_tok))
        h_in = ((q_tok, hq), (k_tok, hk), (v_tok, hv), (bs, w.block_sizes.pin_memory()),
                (r2t, w.row_to_token.pin_memory()))
    else:
        h_in = tuple((d_, h_.pin_memory()) for d_, h_ in zip(tiles, (w.q, w.k, w.v))) + \
            ((bs, w.block_sizes.pin_memory()),)
    # with the GPU selection the selection arrays are outputs, not inputs
    if not select:
        h_in = h_in + ((idx, w.q2k_idx.pin_memory()), (num, w.q2k_num.pin_memory()))
    hout = torch.empty((B, H, Sp, D), dtype=torch.bfloat16).pin_memory()
    if untile:  # the gate is an input too, and the token-major output is read back
        hgate = gate.cpu().pin_memory()
        h_in = h_in + ((gate, hgate),)
        hout = torch.empty((B, S, H, D), dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty((B, H, Sp), dtype=torch.float32).pin_memory() if lse is not None else None
    h2d = sum(h_.numel() * h_.element_size() for _, h_ in h_in)
    d2h = hout.numel() * 2 + (hlse.numel() * 4 if hlse is not None else 0)

    def e2e_step():
        for d_, h_ in h_in:
            d_.copy_(h_, non_blocking=True)
        step()
        hout.copy_(out_tok if untile else out, non_blocking=True)
        if hlse is not None:
            hlse.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    barrier()
    e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e_ms.append((e0, e1))
    barrier()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e_ms) / len(e_ms), dev)

    # ---------------------------------------------------------------- other workloads (outside the step)
    extra = {}
    if args.extra and rank == 0:
        for label, c, tile, hd in EXTRA_WORKLOADS:
            if (c, tile or 128, hd or 128) == (cfg, args.tile or 128, args.head_dim or 128):
                continue  # the headline workload itself
            extra[label] = time_workload(vsa, W.make_workload(c, tile=tile, head_dim=hd), dev, args.extra_steps,
                                         3, flush)

    peak, hbm, src = _peaks()
    attn_avg = sum(attn_ms) / len(attn_ms)
    achieved = eff / (attn_avg / 1e3) / 1e12
    traffic = ATTN_TRAFFIC.get((w.name, _attn_source_hash()))
    if rank == 0:
        config = config_dict(w, eff)
        line = {
            "metric": METRIC, "value": aggregate(eff, world, ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config,
            "attn_ms": attn_avg,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{src} bf16 burst (cuBLAS)",
                         "kernel": f"attn_fwd_kernel<{min(T, 128)},{D},"
                                   f"{'paired' if route.get('layout') == vsa.VSA_LAYOUT_PAIRED else 'split'}>"},
            "e2e": {"value": aggregate(eff, world, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            # per step: [tile layout,] [tile pooling, selection,] work-ordering sort, attention,
            # [split-tail merge,] [un-tiling]
            "gpu_launches": ((1 if token else 0) + 2 + (2 if select else 0) + (1 if route.get("tail_parts", 0) > 1 else 0)
                             + (1 if untile else 0)) * args.steps,
            "clocks": clk.summary(),
            "route": route,
            "steps_tail_full": steps_tail_full,
        }
        if token:
            lay_avg = sum(layout_ms) / len(layout_ms)
            lay_gbs = layout_bytes(w) / (lay_avg / 1e3) / 1e9
            line["layout_ms"] = lay_avg
            line["layout_roofline"] = {"bound": "hbm", "achieved": lay_gbs, "peak": hbm, "unit": "GB/s",
                                       "frac": lay_gbs / hbm, "bytes": layout_bytes(w),
                                       "peak_source": f"{src} HBM copy", "kernel": "layout_kernel"}
        if select:
            sel_avg = sum(select_ms) / len(select_ms)
            pool_bytes = pooled_bytes(w)
            line["select_ms"] = sel_avg
            line["select_roofline"] = {
                "bound": "hbm", "achieved": pool_bytes / (sel_avg / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": pool_bytes / (sel_avg / 1e3) / 1e9 / hbm, "bytes": pool_bytes,
                "kernel": "pool_kernel + select_kernel (bytes: valid rows of q and k read once)"}
            line["config"]["step"] = "tile layout + coarse top-k selection + work ordering + tcgen05 attention"
            line["config"]["topk"] = topk
        if untile:
            ut_avg = sum(untile_ms) / len(untile_ms)
            ut_bytes = 3 * B * S * H * D * 2 + 4 * NT * T  # output rows and gate read, token output written, map
            line["untile_ms"] = ut_avg
            line["untile_roofline"] = {
                "bound": "hbm", "achieved": ut_bytes / (ut_avg / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": ut_bytes / (ut_avg / 1e3) / 1e9 / hbm, "bytes": ut_bytes, "kernel": "untile_kernel (gated)"}
            line["config"]["step"] += " + un-tiling with gate"
        if bwd_line is not None:
            line["bwd"] = bwd_line
        if extra:
            line["workloads"] = extra
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_oracle_run(w, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tile", type=int, default=None, choices=[64, 128, 256],
                    help="dense-limit workload only: tile size (default 128)")
    ap.add_argument("--head-dim", type=int, default=None, choices=[64, 128],
                    help="dense-limit workload only: head_dim (default 128)")
    ap.add_argument("--no-bwd", dest="bwd", action="store_false",
                    help="skip the backward timing (reported under \"bwd\", outside the step)")
    ap.add_argument("--no-extra", dest="extra", action="store_false",
                    help="skip timing the other workloads (reported under \"workloads\")")
    ap.add_argument("--extra-steps", type=int, default=20)
    ap.add_argument("--untile", action="store_true",
                    help="end the step with the un-tiling of the output times a gate")
    ap.add_argument("--select", action="store_true",
                    help="video-grid workload only: select the key tiles on the GPU inside the step")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if (args.tile not in (None, 128) or args.head_dim not in (None, 128)) and args.config != 5:
        ap.error("--tile and --head-dim re-shape the dense-limit workload (--config 5) only")
    if args.select and args.config != 4:
        ap.error("--select needs the video-grid workload (--config 4)")
    if args.impl == "reference":
        run_reference(args, args.config)
    else:
        run_ours(args, args.config)


if __name__ == "__main__":
    main()
