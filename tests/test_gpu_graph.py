"""The forward path captured in a CUDA graph: tile layout, work ordering and
attention replay from the graph with the same results as eager calls (the
work counter is reset by the ordering kernel on every replay), and a replay
after new inputs are copied in reflects the new inputs."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_gathered_gb300 as V
    return V


def test_forward_replays_from_a_cuda_graph(vsa):
    w = W.make_workload(2)
    dev = "cuda"
    B, H, D, T, NT, S = w.B, w.H, w.D, w.T, w.NT, w.S
    q_tok, k_tok, v_tok = (x.to(dev) for x in (w.q_tok, w.k_tok, w.v_tok))
    r2t = w.row_to_token.to(dev)
    idx, num, bs = w.q2k_idx.to(dev), w.q2k_num.to(dev), w.block_sizes.to(dev)
    tiles = [torch.empty((B, H, NT * T, D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    out = torch.empty((B, H, NT * T, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, NT * T), dtype=torch.float32, device=dev)
    dims = vsa.make_dims(B, H, NT, T, D, idx.shape[-1], w.scale)
    ws = torch.empty(vsa.vsa_block_sparse_workspace_size(dims), dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream()

    def run(stream):
        vsa.vsa_tile_layout(q_tok, k_tok, v_tok, tiles[0], tiles[1], tiles[2], r2t, B, S, H, D, NT, T, stream)
        vsa.vsa_block_sparse_fwd(tiles[0], tiles[1], tiles[2], idx, num, bs, out, lse, dims, ws, stream)

    # eager reference (also does the one-time per-device setup outside capture)
    with torch.cuda.stream(side):
        run(side)
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run(side)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert vsa.vsa_check_device_status() == 0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse)
    # new inputs copied into the captured buffers show up in the next replay
    q_tok.copy_(torch.flip(q_tok, dims=[1]))
    graph.replay()
    torch.cuda.synchronize()
    assert not torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    with torch.cuda.stream(side):
        run(side)
    torch.cuda.synchronize()
    eager = out.clone()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
