"""The failure path of the bounded waits, on the GPU, without faulting it:
a warp waits on a barrier phase that nothing completes, gives up after a
short limit, reports VSA_ERR_TIMEOUT through the device status word and
returns; the context stays usable for the next call."""
import time

import pytest
import torch

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


def test_completed_phase_is_not_a_timeout(vsa):
    assert vsa.vsa_wait_probe(True, 20000) == vsa.VSA_OK
    assert vsa.vsa_check_device_status() == vsa.VSA_OK


def test_wait_that_nothing_completes_times_out(vsa):
    t0 = time.perf_counter()
    assert vsa.vsa_wait_probe(False, 20000) == vsa.VSA_OK  # 20 ms
    st = vsa.vsa_check_device_status()
    dt = time.perf_counter() - t0
    assert st == vsa.VSA_ERR_TIMEOUT
    assert 0.015 < dt < 5.0
    # the word was cleared by the read, and the device keeps working
    assert vsa.vsa_check_device_status() == vsa.VSA_OK
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn((1, 1, 128, 64), generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    idx = torch.zeros((1, 1, 1, 1), dtype=torch.int32, device="cuda")
    num = torch.ones((1, 1, 1), dtype=torch.int32, device="cuda")
    bs = torch.full((1,), 128, dtype=torch.int32, device="cuda")
    out = vsa.block_sparse_attention(q, k, v, idx, num, bs, 128)
    ref = torch.softmax(q.float()[0, 0] @ k.float()[0, 0].T / 8.0, -1) @ v.float()[0, 0]
    assert (out.float()[0, 0] - ref).abs().max().item() < 2e-2
    assert vsa.vsa_check_device_status() == vsa.VSA_OK
