"""Device-side failure detection, exercised without faulting or hanging the GPU.

The test hook MOE_FLAG_TEST_TIMEOUT makes the gate/up GEMM skip its first operand
load, so one pipeline stage never fills.  Every wait in the kernel is bounded: the MMA
wait gives up after 20 ms, the kernel drains the copies it did issue, frees its tensor
memory and returns; the call's status word then holds MOE_ERR_TIMEOUT.  The context
must stay usable: the next normal call succeeds and reproduces the earlier result.
"""
import pytest
import torch

from latent_moe_layer_rmsnorm_gb300 import _lib as L
from latent_moe_layer_rmsnorm_gb300 import synth

pytestmark = pytest.mark.gpu

WAIT_MMA_FULL = 2
WAIT_PRODUCER_EMPTY = 1
WAIT_EPI_TMEM_FULL = 4


def test_bounded_wait_reports_timeout_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    build.build()
    shape = synth.Shape("err_bf16", T=96, d=512, p=256, E=8, top_k=2, I=256)
    inp = {k: v.cuda() for k, v in synth.make_inputs(shape, seed=4, device="cpu").items()}
    layer = LatentMoE(shape, inp, out="f32")
    good = layer.forward(inp["x"]).clone()
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)

    layer.forward(inp["x"], flags=L.MOE_FLAG_TEST_TIMEOUT)
    status, detail = layer.read_status()
    assert status == L.MOE_ERR_TIMEOUT
    assert detail in (WAIT_MMA_FULL, WAIT_PRODUCER_EMPTY, WAIT_EPI_TMEM_FULL)
    # read_status cleared the word; the context still works and gives the same bits
    again = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    assert torch.equal(again, good)


def test_invalid_replay_ids_are_reported_not_written():
    """Expert ids outside [0, E) in a routing replay are counted nowhere, written
    nowhere, and reported as MOE_ERR_DEVICE_CHECK."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    build.build()
    shape = synth.Shape("err_bf16", T=64, d=512, p=256, E=8, top_k=2, I=256)
    inp = {k: v.cuda() for k, v in synth.make_inputs(shape, seed=5, device="cpu").items()}
    layer = LatentMoE(shape, inp, out="f32")
    ids, w = layer.route(inp["x"])
    ids[3, 1] = 99
    ids[10, 0] = -4
    layer.forward(inp["x"], ids=ids, w=w)
    status, detail = layer.read_status()
    assert status == L.MOE_ERR_DEVICE_CHECK and detail == 16
    ok_ids, ok_w = layer.route(inp["x"])
    layer.forward(inp["x"], ids=ok_ids, w=ok_w)
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
