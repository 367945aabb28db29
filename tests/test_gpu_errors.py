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


# ---- value-range checks of the FP16 / NVFP4 intermediates ----------------------------------
CHECK_H_RANGE, CHECK_U_RANGE, CHECK_C_RANGE, CHECK_S_RANGE = 18, 19, 20, 21


def _layer(shape, seed, **over):
    from latent_moe_layer_rmsnorm_gb300 import build
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    build.build()
    host = synth.make_inputs(shape, seed=seed, device="cpu")
    host.update(over)
    inp = {k: v.cuda() for k, v in host.items()}
    return LatentMoE(shape, inp, out="f32"), inp


def test_fp16_overflow_of_h_is_reported():
    """A row with one large entry normalises to sqrt(d) at that entry; with a gain of
    4000 there, h = 32 * 4000 at d = 1024, beyond FP16's 65504: the full-width norm
    reports it instead of storing inf for the pooler.  The other rows stay in range,
    and the next call with ordinary gains reads MOE_OK."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    shape = synth.Shape("err_bf16", T=32, d=1024, p=256, E=8, top_k=2, I=256)
    host = synth.make_inputs(shape, seed=6, device="cpu")
    g_in = host["g_in"].clone()
    g_in[0] = 4000.0
    x = host["x"].clone()
    x[0] = 0
    x[0, 0] = 100.0
    layer, inp = _layer(shape, 6, g_in=g_in, x=x)
    layer.forward(inp["x"])
    assert layer.read_status() == (L.MOE_ERR_DEVICE_CHECK, CHECK_H_RANGE)
    x2 = inp["x"].clone()
    x2[0] = inp["x"][1]                # no spike: |h| stays far below the FP16 maximum
    layer.forward(x2)
    assert layer.read_status() == (0, 0)


def test_fp16_overflow_of_c_from_replay_weights_is_reported():
    """Replayed route weights of 5e4 each make c = sum_j w_j * RMSNorm(y_j) reach ~1e5,
    beyond FP16: the combine reports it.  The same ids with the router's weights are
    fine."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    shape = synth.Shape("err_bf16", T=32, d=512, p=256, E=8, top_k=2, I=256)
    layer, inp = _layer(shape, 7)
    ids, w = layer.route(inp["x"])
    layer.forward(inp["x"], ids=ids, w=torch.full_like(w, 5e4))
    assert layer.read_status() == (L.MOE_ERR_DEVICE_CHECK, CHECK_C_RANGE)
    layer.forward(inp["x"], ids=ids, w=w)
    assert layer.read_status() == (0, 0)


def test_nvfp4_requant_scale_saturation_is_reported():
    """A static global scale for the requantised SwiGLU output that is far too small
    (1e-7 instead of 64 / 2688) would clip every block's scale at 448: the gate/up
    epilogue reports it.  The calibrated scale reads MOE_OK."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    shape = synth.Shape("err_nvfp4", T=64, d=512, p=256, E=4, top_k=2, I=256, expert="nvfp4")
    good = synth.nvfp4_act2_scales(shape, "cpu")
    layer, inp = _layer(shape, 8, gs_act2=torch.full_like(good, 1e-7))
    layer.forward(inp["x"])
    assert layer.read_status() == (L.MOE_ERR_DEVICE_CHECK, CHECK_S_RANGE)
    layer2, inp2 = _layer(shape, 8)
    layer2.forward(inp2["x"])
    assert layer2.read_status() == (0, 0)
