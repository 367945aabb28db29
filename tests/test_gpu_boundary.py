"""The block boundary on the GPU (moe_boundary) against the oracle: the sandwich post-norm
of the block output, the residual add and the next block's pre-norm ("vLLM 对 Muse Spark
Open 的 Day 0 支持", section "三明治归一化"; "SGLang and Miles Add Day-0 Support for Muse
Spark Open", section "Kernel Optimizations").

x' is compared with the oracle on the same inputs, h' with the oracle's pre-norm of the
GPU's own stored x' (stage-wise): each stored value equal to the oracle's or one unit
of the storage format away (FP32 sums in a different order than float64 may flip a
rounding), on at most 1 % of the elements for BF16 storage.  Row counts cover one row, the cluster path
(few rows: several CTAs share each row through distributed shared memory) and the
one-CTA-per-row path.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F

pytestmark = pytest.mark.gpu


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    build.build()


def unit(v, kind):
    bits = {"bf16": 7, "f32": 23}[kind]
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 1e-30)
    return np.exp2(np.floor(np.log2(a)) - bits)


def assert_one_unit(name, gpu, ref, kind):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(gpu - ref)
    u = unit(np.maximum(np.abs(gpu), np.abs(ref)), kind)
    bad = d > u * (1 + 1e-9) + 1e-6 * float(np.sqrt(np.mean(ref * ref)))
    assert not np.any(bad), (name, int(bad.sum()), float(d[bad].max()))
    frac = float(np.mean(d > 0))
    if kind == "bf16":
        # a BF16 rounding flips only where FP32 and float64 straddle a boundary; FP32
        # storage shows every last-bit difference of the FP32 arithmetic instead
        assert frac <= 0.01, (name, frac)
    return frac


def run_case(T, d, act, out, gated, inplace=False, seed=0):
    from latent_moe_layer_rmsnorm_gb300 import synth
    from latent_moe_layer_rmsnorm_gb300 import _lib as L
    gen = torch.Generator(device="cpu").manual_seed(1000 + seed)
    xdt = torch.float32 if act == "f32" else torch.bfloat16
    ydt = torch.float32 if out == "f32" else torch.bfloat16
    x = torch.randn((T, d), generator=gen).to(xdt)
    y = (torch.randn((T, d), generator=gen) * 3.0).to(ydt)
    g_post = torch.rand(d, generator=gen) + 0.5
    g_next = torch.rand(d, generator=gen) + 0.5
    gate = (torch.rand(d, generator=gen) * 2.0 - 0.5) if gated else None
    shape = synth.Shape("boundary", T=T, d=d, p=128, E=8, top_k=2, I=128,
                        act="f32" if act == "f32" else "bf16",
                        expert="f32" if act == "f32" else "bf16")
    cfg = L.moe_config_t(T=T, d=d, p=128, E=8, top_k=2, I=128, eps=shape.eps,
                         act=L.MOE_F32 if act == "f32" else L.MOE_BF16,
                         expert=L.MOE_F32 if act == "f32" else L.MOE_BF16,
                         out=L.MOE_F32 if out == "f32" else L.MOE_BF16, flags=0)
    xd, yd = x.cuda(), y.cuda()
    gp, gn = g_post.cuda(), g_next.cuda()
    gt = gate.cuda() if gated else None
    x_out = xd if inplace else torch.empty_like(xd)
    h_next = torch.empty_like(xd)
    st = torch.cuda.current_stream().cuda_stream
    x_before = xd.clone()
    rc = L.moe_boundary(cfg, xd.data_ptr(), yd.data_ptr(), gp.data_ptr(),
                        None if gt is None else gt.data_ptr(), gn.data_ptr(),
                        x_out.data_ptr(), h_next.data_ptr(), st)
    assert rc == L.MOE_OK
    torch.cuda.synchronize()
    kind = "f32" if act == "f32" else "bf16"
    xr, _ = oracle.boundary(x_before.float().cpu().numpy(), y.float().numpy(), g_post.numpy(),
                            g_next.numpy(), shape.eps,
                            gate=None if gate is None else gate.numpy(), act=kind)
    xg = x_out.float().cpu().numpy()
    fx = assert_one_unit("x_out", xg, xr, kind)
    hr = oracle.store(oracle.rmsnorm(xg, g_next.numpy(), shape.eps), kind)
    fh = assert_one_unit("h_next", h_next.float().cpu().numpy(), hr, kind)
    return fx, fh


@pytest.mark.parametrize("T", [1, 64, 1000])
@pytest.mark.parametrize("d", [256, 8192])
def test_boundary_bf16_stream(T, d):
    need_gpu()
    for out in ("f32", "bf16"):
        for gated in (False, True):
            run_case(T, d, "bf16", out, gated, seed=T + d)


def test_boundary_f32_stream_and_in_place():
    need_gpu()
    run_case(300, 1024, "f32", "f32", True, seed=3)
    run_case(64, 8192, "bf16", "bf16", True, inplace=True, seed=4)
    run_case(2, 32768, "bf16", "f32", False, seed=5)      # widest rows: 4+ CTAs per row


def test_boundary_after_the_block():
    """The boundary applied to moe_forward's own output equals the oracle's boundary of
    the oracle's block output (end to end, within the block's own tolerance)."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300 import synth
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    from harness import fix_margins, oracle_view, rel_err, to_np
    shape = synth.Shape("mid_bf16", T=300, d=1024, p=1024, E=16, top_k=4, I=512)
    inp = synth.make_inputs(shape, seed=6, device="cpu")
    fix_margins(inp, shape, seed=6)
    dev = {k: v.cuda() for k, v in inp.items()}
    layer = LatentMoE(shape, dev, out="f32")
    y = layer.forward(dev["x"])
    gen = torch.Generator(device="cpu").manual_seed(7)
    g_post = (torch.rand(shape.d, generator=gen) + 0.5)
    g_next = (torch.rand(shape.d, generator=gen) + 0.5)
    x_out, h_next = layer.boundary(dev["x"], y, g_post.cuda(), g_next.cuda())
    torch.cuda.synchronize()
    ref = oracle.moe_forward(oracle_view(inp), top_k=shape.top_k, eps=shape.eps, act="bf16",
                             expert="bf16", out="f32")
    xr, hr = oracle.boundary(to_np(inp["x"]), ref, g_post.numpy(), g_next.numpy(), shape.eps,
                             act="bf16")
    # the block's own bound (1e-2 of rms) plus one BF16 unit of each stored value: an
    # error far below a unit can still flip a rounding of x'; h' also carries a flipped
    # unit of x' scaled by its norm factor and gain
    rs = 1.0 / np.sqrt(np.mean(xr * xr, axis=-1, keepdims=True) + shape.eps)
    carried = unit(np.abs(xr), "bf16") * rs * g_next.numpy()
    for name, g, r, extra in (("x_out", to_np(x_out), xr, 0.0),
                              ("h_next", to_np(h_next), hr, carried)):
        rms = float(np.sqrt(np.mean(r * r)))
        bad = np.abs(g - r) > (1e-2 * rms + unit(np.abs(r), "bf16") + extra) * (1 + 1e-9)
        assert not np.any(bad), (name, int(bad.sum()), rel_err(g, r))
