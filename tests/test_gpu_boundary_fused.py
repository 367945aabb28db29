"""The block and its boundary in one call (moe_forward_boundary): the post-norm of the block
output, the residual add and the next block's pre-norm run inside the unpooler GEMM's
kernel ("SGLang and Miles Add Day-0 Support for Muse Spark Open", section "Kernel
Optimizations": post-FFN norm, gated residual add and pre-attention norm fused; "vLLM 对
Muse Spark Open 的 Day 0 支持", section "三明治归一化").

Per case: the block output y equals moe_forward's bit for bit (same kernels); x' against
the oracle's boundary of the GPU's own y and x, and h' against the oracle's pre-norm of
the GPU's stored x', each stored value equal or one unit of the storage format apart
(BF16: on at most 1 % of the elements); the tile counters show that the row pass ran in
the unpooler (every 32-row block counted d / 256 column tiles) or, for shapes whose
unpooler runs split-K, that the separate pass ran instead (counters untouched).
"""
import numpy as np
import pytest
import torch

import oracle
from harness import fix_margins, to_np

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
        assert frac <= 0.01, (name, frac)
    return frac


def run_fused(T, act, out, gated, inplace, seed, expect_fused, d=8192, p=256, expert=None,
              replay=False):
    from latent_moe_layer_rmsnorm_gb300 import synth
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.Shape("fused_boundary", T=T, d=d, p=p, E=8, top_k=2, I=256,
                        act=act, expert=expert or act)
    inp = synth.make_inputs(shape, seed=seed, device="cpu")
    fix_margins(inp, shape, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    layer = LatentMoE(shape, dev, out=out)
    gen = torch.Generator(device="cpu").manual_seed(100 + seed)
    g_post = torch.rand(d, generator=gen) + 0.5
    g_next = torch.rand(d, generator=gen) + 0.5
    gate = (torch.rand(d, generator=gen) * 2.0 - 0.5) if gated else None
    x = dev["x"]
    x_before = x.clone()
    ids = w = None
    if replay:                  # routes passed in: the router's own, replayed
        ids, w = layer.route(x)
    y_ref = layer.forward(x, ids=ids, w=w)
    torch.cuda.synchronize()
    y, x_out, h_next = layer.forward_boundary(
        x, g_post.cuda(), g_next.cuda(), gate=None if gate is None else gate.cuda(),
        ids=ids, w=w, x_out=x if inplace else None)
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    assert torch.equal(y, y_ref)
    if inplace:
        assert x_out.data_ptr() == x.data_ptr()

    cnt = layer.intermediate("bnd_cnt", T).cpu().numpy()
    nblk = 8 * ((T + 255) // 256)
    if expect_fused:
        assert np.all(cnt[:nblk] == d // 256), cnt[:nblk]
        assert cnt[nblk] >= (T + 1) // 2          # every 2-row item claimed
    else:
        assert not np.any(cnt), cnt

    kind = "f32" if act == "f32" else "bf16"
    xr, _ = oracle.boundary(to_np(x_before), to_np(y), g_post.numpy(), g_next.numpy(),
                            shape.eps, gate=None if gate is None else gate.numpy(), act=kind)
    xg = to_np(x_out)
    fx = assert_one_unit("x_out", xg, xr, kind)
    hr = oracle.store(oracle.rmsnorm(xg, g_next.numpy(), shape.eps), kind)
    fh = assert_one_unit("h_next", to_np(h_next), hr, kind)
    return fx, fh


@pytest.mark.parametrize("T,out,gated,inplace", [
    (600, "bf16", False, False),      # 3 pair-tile bands, the last ragged (88 rows)
    (600, "f32", True, True),         # gated residual, x updated in place
    (1024, "bf16", True, False),
    (257, "f32", False, False),       # one row in the last band
])
def test_fused_boundary_bf16_stream(T, out, gated, inplace):
    need_gpu()
    fx, fh = run_fused(T, "bf16", out, gated, inplace, seed=T, expect_fused=True)
    print("fused boundary bf16", T, out, f"x' flips {fx:.1e}  h' flips {fh:.1e}")


def test_fused_boundary_f32_stream():
    """FP32 activations: the unpooler on TF32 CTA pairs, FP32 rows in the row pass."""
    need_gpu()
    run_fused(600, "f32", "f32", True, False, seed=11, expect_fused=True)


def test_fused_boundary_nvfp4_experts():
    """NVFP4 experts: the unpooler, and so the row pass, are those of the BF16 stream."""
    need_gpu()
    run_fused(600, "bf16", "bf16", True, False, seed=15, expect_fused=True, expert="nvfp4")


def test_fused_boundary_with_replayed_routes():
    """Routes passed in (routing replay) through the fused call: the same block output as
    moe_forward with those routes, and the row pass on it."""
    need_gpu()
    run_fused(700, "bf16", "f32", False, False, seed=16, expect_fused=True, replay=True)


def test_small_batches_run_the_pass():
    """Decode-sized batches whose unpooler splits K (here p = 1024: four slices) run the
    boundary as its own pass after the block, with the same results; with p = 256 the
    unpooler cannot split and a 64-token batch keeps the fused row pass."""
    need_gpu()
    run_fused(64, "bf16", "bf16", True, False, seed=12, expect_fused=False, p=1024)
    run_fused(1, "bf16", "f32", False, True, seed=13, expect_fused=False, p=1024)
    run_fused(64, "bf16", "bf16", False, False, seed=14, expect_fused=True)


def test_widths_off_the_pair_tiles_run_the_pass():
    """d not a multiple of 256 (d = 1152: 128-column unpooler tiles on single CTAs): the
    boundary runs as its own pass after the block, with the same results."""
    need_gpu()
    run_fused(600, "bf16", "bf16", True, True, seed=17, expect_fused=False, d=1152)


def test_fused_equals_separate_calls():
    """moe_forward + moe_boundary and moe_forward_boundary agree: y bit for bit; x' equal
    or one BF16 unit apart (the two sum the row's squares in different orders) on at most
    1 % of the elements; h' the same, plus the difference of x' it carries (scaled by the
    row's norm factor and gain) where x' differs."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300 import synth
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.Shape("fused_boundary", T=1000, d=8192, p=256, E=8, top_k=2, I=256)
    inp = synth.make_inputs(shape, seed=21, device="cpu")
    dev = {k: v.cuda() for k, v in inp.items()}
    layer = LatentMoE(shape, dev, out="bf16")
    gen = torch.Generator(device="cpu").manual_seed(22)
    g_post = (torch.rand(shape.d, generator=gen) + 0.5).cuda()
    g_next = (torch.rand(shape.d, generator=gen) + 0.5).cuda()
    y1 = layer.forward(dev["x"])
    x1, h1 = layer.boundary(dev["x"], y1, g_post, g_next)
    y2, x2, h2 = layer.forward_boundary(dev["x"], g_post, g_next)
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    assert torch.equal(y1, y2)
    xa, xb = to_np(x2), to_np(x1)
    # where x and gate * a cancel, the few 2^-24 of rounding the two paths' FP32 sums
    # carry can exceed a BF16 unit of the small result: allow 2^-20 of the terms
    yv = to_np(y1)
    rs_y = 1.0 / np.sqrt(np.mean(yv * yv, axis=-1, keepdims=True) + shape.eps)
    terms = np.abs(to_np(dev["x"])) + np.abs(yv * rs_y * to_np(g_post))
    d = np.abs(xa - xb)
    u = unit(np.maximum(np.abs(xa), np.abs(xb)), "bf16")
    assert np.all(d <= (u + terms * 2.0 ** -20) * (1 + 1e-9)), int(np.sum(d > u))
    assert float(np.mean(d > 0)) <= 0.01
    ha, hb = to_np(h2), to_np(h1)
    rs = 1.0 / np.sqrt(np.mean(xb * xb, axis=-1, keepdims=True) + shape.eps)
    carried = np.abs(xa - xb) * rs * to_np(g_next)
    u = unit(np.maximum(np.abs(ha), np.abs(hb)), "bf16")
    bad = np.abs(ha - hb) > (u + carried) * (1 + 1e-6)
    assert not np.any(bad), ("h_next", int(bad.sum()))
    assert float(np.mean(ha != hb)) <= 0.01


def test_repeated_calls_are_deterministic():
    """The counters are cleared by every call: back-to-back calls give identical bits."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300 import synth
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.Shape("fused_boundary", T=700, d=8192, p=256, E=8, top_k=2, I=256)
    inp = synth.make_inputs(shape, seed=31, device="cpu")
    dev = {k: v.cuda() for k, v in inp.items()}
    layer = LatentMoE(shape, dev, out="bf16")
    g = (torch.rand(shape.d, generator=torch.Generator().manual_seed(32)) + 0.5).cuda()
    first = [t.clone() for t in layer.forward_boundary(dev["x"], g, g)]
    for _ in range(3):
        again = layer.forward_boundary(dev["x"], g, g)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)


def test_bounded_waits_in_the_fused_kernel():
    """With the test hook MOE_FLAG_TEST_TIMEOUT the fused unpooler's tiles never complete
    (each pair's first operand load is withheld, as in the gate/up GEMM): every wait in
    the kernel, the row workers' included, runs out after 20 ms, the call reports
    MOE_ERR_TIMEOUT, and the next normal call on the same context gives the same bits as
    before."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300 import _lib as L
    from latent_moe_layer_rmsnorm_gb300 import synth
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.Shape("fused_boundary", T=600, d=8192, p=256, E=8, top_k=2, I=256)
    inp = synth.make_inputs(shape, seed=41, device="cpu")
    dev = {k: v.cuda() for k, v in inp.items()}
    layer = LatentMoE(shape, dev, out="bf16")
    g = (torch.rand(shape.d, generator=torch.Generator().manual_seed(42)) + 0.5).cuda()
    good = [t.clone() for t in layer.forward_boundary(dev["x"], g, g)]
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    layer.forward_boundary(dev["x"], g, g, flags=L.MOE_FLAG_TEST_TIMEOUT)
    status, detail = layer.read_status()
    assert status == L.MOE_ERR_TIMEOUT
    assert detail in (1, 2, 4, 7), detail
    again = layer.forward_boundary(dev["x"], g, g)
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    for a, b in zip(good, again):
        assert torch.equal(a, b)


def test_fused_call_captures_into_a_cuda_graph():
    """moe_forward_boundary (its counter reset included) captures into a CUDA graph:
    replays give the eager call's bits, again and again (the counters start from zero on
    every replay), and follow a new input written into the captured buffer."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300 import synth
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.Shape("fused_boundary", T=600, d=8192, p=256, E=8, top_k=2, I=256)
    inp = synth.make_inputs(shape, seed=51, device="cpu")
    dev = {k: v.cuda() for k, v in inp.items()}
    layer = LatentMoE(shape, dev, out="bf16")
    g = (torch.rand(shape.d, generator=torch.Generator().manual_seed(52)) + 0.5).cuda()
    x = dev["x"].clone()
    eager = [t.clone() for t in layer.forward_boundary(x, g, g)]
    flipped = x.flip(0).contiguous()
    other = [t.clone() for t in layer.forward_boundary(flipped, g, g)]
    y, xo, hn = (torch.empty_like(t) for t in eager)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm the call on the capture stream first
        layer.forward_boundary(x, g, g, y=y, x_out=xo, h_next=hn)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward_boundary(x, g, g, y=y, x_out=xo, h_next=hn)
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip((y, xo, hn), eager):
            assert torch.equal(a, b)
    x.copy_(flipped)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip((y, xo, hn), other):
        assert torch.equal(a, b)
    assert layer.read_status() == (0, 0)
