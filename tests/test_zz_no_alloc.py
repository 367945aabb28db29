"""moe_route_noalloc: routing for callers that cannot allocate device memory (an engine
whose memory is all reserved at start-up, a plugin host that forbids allocations, a
replayed graph that must not grow its pool).  Its scratch lives in a fixed array inside
the library, so it takes no workspace.

Checked through the C ABI against moe_route, the entry point with a caller-provided
workspace: identical expert ids and route weights within the tolerance the other GPU
tests use, on two calls in a row (the second call meets the first call's leftovers in
the shared array).  This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from latent_moe_layer_rmsnorm_gb300 import _lib as L
from latent_moe_layer_rmsnorm_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_W = 5e-4        # same bound as the other GPU tests' route-weight checks


# (T, d, E, top_k): a small case; one token and a decode batch at the full width (the
# router's reduction split over K slices, partial logits in the array); the documented
# limit T * d = 2^21 at d = 8192 with 256 experts (fewer K slices than moe_route takes,
# so the sums differ in order); and a long batch of narrow rows, where the router runs
# unsplit on one CTA per 128 tokens with all 256 experts in one tile.
CASES = [(200, 1024, 32, 6), (1, 8192, 256, 8), (64, 8192, 256, 8), (256, 8192, 256, 8),
         (8192, 256, 256, 8)]


@pytest.mark.parametrize("T,d,E,k", CASES, ids=lambda v: str(v))
def test_noalloc_route_matches_workspace_route(T, d, E, k):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from harness import fix_margins
    from latent_moe_layer_rmsnorm_gb300 import build
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    build.build()
    # narrow experts: only the router's shapes matter here
    shape = synth.Shape("noalloc_bf16", T=T, d=d, p=256, E=E, top_k=k, I=256)
    host = synth.make_inputs(shape, seed=21, device="cpu")
    fix_margins(host, shape, seed=21)        # unique top-k sets across summation orders
    inp = {key: v.cuda() for key, v in host.items()}
    layer = LatentMoE(shape, inp, out="f32")
    x = inp["x"]
    ids_ref, w_ref = layer.route(x)
    cfg = layer.config(shape.T)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        ids = torch.full((shape.T, shape.top_k), -1, dtype=torch.int32, device="cuda")
        w = torch.full((shape.T, shape.top_k), -1.0, dtype=torch.float32, device="cuda")
        st = L.moe_route_noalloc(cfg, layer.W, x.data_ptr(), ids.data_ptr(), w.data_ptr(),
                                 stream)
        assert st == L.MOE_OK, (call, L.status_string(st))
        assert L.moe_read_noalloc_status(stream) == (L.MOE_OK, 0), call
        assert torch.equal(ids.cpu(), ids_ref.cpu()), call
        np.testing.assert_allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=0, atol=TOL_W)


def test_noalloc_route_rejects_calls_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cfg = L.moe_config_t(T=257, d=8192, p=4096, E=256, top_k=8, I=4096, eps=1e-6,
                         act=L.MOE_BF16, expert=L.MOE_BF16, out=L.MOE_BF16, flags=0)
    fake = 1 << 20
    W = L.moe_weights_t(g_in=fake, w_router=fake, w_pool=fake, g_pool=fake, w13=fake,
                        w2=fake, g_exp=fake, w_unpool=fake)
    assert L.moe_route_noalloc(cfg, W, fake, fake, fake, None) == L.MOE_ERR_WORKSPACE
