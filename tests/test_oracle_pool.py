"""The test-side helpers of the full-size parity tests, on the CPU: the pool's expert
map gives the oracle the same result as running the per-expert steps in process, and
the layout helpers invert the chunked scale layout the GPU tests read."""
import numpy as np

import oracle
import oracle_pool
from harness import oracle_view
from latent_moe_layer_rmsnorm_gb300 import synth
from test_gpu_nvfp4 import unchunk_sf


def test_expert_map_equals_in_process_steps():
    for expert in ("bf16", "nvfp4"):
        shape = synth.Shape("p", T=12, d=256, p=128, E=5, top_k=2, I=256, expert=expert)
        view = oracle_view(synth.make_inputs(shape, seed=3))
        kw = dict(top_k=2, eps=shape.eps, act="bf16", expert=expert, out="f32",
                  return_parts=True)
        a = oracle.moe_forward(view, **kw)
        emap = oracle_pool.ExpertMap(shape, 3, digest=True)
        dense = {k: v for k, v in view.items() if k not in ("w_gate", "w_up", "w_down")}
        b = oracle.moe_forward(dense, **kw, expert_map=emap)
        np.testing.assert_array_equal(a["out"], b["out"])
        np.testing.assert_array_equal(a["y"], b["y"])
        if expert == "nvfp4":
            assert set(emap.digests) == set(np.unique(a["ids"]).tolist())


def test_scale_chunking_round_trip():
    rng = np.random.default_rng(0)
    sf = rng.integers(0, 256, size=(256, 32)).astype(np.uint8)
    flat = oracle_pool.chunk_scales(sf)
    np.testing.assert_array_equal(unchunk_sf(flat, 256, 32 * 16), sf)
