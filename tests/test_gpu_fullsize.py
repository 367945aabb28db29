"""GPU parity at the full workload sizes, in the launch configuration the benchmark
times (one moe_forward over the whole batch).

* prefill chunk (T=16384, d=8192, p=4096, E=256, k=8, I=4096, BF16): expert ids of
  ALL tokens exactly (router margins >= 1e-3 after redraws), route weights, and the
  full output of sampled tokens (the oracle computes them one by one; rows are
  independent), including tokens routed to the busiest and the rarest expert.
* decode batch (T=64, same widths): every token in full.

Bound: max|gpu - ref| / rms(ref) <= 1e-2 (BF16 storage; the rounding-chain oracle).
"""
import numpy as np
import pytest
import torch

import oracle
from harness import fix_margins, oracle_view, rel_err, to_np
from latent_moe_layer_rmsnorm_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 1e-2
TOL_W = 5e-4


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    build.build()


def run_full(shape, seed):
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    inp = synth.make_inputs(shape, seed=seed, device="cuda")
    fix_margins(inp, shape, seed=seed)
    layer = LatentMoE(shape, inp, out="f32")
    out = layer.forward(inp["x"])
    ids, w = layer.route(inp["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    return inp, layer, out, ids.cpu().numpy(), to_np(w)


def oracle_rows(inp, shape, tokens):
    view = oracle_view(inp, lazy=True)
    return oracle.moe_forward(view, top_k=shape.top_k, eps=shape.eps, act=shape.act,
                              expert=shape.expert, out="f32", chain=True, tokens=tokens,
                              return_parts=True)


def test_prefill_chunk():
    need_gpu()
    shape = synth.PREFILL_BF16
    inp, layer, out, ids, w = run_full(shape, seed=0)
    # routing of every token
    x = to_np(inp["x"])
    h = oracle.rmsnorm(x, to_np(inp["g_in"]), shape.eps)
    logits = oracle.router_logits(h, to_np(inp["w_router"]))
    del x, h
    rid, rw = oracle.topk_route(logits, shape.top_k)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(w, rw, rtol=0, atol=TOL_W)
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    busiest, rarest = int(np.argmax(counts)), int(np.argmin(counts))
    print("expert load: mean", counts.mean(), "max", counts.max(), "min", counts.min())
    # sampled tokens, spread over the batch and the M tiles, plus the extremes
    tok = [0, 1, 127, 128, 5000, 9999, 16383]
    tok.append(int(np.nonzero((ids == busiest).any(1))[0][0]))
    tok.append(int(np.nonzero((ids == rarest).any(1))[0][-1]))
    tok = sorted(set(tok))
    ref = oracle_rows(inp, shape, tok)
    np.testing.assert_array_equal(ref["ids"], ids[tok])
    got = to_np(out[torch.as_tensor(tok, device=out.device)])
    err = rel_err(got, ref["out"])
    c_gpu = to_np(layer.intermediate("c", shape.T)[torch.as_tensor(tok, device=out.device)])
    c_err = rel_err(c_gpu, ref["c"])
    print(f"prefill sampled tokens {tok}: out err {err:.2e}, c err {c_err:.2e}")
    assert err <= TOL


def test_decode_batch():
    need_gpu()
    shape = synth.DECODE_BF16
    inp, layer, out, ids, w = run_full(shape, seed=1)
    tok = list(range(shape.T))
    ref = oracle_rows(inp, shape, tok)
    np.testing.assert_array_equal(ids, ref["ids"])
    np.testing.assert_allclose(w, ref["w"], rtol=0, atol=TOL_W)
    err = rel_err(to_np(out), ref["out"])
    touched = len(np.unique(ids))
    print(f"decode: {touched} experts touched, out err {err:.2e}")
    assert err <= TOL


def test_skewed_routing():
    """Zipf-skewed routing (T=8192): the busiest expert spans tens of 128-row tiles,
    many experts are empty.  Ids of all tokens exactly; sampled tokens in full,
    including tokens of the busiest and of the least-loaded non-empty expert."""
    need_gpu()
    shape = synth.SKEWED_BF16
    inp, layer, out, ids, w = run_full(shape, seed=2)
    x = to_np(inp["x"])
    h = oracle.rmsnorm(x, to_np(inp["g_in"]), shape.eps)
    logits = oracle.router_logits(h, to_np(inp["w_router"]))
    del x, h
    rid, rw = oracle.topk_route(logits, shape.top_k)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(w, rw, rtol=0, atol=TOL_W)
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    ratio = counts.max() / counts.mean()
    empty = float(np.mean(counts == 0))
    print(f"skewed load: max/mean {ratio:.1f}, empty experts {empty:.2f}")
    assert ratio >= 10 and empty >= 0.05
    busiest = int(np.argmax(counts))
    nonempty = np.nonzero(counts)[0]
    rarest = int(nonempty[np.argmin(counts[nonempty])])
    tok = [0, 4095, 8191]
    tok += [int(t) for t in np.nonzero((ids == busiest).any(1))[0][[0, -1]]]
    tok.append(int(np.nonzero((ids == rarest).any(1))[0][0]))
    tok = sorted(set(tok))
    ref = oracle_rows(inp, shape, tok)
    got = to_np(out[torch.as_tensor(tok, device=out.device)])
    err = rel_err(got, ref["out"])
    print(f"skewed sampled tokens {tok}: out err {err:.2e}")
    assert err <= TOL
