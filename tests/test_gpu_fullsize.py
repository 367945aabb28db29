"""GPU parity at the full workload sizes, in the launch configuration the benchmark
times (one moe_forward over the whole batch).

* prefill chunk (T=16384, d=8192, p=4096, E=256, k=8, I=4096, BF16): expert ids of
  ALL tokens exactly (router margins >= 1e-3 after redraws), route weights, and the
  full output of 256 sampled tokens (the oracle computes them one by one, rows being
  independent): spread over the batch, plus tokens routed to the busiest and to the
  rarest expert.
* decode batch (T=64, same widths): every token in full.
* skewed routing (T=8192): ids of all tokens; 256 sampled tokens including the busiest
  expert's first and last rows and the least-loaded non-empty expert's.

Bound: max|gpu - ref| / rms(ref) <= 1e-2 (BF16 storage; the rounding-chain oracle).
The oracle's per-expert steps run in worker processes (tests/oracle_pool.py).
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pool
from harness import fullsize_inputs, oracle_view, rel_err, to_np
from latent_moe_layer_rmsnorm_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 1e-2
TOL_W = 5e-4
EXPERT_SEED = 0          # one expert set for every full-size test (drawn once per session)
SAMPLE = 256


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    build.build()


def run_full(shape, seed):
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    host, dev = fullsize_inputs(shape, seed, EXPERT_SEED)
    layer = LatentMoE(shape, dev, out="f32", keep_canonical=False)
    out = layer.forward(dev["x"])
    ids, w = layer.route(dev["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    return host, layer, out, ids.cpu().numpy(), to_np(w)


def all_routes(host, shape):
    h = oracle.rmsnorm(to_np(host["x"]), to_np(host["g_in"]), shape.eps)
    return oracle.topk_route(oracle.router_logits(h, to_np(host["w_router"])), shape.top_k)


def sample_tokens(ids: np.ndarray, n: int, E: int) -> list:
    """n tokens: the first and last 4 rows of the busiest expert, up to 8 rows of the
    least-loaded non-empty expert, the rest spread evenly over the batch."""
    T = ids.shape[0]
    counts = np.bincount(ids.reshape(-1), minlength=E)
    busiest = int(np.argmax(counts))
    nonempty = np.nonzero(counts)[0]
    rarest = int(nonempty[np.argmin(counts[nonempty])])
    tb = np.nonzero((ids == busiest).any(1))[0]
    tr = np.nonzero((ids == rarest).any(1))[0]
    out = set(tb[:4].tolist() + tb[-4:].tolist() + tr[:8].tolist())
    for t in np.linspace(0, T - 1, n).round().astype(int).tolist():
        if len(out) >= n:
            break
        out.add(t)
    t = 0
    while len(out) < n:          # fill up (a spread point may repeat an extreme's row)
        out.add(t)
        t += 1
    return sorted(out)


def compare(layer, host, shape, out, ids, tok, label):
    view = oracle_view(host)
    emap = oracle_pool.ExpertMap(shape, EXPERT_SEED)
    ref = oracle.moe_forward(view, top_k=shape.top_k, eps=shape.eps, act=shape.act,
                             expert=shape.expert, out="f32", chain=True, tokens=tok,
                             return_parts=True, expert_map=emap)
    np.testing.assert_array_equal(ref["ids"], ids[tok])
    sel = torch.as_tensor(tok, device=out.device)
    err = rel_err(to_np(out[sel]), ref["out"])
    c_err = rel_err(to_np(layer.intermediate("c", shape.T)[sel]), ref["c"])
    per_tok = np.max(np.abs(to_np(out[sel]) - ref["out"]), axis=1) / np.sqrt(np.mean(ref["out"] ** 2))
    print(f"{label}: {len(tok)} sampled tokens, out err {err:.2e} (median token "
          f"{np.median(per_tok):.2e}), c err {c_err:.2e}")
    assert err <= TOL


def test_prefill_chunk():
    need_gpu()
    shape = synth.PREFILL_BF16
    host, layer, out, ids, w = run_full(shape, seed=0)
    rid, rw = all_routes(host, shape)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(w, rw, rtol=0, atol=TOL_W)
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    print("expert load: mean", counts.mean(), "max", counts.max(), "min", counts.min())
    tok = sample_tokens(ids, SAMPLE, shape.E)
    assert len(tok) >= SAMPLE
    compare(layer, host, shape, out, ids, tok, "prefill")


def test_decode_batch():
    need_gpu()
    shape = synth.DECODE_BF16
    host, layer, out, ids, w = run_full(shape, seed=1)
    rid, rw = all_routes(host, shape)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(w, rw, rtol=0, atol=TOL_W)
    print(f"decode: {len(np.unique(ids))} experts touched")
    compare(layer, host, shape, out, ids, list(range(shape.T)), "decode")


def test_skewed_routing():
    """Zipf-skewed routing (T=8192): the busiest expert spans tens of 128-row tiles,
    many experts are empty."""
    need_gpu()
    shape = synth.SKEWED_BF16
    host, layer, out, ids, w = run_full(shape, seed=2)
    rid, rw = all_routes(host, shape)
    np.testing.assert_array_equal(ids, rid)
    np.testing.assert_allclose(w, rw, rtol=0, atol=TOL_W)
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    ratio = counts.max() / counts.mean()
    empty = float(np.mean(counts == 0))
    print(f"skewed load: max/mean {ratio:.1f}, empty experts {empty:.2f}")
    assert ratio >= 10 and empty >= 0.05
    tok = sample_tokens(ids, SAMPLE, shape.E)
    compare(layer, host, shape, out, ids, tok, "skewed")


def zipf_routes(T: int, E: int, k: int, s: float, seed: int):
    """External routes for T tokens: k distinct experts per token drawn without
    replacement from a Zipf(s) popularity over a seeded permutation of the expert ids
    (Gumbel top-k on the log probabilities), with positive weights that sum to 1.  The
    ordering within a token is by weight, largest first."""
    rng = np.random.default_rng(seed)
    rank = rng.permutation(E) + 1
    logp = -s * np.log(rank.astype(np.float64))
    g = logp[None, :] + rng.gumbel(size=(T, E))
    ids = np.argsort(-g, axis=1)[:, :k].astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T)
    w = -np.sort(-w, axis=1)
    return ids, w.astype(np.float32)


def test_routing_replay_and_external_routes_at_scale():
    """The prefill chunk with routing passed in ("vLLM 对 Muse Spark Open 的 Day 0 支持",
    section "vLLM 中的强化学习": rollout routing replay): the router's own ids and
    weights replayed give bit-identical output; Zipf-skewed external routes (no token's
    experts from the router) match the oracle on 64 sampled tokens, including the
    most- and least-loaded experts' tokens, and are deterministic."""
    need_gpu()
    shape = synth.PREFILL_BF16
    host, layer, out, ids, w = run_full(shape, seed=0)
    dev_x = host["x"].cuda()
    ids_t = torch.as_tensor(ids, device="cuda")
    w_t = torch.as_tensor(w, device="cuda")
    rep = layer.forward(dev_x, ids=ids_t, w=w_t)
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    assert torch.equal(rep, out)
    ext_ids, ext_w = zipf_routes(shape.T, shape.E, shape.top_k, 1.2, seed=99)
    ei, ew = torch.as_tensor(ext_ids, device="cuda"), torch.as_tensor(ext_w, device="cuda")
    a = layer.forward(dev_x, ids=ei, w=ew).clone()
    b = layer.forward(dev_x, ids=ei, w=ew)
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    assert torch.equal(a, b)
    counts = np.bincount(ext_ids.reshape(-1), minlength=shape.E)
    print(f"external routes: busiest expert {counts.max()} rows ({counts.max() / counts.mean():.1f}x "
          f"mean), {int(np.sum(counts == 0))} experts empty")
    tok = sample_tokens(ext_ids, 64, shape.E)
    view = oracle_view(host)
    ref = oracle.moe_forward(view, top_k=shape.top_k, eps=shape.eps, act="bf16", expert="bf16",
                             out="f32", chain=True, tokens=tok, ids=ext_ids[tok],
                             weights=ext_w[tok], expert_map=oracle_pool.ExpertMap(shape, EXPERT_SEED))
    err = rel_err(to_np(a[torch.as_tensor(tok, device="cuda")]), ref)
    print(f"external routes: {len(tok)} sampled tokens, out err {err:.2e}")
    assert err <= TOL


def test_boundary_in_the_unpooler_at_scale():
    """The prefill chunk through moe_forward_boundary, in the bench's configuration (BF16
    stream and output): the row workers of all 76 CTA pairs claim 8192 two-row items
    while the unpooler's tiles complete.  The block output equals moe_forward's bit for
    bit; x' and h' equal moe_forward + moe_boundary's within one BF16 unit on at most 1 %
    of the elements (h' also carrying any x' difference, scaled by the row's norm factor
    and gain); 256 sampled rows against the oracle's boundary of the GPU's own y; every
    32-row block counted its 32 column tiles; repeated calls give the same bits."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.PREFILL_BF16
    host, dev = fullsize_inputs(shape, 0, EXPERT_SEED)
    layer = LatentMoE(shape, dev, out="bf16", keep_canonical=False)
    T, d = shape.T, shape.d
    gen = torch.Generator(device="cpu").manual_seed(5)
    g_post = torch.rand(d, generator=gen) + 0.5
    g_next = torch.rand(d, generator=gen) + 0.5
    gate = torch.rand(d, generator=gen) * 2.0 - 0.5
    gp, gn, gt = g_post.cuda(), g_next.cuda(), gate.cuda()
    x = dev["x"]
    y1 = layer.forward(x)
    x1, h1 = layer.boundary(x, y1, gp, gn, gate=gt)
    y2, x2, h2 = layer.forward_boundary(x, gp, gn, gate=gt)
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    cnt = layer.intermediate("bnd_cnt", T).cpu().numpy()
    assert np.all(cnt[:8 * ((T + 255) // 256)] == d // 256)
    assert torch.equal(y1, y2)

    def unit(v):
        return torch.exp2(torch.floor(torch.log2(v.abs().clamp_min(1e-30))) - 7)

    # x' = bf16(x + gate * y * rs * g_post): the two paths' FP32 values differ by a few
    # units of 2^-24 of the terms added (rs from sums in another order), which where the
    # terms cancel is more than a BF16 unit of the small result
    a, b = x2.float(), x1.float()
    yv = y2.float()
    rs_y = torch.rsqrt((yv * yv).mean(dim=1, keepdim=True) + shape.eps)
    terms = x.float().abs() + (gt * (yv * rs_y * gp)).abs()
    u_x = unit(torch.maximum(a.abs(), b.abs()))
    dx = (a - b).abs()
    over = dx > u_x * (1 + 1e-6)
    print(f"x' beyond one unit: {int(over.sum())} elements, worst {float((dx / terms)[over].max()) if bool(over.any()) else 0.0:.2e} of the terms")
    assert bool((dx <= (u_x + terms * 2.0 ** -20) * (1 + 1e-6)).all())
    fx = float((dx > 0).float().mean())
    rs = torch.rsqrt((b * b).mean(dim=1, keepdim=True) + shape.eps)
    ha, hb = h2.float(), h1.float()
    tol = unit(torch.maximum(ha.abs(), hb.abs())) + dx * rs * gn
    assert bool(((ha - hb).abs() <= tol * (1 + 1e-6)).all())
    fh = float((ha != hb).float().mean())
    print(f"fused boundary at scale: x' differs from the pass on {fx:.1e}, h' on {fh:.1e}")
    assert fx <= 0.01 and fh <= 0.01

    rows = np.linspace(0, T - 1, 256).round().astype(int)
    sel = torch.as_tensor(rows, device="cuda")
    xr, _ = oracle.boundary(to_np(host["x"])[rows], to_np(y2[sel]), g_post.numpy(),
                            g_next.numpy(), shape.eps, gate=gate.numpy(), act="bf16")
    xg = to_np(x2[sel])
    assert np.all(np.abs(xg - xr) <= (np.exp2(np.floor(np.log2(np.maximum(
        np.maximum(np.abs(xg), np.abs(xr)), 1e-30))) - 7) + to_np(terms[sel]) * 2.0 ** -20)
        * (1 + 1e-9))
    hr = oracle.store(oracle.rmsnorm(xg, g_next.numpy(), shape.eps), "bf16")
    hg = to_np(h2[sel])
    assert np.all(np.abs(hg - hr) <= np.exp2(np.floor(np.log2(np.maximum(
        np.maximum(np.abs(hg), np.abs(hr)), 1e-30))) - 7) * (1 + 1e-9))

    again = layer.forward_boundary(x, gp, gn, gate=gt)
    torch.cuda.synchronize()
    for u, v in zip((y2, x2, h2), again):
        assert torch.equal(u, v)
