"""GPU parity of the CUDA path against the CPU oracle on small and ragged shapes.

Every case compares the C-ABI call (through the thin binding) with the oracle's
precision-chain result, element by element: expert ids exactly (inputs are
redrawn until every top-(k+1) router gap is >= 1e-3), route weights, every stored
intermediate and the output.  Output gate: max|gpu - ref| / rms(ref) <= 1e-2 for
BF16 storage (the benchmark spec's bound), and a tighter bound where the arithmetic
allows it (each is derived next to its constant).
"""
import numpy as np
import pytest
import torch

import oracle
from harness import fix_margins, oracle_kwargs, oracle_view, rel_err, to_np
from latent_moe_layer_rmsnorm_gb300 import synth

pytestmark = pytest.mark.gpu

# BF16 storage: outputs agree with the rounding-chain oracle to a few BF16 units of
# the intermediates; 1e-2 is the benchmark spec's bound.  Measured values are printed.
TOL_BF16 = 1e-2
# FP32 storage with TF32 GEMM operands (both sides round at the same points): the
# residual is FP32-vs-FP64 accumulation plus rare TF32 rounding flips, ~1e-4.
TOL_F32 = 2e-3

TINY_BF16 = synth.TINY_F32.replace(name="tiny_bf16", act="bf16", expert="bf16")
MID_BF16 = synth.Shape("mid_bf16", T=300, d=512, p=256, E=16, top_k=4, I=384)
SHAPES = {"tiny_f32": synth.TINY_F32, "tiny_bf16": TINY_BF16, "mid_bf16": MID_BF16}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    build.build()


def make_case(shape, seed=0):
    inp = synth.make_inputs(shape, seed=seed, device="cpu")
    fix_margins(inp, shape, seed=seed)
    return inp


def gpu_layer(shape, inp, out="f32"):
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    dev = {k: v.cuda() for k, v in inp.items()}
    return LatentMoE(shape, dev, out=out), dev


def tol_for(shape):
    return TOL_F32 if shape.act == "f32" else TOL_BF16


def check_dispatch(layer, T, ids):
    """Counting-sort invariants: offsets are the exclusive scan of the expert counts,
    src is a permutation, each expert's rows are in (token, slot) order, inv inverts src."""
    k = layer.shape.top_k
    E = layer.shape.E
    row_off = to_np(layer.intermediate("row_off", T)).astype(np.int64)
    src = layer.intermediate("src", T).cpu().numpy().astype(np.int64)
    inv = layer.intermediate("inv", T).cpu().numpy().astype(np.int64)
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    np.testing.assert_array_equal(row_off, np.concatenate([[0], np.cumsum(counts)]))
    assert sorted(src.tolist()) == list(range(T * k))
    np.testing.assert_array_equal(inv[src], np.arange(T * k))
    for e in range(E):
        seg = src[row_off[e]: row_off[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(flat[seg] == e)
    return src


@pytest.mark.parametrize("name", list(SHAPES))
def test_layer_matches_oracle(name):
    need_gpu()
    shape = SHAPES[name]
    inp = make_case(shape)
    ref = oracle.moe_forward(oracle_view(inp), **oracle_kwargs(shape, "f32"), chain=True,
                             return_parts=True)
    layer, dev = gpu_layer(shape, inp, out="f32")
    T, k = shape.T, shape.top_k
    out = layer.forward(dev["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)

    ids = layer.intermediate("ids", T).cpu().numpy()
    np.testing.assert_array_equal(ids, ref["ids"])
    np.testing.assert_allclose(to_np(layer.intermediate("w", T)), ref["w"], rtol=0, atol=2e-6)
    src = check_dispatch(layer, T, ids)
    tok, slot = src // k, src % k

    errs = {}
    errs["pooled"] = rel_err(to_np(layer.intermediate("pooled", T)), ref["pooled"])
    errs["u"] = rel_err(to_np(layer.intermediate("a_perm", T)), ref["u"][tok])
    errs["s"] = rel_err(to_np(layer.intermediate("s", T)), ref["s"][tok, slot])
    errs["y"] = rel_err(to_np(layer.intermediate("y", T)), ref["y"][tok, slot])
    errs["c"] = rel_err(to_np(layer.intermediate("c", T)), ref["c"])
    errs["out"] = rel_err(to_np(out), ref["out"])
    print(name, {k_: f"{v:.2e}" for k_, v in errs.items()})
    for stage, e in errs.items():
        assert e <= tol_for(shape), (stage, e, errs)


@pytest.mark.parametrize("name", ["tiny_bf16", "mid_bf16", "tiny_f32"])
@pytest.mark.parametrize("T", [1, 63, 65, 129])
def test_ragged_token_counts(name, T):
    need_gpu()
    shape = SHAPES[name].replace(T=T)
    inp = make_case(shape, seed=T)
    ref = oracle.moe_forward(oracle_view(inp), **oracle_kwargs(shape, "f32"), chain=True,
                             return_parts=True)
    layer, dev = gpu_layer(shape, inp, out="f32")
    out = layer.forward(dev["x"])
    ids, w = layer.route(dev["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref["ids"])
    np.testing.assert_allclose(to_np(w), ref["w"], rtol=0, atol=2e-6)
    assert out.shape == (T, shape.d)      # the pooler keeps the token count
    assert rel_err(to_np(out), ref["out"]) <= tol_for(shape)


def test_bf16_output_mode():
    """BF16 output: each element within tolerance*rms + one BF16 unit of the reference
    (an FP32-vs-FP64 difference can move a final rounding by one unit)."""
    need_gpu()
    shape = MID_BF16
    inp = make_case(shape, seed=5)
    ref = oracle.moe_forward(oracle_view(inp), **oracle_kwargs(shape, "bf16"), chain=True)
    layer, dev = gpu_layer(shape, inp, out="bf16")
    out = to_np(layer.forward(dev["x"]))
    rms = np.sqrt(np.mean(ref ** 2))
    ulp = np.abs(ref) * 2.0 ** -7
    assert np.all(np.abs(out - ref) <= TOL_BF16 * rms + ulp)


def test_routing_replay_and_determinism():
    """Passing the router's own ids/weights back reproduces the output bit for bit, and
    two identical calls give identical bits."""
    need_gpu()
    shape = MID_BF16
    inp = make_case(shape, seed=11)
    layer, dev = gpu_layer(shape, inp)
    a = layer.forward(dev["x"]).clone()
    b = layer.forward(dev["x"]).clone()
    ids, w = layer.route(dev["x"])
    c = layer.forward(dev["x"], ids=ids, w=w).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(a, c)


def test_external_routes_match_oracle():
    """Routing replay with routes that are not the router's own (random ids/weights)."""
    need_gpu()
    shape = MID_BF16
    inp = make_case(shape, seed=12)
    g = torch.Generator().manual_seed(3)
    ids = torch.stack([torch.randperm(shape.E, generator=g)[: shape.top_k]
                       for _ in range(shape.T)]).to(torch.int32)
    w = torch.rand((shape.T, shape.top_k), generator=g)
    ref = oracle.moe_forward(oracle_view(inp), **oracle_kwargs(shape, "f32"), chain=True,
                             ids=ids.numpy(), weights=w.numpy().astype(np.float64))
    layer, dev = gpu_layer(shape, inp)
    out = layer.forward(dev["x"], ids=ids.cuda(), w=w.cuda())
    assert rel_err(to_np(out), ref) <= TOL_BF16


def test_relabelling_is_bit_exact():
    """Permuting experts (router rows, expert weights, gains) permutes the chosen ids and
    leaves the output bit-identical: each row's arithmetic does not depend on where the
    dispatch places it."""
    need_gpu()
    shape = MID_BF16
    inp = make_case(shape, seed=13)
    perm = torch.randperm(shape.E, generator=torch.Generator().manual_seed(1))
    relab = dict(inp)
    for key in ("w_router", "w_gate", "w_up", "w_down", "g_exp"):
        relab[key] = inp[key][perm].contiguous()
    la, da = gpu_layer(shape, inp)
    lb, db = gpu_layer(shape, relab)
    oa, ob = la.forward(da["x"]), lb.forward(db["x"])
    ia, _ = la.route(da["x"])
    ib, _ = lb.route(db["x"])
    torch.cuda.synchronize()
    assert torch.equal(oa, ob)
    inv = torch.argsort(perm).to(torch.int32)
    assert torch.equal(inv[ia.cpu().long()], ib.cpu())


def test_token_permutation_is_bit_exact():
    need_gpu()
    shape = MID_BF16
    inp = make_case(shape, seed=14)
    layer, dev = gpu_layer(shape, inp)
    perm = torch.randperm(shape.T, generator=torch.Generator().manual_seed(2)).cuda()
    a = layer.forward(dev["x"]).clone()
    b = layer.forward(dev["x"][perm].contiguous()).clone()
    torch.cuda.synchronize()
    assert torch.equal(a[perm], b)


def test_single_token_calls_equal_batch_rows():
    need_gpu()
    shape = TINY_BF16
    inp = make_case(shape, seed=15)
    layer, dev = gpu_layer(shape, inp)
    full = layer.forward(dev["x"]).clone()
    for t in (0, 17, 63):
        one = layer.forward(dev["x"][t: t + 1].contiguous()).clone()
        assert torch.equal(one[0], full[t])


def test_zero_rows():
    """x = 0: ids 0..k-1 (ties to the lower id), w = 1/k, output exactly 0."""
    need_gpu()
    shape = MID_BF16
    inp = make_case(shape, seed=16)
    inp["x"][[0, 7, 299]] = 0
    layer, dev = gpu_layer(shape, inp)
    out = layer.forward(dev["x"])
    ids, w = layer.route(dev["x"])
    torch.cuda.synchronize()
    for t in (0, 7, 299):
        assert ids[t].tolist() == list(range(shape.top_k))
        assert torch.all(w[t] == 1.0 / shape.top_k)
        assert torch.all(out[t] == 0)


def test_empty_and_crowded_experts():
    """Routes that leave most experts empty and put > 128 rows (several M tiles, a
    ragged tail) on others."""
    need_gpu()
    shape = MID_BF16
    inp = make_case(shape, seed=17)
    T, k = shape.T, shape.top_k
    ids = torch.zeros((T, k), dtype=torch.int32)
    for t in range(T):
        ids[t] = torch.tensor([3, 9, 10, 15])[:k] if t % 3 else torch.tensor([0, 3, 5, 9])[:k]
    w = torch.full((T, k), 1.0 / k)
    ref = oracle.moe_forward(oracle_view(inp), **oracle_kwargs(shape, "f32"), chain=True,
                             ids=ids.numpy(), weights=w.numpy().astype(np.float64))
    layer, dev = gpu_layer(shape, inp)
    out = layer.forward(dev["x"], ids=ids.cuda(), w=w.cuda())
    assert rel_err(to_np(out), ref) <= TOL_BF16
    check_dispatch(layer, T, ids.numpy())
