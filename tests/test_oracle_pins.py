"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test states what it pins.  Sources: "SGLang and Miles Add Day-0 Support for
Muse Spark Open", section "MoE with Pooler, Unpooler and Per-Expert
Normalization" (router on the full-width vector; pooled input normalised; every
selected expert output normalised before its routing weight and the sum; the
combined vector unpooled; the pooler keeps the token count; normalising the sum
instead would change the result) and "vLLM 对 Muse Spark Open 的 Day 0 支持" (vLLM Day-0 support for Muse Spark Open), sections
"潜空间 MoE" (shared pooler/unpooler, 8192 <-> 4096) and "Nvidia" (TF32 router GEMM
on the norm's FP32 output).  Closed forms, invariances, brute force and library
routines (scipy) supply the expected values.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import formats as F
from latent_moe_layer_rmsnorm_gb300 import synth
from harness import oracle_view, fix_margins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(T=16, d=32, p=16, E=6, k=2, I=24, seed=0, act="f32", expert="f32"):
    shape = synth.Shape("t", T=T, d=d, p=p, E=E, top_k=k, I=I, act=act, expert=expert)
    inp = synth.make_inputs(shape, seed=seed, device="cpu")
    return shape, inp


def fwd(inp, shape, **kw):
    args = dict(top_k=shape.top_k, eps=shape.eps, act=shape.act, expert=shape.expert,
                out="f32", chain=False)
    args.update(kw)
    return oracle.moe_forward(oracle_view(inp) if not isinstance(inp["x"], np.ndarray)
                              else inp, **args)


def np_inputs(inp):
    return oracle_view(inp)


# ---- the hand-worked example -----------------------------------------------------

def test_hand_worked_example():
    """A 2-wide, 2-expert case worked on paper (tests/golden/hand_worked_k2.json).

    x=[2,-2] -> h=[1,-1]; logits=[1,0] -> w=softmax([1,0]); u=[1,-1]; expert 0
    gives y ∝ [1,1], expert 1 y ∝ [1,-1], both with positive SwiGLU output, so
    their per-expert norms are [1,1] and [1,-1]; c = [1, tanh(1/2)];
    out = W_unpool c.
    """
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_k2.json")))
    inp = {k: np.array(v, dtype=np.float64) for k, v in g.items()
           if k.startswith(("x", "g_", "w_"))}
    dims = g["dims"]
    parts = oracle.moe_forward(inp, top_k=dims["top_k"], eps=dims["eps"], act="f32",
                               expert="f32", chain=False, return_parts=True)
    e = math.e
    t = math.tanh(0.5)
    np.testing.assert_allclose(parts["h"], g["expected"]["h"], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(parts["ids"], g["expected"]["ids"])
    np.testing.assert_allclose(parts["w"], [[e / (1 + e), 1 / (1 + e)]], rtol=1e-15)
    np.testing.assert_allclose(parts["u"], g["expected"]["u"], atol=1e-15)
    np.testing.assert_allclose(parts["c"], [[1.0, t]], rtol=1e-14)
    np.testing.assert_allclose(parts["out"], [[1 + 2 * t, 3 + 4 * t]], rtol=1e-14)
    # normalising the sum instead gives something else (the page rules it out)
    alt = oracle.moe_forward(inp, top_k=2, eps=0.0, act="f32", expert="f32", chain=False,
                             norm_after_sum=True)
    assert np.max(np.abs(alt - parts["out"])) > 0.1


# ---- RMSNorm ---------------------------------------------------------------------

def test_rmsnorm_closed_form():
    """A constant row a gives a / sqrt(a^2 + eps) * g in every position."""
    g = np.linspace(0.5, 1.5, 7)
    for a in (-3.0, 1e-3, 2.5):
        v = np.full((1, 7), a)
        out = oracle.rmsnorm(v, g, 1e-6)
        np.testing.assert_allclose(out[0], a / math.sqrt(a * a + 1e-6) * g, rtol=1e-15)
    # rms of the normalised row (unit gain) is sqrt(ms / (ms + eps))
    rng = np.random.default_rng(1)
    v = rng.normal(size=(5, 64))
    out = oracle.rmsnorm(v, np.ones(64), 1e-6)
    ms = np.mean(v * v, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(out * out, axis=1)),
                               np.sqrt(ms / (ms + 1e-6)), rtol=1e-13)


def test_zero_row():
    """x = 0: h = 0, logits all 0, ids 0..k-1 (ties to the lower id), w = 1/k, out = 0."""
    shape, inp = tiny()
    inp["x"][3] = 0
    parts = fwd(inp, shape, return_parts=True)
    np.testing.assert_array_equal(parts["ids"][3], np.arange(shape.top_k))
    np.testing.assert_allclose(parts["w"][3], 1.0 / shape.top_k, rtol=1e-15)
    assert np.all(parts["out"][3] == 0.0)


# ---- router ----------------------------------------------------------------------

def test_router_logits_basis_weights():
    """Router rows that are scaled basis vectors pick single components of h.

    W_r[e] = c_e * delta(i_e)  =>  logits[t, e] = tf32(h[t, i_e]) * tf32(c_e),
    which pins the operand roles (h row, W_r row) and the index order.
    """
    rng = np.random.default_rng(2)
    h = rng.normal(size=(4, 10))
    picks = [7, 0, 3]
    c = [0.5, 2.0, -1.0]
    w = np.zeros((3, 10))
    for e, (i, ce) in enumerate(zip(picks, c)):
        w[e, i] = ce
    logits = oracle.router_logits(h, w)
    for e, (i, ce) in enumerate(zip(picks, c)):
        np.testing.assert_array_equal(logits[:, e], F.tf32_rna(F.fp32(h[:, i])) * ce)


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 2), (8, 3), (3, 3)])
def test_topk_brute_force(E, k):
    """The chosen set maximises the summed logits over all C(E,k) subsets; slots are
    in descending logit order; weights equal scipy's softmax of the chosen logits."""
    rng = np.random.default_rng(E * 10 + k)
    logits = rng.normal(size=(40, E))
    ids, w = oracle.topk_route(logits, k)
    for t in range(logits.shape[0]):
        best = max(itertools.combinations(range(E), k), key=lambda s: logits[t, list(s)].sum())
        assert set(ids[t]) == set(best)
        assert np.all(np.diff(logits[t, ids[t]]) <= 0)
        np.testing.assert_allclose(w[t], scipy.special.softmax(logits[t, ids[t]]), rtol=1e-13)
        # softmax over all E, then renormalised over the chosen k: same numbers
        full = scipy.special.softmax(logits[t])
        np.testing.assert_allclose(w[t], full[ids[t]] / full[ids[t]].sum(), rtol=1e-13)


def test_topk_ties_go_to_lower_id():
    logits = np.array([[1.0, 3.0, 3.0, 0.0, 3.0]])
    ids, w = oracle.topk_route(logits, 3)
    np.testing.assert_array_equal(ids[0], [1, 2, 4])
    np.testing.assert_allclose(w[0], [1 / 3] * 3, rtol=1e-15)


def test_route_margin():
    logits = np.array([[5.0, 1.0, 4.0, 4.5, 0.0]])
    # sorted 5, 4.5, 4, 1, 0 ; top-3 (k=2) gaps 0.5, 0.5
    assert oracle.route_margin(logits, 2)[0] == 0.5
    assert oracle.route_margin(logits, 3)[0] == 0.5
    assert oracle.route_margin(logits, 4)[0] == 0.5
    assert oracle.route_margin(np.array([[1.0, 1.0 + 1e-4, -2]]), 1)[0] == pytest.approx(1e-4)


# ---- experts ---------------------------------------------------------------------

def test_silu_matches_library():
    a = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(oracle.silu(a), a * scipy.special.expit(a), rtol=1e-14,
                               atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0


def test_expert_identity_weights():
    """p = I with W_gate = g*Id (large g), W_up = Id, W_down = Id:
    s_i = silu(g u_i) u_i -> g u_i^2 for u_i > 0 and ~0 for u_i < 0; y = s."""
    u = np.array([[0.5, -0.25, 2.0, -1.0]])
    eye = np.eye(4)
    s = oracle.expert_swiglu(u, 40.0 * eye, eye)
    ref = 40.0 * u * scipy.special.expit(40.0 * u) * u
    np.testing.assert_allclose(s, ref, rtol=1e-14)
    np.testing.assert_allclose(oracle.expert_down(s, eye), s, rtol=0)
    # a permutation matrix as W_down permutes the outputs (operand orientation)
    P = eye[[2, 0, 3, 1]]
    np.testing.assert_allclose(oracle.expert_down(s, P), s[:, [2, 0, 3, 1]], rtol=0)


# ---- block-level invariances -----------------------------------------------------

def _scaled(inp, key, c, expert=None):
    """Copy of the inputs (as float64 numpy) with one tensor, or one expert's slice,
    multiplied by c exactly."""
    out = {k: np.asarray(v, dtype=np.float64) for k, v in np_inputs(inp).items()}
    if expert is None:
        out[key] = out[key] * c
    else:
        out[key] = out[key].copy()
        out[key][expert] *= c
    return out


def test_scale_invariances_pin_norm_placement():
    """Each RMSNorm removes a positive scale in front of it (up to eps):
    x*c (full-width norm), W_pool*c (pooled-input norm), one expert's W_down*c or
    W_up*c (per-expert norm).  W_unpool*c scales the output; W_gate*c does not
    cancel (SwiGLU is not homogeneous in the gate)."""
    shape, inp = tiny(T=24, E=5, k=3)
    # eps = 0 makes each invariance exact up to float64 rounding
    base = fwd(inp, shape, eps=0.0)
    scale = float(np.sqrt(np.mean(base ** 2)))
    for key, expert, c in [("x", None, 3.0), ("w_pool", None, 0.3), ("w_down", 2, 7.0),
                           ("w_up", 4, 0.1), ("w_down", 0, 5.0)]:
        got = fwd(_scaled(inp, key, c, expert), shape, eps=0.0)
        assert np.max(np.abs(got - base)) / scale < 1e-9, (key, expert)
    got = fwd(_scaled(inp, "w_unpool", 2.5), shape, eps=0.0)
    np.testing.assert_allclose(got, 2.5 * base, rtol=1e-12, atol=1e-12 * scale)
    ids = fwd(inp, shape, return_parts=True)["ids"]
    e_used = int(ids[0, 0])
    got = fwd(_scaled(inp, "w_gate", 3.0, e_used), shape, eps=0.0)
    assert np.max(np.abs(got - base)) / scale > 1e-3


def test_norm_before_weighting_differs_from_norm_after_sum():
    """The page: normalising the combined output would change the computation.
    With unit per-expert gains the two orders must differ by far more than the
    rounding-chain error."""
    shape, inp = tiny(T=32, E=6, k=3)
    inp["g_exp"] = torch.ones_like(inp["g_exp"])
    a = fwd(inp, shape)
    b = fwd(inp, shape, norm_after_sum=True)
    chain = fwd(inp, shape, chain=True)
    rms = float(np.sqrt(np.mean(a ** 2)))
    diff_order = np.max(np.abs(a - b)) / rms
    diff_chain = np.max(np.abs(a - chain)) / rms
    assert diff_order > 0.05
    assert diff_chain < diff_order / 20


def test_top1_is_the_single_chosen_expert():
    """k = 1: the weight is exactly 1 and the output equals a one-expert layer built
    from the chosen expert alone (no routing involved)."""
    shape, inp = tiny(T=12, E=5, k=1)
    parts = fwd(inp, shape, return_parts=True)
    assert np.all(parts["w"] == 1.0)
    for t in range(shape.T):
        e = int(parts["ids"][t, 0])
        one = dict(inp)
        for key in ("w_gate", "w_up", "w_down", "g_exp"):
            one[key] = inp[key][e: e + 1]
        one["w_router"] = inp["w_router"][e: e + 1]
        one["x"] = inp["x"][t: t + 1]
        single = fwd(one, shape.replace(E=1), top_k=1)
        np.testing.assert_allclose(parts["out"][t: t + 1], single, rtol=1e-13, atol=1e-13)
    # with k=1 the router scale does not matter; with k=2 it does (weights change)
    a = fwd(_scaled(inp, "w_router", 3.0), shape)
    np.testing.assert_allclose(a, parts["out"], rtol=1e-13, atol=1e-13)
    shape2, inp2 = tiny(T=12, E=5, k=2)
    b0 = fwd(inp2, shape2)
    b1 = fwd(_scaled(inp2, "w_router", 3.0), shape2)
    assert np.max(np.abs(b0 - b1)) > 1e-3


def test_expert_relabelling():
    """Permuting expert ids together with router rows, expert weights and gains
    leaves the output unchanged and permutes the chosen ids."""
    shape, inp = tiny(T=20, E=7, k=3)
    perm = torch.tensor([3, 6, 0, 5, 1, 4, 2])
    relab = dict(inp)
    for key in ("w_router", "w_gate", "w_up", "w_down", "g_exp"):
        relab[key] = inp[key][perm]
    a = fwd(inp, shape, return_parts=True)
    b = fwd(relab, shape, return_parts=True)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-13, atol=1e-13)
    inv = torch.argsort(perm).numpy()
    np.testing.assert_array_equal(inv[a["ids"]], b["ids"])


def test_rows_are_independent():
    """The pooler keeps the token count; each row is computed alone: a per-row call
    equals the batched row, and permuting tokens permutes the output rows."""
    shape, inp = tiny(T=9)
    full = fwd(inp, shape)
    assert full.shape == (shape.T, shape.d)
    for t in (0, 4, 8):
        np.testing.assert_allclose(fwd(inp, shape, tokens=[t]), full[t: t + 1], rtol=1e-12,
                                   atol=1e-13)
    perm = np.array([5, 2, 8, 0, 1, 7, 3, 6, 4])
    np.testing.assert_allclose(fwd(inp, shape, tokens=perm), full[perm], rtol=1e-14,
                               atol=1e-14)


def test_unit_gain_bound():
    """Unit per-expert gains: rms(c_t) <= 1 (triangle inequality, weights sum to 1),
    with equality when every chosen expert is the same function (then c = N(y))."""
    shape, inp = tiny(T=30, E=6, k=3)
    inp["g_exp"] = torch.ones_like(inp["g_exp"])
    parts = fwd(inp, shape, return_parts=True)
    rms_c = np.sqrt(np.mean(parts["c"] ** 2, axis=1))
    assert np.all(rms_c <= 1.0 + 1e-12)
    assert np.all(rms_c < 0.999)
    same = dict(inp)
    for key in ("w_gate", "w_up", "w_down"):
        same[key] = inp[key][:1].expand_as(inp[key]).clone()
    parts = fwd(same, shape, return_parts=True, eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(parts["c"] ** 2, axis=1)), 1.0, rtol=1e-13)


def test_brute_force_loops():
    """A pure-Python loop over tokens, slots and matrix entries (no numpy algebra) on
    a tiny case equals the oracle, pinning its grouping by expert and its matrix
    orientations."""
    shape, inp = tiny(T=3, d=6, p=4, E=4, k=2, I=5, seed=3)
    v = np_inputs(inp)
    eps = shape.eps

    def norm(vec, g):
        vec = [float(a) for a in vec]
        ms = sum(a * a for a in vec) / len(vec)
        return [a / math.sqrt(ms + eps) * float(gg) for a, gg in zip(vec, g)]

    def matvec(m, vec):
        return [sum(float(m[r][c]) * vec[c] for c in range(len(vec))) for r in range(len(m))]

    ref = fwd(inp, shape, return_parts=True)
    for t in range(shape.T):
        h = norm(list(v["x"][t]), v["g_in"])
        u = norm(matvec(v["w_pool"], h), v["g_pool"])
        c = [0.0] * shape.p
        for j in range(shape.top_k):
            e = int(ref["ids"][t, j])
            a = matvec(v["w_gate"][e], u)
            b = matvec(v["w_up"][e], u)
            s = [ai / (1 + math.exp(-ai)) * bi for ai, bi in zip(a, b)]
            y = norm(matvec(v["w_down"][e], s), v["g_exp"][e])
            c = [ci + float(ref["w"][t, j]) * yi for ci, yi in zip(c, y)]
        out = matvec(v["w_unpool"], c)
        np.testing.assert_allclose(ref["out"][t], out, rtol=1e-12, atol=1e-12)


def test_routing_replay_equals_internal_route():
    """Passing the router's own ids/weights back in reproduces the output."""
    shape, inp = tiny(T=10)
    parts = fwd(inp, shape, return_parts=True)
    again = fwd(inp, shape, ids=parts["ids"], weights=parts["w"])
    np.testing.assert_array_equal(again, parts["out"])


def test_chain_stays_close_to_exact():
    """The storage-rounding chain (BF16 intermediates) moves the output by about the
    BF16 resolution, not more: max error / rms well under 1e-2."""
    shape, inp = tiny(T=32, d=64, p=32, E=6, k=2, I=48, act="bf16", expert="bf16")
    exact = fwd(inp, shape, chain=False)
    chain = fwd(inp, shape, chain=True)
    rms = float(np.sqrt(np.mean(exact ** 2)))
    err = np.max(np.abs(chain - exact)) / rms
    assert 1e-5 < err < 2e-2


def test_chain_stores_expert_outputs_where_the_kernels_do():
    """The chain keeps y, the per-expert norm's input, on the FP16 grid for BF16 experts
    (and s too: every activation between the GEMMs is FP16 there) and in FP32 for FP32
    experts, and the norm then reads those stored values."""
    shape, inp = tiny(T=16, d=64, p=32, E=6, k=2, I=48, act="bf16", expert="bf16")
    parts = fwd(inp, shape, chain=True, return_parts=True)
    y = parts["y"]
    assert np.array_equal(F.fp16(y), y) and not np.array_equal(F.bf16(y), y)
    assert np.array_equal(F.fp16(parts["s"]), parts["s"])
    assert not np.array_equal(F.bf16(parts["u"]), parts["u"])      # u is FP16, finer
    shape32, inp32 = tiny(T=16, d=64, p=32, E=6, k=2, I=48)
    y32 = fwd(inp32, shape32, chain=True, return_parts=True)["y"]
    assert np.array_equal(F.fp32(y32), y32) and not np.array_equal(F.bf16(y32), y32)
    # the combine normalises exactly the stored rows
    c = oracle.combine(y, parts["ids"], parts["w"], oracle_view(inp)["g_exp"], shape.eps)
    assert np.allclose(c, parts["c"], rtol=1e-3, atol=1e-3 * float(np.abs(c).max()))


def test_margin_repair_makes_routes_unique():
    shape, inp = tiny(T=64, E=8, k=2)
    fix_margins(inp, shape, seed=0, min_gap=1e-3)
    _, _, logits = oracle.route(np_inputs(inp), top_k=shape.top_k, eps=shape.eps)
    assert np.all(oracle.route_margin(logits, shape.top_k) >= 1e-3)
