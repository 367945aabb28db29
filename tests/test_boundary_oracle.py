"""Pins of the oracle's block boundary (post-norm, residual add, next pre-norm) against
facts that do not come from the oracle: a row worked out on paper, closed forms and
invariances.  Sources: "vLLM 对 Muse Spark Open 的 Day 0 支持" (vLLM Day-0 support for Muse
Spark Open), section "三明治归一化" (a norm before and after the block: x + post_norm(F(norm
(x)))), and "SGLang and Miles Add Day-0 Support for Muse Spark Open", section "Kernel
Optimizations" (post-FFN norm, gated residual add and pre-attention norm in one pass).
"""
import json
import math
import os

import numpy as np

import oracle
from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _row(rng, d, scale=1.0):
    return rng.standard_normal((3, d)) * scale


def test_hand_worked_boundary():
    """A 2-wide row computed on paper (tests/golden/boundary_hand_worked.json), with and
    without a per-channel gate."""
    g = json.load(open(os.path.join(GOLDEN, "boundary_hand_worked.json")))
    ev = lambda e: eval(e, {"sqrt": math.sqrt})
    for case in g["cases"]:
        xn, hn = oracle.boundary(np.array(g["x"]), np.array(g["y"]), g["g_post"], g["g_next"],
                                 g["eps"], gate=case["gate"], act="f64")
        np.testing.assert_allclose(xn, [[ev(v) for v in case["x_new"][0]]], rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(hn, [[ev(v) for v in case["h_next"][0]]], rtol=1e-14, atol=1e-14)


def test_post_norm_makes_the_block_output_scale_free():
    """Scaling the block output by any c > 0 leaves both results unchanged (eps = 0):
    the output enters only through a norm."""
    rng = np.random.default_rng(1)
    d = 64
    x, y = _row(rng, d), _row(rng, d)
    gp, gn = rng.uniform(0.5, 1.5, d), rng.uniform(0.5, 1.5, d)
    base = oracle.boundary(x, y, gp, gn, 0.0, act="f64")
    for c in (1e-3, 0.7, 250.0):
        xs, hs = oracle.boundary(x, c * y, gp, gn, 0.0, act="f64")
        np.testing.assert_allclose(xs, base[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(hs, base[1], rtol=1e-12, atol=1e-12)


def test_zero_gate_passes_the_residual_through():
    """gate = 0: the residual stream is x unchanged and the next pre-norm is the plain
    RMSNorm of x (a scaled copy of x whose mean square is 1 with unit gains)."""
    rng = np.random.default_rng(2)
    d = 32
    x, y = _row(rng, d, 3.0), _row(rng, d)
    xn, hn = oracle.boundary(x, y, np.ones(d), np.ones(d), 0.0, gate=np.zeros(d), act="f64")
    np.testing.assert_array_equal(xn, x)
    np.testing.assert_allclose(np.mean(hn * hn, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(hn * np.sqrt(np.mean(x * x, axis=-1, keepdims=True)), x, rtol=1e-12)


def test_residual_adds_the_normalised_output():
    """Unit gains, plain residual: x' - x has mean square exactly 1 (eps = 0) and points
    along y; a negative gate subtracts it."""
    rng = np.random.default_rng(3)
    d = 48
    x, y = _row(rng, d), _row(rng, d, 5.0)
    xn, _ = oracle.boundary(x, y, np.ones(d), np.ones(d), 0.0, act="f64")
    delta = xn - x
    np.testing.assert_allclose(np.mean(delta * delta, axis=-1), 1.0, rtol=1e-12)
    cos = np.sum(delta * y, axis=-1) / np.linalg.norm(delta, axis=-1) / np.linalg.norm(y, axis=-1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-12)
    xm, _ = oracle.boundary(x, y, np.ones(d), np.ones(d), 0.0, gate=-np.ones(d), act="f64")
    np.testing.assert_allclose(xm - x, -delta, rtol=1e-12, atol=1e-15)


def test_eps_bounds_the_pre_norm():
    """With unit gains the next pre-norm's mean square is ms / (ms + eps) < 1, the closed
    form of v / sqrt(mean(v^2) + eps)."""
    rng = np.random.default_rng(4)
    d = 16
    x, y = _row(rng, d, 1e-3), _row(rng, d)
    eps = 1e-6
    xn, hn = oracle.boundary(x, y, np.ones(d), np.ones(d), eps, gate=np.zeros(d), act="f64")
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(hn * hn, axis=-1), ms / (ms + eps), rtol=1e-12)


def test_pre_norm_reads_the_stored_residual():
    """With BF16 storage the next pre-norm is taken on x' as stored (what an unfused
    next block would read), and both results are representable in BF16."""
    rng = np.random.default_rng(5)
    d = 256
    x = F.bf16(_row(rng, d))
    y = _row(rng, d)
    gp, gn = rng.uniform(0.5, 1.5, d), rng.uniform(0.5, 1.5, d)
    xn, hn = oracle.boundary(x, y, gp, gn, 1e-6, act="bf16")
    np.testing.assert_array_equal(F.bf16(xn), xn)
    np.testing.assert_array_equal(F.bf16(hn), hn)
    # the unrounded residual gives a different pre-norm on some element: storage matters
    x64, _ = oracle.boundary(x, y, gp, gn, 1e-6, act="f64")
    assert not np.array_equal(x64, xn)
    _, h_from_stored = oracle.boundary(xn, np.zeros_like(y), gp, gn, 1e-6,
                                       gate=np.zeros(d), act="bf16")
    np.testing.assert_array_equal(h_from_stored, hn)
