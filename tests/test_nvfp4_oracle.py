"""Pins of the oracle's NVFP4 quantiser ("SGLang and Miles Add Day-0 Support for Muse
Spark Open", section "NVFP4 as a third MMA kind": E2M1 values, one UE4M3 scale per 16
elements, FP32 global scale) against closed forms and the format definitions."""
import numpy as np
import pytest

import oracle
from oracle import formats as F
from oracle import nvfp4 as Q


def test_constant_block_is_exact():
    """A tensor of one value c: g = c/2688, the block scale is 448 (code 0x7e), every
    code is 6, and the value comes back exactly (up to the FP32 rounding of g)."""
    for c in (0.75, 3.0, 1e-3):
        w = np.full((2, 32), c, dtype=np.float32)
        q, sf, g = Q.quantize_tensor(w)
        assert np.all(sf == 0x7E)
        assert np.all(q == 7)
        np.testing.assert_allclose(Q.dequantize(q, sf, g), c, rtol=2 ** -23)


def test_zero_tensor_and_zero_row():
    q, sf, g = Q.quantize_tensor(np.zeros((3, 16)))
    assert g == 0 and np.all(q == 0) and np.all(sf == 0)
    x = np.ones((2, 16), dtype=np.float32)
    x[1] = 0
    q, sf, g = Q.quantize_rows(x)
    assert g[1] == 0 and np.all(q[1] == 0) and np.all(sf[1] == 0)
    assert np.all(Q.dequantize(q, sf, g)[1] == 0)


def test_representable_values_round_trip():
    """Values e2m1 * ue4m3 * g with a +-6 in every block quantise to themselves."""
    rng = np.random.default_rng(0)
    rows, K = 8, 64
    codes = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    codes[:, ::16] = 7                        # the block maximum is 6 * scale
    sf = rng.integers(0x20, 0x60, size=(rows, K // 16)).astype(np.uint8)
    sf[0, 0] = 0x7E                           # one block at the top scale: g is exact
    g = np.float32(0.01)
    x = Q.dequantize(codes, sf, g).astype(np.float32)
    q2, sf2 = Q.quantize_blocks(x, np.full(rows, g, np.float32))
    np.testing.assert_array_equal(sf2, sf)
    np.testing.assert_array_equal(F.e2m1_decode(q2), F.e2m1_decode(codes))


def test_error_bound():
    """Each element is within half an E2M1 grid step of its scaled value, except at the
    top of a block whose scale rounded down, where it saturates at 6 * scale; the block
    scale itself is within 1/16 (half a UE4M3 step) of bmax / 6."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 256)) * rng.lognormal(0, 2, (64, 1))).astype(np.float32)
    q, sf, g = Q.quantize_rows(x)
    d = Q.dequantize(q, sf, g)
    S = (F.ue4m3_decode(sf) * g[:, None]).repeat(16, axis=1)          # scale * g
    a = np.abs(x) / S
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    bound = np.maximum(0.5 * step * S, np.abs(x) - 6 * S) * (1 + 1e-5)
    assert np.all(np.abs(d - x) <= bound)
    bmax = np.abs(x).reshape(64, 16, 16).max(-1)
    rel = np.abs(F.ue4m3_decode(sf) * g[:, None] * 6 - bmax) / bmax
    assert np.all(rel <= 1 / 16 + 1e-6)


def test_power_of_two_scaling_is_exact():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    q1, s1, g1 = Q.quantize_tensor(x)
    q2, s2, g2 = Q.quantize_tensor(x * np.float32(8.0))
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)
    assert g2 == g1 * 8


def test_reciprocal_table():
    """The 256-entry table ("The NVFP4 requantization reciprocal table"): 1/scale by IEEE
    division for every finite nonzero code, 0 for the zero code."""
    t = Q.recip_table()
    vals = F.ue4m3_decode(np.arange(1, 0x7F))
    np.testing.assert_array_equal(t[1:0x7F], (np.float32(1) / vals.astype(np.float32)))
    assert t[0] == 0 and t[0x38] == 1.0 and t[0x7E] == np.float32(1 / 448)


def test_nvfp4_layer_close_to_bf16_layer():
    """The NVFP4 block stays close to the unquantised block (FP4 noise ~ 10 % per
    quantisation is damped by the norms) and its routing equals the BF16 routing (the
    router is not quantised)."""
    from latent_moe_layer_rmsnorm_gb300 import synth
    from harness import oracle_view
    shape = synth.Shape("q", T=24, d=256, p=128, E=6, top_k=2, I=256, expert="nvfp4")
    inp = synth.make_inputs(shape, seed=0)
    view = oracle_view(inp)
    a = oracle.moe_forward(view, top_k=2, eps=shape.eps, act="bf16", expert="nvfp4",
                           return_parts=True)
    b = oracle.moe_forward(view, top_k=2, eps=shape.eps, act="bf16", expert="bf16",
                           chain=False, return_parts=True)
    np.testing.assert_array_equal(a["ids"], b["ids"])
    rel = np.sqrt(np.mean((a["out"] - b["out"]) ** 2) / np.mean(b["out"] ** 2))
    assert 0.01 < rel < 0.3
