"""Pins of the oracle's number-format helpers against their definitions and
library conversions (torch's FP32->BF16 cast rounds to nearest even)."""
import numpy as np
import torch

from oracle import formats as F


def test_bf16_matches_torch_cast():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(size=20000) * 10.0 ** rng.integers(-8, 8, 20000),
                        [0.0, -0.0, 1.0, -1.5, 3.0e38]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(F.bf16(v.astype(np.float64)), ref.astype(np.float64))


def test_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1
    assert F.bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6 -> the even one, 1 + 2^-6
    assert F.bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert F.bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -30]))[0] == 1 + 2.0 ** -7
    assert F.bf16(np.array([-(1 + 2.0 ** -8)]))[0] == -1.0


def test_tf32_rounds_ties_away():
    # TF32 keeps 10 mantissa bits: ulp(1) = 2^-10
    assert F.tf32_rna(np.array([1 + 2.0 ** -11]))[0] == 1 + 2.0 ** -10
    assert F.tf32_rna(np.array([-(1 + 2.0 ** -11)]))[0] == -(1 + 2.0 ** -10)
    assert F.tf32_rna(np.array([1 + 2.0 ** -11 - 2.0 ** -23]))[0] == 1.0
    assert F.tf32_rna(np.array([1 + 3 * 2.0 ** -11]))[0] == 1 + 2 * 2.0 ** -10
    v = np.random.default_rng(1).normal(size=1000)
    r = F.tf32_rna(v)
    assert np.all((r.astype(np.float32).view(np.uint32) & 0x1FFF) == 0)
    assert np.all(np.abs(r - v) <= np.abs(v) * 2.0 ** -11 * (1 + 1e-6))


def test_e2m1_table_and_round_trip():
    vals = F.e2m1_decode(np.arange(16))
    np.testing.assert_array_equal(vals[:8], [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    np.testing.assert_array_equal(vals[8:], -vals[:8])
    codes = F.e2m1_encode(vals)
    np.testing.assert_array_equal(F.e2m1_decode(codes), vals)


def test_e2m1_ties_and_saturation():
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in ties.items():
        assert F.e2m1_decode(F.e2m1_encode(np.array([v])))[0] == want, v
        assert F.e2m1_decode(F.e2m1_encode(np.array([-v])))[0] == -want, v
    assert F.e2m1_decode(F.e2m1_encode(np.array([100.0])))[0] == 6.0
    assert F.e2m1_decode(F.e2m1_encode(np.array([-7.0])))[0] == -6.0
    assert F.e2m1_encode(np.array([-0.1]))[0] == 8          # -0 keeps its sign
    assert F.e2m1_encode(np.array([0.1]))[0] == 0


def test_e2m1_encode_is_nearest_even_on_a_dense_sweep():
    """The encoder against the format's definition, applied by brute force: the nearest
    of the eight magnitudes, ties to the one with an even index (mantissa bit 0),
    saturating at 6.  The sweep covers every midpoint and its FP32 neighbours."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (grid[1:] + grid[:-1]) / 2
    near = np.concatenate([np.nextafter(mids.astype(np.float32), np.float32(-1)),
                           np.nextafter(mids.astype(np.float32), np.float32(9))])
    v = np.concatenate([np.linspace(0, 8, 160001), mids, near.astype(np.float64), grid])
    v = np.concatenate([v, -v])
    a = np.minimum(np.abs(v), 6.0)
    best = np.empty(len(v), dtype=np.int64)
    for i, x in enumerate(a):
        d = np.abs(grid - x)
        cand = np.nonzero(d == d.min())[0]
        best[i] = cand[0] if len(cand) == 1 else cand[cand % 2 == 0][0]
    want = np.where(np.signbit(v), -grid[best], grid[best])
    np.testing.assert_array_equal(F.e2m1_decode(F.e2m1_encode(v)), want)


def test_ue4m3_table_and_round_trip():
    codes = np.arange(0x7F)
    vals = F.ue4m3_decode(codes)
    assert vals[0] == 0.0 and vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6
    assert vals[0x38] == 1.0 and vals[0x7E] == 448.0
    assert np.all(np.diff(vals) > 0)
    np.testing.assert_array_equal(F.ue4m3_encode(vals), codes)


def test_ue4m3_rounding():
    # between 1 (0x38) and 1.125 (0x39): the tie goes to the even code 0x38
    assert F.ue4m3_encode(np.array([1.0625]))[0] == 0x38
    # between 1.125 (0x39) and 1.25 (0x3a): tie -> 0x3a
    assert F.ue4m3_encode(np.array([1.1875]))[0] == 0x3A
    assert F.ue4m3_encode(np.array([1.05]))[0] == 0x38
    assert F.ue4m3_encode(np.array([1.07]))[0] == 0x39
    assert F.ue4m3_encode(np.array([1e9]))[0] == 0x7E
    assert F.ue4m3_encode(np.array([-1.0]))[0] == 0


def test_fp16_matches_torch_cast():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.normal(size=20000) * 10.0 ** rng.integers(-9, 4, 20000),
                        [0.0, 1.0, 65504.0, 2.0 ** -24, 3 * 2.0 ** -26]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float16).to(torch.float32).numpy()
    np.testing.assert_array_equal(F.fp16(v.astype(np.float64)), ref.astype(np.float64))
    # bf16 values of ordinary magnitude are exact in fp16 (3 more significand bits)
    b = F.bf16(rng.normal(size=5000) * 0.02)
    big = np.abs(b) >= 2.0 ** -17
    np.testing.assert_array_equal(F.fp16(b)[big], b[big])
