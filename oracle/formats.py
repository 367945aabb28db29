"""Number formats used by the oracle, written from their definitions.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; it exists
so the CPU oracle can reproduce the rounding points at which the GPU path stores
values.  Every function works on float64 numpy arrays and returns float64 arrays
holding exactly representable values of the target format.

Definitions followed:
* BF16: 1 sign, 8 exponent, 7 stored mantissa bits (8 significant bits);
  conversion rounds to nearest, ties to even.
* TF32: FP32 with the low 13 mantissa bits dropped (11 significant bits); the
  GPU path converts with round-to-nearest, ties AWAY from zero (`cvt.rna.tf32.f32`),
  which is the rounding the oracle mirrors.
* FP32: IEEE binary32, round to nearest even (numpy's cast).
* FP16: IEEE binary16 (11 significant bits, subnormals 2^-24 apart below 2^-14),
  round to nearest even (numpy's cast from float64).
* E2M1 (FP4): sign + 2-bit exponent + 1-bit mantissa, magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}; NVFP4 encodes by round-to-nearest-even on that
  grid, saturating at 6.  ("SGLang and Miles Add Day-0 Support for Muse Spark
  Open", section "NVFP4 as a third MMA kind": dense FP4 operands with an E4M3
  scale per 16 elements.)
* UE4M3 (unsigned FP8 E4M3 block scale): exponent bias 7, 3 mantissa bits,
  subnormals 2^-6 * m/8, largest finite 448; round to nearest even, saturating.
"""
from __future__ import annotations

import numpy as np


def _round_mantissa_rne(x: np.ndarray, keep: int) -> np.ndarray:
    """Round float64 values to `keep` stored mantissa bits, nearest-even.

    Works on the binary64 encoding: the dropped 52-keep bits decide.  Assumes the
    result's exponent is inside the target's normal range (true for every value
    this project rounds: all non-zero values are far above 2^-126).
    """
    x = np.asarray(x, dtype=np.float64)
    bits = x.view(np.uint64).copy()
    drop = np.uint64(52 - keep)
    one = np.uint64(1)
    lsb = (bits >> drop) & one
    half_minus_one = (one << (drop - one)) - one
    bits = bits + half_minus_one + lsb
    bits &= ~((one << drop) - one)
    out = bits.view(np.float64)
    return np.where(np.isfinite(x), out, x)


def bf16(x) -> np.ndarray:
    """Round to BF16 (nearest even)."""
    return _round_mantissa_rne(x, 7)


def fp32(x) -> np.ndarray:
    """Round to IEEE binary32 (nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def fp16(x) -> np.ndarray:
    """Round to IEEE binary16 (nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def tf32_rna(x) -> np.ndarray:
    """Round FP32 values to TF32 with ties away from zero.

    The input is first taken to FP32 (it already is, for the values the GPU
    stores); then half a TF32 unit is added to the magnitude and the low 13
    mantissa bits are cleared.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).copy()
    finite = np.isfinite(f)
    bits = np.where(finite, (bits + np.uint32(1 << 12)) & np.uint32(0xFFFFE000), bits)
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


# ---- FP4 (E2M1) -------------------------------------------------------------------

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(code) -> np.ndarray:
    """4-bit code (bit 3 = sign, bits 2..0 = magnitude index) -> value."""
    code = np.asarray(code, dtype=np.int64)
    mag = E2M1_MAGNITUDES[code & 7]
    return np.where(code & 8, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """Nearest E2M1 code, ties to the even code (even mantissa bit), saturating at 6.

    The grid steps are 0.5 on [0, 2], 1 on [2, 4] and 2 on [4, 6]; on a tie the
    code whose mantissa bit is 0 wins (0.25->0, 0.75->1, 1.25->1, 1.75->2,
    2.5->2, 3.5->4, 5->4).
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    # The magnitude index is the number of midpoints between neighbouring grid values
    # that |v| has passed.  At a midpoint itself the neighbour with an even index
    # (mantissa bit 0) wins: the index moves up at the midpoints below the even
    # indices 2, 4, 6 (0.75, 1.75, 3.5: ">=") and stays at the midpoints above the
    # even indices 0, 2, 4, 6 (0.25, 1.25, 2.5, 5: ">").  Values above 5 give index 7
    # (6), so magnitudes beyond 6 saturate.
    best = ((a > 0.25).astype(np.int64) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
            + (a > 2.5) + (a >= 3.5) + (a > 5.0))
    # the sign bit follows the input's sign, also when the magnitude rounds to zero
    # (as for IEEE conversions: -0.1 -> -0)
    return (best | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


# ---- UE4M3 (block scale) ----------------------------------------------------------

def ue4m3_decode(code) -> np.ndarray:
    """8-bit unsigned E4M3 code -> value (code 0x7f would be NaN; never produced)."""
    code = np.asarray(code, dtype=np.int64)
    e = (code >> 3) & 0xF
    m = code & 7
    sub = np.ldexp(m / 8.0, -6)
    nrm = np.ldexp(1.0 + m / 8.0, e - 7)
    return np.where(e == 0, sub, nrm)


_UE4M3_ALL = ue4m3_decode(np.arange(0x7F))  # 0x00..0x7e, ascending, finite


def ue4m3_encode(v) -> np.ndarray:
    """Nearest UE4M3 code (ties to even code), saturating at 448; negatives -> 0."""
    v = np.clip(np.asarray(v, dtype=np.float64), 0.0, 448.0)
    idx = np.searchsorted(_UE4M3_ALL, v)           # first grid value >= v
    idx = np.clip(idx, 1, len(_UE4M3_ALL) - 1)
    lo, hi = _UE4M3_ALL[idx - 1], _UE4M3_ALL[idx]
    pick_hi = (v - lo > hi - v) | ((v - lo == hi - v) & ((idx & 1) == 0))
    code = np.where(pick_hi, idx, idx - 1)
    code = np.where(v >= _UE4M3_ALL[-1], len(_UE4M3_ALL) - 1, code)
    return code.astype(np.uint8)
