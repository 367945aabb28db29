"""NVFP4 quantisation for the oracle (test infrastructure only).

NVFP4 ("SGLang and Miles Add Day-0 Support for Muse Spark Open", section "NVFP4 as a
third MMA kind"): dense FP4 (E2M1) values with one UE4M3 scale per 16 elements along
K, and an FP32 global scale per tensor (weights) or per token (activations; "per-token
FP32 input scales are applied to the first GEMM's accumulators").  A stored value is
    v = e2m1(code) * ue4m3(scale_code) * g.

Quantising decides integer codes, so the oracle takes those decisions in the
kernel's precision: every step below is an IEEE FP32 operation in the same order the
quantiser kernels use (numpy float32 arithmetic is correctly rounded):

    g      = amax / 2688                (2688 = 6 * 448; or a given static scale)
    sf     = ue4m3_rne_sat( bmax / (6 * g) )              bmax = max |x| of the block
    r      = recip(sf) * (1 / g)        recip(sf) = 1 / ue4m3(sf), recip(0) = 0
    code   = e2m1_rne_sat( x * r )

g = 0 (an all-zero tensor or row) gives codes 0 and scale codes 0.
"""
from __future__ import annotations

import numpy as np

from . import formats as F

F32 = np.float32
BLOCK = 16
E2M1_MAX_TIMES_E4M3_MAX = 2688.0


def recip_table() -> np.ndarray:
    """FP32 reciprocal of every UE4M3 code (0 for code 0), IEEE division; codes 0x7f..
    are not produced by the quantiser and map to 0."""
    vals = F.ue4m3_decode(np.arange(256) & 0x7F).astype(F32)
    out = np.zeros(256, dtype=F32)
    ok = (np.arange(256) > 0) & (np.arange(256) < 0x7F)
    out[ok] = (F32(1.0) / vals[ok]).astype(F32)
    return out


_RECIP = recip_table()


def global_scale(amax) -> np.ndarray:
    return (np.asarray(amax, dtype=F32) / F32(E2M1_MAX_TIMES_E4M3_MAX)).astype(F32)


def quantize_blocks(x: np.ndarray, g: np.ndarray):
    """x [..., K] (FP32 values), g broadcastable to x[..., 0]: (codes [..., K] uint8,
    scale codes [..., K/16] uint8)."""
    x = np.asarray(x, dtype=F32)
    K = x.shape[-1]
    assert K % BLOCK == 0
    xb = x.reshape(*x.shape[:-1], K // BLOCK, BLOCK)
    g = np.asarray(g, dtype=F32)[..., None]                       # per block row
    bmax = np.max(np.abs(xb), axis=-1)
    six_g = (F32(6.0) * g).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(six_g > 0, bmax / six_g, F32(0.0)).astype(F32)
        inv_g = np.where(g > 0, F32(1.0) / g, F32(0.0)).astype(F32)
    sf = F.ue4m3_encode(ratio.astype(np.float64))
    r = (_RECIP[sf] * inv_g).astype(F32)
    q = F.e2m1_encode((xb * r[..., None]).astype(F32).astype(np.float64))
    return q.reshape(x.shape), sf


def dequantize(codes: np.ndarray, sf: np.ndarray, g) -> np.ndarray:
    """Stored NVFP4 values, float64."""
    v = F.e2m1_decode(codes)
    K = v.shape[-1]
    s = F.ue4m3_decode(sf)
    v = v.reshape(*v.shape[:-1], K // BLOCK, BLOCK) * s[..., None]
    return v.reshape(codes.shape) * np.asarray(g, dtype=np.float64)[..., None]


def quantize_tensor(w: np.ndarray):
    """A weight matrix with one global scale: (codes, scale codes, g)."""
    w = np.asarray(w, dtype=F32)
    g = global_scale(np.max(np.abs(w)))
    q, sf = quantize_blocks(w, g)
    return q, sf, g


def quantize_rows(x: np.ndarray):
    """Activations with a global scale per row (token): (codes, scale codes, g [rows])."""
    x = np.asarray(x, dtype=F32)
    g = global_scale(np.max(np.abs(x), axis=-1))
    q, sf = quantize_blocks(x, g)
    return q, sf, g


def quantize_static(x: np.ndarray, g: float):
    """Activations with a given static global scale (the requantised SwiGLU output)."""
    x = np.asarray(x, dtype=F32)
    q, sf = quantize_blocks(x, np.full(x.shape[:-1], g, dtype=F32))
    return q, sf


# ---- how close each rounding decision is to changing ---------------------------------

_E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
_UE4M3_MIDPOINTS = (F.ue4m3_decode(np.arange(1, 0x7F)) + F.ue4m3_decode(np.arange(0, 0x7E))) / 2


def decision_margins(x: np.ndarray, g: np.ndarray):
    """Distances, in the units of x, from the two kinds of rounding decision that
    quantize_blocks(x, g) takes to the points where those decisions would change.

    elem [..., K]: for each element, |x * r - m| / r, where r is the element's block
    multiplier (recip(scale) / g, as in quantize_blocks) and m is the E2M1 rounding
    midpoint nearest to |x * r|: how far x may move before its code changes (block
    scale held).  inf where r = 0 (a zero block or g = 0).
    block [..., K/16]: for each block, |bmax / (6 g) - m'| * 6 g, m' the UE4M3 midpoint
    nearest to bmax / (6 g): how far the block maximum may move before the block's
    scale code changes.  inf where g = 0.

    When two computations of x differ by less than these distances, they quantise to
    the same codes.  Arithmetic in float64 on the FP32 quantities of quantize_blocks.
    """
    x = np.asarray(x, dtype=F32)
    K = x.shape[-1]
    xb = x.reshape(*x.shape[:-1], K // BLOCK, BLOCK).astype(np.float64)
    g32 = np.asarray(g, dtype=F32)[..., None]
    bmax = np.max(np.abs(xb), axis=-1)
    six_g = (F32(6.0) * g32).astype(F32).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(six_g > 0, bmax / six_g, 0.0)
        inv_g = np.where(g32 > 0, F32(1.0) / g32, F32(0.0)).astype(F32)
    sf = F.ue4m3_encode(ratio.astype(F32).astype(np.float64))
    r = (_RECIP[sf] * inv_g).astype(F32).astype(np.float64)
    v = np.abs(xb) * r[..., None]
    d_elem = np.min(np.abs(v[..., None] - _E2M1_MIDPOINTS), axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        elem = np.where(r[..., None] > 0, d_elem / r[..., None], np.inf)
        d_blk = np.min(np.abs(ratio[..., None] - _UE4M3_MIDPOINTS), axis=-1)
        block = np.where(six_g > 0, d_blk * six_g, np.inf)
    return elem.reshape(x.shape), block
