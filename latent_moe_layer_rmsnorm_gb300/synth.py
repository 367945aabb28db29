"""Seeded synthetic inputs for the latent-MoE layer.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic (no norm, routing, projection or activation).  Both the CUDA
path and the CPU oracle take their inputs from here, so the two never share any
step of the computation.

Workloads follow the MoE-block description of "SGLang and Miles Add Day-0 Support
for Muse Spark Open" (section "MoE with Pooler, Unpooler and Per-Expert
Normalization") and the dimensions of "vLLM 对 Muse Spark Open 的 Day 0 支持" (vLLM Day-0 support for Muse Spark Open) (section
"潜空间 MoE": pooler 8192 x 4096, 256 experts per layer):

* activations x ~ N(0, 1)
* every weight ~ N(0, std = 1/sqrt(fan_in)), fan_in = the reduction width
  (d for router and pooler, p for gate/up and unpooler, I for down)
* RMSNorm gains ~ U(0.5, 1.5)
* router weights are FP32; the other tensors are stored in the workload's
  activation/weight dtype (values drawn in FP32, then rounded once).

All tensors are canonical (un-packed) and row-major:
  x [T,d], g_in [d], w_router [E,d], w_pool [p,d], g_pool [p],
  w_gate [E,I,p], w_up [E,I,p], w_down [E,p,I], g_exp [E,p], w_unpool [d,p].
Gains are always returned as FP32 tensors (holding values of the storage dtype).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Shape:
    """Dimensions and dtypes of one latent-MoE workload."""
    name: str
    T: int          # tokens
    d: int          # model width
    p: int          # pooled (expert) width
    E: int          # routed experts
    top_k: int      # experts per token
    I: int          # SwiGLU intermediate width
    act: str = "bf16"      # "bf16" or "f32": storage of x / projections
    expert: str = "bf16"   # "bf16", "f32" (TF32 MMA) or "nvfp4"
    eps: float = 1e-6
    zipf_s: float = 0.0    # > 0: skewed routing (Zipf exponent of the expert offsets)

    def replace(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


# The five workloads.  T=16384 is one 16K prefill chunk (the SGLang page's
# sequence-parallel prefill measurement); d/p/E/I are the decoder's layer sizes.
TINY_F32 = Shape("tiny_f32", T=64, d=256, p=128, E=8, top_k=2, I=256,
                 act="f32", expert="f32")
PREFILL_BF16 = Shape("prefill_bf16", T=16384, d=8192, p=4096, E=256, top_k=8, I=4096)
DECODE_BF16 = Shape("decode_bf16", T=64, d=8192, p=4096, E=256, top_k=8, I=4096)
PREFILL_NVFP4 = Shape("prefill_nvfp4", T=16384, d=8192, p=4096, E=256, top_k=8, I=4096,
                      expert="nvfp4")
SKEWED_BF16 = Shape("skewed_bf16", T=8192, d=8192, p=4096, E=256, top_k=8, I=4096,
                    zipf_s=1.2)

# A 1/16 slice of the prefill chunk with the same per-expert load (512 rows per expert)
# and widths: small enough (~2 GB on the device) for full profiler captures.
PREFILL_SLICE_BF16 = Shape("prefill_slice_bf16", T=1024, d=8192, p=4096, E=16, top_k=8,
                           I=4096)

PREFILL_SLICE_NVFP4 = PREFILL_SLICE_BF16.replace(name="prefill_slice_nvfp4", expert="nvfp4")
# A 1/8 slice (512 rows per expert as well) whose expert outputs (16384 rows x 8 KB =
# 134 MB) exceed L2, for captures of the memory-bound kernels between the GEMMs.
PREFILL_EIGHTH_BF16 = Shape("prefill_eighth_bf16", T=2048, d=8192, p=4096, E=32, top_k=8,
                            I=4096)
# The block boundary on 4096 full-width rows (x, the block output, x' and h': 256 MB in
# all) with narrow experts, for captures of moe_boundary.
BOUNDARY_BF16 = Shape("boundary_bf16", T=4096, d=8192, p=256, E=8, top_k=2, I=256)
# Decode with NVFP4 experts: the weight stream is 4.5 bits per weight instead of 16.
DECODE_NVFP4 = DECODE_BF16.replace(name="decode_nvfp4", expert="nvfp4")
# Decode with narrow experts (I = 256): the norm, router, pooler, dispatch, combine and
# unpooler see exactly the decode batch's shapes, with ~1.7 GB on the device, for full
# profiler captures of those kernels.
DECODE_SLICE_BF16 = DECODE_BF16.replace(name="decode_slice_bf16", I=256)

WORKLOADS = {s.name: s for s in (TINY_F32, PREFILL_BF16, DECODE_BF16, PREFILL_NVFP4,
                                 SKEWED_BF16, PREFILL_SLICE_BF16, PREFILL_SLICE_NVFP4,
                                 DECODE_NVFP4, PREFILL_EIGHTH_BF16, BOUNDARY_BF16,
                                 DECODE_SLICE_BF16)}


def storage_dtype(kind: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32, "nvfp4": torch.bfloat16}[kind]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


_STREAM_IDS = {"x": 1, "g_in": 2, "w_router": 3, "w_pool": 4, "g_pool": 5, "w_gate": 6,
               "w_up": 7, "w_down": 8, "g_exp": 9, "w_unpool": 10}


def _stream_seed(seed: int, name: str, expert: int = 0) -> int:
    """Independent seed per (workload seed, tensor, expert): any tensor or expert can be
    drawn on its own, in any order."""
    return (int(seed) * 1000003 + _STREAM_IDS[name] * 65537 + expert * 257) % (1 << 62)


def _normal(shape, std, gen, device, out_dtype):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(out_dtype)


def _uniform_gain(shape, gen, device, store_dtype):
    t = torch.rand(shape, generator=gen, device=device, dtype=torch.float32) + 0.5
    # round to the storage dtype, then hold it in FP32 (the library takes FP32 gains)
    return t.to(store_dtype).to(torch.float32)


def make_expert(shape: Shape, seed: int, e: int, device="cpu") -> dict:
    """Gate, up and down matrices of expert e: [I,p], [I,p], [p,I]."""
    exp = storage_dtype(shape.expert)
    p, I = shape.p, shape.I
    return {
        "w_gate": _normal((I, p), 1.0 / math.sqrt(p), _gen(_stream_seed(seed, "w_gate", e), device),
                          device, exp),
        "w_up": _normal((I, p), 1.0 / math.sqrt(p), _gen(_stream_seed(seed, "w_up", e), device),
                        device, exp),
        "w_down": _normal((p, I), 1.0 / math.sqrt(I), _gen(_stream_seed(seed, "w_down", e), device),
                          device, exp),
    }


def make_dense(shape: Shape, seed: int = 0, device="cpu") -> dict:
    """Every input except the expert matrices."""
    act = storage_dtype(shape.act)
    T, d, p, E = shape.T, shape.d, shape.p, shape.E
    g = lambda name: _gen(_stream_seed(seed, name), device)  # noqa: E731
    out = {
        "x": _normal((T, d), 1.0, g("x"), device, act),
        "g_in": _uniform_gain((d,), g("g_in"), device, act),
        "w_router": _normal((E, d), 1.0 / math.sqrt(d), g("w_router"), device, torch.float32),
        "w_pool": _normal((p, d), 1.0 / math.sqrt(d), g("w_pool"), device, act),
        "g_pool": _uniform_gain((p,), g("g_pool"), device, act),
        "g_exp": _uniform_gain((E, p), g("g_exp"), device, act),
        "w_unpool": _normal((d, p), 1.0 / math.sqrt(p), g("w_unpool"), device, act),
    }
    if shape.zipf_s > 0:
        apply_zipf_skew(out, shape, seed)
    return out


# Static global scale of the requantised SwiGLU output s for NVFP4 experts, one per
# expert.  The pages give no rule for it (a per-token scale would need a row maximum
# across all output tiles of the gate/up GEMM); a static calibrated scale is the usual
# choice.  For these inputs |s| stays far below 64, so g = 64 / (6 * 448) keeps every
# block scale inside the UE4M3 range without saturating.
NVFP4_S_AMAX = 64.0


def nvfp4_act2_scales(shape: Shape, device="cpu") -> torch.Tensor:
    return torch.full((shape.E,), NVFP4_S_AMAX / 2688.0, dtype=torch.float32, device=device)


def make_inputs(shape: Shape, seed: int = 0, device="cpu") -> dict:
    """Draw every input of one layer call.  Deterministic for (shape, seed, device).

    Expert tensors are drawn one expert at a time, so the FP32 staging buffer stays
    one expert large even for the 24 GB expert weight set.
    """
    out = make_dense(shape, seed, device)
    exp = storage_dtype(shape.expert)
    E, p, I = shape.E, shape.p, shape.I
    w_gate = torch.empty((E, I, p), dtype=exp, device=device)
    w_up = torch.empty((E, I, p), dtype=exp, device=device)
    w_down = torch.empty((E, p, I), dtype=exp, device=device)
    for e in range(E):
        m = make_expert(shape, seed, e, device)
        w_gate[e], w_up[e], w_down[e] = m["w_gate"], m["w_up"], m["w_down"]
    out["w_gate"], out["w_up"], out["w_down"] = w_gate, w_up, w_down
    if shape.expert == "nvfp4":
        out["gs_act2"] = nvfp4_act2_scales(shape, device)
    return out


def redraw_rows(x: torch.Tensor, rows, seed: int, shape: Shape | None = None,
                base_seed: int = 0) -> None:
    """Replace the listed rows of x with fresh N(0,1) draws (in place).

    Used to resample tokens whose router margins are too small for an
    index-exact comparison; which rows is decided by the caller.  For a skewed
    workload (shape.zipf_s > 0) the fresh rows get the same shared-direction mixing
    as the originals (base_seed = the seed the inputs were made with).
    """
    if len(rows) == 0:
        return
    gen = _gen(seed, x.device)
    idx = torch.as_tensor(list(rows), dtype=torch.long, device=x.device)
    fresh = torch.randn((len(rows), x.shape[1]), generator=gen, device=x.device,
                        dtype=torch.float32)
    if shape is not None and shape.zipf_s > 0:
        v = _skew_direction(shape.d, base_seed, x.device)
        fresh = (fresh + SKEW_BETA * v) / math.sqrt(1.0 + SKEW_BETA * SKEW_BETA)
    x[idx] = fresh.to(x.dtype)


def zipf_offsets(E: int, s: float, strength: float, seed: int) -> torch.Tensor:
    """Per-expert logit offsets b_e = -strength * s * ln(rank_e), FP32 on the CPU.

    rank_e (1..E) is a seeded permutation, so the popular experts are scattered
    over the id range.  strength scales the whole Zipf profile.
    """
    gen = _gen(seed + 7919, "cpu")
    ranks = torch.randperm(E, generator=gen).to(torch.float64) + 1.0
    return (-strength * s * torch.log(ranks)).to(torch.float32)


# Strength of the Zipf profile for the skewed workload: with it the busiest expert
# gets about 20x the mean load at T=8192, E=256, k=8 (19.8x, 18 % of experts empty on
# the CPU-drawn inputs); the achieved load profile is measured and reported with every
# run rather than assumed.
SKEW_STRENGTH = 0.35
SKEW_BETA = 1.0


def _skew_direction(d: int, seed: int, device) -> torch.Tensor:
    gen = _gen(seed * 7 + 104729, device)
    return (torch.randint(0, 2, (d,), generator=gen, device=device, dtype=torch.int32) * 2 - 1
            ).to(torch.float32)


def apply_zipf_skew(inp: dict, shape: Shape, seed: int, strength: float = SKEW_STRENGTH,
                    beta: float = SKEW_BETA) -> torch.Tensor:
    """Realise a per-expert router offset through the data (the layer has no router bias).

    A shared direction v (entries +-1) is mixed into every token,
    x_t <- (x_t + beta*v) / sqrt(1 + beta^2), and router row e gets
    b_e * v / (v . v) added, so the router sees roughly b_e extra logit for
    expert e on every token.  Returns the offsets b.
    """
    device = inp["x"].device
    d = shape.d
    v = _skew_direction(d, seed, device)
    x = inp["x"].to(torch.float32)
    x = (x + beta * v) / math.sqrt(1.0 + beta * beta)
    inp["x"] = x.to(inp["x"].dtype)
    b = zipf_offsets(shape.E, shape.zipf_s, strength, seed).to(device)
    # the router sees h = rmsnorm(x) * g_in, so v is pre-divided by g_in and by its
    # share of the normalised row (beta / sqrt(1+beta^2))
    vg = v / inp["g_in"]
    scale = math.sqrt(1.0 + beta * beta) / beta / float((v * v).sum())
    inp["w_router"] = (inp["w_router"] + scale * b[:, None] * vg[None, :]).to(torch.float32)
    return b
