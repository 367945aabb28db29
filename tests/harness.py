"""Helpers shared by the tests: numpy views of generated inputs and margin repair.

The oracle gets numpy arrays; generated tensors (BF16 or FP32, CPU or GPU) are
widened to FP32 (exact) before the oracle sees them.  Expert tensors are wrapped
so that only the experts the oracle touches are copied to the host.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from latent_moe_layer_rmsnorm_gb300 import synth


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float32).cpu().numpy()


class LazyExperts:
    """w[e] -> numpy FP32 copy of one expert's matrix, copied to the host on demand
    (nothing is cached: the full expert set can be tens of GB)."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __getitem__(self, e):
        return to_np(self.t[int(e)])

    def __len__(self):
        return self.t.shape[0]


EXPERT_KEYS = ("w_gate", "w_up", "w_down")


def oracle_view(inp: dict, lazy: bool = False) -> dict:
    out = {}
    for k, v in inp.items():
        if not isinstance(v, torch.Tensor):
            continue
        if k in EXPERT_KEYS and lazy:
            out[k] = LazyExperts(v)
        else:
            out[k] = to_np(v)
    return out


def oracle_kwargs(shape: synth.Shape, out: str = "f32") -> dict:
    return dict(top_k=shape.top_k, eps=shape.eps, act=shape.act, expert=shape.expert,
                out=out)


def fix_margins(inp: dict, shape: synth.Shape, seed: int, min_gap: float = 1e-3,
                max_rounds: int = 50) -> int:
    """Redraw tokens whose top-(k+1) router logits are closer than min_gap.

    The gaps are measured on the oracle's logits (TF32 operands, float64 sums), so
    every remaining token has a unique expert set and slot order with margin to
    spare over FP32 accumulation noise.  Returns the number of redraws.
    """
    redraws = 0
    w_router = to_np(inp["w_router"])
    g_in = to_np(inp["g_in"])
    rows = np.arange(shape.T)
    for r in range(max_rounds):
        x = to_np(inp["x"][torch.as_tensor(rows, device=inp["x"].device)])
        h = oracle.rmsnorm(x, g_in, shape.eps)
        logits = oracle.router_logits(h, w_router)
        bad = rows[oracle.route_margin(logits, shape.top_k) < min_gap]
        if len(bad) == 0:
            return redraws
        synth.redraw_rows(inp["x"], bad, seed=seed * 1000003 + 7 * r + 1, shape=shape,
                          base_seed=seed)
        redraws += len(bad)
        rows = bad
    raise RuntimeError("router margins could not be repaired")


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max |gpu - ref| / rms(ref)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(gpu - ref)) / max(rms, 1e-300))


# ---- full-size inputs --------------------------------------------------------------------
# Expert matrices are drawn on the CPU one expert at a time with the generator's
# per-expert recipe (the draw the oracle's worker processes repeat) and kept on the GPU
# for the session: the full-size tests share one expert set per (seed, widths, dtype).
_EXPERTS = {}


def gpu_experts(shape: synth.Shape, seed: int) -> dict:
    key = (seed, shape.E, shape.p, shape.I, synth.storage_dtype(shape.expert))
    if key not in _EXPERTS:
        _EXPERTS.clear()
        torch.cuda.empty_cache()
        dt = synth.storage_dtype(shape.expert)
        E, p, I = shape.E, shape.p, shape.I
        out = {"w_gate": torch.empty((E, I, p), dtype=dt, device="cuda"),
               "w_up": torch.empty((E, I, p), dtype=dt, device="cuda"),
               "w_down": torch.empty((E, p, I), dtype=dt, device="cuda")}
        for e in range(E):
            m = synth.make_expert(shape, seed, e, "cpu")
            for k in out:
                out[k][e].copy_(m[k])
        _EXPERTS[key] = out
    return _EXPERTS[key]


def fullsize_inputs(shape: synth.Shape, seed: int, expert_seed: int = 0):
    """(host inputs without the expert matrices, device inputs with them).  The dense
    inputs are drawn on the CPU and their router margins repaired there; the experts
    come from gpu_experts(shape, expert_seed)."""
    host = synth.make_dense(shape, seed, "cpu")
    fix_margins(host, shape, seed=seed)
    if shape.expert == "nvfp4":
        host["gs_act2"] = synth.nvfp4_act2_scales(shape, "cpu")
    dev = {k: v.cuda() for k, v in host.items()}
    dev.update(gpu_experts(shape, expert_seed))
    return host, dev
