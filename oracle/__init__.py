"""CPU float64 oracle of the latent-MoE block (test infrastructure only).

Only `tests/`, the package smoke check and the benchmark's CPU-baseline leg may
import this package; the library never does.
"""
from .moe_oracle import (moe_forward, route, rmsnorm, router_logits, topk_route,
                         route_margin, expert_swiglu, expert_down, silu, pool, unpool,
                         combine, storage_kinds, store, nvfp4_expert_weights,
                         nvfp4_expert_rows, nvfp4_expert, chain_expert, expert_input,
                         boundary)
from . import formats
from . import nvfp4

__all__ = ["moe_forward", "route", "rmsnorm", "router_logits", "topk_route",
           "route_margin", "expert_swiglu", "expert_down", "silu", "pool", "unpool",
           "combine", "storage_kinds", "store", "formats", "nvfp4", "nvfp4_expert_weights",
           "nvfp4_expert_rows", "nvfp4_expert", "chain_expert", "expert_input",
           "boundary"]
