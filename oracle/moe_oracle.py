"""CPU oracle of the latent mixture-of-experts block, in float64.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  The library never does, and
this module imports nothing from the library.

What it computes is the plain definition of the block, taken from "SGLang and Miles
Add Day-0 Support for Muse Spark Open", section "MoE with Pooler, Unpooler and
Per-Expert Normalization", with the widths of "vLLM 对 Muse Spark Open 的 Day 0 支持" (vLLM Day-0 support for Muse Spark Open),
section "潜空间 MoE", and the router precision of the same page's "Nvidia" section:

    h_t   = RMSNorm_{g_in}(x_t)                       full-width norm
    l_t   = W_r h_t                                   router logits (TF32 operands)
    (e_t, w_t) = top-k of softmax(l_t), renormalised   k experts, weights sum to 1
    u_t   = RMSNorm_{g_pool}(W_pool h_t)              pooler 8192->4096, then the
                                                      pooled-input norm
    y_tj  = W_down_e (silu(W_gate_e u_t) * W_up_e u_t) routed SwiGLU expert e = e_tj
    c_t   = sum_j w_tj * RMSNorm_{g_exp[e_tj]}(y_tj)   per-expert norm BEFORE the
                                                      weighting, sum in order j
    out_t = W_unpool c_t                              unpooler 4096->8192

with RMSNorm_g(v) = v / sqrt(mean(v^2) + eps) * g and silu(a) = a * sigmoid(a).

Dispatching tokens to experts and running grouped GEMMs reaches exactly this
per-token result (up to rounding order), so the oracle computes it token by
token with dense float64 products (numpy matmul as the only library step) and
no blocking, fusion or reordering.

Two modes:
* chain=False ("exact"): float64 throughout.  Router operands are still rounded
  to TF32 (ties away), because the page fixes a TF32 router GEMM fed by the
  norm's FP32 output, and the routing decision must be taken in the precision
  the kernel uses.
* chain=True ("precision chain", the parity gate): float64 arithmetic, with every
  value rounded where the GPU path stores it (see `storage_kinds`): h (FP32 for
  the router; FP16, or TF32 in FP32 mode, for the pooler), pooled (FP32), u and c
  (FP16 / TF32), s (FP16 / TF32), y (FP16, FP32 for FP32 experts: the values the fused
  post-per-expert norm squares) and out; the weights meet the GEMMs in the same formats
  (FP16 copies of the pooler, gate/up, down and unpooler weights).  The page fixes the
  FP32 norm and route-weighted sum; the storage types are the kernel's.

Readings of points the pages leave open (each is also listed with the design
notes): softmax over all E logits, top-k, renormalised (= softmax over the k
chosen logits); slots ordered by logit, ties to the lower expert id; no biases;
every norm has a learned gain; per-expert gains are [E, p]; eps inside the
square root.

NVFP4 experts (block-scaled FP4, "NVFP4 as a third MMA kind") are emulated in
`nvfp4.py`.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import nvfp4 as Q


# ---- storage rounding --------------------------------------------------------------

def _store(v: np.ndarray, kind: str) -> np.ndarray:
    """Round float64 values to the storage format `kind` of the GPU path."""
    if kind == "f64":
        return v
    if kind == "f32":
        return F.fp32(v)
    if kind == "bf16":
        return F.bf16(v)
    if kind == "f16":
        return F.fp16(v)
    if kind == "tf32":          # FP32 storage, pre-rounded for a TF32 MMA operand
        return F.tf32_rna(F.fp32(v))
    raise ValueError(kind)


store = _store


def as_f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---- the steps ---------------------------------------------------------------------

def rmsnorm(v: np.ndarray, g, eps: float) -> np.ndarray:
    """Row-wise RMSNorm with gain: v / sqrt(mean(v^2) + eps) * g."""
    v = as_f64(v)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * as_f64(g)


def router_logits(h: np.ndarray, w_router) -> np.ndarray:
    """logits[t, e] = sum_i tf32(h[t, i]) * tf32(W_r[e, i]).

    "vLLM 对 Muse Spark Open 的 Day 0 支持", section "Nvidia": the router GEMM is TF32, fed by the
    norm's FP32 output.  h is first stored as FP32, then both operands are
    rounded to TF32; products and the sum are float64.
    """
    a = F.tf32_rna(F.fp32(h))
    b = F.tf32_rna(as_f64(w_router))
    return a @ b.T


def topk_route(logits: np.ndarray, k: int):
    """Top-k experts per row and their renormalised softmax weights.

    Slots are ordered by logit, largest first; equal logits go to the lower id.
    softmax over all E followed by renormalisation over the chosen k equals the
    softmax over the chosen logits, which is what is computed here.
    """
    logits = as_f64(logits)
    order = np.argsort(-logits, axis=-1, kind="stable")
    ids = order[:, :k]
    chosen = np.take_along_axis(logits, ids, axis=-1)
    z = np.exp(chosen - chosen[:, :1])
    w = z / np.sum(z, axis=-1, keepdims=True)
    return ids.astype(np.int32), w


def route_margin(logits: np.ndarray, k: int) -> np.ndarray:
    """Smallest gap between consecutive sorted logits among the top min(k+1, E).

    A row whose margin exceeds the routing noise has a unique top-k set and a
    unique slot order.
    """
    s = -np.sort(-as_f64(logits), axis=-1)
    m = min(k + 1, s.shape[-1])
    if m < 2:
        return np.full(s.shape[0], np.inf)
    return np.min(s[:, : m - 1] - s[:, 1:m], axis=-1)


def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def expert_swiglu(u: np.ndarray, w_gate_e, w_up_e) -> np.ndarray:
    """s = silu(W_gate u) * W_up u for rows u [n, p]; W_gate, W_up are [I, p]."""
    a = u @ as_f64(w_gate_e).T
    b = u @ as_f64(w_up_e).T
    return silu(a) * b


def expert_down(s: np.ndarray, w_down_e) -> np.ndarray:
    """y = W_down s for rows s [n, I]; W_down is [p, I]."""
    return s @ as_f64(w_down_e).T


def pool(h: np.ndarray, w_pool) -> np.ndarray:
    """pooled = W_pool h for rows h [n, d]; W_pool is [p, d] (the pooler, 8192 -> 4096)."""
    return as_f64(h) @ as_f64(w_pool).T


def unpool(c: np.ndarray, w_unpool) -> np.ndarray:
    """out = W_unpool c for rows c [n, p]; W_unpool is [d, p] (the unpooler)."""
    return as_f64(c) @ as_f64(w_unpool).T


def combine(y: np.ndarray, ids: np.ndarray, wts: np.ndarray, g_exp, eps: float) -> np.ndarray:
    """c_t = sum_j w_tj * RMSNorm_{g_exp[e_tj]}(y_tj), summed in slot order j = 0..k-1.

    y is [n, k, p] (slot j of token t = output of expert ids[t, j]).  Each expert
    output is normalised with its own gain before the weighting (the page's
    per-expert RMSNorm before the routing-weighted sum).
    """
    g_exp = as_f64(g_exp)
    n, k, p = y.shape
    c = np.zeros((n, p))
    for j in range(k):
        c = c + as_f64(wts)[:, j: j + 1] * rmsnorm(y[:, j], g_exp[np.asarray(ids)[:, j]], eps)
    return c


# ---- between two blocks ----------------------------------------------------------------

def boundary(x: np.ndarray, y: np.ndarray, g_post, g_next, eps: float, gate=None,
             act: str = "bf16"):
    """What follows the block in the decoder: the sandwich post-norm, the residual add and
    the next block's pre-norm ("vLLM 对 Muse Spark Open 的 Day 0 支持", section "三明治归一化":
    x + post_norm(F(norm(x))); "SGLang and Miles Add Day-0 Support for Muse Spark Open",
    section "Kernel Optimizations": post-FFN norm, gated residual add and pre-attention
    norm form one elementwise chain).

        a_t  = RMSNorm_{g_post}(y_t)            y = the block's output F(norm(x))
        x'_t = x_t + gate * a_t                 gate per channel; None = plain residual
        h'_t = RMSNorm_{g_next}(x'_t)           on x' as stored in the residual stream

    The pages name the residual "gated" without giving the gate's form; a per-channel
    gate vector is the reading taken (None gives the plain residual of the sandwich
    form).  x' and h' are stored in the residual-stream format `act` ("bf16", "f32" or
    "f64" for no rounding); returns (x', h') as float64 arrays.
    """
    a = rmsnorm(y, g_post, eps)
    if gate is not None:
        a = a * as_f64(gate)
    xn = _store(as_f64(x) + a, act)
    hn = _store(rmsnorm(xn, g_next, eps), act)
    return xn, hn


# ---- the layer ---------------------------------------------------------------------

def storage_kinds(act: str, expert: str, out: str, chain: bool) -> dict:
    """Where the GPU path stores each intermediate, as `_store` kinds."""
    if not chain:
        return dict(h_pool="f64", pooled="f64", u="f64", s="f64", y="f64", c="f64",
                    out="f64", w_proj="f64", w_gate_up="f64", w_down="f64")
    tc = act == "f32"            # FP32 activations run their GEMMs on TF32 operands
    te = expert == "f32"
    # BF16 configurations store every activation between the GEMMs (h, u, s, y, c) in
    # FP16 and meet FP16 copies of the weights (exact for |w| >= 2^-17).  The pages fix
    # the per-expert norm and the weighted sum in FP32 but not the format the expert
    # outputs y wait in before them: FP16 (FP32 for FP32 experts), normalised from the
    # stored values.
    return dict(
        h_pool="tf32" if tc else "f16",
        pooled="f32",
        u="tf32" if te else "f16",
        s="tf32" if te else "f16",
        y="f32" if te else "f16",             # expert outputs, the per-expert norm's input
        c="tf32" if tc else "f16",
        out=out,
        w_proj="tf32" if tc else "f16",
        w_gate_up="tf32" if te else "f16",
        w_down="tf32" if te else "f16",
    )


def nvfp4_expert_weights(w_gate_e, w_up_e, w_down_e):
    """Quantise one expert as the library does: gate and up share one global scale
    (they form one gate/up matrix), down has its own.  Returns dequantised float64
    matrices and the quantised codes."""
    gu = np.concatenate([as_f64(w_gate_e), as_f64(w_up_e)], axis=0).astype(np.float32)
    g13 = Q.global_scale(np.max(np.abs(gu)))
    q13, sf13 = Q.quantize_blocks(gu, g13)
    d13 = Q.dequantize(q13, sf13, g13)
    I = d13.shape[0] // 2
    q2, sf2, g2 = Q.quantize_tensor(as_f64(w_down_e))
    return dict(gate=d13[:I], up=d13[I:], down=Q.dequantize(q2, sf2, g2), q13=q13, sf13=sf13,
                g13=g13, q2=q2, sf2=sf2, g2=g2)


def nvfp4_expert_rows(u_rows: np.ndarray, wq: dict, gamma: float) -> dict:
    """One NVFP4 expert on its dispatched rows ("SGLang and Miles Add Day-0 Support for
    Muse Spark Open", section "NVFP4 as a third MMA kind").

    u_rows are the stored (dequantised) NVFP4 activations, so the per-token scale is
    already inside them: a and b are the first GEMM's accumulators times that scale
    and the weights' shared W13 scale (both carried by the dequantised operands).
        s     = fp32(silu(a) * b),  a = W_gate u, b = W_up u
        s_q   = NVFP4 of s with the static global scale gamma (scale codes per 16)
        y     = fp16(W_down s_q)   (W_down dequantised with its own global scale)
    Returns s (FP32 values before the requantisation), its codes qs / scale codes sfs,
    the dequantised s_deq and y.
    """
    s = F.fp32(expert_swiglu(u_rows, wq["gate"], wq["up"]))
    qs, sfs = Q.quantize_static(s, gamma)
    s_deq = Q.dequantize(qs, sfs, np.float32(gamma))
    y = F.fp16(expert_down(s_deq, wq["down"]))
    return dict(s=s, qs=qs, sfs=sfs, s_deq=s_deq, y=y)


def nvfp4_expert(w_gate_e, w_up_e, w_down_e, u_rows, gamma) -> dict:
    """nvfp4_expert_rows with expert e's weights quantised by nvfp4_expert_weights."""
    return nvfp4_expert_rows(u_rows, nvfp4_expert_weights(w_gate_e, w_up_e, w_down_e), gamma)


def chain_expert(w_gate_e, w_up_e, w_down_e, u_rows, st: dict) -> dict:
    """One BF16 / FP32 expert on its rows, rounded where the GPU path stores values:
    s = store(silu(W_gate u) * W_up u), y = store(W_down s) (storage kinds `st`)."""
    wg = _store(as_f64(w_gate_e), st["w_gate_up"])
    wu = _store(as_f64(w_up_e), st["w_gate_up"])
    wd = _store(as_f64(w_down_e), st["w_down"])
    s = _store(expert_swiglu(u_rows, wg, wu), st["s"])
    return dict(s=s, y=_store(expert_down(s, wd), st["y"]))


def moe_forward(inp: dict, *, top_k: int, eps: float, act: str = "bf16",
                expert: str = "bf16", out: str = "f32", chain: bool = True,
                tokens=None, ids=None, weights=None, norm_after_sum: bool = False,
                return_parts: bool = False, expert_map=None, pooled=None):
    """The latent-MoE block for the rows `tokens` of inp["x"] (all rows if None).

    inp holds x [T,d], g_in [d], w_router [E,d], w_pool [p,d], g_pool [p],
    w_gate/w_up [E,I,p], w_down [E,p,I], g_exp [E,p], w_unpool [d,p]; expert
    tensors only need to support w[e] (one expert at a time is converted).
    `ids`/`weights` ([n,k]) replace the router when given (routing replay).
    `norm_after_sum=True` computes the variant that normalises the combined vector
    instead of each expert output, which the page rules out; it exists so tests
    can show the two orders differ.
    Returns out [n, d] (float64 holding values of the output storage type), or a
    dict of every intermediate with return_parts.

    expert="nvfp4": expert weights are quantised to NVFP4 (nvfp4.py) and used
    dequantised; the expert input u is quantised per token on the fly and the SwiGLU
    output s is requantised with the static per-expert global scale inp["gs_act2"][e]
    (the page gives no rule for that scale; see the design notes), as the kernels do.

    expert_map (optional) evaluates the per-expert step elsewhere (e.g. in worker
    processes): it receives a list of tasks (e, u_rows, arg) and must return, in the
    same order, what `chain_expert(w_gate[e], w_up[e], w_down[e], u_rows, arg)` (or,
    for NVFP4 experts, `nvfp4_expert(..., u_rows, arg)`) returns for expert e's
    weights.  It only decides where the step runs; None runs it here on inp's weights.

    pooled (NVFP4 experts only, optional): the pooler's FP32 output rows [n, p] to start
    the expert chain from, instead of computing them from x: a stage-wise comparison
    starts each stage from the stored input of that stage.  Routing still comes from x.
    """
    if expert == "nvfp4":
        return _forward_nvfp4(inp, top_k=top_k, eps=eps, out=out, tokens=tokens, ids=ids,
                              weights=weights, return_parts=return_parts,
                              expert_map=expert_map, pooled=pooled)
    st = storage_kinds(act, expert, out, chain)
    x = as_f64(inp["x"])
    if tokens is not None:
        x = x[np.asarray(tokens)]
    n = x.shape[0]

    h = rmsnorm(x, inp["g_in"], eps)
    if ids is None:
        logits = router_logits(h, inp["w_router"])
        ids, wts = topk_route(logits, top_k)
    else:
        logits = None
        ids = np.asarray(ids, dtype=np.int32)
        wts = as_f64(weights)
        top_k = ids.shape[1]

    h_pool = _store(F.fp32(h) if chain else h, st["h_pool"])
    w_pool = _store(as_f64(inp["w_pool"]), st["w_proj"])
    pooled = _store(pool(h_pool, w_pool), st["pooled"])
    u = _store(rmsnorm(pooled, inp["g_pool"], eps), st["u"])

    p = u.shape[1]
    g_exp = as_f64(inp["g_exp"])
    experts = [int(e) for e in np.unique(ids)]
    tasks = [(e, u[np.nonzero(ids == e)[0]], st) for e in experts]
    if expert_map is None:
        results = [chain_expert(inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e], ur, a)
                   for e, ur, a in tasks]
    else:
        results = expert_map(tasks)
    y_all = np.zeros((n, top_k, p))
    s_all = None
    for e, r in zip(experts, results):
        rows, slots = np.nonzero(ids == e)
        if return_parts:
            if s_all is None:
                s_all = np.zeros((n, top_k, r["s"].shape[1]))
            s_all[rows, slots] = r["s"]
        y_all[rows, slots] = r["y"]

    if not norm_after_sum:
        c = combine(y_all, ids, wts, g_exp, eps)
    else:
        c = np.zeros((n, p))
        for j in range(top_k):
            c = c + wts[:, j: j + 1] * y_all[:, j]
        c = rmsnorm(c, np.ones(p), eps)
    c = _store(c, st["c"])
    w_unpool = _store(as_f64(inp["w_unpool"]), st["w_proj"])
    res = _store(unpool(c, w_unpool), st["out"])
    if not return_parts:
        return res
    return dict(out=res, h=h, logits=logits, ids=ids, w=wts, pooled=pooled, u=u,
                s=s_all, y=y_all, c=c)


def route(inp: dict, *, top_k: int, eps: float, tokens=None):
    """Router only: (ids [n,k] int32, weights [n,k] float64, logits [n,E])."""
    x = as_f64(inp["x"])
    if tokens is not None:
        x = x[np.asarray(tokens)]
    logits = router_logits(rmsnorm(x, inp["g_in"], eps), inp["w_router"])
    ids, w = topk_route(logits, top_k)
    return ids, w, logits


def expert_input(inp: dict, *, eps: float, tokens=None, h=None):
    """The NVFP4 experts' input before quantisation, on the BF16 chain: h = RMSNorm(x),
    stored FP16 for the pooler; pooled = W_pool h (FP16 weights), stored FP32; u32 =
    RMSNorm_{g_pool}(pooled) rounded to FP32, the value the activation quantiser reads.
    Returns (h, pooled, u32) for the rows `tokens` (all if None); h may be given."""
    st = storage_kinds("bf16", "bf16", "f32", True)
    if h is None:
        x = as_f64(inp["x"])
        if tokens is not None:
            x = x[np.asarray(tokens)]
        h = rmsnorm(x, inp["g_in"], eps)
    h_pool = _store(F.fp32(h), st["h_pool"])
    pooled = _store(pool(h_pool, _store(as_f64(inp["w_pool"]), st["w_proj"])), st["pooled"])
    return h, pooled, F.fp32(rmsnorm(pooled, inp["g_pool"], eps))


def _forward_nvfp4(inp, *, top_k, eps, out, tokens, ids, weights, return_parts,
                   expert_map=None, pooled=None):
    """The block with NVFP4 experts; storage points as in the BF16 chain except the
    expert operands: u and s are NVFP4 (u quantised from its FP32 value with a per-token
    scale, s with the static per-expert scale inp["gs_act2"]); y FP16."""
    st = storage_kinds("bf16", "bf16", out, True)
    x = as_f64(inp["x"])
    if tokens is not None:
        x = x[np.asarray(tokens)]
    n = x.shape[0]
    h = rmsnorm(x, inp["g_in"], eps)
    if ids is None:
        ids, wts = topk_route(router_logits(h, inp["w_router"]), top_k)
    else:
        ids = np.asarray(ids, dtype=np.int32)
        wts = as_f64(weights)
        top_k = ids.shape[1]
    if pooled is None:
        _, pooled, u32 = expert_input(inp, eps=eps, h=h)
    else:
        pooled = F.fp32(as_f64(pooled))
        u32 = F.fp32(rmsnorm(pooled, inp["g_pool"], eps))
    qu, sfu, alpha = Q.quantize_rows(u32)
    u = Q.dequantize(qu, sfu, alpha)
    p = u.shape[1]
    gs2 = as_f64(inp["gs_act2"])
    experts = [int(e) for e in np.unique(ids)]
    tasks = [(e, u[np.nonzero(ids == e)[0]], float(gs2[e])) for e in experts]
    if expert_map is None:
        results = [nvfp4_expert(inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e], ur, g)
                   for e, ur, g in tasks]
    else:
        results = expert_map(tasks)
    y_all = np.zeros((n, top_k, p))
    s_all = qs_all = sfs_all = None
    for e, r in zip(experts, results):
        rows, slots = np.nonzero(ids == e)
        if return_parts:
            if s_all is None:
                I = r["s"].shape[1]
                s_all = np.zeros((n, top_k, I))
                qs_all = np.zeros((n, top_k, I), dtype=np.uint8)
                sfs_all = np.zeros((n, top_k, I // Q.BLOCK), dtype=np.uint8)
            s_all[rows, slots] = r["s"]
            qs_all[rows, slots] = r["qs"]
            sfs_all[rows, slots] = r["sfs"]
        y_all[rows, slots] = r["y"]
    c = _store(combine(y_all, ids, wts, inp["g_exp"], eps), st["c"])
    res = _store(unpool(c, _store(as_f64(inp["w_unpool"]), st["w_proj"])), st["out"])
    if not return_parts:
        return res
    return dict(out=res, h=h, ids=ids, w=wts, pooled=pooled, u32=u32, qu=qu, sfu=sfu, u=u,
                alpha=alpha, s=s_all, qs=qs_all, sfs=sfs_all, y=y_all, c=c)
