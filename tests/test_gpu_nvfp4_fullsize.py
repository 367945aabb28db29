"""NVFP4 experts at the full workload sizes against the oracle that quantises the same
weights itself and dequantises them ("SGLang and Miles Add Day-0 Support for Muse Spark
Open", section "NVFP4 as a third MMA kind").

* decode batch (T=64, d=8192, p=4096, E=256, k=8, I=4096): every token in full;
* prefill chunk (T=16384): ids of all tokens exactly, and 64 sampled tokens in full,
  spread over the batch plus tokens of the busiest and the rarest expert.

Both check, bit for bit, the GPU's quantised weights of every routed expert against
the oracle's quantiser (a digest in the library's layout, tests/oracle_pool.py), the
activation codes, block scales and per-token scales of the compared tokens, and that
every requantised SwiGLU code that differs from the oracle's sits at a rounding
decision the FP32 accumulation noise can tip.  Bound: max|gpu - ref| / rms(ref) <=
3e-2 over all outputs of the compared tokens.

Unique decisions.  Quantising decides integer codes from FP32 values that the GPU and
the oracle compute with different rounding (the pooler GEMM's FP32 accumulation, the
norm's FP32 arithmetic), so, like the router's top-k, a code is only a unique result
when its value is not within that noise of a rounding midpoint.  One activation code
flipped by the noise moves a token's u by up to a third of its block maximum, and
every expert output of the token with it (about 4e-2 of rms at the output).  So, as the
router ids are compared on tokens whose top-k gaps exceed 1e-3, the outputs are
compared on tokens whose activation quantisation decisions are all at least EPS_U (of
the row's rms) from a midpoint: decode tokens closer than that are redrawn, prefill
tokens closer than that are not sampled.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pool
from oracle import formats as F
from oracle import nvfp4 as Q
from harness import fix_margins, fullsize_inputs, gpu_experts, oracle_view, rel_err, to_np
from latent_moe_layer_rmsnorm_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_NVFP4 = 3e-2
EXPERT_SEED = 0
# Distance (relative to the rms of the token's u row) that every activation rounding
# decision of a compared token keeps from its midpoint.  It bounds the difference
# between the GPU's and the oracle's FP32 u: the pooler GEMM's FP32 accumulation over
# d = 8192 products and the norm's FP32 arithmetic, measured far below it.
EPS_U = 2e-5
# A requantised SwiGLU code may differ from the oracle's only where the oracle's value
# is this close (relative to the rms of its row) to a rounding midpoint: the gate/up
# GEMM's FP32 accumulation (K = 4096) and the FP32 SwiGLU arithmetic stay below it.
EPS_S_VALID = 1e-4


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    build.build()


def u_margin(u32: np.ndarray) -> np.ndarray:
    """Per token: the smallest distance of an activation rounding decision from its
    midpoint, relative to the rms of the token's u row."""
    _, _, alpha = Q.quantize_rows(u32)
    elem, blk = Q.decision_margins(u32, alpha)
    rms = np.sqrt(np.mean(u32.astype(np.float64) ** 2, axis=1))
    return np.minimum(elem.min(axis=1), blk.min(axis=1)) / np.maximum(rms, 1e-30)


def unpack_codes(b: np.ndarray) -> np.ndarray:
    out = np.empty((b.shape[0], b.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = b & 15
    out[:, 1::2] = b >> 4
    return out


def sf_rows(sf: np.ndarray, rows: np.ndarray, K: int) -> np.ndarray:
    """Scale codes [len(rows), K/16] of the given rows from the chunked layout."""
    r = np.asarray(rows, dtype=np.int64)[:, None]
    g = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4
    return sf[off]


def check_layer(layer, host, shape, out, tok, label):
    """Compare the tokens `tok` of a finished NVFP4 forward with the oracle."""
    T, k, p, I = shape.T, shape.top_k, shape.p, shape.I
    view = oracle_view(host)
    emap = oracle_pool.ExpertMap(shape, EXPERT_SEED, digest=True)
    ref = oracle.moe_forward(view, top_k=k, eps=shape.eps, act="bf16", expert="nvfp4",
                             out="f32", tokens=tok, return_parts=True, expert_map=emap)
    ids = layer.intermediate("ids", T).cpu().numpy()
    np.testing.assert_array_equal(ids[tok], ref["ids"])
    # quantised weights of every routed expert, bit for bit
    for e, dg in sorted(emap.digests.items()):
        assert oracle_pool.gpu_nvfp4_digest(layer, e) == dg, f"weights of expert {e}"
    # pooled rows: only the FP32 accumulation order differs
    pooled = to_np(layer.intermediate("pooled", T))[tok]
    pool_noise = float(np.max(np.abs(pooled - ref["pooled"])) /
                       np.sqrt(np.mean(ref["pooled"] ** 2)))
    # activation codes, block scales and per-token scales of every dispatched row
    inv = layer.intermediate("inv", T).cpu().numpy().astype(np.int64).reshape(T, k)[tok]
    rows = inv.reshape(-1)
    tok_of_row = np.repeat(np.arange(len(tok)), k)
    a_perm = layer.intermediate("a_perm", T).cpu().numpy()
    u_codes = unpack_codes(a_perm[rows])
    u_flip = F.e2m1_decode(u_codes) != F.e2m1_decode(ref["qu"][tok_of_row])
    sfu_gpu = sf_rows(layer.intermediate("sf_u", T).cpu().numpy(), rows, p)
    alpha = to_np(layer.intermediate("alpha", T))[rows]
    a_rel = float(np.max(np.abs(alpha - ref["alpha"][tok_of_row]) / ref["alpha"][tok_of_row]))
    print(f"{label}: pooled noise {pool_noise:.1e} of rms; u codes {int(u_flip.sum())} of "
          f"{u_flip.size} differ, {int(np.sum(sfu_gpu != ref['sfu'][tok_of_row]))} block "
          f"scales differ; per-token scales within {a_rel:.1e}")
    assert not u_flip.any()
    np.testing.assert_array_equal(sfu_gpu, ref["sfu"][tok_of_row])
    np.testing.assert_allclose(alpha, ref["alpha"][tok_of_row], rtol=1e-6)
    # requantised SwiGLU codes: equal, or at a decision the noise can tip
    s_gpu = F.e2m1_decode(unpack_codes(layer.intermediate("s", T).cpu().numpy()[rows]))
    sfs_gpu = sf_rows(layer.intermediate("sf_s", T).cpu().numpy(), rows, I)
    s_ref = ref["s"].reshape(-1, I)
    qs_ref = F.e2m1_decode(ref["qs"].reshape(-1, I))
    sfs_ref = ref["sfs"].reshape(-1, I // 16)
    gam = view["gs_act2"][ref["ids"].reshape(-1)]
    elem, blk = Q.decision_margins(s_ref, gam)
    rms_s = np.sqrt(np.mean(s_ref ** 2, axis=1, keepdims=True))
    blk_flip = sfs_gpu != sfs_ref
    code_flip = (s_gpu != qs_ref) & ~np.repeat(blk_flip, 16, axis=1)
    assert np.all(blk[blk_flip] < EPS_S_VALID * rms_s.repeat(I // 16, axis=1)[blk_flip])
    assert np.all(elem[code_flip] < EPS_S_VALID * rms_s.repeat(I, axis=1)[code_flip])
    near = int(np.sum(elem < EPS_S_VALID * rms_s))
    # end to end, every output of the compared tokens
    got = to_np(out[torch.as_tensor(tok, device=out.device)])
    err = rel_err(got, ref["out"])
    per_tok = np.max(np.abs(got - ref["out"]), axis=1) / np.sqrt(np.mean(ref["out"] ** 2))
    worst = int(np.argmax(per_tok))
    print(f"{label}: {len(tok)} tokens, {len(emap.digests)} experts' weights equal; pooled "
          f"noise {pool_noise:.1e} of rms; s codes: {int(code_flip.sum())} flipped, "
          f"{int(blk_flip.sum())} block scales flipped, of {s_gpu.size} ({near} oracle "
          f"values within {EPS_S_VALID:g} rms of a midpoint); end to end {err:.2e} "
          f"(worst token {tok[worst]}: {per_tok[worst]:.2e}, median "
          f"{np.median(per_tok):.2e})")
    assert err <= TOL_NVFP4


def test_nvfp4_decode_full():
    """All 64 decode tokens; tokens whose activation quantisation is within EPS_U of a
    rounding midpoint are redrawn first, as tokens with close router logits are."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.DECODE_NVFP4
    seed = 21
    host = synth.make_dense(shape, seed, "cpu")
    fix_margins(host, shape, seed=seed)
    host["gs_act2"] = synth.nvfp4_act2_scales(shape, "cpu")
    redrawn = 0
    for r in range(40):
        _, _, u32 = oracle.expert_input(oracle_view(host), eps=shape.eps)
        bad = np.nonzero(u_margin(u32) < EPS_U)[0]
        if len(bad) == 0:
            break
        synth.redraw_rows(host["x"], bad.tolist(), seed=seed * 7919 + 31 * r + 1)
        redrawn += len(bad)
        fix_margins(host, shape, seed=seed + 1000 * (r + 1))
    else:
        pytest.fail("activation quantisation margins could not be repaired")
    print(f"decode: {redrawn} token draws replaced for quantisation margins")
    dev = {k: v.cuda() for k, v in host.items()}
    dev.update(gpu_experts(shape, EXPERT_SEED))
    layer = LatentMoE(shape, dev, out="f32", keep_canonical=False)
    out = layer.forward(dev["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    check_layer(layer, host, shape, out, list(range(shape.T)), "nvfp4 decode")


def test_nvfp4_prefill_chunk_sampled():
    """The prefill chunk: ids of all tokens exactly, 64+ tokens in full."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.PREFILL_NVFP4
    host, dev = fullsize_inputs(shape, 23, EXPERT_SEED)
    layer = LatentMoE(shape, dev, out="f32", keep_canonical=False)
    out = layer.forward(dev["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    T = shape.T
    ids = layer.intermediate("ids", T).cpu().numpy()
    h = oracle.rmsnorm(to_np(host["x"]), to_np(host["g_in"]), shape.eps)
    rid, _ = oracle.topk_route(oracle.router_logits(h, to_np(host["w_router"])), shape.top_k)
    del h
    np.testing.assert_array_equal(ids, rid)
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    busiest = int(np.argmax(counts))
    nonempty = np.nonzero(counts)[0]
    rarest = int(nonempty[np.argmin(counts[nonempty])])
    # candidates: 192 spread over the batch, then the busiest and rarest experts' rows
    spread = np.linspace(0, T - 1, 192).round().astype(int).tolist()
    tb = np.nonzero((ids == busiest).any(1))[0][:16].tolist()
    tr = np.nonzero((ids == rarest).any(1))[0][:16].tolist()
    cand = sorted(set(spread + tb + tr))
    _, _, u32 = oracle.expert_input(oracle_view(host), eps=shape.eps, tokens=cand)
    ok = dict(zip(cand, u_margin(u32) >= EPS_U))
    tok = [t for t in spread if ok[t]][:64]
    tok += [t for t in tb if ok[t]][:2] + [t for t in tr if ok[t]][:2]
    tok = sorted(set(tok))
    skipped = sum(1 for t in cand if not ok[t])
    print(f"prefill: {skipped} of {len(cand)} candidate tokens left out for quantisation "
          f"margins")
    assert len(tok) >= 64 and any(t in tok for t in tb) and any(t in tok for t in tr)
    check_layer(layer, host, shape, out, tok, "nvfp4 prefill")
