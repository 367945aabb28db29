"""NVFP4 experts at the full workload sizes against the oracle that quantises the same
weights itself and dequantises them ("SGLang and Miles Add Day-0 Support for Muse Spark
Open", section "NVFP4 as a third MMA kind").

* decode batch (T=64, d=8192, p=4096, E=256, k=8, I=4096): every token in full;
* prefill chunk (T=16384): ids of all tokens exactly, and 64 sampled tokens in full,
  spread over the batch plus tokens of the busiest and the rarest expert.

Both check, bit for bit, the GPU's quantised weights of every routed expert against
the oracle's own quantiser (a digest in the library's layout, tests/oracle_pool.py).

Where the comparison starts.  Quantising decides integer codes, and the first codes
(the per-token activation quantisation) are decided from u = RMSNorm(W_pool h), whose
FP32 value the GPU's pooler GEMM reaches with tensor-core accumulation noise: measured
up to 1.1e-4 of the rms of the pooled rows over d = 8192 products.  Quantising the GPU's
own pooled rows with the oracle reproduces every activation code the GPU chose (0
differences measured), while quantising the oracle's pooled rows flips a few codes that
sit within that noise of a rounding midpoint; one such flip moves every expert output of
its token (about 4e-2 of rms at the output).  Both results are correct quantisations of
the pooled rows, so the test compares what is unique at each stage:
  1. x -> pooled: the GPU's stored pooled rows against the oracle's, within the FP32
     accumulation bound TOL_POOLED (and the routing: ids exactly);
  2. pooled -> out: the oracle's NVFP4 chain started from the GPU's stored pooled rows
     (moe_forward(..., pooled=...)): activation codes, block scales and per-token scales
     bit for bit; each requantised SwiGLU code that differs must sit within EPS_S_VALID
     of its row's rms of a rounding midpoint (the gate/up GEMM's accumulation noise); and
     max|gpu - ref| / rms(ref) <= 3e-2 over all outputs of the compared tokens.
The end-to-end error against the oracle started from x is printed beside them.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pool
from oracle import formats as F
from oracle import nvfp4 as Q
from harness import fullsize_inputs, oracle_view, rel_err, to_np
from latent_moe_layer_rmsnorm_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_NVFP4 = 3e-2
EXPERT_SEED = 0
# FP32 accumulation of d = 8192 FP16 products on the tensor cores, relative to the rms of
# the pooled rows: measured 5.2e-5 (decode, split K) and 1.1e-4 (prefill)
TOL_POOLED = 5e-4
# A requantised SwiGLU code may differ from the oracle's only where the oracle's value
# is this close (relative to the rms of its row) to a rounding midpoint: the gate/up
# GEMM's FP32 accumulation (K = 4096) and the FP32 SwiGLU arithmetic stay below it.
EPS_S_VALID = 1e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    build.build()


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
    ids = layer.intermediate("ids", T).cpu().numpy()
    # stage 1: x -> pooled
    pooled = to_np(layer.intermediate("pooled", T))[tok]
    _, pooled_ref, _ = oracle.expert_input(view, eps=shape.eps, tokens=tok)
    pool_noise = rel_err(pooled, pooled_ref)
    # stage 2: pooled -> out, the oracle started from the GPU's pooled rows
    emap = oracle_pool.ExpertMap(shape, EXPERT_SEED, digest=True)
    ref = oracle.moe_forward(view, top_k=k, eps=shape.eps, act="bf16", expert="nvfp4",
                             out="f32", tokens=tok, return_parts=True, expert_map=emap,
                             pooled=pooled)
    np.testing.assert_array_equal(ids[tok], ref["ids"])
    for e, dg in sorted(emap.digests.items()):
        assert oracle_pool.gpu_nvfp4_digest(layer, e) == dg, f"weights of expert {e}"
    inv = layer.intermediate("inv", T).cpu().numpy().astype(np.int64).reshape(T, k)[tok]
    rows = inv.reshape(-1)
    tok_of_row = np.repeat(np.arange(len(tok)), k)
    u_codes = unpack_codes(layer.intermediate("a_perm", T).cpu().numpy()[rows])
    u_flip = F.e2m1_decode(u_codes) != F.e2m1_decode(ref["qu"][tok_of_row])
    sfu_gpu = sf_rows(layer.intermediate("sf_u", T).cpu().numpy(), rows, p)
    alpha = to_np(layer.intermediate("alpha", T))[rows]
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
    worst_s = max(float(np.max((blk / rms_s)[blk_flip], initial=0.0)),
                  float(np.max((elem / rms_s)[code_flip], initial=0.0)))
    # end to end over every output of the compared tokens
    got = to_np(out[torch.as_tensor(tok, device=out.device)])
    err = rel_err(got, ref["out"])
    per_tok = np.max(np.abs(got - ref["out"]), axis=1) / np.sqrt(np.mean(ref["out"] ** 2))
    worst = int(np.argmax(per_tok))
    # the same tokens against the oracle started from x (printed, not a gate)
    ref_x = oracle.moe_forward(view, top_k=k, eps=shape.eps, act="bf16", expert="nvfp4",
                               out="f32", tokens=tok, expert_map=emap)
    err_x = rel_err(got, ref_x)
    print(f"{label}: {len(tok)} tokens, {len(emap.digests)} experts' weights equal; pooled "
          f"{pool_noise:.1e} of rms; u codes {int(u_flip.sum())} of {u_flip.size} differ; "
          f"s codes {int(code_flip.sum())} and block scales {int(blk_flip.sum())} differ of "
          f"{s_gpu.size} (largest margin {worst_s:.1e} of rms); end to end {err:.2e} "
          f"(worst token {tok[worst]}: {per_tok[worst]:.2e}, median {np.median(per_tok):.2e}); "
          f"from x {err_x:.2e}")
    assert pool_noise <= TOL_POOLED
    assert not u_flip.any()
    np.testing.assert_array_equal(sfu_gpu, ref["sfu"][tok_of_row])
    np.testing.assert_allclose(alpha, ref["alpha"][tok_of_row], rtol=1e-6)
    assert worst_s < EPS_S_VALID
    assert err <= TOL_NVFP4


def test_nvfp4_decode_full():
    """All 64 decode tokens."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    shape = synth.DECODE_NVFP4
    host, dev = fullsize_inputs(shape, 21, EXPERT_SEED)
    layer = LatentMoE(shape, dev, out="f32", keep_canonical=False)
    out = layer.forward(dev["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    ids = layer.intermediate("ids", shape.T).cpu().numpy()
    rid, _, _ = oracle.route(oracle_view(host), top_k=shape.top_k, eps=shape.eps)
    np.testing.assert_array_equal(ids, rid)
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
    tb = np.nonzero((ids == busiest).any(1))[0]
    tr = np.nonzero((ids == rarest).any(1))[0]
    tok = set(np.linspace(0, T - 1, 64).round().astype(int).tolist())
    tok |= set(tb[[0, -1]].tolist()) | set(tr[[0, -1]].tolist())
    check_layer(layer, host, shape, out, sorted(tok), "nvfp4 prefill")
