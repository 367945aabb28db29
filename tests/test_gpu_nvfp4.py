"""NVFP4 experts on the GPU against the oracle ("SGLang and Miles Add Day-0 Support for
Muse Spark Open", section "NVFP4 as a third MMA kind"; "The NVFP4 requantization
reciprocal table").

* weight quantiser: codes, block scales and global scales bit-exact (integer output;
  both sides decide in the same FP32 op order);
* stage-wise: the activation quantiser, the block-scaled gate/up GEMM with its SwiGLU +
  requantisation epilogue and the block-scaled down GEMM, each from the GPU's own input;
* end to end against the oracle that dequantises the same NVFP4 weights and emulates
  the activation quantisation, started from the GPU's stored pooled rows (the quantiser's
  input, as in the full-size tests): max|gpu - ref| / rms(ref) <= 3e-2 (the NVFP4 bound).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F
from oracle import nvfp4 as Q
from harness import fix_margins, oracle_view, rel_err, to_np
from latent_moe_layer_rmsnorm_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_NVFP4 = 3e-2
SMALL = synth.Shape("nvfp4_small", T=200, d=1024, p=512, E=8, top_k=4, I=512, expert="nvfp4")
# several 128-row tiles per expert
MID = synth.Shape("nvfp4_mid", T=600, d=1024, p=512, E=8, top_k=4, I=512, expert="nvfp4")
# the decode structure (two rows per expert on average, most 128-row tiles nearly empty)
# at widths the stage-wise oracle handles per expert in seconds
DECODE_LIKE = synth.Shape("nvfp4_decode_like", T=16, d=1024, p=512, E=64, top_k=8, I=512,
                          expert="nvfp4")
# Zipf-skewed routing: empty experts, experts of one row and experts of several tiles in
# one call (T x k = 4096 < 256 x E: one-CTA kernels; the pair test forces pairs)
SKEWED = synth.Shape("nvfp4_skewed", T=1024, d=1024, p=512, E=32, top_k=4, I=512,
                     expert="nvfp4", zipf_s=1.2)


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from latent_moe_layer_rmsnorm_gb300 import build
    build.build()


def unchunk_sf(sf: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Chunked scale layout (see latent_moe.h) -> [rows, K/16]."""
    r = np.arange(rows)[:, None]
    g = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4
    return sf[off]


def unpack_codes(b: np.ndarray) -> np.ndarray:
    """[rows, K/2] bytes -> [rows, K] E2M1 codes (even element in the low nibble)."""
    out = np.empty((b.shape[0], b.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = b & 15
    out[:, 1::2] = b >> 4
    return out


def w13_row_map(I: int) -> np.ndarray:
    """Packed gate/up row -> row of [gate; up] (interleaved in blocks of 64)."""
    r = np.arange(2 * I)
    b, i = r // 128, r % 128
    return np.where(i < 64, b * 64 + i, I + b * 64 + (i - 64))


def build(shape, seed):
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    inp = synth.make_inputs(shape, seed=seed, device="cpu")
    fix_margins(inp, shape, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    return inp, dev, LatentMoE(shape, dev, out="f32")


def test_weight_quantizer_bit_exact():
    need_gpu()
    shape = SMALL
    inp, dev, layer = build(shape, 0)
    torch.cuda.synchronize()
    E, I, p = shape.E, shape.I, shape.p
    codes13 = layer.w13.cpu().numpy().reshape(E, 2 * I, p // 2)
    sf13 = layer.sf13.cpu().numpy()
    codes2 = layer.w2.cpu().numpy().reshape(E, p, I // 2)
    sf2 = layer.sf2.cpu().numpy()
    gs13, gs2 = layer.gs13.cpu().numpy(), layer.gs2.cpu().numpy()
    view = oracle_view(inp)
    rmap = w13_row_map(I)
    sf13_rows = unchunk_sf(sf13, E * 2 * I, p).reshape(E, 2 * I, p // 16)
    sf2_rows = unchunk_sf(sf2, E * p, I).reshape(E, p, I // 16)
    for e in range(E):
        ref = oracle.nvfp4_expert_weights(view["w_gate"][e], view["w_up"][e], view["w_down"][e])
        assert gs13[e] == ref["g13"] and gs2[e] == ref["g2"], e
        np.testing.assert_array_equal(unpack_codes(codes13[e]), ref["q13"][rmap])
        np.testing.assert_array_equal(sf13_rows[e], ref["sf13"][rmap])
        np.testing.assert_array_equal(unpack_codes(codes2[e]), ref["q2"])
        np.testing.assert_array_equal(sf2_rows[e], ref["sf2"])


# E2M1 rounding decisions in units of the block scale: the seven midpoints (ties go to
# the even code) and values 2^-5 (relative) to either side of them, then the block maximum.
SWEEP_M = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0,
           0.25 * (1 + 2 ** -5), 0.75 * (1 - 2 ** -5), 1.25 * (1 + 2 ** -5),
           1.75 * (1 - 2 ** -5), 2.5 * (1 + 2 ** -5), 3.5 * (1 - 2 ** -5), 5.0 * (1 + 2 ** -5)]
# block scales (UE4M3 values; the powers of two keep every element exact in BF16, so the
# midpoints are exact ties), including the largest (448) that fixes the tensor's amax
SWEEP_S = [448.0, 2.0 ** -6, 2.0 ** -3, 0.5, 1.0, 2.0, 8.0, 64.0, 1.5, 3.75, 26.0, 0.0]


def sweep_matrix(rows: int, K: int, seed: int) -> torch.Tensor:
    """A [rows, K] BF16 weight whose 16-element blocks sit on E2M1 rounding boundaries:
    with beta = 2^-8 (tensor amax 6 * 448 * 2^-8 = 10.5, in the first block), a block
    of scale S holds 6 * S * beta and then m * S * beta for m in SWEEP_M, signs and
    order shuffled per block (S = 0: an all-zero block)."""
    rng = np.random.default_rng(seed)
    beta = 2.0 ** -8
    out = np.zeros((rows, K), np.float64)
    nb = K // 16
    for r in range(rows):
        for b in range(nb):
            S = SWEEP_S[(r * nb + b) % len(SWEEP_S)] if (r, b) != (0, 0) else 448.0
            vals = np.array([6.0] + SWEEP_M + [6.0 * (1 - 2 ** -6)]) * S * beta
            vals = vals[rng.permutation(16)] * rng.choice([-1.0, 1.0], 16)
            out[r, 16 * b:16 * b + 16] = vals
    return torch.from_numpy(out).to(torch.bfloat16)


def test_quantizer_rounding_sweep_bit_exact():
    """The device encoder (shared by the weight quantiser, the activation quantiser and
    the SwiGLU requantisation) against the oracle's on exact E2M1 ties, values just past
    them, block scales across the UE4M3 range and all-zero blocks: codes, block scales
    and global scales bit for bit."""
    need_gpu()
    shape = SMALL
    E, I, p = shape.E, shape.I, shape.p
    inp = synth.make_inputs(shape, seed=0, device="cpu")
    for e in range(E):
        inp["w_gate"][e] = sweep_matrix(I, p, 100 + e)
        inp["w_up"][e] = sweep_matrix(I, p, 200 + e)
        inp["w_down"][e] = sweep_matrix(p, I, 300 + e)
    from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
    dev = {k: v.cuda() for k, v in inp.items()}
    layer = LatentMoE(shape, dev, out="f32")
    torch.cuda.synchronize()
    codes13 = layer.w13.cpu().numpy().reshape(E, 2 * I, p // 2)
    sf13 = unchunk_sf(layer.sf13.cpu().numpy(), E * 2 * I, p).reshape(E, 2 * I, p // 16)
    codes2 = layer.w2.cpu().numpy().reshape(E, p, I // 2)
    sf2 = unchunk_sf(layer.sf2.cpu().numpy(), E * p, I).reshape(E, p, I // 16)
    gs13, gs2 = layer.gs13.cpu().numpy(), layer.gs2.cpu().numpy()
    view = oracle_view(inp)
    rmap = w13_row_map(I)
    ties = 0
    for e in range(E):
        ref = oracle.nvfp4_expert_weights(view["w_gate"][e], view["w_up"][e], view["w_down"][e])
        assert gs13[e] == ref["g13"] == np.float32(2.0 ** -8), e
        assert gs2[e] == ref["g2"] == np.float32(2.0 ** -8), e
        np.testing.assert_array_equal(unpack_codes(codes13[e]), ref["q13"][rmap])
        np.testing.assert_array_equal(sf13[e], ref["sf13"][rmap])
        np.testing.assert_array_equal(unpack_codes(codes2[e]), ref["q2"])
        np.testing.assert_array_equal(sf2[e], ref["sf2"])
        # the sweep really lands on ties: codes of exact midpoints are even
        mags = np.abs(view["w_down"][e]).reshape(p, I // 16, 16)
        blk = mags.max(axis=2, keepdims=True)
        rel = np.where(blk > 0, mags / np.where(blk > 0, blk, 1) * 6.0, 0)
        ties += int(np.isin(rel, [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]).sum())
    assert ties > 0


@pytest.mark.parametrize("shape", [SMALL, MID, DECODE_LIKE, SKEWED], ids=lambda s: s.name)
def test_nvfp4_stages_and_layer(shape):
    need_gpu()
    inp, dev, layer = build(shape, 1)
    T, k, E, I, p = shape.T, shape.top_k, shape.E, shape.I, shape.p
    out = layer.forward(dev["x"])
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    view = oracle_view(inp)
    ref = oracle.moe_forward(view, top_k=k, eps=shape.eps, act="bf16", expert="nvfp4",
                             out="f32", return_parts=True)
    ids = layer.intermediate("ids", T).cpu().numpy()
    np.testing.assert_array_equal(ids, ref["ids"])
    row_off = layer.intermediate("row_off", T).cpu().numpy().astype(np.int64)
    row_cnt = layer.intermediate("row_cnt", T).cpu().numpy().astype(np.int64)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    np.testing.assert_array_equal(row_cnt[:E], counts)
    assert np.all(row_off[:E] % 128 == 0)                   # 128-aligned expert rows
    inv = layer.intermediate("inv", T).cpu().numpy().astype(np.int64).reshape(T, k)
    pooled = to_np(layer.intermediate("pooled", T))
    R = 128 * ((T * k + 127) // 128 + E)

    # activation quantiser, from the GPU's pooled rows
    u_codes = unpack_codes(layer.intermediate("a_perm", T).cpu().numpy())
    sf_u = unchunk_sf(layer.intermediate("sf_u", T).cpu().numpy(), R, p)
    alpha = to_np(layer.intermediate("alpha", T))
    u32 = F.fp32(oracle.rmsnorm(pooled, view["g_pool"], shape.eps))
    qu, sfu, al = Q.quantize_rows(u32)
    rows_t = inv.reshape(-1)
    tok = np.repeat(np.arange(T), k)
    np.testing.assert_allclose(alpha[rows_t], al[tok], rtol=2e-6)
    deq_gpu = Q.dequantize(u_codes[rows_t], sf_u[rows_t], alpha[rows_t])
    deq_ref = Q.dequantize(qu[tok], sfu[tok], al[tok])
    code_match = float(np.mean(u_codes[rows_t] == qu[tok]))
    # a value near a rounding boundary may land one E2M1 step (<= 2 x scale) away, and a
    # block maximum near a UE4M3 boundary may change its block's scale by one step (1/8)
    scale = np.maximum(F.ue4m3_decode(sfu[tok]), F.ue4m3_decode(sf_u[rows_t]))
    step = scale.repeat(16, axis=1) * al[tok][:, None] * 2.0
    assert np.all(np.abs(deq_gpu - deq_ref) <= step * (1 + 1e-6) + 0.13 * np.abs(deq_ref))
    assert code_match > 0.99, code_match

    # gate/up GEMM + SwiGLU + requantisation, from the GPU's own u
    s_codes = unpack_codes(layer.intermediate("s", T).cpu().numpy())
    sf_s = unchunk_sf(layer.intermediate("sf_s", T).cpu().numpy(), R, I)
    y = to_np(layer.intermediate("y", T))
    gs_act2 = view["gs_act2"]
    s_match, s_total, y_err, y_flips, y_n = 0, 0, 0.0, 0, 0
    for e in range(E):
        rows = np.arange(row_off[e], row_off[e] + row_cnt[e])
        if len(rows) == 0:
            continue
        wq = oracle.nvfp4_expert_weights(view["w_gate"][e], view["w_up"][e], view["w_down"][e])
        u_deq = Q.dequantize(u_codes[rows], sf_u[rows], alpha[rows])
        s_ref = F.fp32(oracle.expert_swiglu(u_deq, wq["gate"], wq["up"]))
        qs, sfs = Q.quantize_static(s_ref, gs_act2[e])
        s_match += int(np.sum(s_codes[rows] == qs))
        s_total += qs.size
        d_gpu = Q.dequantize(s_codes[rows], sf_s[rows], np.float32(gs_act2[e]))
        d_ref = Q.dequantize(qs, sfs, np.float32(gs_act2[e]))
        stp = np.maximum(F.ue4m3_decode(sfs), F.ue4m3_decode(sf_s[rows])).repeat(16, axis=1)
        assert np.all(np.abs(d_gpu - d_ref)
                      <= 2.0 * stp * gs_act2[e] * (1 + 1e-6) + 0.13 * np.abs(d_ref) + 1e-12)
        # down GEMM, from the GPU's own s; y is stored in FP16: equal to the rounded exact
        # sum, or one FP16 unit away where FP32 accumulation crossed a rounding boundary
        y_exact = oracle.expert_down(d_gpu, wq["down"])
        y_ref = F.fp16(y_exact)
        d = np.abs(y[rows] - y_ref)
        mag = np.maximum(np.maximum(np.abs(y[rows]), np.abs(y_ref)), 1e-30)
        one = np.maximum(np.exp2(np.floor(np.log2(mag)) - 10), 2.0 ** -24)
        floor = 3e-5 * float(np.sqrt(np.mean(y_exact * y_exact)))
        assert np.all(d <= one * (1 + 1e-9) + floor), (e, float(d.max()))
        y_flips += int(np.sum(d > 0))
        y_n += d.size
        y_err = max(y_err, rel_err(y[rows], y_exact))
    assert s_match / s_total > 0.97, s_match / s_total
    assert y_flips / y_n <= 0.01, y_flips / y_n

    # end to end from the GPU's stored pooled rows (the activation codes are decided from
    # them; the oracle's own pooled rows differ by the pooler's FP32 accumulation noise,
    # which can tip a code at a rounding midpoint: the error from x is printed beside)
    ref_p = oracle.moe_forward(view, top_k=k, eps=shape.eps, act="bf16", expert="nvfp4",
                               out="f32", pooled=pooled)
    e2e = rel_err(to_np(out), ref_p)
    e2e_x = rel_err(to_np(out), ref["out"])
    print(f"nvfp4 {shape.name}: u codes {code_match:.4f} equal, s codes "
          f"{s_match / s_total:.4f} equal, y {y_err:.1e}, end to end {e2e:.2e} "
          f"(from x {e2e_x:.2e})")
    assert e2e <= TOL_NVFP4


@pytest.mark.parametrize("shape", [SMALL, MID, DECODE_LIKE, SKEWED], ids=lambda s: s.name)
def test_pair_kernel_matches_one_cta_kernel(shape):
    """The CTA-pair NVFP4 GEMMs (MOE_FLAG_NVFP4_PAIR: 256 x 256 tiles, each CTA staging
    half of the weight tile) against the one-CTA kernels (MOE_FLAG_NVFP4_ONE_CTA) on the
    same inputs: requantised SwiGLU codes and scales, expert outputs and the layer
    output; the default choice (one CTA for gate/up, pairs for the down GEMM once the
    experts average 256 rows) gives the same output.  The shapes give experts with an
    odd number of 128-row blocks, whose last pair tile has rows in one CTA only, and
    (decode-like) experts of one or two rows."""
    need_gpu()
    from latent_moe_layer_rmsnorm_gb300 import _lib as L
    inp, dev, layer = build(shape, 2)
    T, I = shape.T, shape.I
    x = dev["x"]
    auto = layer.forward(x).clone()
    one = layer.forward(x, flags=L.MOE_FLAG_NVFP4_ONE_CTA).clone()
    s_one = layer.intermediate("s", T)
    sf_one = layer.intermediate("sf_s", T)
    y_one = layer.intermediate("y", T)
    pair = layer.forward(x, flags=L.MOE_FLAG_NVFP4_PAIR).clone()
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    row_off = layer.intermediate("row_off", T).cpu().numpy().astype(np.int64)
    row_cnt = layer.intermediate("row_cnt", T).cpu().numpy().astype(np.int64)
    rows = np.concatenate([np.arange(row_off[e], row_off[e] + row_cnt[e])
                           for e in range(shape.E)]).astype(np.int64)
    odd = int(np.sum(((row_cnt[:shape.E] + 127) // 128) % 2 == 1))
    s_pair, y_pair = layer.intermediate("s", T), layer.intermediate("y", T)
    rs = torch.as_tensor(rows)
    same_s = torch.equal(s_pair[rs], s_one[rs])
    same_y = torch.equal(y_pair[rs], y_one[rs])
    sf_rows_idx = unchunk_sf(np.arange(len(sf_one)), 128 * ((T * shape.top_k + 127) // 128 + shape.E),
                             I)[rows].reshape(-1)
    same_sf = np.array_equal(layer.intermediate("sf_s", T).cpu().numpy()[sf_rows_idx],
                             sf_one.cpu().numpy()[sf_rows_idx])
    err = rel_err(to_np(pair), to_np(one))
    print(f"pair vs one-CTA ({shape.name}, {odd} experts with an odd block count): s codes "
          f"{'equal' if same_s else 'differ'}, scales {'equal' if same_sf else 'differ'}, y "
          f"{'equal' if same_y else 'differs'}, out {err:.1e}")
    # same operands, same K order per output element: the pair MMA gives the same sums
    assert same_s and same_sf and same_y
    assert torch.equal(pair, one)
    assert torch.equal(auto, one)


def test_nvfp4_rows_do_not_depend_on_the_batch():
    """NVFP4 experts keep the block's row independence bit for bit: each token's
    activation scale, codes and expert products are its own, so a single-token call (one
    row per expert: the one-CTA down GEMM storing rows directly) and a permuted batch
    (other tile placements) give the batch rows (T x k = 2400 >= 256 x E: the down GEMM
    on CTA pairs) exactly."""
    need_gpu()
    shape = MID
    inp, dev, layer = build(shape, 5)
    x = dev["x"]
    full = layer.forward(x).clone()
    perm = torch.randperm(shape.T, generator=torch.Generator().manual_seed(3)).cuda()
    permuted = layer.forward(x[perm].contiguous()).clone()
    singles = [layer.forward(x[t:t + 1].contiguous()).clone() for t in (0, 77, shape.T - 1)]
    torch.cuda.synchronize()
    assert layer.read_status() == (0, 0)
    assert torch.equal(permuted, full[perm])
    for one, t in zip(singles, (0, 77, shape.T - 1)):
        assert torch.equal(one[0], full[t]), t
