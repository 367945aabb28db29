"""Pins of the oracle's NVFP4 expert chain (`nvfp4_expert_weights`, `nvfp4_expert_rows`
and the NVFP4 branch of `moe_forward`) against facts that do not come from the oracle.

Source: "SGLang and Miles Add Day-0 Support for Muse Spark Open", section "NVFP4 as a
third MMA kind": dense E2M1 operands, one UE4M3 scale per 16 elements along K, FP32
global scales, the per-token FP32 input scales applied to the first GEMM's
accumulators.  Readings of this library: gate and up share one global scale (one
gate/up matrix), the per-token scale is amax / (6 * 448), and the requantised SwiGLU
output has a static per-expert scale gamma.

* a hand-worked case (tests/golden/nvfp4_hand_worked_k1.json) fixes where the per-token
  scale, the shared W13 scale, gamma and the W2 scale enter, value by value;
* weights already on the NVFP4 grid come back unchanged (shared W13 scale, row layout);
* on inputs that every quantisation represents exactly, the NVFP4 chain equals the BF16
  experts' chain;
* scaling one expert's W_down by 2^k moves only its W2 scale, and the per-expert norm
  cancels it: identical output;
* scaling gamma by 2^k (block scales staying in the normal UE4M3 range) leaves the
  requantised values, and so the output, unchanged.
"""
import json
import os

import numpy as np

import oracle
from oracle import formats as F
from oracle import nvfp4 as Q
from harness import oracle_view
from latent_moe_layer_rmsnorm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def hand_worked():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_hand_worked_k1.json")))
    d = g["dims"]
    n = d["d"]

    def dense(entries, rows, cols):
        m = np.zeros((rows, cols))
        for r, c, v in entries:
            m[r, c] = v
        return m

    inp = {
        "x": np.array(g["x"]), "g_in": np.array(g["g_in"]),
        "w_router": np.ones((1, n)), "w_pool": np.eye(n), "g_pool": np.array(g["g_pool"]),
        "w_gate": dense(g["w_gate_entries"], d["I"], d["p"])[None],
        "w_up": dense(g["w_up_entries"], d["I"], d["p"])[None],
        "w_down": dense(g["w_down_entries"], d["p"], d["I"])[None],
        "g_exp": np.ones((1, d["p"])), "w_unpool": np.eye(n),
        "gs_act2": np.array([g["gamma"]]),
    }
    return g, inp


def test_hand_worked_nvfp4_chain():
    """Every stage of the NVFP4 chain on the hand-worked case."""
    g, inp = hand_worked()
    ex = g["expected"]
    parts = oracle.moe_forward(inp, top_k=1, eps=0.0, act="bf16", expert="nvfp4", out="f32",
                               return_parts=True)
    np.testing.assert_array_equal(parts["ids"], [[0]])
    np.testing.assert_array_equal(parts["w"], [[1.0]])
    # per-token scale: amax / 2688 = 1/448 up to its FP32 rounding; block scale 448
    np.testing.assert_allclose(parts["alpha"] * 448, ex["alpha_times_448"], rtol=1e-7)
    np.testing.assert_array_equal(F.e2m1_decode(parts["qu"][0]), ex["u_codes"])
    np.testing.assert_array_equal(F.ue4m3_decode(parts["sfu"][0]), [ex["u_scale"]])
    # dequantised u carries the per-token scale once: u_deq = codes * 448 * alpha
    np.testing.assert_allclose(parts["u"][0], ex["u_codes"], rtol=1e-7)
    # expert weights: shared W13 scale 2^-6 and W2 scale 2^-4, both exact
    wq = oracle.nvfp4_expert_weights(inp["w_gate"][0], inp["w_up"][0], inp["w_down"][0])
    assert wq["g13"] == ex["g13"] and wq["g2"] == ex["g2"]
    # SwiGLU output before requantisation (FP32): 24 * b, within the FP32 unit that the
    # rounded per-token scale can move it by
    np.testing.assert_allclose(parts["s"][0, 0], ex["s"], rtol=2e-7, atol=0)
    np.testing.assert_array_equal(F.e2m1_decode(parts["qs"][0, 0]), ex["s_codes"])
    np.testing.assert_array_equal(F.ue4m3_decode(parts["sfs"][0, 0]), [ex["s_scale"]])
    # expert output, stored FP16, carries gamma and the W2 scale: exactly +-2016
    np.testing.assert_array_equal(parts["y"][0, 0], ex["y"])
    np.testing.assert_array_equal(parts["out"][0], ex["out"])


def test_hand_worked_requantisation_changes_s():
    """The same case with gamma = 0.35: the block scale of s rounds to 72, the codes stay
    s / 24 and the dequantised s is 1.05 s, so y = fp16(+-2016 * 1.05) = +-2116: the
    down GEMM reads the requantised s, and y is stored in FP16."""
    g, inp = hand_worked()
    var = g["variant_gamma_0_35"]
    inp["gs_act2"] = np.array([var["gamma"]], dtype=np.float32)
    ex = var["expected"]
    parts = oracle.moe_forward(inp, top_k=1, eps=0.0, act="bf16", expert="nvfp4", out="f32",
                               return_parts=True)
    np.testing.assert_array_equal(F.e2m1_decode(parts["qs"][0, 0]), ex["s_codes"])
    np.testing.assert_array_equal(F.ue4m3_decode(parts["sfs"][0, 0]), [ex["s_scale"]])
    np.testing.assert_array_equal(parts["y"][0, 0], ex["y"])
    np.testing.assert_array_equal(parts["out"][0], ex["out"])


def test_hand_worked_scale_placement_is_visible():
    """The hand-worked values change when a scale is applied in the wrong place, so the
    test above constrains each: a per-token scale applied a second time leaves a tiny
    gate input (silu no longer the identity), and dropping gamma from the dequantised s
    multiplies y by 1/gamma."""
    g, inp = hand_worked()
    ex = g["expected"]
    wq = oracle.nvfp4_expert_weights(inp["w_gate"][0], inp["w_up"][0], inp["w_down"][0])
    u = np.array(ex["u_codes"])[None]
    good = oracle.nvfp4_expert_rows(u, wq, g["gamma"])
    np.testing.assert_array_equal(good["y"][0], ex["y"])
    twice = oracle.nvfp4_expert_rows(u / 448.0, wq, g["gamma"])
    assert np.max(np.abs(twice["s"][0] - ex["s"])) > 100
    s_deq_no_gamma = Q.dequantize(good["qs"], good["sfs"], 1.0)
    y_no_gamma = F.fp16(oracle.expert_down(s_deq_no_gamma, wq["down"]))
    np.testing.assert_array_equal(y_no_gamma[0], np.array(ex["y"]) / g["gamma"])


def test_nvfp4_equals_bf16_chain_on_representable_inputs():
    """On the hand-worked inputs every NVFP4 quantisation is exact (u, s and the weights
    on their grids), and the BF16 experts' chain stores the same values exactly (FP16 u,
    s and y): the two chains give the same expert outputs and the same layer output."""
    g, inp = hand_worked()
    a = oracle.moe_forward(inp, top_k=1, eps=0.0, act="bf16", expert="nvfp4", out="f32",
                           return_parts=True)
    b = oracle.moe_forward(inp, top_k=1, eps=0.0, act="bf16", expert="bf16", out="f32",
                           chain=True, return_parts=True)
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["out"], b["out"])


def test_stored_values_lie_on_their_grids():
    """On random inputs the chain stores u and y in their formats: u re-quantises to
    itself with its own per-token scale (it is an NVFP4 value, not the FP32 norm
    output), and y is an FP16 value."""
    shape, view = small_nvfp4(2)
    parts = oracle.moe_forward(view, top_k=2, eps=shape.eps, act="bf16", expert="nvfp4",
                               out="f32", return_parts=True)
    u, alpha = parts["u"], parts["alpha"]
    q, sf = Q.quantize_blocks(u.astype(np.float32), alpha)
    np.testing.assert_array_equal(Q.dequantize(q, sf, alpha), u)
    assert np.mean(u != parts["u32"]) > 0.5
    y = parts["y"]
    np.testing.assert_array_equal(F.fp16(y), y)


def grid_weights(rng, rows, K, beta, top_scale):
    """A matrix already on the NVFP4 grid: codes x UE4M3 block scale x beta, with a
    code-6 element in every non-zero block (so the block maximum is 6 * scale); the
    largest block scale is `top_scale`."""
    codes = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    nb = K // 16
    codes[:, ::16] = rng.choice([7, 15], size=(rows, nb))        # +-6 heads every block
    scales = rng.integers(0x30, 0x70, size=(rows, nb)).astype(np.uint8)
    scales = np.minimum(scales, F.ue4m3_encode(np.array([top_scale]))[0])
    scales[0, 0] = F.ue4m3_encode(np.array([top_scale]))[0]
    return Q.dequantize(codes, scales, beta), codes, scales


def test_grid_weights_come_back_unchanged():
    """Gate and up share one global scale: with the W13 maximum in `up` (block scale
    448) and gate's largest block scale 320, the shared scale is beta exactly and both
    come back unchanged.  Separate scales would give gate a scale of 320/448 * beta,
    which is not exact in FP32, and change its values.  W_down with its own beta2."""
    rng = np.random.default_rng(5)
    I, p = 32, 64
    beta, beta2 = 2.0 ** -9, 2.0 ** -6
    gate, qg, sg = grid_weights(rng, I, p, beta, 320.0)
    up, qu, su = grid_weights(rng, I, p, beta, 448.0)
    down, qd, sd = grid_weights(rng, p, I, beta2, 448.0)
    wq = oracle.nvfp4_expert_weights(gate, up, down)
    assert wq["g13"] == beta and wq["g2"] == beta2
    np.testing.assert_array_equal(wq["gate"], gate)
    np.testing.assert_array_equal(wq["up"], up)
    np.testing.assert_array_equal(wq["down"], down)
    # rows stay in place: [gate; up] codes and scales are the constructed ones
    np.testing.assert_array_equal(F.e2m1_decode(wq["q13"]),
                                  F.e2m1_decode(np.concatenate([qg, qu])))
    np.testing.assert_array_equal(wq["sf13"], np.concatenate([sg, su]))
    np.testing.assert_array_equal(F.e2m1_decode(wq["q2"]), F.e2m1_decode(qd))
    np.testing.assert_array_equal(wq["sf2"], sd)
    # the same matrices with gate scaled separately would not be exact
    g_sep = Q.global_scale(np.max(np.abs(gate)))
    q_sep, s_sep = Q.quantize_blocks(gate.astype(np.float32), np.full(I, g_sep, np.float32))
    assert not np.array_equal(Q.dequantize(q_sep, s_sep, g_sep), gate)


def small_nvfp4(seed=0):
    shape = synth.Shape("q", T=24, d=256, p=128, E=6, top_k=2, I=256, expert="nvfp4")
    return shape, oracle_view(synth.make_inputs(shape, seed=seed))


def test_down_scale_moves_only_beta2_and_cancels():
    """W_down of one expert times 2^3: its E2M1 codes and block scales are unchanged, its
    global scale is 8x, y is 8x (exact in FP16), and the per-expert norm (eps = 0)
    returns identical output."""
    shape, view = small_nvfp4()
    e = int(oracle.route(view, top_k=2, eps=0.0)[0][0, 0])    # an expert that is used
    w1 = oracle.nvfp4_expert_weights(view["w_gate"][e], view["w_up"][e], view["w_down"][e])
    v2 = dict(view)
    v2["w_down"] = view["w_down"].copy()
    v2["w_down"][e] = view["w_down"][e] * 8.0
    w2 = oracle.nvfp4_expert_weights(v2["w_gate"][e], v2["w_up"][e], v2["w_down"][e])
    np.testing.assert_array_equal(w1["q2"], w2["q2"])
    np.testing.assert_array_equal(w1["sf2"], w2["sf2"])
    assert w2["g2"] == 8 * w1["g2"]
    kw = dict(top_k=2, eps=0.0, act="bf16", expert="nvfp4", out="f32", return_parts=True)
    a = oracle.moe_forward(view, **kw)
    b = oracle.moe_forward(v2, **kw)
    used = a["ids"] == e
    assert used.any()
    np.testing.assert_array_equal(b["y"][used], 8 * a["y"][used])
    np.testing.assert_array_equal(b["out"], a["out"])


def test_requant_scale_power_of_two_leaves_output_unchanged():
    """gamma / 2 for every expert doubles each s block's scale code value (the block
    ratios stay inside the normal UE4M3 range, checked), so the E2M1 codes and the
    dequantised s are unchanged, and so is the output.  A chain that quantised with
    gamma but dequantised without it (or the reverse) would fail here."""
    shape, view = small_nvfp4(1)
    kw = dict(top_k=2, eps=shape.eps, act="bf16", expert="nvfp4", out="f32",
              return_parts=True)
    a = oracle.moe_forward(view, **kw)
    gam = view["gs_act2"].astype(np.float64)
    used = np.abs(a["s"]).reshape(-1, 16).max(-1)
    used = used[used > 0]
    ratio = used / (6 * gam.min())
    assert ratio.min() >= 2.0 ** -6 and ratio.max() * 2 <= 448   # normal range, both sides
    v2 = dict(view)
    v2["gs_act2"] = (view["gs_act2"] / 2).astype(np.float32)
    b = oracle.moe_forward(v2, **kw)
    np.testing.assert_array_equal(F.e2m1_decode(a["qs"]), F.e2m1_decode(b["qs"]))
    np.testing.assert_array_equal(F.ue4m3_decode(b["sfs"]), 2 * F.ue4m3_decode(a["sfs"]))
    np.testing.assert_array_equal(b["y"], a["y"])
    np.testing.assert_array_equal(b["out"], a["out"])


def test_decision_margins():
    """The margins name the distance to the nearest decision change: a value just
    below an E2M1 midpoint has a small element margin and crosses it when moved by more
    than that margin; a block whose ratio sits near a UE4M3 midpoint has a small block
    margin."""
    g = np.float32(1.0 / 2688)          # six_g = 1/448: block ratio = 448 * bmax
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 1.0                                   # block max: ratio 448, scale 448
    x[0, 1] = np.float32(1.25 / 6 - 1e-6)           # just under the 1.25 midpoint
    elem, blk = Q.decision_margins(x, np.array([g]))
    assert elem[0, 1] < 2e-6 and elem[0, 2] >= 0.25 / 6 * 0.999
    q0, _ = Q.quantize_blocks(x, np.array([g]))
    x2 = x.copy()
    x2[0, 1] += np.float32(2 * elem[0, 1])
    q1, _ = Q.quantize_blocks(x2, np.array([g]))
    assert q0[0, 1] != q1[0, 1] and np.all(q0[0, 2:] == q1[0, 2:])
    # block ratio 432 sits on the UE4M3 midpoint between 416 and 448
    y = np.zeros((1, 16), np.float32)
    y[0, 0] = np.float32(432.0 / 448)
    _, blk2 = Q.decision_margins(y, np.array([g]))
    assert blk2[0, 0] < 1e-6
    assert blk[0, 0] > 0.03                         # 448 is 16 away from the midpoint 432
