"""The benchmark's byte and FLOP counts for the expert GEMMs, on CPU: the algorithmic
bytes of one launch and which roofline (tensor or HBM) each workload falls under."""
import bench
from latent_moe_layer_rmsnorm_gb300 import synth


def test_gate_up_bytes_of_the_profiled_slice():
    # 16 experts x (4096 x 8192) FP16 W13, 8192 dispatched FP16 rows of 4096 in, 8192 BF16
    # rows of 4096 out: the 1.208 GB counted by hand for the ncu capture of this slice
    s = synth.PREFILL_SLICE_BF16
    b = bench.expert_gemm_bytes(s, 16, s.T)["gemm1_gate_up_swiglu"]
    assert b == 16 * 4096 * 8192 * 2 + 8192 * 4096 * 2 + 8192 * 4096 * 2
    assert abs(b / 1e9 - 1.208) < 1e-3


def test_down_bytes_include_output_rows_and_partials():
    s = synth.PREFILL_SLICE_BF16
    b = bench.expert_gemm_bytes(s, 16, s.T)["gemm2_down"]
    R = s.T * s.top_k
    assert b == 16 * 4096 * 4096 * 2 + R * 4096 * 2 + R * 4096 * 2 + R * 32 * 4
    f = synth.TINY_F32           # FP32 experts: FP32 weights, s and y
    bf = bench.expert_gemm_bytes(f, f.E, f.T)["gemm2_down"]
    Rf = f.T * f.top_k
    assert bf == f.E * f.I * f.p * 4 + Rf * f.I * 4 + Rf * f.p * 4 + Rf * (f.p // 128) * 4


def test_nvfp4_bytes_are_codes_plus_block_scales():
    s = synth.PREFILL_SLICE_NVFP4
    b = bench.expert_gemm_bytes(s, 16, s.T)["gemm1_gate_up_swiglu"]
    R = s.T * s.top_k
    per_elem = 0.5 + 1 / 16
    assert b == (16 * 4096 * 8192 + R * 4096 + R * 4096) * per_elem


def _intensity(shape, touched):
    fl = bench.flops_per_token(shape)["gemm1_gate_up_swiglu"] * shape.T
    return fl / bench.expert_gemm_bytes(shape, touched, shape.T)["gemm1_gate_up_swiglu"]


def test_decode_streams_weights_and_prefill_is_compute_bound():
    ridge_bf16 = 1700e12 / 6763e9
    ridge_fp4 = 6 * ridge_bf16
    # 64 tokens x top-8 over 256 experts touch about 221 experts
    assert _intensity(synth.DECODE_BF16, 221) < 5 < ridge_bf16
    assert _intensity(synth.DECODE_NVFP4, 221) < ridge_fp4
    assert _intensity(synth.PREFILL_BF16, 256) > ridge_bf16
    assert _intensity(synth.PREFILL_NVFP4, 256) > ridge_fp4


def test_projection_bytes_at_decode_are_the_weights():
    s = synth.DECODE_BF16
    b = bench.projection_bytes(s, s.T)
    assert b["pool"] == 4096 * 8192 * 2 + 64 * 8192 * 2 + 64 * 4096 * 4
    assert b["unpool"] == 8192 * 4096 * 2 + 64 * 4096 * 2 + 64 * 8192 * 2
    assert b["router"] == 256 * 8192 * 4 + 64 * 8192 * 4 + 64 * 8 * 8
    # at 64 tokens the weights are more than 95 % of each projection's bytes
    assert 4096 * 8192 * 2 / b["pool"] > 0.95


def test_peak_follows_the_timed_region():
    """A kernel timed in a region shorter than SUSTAINED_MIN_S runs at the boost clock
    and is measured against the burst BF16 peak; a region of at least that long, against
    the sustained one.  NVFP4 GEMMs take the nominal FP4/BF16 ratio of either."""
    peaks = {"bf16_tflops": 1876.1, "bf16_tflops_sustained": 1706.8, "hbm_gbs": 6778.7}
    p, why = bench.tensor_peak(peaks, "measured", 0.24, nvfp4=False)
    assert p == 1876.1 and "bf16_tflops (" in why
    p, why = bench.tensor_peak(peaks, "measured", bench.SUSTAINED_MIN_S, nvfp4=False)
    assert p == 1706.8 and "sustained" in why
    p, why = bench.tensor_peak(peaks, "measured", 0.5, nvfp4=True)
    assert p == 1876.1 * bench.FP4_PER_BF16 and "measured FP4 MMA issue rate" in why


def test_roofline_frac_is_achieved_over_peak():
    """The line's frac is reproducible from its own achieved and peak."""
    s = synth.PREFILL_BF16
    stage_ms = {"norm": 0.2, "router": 0.14, "pool": 0.65, "dispatch": 0.26,
                "gemm1_gate_up_swiglu": 6.6, "gemm2_down": 3.2, "combine": 0.33, "unpool": 0.64}
    peaks = {"bf16_tflops": 1876.1, "bf16_tflops_sustained": 1706.8, "hbm_gbs": 6778.7}
    roof, tfl, _ = bench.roofline_of(s, s.T, stage_ms, 256, 0.25, peaks, "measured", "x")
    assert roof["bound"] == "tensor" and roof["kernel"] == "gemm1_gate_up_swiglu"
    assert roof["peak"] == 1876.1
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    fl = bench.flops_per_token(s)["gemm1_gate_up_swiglu"] * s.T
    assert abs(roof["achieved"] - fl / 6.6e-3 / 1e12) < 0.1
