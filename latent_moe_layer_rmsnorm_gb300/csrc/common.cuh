// common.cuh -- device helpers for sm_103a: mbarriers, TMA, tcgen05 (TMEM + MMA),
// bounded waits and the workspace status word.  Inline PTX written from the PTX ISA.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lmoe {

// ---- status word (first bytes of the workspace) ------------------------------------
// status[0]: first error code (moe_status_t), status[1]: detail (which wait/check).
enum : int { ST_OK = 0, ST_TIMEOUT = 5, ST_DEVICE_CHECK = 6 };
enum : int {
  WAIT_PRODUCER_EMPTY = 1,
  WAIT_MMA_FULL = 2,
  WAIT_MMA_TMEM_EMPTY = 3,
  WAIT_EPI_TMEM_FULL = 4,
  WAIT_DRAIN = 5,
  WAIT_COMBINE = 6,
  WAIT_BOUNDARY_ROWS = 7,   // the unpooler's row workers: a 32-row block never completed
  CHECK_EXPERT_ID = 16,
  CHECK_ROW = 17,
  // a stored intermediate left its format's range: a non-finite row, a value above the
  // FP16 maximum (h, u, c), or an s block whose NVFP4 scale saturated under its static
  // global scale
  CHECK_H_RANGE = 18,
  CHECK_U_RANGE = 19,
  CHECK_C_RANGE = 20,
  CHECK_S_RANGE = 21,
};

// Largest finite FP16 value: the FP16 intermediates (h, u, c) are checked against it.
constexpr float F16_MAX = 65504.0f;

__device__ __forceinline__ void report_error(int* status, int code, int detail) {
  if (status == nullptr) return;
  if (atomicCAS(status, 0, code) == 0) status[1] = detail;
}

// ---- programmatic dependent launch ----------------------------------------------------
// The kernels of one forward are launched so that each may start while its predecessor
// in the stream is still finishing (prologue: barrier set-up, tensor-map prefetch, TMEM
// allocation).  pdl_wait() blocks until every earlier grid of the stream has completed
// and its memory is visible: each kernel calls it before its first access to global
// memory, so no kernel completes before its predecessors and every read sees the
// writes before it.  pdl_allow_next() lets the next grid be scheduled (it then waits in
// its own pdl_wait).  Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_allow_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed.  Gives up after
// `limit_ns` (or as soon as another role raised the CTA's abort flag), records the
// failure in the status word and returns false.  Every pipeline wait goes through
// here, so a missing arrival ends the kernel with an error instead of a hang.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, int* status,
                                                  int where, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        report_error(status, ST_TIMEOUT, where);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// ---- TMA ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Ask L2 for the box at (c0, c1) of a tensor map (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// 2-D tiled load: box at (c0 = inner/element index, c1 = row) into smem, completing
// `bytes` of transaction count on `bar`.  c0 * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map,
                                                 uint64_t* bar, int32_t c0, int32_t c1,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
      "l"(policy)
      : "memory");
}

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16),
// completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// TMA store of a shared-memory box (written by the generic proxy: fence first) in its own
// bulk group; wait_read: earlier stores have read their source, wait_all: they are done.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t c0,
                                             int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the previous stores have read their shared-memory source
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- tcgen05: tensor memory ---------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns per thread (thread i <-> lane base+i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Each lane writes 16 consecutive 32-bit columns of its own TMEM lane (the warp's
// 32-lane quadrant).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- tcgen05: MMA -------------------------------------------------------------------
// Shared-memory matrix descriptor for a K-major operand tile stored with the 128-byte
// swizzle (rows of 128 B, 8-row / 1024-B swizzle atoms stacked along M/N):
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4 (unused here)
//   bits 32-45 stride byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-47 descriptor version 1     bits 61-63 layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor, dense MMA with FP32 accumulation, both operands K-major:
//   bits 4-5 D format (1 = F32); bits 7-9 / 10-12 A / B format (kind::f16: 0 = F16,
//   1 = BF16; kind::tf32: 2 = TF32); bits 17-22 N >> 3; bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f32acc(uint32_t ab_format, uint32_t m,
                                                    uint32_t n) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((n >> 3) << 17) |
         ((m >> 4) << 24);
}

template <bool TF32>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  if constexpr (TF32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Block-scaled FP4 MMA (NVFP4: E2M1 operands, one UE4M3 scale per 16 elements of K):
// scale_a / scale_b are the TMEM addresses of this K=64 step's scales (A row r: lane r,
// column scale_a + r/32; B column n: lane n%32, column scale_b + n/32; 4 bytes = the 4
// blocks of 16): the layout a tcgen05.cp .32x128b.warpx4 of a 4x32 chunk leaves.
__device__ __forceinline__ void mma_issue_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t scale_a, uint32_t scale_b,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(scale_a), "r"(scale_b), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of the block-scaled kind: A/B format E2M1 (1), scale format
// UE4M3 (bit 23 = 0), scale-data ids 0, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_nvf4(uint32_t m, uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Shared-memory descriptor of an unswizzled operand: 8-row x 16-byte core matrices,
// `lbo` bytes apart along the 16-byte dimension and `sbo` bytes apart along rows.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(lbo >> 4) << 16;
  d |= static_cast<uint64_t>(sbo >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  return d;
}

// Arrive once on `bar` when every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ---- small numeric helpers ----------------------------------------------------------
// FP32 -> TF32 with round to nearest, ties away from zero: add half a TF32 unit to
// the magnitude and clear the 13 dropped mantissa bits (finite inputs).
__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7F800000u) != 0x7F800000u) b = (b + 0x1000u) & 0xFFFFE000u;
  return __uint_as_float(b);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Storage formats of GEMM outputs.  FP16 holds the expert GEMMs' outputs (s, y) of BF16
// configurations: 3 more significand bits than BF16 at the same size.
enum OutFmt : int { OUT_BF16 = 0, OUT_F32 = 1, OUT_TF32 = 2, OUT_F16 = 3 };

// The value an output holds once stored in format `fmt` (round to nearest even for BF16
// and FP16; FP32 keeps it).  Epilogues square this value, so a row's sums of squares
// describe the stored row.
__device__ __forceinline__ float stored_value(float v, int fmt) {
  if (fmt == OUT_BF16) return __bfloat162float(__float2bfloat16_rn(v));
  if (fmt == OUT_F16) return __half2float(__float2half_rn(v));
  return v;
}

// ss + the sum of squares of 16 values as stored in format `fmt`, one branch on the
// format for all 16 (the format is the same for every thread of a launch).
__device__ __forceinline__ float add_stored_squares(float ss, const float (&v)[16], int fmt) {
  if (fmt == OUT_F16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) { const float q = __half2float(__float2half_rn(v[i])); ss = fmaf(q, q, ss); }
  } else if (fmt == OUT_BF16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float q = __bfloat162float(__float2bfloat16_rn(v[i]));
      ss = fmaf(q, q, ss);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
  }
  return ss;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two FP32 values -> two E2M1 codes (round to nearest even, saturating at 6), `lo` in
// bits 0-3 (the even K element), `hi` in bits 4-7.
__device__ __forceinline__ uint32_t pack_e2m1x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1,
                                                        cudaRoundNearest));
}

// Non-negative FP32 -> UE4M3 code (round to nearest even, saturating at 448).
__device__ __forceinline__ uint32_t encode_ue4m3(float v) {
  return static_cast<uint32_t>(
             __nv_cvt_float2_to_fp8x2(make_float2(v, 0.0f), __NV_SATFINITE, __NV_E4M3)) &
         0xFFu;
}

// UE4M3 code -> value, from the format: bias 7, 3 mantissa bits, subnormals m * 2^-9.
// Built from the FP32 bit fields (exact).
__device__ __forceinline__ float decode_ue4m3(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e == 0 ? static_cast<float>(m) * 0.001953125f
                : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// 1 / scale for a UE4M3 code (IEEE division), 0 for the zero code and the NaN codes.
__device__ __forceinline__ float recip_ue4m3(uint32_t c) {
  c &= 0xFFu;
  return (c == 0 || (c & 0x7Fu) == 0x7Fu || c > 0x7Fu) ? 0.0f : 1.0f / decode_ue4m3(c);
}

// NVFP4 quantisation of one block of 16 FP32 values with global scale g (six_g =
// 6*g and inv_g = 1/g in FP32, both 0 when g == 0): returns the scale code and writes
// 8 bytes of E2M1 codes (element 2i in the low nibble of byte i).  The op order is
// the reference order: sf = ue4m3(bmax / six_g); r = recip(sf) * inv_g;
// code = e2m1(x * r).  ratio_out (optional) receives bmax / six_g: above 464 the scale
// saturated at 448 (the largest UE4M3 value) instead of rounding.
__device__ __forceinline__ uint32_t quantize16(const float (&x)[16], float six_g, float inv_g,
                                               uint2& codes, const float* recip_tab,
                                               float* ratio_out = nullptr) {
  float bmax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(x[i]));
  const float ratio = six_g > 0.f ? bmax / six_g : 0.f;
  if (ratio_out) *ratio_out = ratio;
  const uint32_t sf = encode_ue4m3(ratio);
  const float r = (recip_tab ? recip_tab[sf] : recip_ue4m3(sf)) * inv_g;
  uint32_t w0 = 0, w1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w0 |= pack_e2m1x2(x[2 * i] * r, x[2 * i + 1] * r) << (8 * i);
    w1 |= pack_e2m1x2(x[8 + 2 * i] * r, x[8 + 2 * i + 1] * r) << (8 * i);
  }
  codes = make_uint2(w0, w1);
  return sf;
}

// Byte offset of scale (row r, 16-element block g) in the chunked scale layout of a
// matrix with K columns: chunk = (r / 128, g / 4), 512 B each, chunks row-block-major;
// inside a chunk byte (r % 32) * 16 + ((r % 128) / 32) * 4 + g % 4.
__device__ __forceinline__ size_t sf_offset(size_t r, int g, int K) {
  const size_t chunk = (r >> 7) * static_cast<size_t>(K >> 6) + (g >> 2);
  return chunk * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (g & 3);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v);
  return __bfloat1622float2(b);
}

}  // namespace lmoe
