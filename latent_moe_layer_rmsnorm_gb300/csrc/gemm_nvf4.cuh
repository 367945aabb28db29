// gemm_nvf4.cuh -- grouped expert GEMMs on NVFP4 operands with tcgen05 block-scaled MMA
// ("SGLang and Miles Add Day-0 Support for Muse Spark Open", "NVFP4 as a third MMA kind":
// E2M1 operands, UE4M3 scale per 16 elements, per-token FP32 input scales applied to the
// first GEMM's accumulators; "The NVFP4 requantization reciprocal table": the SwiGLU
// output is requantised to NVFP4 between the two GEMMs with a 256-entry FP32 table of
// scale reciprocals in shared memory).
//
//   gate/up  u [rows, p] x W13_e [2I, p] (gate/up rows interleaved in blocks of 64)
//            epilogue: a, b = acc * alpha[row] * beta13[e]; s = silu(a) * b; s -> NVFP4
//            with the static global scale gamma[e] (codes + chunked scales)
//   down     s [rows, I] x W2_e [p, I]; epilogue y = acc * gamma[e] * beta2[e] (FP16)
//
// The pipeline of gemm_tcgen05.cuh (TMA producer warp, one MMA-issuing thread, epilogue
// warps, bounded waits) with per-stage scale tiles: the producer bulk-copies the 4 scale
// chunks (512 B each) of the A and B tiles first, on a barrier of their own, then the
// operand tiles, and four scale warps (one per TMEM lane quadrant) write the chunks into
// TMEM with tcgen05.st while the operands still arrive, each quadrant getting the same
// 32 lanes x 16 columns per operand that a tcgen05.cp .32x128b.warpx4 of the chunks
// would leave.  Copying them with tcgen05.cp instead costs about 50 tensor-pipe cycles
// per chunk, more than the 4 MMAs of the slice take (measured on GB300).  The MMA thread
// issues 4 block-scaled MMAs (K = 64 each) per 128-byte K slice once its operands and
// scales are in place.  Tiles are 128 rows x 256 columns: per K slice 16 KB of A, 32 KB
// of B and 6 KB of scales for 128 x 256 x 256 MACs, a quarter fewer bytes per MAC than
// 128 x 128 tiles (the kernel is bound by the rate operands reach shared memory, about
// 52-64 B/clk per SM measured).  TMEM then holds one 256-column accumulator (columns
// [0, 256)) and a ring of per-stage scale columns after it, so the next tile's MMAs wait
// until the epilogue has read the accumulator: eight epilogue warps (two per lane
// quadrant, one per 128-column half) read it first (the gate/up epilogue forms its row's
// 64 SwiGLU values in registers) and hand it back before requantising and storing.
// A rows are 128-aligned per expert (padded dispatch), so a tile's scales are whole chunks.
#pragma once

#include "gemm_tcgen05.cuh"

namespace lmoe {

constexpr int NV_BN = 256;
// shared-memory ring depth: the gate/up kernel (no y staging boxes) fits 4 stages, which
// keep TMA loading further ahead while its epilogue runs between tiles (measured on
// GB300: 2.41 -> 2.06 ms for the prefill gate/up GEMM); the down kernel needs the
// boxes and keeps 3
constexpr int NV_MAX_STAGES = 4;
constexpr int NV_A_STAGE = GEMM_BM * 128;    // 128 rows x 256 FP4
constexpr int NV_B_STAGE = NV_BN * 128;
constexpr int NV_SFA_STAGE = 4 * 512;        // 4 scale chunks (K = 64 steps) of 128 A rows
constexpr int NV_SFB_STAGE = 8 * 512;        // the same for both 128-row halves of B
constexpr int NV_SF_COL0 = 256;
constexpr int NV_SF_COLS = 48;               // per stage: 16 (A) + 32 (B)
// warps 0 TMA, 1 MMA, 2 TMEM owner, 4-7 epilogue (columns 0-127), 8-11 scales,
// 12-15 epilogue (columns 128-255)
constexpr int NV_THREADS = 512;
// NVFP4 W13 rows interleave gate and up in blocks of 64: each 128-column half of a tile
// holds 64 gate columns and the matching 64 up columns (the layout moe_quantize_nvfp4
// writes and include/latent_moe.h documents)
constexpr int NV_W13_GROUP = 64;

// STORE_Y writes y through TMA store boxes (3-stage ring); STORE_Y_ROWS writes each valid
// row with plain 16-byte stores and keeps a 4-stage ring (no boxes): the down GEMM when
// tiles hold few rows (decode), where the weight stream is all that matters.
enum NvEpi : int { NV_EPI_SWIGLU_Q = 0, NV_EPI_STORE_Y = 1, NV_EPI_STORE_Y_ROWS = 2 };

struct NvSmem {
  GemmSmem g;                // barriers and schedule (its `full`/`empty` sized for GEMM_STAGES)
  uint64_t full[NV_MAX_STAGES];       // the stage's operand tiles landed
  uint64_t sfull[NV_MAX_STAGES];      // its scale chunks landed (copied first)
  uint64_t empty[NV_MAX_STAGES];
  uint64_t sf_ready[NV_MAX_STAGES];   // the 4 scale warps have written the stage's scales
  float recip[256];
};

// The down GEMM's epilogue writes y through shared memory: each epilogue warp stages a
// 32-row x 64-column FP16 box (4 KB, 128-byte swizzle) and stores it with TMA, instead of
// 32 rows of 16-byte pieces per store instruction (those stores cost about a third of
// the kernel's time, measured).  Expert rows are padded to 128 per expert, so a box never
// reaches another expert's rows; rows past an expert's last token are padding.
constexpr int NV_Y_BOX = 32 * 128;

template <int EPI> __host__ __device__ constexpr int nv_stages() {
  return EPI == NV_EPI_STORE_Y ? 3 : 4;
}
template <int EPI> __host__ __device__ constexpr int nv_boxes() {
  return EPI == NV_EPI_STORE_Y ? 8 : 0;
}
template <int EPI>
constexpr size_t nvf4_smem_bytes_for() {
  return 1024 + size_t(nv_stages<EPI>()) * (NV_A_STAGE + NV_B_STAGE + NV_SFA_STAGE + NV_SFB_STAGE) +
         size_t(nv_boxes<EPI>()) * NV_Y_BOX + sizeof(NvSmem);
}
// one dynamic shared-memory size for every variant: the largest
constexpr size_t nvf4_smem_bytes() {
  return nvf4_smem_bytes_for<NV_EPI_SWIGLU_Q>() > nvf4_smem_bytes_for<NV_EPI_STORE_Y>()
             ? nvf4_smem_bytes_for<NV_EPI_SWIGLU_Q>()
             : nvf4_smem_bytes_for<NV_EPI_STORE_Y>();
}
static_assert(nvf4_smem_bytes_for<NV_EPI_STORE_Y_ROWS>() <= nvf4_smem_bytes(), "row-store size");
static_assert(nvf4_smem_bytes() <= 232448, "more than 227 KB of shared memory per CTA");
static_assert(NV_SF_COL0 + NV_MAX_STAGES * NV_SF_COLS <= GEMM_TMEM_COLS, "scale ring past TMEM");



// The tile's scalars for row r, read before the epilogue waits for the accumulator so
// their latency hides behind the tile's MMAs.  SwiGLU: x0 = per-token activation scale x
// the expert's W13 scale, x1 = the expert's static scale of s.  Down: x0 = the expert's
// W2 scale x the scale of s.  Every row of a tile lies inside the expert's 128-row
// padded block, so the per-row scale array (one entry per padded row) covers it even
// when the row holds no token.
template <int EPI>
__device__ __forceinline__ void nvf4_scalars(const GemmParams& P, const TileCoord& tc, int r,
                                             float& x0, float& x1) {
  if constexpr (EPI == NV_EPI_SWIGLU_Q) {
    x0 = P.row_scale[static_cast<size_t>(tc.a_row + r)] * P.grp_scale[tc.e];
    x1 = P.out_scale[tc.e];
  } else {
    x0 = P.grp_scale[tc.e] * P.out_scale[tc.e];
    x1 = 0.f;
  }
}

// One warp's 32 rows of one 128-column block of the accumulator (taddr points at its
// first column); `col0` is the block's first output column: of s (64 SwiGLU outputs per
// block) for the gate/up GEMM, of y for the down GEMM.  x0, x1 from nvf4_scalars.
// `release()` is called once by every thread as soon as its last TMEM read has completed,
// before the rest of the epilogue, so the MMAs of the next tile can start under it: the
// gate/up GEMM holds the 64 SwiGLU values of its row in registers and requantises them
// after the release; the down GEMM releases after its last accumulator load.
template <int EPI, typename Release>
__device__ __forceinline__ void nvf4_epilogue(const GemmParams& P, const TileCoord& tc,
                                              uint32_t taddr, int r, int col0, const float* recip,
                                              const CUtensorMap* tmY, uint8_t* ybox, float x0,
                                              float x1, Release&& release) {
  const bool row_ok = r < tc.valid;
  const size_t row = static_cast<size_t>(tc.a_row + r);
  if (r - (r & 31) >= tc.valid) {   // the warp's 32 rows are all padding: nothing to store
    release();
    return;
  }
  if constexpr (EPI == NV_EPI_SWIGLU_Q) {
    // columns [0, 64) of the block gate, [64, 128) up, of output features col0 ..
    const float sc = x0;
    const float gam = x1;
    float sv[64];
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
      uint32_t g[16], u[16];
      tmem_ld16(taddr + c0, g);
      tmem_ld16(taddr + 64 + c0, u);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = __uint_as_float(g[i]) * sc, b = __uint_as_float(u[i]) * sc;
        sv[c0 + i] = __fdividef(a, 1.0f + __expf(-a)) * b;   // silu(a) * b
      }
    }
    release();
    const float six_g = 6.0f * gam;
    const float inv_g = gam > 0.f ? 1.0f / gam : 0.f;
    const int I = P.ld_out;
    uint8_t* codes = static_cast<uint8_t*>(P.out) + row * (I / 2);
    // two quantisation blocks at a time: their chains are independent
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      const float(&s0)[16] = *reinterpret_cast<const float(*)[16]>(sv + c0);
      const float(&s1)[16] = *reinterpret_cast<const float(*)[16]>(sv + c0 + 16);
      uint2 q0, q1;
      float ratio0, ratio1, fin = 0.f;
      const uint32_t code0 = quantize16(s0, six_g, inv_g, q0, recip, &ratio0);
      const uint32_t code1 = quantize16(s1, six_g, inv_g, q1, recip, &ratio1);
#pragma unroll
      for (int i = 0; i < 16; ++i) fin = fmaf(s0[i] + s1[i], 0.f, fin);   // NaN unless finite
      // a block whose ratio passed 464 saturated its scale at 448 instead of rounding: its
      // static global scale is too small for it (or s is not finite)
      if (row_ok && !(fmaxf(ratio0, ratio1) <= 464.f && fin == 0.f))
        report_error(P.status, ST_DEVICE_CHECK, CHECK_S_RANGE);
      if (row_ok) {
        const int col = col0 + c0;
        *reinterpret_cast<uint4*>(codes + col / 2) = make_uint4(q0.x, q0.y, q1.x, q1.y);
        P.out_sf[sf_offset(row, col / 16, I)] = static_cast<uint8_t>(code0);
        P.out_sf[sf_offset(row, col / 16 + 1, I)] = static_cast<uint8_t>(code1);
      }
    }
  } else if constexpr (EPI == NV_EPI_STORE_Y_ROWS) {
    const float sc = x0;
    float ss = 0.f;     // the block is one 128-column block of the row (row_ssq)
    __half* yrow = static_cast<__half*>(P.out) + row * P.ld_out + col0;
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 64) {
      uint32_t a0[16], a1[16], a2[16], a3[16];
      tmem_ld16(taddr + c0, a0);
      tmem_ld16(taddr + c0 + 16, a1);
      tmem_ld16(taddr + c0 + 32, a2);
      tmem_ld16(taddr + c0 + 48, a3);
      tmem_ld_wait();
      if (c0 == 64) release();
      float v[64];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        v[i] = __uint_as_float(a0[i]) * sc;
        v[16 + i] = __uint_as_float(a1[i]) * sc;
        v[32 + i] = __uint_as_float(a2[i]) * sc;
        v[48 + i] = __uint_as_float(a3[i]) * sc;
      }
      if (row_ok) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float* w = v + 8 * j;
          *reinterpret_cast<uint4*>(yrow + c0 + 8 * j) =
              make_uint4(pack_f16x2(w[0], w[1]), pack_f16x2(w[2], w[3]),
                         pack_f16x2(w[4], w[5]), pack_f16x2(w[6], w[7]));
        }
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) { const float q = stored_value(v[i], OUT_F16); ss = fmaf(q, q, ss); }
    }
    if (P.row_ssq && row_ok) P.row_ssq[row * (P.N >> 7) + (col0 >> 7)] = ss;
  } else {
    const float sc = x0;
    const int lane = r & 31;
    float ss = 0.f;     // the block is one 128-column block of the row (row_ssq)
    // one 32-row x 64-column FP16 staging box per TMEM wait: row `lane`, 16-byte chunk j
    // (columns 8j..8j+7) at chunk (j ^ lane % 8), the 128-byte swizzle of the tensor map
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 64) {
      uint32_t a0[16], a1[16], a2[16], a3[16];
      tmem_ld16(taddr + c0, a0);
      tmem_ld16(taddr + c0 + 16, a1);
      tmem_ld16(taddr + c0 + 32, a2);
      tmem_ld16(taddr + c0 + 48, a3);
      tmem_ld_wait();
      if (c0 == 64) release();
      float v[64];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        v[i] = __uint_as_float(a0[i]) * sc;
        v[16 + i] = __uint_as_float(a1[i]) * sc;
        v[32 + i] = __uint_as_float(a2[i]) * sc;
        v[48 + i] = __uint_as_float(a3[i]) * sc;
      }
      if (lane == 0) tma_store_wait_read();      // the box's previous store has read it
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float* w = v + 8 * j;
        const uint4 o = make_uint4(pack_f16x2(w[0], w[1]), pack_f16x2(w[2], w[3]),
                                   pack_f16x2(w[4], w[5]), pack_f16x2(w[6], w[7]));
        *reinterpret_cast<uint4*>(ybox + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        tma_store_2d(tmY, ybox, col0 + c0, tc.a_row + (r - lane));
#pragma unroll
      for (int i = 0; i < 64; ++i) { const float q = stored_value(v[i], OUT_F16); ss = fmaf(q, q, ss); }
    }
    if (P.row_ssq && row_ok) P.row_ssq[row * (P.N >> 7) + (col0 >> 7)] = ss;
  }
}

template <int EPI>
__global__ void __launch_bounds__(NV_THREADS, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmY, const GemmParams P) {
  constexpr int NS = nv_stages<EPI>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + NS * NV_A_STAGE;
  uint8_t* sSA = sB + NS * NV_B_STAGE;
  uint8_t* sSB = sSA + NS * NV_SFA_STAGE;
  uint8_t* sY = sSB + NS * NV_SFB_STAGE;    // staging boxes (down GEMM only), 1 KB aligned
  NvSmem* N = reinterpret_cast<NvSmem*>(sY + nv_boxes<EPI>() * NV_Y_BOX);
  GemmSmem* S = &N->g;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&N->full[s], 1);
      mbar_init(&N->sfull[s], 1);
      mbar_init(&N->empty[s], 1);
      mbar_init(&N->sf_ready[s], 4);
    }
    mbar_init(&S->tfull[0], 1);       // one accumulator: the [0] barriers only
    mbar_init(&S->tempty[0], 8);
    mbar_init(&S->drain, 1);
    S->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  for (int i = threadIdx.x; i < 256; i += blockDim.x) N->recip[i] = recip_ue4m3(i);
  pdl_wait();          // the inputs and tables are the previous kernels' outputs
  pdl_allow_next();
  for (int i = threadIdx.x; i <= P.groups; i += blockDim.x) {
    S->mt_off[i] = P.mt_off[i];
    S->row_off[i] = P.row_off[i];
    S->row_cnt[i] = P.row_cnt[i];
  }
  if (warp == 2) tmem_alloc(&S->tmem_base, GEMM_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = S->tmem_base;
  const int num_tiles = gemm_num_tiles(P, S);
  const int kblocks = P.K / 256;               // 256 FP4 = 128 bytes per stage
  const int kchunks = P.K / 64;                // scale chunks per 128-row block
  const uint64_t limit = P.timeout_ns;
  volatile int* abort_flag = &S->abort_flag;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    // the scale chunks go first, on their own barrier, so the scale warps can move them
    // into TMEM while the operand tiles are still arriving
    const uint32_t bytes = NV_A_STAGE + NV_B_STAGE;
    int stage = 0;
    uint32_t phase = 0;
    int last_phase[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) last_phase[s] = -1;
    for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
      const TileCoord tc = gemm_tile(P, S, t);
      const uint8_t* sfa = P.sf_a + (static_cast<size_t>(tc.a_row >> 7) * kchunks) * 512;
      const uint8_t* sfb = P.sf_b + (static_cast<size_t>(tc.b_row >> 7) * kchunks) * 512;
      const uint8_t* sfb1 = sfb + static_cast<size_t>(kchunks) * 512;   // rows 128-255
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&N->empty[stage], phase ^ 1, abort_flag, P.status,
                               WAIT_PRODUCER_EMPTY, limit))
          goto producer_done;
        mbar_arrive_expect_tx(&N->sfull[stage], NV_SFA_STAGE + NV_SFB_STAGE);
        bulk_load(sSA + stage * NV_SFA_STAGE, sfa + kb * NV_SFA_STAGE, NV_SFA_STAGE,
                  &N->sfull[stage]);
        bulk_load(sSB + stage * NV_SFB_STAGE, sfb + kb * 2048, 2048, &N->sfull[stage]);
        bulk_load(sSB + stage * NV_SFB_STAGE + 2048, sfb1 + kb * 2048, 2048, &N->sfull[stage]);
        mbar_arrive_expect_tx(&N->full[stage], bytes);
        tma_load_2d(sA + stage * NV_A_STAGE, &tmA, &N->full[stage], kb * 128, tc.a_row);
        tma_load_2d(sB + stage * NV_B_STAGE, &tmB, &N->full[stage], kb * 128, tc.b_row);
        last_phase[stage] = static_cast<int>(phase);
        if (++stage == NS) { stage = 0; phase ^= 1; }
      }
    }
  producer_done:
    if (*abort_flag) {
      volatile int never = 0;
      for (int s = 0; s < NS; ++s)
        if (last_phase[s] >= 0) {
          mbar_wait_bounded(&N->full[s], static_cast<uint32_t>(last_phase[s]), &never, nullptr,
                            WAIT_DRAIN, limit);
          mbar_wait_bounded(&N->sfull[s], static_cast<uint32_t>(last_phase[s]), &never, nullptr,
                            WAIT_DRAIN, limit);
        }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = idesc_nvf4(GEMM_BM, NV_BN);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      if (!mbar_wait_bounded(&S->tempty[0], (it & 1) ^ 1, abort_flag, P.status,
                             WAIT_MMA_TMEM_EMPTY, limit))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&N->full[stage], phase, abort_flag, P.status, WAIT_MMA_FULL,
                               limit)) {
          ok = false;
          break;
        }
        if (!mbar_wait_bounded(&N->sf_ready[stage], phase, abort_flag, P.status,
                               WAIT_MMA_FULL, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_col = tmem_base + NV_SF_COL0 + stage * NV_SF_COLS;
        const uint32_t a0 = smem_u32(sA + stage * NV_A_STAGE);
        const uint32_t b0 = smem_u32(sB + stage * NV_B_STAGE);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mma_issue_nvf4(d_tmem, sdesc_sw128(a0 + 32 * j), sdesc_sw128(b0 + 32 * j), idesc,
                         sf_col + 4 * j, sf_col + 16 + 8 * j, (kb | j) != 0);
        }
        mma_commit(&N->empty[stage]);
        if (++stage == NS) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit(&S->tfull[0]);
    }
    mma_commit(&S->drain);
    {
      volatile int never = 0;
      mbar_wait_bounded(&S->drain, 0, &never, P.status, WAIT_DRAIN, limit);
    }
  } else if (warp >= 8 && warp < 12) {
    // ---------------- scale warps: stage scales -> TMEM (quadrant warp % 4) ----------
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&N->sfull[stage], phase, abort_flag, P.status, WAIT_MMA_FULL,
                               limit)) {
          ok = false;
          break;
        }
        // lane l: row l of each 512-byte chunk (16 bytes = 4 columns).  A: chunk j ->
        // columns 4j..; B (N = 256): K step j takes 8 columns, rows 0-127 (chunk j of the
        // first half) then rows 128-255 (chunk j of the second half)
        uint32_t va[16], vb0[16], vb1[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(sSA + stage * NV_SFA_STAGE + 512 * j + 16 * lane);
          va[4 * j] = a.x; va[4 * j + 1] = a.y; va[4 * j + 2] = a.z; va[4 * j + 3] = a.w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint8_t* sb = sSB + stage * NV_SFB_STAGE;
          const uint4 b0 = *reinterpret_cast<const uint4*>(sb + 512 * j + 16 * lane);
          const uint4 b1 = *reinterpret_cast<const uint4*>(sb + 2048 + 512 * j + 16 * lane);
          uint32_t* v = j < 2 ? vb0 : vb1;
          const int o = 8 * (j & 1);
          v[o] = b0.x; v[o + 1] = b0.y; v[o + 2] = b0.z; v[o + 3] = b0.w;
          v[o + 4] = b1.x; v[o + 5] = b1.y; v[o + 6] = b1.z; v[o + 7] = b1.w;
        }
        const uint32_t sf_col = tmem_base + NV_SF_COL0 + stage * NV_SF_COLS + lane_base;
        tmem_st16(sf_col, va);
        tmem_st16(sf_col + 16, vb0);
        tmem_st16(sf_col + 32, vb1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&N->sf_ready[stage]);
        if (++stage == NS) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
    }
  } else if (warp >= 4) {
    // ---------------- epilogue: warps 4-7 columns 0-127, 12-15 columns 128-255 -------
    const int q = warp & 3;
    const int hh = warp >= 12 ? 1 : 0;
    const int r = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const TileCoord tc = gemm_tile(P, S, t);
      float x0, x1;
      nvf4_scalars<EPI>(P, tc, r, x0, x1);        // in flight while the MMAs run
      if (!mbar_wait_bounded(&S->tfull[0], it & 1, abort_flag, P.status, WAIT_EPI_TMEM_FULL,
                             limit))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + hh * 128 + (static_cast<uint32_t>(q * 32) << 16);
      const int col0 = EPI == NV_EPI_SWIGLU_Q ? tc.n_blk * (NV_BN / 2) + hh * 64
                                              : tc.n_blk * NV_BN + hh * 128;
      nvf4_epilogue<EPI>(P, tc, taddr, r, col0, N->recip, &tmY, sY + (hh * 4 + q) * NV_Y_BOX,
                         x0, x1, [&] {
                           tc_fence_before();
                           __syncwarp();
                           if (lane == 0) mbar_arrive(&S->tempty[0]);
                         });
    }
    if (EPI == NV_EPI_STORE_Y && lane == 0) tma_store_wait_all();   // y fully written
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, GEMM_TMEM_COLS);
  }
}

}  // namespace lmoe
