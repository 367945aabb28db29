// gemm_nvf4_pair.cuh -- the NVFP4 grouped expert GEMMs of gemm_nvf4.cuh on CTA pairs
// (tcgen05.mma.cta_group::2 with block scaling; "SGLang and Miles Add Day-0 Support for
// Muse Spark Open", "NVFP4 as a third MMA kind").
//
// A cluster of two CTAs computes a 256 x 256 output tile: CTA r stages A rows 128r ..
// 128r+127 of the tile and B rows 128r .. 128r+127 (half of the N = 256 weight rows) in
// its own shared memory, the leader (rank 0) issues M = 256, N = 256 block-scaled MMAs
// that read both halves, and each CTA's TMEM receives its 128 rows x 256 columns.  Per
// CTA and K slice (256 FP4 values) that is 16 KB of A, 16 KB of B and 6 KB of scale
// chunks for 128 x 256 x 256 MACs, against 54 KB on one CTA.
//
// Measured on a GB300 at a prefill chunk (131072 expert rows over 256 experts, p = I =
// 4096): the down GEMM takes 1.07 ms on pairs against 1.26 ms on single CTAs, the gate/up
// GEMM 2.28 against 2.16 ms (its SwiGLU + requantisation epilogue is longer, and with
// one accumulator the MMAs wait for it).  Timing copies with parts removed show what
// bounds both: without epilogues the gate/up GEMM takes 1.76 ms on pairs and 1.69 ms on
// single CTAs, without MMAs as well 1.57 and 1.41 ms.  Operand delivery, not the tensor
// pipe, sets the pace, and a stage takes about as long on a pair (38 KB per CTA) as on
// one CTA (54 KB), about 850 clocks: the round trip of a ring slot through the barriers
// of both CTAs, more than its bytes, is the limit.  A 256 x 128 variant with two
// accumulators (the epilogue under the next tile's MMAs) measured slower still (3.2 ms):
// half the MACs per stage at the same round trip.
//
// Scales: each CTA's TMEM holds the scales of its own 128 A rows and of all 256 B
// columns (the placement the pair MMA reads), so each CTA bulk-copies its own A scale
// chunks and both B halves' chunks into its shared memory (completing on its own
// barrier `sfull`), and its four scale warps write them into its TMEM exactly as in the
// single-CTA kernel, then arrive on the leader's `sf_ready` (8 arrivals per stage).
//
// Tiles: an expert's rows start on a 128-row boundary (padded dispatch) and its tiles
// cover them in steps of 256 rows (mt_off = prefix of ceil(rows / 256)).  When an
// expert's last tile holds at most 128 rows, the second CTA has no rows of it: it loads
// no A rows or A scales (the leader expects the smaller byte count), its half of the
// MMA output is never stored, and it only contributes its B half.
//
// Protocol (every wait bounded):
//   full[s]     leader only: armed by the leader with both CTAs' operand bytes; both
//               CTAs' .cta_group::2 TMA loads complete on it
//   sfull[s]    each CTA: its own scale chunks (bulk copies) landed
//   sf_ready[s] leader only: both CTAs' scale warps have written stage s's scales
//   empty[s]    both CTAs: the leader's commit multicasts when stage s's MMAs are done
//   tfull       both CTAs: multicast commit after a tile's last MMA
//   tempty      leader only: the 8 epilogue warps of each CTA arrive (the peer remotely)
// The follower's arrivals (scales written, accumulator read) publish TMEM that tcgen05
// operations completed before the arrive (tcgen05.wait::st / wait::ld) and that only the
// tensor core touches next, so they carry the default CTA scope of release: a release at
// cluster scope (a cluster-wide fence per stage and warp) measured as the bottleneck of
// the pipeline (ncu: 4.5 membar stalls per issued instruction, the kernel at half the
// one-CTA kernel's speed).
#pragma once

#include "gemm_nvf4.cuh"
#include "gemm_pair.cuh"

namespace lmoe {

constexpr int NVP_STAGES = 5;                       // 5 x 38 KB (+ 32 KB y boxes) fit
constexpr int NVP_A_STAGE = GEMM_BM * 128;          // 128 rows x 256 FP4
constexpr int NVP_B_STAGE = 128 * 128;              // this CTA's 128 of the 256 B rows
constexpr int NVP_SF_STAGE = NV_SFA_STAGE + NV_SFB_STAGE;   // 2 KB A + 4 KB B
constexpr int NVP_SF_COL0 = 256;
static_assert(NVP_SF_COL0 + NVP_STAGES * NV_SF_COLS <= GEMM_TMEM_COLS, "scale ring past TMEM");

struct NvPairSmem {
  uint64_t full[NVP_STAGES];
  uint64_t sfull[NVP_STAGES];
  uint64_t sf_ready[NVP_STAGES];
  uint64_t empty[NVP_STAGES];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  float recip[256];
};

template <int EPI>
constexpr size_t nvf4_pair_smem_bytes_for() {
  return 1024 + size_t(NVP_STAGES) * (NVP_A_STAGE + NVP_B_STAGE + NVP_SF_STAGE) +
         size_t(nv_boxes<EPI>()) * NV_Y_BOX + sizeof(NvPairSmem);
}
constexpr size_t nvf4_pair_smem_bytes() {
  return nvf4_pair_smem_bytes_for<NV_EPI_SWIGLU_Q>() > nvf4_pair_smem_bytes_for<NV_EPI_STORE_Y>()
             ? nvf4_pair_smem_bytes_for<NV_EPI_SWIGLU_Q>()
             : nvf4_pair_smem_bytes_for<NV_EPI_STORE_Y>();
}
static_assert(nvf4_pair_smem_bytes() <= 232448, "more than 227 KB of shared memory per CTA");

// Pair block-scaled MMA, issued by the leader: D (M = 256 over both CTAs' TMEM) from A and
// B halves at the same shared-memory offsets in both CTAs and the scales at the same TMEM
// columns in both.
__device__ __forceinline__ void mma_issue_nvf4_pair(uint32_t d_tmem, uint64_t adesc,
                                                    uint64_t bdesc, uint32_t idesc,
                                                    uint32_t scale_a, uint32_t scale_b,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(scale_a), "r"(scale_b), "r"(accumulate)
      : "memory");
}


// Pair tile t -> this CTA's rows.  `half`: the tile's second CTA holds no rows of the
// expert (its valid count is <= 0 then).
__device__ __forceinline__ TileCoord nvp_tile(const GemmParams& P, int t, uint32_t rank,
                                              bool& half) {
  const int nb = P.N / NV_BN;
  int lo = 0, hi = P.groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(P.mt_off + mid) * nb <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mt_e = __ldg(P.mt_off + e);
  const int np_e = __ldg(P.mt_off + e + 1) - mt_e;
  const int local = t - mt_e * nb;
  TileCoord c;
  c.split = 0;
  c.n_blk = local / np_e;
  const int pr = local - c.n_blk * np_e;
  const int left = __ldg(P.row_cnt + e) - pr * 256;
  half = left <= 128;
  c.a_row = __ldg(P.row_off + e) + pr * 256 + 128 * static_cast<int>(rank);
  c.b_row = e * P.N + c.n_blk * NV_BN;               // the tile's first B row
  c.valid = min(128, left - 128 * static_cast<int>(rank));
  c.e = e;
  return c;
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NV_THREADS, 1)
    gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmY, const GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + NVP_STAGES * NVP_A_STAGE;
  uint8_t* sSF = sB + NVP_STAGES * NVP_B_STAGE;        // per stage: A chunks, then B chunks
  uint8_t* sY = sSF + NVP_STAGES * NVP_SF_STAGE;       // staging boxes (down GEMM only)
  NvPairSmem* S = reinterpret_cast<NvPairSmem*>(sY + nv_boxes<EPI>() * NV_Y_BOX);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NVP_STAGES; ++s) {
      mbar_init(&S->full[s], 1);
      mbar_init(&S->sfull[s], 1);
      mbar_init(&S->sf_ready[s], 8);
      mbar_init(&S->empty[s], 1);
    }
    mbar_init(&S->tfull, 1);
    mbar_init(&S->tempty, 16);
    mbar_init(&S->drain, 1);
    S->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  for (int i = threadIdx.x; i < 256; i += blockDim.x) S->recip[i] = recip_ue4m3(i);
  pdl_wait();          // the inputs and tables are the previous kernels' outputs
  pdl_allow_next();
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&S->tmem_base)),
                 "r"(GEMM_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();

  const uint32_t tmem_base = S->tmem_base;
  const int nb = P.N / NV_BN;
  const int num_tiles = __ldg(P.mt_off + P.groups) * nb;
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;
  const int kblocks = P.K / 256;               // 256 FP4 = 128 bytes per stage
  const int kchunks = P.K / 64;                // scale chunks per 128-row block
  const uint64_t limit = P.timeout_ns;
  volatile int* abort_flag = &S->abort_flag;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool issued_any = false;
    int last_sf_phase[NVP_STAGES];   // parity of the last scale load into each stage
#pragma unroll
    for (int s = 0; s < NVP_STAGES; ++s) last_sf_phase[s] = -1;
    for (int t = cluster_id; t < num_tiles && !*abort_flag; t += num_clusters) {
      bool half;
      const TileCoord tc = nvp_tile(P, t, rank, half);
      const bool load_a = tc.valid > 0;
      const uint8_t* sfa = P.sf_a + (static_cast<size_t>(tc.a_row >> 7) * kchunks) * 512;
      const uint8_t* sfb = P.sf_b + (static_cast<size_t>(tc.b_row >> 7) * kchunks) * 512;
      const uint8_t* sfb1 = sfb + static_cast<size_t>(kchunks) * 512;   // rows 128-255
      const uint32_t op_bytes = (half ? 3u : 4u) * NVP_A_STAGE;   // A + B of both CTAs
      const uint32_t sf_bytes = (load_a ? NV_SFA_STAGE : 0) + NV_SFB_STAGE;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&S->empty[stage], phase ^ 1, abort_flag, P.status,
                               WAIT_PRODUCER_EMPTY, limit))
          goto producer_done;
        const uint32_t bar = mapa_shared(smem_u32(&S->full[stage]), 0);
        if (leader) mbar_arrive_expect_tx(&S->full[stage], op_bytes);
        uint8_t* sf = sSF + stage * NVP_SF_STAGE;
        // scale chunks first, so the scale warps can start while the operands arrive
        mbar_arrive_expect_tx(&S->sfull[stage], sf_bytes);
        if (load_a) bulk_load(sf, sfa + kb * NV_SFA_STAGE, NV_SFA_STAGE, &S->sfull[stage]);
        bulk_load(sf + NV_SFA_STAGE, sfb + kb * 2048, 2048, &S->sfull[stage]);
        bulk_load(sf + NV_SFA_STAGE + 2048, sfb1 + kb * 2048, 2048, &S->sfull[stage]);
        if (load_a) tma_load_2d_pair(sA + stage * NVP_A_STAGE, &tmA, bar, kb * 128, tc.a_row);
        tma_load_2d_pair(sB + stage * NVP_B_STAGE, &tmB, bar, kb * 128,
                         tc.b_row + 128 * static_cast<int>(rank));
        last_sf_phase[stage] = static_cast<int>(phase);
        issued_any = true;
        if (++stage == NVP_STAGES) { stage = 0; phase ^= 1; }
      }
    }
  producer_done:
    if (*abort_flag && issued_any) {
      // the scale copies complete on this CTA's own barriers: wait for them (bounded);
      // operand copies complete on the leader's: give those ample time to land before
      // the teardown barrier
      volatile int never = 0;
      for (int s = 0; s < NVP_STAGES; ++s)
        if (last_sf_phase[s] >= 0)
          mbar_wait_bounded(&S->sfull[s], static_cast<uint32_t>(last_sf_phase[s]), &never,
                            nullptr, WAIT_DRAIN, limit);
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) { }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------- MMA issuer (leader) ----------------
    const uint32_t idesc = idesc_nvf4(256, NV_BN);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters, ++it) {
      if (!mbar_wait_bounded(&S->tempty, (it & 1) ^ 1, abort_flag, P.status,
                             WAIT_MMA_TMEM_EMPTY, limit))
        break;
      tc_fence_after();
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&S->full[stage], phase, abort_flag, P.status, WAIT_MMA_FULL,
                               limit) ||
            !mbar_wait_bounded(&S->sf_ready[stage], phase, abort_flag, P.status,
                               WAIT_MMA_FULL, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_col = tmem_base + NVP_SF_COL0 + stage * NV_SF_COLS;
        const uint32_t a0 = smem_u32(sA + stage * NVP_A_STAGE);
        const uint32_t b0 = smem_u32(sB + stage * NVP_B_STAGE);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_issue_nvf4_pair(tmem_base, sdesc_sw128(a0 + 32 * j), sdesc_sw128(b0 + 32 * j),
                              idesc, sf_col + 4 * j, sf_col + 16 + 8 * j, (kb | j) != 0);
        mma_commit_pair(&S->empty[stage]);
        if (++stage == NVP_STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit_pair(&S->tfull);
    }
    mma_commit_pair_local(&S->drain);
    {
      volatile int never = 0;
      mbar_wait_bounded(&S->drain, 0, &never, P.status, WAIT_DRAIN, limit);
    }
  } else if (warp >= 8 && warp < 12) {
    // ---------------- scale warps (both CTAs): stage scales -> own TMEM ----------------
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ready = mapa_shared(smem_u32(&S->sf_ready[0]), 0);
    int stage = 0;
    uint32_t phase = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters) {
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&S->sfull[stage], phase, abort_flag, P.status, WAIT_MMA_FULL,
                               limit)) {
          ok = false;
          break;
        }
        // lane l: row l of each 512-byte chunk (16 bytes = 4 columns), as in the one-CTA
        // kernel (A chunks whose rows this CTA does not hold are not read by any store)
        const uint8_t* sf = sSF + stage * NVP_SF_STAGE;
        uint32_t va[16], vb0[16], vb1[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(sf + 512 * j + 16 * lane);
          va[4 * j] = a.x; va[4 * j + 1] = a.y; va[4 * j + 2] = a.z; va[4 * j + 3] = a.w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint8_t* sb = sf + NV_SFA_STAGE;
          const uint4 b0 = *reinterpret_cast<const uint4*>(sb + 512 * j + 16 * lane);
          const uint4 b1 = *reinterpret_cast<const uint4*>(sb + 2048 + 512 * j + 16 * lane);
          uint32_t* v = j < 2 ? vb0 : vb1;
          const int o = 8 * (j & 1);
          v[o] = b0.x; v[o + 1] = b0.y; v[o + 2] = b0.z; v[o + 3] = b0.w;
          v[o + 4] = b1.x; v[o + 5] = b1.y; v[o + 6] = b1.z; v[o + 7] = b1.w;
        }
        const uint32_t sf_col = tmem_base + NVP_SF_COL0 + stage * NV_SF_COLS + lane_base;
        tmem_st16(sf_col, va);
        tmem_st16(sf_col + 16, vb0);
        tmem_st16(sf_col + 32, vb1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&S->sf_ready[stage]);
          else mbar_arrive_cluster(ready + stage * 8);
        }
        if (++stage == NVP_STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
    }
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs, own rows): warps 4-7 columns 0-127,
    // 12-15 columns 128-255 ----------------
    const int q = warp & 3;
    const int hh = warp >= 12 ? 1 : 0;
    const int r = q * 32 + lane;
    const uint32_t tempty = mapa_shared(smem_u32(&S->tempty), 0);
    int it = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters, ++it) {
      bool half;
      const TileCoord tc = nvp_tile(P, t, rank, half);
      float x0 = 0.f, x1 = 0.f;
      if (tc.valid > 0) nvf4_scalars<EPI>(P, tc, r, x0, x1);   // in flight during the MMAs
      if (!mbar_wait_bounded(&S->tfull, it & 1, abort_flag, P.status, WAIT_EPI_TMEM_FULL,
                             limit))
        break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + hh * 128 + (static_cast<uint32_t>(q * 32) << 16);
      const int col0 = EPI == NV_EPI_SWIGLU_Q ? tc.n_blk * (NV_BN / 2) + hh * 64
                                              : tc.n_blk * NV_BN + hh * 128;
      auto release = [&] {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&S->tempty);
          else mbar_arrive_cluster(tempty);
        }
      };
      if (tc.valid > 0)
        nvf4_epilogue<EPI>(P, tc, taddr, r, col0, S->recip, &tmY, sY + (hh * 4 + q) * NV_Y_BOX,
                           x0, x1, release);
      else
        release();
    }
    if (EPI == NV_EPI_STORE_Y && lane == 0) tma_store_wait_all();   // y fully written
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(GEMM_TMEM_COLS)
                 : "memory");
  }
}

}  // namespace lmoe
