// gemm_pair.cuh -- the tcgen05 GEMM of gemm_tcgen05.cuh on CTA pairs (cta_group::2).
//
// A cluster of two CTAs computes one 256 x 256 output tile: CTA r holds A rows
// 128r .. 128r+127 and B rows 128r .. 128r+127 of the tile in its own shared memory, the
// leader (rank 0) issues M = 256, N = 256 MMAs that read both halves, and each CTA's TMEM
// receives its 128 rows x 256 columns.  Per CTA and K slice that is 32 KB of operands for
// 128 x 256 x 64 MACs, against 48 KB on one CTA: the expert and projection GEMMs are
// bound by operand delivery into shared memory, so this is the tile shape that moves them.
//
// Grouped (per-expert) GEMMs tile each expert's rows in 256-row pair tiles.  An expert's
// last tile with at most 128 rows left runs as an M = 128 pair MMA instead, so a remainder
// costs no more MMA work than a 128-row single-CTA tile would.  CTA r then holds A rows
// 64r .. 64r+63 (a 64-row TMA box), and its 64 x 256 block of D is folded onto the 128
// TMEM lanes: lane i holds row i, columns 0-127, and lane 64 + i holds row i, columns
// 128-255, both in TMEM columns 0-127 (measured on the hardware).  The gate/up GEMM
// therefore loads its B half as [gate 64 rows; up 64 rows] in those tiles, so that each
// lane sees the gate and up columns its SwiGLU outputs need.
//
// Protocol (every wait bounded):
//   full[s]    leader only: the leader arms it with both CTAs' bytes; both CTAs' TMA
//              loads (.cta_group::2) complete on it
//   empty[s]   both CTAs: the leader's tcgen05.commit multicasts to both when the MMAs
//              reading stage s are done
//   tfull[a]   both CTAs: multicast commit after a tile's last MMA
//   tempty[a]  leader only: 4 epilogue warps of each CTA arrive (the peer remotely)
// A cluster barrier after set-up and before teardown keeps both CTAs alive while the
// other may still touch their shared memory or barriers.
#pragma once

#include "gemm_tcgen05.cuh"

namespace lmoe {

// Six 32 KB stages (a seventh measured neutral) and four 4 KB output boxes; the
// per-expert tables stay in global memory (L1-cached reads).
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_BOX = 32 * 128;            // one epilogue warp's 32 rows x 128 bytes
constexpr int PAIR_STAGE = 2 * 128 * 128;     // A 128 rows + B 128 rows of 128 bytes

struct PairSmem {
  uint64_t full[PAIR_STAGES];
  uint64_t empty[PAIR_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t pair_smem_bytes() {
  return 1024 + size_t(PAIR_STAGES) * PAIR_STAGE + 4 * PAIR_BOX + sizeof(PairSmem);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory object in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive;\n\tbarrier.cluster.wait;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t leader_bar, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(leader_bar), "r"(c0), "r"(c1)
      : "memory");
}

template <bool TF32>
__device__ __forceinline__ void mma_issue_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  if constexpr (TF32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Arrive once on `bar` (same offset) in both CTAs of the pair when the leader's MMAs
// issued so far are complete.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Arrive once on the leader's own `bar` when its MMAs so far are complete.
__device__ __forceinline__ void mma_commit_pair_local(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Arrive on a barrier of the cluster (any CTA's) with the default CTA scope of release.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Pair tile t -> this CTA's rows; `small` marks an M = 128 tile (64 rows per CTA).
// Dense: 256-row tiles over M.  Grouped: ceil(rows / 256) tiles per expert (mt_off holds
// the prefix sum of those counts).
__device__ __forceinline__ TileCoord pair_tile(const GemmParams& P, const PairSmem* S, int t,
                                               uint32_t rank, bool& small) {
  const int nb = P.N / P.bn;
  TileCoord c;
  c.split = 0;
  small = false;
  if (P.groups == 0) {
    const int m_pair = t / nb;
    c.n_blk = t - m_pair * nb;
    c.a_row = m_pair * 256 + 128 * static_cast<int>(rank);
    c.b_row = c.n_blk * P.bn + 128 * static_cast<int>(rank);
    c.valid = min(GEMM_BM, P.M - c.a_row);
    c.e = 0;
    return c;
  }
  int lo = 0, hi = P.groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(P.mt_off + mid) * nb <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mt_e = __ldg(P.mt_off + e);
  const int np_e = __ldg(P.mt_off + e + 1) - mt_e;
  const int local = t - mt_e * nb;
  c.n_blk = local / np_e;
  const int pr = local - c.n_blk * np_e;
  const int left = __ldg(P.row_cnt + e) - pr * 256;   // rows of this expert from the tile on
  small = left <= 128;
  const int half = small ? 64 : 128;
  c.a_row = __ldg(P.row_off + e) + pr * 256 + half * static_cast<int>(rank);
  c.b_row = e * P.N + c.n_blk * P.bn + 128 * static_cast<int>(rank);
  c.valid = min(half, left - half * static_cast<int>(rank));
  c.e = e;
  return c;
}

// Epilogue of an M = 128 tile for one warp: row `r` (0-63) of this CTA's rows, column
// half `h` of the 256-wide tile, read from TMEM columns 0-127 of the warp's lanes.
template <int EPI>
__device__ __forceinline__ void pair_small_epilogue(const GemmParams& P, const TileCoord& tc,
                                                    uint32_t taddr, int r, int h) {
  const bool row_ok = r < tc.valid;
  const size_t row = static_cast<size_t>(tc.a_row + r);
  if constexpr (EPI == EPI_SWIGLU) {
    // TMEM columns 0-63: gate, 64-127: the matching up; outputs h*64 .. h*64+63
    const size_t base = row * P.ld_out + static_cast<size_t>(tc.n_blk) * (P.bn >> 1) + h * 64;
    for (int c0 = 0; c0 < 64; c0 += 16) {
      uint32_t g[16], u[16];
      tmem_ld16(taddr + c0, g);
      tmem_ld16(taddr + 64 + c0, u);
      tmem_ld_wait();
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = __uint_as_float(g[i]);
        v[i] = __fdividef(a, 1.0f + __expf(-a)) * __uint_as_float(u[i]);   // silu(a) * b
      }
      if (row_ok) store16(P.out, base + c0, P.out_fmt, v);
    }
  } else {
    const size_t base = row * P.ld_out + static_cast<size_t>(tc.n_blk) * P.bn + h * 128;
    float ss = 0.f;
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t a[16], b[16];
      tmem_ld16(taddr + c0, a);
      tmem_ld16(taddr + c0 + 16, b);
      tmem_ld_wait();
      float va[16], vb[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) { va[i] = __uint_as_float(a[i]); vb[i] = __uint_as_float(b[i]); }
      if (row_ok) {
        store16(P.out, base + c0, P.out_fmt, va);
        store16(P.out, base + c0 + 16, P.out_fmt, vb);
      }
      const int rb = P.out_fmt;                    // squared as stored
      ss = add_stored_squares(ss, va, rb);
      ss = add_stored_squares(ss, vb, rb);
    }
    // same column order as the full-tile epilogue, so the block sums agree bit for bit
    if (P.row_ssq && row_ok)
      P.row_ssq[row * (P.N >> 7) + ((tc.n_blk * P.bn) >> 7) + h] = ss;
  }
}

// Put 16 consecutive output values of row `lane` into the warp's staging box at byte
// offset `off` of the row (128-byte swizzle: 16-byte chunk j lands at chunk j ^ lane % 8).
__device__ __forceinline__ void box_put16(uint8_t* box, int lane, int off, int fmt,
                                          const float (&v)[16]) {
  uint8_t* row = box + lane * 128;
  if (fmt == OUT_F16) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = (off >> 4) + h;
      const float* w = v + 8 * h;
      const uint4 o = make_uint4(pack_f16x2(w[0], w[1]), pack_f16x2(w[2], w[3]),
                                 pack_f16x2(w[4], w[5]), pack_f16x2(w[6], w[7]));
      *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) = o;
    }
  } else if (fmt == OUT_BF16) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = (off >> 4) + h;
      const float* w = v + 8 * h;
      const uint4 o = make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                                 pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7]));
      *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) = o;
    }
  } else {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int j = (off >> 4) + h;
      float w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = fmt == OUT_TF32 ? tf32_rna(v[4 * h + i]) : v[4 * h + i];
      *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) = make_float4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Epilogue of one warp whose 32 rows of a full-height tile are all valid: values go
// through the warp's shared-memory box and leave as 32-row x 128-byte TMA stores (a row
// segment per store instead of 16 bytes of each of 32 rows per store instruction).
// Same values, and for the down GEMM the same 128-column sums of squares in the same
// column order, as gemm_epilogue.
template <int EPI>
__device__ __forceinline__ void pair_epilogue_boxes(const GemmParams& P, const TileCoord& tc,
                                                    uint32_t taddr, int q, int lane,
                                                    const CUtensorMap* tmOut, uint8_t* box) {
  const int es = (P.out_fmt == OUT_BF16 || P.out_fmt == OUT_F16) ? 2 : 4;
  const int per_box = 128 / es;                       // values per box row
  const int row0 = tc.a_row + 32 * q;
  const size_t row = static_cast<size_t>(row0 + lane);
  auto put = [&](int col, const float (&v)[16], int col_base) {
    const int off = ((col - col_base) % per_box) * es;
    if (off == 0) {
      if (lane == 0) tma_store_wait_read();
      __syncwarp();
    }
    box_put16(box, lane, off, P.out_fmt, v);
    if (off + 16 * es == 128) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tma_store_2d(tmOut, box, col - (col - col_base) % per_box, row0);
    }
  };
  if constexpr (EPI == EPI_STORE) {
    const int col_base = tc.n_blk * P.bn;
    float ss = 0.f;
    for (int c0 = 0; c0 < P.bn; c0 += 32) {
      uint32_t a[16], b[16];
      tmem_ld16(taddr + c0, a);
      tmem_ld16(taddr + c0 + 16, b);
      tmem_ld_wait();
      float va[16], vb[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) { va[i] = __uint_as_float(a[i]); vb[i] = __uint_as_float(b[i]); }
      put(col_base + c0, va, col_base);
      put(col_base + c0 + 16, vb, col_base);
      if (P.row_ssq) {                                // squared as stored
        const int rb = P.out_fmt;
        ss = add_stored_squares(ss, va, rb);
        ss = add_stored_squares(ss, vb, rb);
        if (((c0 + 32) & 127) == 0) {
          P.row_ssq[row * (P.N >> 7) + ((col_base + c0) >> 7)] = ss;
          ss = 0.f;
        }
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {   // gate columns [0, bn/2), up [bn/2, bn)
    const int half = P.bn >> 1;
    const int col_base = tc.n_blk * half;
    for (int c0 = 0; c0 < half; c0 += 16) {
      uint32_t g[16], u[16];
      tmem_ld16(taddr + c0, g);
      tmem_ld16(taddr + half + c0, u);
      tmem_ld_wait();
      float s[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = __uint_as_float(g[i]);
        s[i] = __fdividef(a, 1.0f + __expf(-a)) * __uint_as_float(u[i]);   // silu(a) * b
      }
      put(col_base + c0, s, col_base);
    }
  }
}

template <int KIND, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmA64,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmB64,
                     const __grid_constant__ CUtensorMap tmOut, const GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* boxes = smem + PAIR_STAGES * PAIR_STAGE;     // 1 KB aligned
  PairSmem* S = reinterpret_cast<PairSmem*>(boxes + 4 * PAIR_BOX);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(&S->full[s], 1);
      mbar_init(&S->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&S->tfull[a], 1);
      mbar_init(&S->tempty[a], 8);
    }
    mbar_init(&S->drain, 1);
    S->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (P.groups > 0) {
      tma_prefetch_desc(&tmA64);
      if (EPI == EPI_SWIGLU) tma_prefetch_desc(&tmB64);
    }
  }
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

  constexpr bool TF32 = KIND == OP_TF32;
  const uint32_t tmem_base = S->tmem_base;
  const int nb = P.N / P.bn;
  const int num_tiles = P.groups == 0 ? ((P.M + 255) / 256) * nb : __ldg(P.mt_off + P.groups) * nb;
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;
  const int kblocks = P.K / (TF32 ? 32 : 64);
  const uint64_t limit = P.timeout_ns;
  volatile int* abort_flag = &S->abort_flag;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool issued_any = false;
    bool skip = P.debug_skip_first_load != 0 && leader;
    for (int t = cluster_id; t < num_tiles && !*abort_flag; t += num_clusters) {
      bool small;
      const TileCoord tc = pair_tile(P, S, t, rank, small);
      const CUtensorMap* ta = small ? &tmA64 : &tmA;
      const uint32_t bytes = small ? 2 * (PAIR_STAGE - 64 * 128) : 2 * PAIR_STAGE;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&S->empty[stage], phase ^ 1, abort_flag, P.status,
                               WAIT_PRODUCER_EMPTY, limit))
          goto producer_done;
        if (skip) {
          skip = false;   // test hook: this stage never fills, so the MMA wait runs out
        } else {
          const uint32_t bar = mapa_shared(smem_u32(&S->full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&S->full[stage], bytes);
          const int kc = kb * (TF32 ? 32 : 64);
          uint8_t* st = smem + stage * PAIR_STAGE;
          tma_load_2d_pair(st, ta, bar, kc, tc.a_row);
          if (EPI == EPI_SWIGLU && small) {
            // this CTA's 128 columns of the block: gate 64r.. and the matching up rows
            const int blk = tc.b_row - 128 * static_cast<int>(rank);
            tma_load_2d_pair(st + 128 * 128, &tmB64, bar, kc, blk + 64 * static_cast<int>(rank));
            tma_load_2d_pair(st + 128 * 128 + 64 * 128, &tmB64, bar, kc,
                             blk + 128 + 64 * static_cast<int>(rank));
          } else {
            tma_load_2d_pair(st + 128 * 128, &tmB, bar, kc, tc.b_row);
          }
          issued_any = true;
        }
        if (++stage == PAIR_STAGES) { stage = 0; phase ^= 1; }
      }
    }
  producer_done:
    if (*abort_flag && issued_any) {
      // copies completing on the leader's barriers cannot be observed here: give any
      // in flight ample time to land before the teardown barrier
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) { }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------- MMA issuer (leader) ----------------
    const uint32_t idesc256 = idesc_f32acc(static_cast<uint32_t>(KIND), 256, P.bn);
    const uint32_t idesc128 = idesc_f32acc(static_cast<uint32_t>(KIND), 128, P.bn);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters, ++it) {
      bool small;
      pair_tile(P, S, t, rank, small);
      const uint32_t idesc = small ? idesc128 : idesc256;
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(&S->tempty[acc], acc_phase ^ 1, abort_flag, P.status,
                             WAIT_MMA_TMEM_EMPTY, limit))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * GEMM_BN_MAX;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&S->full[stage], phase, abort_flag, P.status, WAIT_MMA_FULL,
                               limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(smem + stage * PAIR_STAGE);
        const uint32_t b0 = a0 + 128 * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_issue_pair<TF32>(d_tmem, sdesc_sw128(a0 + 32 * k), sdesc_sw128(b0 + 32 * k), idesc,
                               (kb | k) != 0);
        mma_commit_pair(&S->empty[stage]);
        if (++stage == PAIR_STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit_pair(&S->tfull[acc]);
    }
    mma_commit_pair_local(&S->drain);
    {
      volatile int never = 0;
      mbar_wait_bounded(&S->drain, 0, &never, P.status, WAIT_DRAIN, limit);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs: own rows) ----------------
    const int q = warp & 3;
    const int r = q * 32 + lane;
    int it = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(&S->tfull[acc], acc_phase, abort_flag, P.status,
                             WAIT_EPI_TMEM_FULL, limit))
        break;
      tc_fence_after();
      bool small;
      const TileCoord tc = pair_tile(P, S, t, rank, small);
      const uint32_t taddr =
          tmem_base + acc * GEMM_BN_MAX + (static_cast<uint32_t>(q * 32) << 16);
      if (small) pair_small_epilogue<EPI>(P, tc, taddr, (q & 1) * 32 + lane, q >> 1);
      else if (P.out_box && tc.valid >= 32 * (q + 1))
        pair_epilogue_boxes<EPI>(P, tc, taddr, q, lane, &tmOut, boxes + q * PAIR_BOX);
      else gemm_epilogue<EPI>(P, tc, taddr, r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // the accumulator's loads have completed (tcgen05.wait::ld): no memory write has
        // to reach the leader, so the arrive needs no cluster-scope release
        if (leader) mbar_arrive(&S->tempty[acc]);
        else mbar_arrive_cluster(mapa_shared(smem_u32(&S->tempty[acc]), 0));
      }
    }
    if (lane == 0) tma_store_wait_all();   // the box stores have landed
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
