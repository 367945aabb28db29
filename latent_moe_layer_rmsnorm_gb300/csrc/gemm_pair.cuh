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
  c.valid = P.pad_rows ? half : min(half, left - half * static_cast<int>(rank));
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

// ---- the block boundary in the unpooler's kernel (EPI_BOUNDARY) --------------------------
// "SGLang and Miles Add Day-0 Support for Muse Spark Open", section "Kernel Optimizations":
// the post-FFN norm, the gated residual add and the next block's pre-attention norm are
// fused.  Here they run inside the unpooler GEMM that produces the block's output.  A
// row's RMS needs all d / 256 column tiles of the row, which different CTA pairs compute,
// so the tile epilogues (warps 4-7) store the output and its per-128-column sums of
// squares as for the plain unpooler and then count, per 32-row block, the tiles stored;
// six more warps of every CTA, idle during the main loop, take 2-row items in order and
// run the row pass on each once its block is complete:
//   a = RMSNorm_{g_post}(out) (sum of squares from the stored partials);
//   x' = x + gate * a, rounded to the residual stream's type and stored;
//   h' = RMSNorm_{g_next}(x' as stored)
// The output rows are reread from L2 within microseconds of their store, and the separate
// pass over [T, d] (its launch and its reread of the output from HBM) is gone.  A worker
// waits only for tiles of the same launch, whose CTAs never wait for a worker; the launch
// is sized so that all its clusters are resident together, and every wait is bounded.
// Measured at the prefill chunk (T = 16384, d = 8192): the row pass's reads (output rows,
// residual rows, gains, x' again) share the path from L2 into the SMs with the GEMM's
// operand copies, which bound the unpooler, and stretch its tiles from 0.59 to 0.71 ms;
// with the tail of the last rows the call takes what moe_forward + moe_boundary take.
constexpr int BND_ITEM_ROWS = 2;
// The fused kernel runs 12 warps: 0 TMA, 1 MMA, 4-7 epilogue as in the plain kernel, and
// the row workers 2, 3 and 8-11 (the epilogue warps join them after their last tile).
constexpr int BND_THREADS = 384;

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 8 consecutive values of a row chunk held as 1 (BF16) or 2 (FP32) 16-byte words
template <bool F32>
struct Chunk8 {
  uint4 w[F32 ? 2 : 1];
};

// Read at L2 (other SMs wrote these values during this launch; L1 may hold none of them)
template <bool F32>
__device__ __forceinline__ void chunk_ldcg(const void* base, size_t i, Chunk8<F32>& c) {
  const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(base) + i * (F32 ? 4 : 2));
  c.w[0] = __ldcg(p);
  if constexpr (F32) c.w[1] = __ldcg(p + 1);
}

template <bool F32>
__device__ __forceinline__ void chunk_unpack(const Chunk8<F32>& c, float (&v)[8]) {
  if constexpr (F32) {
    v[0] = __uint_as_float(c.w[0].x); v[1] = __uint_as_float(c.w[0].y);
    v[2] = __uint_as_float(c.w[0].z); v[3] = __uint_as_float(c.w[0].w);
    v[4] = __uint_as_float(c.w[1].x); v[5] = __uint_as_float(c.w[1].y);
    v[6] = __uint_as_float(c.w[1].z); v[7] = __uint_as_float(c.w[1].w);
  } else {
    float2 f;
    f = unpack_bf16x2(c.w[0].x); v[0] = f.x; v[1] = f.y;
    f = unpack_bf16x2(c.w[0].y); v[2] = f.x; v[3] = f.y;
    f = unpack_bf16x2(c.w[0].z); v[4] = f.x; v[5] = f.y;
    f = unpack_bf16x2(c.w[0].w); v[6] = f.x; v[7] = f.y;
  }
}

// Store 8 values (BF16: rounded to nearest even), streaming or plain
template <bool F32, bool STREAM>
__device__ __forceinline__ void chunk_store(void* base, size_t i, const float (&o)[8]) {
  uint4* p = reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + i * (F32 ? 4 : 2));
  if constexpr (F32) {
    const uint4 a = make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                               __float_as_uint(o[3]));
    const uint4 b = make_uint4(__float_as_uint(o[4]), __float_as_uint(o[5]), __float_as_uint(o[6]),
                               __float_as_uint(o[7]));
    if constexpr (STREAM) { __stcs(p, a); __stcs(p + 1, b); } else { p[0] = a; p[1] = b; }
  } else {
    const uint4 q = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                               pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
    if constexpr (STREAM) __stcs(p, q); else *p = q;
  }
}

__device__ __forceinline__ void load_vec8(const float* g, int col, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(g + col));
  const float4 b = __ldg(reinterpret_cast<const float4*>(g + col) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// The row pass on rows row0 and row1 (row1 == row0 for a lone last row) by one warp, in
// lockstep so that each gain vector is read once for both: lane l takes the 8-value
// chunks l, l + 32, ..., and every load of an iteration (U chunks of the gains and of
// both rows' output and x) is issued before the first is used.  The gains do not fit
// beside the GEMM's shared memory in L1, so they come from L2.
template <bool XF, bool YF>
__device__ __forceinline__ void boundary_rows(const GemmParams& P, int row0, int row1, int lane) {
  constexpr int U = 2;
  const BoundaryArgs& B = P.bnd;
  const int d = P.N;
  const int nch = d >> 3;
  const size_t base[2] = {static_cast<size_t>(row0) * d, static_cast<size_t>(row1) * d};
  const bool gated = B.gate != nullptr;
  // 1. sums of squares of the stored output rows, from their 128-column partials
  float rs_y[2], ss2[2] = {0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float* part = P.row_ssq + static_cast<size_t>(r ? row1 : row0) * (d >> 7);
    float ss = 0.f;
    for (int j = lane; j < (d >> 7); j += 32) ss += __ldcg(part + j);
    rs_y[r] = rsqrtf(warp_sum(ss) / static_cast<float>(d) + B.eps);
  }
  // 2. residual add, rounded to the stream's type
  for (int c0 = lane; c0 < nch; c0 += 32 * U) {
    Chunk8<YF> yc[U][2];
    Chunk8<XF> xc[U][2];
    float gp[U][8], gt[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 32 * u;
      if (c < nch) {
        load_vec8(B.g_post, 8 * c, gp[u]);
        if (gated) load_vec8(B.gate, 8 * c, gt[u]);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          chunk_ldcg<YF>(P.out, base[r] + 8 * c, yc[u][r]);
          chunk_ldcg<XF>(B.x, base[r] + 8 * c, xc[u][r]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 32 * u;
      if (c >= nch) continue;
      if (!gated) {
#pragma unroll
        for (int j = 0; j < 8; ++j) gt[u][j] = 1.f;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float yv[8], xv[8], o[8];
        chunk_unpack<YF>(yc[u][r], yv);
        chunk_unpack<XF>(xc[u][r], xv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          o[j] = xv[j] + gt[u][j] * (yv[j] * rs_y[r] * gp[u][j]);
          if (!XF) o[j] = __bfloat162float(__float2bfloat16_rn(o[j]));
          ss2[r] = fmaf(o[j], o[j], ss2[r]);
        }
        chunk_store<XF, false>(B.x_out, base[r] + 8 * c, o);
      }
    }
  }
  float rs_x[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) rs_x[r] = rsqrtf(warp_sum(ss2[r]) / static_cast<float>(d) + B.eps);
  // 3. the next block's pre-norm on x' as stored (each lane rereads its own chunks)
  for (int c0 = lane; c0 < nch; c0 += 32 * U) {
    Chunk8<XF> xc[U][2];
    float gn[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 32 * u;
      if (c < nch) {
        load_vec8(B.g_next, 8 * c, gn[u]);
#pragma unroll
        for (int r = 0; r < 2; ++r) chunk_ldcg<XF>(B.x_out, base[r] + 8 * c, xc[u][r]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 32 * u;
      if (c >= nch) continue;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float v[8], o[8];
        chunk_unpack<XF>(xc[u][r], v);
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = v[j] * rs_x[r] * gn[u][j];
        chunk_store<XF, true>(B.h_next, base[r] + 8 * c, o);
      }
    }
  }
}

// Row worker (one warp): claim items in order, wait (bounded) until the item's 32-row
// block has all its column tiles stored, run the row pass.  Returns when every item is
// claimed, or on a timeout / abort.
template <bool XF, bool YF>
__device__ void boundary_worker(const GemmParams& P, int lane, volatile int* abort_flag) {
  const BoundaryArgs& B = P.bnd;
  const int M = P.M;
  const int tiles_n = P.N / P.bn;
  int* claim = B.count + ((M + 255) / 256) * 8;
  const int n_items = (M + BND_ITEM_ROWS - 1) / BND_ITEM_ROWS;
  for (;;) {
    int item = 0;
    if (lane == 0) item = atomicAdd(claim, 1);
    item = __shfl_sync(0xFFFFFFFFu, item, 0);
    if (item >= n_items) return;
    const int row0 = item * BND_ITEM_ROWS;
    const int row1 = min(row0 + 1, M - 1);
    const int* cnt = B.count + (row0 >> 5);
    int ok = 1;
    if (lane == 0 && ld_acquire_gpu(cnt) < tiles_n) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(cnt) < tiles_n) {
        __nanosleep(256);
        if (*abort_flag) { ok = 0; break; }
        if (globaltimer_ns() - t0 > P.timeout_ns) {
          report_error(P.status, ST_TIMEOUT, WAIT_BOUNDARY_ROWS);
          *abort_flag = 1;
          ok = 0;
          break;
        }
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) return;
    (void)ld_acquire_gpu(cnt);     // each lane acquires the block's stores
    boundary_rows<XF, YF>(P, row0, row1, lane);
  }
}

__device__ __forceinline__ void boundary_worker_any(const GemmParams& P, int lane,
                                                    volatile int* abort_flag) {
  const bool yf = P.out_fmt == OUT_F32;
  if (P.bnd.x_f32) {
    if (yf) boundary_worker<true, true>(P, lane, abort_flag);
    else boundary_worker<true, false>(P, lane, abort_flag);
  } else {
    if (yf) boundary_worker<false, true>(P, lane, abort_flag);
    else boundary_worker<false, false>(P, lane, abort_flag);
  }
}

template <int EPI>
constexpr int pair_threads() { return EPI == EPI_BOUNDARY ? BND_THREADS : GEMM_THREADS; }

template <int KIND, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads<EPI>(), 1)
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
  } else if (EPI == EPI_BOUNDARY && (warp == 2 || warp == 3 || warp >= 8)) {
    // ---------------- boundary row workers (both CTAs) ----------------
    boundary_worker_any(P, lane, abort_flag);
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
      constexpr int EPI_T = EPI == EPI_BOUNDARY ? EPI_STORE : EPI;
      if (small) pair_small_epilogue<EPI_T>(P, tc, taddr, (q & 1) * 32 + lane, q >> 1);
      else if (P.out_box && tc.valid >= 32 * (q + 1))
        pair_epilogue_boxes<EPI_T>(P, tc, taddr, q, lane, &tmOut, boxes + q * PAIR_BOX);
      else gemm_epilogue<EPI_T>(P, tc, taddr, r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // the accumulator's loads have completed (tcgen05.wait::ld): no memory write has
        // to reach the leader, so the arrive needs no cluster-scope release
        if (leader) mbar_arrive(&S->tempty[acc]);
        else mbar_arrive_cluster(mapa_shared(smem_u32(&S->tempty[acc]), 0));
      }
      if constexpr (EPI == EPI_BOUNDARY) {
        // this warp's 32 rows of the tile (values and sums of squares) are stored: make
        // the stores visible GPU-wide, then count the tile for the row workers
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          tma_store_wait_all();
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          red_release_gpu_add(P.bnd.count + (tc.a_row >> 5) + q, 1);
        }
        __syncwarp();
      }
    }
    if (lane == 0) tma_store_wait_all();   // the box stores have landed
    if constexpr (EPI == EPI_BOUNDARY) boundary_worker_any(P, lane, abort_flag);
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
