// gemm_swap.cuh -- grouped expert GEMMs with the weights on the MMA's M side and the
// expert's tokens on N ("swap AB"), for the BF16/FP16 and TF32 expert paths.
//
// With tokens on M, the last 128-row tile of every expert is partly empty (about 12 % of
// the MMA work at ~512 rows per expert).  On the N side the tile width can shrink to
// the tokens present, rounded up to 16, so the MMA work follows the routed work:
//
//   gate/up   W13 block [256 rows = 128 gate + 128 up] x tokens [TN = 128]:
//             two M = 128 MMAs per K step into two TMEM accumulators (gate, up),
//             epilogue: thread i owns feature i of the block, s[token][f] = silu(g) * u
//   down      W2 block [128 rows of p] x tokens [TN = 256], epilogue y[token][f] (FP32)
//
// Pipeline as in gemm_tcgen05.cuh: TMA producer warp (weight tile + token tile per
// 128-byte K slice, 4 stages of 48 KB), one MMA-issuing thread, double-buffered TMEM
// accumulators (2 x 256 columns), four epilogue warps, every wait bounded.
#pragma once

#include "gemm_tcgen05.cuh"

namespace lmoe {

enum SwapEpi : int { SWAP_SWIGLU = 0, SWAP_STORE = 1 };

constexpr int SWAP_STAGE = 384 * 128;   // weight rows + token rows, 128 bytes each
constexpr int SWAP_STAGES = 4;

template <int EPI>
struct SwapShape {
  static constexpr int W_ROWS = EPI == SWAP_SWIGLU ? 256 : 128;   // weight rows per tile
  static constexpr int TN = EPI == SWAP_SWIGLU ? 128 : 256;       // tokens per tile
};

constexpr size_t swap_smem_bytes() {
  return 1024 + size_t(SWAP_STAGES) * SWAP_STAGE + sizeof(GemmSmem);
}

struct SwapTile {
  int tok_row;   // first dispatched row (token) of the tile
  int w_row;     // first weight row
  int valid;     // tokens of the tile (<= TN)
  int w_blk;     // weight block index within the expert
  int e;
};

// Tile t -> (expert, weight block, token block); expert by expert, and inside an expert
// weight block by weight block, so CTAs in flight share a weight tile through L2.
template <int EPI>
__device__ __forceinline__ SwapTile swap_tile(const GemmParams& P, const GemmSmem* S, int t) {
  constexpr int TN = SwapShape<EPI>::TN;
  constexpr int WR = SwapShape<EPI>::W_ROWS;
  const int nw = P.N / WR;
  int lo = 0, hi = P.groups - 1;
  while (lo < hi) {   // largest e with tile_off[e] <= t, tile_off[e] = mt_off[e] * nw
    const int mid = (lo + hi + 1) >> 1;
    if (S->mt_off[mid] * nw <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int nt_e = S->mt_off[e + 1] - S->mt_off[e];
  const int local = t - S->mt_off[e] * nw;
  SwapTile c;
  c.w_blk = local / nt_e;
  const int j = local - c.w_blk * nt_e;
  c.tok_row = S->row_off[e] + j * TN;
  c.valid = min(TN, S->row_cnt[e] - j * TN);
  c.w_row = e * P.N + c.w_blk * WR;
  c.e = e;
  return c;
}

template <int EPI>
__device__ __forceinline__ void swap_epilogue(const GemmParams& P, const SwapTile& tc,
                                              uint32_t taddr, int i) {
  const int f = tc.w_blk * 128 + i;       // output feature owned by this thread
  if constexpr (EPI == SWAP_SWIGLU) {
    for (int c0 = 0; c0 < tc.valid; c0 += 16) {
      uint32_t g[16], u[16];
      tmem_ld16(taddr + c0, g);
      tmem_ld16(taddr + 128 + c0, u);
      tmem_ld_wait();
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        if (c0 + jj < tc.valid) {
          const float a = __uint_as_float(g[jj]);
          const float b = __uint_as_float(u[jj]);
          const float s = __fdividef(a, 1.0f + __expf(-a)) * b;      // silu(a) * b
          const size_t idx = static_cast<size_t>(tc.tok_row + c0 + jj) * P.ld_out + f;
          if (P.out_fmt == OUT_F16)
            reinterpret_cast<__half*>(P.out)[idx] = __float2half_rn(s);
          else if (P.out_fmt == OUT_BF16)
            reinterpret_cast<__nv_bfloat16*>(P.out)[idx] = __float2bfloat16_rn(s);
          else
            reinterpret_cast<float*>(P.out)[idx] = tf32_rna(s);
        }
      }
    }
  } else {
    for (int c0 = 0; c0 < tc.valid; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(taddr + c0, v);
      tmem_ld_wait();
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        if (c0 + jj < tc.valid) {
          const size_t idx = static_cast<size_t>(tc.tok_row + c0 + jj) * P.ld_out + f;
          if (P.out_fmt == OUT_F16)
            reinterpret_cast<__half*>(P.out)[idx] = __float2half_rn(__uint_as_float(v[jj]));
          else if (P.out_fmt == OUT_BF16)
            reinterpret_cast<__nv_bfloat16*>(P.out)[idx] = __float2bfloat16_rn(__uint_as_float(v[jj]));
          else
            reinterpret_cast<float*>(P.out)[idx] = __uint_as_float(v[jj]);
        }
      }
    }
  }
}

template <int KIND, int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmX, const GemmParams P) {
  constexpr int WR = SwapShape<EPI>::W_ROWS;
  constexpr int TN = SwapShape<EPI>::TN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  GemmSmem* S = reinterpret_cast<GemmSmem*>(smem + SWAP_STAGES * SWAP_STAGE);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SWAP_STAGES; ++s) {
      mbar_init(&S->full[s], 1);
      mbar_init(&S->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&S->tfull[a], 1);
      mbar_init(&S->tempty[a], 4);
    }
    mbar_init(&S->drain, 1);
    S->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  pdl_wait();          // the inputs and tables are the previous kernels' outputs
  pdl_allow_next();
  for (int i = threadIdx.x; i <= P.groups; i += blockDim.x) {
    S->mt_off[i] = P.mt_off[i];    // token tiles (of TN) per expert, prefix sums
    S->row_off[i] = P.row_off[i];
    S->row_cnt[i] = P.row_cnt[i];
  }
  if (warp == 2) tmem_alloc(&S->tmem_base, GEMM_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  constexpr bool TF32 = KIND == OP_TF32;
  const uint32_t tmem_base = S->tmem_base;
  const int num_tiles = S->mt_off[P.groups] * (P.N / WR);
  const int kblocks = P.K / (TF32 ? 32 : 64);
  const uint64_t limit = P.timeout_ns;
  volatile int* abort_flag = &S->abort_flag;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: weight tile, then token tile ----------------
    const uint32_t bytes = (WR + TN) * 128;
    int stage = 0;
    uint32_t phase = 0;
    int last_phase[SWAP_STAGES];
#pragma unroll
    for (int s = 0; s < SWAP_STAGES; ++s) last_phase[s] = -1;
    bool skip = P.debug_skip_first_load != 0;
    for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
      const SwapTile tc = swap_tile<EPI>(P, S, t);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&S->empty[stage], phase ^ 1, abort_flag, P.status,
                               WAIT_PRODUCER_EMPTY, limit))
          goto producer_done;
        if (skip) {
          skip = false;   // test hook: this stage never fills, so the MMA wait runs out
        } else {
          mbar_arrive_expect_tx(&S->full[stage], bytes);
          const int kc = kb * (TF32 ? 32 : 64);
          uint8_t* st = smem + stage * SWAP_STAGE;
          tma_load_2d(st, &tmW, &S->full[stage], kc, tc.w_row);
          tma_load_2d(st + WR * 128, &tmX, &S->full[stage], kc, tc.tok_row);
          last_phase[stage] = static_cast<int>(phase);
        }
        if (++stage == SWAP_STAGES) { stage = 0; phase ^= 1; }
      }
    }
  producer_done:
    if (*abort_flag) {
      volatile int never = 0;
      for (int s = 0; s < SWAP_STAGES; ++s)
        if (last_phase[s] >= 0)
          mbar_wait_bounded(&S->full[s], static_cast<uint32_t>(last_phase[s]), &never, nullptr,
                            WAIT_DRAIN, limit);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const SwapTile tc = swap_tile<EPI>(P, S, t);
      const uint32_t n_mma = static_cast<uint32_t>((tc.valid + 15) & ~15);
      const uint32_t idesc = idesc_f32acc(static_cast<uint32_t>(KIND), GEMM_BM, n_mma);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(&S->tempty[acc], acc_phase ^ 1, abort_flag, P.status,
                             WAIT_MMA_TMEM_EMPTY, limit))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * 256;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&S->full[stage], phase, abort_flag, P.status, WAIT_MMA_FULL,
                               limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t w0 = smem_u32(smem + stage * SWAP_STAGE);
        const uint32_t x0 = w0 + WR * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t xd = sdesc_sw128(x0 + 32 * k);
          mma_issue<TF32>(d_tmem, sdesc_sw128(w0 + 32 * k), xd, idesc, (kb | k) != 0);
          if constexpr (EPI == SWAP_SWIGLU)   // up rows: the second 128 weight rows
            mma_issue<TF32>(d_tmem + 128, sdesc_sw128(w0 + 128 * 128 + 32 * k), xd, idesc,
                            (kb | k) != 0);
        }
        mma_commit(&S->empty[stage]);
        if (++stage == SWAP_STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit(&S->tfull[acc]);
    }
    mma_commit(&S->drain);
    {
      volatile int never = 0;
      mbar_wait_bounded(&S->drain, 0, &never, P.status, WAIT_DRAIN, limit);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue: thread i <-> weight row (feature) i ----------------
    const int q = warp & 3;
    const int i = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(&S->tfull[acc], acc_phase, abort_flag, P.status,
                             WAIT_EPI_TMEM_FULL, limit))
        break;
      tc_fence_after();
      const SwapTile tc = swap_tile<EPI>(P, S, t);
      const uint32_t taddr = tmem_base + acc * 256 + (static_cast<uint32_t>(q * 32) << 16);
      swap_epilogue<EPI>(P, tc, taddr, i);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S->tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, GEMM_TMEM_COLS);
  }
}

}  // namespace lmoe
