// gemm_tcgen05.cuh -- persistent tcgen05/TMEM GEMM, D[m,n] = sum_k A[m,k] * B[n,k],
// both operands K-major, fed by TMA, for every projection of the latent-MoE block:
//
//   router  h32 [T,d] x W_r [E,d]          TF32, epilogue = top-k + renormalised softmax
//   pooler  h16 [T,d] x W_pool [p,d]        FP16, epilogue = FP32 store
//   gate/up A_perm [Tk,p] x W13_e [2I,p]    FP16, grouped by expert, epilogue = SwiGLU
//   down    s [Tk,I] x W2_e [p,I]           BF16, grouped by expert, epilogue = FP32 store
//   unpool  c [T,p] x W_unpool [d,p]        FP16, epilogue = store
// (FP32 configurations run every projection on TF32 operands.)
//
// ("SGLang and Miles Add Day-0 Support for Muse Spark Open": section "MoE with Pooler,
// Unpooler and Per-Expert Normalization" for the steps; "Kernel Optimizations" for the
// grouped expert GEMM that computes only routed work and the top-k on CUDA.)
//
// One CTA per SM walks a static tile list.  Warp roles:
//   warp 0 (one lane)  TMA producer: A and B 128-byte-swizzled K-slices into a
//                      STAGES-deep shared-memory ring (full/empty mbarriers)
//   warp 1 (one lane)  MMA issuer: 4 x tcgen05.mma (M=128, N=bn, K=32 bytes) per slice
//                      into one of two TMEM accumulators (2 x 256 columns)
//   warp 2             allocates / frees the 512 TMEM columns
//   warps 4..7         epilogue: thread i owns accumulator row i (TMEM lane i), loads
//                      16 columns at a time with tcgen05.ld and writes the result
// The double-buffered accumulator lets the epilogue of tile i overlap the MMAs of i+1.
#pragma once

#include "common.cuh"

namespace lmoe {

constexpr int GEMM_BM = 128;
constexpr int GEMM_BN_MAX = 256;
constexpr int GEMM_STAGES = 4;
constexpr int GEMM_THREADS = 256;
constexpr int GEMM_A_STAGE = GEMM_BM * 128;      // 16 KB: 128 rows x 128 B
constexpr int GEMM_B_STAGE = GEMM_BN_MAX * 128;  // 32 KB: up to 256 rows x 128 B
constexpr int GEMM_MAX_GROUPS = 256;
constexpr int GEMM_TMEM_COLS = 512;
constexpr int ROUTER_MAX_K = 8;

// EPI_BOUNDARY: EPI_STORE plus the block boundary's row pass (CTA-pair kernel only)
enum EpiKind : int { EPI_ROUTER = 0, EPI_STORE = 1, EPI_SWIGLU = 2, EPI_BOUNDARY = 3 };
// Operand kinds; the values of the first three are the instruction-descriptor format
// codes of kind::f16 / kind::tf32.  OP_NVF4: packed E2M1 operands (gemm_nvf4.cuh).
enum OpKind : int { OP_F16 = 0, OP_BF16 = 1, OP_TF32 = 2, OP_NVF4 = 3 };

// The block boundary fused into the unpooler (gemm_pair_kernel<KIND, EPI_BOUNDARY>):
// the residual stream, the gains and gate of the two norms, the row pass's outputs, and
// the counters through which the tile epilogues tell the row workers that a 32-row block
// of the output is stored in full.
struct BoundaryArgs {
  const void* x;         // [M, N] residual stream entering the block (act type)
  void* x_out;           // [M, N] x + gate * RMSNorm_{g_post}(out); may be x
  void* h_next;          // [M, N] RMSNorm_{g_next}(x_out)
  const float* g_post;
  const float* gate;     // NULL: plain residual
  const float* g_next;
  int* count;            // [8 * ceil(M / 256)] tiles stored per 32-row block, then one
                         // item counter; zero before the launch
  float eps;
  int x_f32;             // residual stream in FP32 (else BF16)
};

struct GemmParams {
  int M;        // dense: rows of A and of the output
  int N;        // output columns (dense) / columns per expert (grouped)
  int K;        // reduction length in elements
  int bn;       // tile width: multiple of 16, <= 256
  int groups;   // 0 = dense; > 0 = grouped over this many experts
  int ksplit;   // dense only: K is split into this many slices (1 = no split); slice s
                // writes its FP32 partial at out + s * split_stride
  size_t split_stride;
  const int* row_off;  // grouped: [groups+1] first A row of each expert (device)
  const int* mt_off;   // grouped: [groups+1] prefix sum of 128-row tiles (device)
  const int* row_cnt;  // grouped: [groups] rows of each expert (device)
  int* status;
  unsigned long long timeout_ns;
  int debug_skip_first_load;  // test hook: never issue the first TMA load
  // epilogue
  void* out;
  int ld_out;
  int out_fmt;
  int E, top_k;         // router
  int32_t* ids;
  float* wts;
  // NVFP4 operands: chunked scale arrays of A and B, and FP32 scales applied to the
  // accumulator: row_scale[row] * grp_scale[e] (gate/up) or grp_scale[e] * out_scale[e]
  const uint8_t* sf_a;
  const uint8_t* sf_b;
  const float* row_scale;
  const float* grp_scale;
  const float* out_scale;   // requantisation global scale (gate/up) / extra factor (down)
  uint8_t* out_sf;          // requantised output: chunked scales (codes go to `out`)
  // expert outputs: per-row sums of squares of each 128-column block of the stored FP32
  // values, at row_ssq[row * (N / 128) + column / 128], each summed in column order
  // (the per-expert RMSNorm reads these instead of a second pass over the row)
  float* row_ssq;
  int out_box;   // CTA-pair kernels: 1 = write full 32-row blocks through the output's
                 // tensor map (the kernel's tmOut) instead of per-thread stores
  BoundaryArgs bnd;   // EPI_BOUNDARY only (its row_ssq: [M, N / 128] of the output)
  int b_const;   // dense: B is a weight, written before the forward began, so the first
                 // ring stages' B tiles are requested before the wait on the previous kernel
  int pad_rows;  // grouped on CTA pairs: the rows of a tile past the expert's last row lie
                 // in its zeroed padding; store them too (the zeros they compute to)
};

struct GemmSmem {
  uint64_t full[GEMM_STAGES];
  uint64_t empty[GEMM_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int mt_off[GEMM_MAX_GROUPS + 1];
  int row_off[GEMM_MAX_GROUPS + 1];
  int row_cnt[GEMM_MAX_GROUPS + 1];
};

constexpr size_t gemm_smem_bytes() {
  return 1024 /* alignment slack */ + size_t(GEMM_STAGES) * (GEMM_A_STAGE + GEMM_B_STAGE) +
         sizeof(GemmSmem);
}

struct TileCoord {
  int a_row;   // first A row (and output row) of the tile
  int b_row;   // first B row
  int valid;   // rows of the tile that belong to it (<= 128)
  int n_blk;   // tile index along N
  int e;       // expert (grouped), 0 for dense
  int split;   // K slice (dense split-K), 0 otherwise
};

__device__ __forceinline__ int gemm_num_tiles(const GemmParams& P, const GemmSmem* S) {
  const int nb = P.N / P.bn;
  if (P.groups == 0) return ((P.M + GEMM_BM - 1) / GEMM_BM) * nb * P.ksplit;
  return S->mt_off[P.groups] * nb;
}

// Tile t -> coordinates.  Grouped tiles run expert by expert, and inside an expert
// N-block by N-block, so the CTAs working at one time share one B tile through L2.
__device__ __forceinline__ TileCoord gemm_tile(const GemmParams& P, const GemmSmem* S, int t) {
  const int nb = P.N / P.bn;
  TileCoord c;
  if (P.groups == 0) {
    c.split = t % P.ksplit;          // consecutive tiles: the slices of one output tile
    const int o = t / P.ksplit;
    const int m_blk = o / nb;
    c.n_blk = o - m_blk * nb;
    c.a_row = m_blk * GEMM_BM;
    c.b_row = c.n_blk * P.bn;
    c.valid = min(GEMM_BM, P.M - c.a_row);
    c.e = 0;
    return c;
  }
  c.split = 0;
  // largest e with mt_off[e] * nb <= t (experts with no rows have empty ranges)
  int lo = 0, hi = P.groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S->mt_off[mid] * nb <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mt_e = S->mt_off[e + 1] - S->mt_off[e];
  const int local = t - S->mt_off[e] * nb;
  c.n_blk = local / mt_e;
  const int m_blk = local - c.n_blk * mt_e;
  c.a_row = S->row_off[e] + m_blk * GEMM_BM;
  c.b_row = e * P.N + c.n_blk * P.bn;
  c.valid = min(GEMM_BM, S->row_cnt[e] - m_blk * GEMM_BM);
  c.e = e;
  return c;
}

// ---- epilogue stores ------------------------------------------------------------------
__device__ __forceinline__ void store16(void* out, size_t idx, int fmt, const float (&v)[16]) {
  if (fmt == OUT_F16) {
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(out) + idx);
    uint4 a, b;
    a.x = pack_f16x2(v[0], v[1]);   a.y = pack_f16x2(v[2], v[3]);
    a.z = pack_f16x2(v[4], v[5]);   a.w = pack_f16x2(v[6], v[7]);
    b.x = pack_f16x2(v[8], v[9]);   b.y = pack_f16x2(v[10], v[11]);
    b.z = pack_f16x2(v[12], v[13]); b.w = pack_f16x2(v[14], v[15]);
    dst[0] = a;
    dst[1] = b;
  } else if (fmt == OUT_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + idx);
    uint4 a, b;
    a.x = pack_bf16x2(v[0], v[1]);   a.y = pack_bf16x2(v[2], v[3]);
    a.z = pack_bf16x2(v[4], v[5]);   a.w = pack_bf16x2(v[6], v[7]);
    b.x = pack_bf16x2(v[8], v[9]);   b.y = pack_bf16x2(v[10], v[11]);
    b.z = pack_bf16x2(v[12], v[13]); b.w = pack_bf16x2(v[14], v[15]);
    dst[0] = a;
    dst[1] = b;
  } else {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + idx);
    float w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = (fmt == OUT_TF32) ? tf32_rna(v[i]) : v[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

// Insert (v, e) into a descending list of K entries.  Strict comparison: an equal
// logit never displaces an earlier (lower) expert id.
__device__ __forceinline__ void topk_insert(float (&val)[ROUTER_MAX_K], int (&id)[ROUTER_MAX_K],
                                            int k, float v, int e) {
#pragma unroll
  for (int j = 0; j < ROUTER_MAX_K; ++j) {
    if (j < k && v > val[j]) {
      const float tv = val[j];
      const int te = id[j];
      val[j] = v;
      id[j] = e;
      v = tv;
      e = te;
    }
  }
}

template <int EPI>
__device__ __forceinline__ void gemm_epilogue(const GemmParams& P, const TileCoord& tc,
                                              uint32_t taddr, int r) {
  const bool row_ok = r < tc.valid;
  const size_t row = static_cast<size_t>(tc.a_row + r);
  if constexpr (EPI == EPI_STORE) {
    const size_t base = row * P.ld_out + static_cast<size_t>(tc.n_blk) * P.bn +
                        static_cast<size_t>(tc.split) * P.split_stride;
    float ss = 0.f;     // sum of squares of the current 128-column block (row_ssq)
    for (int c0 = 0; c0 < P.bn; c0 += 32) {    // bn is a multiple of 16
      const bool two = c0 + 16 < P.bn;          // uniform across the warp
      uint32_t a[16], b[16];
      tmem_ld16(taddr + c0, a);
      if (two) tmem_ld16(taddr + c0 + 16, b);
      tmem_ld_wait();
      float va[16], vb[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) { va[i] = __uint_as_float(a[i]); vb[i] = __uint_as_float(b[i]); }
      if (row_ok) {
        store16(P.out, base + c0, P.out_fmt, va);
        if (two) store16(P.out, base + c0 + 16, P.out_fmt, vb);
      }
      if (P.row_ssq) {          // expert outputs (bn is 128 or 256), squared as stored
        const int rb = P.out_fmt;
        ss = add_stored_squares(ss, va, rb);
        ss = add_stored_squares(ss, vb, rb);
        if (((c0 + 32) & 127) == 0) {
          if (row_ok)
            P.row_ssq[row * (P.N >> 7) + ((tc.n_blk * P.bn + c0) >> 7)] = ss;
          ss = 0.f;
        }
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // columns [0, bn/2) hold gate rows, [bn/2, bn) the matching up rows.  silu divides
    // with __fdividef (a few ulp of FP32, far below the BF16/TF32/NVFP4 storage of s):
    // the correctly rounded FP32 division made the NVFP4 gate/up epilogue the bound of
    // its GEMM (4.20 -> 2.81 ms at prefill, measured)
    const int half = P.bn >> 1;
    const size_t base = row * P.ld_out + static_cast<size_t>(tc.n_blk) * half;
    for (int c0 = 0; c0 < half; c0 += 16) {
      uint32_t g[16], u[16];
      tmem_ld16(taddr + c0, g);
      tmem_ld16(taddr + half + c0, u);
      tmem_ld_wait();
      float s[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = __uint_as_float(g[i]);
        const float b = __uint_as_float(u[i]);
        s[i] = __fdividef(a, 1.0f + __expf(-a)) * b;     // silu(a) * b
      }
      if (row_ok) store16(P.out, base + c0, P.out_fmt, s);
    }
  } else {  // EPI_ROUTER: logits of one token -> top-k ids and renormalised softmax
    float val[ROUTER_MAX_K];
    int id[ROUTER_MAX_K];
#pragma unroll
    for (int j = 0; j < ROUTER_MAX_K; ++j) { val[j] = -INFINITY; id[j] = 0; }
    const int k = P.top_k;
    for (int c0 = 0; c0 < P.bn; c0 += 16) {
      uint32_t a[16];
      tmem_ld16(taddr + c0, a);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int e = c0 + i;
        if (e < P.E) topk_insert(val, id, k, __uint_as_float(a[i]), e);
      }
    }
    if (row_ok) {
      float z[ROUTER_MAX_K];
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < ROUTER_MAX_K; ++j) {
        z[j] = (j < k) ? __expf(val[j] - val[0]) : 0.f;
        sum += z[j];
      }
      const float inv = 1.0f / sum;
#pragma unroll
      for (int j = 0; j < ROUTER_MAX_K; ++j) {
        if (j < k) {
          P.ids[row * k + j] = id[j];
          P.wts[row * k + j] = z[j] * inv;
        }
      }
    }
  }
}

template <int KIND, int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + GEMM_STAGES * GEMM_A_STAGE;
  GemmSmem* S = reinterpret_cast<GemmSmem*>(sB + GEMM_STAGES * GEMM_B_STAGE);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < GEMM_STAGES; ++s) {
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
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  // A weight operand does not depend on the kernels before this one: the producer puts
  // the B halves of the first ring stages in flight, and asks L2 for the rest of its first
  // tile's B, while the previous kernel is still running (at decode the projections and
  // the router stream their weights once, and the wait is most of their time).
  int preloaded = 0;
  if (P.b_const && P.groups == 0 && P.debug_skip_first_load == 0 && warp == 0 && lane == 0 &&
      static_cast<int>(blockIdx.x) < gemm_num_tiles(P, nullptr)) {
    constexpr int KB = KIND == OP_TF32 ? 32 : 64;
    const int kb0 = P.K / KB / P.ksplit;
    const TileCoord tc = gemm_tile(P, nullptr, static_cast<int>(blockIdx.x));
    preloaded = kb0 < GEMM_STAGES ? kb0 : GEMM_STAGES;
    for (int s = 0; s < preloaded; ++s) {
      mbar_arrive_expect_tx(&S->full[s], GEMM_A_STAGE + P.bn * 128);
      tma_load_2d(sB + s * GEMM_B_STAGE, &tmB, &S->full[s], (tc.split * kb0 + s) * KB, tc.b_row);
    }
    for (int kb = preloaded; kb < kb0; ++kb)
      tma_prefetch_l2_2d(&tmB, (tc.split * kb0 + kb) * KB, tc.b_row);
  }
  pdl_wait();          // the inputs and tables are the previous kernels' outputs
  pdl_allow_next();
  if (P.groups > 0) {
    for (int i = threadIdx.x; i <= P.groups; i += blockDim.x) {
      S->mt_off[i] = P.mt_off[i];
      S->row_off[i] = P.row_off[i];
      S->row_cnt[i] = P.row_cnt[i];
    }
  }
  if (warp == 2) tmem_alloc(&S->tmem_base, GEMM_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = S->tmem_base;
  const int num_tiles = gemm_num_tiles(P, S);
  constexpr bool TF32 = KIND == OP_TF32;
  const int kblocks = P.K / (TF32 ? 32 : 64) / (P.groups == 0 ? P.ksplit : 1);
  const uint64_t limit = P.timeout_ns;
  volatile int* abort_flag = &S->abort_flag;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    const uint32_t bytes = GEMM_A_STAGE + P.bn * 128;
    int stage = 0;
    uint32_t phase = 0;
    int last_phase[GEMM_STAGES];   // parity of the last load issued into each stage
#pragma unroll
    for (int s = 0; s < GEMM_STAGES; ++s) last_phase[s] = s < preloaded ? 0 : -1;
    bool skip = P.debug_skip_first_load != 0;
    for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
      const TileCoord tc = gemm_tile(P, S, t);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&S->empty[stage], phase ^ 1, abort_flag, P.status,
                               WAIT_PRODUCER_EMPTY, limit))
          goto producer_done;
        if (skip) {
          skip = false;   // test hook: this stage never fills, so the MMA wait runs out
        } else if (t == static_cast<int>(blockIdx.x) && kb < preloaded) {
          // B is in flight since before the wait; the stage's barrier already expects both
          const int kc = (tc.split * kblocks + kb) * (TF32 ? 32 : 64);
          tma_load_2d(sA + stage * GEMM_A_STAGE, &tmA, &S->full[stage], kc, tc.a_row);
          last_phase[stage] = static_cast<int>(phase);
        } else {
          mbar_arrive_expect_tx(&S->full[stage], bytes);
          const int kc = (tc.split * kblocks + kb) * (TF32 ? 32 : 64);
          tma_load_2d(sA + stage * GEMM_A_STAGE, &tmA, &S->full[stage], kc, tc.a_row);
          tma_load_2d(sB + stage * GEMM_B_STAGE, &tmB, &S->full[stage], kc, tc.b_row);
          last_phase[stage] = static_cast<int>(phase);
        }
        if (++stage == GEMM_STAGES) { stage = 0; phase ^= 1; }
      }
    }
  producer_done:
    if (*abort_flag) {
      // Never leave a copy in flight: the last load issued into each stage completes
      // that stage's phase when it lands (nothing else arrives on it any more).
      volatile int never = 0;
      for (int s = 0; s < GEMM_STAGES; ++s)
        if (last_phase[s] >= 0)
          mbar_wait_bounded(&S->full[s], static_cast<uint32_t>(last_phase[s]), &never, nullptr,
                            WAIT_DRAIN, limit);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = idesc_f32acc(static_cast<uint32_t>(KIND), GEMM_BM, P.bn);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
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
        const uint32_t a0 = smem_u32(sA + stage * GEMM_A_STAGE);
        const uint32_t b0 = smem_u32(sB + stage * GEMM_B_STAGE);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          mma_issue<TF32>(d_tmem, sdesc_sw128(a0 + 32 * k), sdesc_sw128(b0 + 32 * k), idesc,
                          (kb | k) != 0);
        }
        mma_commit(&S->empty[stage]);
        if (++stage == GEMM_STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      mma_commit(&S->tfull[acc]);
    }
    // all MMAs this thread issued have completed once `drain` flips
    mma_commit(&S->drain);
    {
      volatile int never = 0;
      mbar_wait_bounded(&S->drain, 0, &never, P.status, WAIT_DRAIN, limit);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int r = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(&S->tfull[acc], acc_phase, abort_flag, P.status,
                             WAIT_EPI_TMEM_FULL, limit))
        break;
      tc_fence_after();
      const TileCoord tc = gemm_tile(P, S, t);
      const uint32_t taddr = tmem_base + acc * GEMM_BN_MAX + (static_cast<uint32_t>(q * 32) << 16);
      gemm_epilogue<EPI>(P, tc, taddr, r);
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
