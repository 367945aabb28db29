// kernels_mem.cuh -- the memory-bound steps of the latent-MoE block:
//   norm_in        full-width RMSNorm of x -> h32 (TF32-rounded FP32, router operand)
//                  and h16 (FP16, pooler operand)
//   dispatch       histogram of expert ids -> per-expert row offsets -> stable
//                  counting-sort positions (token-major order) and the inverse map
//   pool_permute   RMSNorm of the pooled row, cast, written to the k permuted rows
//                  of the expert GEMM input
//   combine        per-expert RMSNorm of each selected expert output, times its route
//                  weight, summed in FP32 in slot order
//   pack           gate/up interleave and weight conversion (BF16 -> FP16, or TF32
//                  rounding for FP32 configurations)
// ("SGLang and Miles Add Day-0 Support for Muse Spark Open": section "MoE with Pooler,
// Unpooler and Per-Expert Normalization"; "The Fused Post-per-expert Norm" for the
// combine; "Kernel Optimizations" for the norm fused into the boundary kernel and the
// packed routing output.)
#pragma once

#include "common.cuh"

namespace lmoe {

constexpr int MEM_THREADS = 256;
constexpr int DISPATCH_CHUNK = 2048;   // (token, slot) pairs per counting-sort chunk
constexpr int MAX_TOPK = 8;

// Sum over the block; every thread gets the result.  `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = (l < (blockDim.x >> 5)) ? red[l] : 0.f;
  s = warp_sum(s);
  return s;
}

// ---- full-width RMSNorm ---------------------------------------------------------------
// One block per token.  Pass 1 sums squares; pass 2 re-reads the row (L1-resident) and
// writes h = x * rsqrt(mean(x^2) + eps) * g twice: TF32-rounded FP32 and FP16 (h16 may be
// null: router-only calls).  |h_i| <= sqrt(d) * max|g| (e.g. 91 * 1.5 at d = 8192) keeps
// h inside FP16 for gains of ordinary size; a row that is not finite, or an h16 value
// above the FP16 maximum (very large gains), is reported as CHECK_H_RANGE.
template <bool ACT_F32>
__global__ void __launch_bounds__(MEM_THREADS)
    norm_in_kernel(const void* __restrict__ x, const float* __restrict__ g,
                   float* __restrict__ h32, __half* __restrict__ h16, int d, float eps,
                   int* status) {
  pdl_wait();
  pdl_allow_next();
  __shared__ float red[32];
  const size_t t = blockIdx.x;
  const int nchunk = d >> 3;  // 8 elements per chunk
  float ss = 0.f;
  for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
    float v[8];
    if constexpr (ACT_F32) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(x) + t * d) + 2 * c;
      const float4 a = src[0], b = src[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
      const uint4 a = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + t * d)[c];
      float2 f;
      f = unpack_bf16x2(a.x); v[0] = f.x; v[1] = f.y;
      f = unpack_bf16x2(a.y); v[2] = f.x; v[3] = f.y;
      f = unpack_bf16x2(a.z); v[4] = f.x; v[5] = f.y;
      f = unpack_bf16x2(a.w); v[6] = f.x; v[7] = f.y;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
  }
  const float total = block_sum(ss, red);
  const float rs = rsqrtf(total / static_cast<float>(d) + eps);
  float hmax = 0.f;
  for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
    float v[8];
    if constexpr (ACT_F32) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(x) + t * d) + 2 * c;
      const float4 a = src[0], b = src[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
      const uint4 a = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + t * d)[c];
      float2 f;
      f = unpack_bf16x2(a.x); v[0] = f.x; v[1] = f.y;
      f = unpack_bf16x2(a.y); v[2] = f.x; v[3] = f.y;
      f = unpack_bf16x2(a.z); v[4] = f.x; v[5] = f.y;
      f = unpack_bf16x2(a.w); v[6] = f.x; v[7] = f.y;
    }
    const float4 g0 = reinterpret_cast<const float4*>(g)[2 * c];
    const float4 g1 = reinterpret_cast<const float4*>(g)[2 * c + 1];
    const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = v[i] * rs * gg[i];
    float4* o32 = reinterpret_cast<float4*>(h32 + t * d) + 2 * c;
    o32[0] = make_float4(tf32_rna(h[0]), tf32_rna(h[1]), tf32_rna(h[2]), tf32_rna(h[3]));
    o32[1] = make_float4(tf32_rna(h[4]), tf32_rna(h[5]), tf32_rna(h[6]), tf32_rna(h[7]));
    if constexpr (!ACT_F32) {
      if (h16 != nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) hmax = fmaxf(hmax, fabsf(h[i]));
        uint4 o;
        o.x = pack_f16x2(h[0], h[1]); o.y = pack_f16x2(h[2], h[3]);
        o.z = pack_f16x2(h[4], h[5]); o.w = pack_f16x2(h[6], h[7]);
        reinterpret_cast<uint4*>(h16 + t * d)[c] = o;
      }
    }
  }
  // total is the same in every thread: a non-finite row is reported once, by thread 0
  if ((threadIdx.x == 0 && !(fabsf(total) < INFINITY)) || !(hmax <= F16_MAX))
    report_error(status, ST_DEVICE_CHECK, CHECK_H_RANGE);
}

// ---- dispatch: counting sort of (token, slot) pairs by expert -------------------------
// 1) per-chunk histograms.  Ids outside [0, E) are counted nowhere and reported.
__global__ void __launch_bounds__(MEM_THREADS)
    dispatch_hist_kernel(const int32_t* __restrict__ ids, int n, int E,
                         int* __restrict__ chunk_counts, int* status) {
  pdl_wait();
  pdl_allow_next();
  __shared__ int hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * DISPATCH_CHUNK;
  const int end = min(base + DISPATCH_CHUNK, n);
  for (int i = base + threadIdx.x; i < end; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else report_error(status, ST_DEVICE_CHECK, CHECK_EXPERT_ID);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[blockIdx.x * E + e] = hist[e];
}

// exclusive scan over the block (blockDim = 256); returns the prefix, *total = sum
__device__ __forceinline__ int block_excl_scan(int v, int* sh, int* total) {
  const int l = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (l >= o) x += y;
  }
  __syncthreads();
  if (l == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = (l < (blockDim.x >> 5)) ? sh[l] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (l >= o) s += y;
    }
    if (l < (blockDim.x >> 5)) sh[l] = s;   // inclusive warp totals
  }
  __syncthreads();
  const int warp_prefix = (w > 0) ? sh[w - 1] : 0;
  *total = sh[(blockDim.x >> 5) - 1];
  return warp_prefix + x - v;
}

// 2) one block: chunk bases per expert, expert row offsets, row counts and 128-row tile
// offsets.  padded != 0 starts every expert's rows on a 128-row boundary (row_off[e] =
// 128 * mt_off[e]), so no 128-row tile spans two experts.
__global__ void __launch_bounds__(256)
    dispatch_scan_kernel(int* __restrict__ chunk_counts, int nchunks, int E,
                         int* __restrict__ row_off, int* __restrict__ mt_off,
                         int* __restrict__ mt2_off, int* __restrict__ row_cnt, int padded) {
  pdl_wait();
  pdl_allow_next();
  __shared__ int sh[32];
  const int e = threadIdx.x;
  int running = 0;
  if (e < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = chunk_counts[c * E + e];
      chunk_counts[c * E + e] = running;
      running += v;
    }
  }
  int total;
  const int off = block_excl_scan(e < E ? running : 0, sh, &total);
  const int mt = (e < E) ? (running + 127) / 128 : 0;
  int mt_total;
  const int mto = block_excl_scan(mt, sh, &mt_total);
  const int mt2 = (e < E) ? (running + 255) / 256 : 0;    // 256-row tiles
  int mt2_total;
  const int mt2o = block_excl_scan(mt2, sh, &mt2_total);
  const int start = padded ? mto * 128 : off;
  if (e < E) {
    row_off[e] = start;
    mt_off[e] = mto;
    mt2_off[e] = mt2o;
    row_cnt[e] = running;
    for (int c = 0; c < nchunks; ++c) chunk_counts[c * E + e] += start;
  }
  if (e == 0) {
    row_off[E] = padded ? mt_total * 128 : total;
    mt_off[E] = mt_total;
    mt2_off[E] = mt2_total;
    row_cnt[E] = total;
  }
}

// 3) one warp per chunk: stable positions in (token, slot) order.  Lanes holding the
// same expert rank themselves by lane order; chunks and rounds run in order, so the
// rows of each expert keep token order.
__global__ void __launch_bounds__(32)
    dispatch_scatter_kernel(const int32_t* __restrict__ ids, int n, int E,
                            const int* __restrict__ chunk_base, int* __restrict__ inv,
                            int* __restrict__ src) {
  pdl_wait();
  pdl_allow_next();
  __shared__ int cnt[256];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cnt[e] = chunk_base[blockIdx.x * E + e];
  __syncwarp();
  const int base = blockIdx.x * DISPATCH_CHUNK;
  const int end = min(base + DISPATCH_CHUNK, n);
  const unsigned lt = (1u << lane) - 1u;
  for (int i0 = base; i0 < end; i0 += 32) {
    const int i = i0 + lane;
    int e = (i < end) ? ids[i] : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & lt);
    const int pos0 = (e >= 0) ? cnt[e] : 0;
    __syncwarp();
    if (e >= 0 && (__ffs(peers) - 1) == lane) cnt[e] = pos0 + __popc(peers);
    __syncwarp();
    if (i < end) {
      if (e >= 0) {
        const int pos = pos0 + rank;
        inv[i] = pos;
        src[pos] = i;
      } else {
        inv[i] = -1;
      }
    }
  }
}

// The three dispatch steps in one block, for batches of at most DISPATCH_CHUNK (token,
// slot) pairs (decode): counts in shared memory, the scan of dispatch_scan_kernel with
// one chunk, then warp 0 places the pairs in (token, slot) order as
// dispatch_scatter_kernel does.  Same maps as the three kernels.
__global__ void __launch_bounds__(256)
    dispatch_small_kernel(const int32_t* __restrict__ ids, int n, int E,
                          int* __restrict__ row_off, int* __restrict__ mt_off,
                          int* __restrict__ mt2_off, int* __restrict__ row_cnt,
                          int* __restrict__ inv, int* __restrict__ src, int padded,
                          int* status) {
  pdl_wait();
  pdl_allow_next();
  __shared__ int cnt[256];
  __shared__ int sh[32];
  const int e = threadIdx.x;
  if (e < 256) cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int id = ids[i];
    if (id >= 0 && id < E) atomicAdd(&cnt[id], 1);
    else report_error(status, ST_DEVICE_CHECK, CHECK_EXPERT_ID);
  }
  __syncthreads();
  const int running = e < E ? cnt[e] : 0;
  int total;
  const int off = block_excl_scan(running, sh, &total);
  int mt_total;
  const int mto = block_excl_scan(e < E ? (running + 127) / 128 : 0, sh, &mt_total);
  int mt2_total;
  const int mt2o = block_excl_scan(e < E ? (running + 255) / 256 : 0, sh, &mt2_total);
  const int start = padded ? mto * 128 : off;
  if (e < E) {
    row_off[e] = start;
    mt_off[e] = mto;
    mt2_off[e] = mt2o;
    row_cnt[e] = running;
  }
  if (e == 0) {
    row_off[E] = padded ? mt_total * 128 : total;
    mt_off[E] = mt_total;
    mt2_off[E] = mt2_total;
    row_cnt[E] = total;
  }
  __syncthreads();                       // every thread has read its count
  if (e < E) cnt[e] = start;             // next free position of each expert
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const unsigned lt = (1u << lane) - 1u;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    int id = (i < n) ? ids[i] : -1;
    if (id >= E) id = -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, id);
    const int rank = __popc(peers & lt);
    const int pos0 = (id >= 0) ? cnt[id] : 0;
    __syncwarp();
    if (id >= 0 && (__ffs(peers) - 1) == lane) cnt[id] = pos0 + __popc(peers);
    __syncwarp();
    if (i < n) {
      if (id >= 0) {
        const int pos = pos0 + rank;
        inv[i] = pos;
        src[pos] = i;
      } else {
        inv[i] = -1;
      }
    }
  }
}

// ---- pooled-input RMSNorm + cast + permute ---------------------------------------------
// One block per token: u = pooled * rsqrt(mean(pooled^2) + eps) * g_pool, written in the
// GEMM operand format (FP16, or TF32-rounded FP32) to the token's k dispatched rows.
// |u_i| <= sqrt(p) * max|g_pool| keeps u inside FP16 for gains of ordinary size; a row
// that is not finite, or an FP16 value above its maximum, is reported as CHECK_U_RANGE.
template <bool OUT_F32>
__global__ void __launch_bounds__(MEM_THREADS)
    pool_permute_kernel(const float* __restrict__ pooled, const float* __restrict__ g,
                        const int* __restrict__ inv, void* __restrict__ a_perm, int p, int k,
                        float eps, int* status, const int* __restrict__ row_off,
                        const int* __restrict__ row_cnt, int zero_blocks) {
  pdl_wait();
  pdl_allow_next();
  if (blockIdx.x < static_cast<unsigned>(zero_blocks)) {
    // blocks 4e .. 4e+3: a quarter each of expert e's padding rows (its rows start on
    // 128-row boundaries), written as zeros, so the grouped GEMMs' tiles that run past the
    // expert's last row multiply zeros: the same results, and far less switching power in
    // the tensor cores, which under the power cap buys clock
    const int e = static_cast<int>(blockIdx.x) >> 2, part = static_cast<int>(blockIdx.x) & 3;
    const size_t es = OUT_F32 ? 4 : 2;
    const size_t r0 = static_cast<size_t>(row_off[e]) + row_cnt[e];
    const size_t n16 = (static_cast<size_t>(row_off[e + 1]) - r0) * p * es / 16;
    const size_t q = (n16 + 3) / 4;
    const size_t i0 = part * q, i1 = n16 < i0 + q ? n16 : i0 + q;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a_perm) + r0 * p * es);
    for (size_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  __shared__ float red[32];
  __shared__ int rows[MAX_TOPK];
  const size_t t = blockIdx.x - zero_blocks;
  if (threadIdx.x < k) rows[threadIdx.x] = inv[t * k + threadIdx.x];
  const int nchunk = p >> 3;
  constexpr int CPT = 4;  // chunks of 8 per thread: p <= 8192
  float v[CPT][8];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * MEM_THREADS;
    if (c < nchunk) {
      const float4* s = reinterpret_cast<const float4*>(pooled + t * p) + 2 * c;
      const float4 a = s[0], b = s[1];
      v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
      v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(v[j][i], v[j][i], ss);
    }
  }
  const float total = block_sum(ss, red);   // also orders rows[] before its use
  const float rs = rsqrtf(total / static_cast<float>(p) + eps);
  float umax = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * MEM_THREADS;
    if (c < nchunk) {
      const float4 g0 = reinterpret_cast<const float4*>(g)[2 * c];
      const float4 g1 = reinterpret_cast<const float4*>(g)[2 * c + 1];
      const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      float u[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = v[j][i] * rs * gg[i];
      if constexpr (OUT_F32) {
        const float4 o0 = make_float4(tf32_rna(u[0]), tf32_rna(u[1]), tf32_rna(u[2]), tf32_rna(u[3]));
        const float4 o1 = make_float4(tf32_rna(u[4]), tf32_rna(u[5]), tf32_rna(u[6]), tf32_rna(u[7]));
        for (int s = 0; s < k; ++s) {
          const int r = rows[s];
          if (r < 0) continue;
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a_perm) + size_t(r) * p) + 2 * c;
          dst[0] = o0;
          dst[1] = o1;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) umax = fmaxf(umax, fabsf(u[i]));
        uint4 o;
        o.x = pack_f16x2(u[0], u[1]); o.y = pack_f16x2(u[2], u[3]);
        o.z = pack_f16x2(u[4], u[5]); o.w = pack_f16x2(u[6], u[7]);
        for (int s = 0; s < k; ++s) {
          const int r = rows[s];
          if (r < 0) continue;
          reinterpret_cast<uint4*>(static_cast<__half*>(a_perm) + size_t(r) * p)[c] = o;
        }
      }
    }
  }
  if ((threadIdx.x == 0 && !(fabsf(total) < INFINITY)) || !(umax <= F16_MAX))
    report_error(status, ST_DEVICE_CHECK, CHECK_U_RANGE);
}

// ---- combine -----------------------------------------------------------------------
// One block per (token, slice of `cols` columns, at most 1024), 8 columns per thread.
// Expert output rows y are FP32, or FP16 when Y_F16 (BF16 and NVFP4 experts).  The down
// GEMM's epilogue left, for every stored expert output row, the sum of squares of each
// 128-column block (row_ssq, [rows, p / 128]).  Thread 0 bulk-copies the token's k row
// slices into shared memory while the warps form r_j = rsqrt(sum / p + eps) from row
// j's blocks (a fixed warp tree); then c = sum_j w_j * r_j * g_exp[e_j] * y_j is
// accumulated in FP32 in slot order j = 0..k-1 and stored as the unpooler's operand:
// FP16 (|c_i| <= sum_j |w_j| * sqrt(p) * max|g_exp|), or TF32-rounded FP32.  Blocks of
// 128 threads and 16 KB (BF16) let 13 of them, and so 13 tokens' copies, be resident
// per SM: measured on GB300 at 4.5 TB/s for the prefill chunk against 3.2 TB/s with
// 256-thread blocks of 4 columns per thread and 2.0-3.0 TB/s for persistent variants
// whose block- or warp-wide steps serialised the dependent reads.
constexpr int COMBINE_MAX_COLS = 1024;
constexpr int COMBINE_VEC = 8;                 // columns per thread

// Columns per block: the largest multiple of 128 that divides p, at most 1024.
inline int combine_cols(int p) {
  for (int c = COMBINE_MAX_COLS; c > 128; c -= 128)
    if (p % c == 0) return c;
  return 128;
}
inline int combine_threads(int cols) { return cols / COMBINE_VEC < 32 ? 32 : cols / COMBINE_VEC; }
inline size_t combine_smem_bytes(int cols, bool y_f16) {
  return size_t(MAX_TOPK) * cols * (y_f16 ? 2 : 4);
}

template <bool C_F32, bool Y_F16>
__global__ void __launch_bounds__(COMBINE_MAX_COLS / COMBINE_VEC)
    combine_kernel(const void* __restrict__ y, const float* __restrict__ row_ssq,
                   const int* __restrict__ inv, const int32_t* __restrict__ ids,
                   const float* __restrict__ wts, const float* __restrict__ g_exp,
                   void* __restrict__ c_out, int p, int cols, int k, int E, float eps,
                   int* status, unsigned long long timeout_ns) {
  pdl_wait();
  pdl_allow_next();
  extern __shared__ __align__(16) uint8_t cmb_smem[];
  __shared__ uint64_t landed;
  __shared__ float sj[MAX_TOPK];     // w_j * r_j
  __shared__ int srow[MAX_TOPK], seid[MAX_TOPK];
  constexpr int YB = Y_F16 ? 2 : 4;   // bytes per stored y value
  const int nq = p / cols;
  const size_t t = blockIdx.x / nq;
  const int col0 = static_cast<int>(blockIdx.x % nq) * cols;
  const uint32_t slice = static_cast<uint32_t>(cols) * YB;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (threadIdx.x < MAX_TOPK) {
    int r = -1, e = 0;
    if (static_cast<int>(threadIdx.x) < k) {
      const int id = ids[t * k + threadIdx.x];
      if (id >= 0 && id < E) { r = inv[t * k + threadIdx.x]; e = id; }
    }
    srow[threadIdx.x] = r;
    seid[threadIdx.x] = e;
  }
  if (threadIdx.x == 0) {
    mbar_init(&landed, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t bytes = 0;
    for (int j = 0; j < k; ++j) bytes += srow[j] >= 0 ? slice : 0;
    mbar_arrive_expect_tx(&landed, bytes);
    for (int j = 0; j < k; ++j)
      if (srow[j] >= 0)
        bulk_load(cmb_smem + j * slice,
                  static_cast<const uint8_t*>(y) + (size_t(srow[j]) * p + col0) * YB, slice,
                  &landed);
  }
  // slot j's 128-column sums of squares, added by a fixed warp tree (warp j mod warps)
  for (int j = w; j < k; j += static_cast<int>(blockDim.x >> 5)) {
    const int parts = p >> 7;
    const int r = srow[j];
    float ss = 0.f;
    if (r >= 0)
      for (int i = l; i < parts; i += 32) ss += row_ssq[size_t(r) * parts + i];
    ss = warp_sum(ss);
    if (l == 0) sj[j] = wts[t * k + j] * rsqrtf(ss / static_cast<float>(p) + eps);
  }
  {
    volatile int never = 0;
    mbar_wait_bounded(&landed, 0, &never, status, WAIT_COMBINE, timeout_ns);
  }
  __syncthreads();
  const int cl = COMBINE_VEC * threadIdx.x;    // this thread's first column of the slice
  if (cl >= cols) return;
  float acc[COMBINE_VEC];
#pragma unroll
  for (int i = 0; i < COMBINE_VEC; ++i) acc[i] = 0.f;
  for (int j = 0; j < k; ++j) {
    if (srow[j] < 0) continue;
    const uint8_t* src = cmb_smem + j * slice + cl * YB;
    float v[COMBINE_VEC];
    if constexpr (Y_F16) {
      const uint4 b = *reinterpret_cast<const uint4*>(src);
      const float2 f0 = unpack_f16x2(b.x), f1 = unpack_f16x2(b.y);
      const float2 f2 = unpack_f16x2(b.z), f3 = unpack_f16x2(b.w);
      v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
      v[4] = f2.x; v[5] = f2.y; v[6] = f3.x; v[7] = f3.y;
    } else {
      const float4 a = *reinterpret_cast<const float4*>(src);
      const float4 b = *reinterpret_cast<const float4*>(src + 16);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    const float* gp = g_exp + size_t(seid[j]) * p + col0 + cl;
    const float4 g0 = *reinterpret_cast<const float4*>(gp);
    const float4 g1 = *reinterpret_cast<const float4*>(gp + 4);
    const float g[COMBINE_VEC] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float sc = sj[j];
#pragma unroll
    for (int i = 0; i < COMBINE_VEC; ++i) acc[i] = fmaf(sc, v[i] * g[i], acc[i]);
  }
  const size_t off = t * p + col0 + cl;
  // c must fit its store: finite, and inside FP16 for BF16 configurations (|c_i| <=
  // sum_j |w_j| * sqrt(p) * max|g_exp|; replayed weights with a large sum can leave it)
  float cmax = 0.f, fin = 0.f;
#pragma unroll
  for (int i = 0; i < COMBINE_VEC; ++i) {
    cmax = fmaxf(cmax, fabsf(acc[i]));
    fin = fmaf(acc[i], 0.f, fin);           // NaN unless every value is finite
  }
  if (!(fin == 0.f && (C_F32 || cmax <= F16_MAX)))
    report_error(status, ST_DEVICE_CHECK, CHECK_C_RANGE);
  if constexpr (C_F32) {
    float* o = static_cast<float*>(c_out) + off;
    *reinterpret_cast<float4*>(o) = make_float4(tf32_rna(acc[0]), tf32_rna(acc[1]),
                                                tf32_rna(acc[2]), tf32_rna(acc[3]));
    *reinterpret_cast<float4*>(o + 4) = make_float4(tf32_rna(acc[4]), tf32_rna(acc[5]),
                                                    tf32_rna(acc[6]), tf32_rna(acc[7]));
  } else {
    uint4 o;
    o.x = pack_f16x2(acc[0], acc[1]);
    o.y = pack_f16x2(acc[2], acc[3]);
    o.z = pack_f16x2(acc[4], acc[5]);
    o.w = pack_f16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(static_cast<__half*>(c_out) + off) = o;
  }
}

// Block sums of squares of stored expert output rows (FP32, or FP16 when Y_F16), for the
// down GEMM variants whose epilogue does not produce them (weight-row tiles): one thread
// per (row, 128 columns), summed in column order like the GEMM epilogues.
template <bool Y_F16>
__global__ void __launch_bounds__(MEM_THREADS)
    row_ssq_kernel(const void* __restrict__ y, int rows, int p, float* __restrict__ row_ssq) {
  pdl_wait();
  pdl_allow_next();
  const int parts = p >> 7;
  const size_t n = size_t(rows) * parts;
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n;
       i += size_t(gridDim.x) * blockDim.x) {
    const size_t e0 = (i / parts) * p + (i % parts) * 128;
    float ss = 0.f;
    if constexpr (Y_F16) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __half*>(y) + e0);
      for (int q = 0; q < 16; ++q) {
        const uint4 v = src[q];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f = unpack_f16x2(w[h]);
          ss = fmaf(f.x, f.x, ss);
          ss = fmaf(f.y, f.y, ss);
        }
      }
    } else {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(y) + e0);
      for (int q = 0; q < 32; ++q) {
        const float4 v = src[q];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
    }
    row_ssq[i] = ss;
  }
}

// ---- block boundary: post-norm + residual + next pre-norm ------------------------------
// "vLLM 对 Muse Spark Open 的 Day 0 支持", section "三明治归一化": the block sits between
// two norms, x + post_norm(F(norm(x))); "SGLang and Miles Add Day-0 Support for Muse Spark
// Open", section "Kernel Optimizations": the post-FFN norm, the gated residual add and
// the pre-attention norm run as one kernel that keeps each row on chip across both
// RMS reductions (here in shared memory), and a cluster of CTAs shares one row through distributed shared memory
// when rows alone do not fill the GPU.
//
//   a = RMSNorm_{g_post}(y);  x' = x + gate * a (gate per channel, or 1);  stored as the
//   residual stream's type;  h' = RMSNorm_{g_next}(x' as stored)
//
// C CTAs (one cluster) share a row: CTA r holds columns [r d/C, (r+1) d/C) (at most
// BND_MAXV * MEM_THREADS) in shared memory.  Both sums of squares go thread -> warp -> CTA (fixed
// order) -> cluster (partials of ranks 0..C-1 added in rank order by every CTA), so all
// CTAs of a row use the same bits.
constexpr int BND_MAXV = 32;   // values per thread: d / C <= 8192

__device__ __forceinline__ float cluster_row_sum(float v, float* red, float* part, int C) {
  const float s = block_sum(v, red);
  if (C == 1) return s;
  if (threadIdx.x == 0) *part = s;
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
  float total = 0.f;
  for (int r = 0; r < C; ++r) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(part)), "r"(r));
    float q;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(q) : "r"(a) : "memory");
    total += q;
  }
  return total;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// 8 consecutive values of a BF16 or FP32 array in shared memory
__device__ __forceinline__ void smem_load8(const uint8_t* base, int idx, int is_f32,
                                           float (&v)[8]) {
  if (is_f32) {
    const float4 a = reinterpret_cast<const float4*>(base)[2 * idx];
    const float4 b = reinterpret_cast<const float4*>(base)[2 * idx + 1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 a = reinterpret_cast<const uint4*>(base)[idx];
    float2 f;
    f = unpack_bf16x2(a.x); v[0] = f.x; v[1] = f.y;
    f = unpack_bf16x2(a.y); v[2] = f.x; v[3] = f.y;
    f = unpack_bf16x2(a.z); v[4] = f.x; v[5] = f.y;
    f = unpack_bf16x2(a.w); v[6] = f.x; v[7] = f.y;
  }
}

// Shared memory of one CTA of the boundary kernel: its x and y slices.
inline size_t boundary_smem_bytes(int cols, int x_f32, int y_f32) {
  return size_t(cols) * ((x_f32 ? 4 : 2) + (y_f32 ? 4 : 2));
}

template <int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(MEM_THREADS)
    boundary_kernel(const void* __restrict__ x, const void* __restrict__ y,
                    const float* __restrict__ g_post, const float* __restrict__ gate,
                    const float* __restrict__ g_next, void* x_out, void* __restrict__ h_next,
                    int d, float eps, int x_f32, int y_f32) {
  extern __shared__ __align__(16) uint8_t bnd_smem[];
  __shared__ float red[32];
  __shared__ float part[2];
  const int rank = C == 1 ? 0 : static_cast<int>(blockIdx.x % C);
  const size_t t = blockIdx.x / C;
  const int cols = d / C;
  const int c0 = rank * cols;
  const int nchunk = cols >> 3;       // 8 values per chunk
  const int xe = x_f32 ? 4 : 2, ye = y_f32 ? 4 : 2;
  uint8_t* sy = bnd_smem;
  uint8_t* sx = bnd_smem + size_t(cols) * ye;
  // the CTA's slices of y and x, fetched with asynchronous 16-byte copies (many in flight,
  // few registers), then the row stays on chip across both reductions
  {
    const uint8_t* gy = static_cast<const uint8_t*>(y) + (t * d + c0) * ye;
    const uint8_t* gx = static_cast<const uint8_t*>(x) + (t * d + c0) * xe;
    const int ny = cols * ye / 16, nx = cols * xe / 16;
    for (int i = threadIdx.x; i < ny; i += blockDim.x) cp_async16(sy + 16 * i, gy + 16 * i);
    for (int i = threadIdx.x; i < nx; i += blockDim.x) cp_async16(sx + 16 * i, gx + 16 * i);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncthreads();
  }
  // 1. sum of squares of the block output
  float ss = 0.f;
  for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
    float v[8];
    smem_load8(sy, c, y_f32, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
  }
  const float rs_y = rsqrtf(cluster_row_sum(ss, red, &part[0], C) / static_cast<float>(d) + eps);
  // 2. residual add, rounded to the stream's type: written out and kept on chip
  float ss2 = 0.f;
  for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
    const int col = c0 + 8 * c;
    float v[8], xv[8];
    smem_load8(sy, c, y_f32, v);
    smem_load8(sx, c, x_f32, xv);
    const float4 p0 = reinterpret_cast<const float4*>(g_post + col)[0];
    const float4 p1 = reinterpret_cast<const float4*>(g_post + col)[1];
    const float gp[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    float gt[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
    if (gate) {
      const float4 q0 = reinterpret_cast<const float4*>(gate + col)[0];
      const float4 q1 = reinterpret_cast<const float4*>(gate + col)[1];
      gt[0] = q0.x; gt[1] = q0.y; gt[2] = q0.z; gt[3] = q0.w;
      gt[4] = q1.x; gt[5] = q1.y; gt[6] = q1.z; gt[7] = q1.w;
    }
    float r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      r[j] = xv[j] + gt[j] * (v[j] * rs_y * gp[j]);
      if (!x_f32) r[j] = __bfloat162float(__float2bfloat16_rn(r[j]));
      ss2 = fmaf(r[j], r[j], ss2);
    }
    const size_t off = t * d + col;
    if (x_f32) {
      const float4 o0 = make_float4(r[0], r[1], r[2], r[3]), o1 = make_float4(r[4], r[5], r[6], r[7]);
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(x_out) + off);
      dst[0] = o0;
      dst[1] = o1;
      reinterpret_cast<float4*>(sx)[2 * c] = o0;
      reinterpret_cast<float4*>(sx)[2 * c + 1] = o1;
    } else {
      uint4 o;
      o.x = pack_bf16x2(r[0], r[1]); o.y = pack_bf16x2(r[2], r[3]);
      o.z = pack_bf16x2(r[4], r[5]); o.w = pack_bf16x2(r[6], r[7]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(x_out) + off) = o;
      reinterpret_cast<uint4*>(sx)[c] = o;
    }
  }
  // 3. the next block's pre-norm on the stored residual (each thread rereads its own
  // chunks, so no barrier is needed between the write above and the read below)
  const float rs_x = rsqrtf(cluster_row_sum(ss2, red, &part[1], C) / static_cast<float>(d) + eps);
  for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
    const int col = c0 + 8 * c;
    float v[8];
    smem_load8(sx, c, x_f32, v);
    const float4 n0 = reinterpret_cast<const float4*>(g_next + col)[0];
    const float4 n1 = reinterpret_cast<const float4*>(g_next + col)[1];
    const float gn[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = v[j] * rs_x * gn[j];
    const size_t off = t * d + col;
    if (x_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(h_next) + off);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    } else {
      uint4 q;
      q.x = pack_bf16x2(o[0], o[1]); q.y = pack_bf16x2(o[2], o[3]);
      q.z = pack_bf16x2(o[4], o[5]); q.w = pack_bf16x2(o[6], o[7]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(h_next) + off) = q;
    }
  }
  // no CTA of the cluster leaves while another may still read its partials
  if (C > 1) asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ---- weight preparation ----------------------------------------------------------------
// Element conversion applied while packing a weight: FP32 -> TF32 (ties away) for FP32
// configurations, BF16 -> FP16 for BF16 ones (exact for |w| >= 2^-17; smaller values
// round to the FP16 subnormal grid, 2^-24 apart).
enum PackConv : int { CONV_TF32 = 0, CONV_BF16_TO_F16 = 1 };

template <int CONV>
__device__ __forceinline__ uint4 pack_convert(uint4 v) {
  if constexpr (CONV == CONV_TF32) {
    v.x = __float_as_uint(tf32_rna(__uint_as_float(v.x)));
    v.y = __float_as_uint(tf32_rna(__uint_as_float(v.y)));
    v.z = __float_as_uint(tf32_rna(__uint_as_float(v.z)));
    v.w = __float_as_uint(tf32_rna(__uint_as_float(v.w)));
  } else {
    float2 f;
    f = unpack_bf16x2(v.x); v.x = pack_f16x2(f.x, f.y);
    f = unpack_bf16x2(v.y); v.y = pack_f16x2(f.x, f.y);
    f = unpack_bf16x2(v.z); v.z = pack_f16x2(f.x, f.y);
    f = unpack_bf16x2(v.w); v.w = pack_f16x2(f.x, f.y);
  }
  return v;
}

// Converted copy of n bytes (a multiple of 16) of a weight tensor.
template <int CONV>
__global__ void convert_copy_kernel(const void* __restrict__ src, void* __restrict__ dst,
                                    size_t n16) {
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n16;
       i += size_t(gridDim.x) * blockDim.x)
    reinterpret_cast<uint4*>(dst)[i] = pack_convert<CONV>(reinterpret_cast<const uint4*>(src)[i]);
}

// One block per destination row of w13 [E, 2I, p]: rows are interleaved in blocks of G:
// dst[e][2G*b + i] = gate[e][G*b + i], dst[e][2G*b + G + i] = up[e][G*b + i].
template <int CONV>
__global__ void pack_w13_kernel(const void* __restrict__ gate, const void* __restrict__ up,
                                void* __restrict__ dst, int I, int p, int G, int elem_bytes) {
  const size_t drow = blockIdx.x;         // e * 2I + r
  const size_t e = drow / (2 * I);
  const int r = static_cast<int>(drow - e * 2 * I);
  const int b = r / (2 * G);
  const int i = r - b * 2 * G;
  const bool is_up = i >= G;
  const size_t srow = e * I + size_t(b) * G + (is_up ? i - G : i);
  const uint8_t* s = static_cast<const uint8_t*>(is_up ? up : gate) + srow * p * elem_bytes;
  uint8_t* o = static_cast<uint8_t*>(dst) + drow * p * elem_bytes;
  const int n16 = p * elem_bytes / 16;
  for (int c = threadIdx.x; c < n16; c += blockDim.x)
    reinterpret_cast<uint4*>(o)[c] = pack_convert<CONV>(reinterpret_cast<const uint4*>(s)[c]);
}

// ---- split-K reductions ----------------------------------------------------------------
// out[i] = sum over s of part[s * n + i], in slice order (deterministic), written as FP32,
// BF16 or TF32-rounded FP32.  n % 4 == 0.
constexpr int SPLITK_BATCH = 8;
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int ksplit, size_t n,
                                     void* __restrict__ out, int fmt) {
  pdl_wait();
  pdl_allow_next();
  for (size_t i = (blockIdx.x * size_t(blockDim.x) + threadIdx.x) * 4; i < n;
       i += size_t(gridDim.x) * blockDim.x * 4) {
    // the first SPLITK_BATCH slices' loads all in flight, then the sums in a fixed order:
    // groups of 4 summed pairwise and added in slice order, then single slices
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[SPLITK_BATCH];
#pragma unroll
    for (int s = 0; s < SPLITK_BATCH; ++s)
      if (s < ksplit) v[s] = *reinterpret_cast<const float4*>(part + s * n + i);
    const int full = ksplit / 4 * 4;
#pragma unroll
    for (int s = 0; s < SPLITK_BATCH; s += 4) {
      if (s + 4 <= full) {
        acc.x += (v[s].x + v[s + 1].x) + (v[s + 2].x + v[s + 3].x);
        acc.y += (v[s].y + v[s + 1].y) + (v[s + 2].y + v[s + 3].y);
        acc.z += (v[s].z + v[s + 1].z) + (v[s + 2].z + v[s + 3].z);
        acc.w += (v[s].w + v[s + 1].w) + (v[s + 2].w + v[s + 3].w);
      }
    }
    int s = SPLITK_BATCH < full ? SPLITK_BATCH : full;
    for (; s + 4 <= full; s += 4) {
      const float4 v0 = *reinterpret_cast<const float4*>(part + (s + 0) * n + i);
      const float4 v1 = *reinterpret_cast<const float4*>(part + (s + 1) * n + i);
      const float4 v2 = *reinterpret_cast<const float4*>(part + (s + 2) * n + i);
      const float4 v3 = *reinterpret_cast<const float4*>(part + (s + 3) * n + i);
      acc.x += (v0.x + v1.x) + (v2.x + v3.x);
      acc.y += (v0.y + v1.y) + (v2.y + v3.y);
      acc.z += (v0.z + v1.z) + (v2.z + v3.z);
      acc.w += (v0.w + v1.w) + (v2.w + v3.w);
    }
#pragma unroll
    for (int j = 0; j < SPLITK_BATCH; ++j)     // single slices after the groups, in order
      if (j >= full && j < ksplit) {
        acc.x += v[j].x; acc.y += v[j].y; acc.z += v[j].z; acc.w += v[j].w;
      }
    for (s = full > SPLITK_BATCH ? full : SPLITK_BATCH; s < ksplit; ++s) {
      const float4 w = *reinterpret_cast<const float4*>(part + s * n + i);
      acc.x += w.x; acc.y += w.y; acc.z += w.z; acc.w += w.w;
    }
    if (fmt == 0) {          // BF16
      uint2 o;
      o.x = pack_bf16x2(acc.x, acc.y);
      o.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + i) = o;
    } else if (fmt == 2) {   // TF32-rounded FP32
      *reinterpret_cast<float4*>(static_cast<float*>(out) + i) =
          make_float4(tf32_rna(acc.x), tf32_rna(acc.y), tf32_rna(acc.z), tf32_rna(acc.w));
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = acc;
    }
  }
}

// Router logits from split-K partials [ksplit][T][ld] (sum in slice order), then the
// top-k (descending, ties to the lower id) and the softmax over the chosen logits.
// One block of 256 threads per token: thread e sums expert e's slices (every load in
// flight at once, ksplit <= ROUTER_MAX_SPLIT), then warp 0 picks the top k, lane l
// holding experts l, l+32, ...
constexpr int ROUTER_MAX_SPLIT = 32;
__global__ void __launch_bounds__(256)
    router_reduce_topk_kernel(const float* __restrict__ part, int ksplit, int T, int ld, int E,
                              int k, int32_t* __restrict__ ids, float* __restrict__ wts) {
  pdl_wait();
  pdl_allow_next();
  __shared__ float logit[256];
  const int t = blockIdx.x;
  const int e = threadIdx.x;
  float sum = 0.f;
  if (e < E) {
    const float* p = part + size_t(t) * ld + e;
    const size_t stride = size_t(T) * ld;
    float q[ROUTER_MAX_SPLIT];
#pragma unroll
    for (int s = 0; s < ROUTER_MAX_SPLIT; ++s) q[s] = s < ksplit ? p[s * stride] : 0.f;
#pragma unroll
    for (int s = 0; s < ROUTER_MAX_SPLIT; ++s)
      if (s < ksplit) sum += q[s];
  }
  logit[e] = sum;
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  constexpr int PER = 8;                 // E <= 256
  float v[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) v[j] = lane + 32 * j < E ? logit[lane + 32 * j] : -INFINITY;
  // k rounds of warp arg-max: larger logit wins, equal logits go to the lower id
  float chosen[MAX_TOPK];
  int chosen_id[MAX_TOPK];
  for (int r = 0; r < k; ++r) {
    float best = -INFINITY;
    int bid = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = lane + 32 * j;
      if (e < E && (v[j] > best || (v[j] == best && e < bid))) { best = v[j]; bid = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bid, o);
      if (ob > best || (ob == best && oi < bid)) { best = ob; bid = oi; }
    }
    chosen[r] = best;
    chosen_id[r] = bid;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (lane + 32 * j == bid) v[j] = -INFINITY;   // remove it (its id is unique)
  }
  if (lane == 0) {
    float z[MAX_TOPK], sum = 0.f;
    for (int r = 0; r < k; ++r) { z[r] = __expf(chosen[r] - chosen[0]); sum += z[r]; }
    const float inv = 1.0f / sum;
    for (int r = 0; r < k; ++r) {
      ids[size_t(t) * k + r] = chosen_id[r];
      wts[size_t(t) * k + r] = z[r] * inv;
    }
  }
}

// ---- NVFP4 ------------------------------------------------------------------------------
// ("SGLang and Miles Add Day-0 Support for Muse Spark Open", "NVFP4 as a third MMA kind":
// E2M1 values, UE4M3 scale per 16 elements, FP32 global scale per tensor / per token.)
constexpr float NVFP4_AMAX_DIV = 2688.0f;   // 6 (largest E2M1) * 448 (largest UE4M3)

// amax of |x| over `n` BF16 values at src + blockIdx.y * stride_y, merged into
// amax_bits[blockIdx.y] (FP32 bits of a non-negative value order like integers, so
// atomicMax is exact and order independent).
__global__ void amax_bf16_kernel(const __nv_bfloat16* __restrict__ src, size_t n,
                                 size_t stride_y, unsigned* __restrict__ amax_bits) {
  __shared__ float red[32];
  const __nv_bfloat16* p = src + blockIdx.y * stride_y;
  float m = 0.f;
  for (size_t i = (blockIdx.x * size_t(blockDim.x) + threadIdx.x) * 8; i < n;
       i += size_t(gridDim.x) * blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(p + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (threadIdx.x == 0) atomicMax(amax_bits + blockIdx.y, __float_as_uint(m));
  }
}

__global__ void zero_u32_kernel(unsigned* p, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0;
}

// g[e] = amax[e] / 2688 (the NVFP4 global scale of one expert's tensor).
__global__ void global_scale_kernel(const unsigned* __restrict__ amax_bits, float* __restrict__ g,
                                    int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) g[i] = __uint_as_float(amax_bits[i]) / NVFP4_AMAX_DIV;
}

// One block per destination row of a quantised expert matrix [E * rows, K]:
//   gate/up (interleaved in blocks of G rows, like the BF16 packing) when `up` is set,
//   a plain matrix otherwise.  Codes: [row][K/2] bytes; scales: chunked layout.
__global__ void quantize_weight_kernel(const __nv_bfloat16* __restrict__ gate,
                                       const __nv_bfloat16* __restrict__ up,
                                       uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                       const float* __restrict__ g, int rows_per_expert, int K,
                                       int G) {
  const size_t drow = blockIdx.x;
  const size_t e = drow / rows_per_expert;
  const int r = static_cast<int>(drow - e * rows_per_expert);
  const __nv_bfloat16* src;
  if (up != nullptr) {     // interleaved: dst rows [2G*b, 2G*b+G) gate, then up
    const int half_rows = rows_per_expert / 2;
    const int b = r / (2 * G), i = r - b * 2 * G;
    const size_t srow = e * half_rows + size_t(b) * G + (i >= G ? i - G : i);
    src = (i >= G ? up : gate) + srow * K;
  } else {
    src = gate + drow * K;
  }
  const float ge = g[e];
  const float six_g = 6.0f * ge;
  const float inv_g = ge > 0.f ? 1.0f / ge : 0.f;
  for (int grp = threadIdx.x; grp < K / 16; grp += blockDim.x) {
    const uint4 a = reinterpret_cast<const uint4*>(src)[2 * grp];
    const uint4 b = reinterpret_cast<const uint4*>(src)[2 * grp + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float x[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      x[2 * j] = f.x;
      x[2 * j + 1] = f.y;
    }
    uint2 q;
    const uint32_t code = quantize16(x, six_g, inv_g, q, nullptr);
    reinterpret_cast<uint2*>(codes + drow * (K / 2))[grp] = q;
    sf[sf_offset(drow, grp, K)] = static_cast<uint8_t>(code);
  }
}

// Pooled-input RMSNorm fused with the per-token NVFP4 quantiser: one block per token;
// u = pooled * rsqrt(mean(pooled^2) + eps) * g_pool in FP32, alpha = max|u| / 2688,
// then E2M1 codes + UE4M3 scales written to each of the token's k dispatched rows
// (alpha too, per row, for the gate/up GEMM's accumulators).  p <= 8192.  A row that is
// not finite is reported as CHECK_U_RANGE.
__global__ void __launch_bounds__(MEM_THREADS)
    pool_quant_kernel(const float* __restrict__ pooled, const float* __restrict__ g,
                      const int* __restrict__ inv, uint8_t* __restrict__ codes,
                      uint8_t* __restrict__ sf, float* __restrict__ alpha_rows, int p, int k,
                      float eps, int* status) {
  pdl_wait();
  pdl_allow_next();
  __shared__ float red[32];
  __shared__ int rows[MAX_TOPK];
  const size_t t = blockIdx.x;
  if (threadIdx.x < k) rows[threadIdx.x] = inv[t * k + threadIdx.x];
  constexpr int GPT = 2;                 // 16-element groups per thread: p <= 8192
  const int ngrp = p >> 4;
  float v[GPT][16];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    const int grp = threadIdx.x + j * MEM_THREADS;
    if (grp < ngrp) {
      const float4* s4 = reinterpret_cast<const float4*>(pooled + t * p) + 4 * grp;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a = s4[q];
        v[j][4 * q] = a.x; v[j][4 * q + 1] = a.y; v[j][4 * q + 2] = a.z; v[j][4 * q + 3] = a.w;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) ss = fmaf(v[j][i], v[j][i], ss);
    }
  }
  const float total = block_sum(ss, red);
  const float rs = rsqrtf(total / static_cast<float>(p) + eps);
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    const int grp = threadIdx.x + j * MEM_THREADS;
    if (grp < ngrp) {
      const float4* g4 = reinterpret_cast<const float4*>(g) + 4 * grp;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 gg = g4[q];
        v[j][4 * q] = v[j][4 * q] * rs * gg.x;
        v[j][4 * q + 1] = v[j][4 * q + 1] * rs * gg.y;
        v[j][4 * q + 2] = v[j][4 * q + 2] * rs * gg.z;
        v[j][4 * q + 3] = v[j][4 * q + 3] * rs * gg.w;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[j][i]));
    }
  }
  // block max (after block_sum's barriers the reduction buffer is free again)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = (threadIdx.x & 31) < (blockDim.x >> 5) ? red[threadIdx.x & 31] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  // a row that is not finite cannot be quantised (its scale would be inf or NaN)
  if (threadIdx.x == 0 && !(fabsf(total) < INFINITY && amax < INFINITY))
    report_error(status, ST_DEVICE_CHECK, CHECK_U_RANGE);
  const float a = amax / NVFP4_AMAX_DIV;
  const float six_a = 6.0f * a;
  const float inv_a = a > 0.f ? 1.0f / a : 0.f;
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    const int grp = threadIdx.x + j * MEM_THREADS;
    if (grp < ngrp) {
      uint2 q;
      const uint32_t code = quantize16(v[j], six_a, inv_a, q, nullptr);
      for (int sl = 0; sl < k; ++sl) {
        const int r = rows[sl];
        if (r < 0) continue;
        reinterpret_cast<uint2*>(codes + size_t(r) * (p / 2))[grp] = q;
        sf[sf_offset(size_t(r), grp, p)] = static_cast<uint8_t>(code);
      }
    }
  }
  if (threadIdx.x < k && rows[threadIdx.x] >= 0) alpha_rows[rows[threadIdx.x]] = a;
}

__global__ void clear_status_kernel(int* status) {
  if (threadIdx.x < 2) status[threadIdx.x] = 0;
}

}  // namespace lmoe
