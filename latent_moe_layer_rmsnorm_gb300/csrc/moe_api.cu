// moe_api.cu -- the C ABI of the latent-MoE block (declared in include/latent_moe.h):
// argument validation, workspace carving, TMA descriptors and the launch sequence.
// Nothing here allocates device memory; every buffer is the caller's.
#include <mutex>

#include "../../include/latent_moe.h"
#include "common.cuh"
#include "gemm_nvf4.cuh"
#include "gemm_nvf4_pair.cuh"
#include "gemm_pair.cuh"
#include "gemm_swap.cuh"
#include "gemm_tcgen05.cuh"
#include "kernels_mem.cuh"

using namespace lmoe;

namespace {


constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;       // 1 s
constexpr unsigned long long TEST_WAIT_LIMIT_NS = 20000000ull;    // 20 ms

enum Stage { STG_NORM = 0, STG_ROUTER, STG_POOL, STG_DISPATCH, STG_GEMM1, STG_GEMM2,
             STG_COMBINE, STG_UNPOOL, STG_COUNT };
const char* const kStageNames[STG_COUNT] = {"norm", "router", "pool", "dispatch",
                                            "gemm1_gate_up_swiglu", "gemm2_down",
                                            "combine", "unpool"};

constexpr int W13_GROUP = 128;   // gate/up interleave block (rows)

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// ---- driver entry point for tensor maps ------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major [rows, inner] operand of the given kind, tiles of box_rows x 128 bytes,
// 128-byte swizzle, zero fill outside the tensor.  TF32 operands are plain FP32 words
// (already rounded), so the copy moves their bits unchanged.
bool make_tmap(CUtensorMap* m, const void* base, int kind, uint64_t inner, uint64_t rows,
               uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const uint32_t es = kind == OP_TF32 ? 4 : kind == OP_NVF4 ? 1 : 2;
  const CUtensorMapDataType dt = kind == OP_TF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : kind == OP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : kind == OP_NVF4 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * es};
  cuuint32_t box[2] = {128u / es, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- per-device cache -------------------------------------------------------------------
struct DevInfo {
  int sms = 0;
  int bnd_clusters = 0;   // CTA pairs of the fused unpooler + boundary kernel that fit at once
  bool ready = false;
};
DevInfo g_dev[64];
std::mutex g_mu;

template <int KIND, int EPI>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gemm_tcgen05_kernel<KIND, EPI>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(gemm_smem_bytes()));
}

moe_status_t device_ready(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& D = g_dev[dev];
  if (!D.ready) {
    if (cudaDeviceGetAttribute(&D.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = set_smem_attr<OP_TF32, EPI_ROUTER>();
    if (e == cudaSuccess) e = set_smem_attr<OP_TF32, EPI_STORE>();
    if (e == cudaSuccess) e = set_smem_attr<OP_TF32, EPI_SWIGLU>();
    if (e == cudaSuccess) e = set_smem_attr<OP_F16, EPI_STORE>();
    if (e == cudaSuccess) e = set_smem_attr<OP_F16, EPI_SWIGLU>();
    const int swap_smem = static_cast<int>(swap_smem_bytes());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_swap_kernel<OP_F16, SWAP_SWIGLU>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, swap_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_swap_kernel<OP_F16, SWAP_STORE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, swap_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_swap_kernel<OP_TF32, SWAP_SWIGLU>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, swap_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_swap_kernel<OP_TF32, SWAP_STORE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, swap_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_nvf4_kernel<NV_EPI_SWIGLU_Q>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(nvf4_smem_bytes()));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_nvf4_kernel<NV_EPI_STORE_Y>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(nvf4_smem_bytes()));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_nvf4_kernel<NV_EPI_STORE_Y_ROWS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(nvf4_smem_bytes()));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel<NV_EPI_SWIGLU_Q>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(nvf4_pair_smem_bytes()));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel<NV_EPI_STORE_Y>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(nvf4_pair_smem_bytes()));
    const int pair_smem = static_cast<int>(pair_smem_bytes());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_pair_kernel<OP_F16, EPI_STORE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_pair_kernel<OP_F16, EPI_SWIGLU>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_pair_kernel<OP_TF32, EPI_STORE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_pair_kernel<OP_TF32, EPI_SWIGLU>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_pair_kernel<OP_TF32, EPI_ROUTER>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_pair_kernel<OP_F16, EPI_BOUNDARY>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_pair_kernel<OP_TF32, EPI_BOUNDARY>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem);
    if (e == cudaSuccess) {
      // the fused unpooler's row workers wait for tiles of other clusters of the same
      // launch, so that launch never holds more clusters than can run at once
      cudaLaunchConfig_t oc{};
      oc.gridDim = dim3(D.sms);
      oc.blockDim = dim3(BND_THREADS);
      oc.dynamicSmemBytes = pair_smem;
      int n16 = 0, n32 = 0;
      if (cudaOccupancyMaxActiveClusters(&n16, gemm_pair_kernel<OP_F16, EPI_BOUNDARY>, &oc) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveClusters(&n32, gemm_pair_kernel<OP_TF32, EPI_BOUNDARY>, &oc) !=
              cudaSuccess) {
        (void)cudaGetLastError();   // no figure: the fused path stays off on this device
        n16 = n32 = 0;
      }
      D.bnd_clusters = std::min(std::min(n16, n32), D.sms / 2);
    }
    // boundary kernel: x and y slices of up to BND_MAXV * MEM_THREADS FP32 columns each
    const int bnd_smem = static_cast<int>(boundary_smem_bytes(BND_MAXV * MEM_THREADS, 1, 1));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(boundary_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bnd_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(boundary_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bnd_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(boundary_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bnd_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(boundary_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bnd_smem);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    D.ready = true;
  }
  *sms = D.sms;
  return MOE_OK;
}

// ---- validation and workspace layout ------------------------------------------------------
moe_status_t validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d <= 0 || c->p <= 0 || c->I <= 0 || c->E <= 0 || c->top_k <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->E) return MOE_ERR_INVALID_ARG;
  if (!(c->eps >= 0.0f) || c->eps > 1.0f) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_BF16 && c->act != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (c->out != MOE_BF16 && c->out != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (c->expert != MOE_BF16 && c->expert != MOE_F32 && c->expert != MOE_NVFP4)
    return MOE_ERR_INVALID_ARG;
  if (c->expert == MOE_NVFP4) {
    if (c->act != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (c->p % 256 || c->I % 256) return MOE_ERR_UNSUPPORTED;
  } else if (c->expert != c->act) {
    return MOE_ERR_UNSUPPORTED;
  }
  if ((c->flags & ~(MOE_FLAG_TEST_TIMEOUT | MOE_FLAG_WEIGHT_TILES | MOE_FLAG_NVFP4_PAIR |
                    MOE_FLAG_NVFP4_ONE_CTA)) != 0)
    return MOE_ERR_INVALID_ARG;
  if ((c->flags & MOE_FLAG_NVFP4_PAIR) && (c->flags & MOE_FLAG_NVFP4_ONE_CTA))
    return MOE_ERR_INVALID_ARG;
  if (c->E > 256 || c->top_k > MAX_TOPK) return MOE_ERR_UNSUPPORTED;
  if (c->d % 128 || c->p % 128 || c->I % 128) return MOE_ERR_UNSUPPORTED;
  if (c->d > 32768 || c->p > 8192 || c->I > 32768) return MOE_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(c->T) * c->top_k;
  if (rows > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(c->E) * 2 * c->I > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

inline int bn_for(int n) { return (n % 256 == 0) ? 256 : 128; }

// K slices for a dense GEMM whose output has too few tiles to fill the GPU (the decode
// regime): aim for ~128 CTAs, each slice at least 4 K blocks (kblk elements each).
int split_for(int T, int N, int bn, int K, int kblk) {
  const int tiles = ((T + GEMM_BM - 1) / GEMM_BM) * (N / bn);
  if (tiles >= 64) return 1;
  int ks = 1;
  while (ks * 2 * tiles <= 128 && K % (ks * 2 * kblk) == 0 && K / (ks * 2) >= 4 * kblk) ks *= 2;
  return ks;
}

struct SplitPlan {
  int router, pool, unpool;
  size_t part_floats;
};

SplitPlan split_plan(const moe_config_t& c) {
  SplitPlan sp{};
  const int Ep = (c.E + 15) / 16 * 16;
  const bool f32 = c.act == MOE_F32;
  sp.router = std::min(split_for(c.T, Ep, Ep, c.d, 32), ROUTER_MAX_SPLIT);
  sp.pool = split_for(c.T, c.p, bn_for(c.p), c.d, f32 ? 32 : 64);
  sp.unpool = split_for(c.T, c.d, bn_for(c.d), c.p, f32 ? 32 : 64);
  size_t m = 0;
  if (sp.router > 1) m = std::max(m, size_t(sp.router) * c.T * Ep);
  if (sp.pool > 1) m = std::max(m, size_t(sp.pool) * c.T * c.p);
  if (sp.unpool > 1) m = std::max(m, size_t(sp.unpool) * c.T * c.d);
  sp.part_floats = m;
  return sp;
}

// 32-row blocks whose column tiles the fused unpooler counts (whole 256-row pair tiles)
inline size_t bnd_blocks(int T) { return size_t(8) * ((T + 255) / 256); }

struct WsLayout {
  size_t status, h32, h16, ids, wts, pooled, chunk, row_off, mt_off, mt2_off, row_cnt, src, inv,
      a_perm, s, y, ssq, c, sf_u, sf_s, alpha, part, bnd_ssq, bnd_cnt, total;
  int nchunks;
  size_t rows;    // dispatched rows (NVFP4: 128-aligned per expert)
};

WsLayout ws_layout(const moe_config_t& c) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t T = c.T, d = c.d, p = c.p, E = c.E, k = c.top_k, I = c.I;
  const size_t ea = c.act == MOE_F32 ? 4 : 2;
  const size_t ee = c.expert == MOE_F32 ? 4 : 2;
  const bool q = c.expert == MOE_NVFP4;
  L.nchunks = static_cast<int>((T * k + DISPATCH_CHUNK - 1) / DISPATCH_CHUNK);
  L.rows = 128 * ((T * k + 127) / 128 + E);   // every expert's rows start on a 128-row boundary
  const size_t R = L.rows;
  L.status = take(256);
  L.h32 = take(T * d * 4);
  L.h16 = take(c.act == MOE_BF16 ? T * d * 2 : 0);
  L.ids = take(T * k * 4);
  L.wts = take(T * k * 4);
  L.pooled = take(T * p * 4);
  L.chunk = take(size_t(L.nchunks) * E * 4);
  L.row_off = take((E + 1) * 4);
  L.mt_off = take((E + 1) * 4);
  L.mt2_off = take((E + 1) * 4);
  L.row_cnt = take((E + 1) * 4);
  L.src = take(R * 4);
  L.inv = take(T * k * 4);
  L.a_perm = take(q ? R * p / 2 : R * p * ee);
  L.s = take(q ? R * I / 2 : R * I * ee);
  L.y = take(R * p * (c.expert == MOE_F32 ? 4 : 2));   // expert outputs: FP16 (FP32 experts: FP32)
  L.ssq = take(R * (p / 128) * 4);   // their sums of squares per 128-column block
  L.c = take(T * p * ea);
  L.sf_u = take(q ? R * p / 16 : 0);
  L.sf_s = take(q ? R * I / 16 : 0);
  L.alpha = take(q ? R * 4 : 0);
  L.part = take(split_plan(c).part_floats * 4);   // split-K partial sums (small T only)
  // moe_forward_boundary with the boundary in the unpooler: the block output's sums of
  // squares per 128 columns, and the per-32-row-block tile counters + the item counter
  L.bnd_ssq = take(T * (d / 128) * 4);
  L.bnd_cnt = take((bnd_blocks(c.T) + 1) * 4);
  L.total = off;
  return L;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status_t check_weights(const moe_config_t& c, const moe_weights_t* W, bool route_only,
                           bool need_router) {
  if (!W) return MOE_ERR_INVALID_ARG;
  const void* need[] = {W->g_in, need_router ? W->w_router : W->g_in};
  for (const void* p : need)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (route_only) return MOE_OK;
  const void* more[] = {W->w_pool, W->g_pool, W->w13, W->w2, W->g_exp, W->w_unpool};
  for (const void* p : more)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (c.expert == MOE_NVFP4) {
    const void* q[] = {W->sf13, W->sf2, W->gs13, W->gs2, W->gs_act2};
    for (const void* p : q)
      if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

inline moe_status_t last_launch() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// One kernel of a forward.  Programmatic stream serialisation lets the kernel be
// scheduled while the previous kernel of the stream is finishing, so its prologue
// (barrier set-up, tensor-map prefetch, TMEM allocation) and launch latency overlap the
// predecessor's tail; every kernel of the step waits for its predecessors (pdl_wait)
// before it touches global memory ("SGLang and Miles Add Day-0 Support for Muse Spark
// Open", section "Kernel Optimizations": launch dependent kernels earlier).
template <typename... KArgs, typename... Args>
moe_status_t launch_step(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t st, Args... args) {
  if (grid.x == 0) return MOE_OK;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

template <int KIND, int EPI>
moe_status_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& P,
                         int grid, cudaStream_t st) {
  if (grid <= 0) return MOE_OK;
  return launch_step(gemm_tcgen05_kernel<KIND, EPI>, dim3(grid), dim3(GEMM_THREADS),
                     gemm_smem_bytes(), st, ta, tb, P);
}

// CTA-pair GEMM: one cluster of 2 CTAs per 256 x 256 tile, up to one cluster per 2 SMs.
// `ta64` / `tb64` map A / B with 64-row boxes (the grouped GEMMs' M = 128 tiles; `tb64`
// only for the gate/up GEMM; both unused when dense).
template <int KIND, int EPI>
// `tout` maps the output in 32-row boxes of 128 bytes: warps whose 32 rows of a tile are
// all valid write through it (P.out_box is set here).
moe_status_t launch_pair(const CUtensorMap& ta, const CUtensorMap& ta64, const CUtensorMap& tb,
                         const CUtensorMap& tb64, const CUtensorMap& tout, GemmParams P,
                         int max_tiles, int sms, cudaStream_t st, bool boxes = true,
                         int max_clusters = 0) {
  const int clusters = std::min(max_clusters > 0 ? max_clusters : sms / 2, max_tiles);
  if (clusters <= 0) return MOE_OK;
  P.out_box = boxes ? 1 : 0;
  return launch_step(gemm_pair_kernel<KIND, EPI>, dim3(2 * clusters), dim3(pair_threads<EPI>()),
                     pair_smem_bytes(), st, ta, ta64, tb, tb64, tout, P);
}

GemmParams base_params(int* status, uint32_t flags) {
  GemmParams P{};
  P.ksplit = 1;
  P.status = status;
  P.timeout_ns = (flags & MOE_FLAG_TEST_TIMEOUT) ? TEST_WAIT_LIMIT_NS : WAIT_LIMIT_NS;
  return P;
}

struct Events {
  cudaEvent_t* ev;
  int n;
  cudaStream_t st;
  void mark(int i) {   // after stage i-1
    if (ev && i < n && ev[i]) cudaEventRecord(ev[i], st);
  }
};

#define MOE_TRY(expr)                \
  do {                               \
    moe_status_t _s = (expr);        \
    if (_s != MOE_OK) return _s;     \
  } while (0)

// Arguments of the block boundary (moe_boundary, moe_forward_boundary): present, 16-byte
// aligned, and no output overlapping an input other than x_out == x (in place); y_written:
// y is an output too (moe_forward_boundary), so it may not overlap x either.
moe_status_t check_boundary_buffers(const moe_config_t& c, const void* x, const void* y,
                                    const float* g_post, const float* gate, const float* g_next,
                                    const void* x_out, const void* h_next, bool y_written) {
  if (!x || !y || !g_post || !g_next || !x_out || !h_next) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(g_post) || !aligned16(g_next) ||
      !aligned16(x_out) || !aligned16(h_next) || (gate && !aligned16(gate)))
    return MOE_ERR_INVALID_ARG;
  const size_t ex = c.act == MOE_F32 ? 4 : 2, ey = c.out == MOE_F32 ? 4 : 2;
  const size_t bx = size_t(c.T) * c.d * ex, by = size_t(c.T) * c.d * ey;
  auto overlap = [](const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
  };
  // x_out may be x itself (in-place residual update); nothing else may overlap
  if ((x_out != x && overlap(x_out, bx, x, bx)) || overlap(x_out, bx, y, by) ||
      (y_written && overlap(x, bx, y, by)) || overlap(h_next, bx, x, bx) ||
      overlap(h_next, bx, y, by) ||
      overlap(h_next, bx, x_out, bx))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// The boundary as its own pass over [T, d] (boundary_kernel<C>).
moe_status_t launch_boundary_pass(const moe_config_t& c, const void* x, const void* y,
                                  const float* g_post, const float* gate, const float* g_next,
                                  void* x_out, void* h_next, cudaStream_t st, int sms) {
  // CTAs per row: enough that a CTA holds at most BND_MAXV * MEM_THREADS columns, and
  // more (up to a cluster of 8) while the rows alone would leave SMs idle
  int C = 1;
  while (C < 8 && (c.d / C > BND_MAXV * MEM_THREADS || static_cast<long long>(c.T) * C < 2 * sms))
    C *= 2;
  const int xf = c.act == MOE_F32, yf = c.out == MOE_F32;
  const unsigned grid = static_cast<unsigned>(c.T) * C;
  const size_t smem = boundary_smem_bytes(c.d / C, xf, yf);
  switch (C) {
    case 1: boundary_kernel<1><<<grid, MEM_THREADS, smem, st>>>(x, y, g_post, gate, g_next, x_out, h_next, c.d, c.eps, xf, yf); break;
    case 2: boundary_kernel<2><<<grid, MEM_THREADS, smem, st>>>(x, y, g_post, gate, g_next, x_out, h_next, c.d, c.eps, xf, yf); break;
    case 4: boundary_kernel<4><<<grid, MEM_THREADS, smem, st>>>(x, y, g_post, gate, g_next, x_out, h_next, c.d, c.eps, xf, yf); break;
    default: boundary_kernel<8><<<grid, MEM_THREADS, smem, st>>>(x, y, g_post, gate, g_next, x_out, h_next, c.d, c.eps, xf, yf); break;
  }
  return last_launch();
}

// The block.  route_only: stop after the router, writing ids_out / w_out.
moe_status_t run_layer(const moe_config_t* cfg, const moe_weights_t* W, const void* x,
                       const int32_t* ids_in, const float* w_in, void* out, int32_t* ids_out,
                       float* w_out, bool route_only, void* ws, size_t ws_bytes,
                       cudaStream_t st, cudaEvent_t* ev, int nev,
                       const BoundaryArgs* bnd = nullptr) {
  MOE_TRY(validate(cfg));
  const moe_config_t& c = *cfg;
  const bool internal_route = route_only || ids_in == nullptr;
  if (!route_only && ((ids_in == nullptr) != (w_in == nullptr))) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_weights(c, W, route_only, internal_route));
  if (!x || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  if (route_only && (!ids_out || !w_out)) return MOE_ERR_INVALID_ARG;
  if (!route_only && (!out || !aligned16(out))) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return MOE_ERR_WORKSPACE;
  const WsLayout L = ws_layout(c);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  Events E{ev, nev, st};
  E.mark(0);
  if (c.T == 0) return MOE_OK;
  int sms = 0;
  MOE_TRY(device_ready(&sms));

  uint8_t* base = static_cast<uint8_t*>(ws);
  if (bnd && cudaMemsetAsync(base + L.bnd_cnt, 0, (bnd_blocks(c.T) + 1) * 4, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  int* status = reinterpret_cast<int*>(base + L.status);
  float* h32 = reinterpret_cast<float*>(base + L.h32);
  __half* h16 = reinterpret_cast<__half*>(base + L.h16);
  const bool act_f32 = c.act == MOE_F32;
  const bool exp_f32 = c.expert == MOE_F32;
  // operand kinds: FP32 configurations run on TF32; BF16 ones store every activation
  // between the GEMMs (h, u, s, y, c) in FP16 and meet FP16 copies of the weights
  const int k_proj = act_f32 ? OP_TF32 : OP_F16;      // pooler, unpooler
  const int k_up = exp_f32 ? OP_TF32 : OP_F16;        // gate/up GEMM
  const int k_down = exp_f32 ? OP_TF32 : OP_F16;      // down GEMM
  const int T = c.T, d = c.d, p = c.p, E_ = c.E, k = c.top_k, I = c.I;
  const int rows = T * k;
  const int mtiles = (T + GEMM_BM - 1) / GEMM_BM;

  // ---- stage: full-width RMSNorm ------------------------------------------------------
  // a router-only call does not need the pooler's FP16 copy of h
  if (act_f32)
    MOE_TRY(launch_step(norm_in_kernel<true>, dim3(T), dim3(MEM_THREADS), 0, st, x, W->g_in, h32,
                        static_cast<__half*>(nullptr), d, c.eps, status));
  else
    MOE_TRY(launch_step(norm_in_kernel<false>, dim3(T), dim3(MEM_THREADS), 0, st, x, W->g_in, h32,
                        route_only ? nullptr : h16, d, c.eps, status));
  E.mark(1);

  // ---- stage: router GEMM (TF32) + top-k ------------------------------------------------
  int32_t* ids = route_only ? ids_out : reinterpret_cast<int32_t*>(base + L.ids);
  float* wts = route_only ? w_out : reinterpret_cast<float*>(base + L.wts);
  const SplitPlan sp = split_plan(c);
  float* part = reinterpret_cast<float*>(base + L.part);
  if (internal_route) {
    const int bn = (E_ + 15) / 16 * 16;
    // split-K partial logits: 128-column tiles when they divide the experts, so twice the
    // CTAs share the 8 MiB GEMV at E = 256
    const int bn_split = bn % 128 == 0 ? 128 : bn;
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, h32, OP_TF32, d, T, GEMM_BM) ||
        !make_tmap(&tb, W->w_router, OP_TF32, d, E_, sp.router > 1 ? bn_split : bn))
      return MOE_ERR_CUDA;
    GemmParams P = base_params(status, c.flags);
    P.M = T; P.N = bn; P.K = d; P.bn = bn; P.groups = 0;
    P.b_const = 1;           // the router weights: loads may start before the norm ends
    if (sp.router > 1) {     // small T: K slices -> partial logits -> sum + top-k
      P.bn = bn_split;
      P.ksplit = sp.router; P.split_stride = size_t(T) * bn;
      P.out = part; P.ld_out = bn; P.out_fmt = OUT_F32;
      MOE_TRY((launch_gemm<OP_TF32, EPI_STORE>(
          ta, tb, P, std::min(sms, mtiles * (bn / bn_split) * sp.router), st)));
      MOE_TRY(launch_step(router_reduce_topk_kernel, dim3(T), dim3(256), 0, st, part,
                          sp.router, T, bn, E_, k, ids, wts));
    } else if (bn == 256) {   // CTA pairs: each CTA loads 128 of the 256 router rows
      P.E = E_; P.top_k = k; P.ids = ids; P.wts = wts;
      CUtensorMap tb2;
      if (!make_tmap(&tb2, W->w_router, OP_TF32, d, E_, 128)) return MOE_ERR_CUDA;
      MOE_TRY((launch_pair<OP_TF32, EPI_ROUTER>(ta, ta, tb2, tb2, ta, P, (T + 255) / 256, sms, st,
                                                false)));
    } else {
      P.E = E_; P.top_k = k; P.ids = ids; P.wts = wts;
      MOE_TRY((launch_gemm<OP_TF32, EPI_ROUTER>(ta, tb, P, std::min(sms, mtiles), st)));
    }
  } else {
    ids = const_cast<int32_t*>(ids_in);
    wts = const_cast<float*>(w_in);
  }
  E.mark(2);
  if (route_only) return MOE_OK;

  // ---- stage: pooler GEMM -> pooled FP32 ------------------------------------------------
  float* pooled = reinterpret_cast<float*>(base + L.pooled);
  {
    CUtensorMap ta, tb;
    const int bn = bn_for(p);
    if (!make_tmap(&ta, act_f32 ? static_cast<const void*>(h32) : h16, k_proj, d, T, GEMM_BM) ||
        !make_tmap(&tb, W->w_pool, k_proj, d, p, bn))
      return MOE_ERR_CUDA;
    GemmParams P = base_params(status, c.flags);
    P.M = T; P.N = p; P.K = d; P.bn = bn; P.groups = 0;
    P.b_const = 1;           // W_pool
    P.out = pooled; P.ld_out = p; P.out_fmt = OUT_F32;
    if (sp.pool > 1) { P.ksplit = sp.pool; P.split_stride = size_t(T) * p; P.out = part; }
    const int grid = std::min(sms, mtiles * (p / bn) * sp.pool);
    if (sp.pool == 1 && bn == 256) {          // CTA pairs: B half-tiles of 128 rows
      CUtensorMap tb2, to;
      if (!make_tmap(&tb2, W->w_pool, k_proj, d, p, 128) ||
          !make_tmap(&to, pooled, OP_TF32, p, T, 32))
        return MOE_ERR_CUDA;
      const int tiles = ((T + 255) / 256) * (p / 256);
      if (act_f32) MOE_TRY((launch_pair<OP_TF32, EPI_STORE>(ta, ta, tb2, tb2, to, P, tiles, sms, st)));
      else MOE_TRY((launch_pair<OP_F16, EPI_STORE>(ta, ta, tb2, tb2, to, P, tiles, sms, st)));
    } else if (act_f32) MOE_TRY((launch_gemm<OP_TF32, EPI_STORE>(ta, tb, P, grid, st)));
    else MOE_TRY((launch_gemm<OP_F16, EPI_STORE>(ta, tb, P, grid, st)));
    if (sp.pool > 1) {
      const size_t n = size_t(T) * p;
      MOE_TRY(launch_step(splitk_reduce_kernel,
                          dim3(static_cast<int>(std::min<size_t>((n / 4 + 255) / 256, 4096))),
                          dim3(256), 0, st, part, sp.pool, n, static_cast<void*>(pooled),
                          static_cast<int>(OUT_F32)));
    }
  }
  E.mark(3);

  // ---- stage: dispatch (counting sort) + pooled RMSNorm + permute ---------------------
  const bool nvf4 = c.expert == MOE_NVFP4;
  // Zero padding rows pay where the expert GEMMs run into the power cap: batches whose
  // experts average a full 256-row pair tile (prefill: +3 % SM clock, both GEMMs 3 %
  // faster).  At decode sizes almost every tile row is padding: zeroing it (and storing
  // it again as s) costs more than it saves, and even unzeroed, 128-row aligned experts
  // make each tile read rows of its own instead of its neighbours' rows already in L2.
  // NVFP4 experts keep the aligned layout always (their scale chunks need it).
  const bool zero_pad = !nvf4 && static_cast<int64_t>(T) * k >= int64_t(256) * E_;
  const int padded = (nvf4 || zero_pad) ? 1 : 0;
  int* chunk = reinterpret_cast<int*>(base + L.chunk);
  int* row_off = reinterpret_cast<int*>(base + L.row_off);
  int* mt_off = reinterpret_cast<int*>(base + L.mt_off);
  int* mt2_off = reinterpret_cast<int*>(base + L.mt2_off);
  int* row_cnt = reinterpret_cast<int*>(base + L.row_cnt);
  int* src = reinterpret_cast<int*>(base + L.src);
  int* inv = reinterpret_cast<int*>(base + L.inv);
  void* a_perm = base + L.a_perm;
  uint8_t* sf_u = base + L.sf_u;
  uint8_t* sf_s = base + L.sf_s;
  float* alpha = reinterpret_cast<float*>(base + L.alpha);
  if (L.nchunks == 1) {     // small batches (decode): the three steps in one block
    MOE_TRY(launch_step(dispatch_small_kernel, dim3(1), dim3(256), 0, st,
                        static_cast<const int32_t*>(ids), rows, E_, row_off, mt_off, mt2_off,
                        row_cnt, inv, src, padded, status));
  } else {
    MOE_TRY(launch_step(dispatch_hist_kernel, dim3(L.nchunks), dim3(MEM_THREADS), 0, st,
                        static_cast<const int32_t*>(ids), rows, E_, chunk, status));
    MOE_TRY(launch_step(dispatch_scan_kernel, dim3(1), dim3(256), 0, st, chunk, L.nchunks, E_,
                        row_off, mt_off, mt2_off, row_cnt, padded));
    MOE_TRY(launch_step(dispatch_scatter_kernel, dim3(L.nchunks), dim3(32), 0, st,
                        static_cast<const int32_t*>(ids), rows, E_,
                        static_cast<const int*>(chunk), inv, src));
  }
  const int zero_blocks = zero_pad ? 4 * E_ : 0;
  if (nvf4)
    MOE_TRY(launch_step(pool_quant_kernel, dim3(T), dim3(MEM_THREADS), 0, st,
                        static_cast<const float*>(pooled), W->g_pool,
                        static_cast<const int*>(inv), static_cast<uint8_t*>(a_perm), sf_u, alpha,
                        p, k, c.eps, status));
  else if (exp_f32)
    MOE_TRY(launch_step(pool_permute_kernel<true>, dim3(T + zero_blocks), dim3(MEM_THREADS), 0,
                        st, static_cast<const float*>(pooled), W->g_pool,
                        static_cast<const int*>(inv), a_perm, p, k, c.eps, status,
                        static_cast<const int*>(row_off), static_cast<const int*>(row_cnt),
                        zero_blocks));
  else
    MOE_TRY(launch_step(pool_permute_kernel<false>, dim3(T + zero_blocks), dim3(MEM_THREADS), 0,
                        st, static_cast<const float*>(pooled), W->g_pool,
                        static_cast<const int*>(inv), a_perm, p, k, c.eps, status,
                        static_cast<const int*>(row_off), static_cast<const int*>(row_cnt),
                        zero_blocks));
  E.mark(4);

  // ---- stage: grouped gate/up GEMM + SwiGLU -------------------------------------------
  void* s_buf = base + L.s;
  const int max_mt = (rows + GEMM_BM - 1) / GEMM_BM + E_;
  const int R = static_cast<int>(L.rows);
  if (nvf4) {
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, a_perm, OP_NVF4, p / 2, R, GEMM_BM) ||
        !make_tmap(&tb, W->w13, OP_NVF4, p / 2, static_cast<uint64_t>(E_) * 2 * I, NV_BN))
      return MOE_ERR_CUDA;
    GemmParams P = base_params(status, c.flags);
    P.N = 2 * I; P.K = p; P.bn = NV_BN; P.groups = E_;
    P.row_off = row_off; P.mt_off = mt_off; P.row_cnt = row_cnt;
    P.out = s_buf; P.ld_out = I;
    P.sf_a = sf_u; P.sf_b = W->sf13; P.row_scale = alpha; P.grp_scale = W->gs13;
    P.out_scale = W->gs_act2; P.out_sf = sf_s;
    if (!(c.flags & MOE_FLAG_NVFP4_PAIR)) {   // default: one CTA per 128 x 256 tile
      const int grid = std::min(sms, max_mt * (2 * I / NV_BN));
      MOE_TRY(launch_step(gemm_nvf4_kernel<NV_EPI_SWIGLU_Q>, dim3(grid), dim3(NV_THREADS),
                          nvf4_smem_bytes(), st, ta, tb, ta, P));
    } else {   // CTA pairs over 256-row tiles of each expert (tile prefix: mt2_off)
      CUtensorMap tb128;      // each CTA of a pair loads 128 of the tile's 256 weight rows
      if (!make_tmap(&tb128, W->w13, OP_NVF4, p / 2, static_cast<uint64_t>(E_) * 2 * I, 128))
        return MOE_ERR_CUDA;
      P.mt_off = mt2_off;
      const int clusters = std::min(sms / 2, (R / 256 + E_) * (2 * I / NV_BN));
      MOE_TRY(launch_step(gemm_nvf4_pair_kernel<NV_EPI_SWIGLU_Q>, dim3(2 * clusters),
                          dim3(NV_THREADS), nvf4_pair_smem_bytes(), st, ta, tb128, ta, P));
    }
  } else if (c.flags & MOE_FLAG_WEIGHT_TILES) {
    // weights on the MMA's M side (256-row W13 blocks: 128 gate + 128 up), tokens on N
    CUtensorMap tw, tx;
    if (!make_tmap(&tw, W->w13, k_up, p, static_cast<uint64_t>(E_) * 2 * I, 256) ||
        !make_tmap(&tx, a_perm, k_up, p, R, 128))
      return MOE_ERR_CUDA;
    GemmParams P = base_params(status, c.flags);
    P.N = 2 * I; P.K = p; P.bn = 256; P.groups = E_;
    P.row_off = row_off; P.mt_off = mt_off; P.row_cnt = row_cnt;
    P.out = s_buf; P.ld_out = I; P.out_fmt = exp_f32 ? OUT_TF32 : OUT_F16;
    P.debug_skip_first_load = (c.flags & MOE_FLAG_TEST_TIMEOUT) ? 1 : 0;
    const int grid = std::min(sms, max_mt * (2 * I / 256));
    if (exp_f32)
      MOE_TRY(launch_step(gemm_swap_kernel<OP_TF32, SWAP_SWIGLU>, dim3(grid), dim3(GEMM_THREADS),
                          swap_smem_bytes(), st, tw, tx, P));
    else
      MOE_TRY(launch_step(gemm_swap_kernel<OP_F16, SWAP_SWIGLU>, dim3(grid), dim3(GEMM_THREADS),
                          swap_smem_bytes(), st, tw, tx, P));
  } else {
    // CTA pairs over 256-row tiles of each expert (M = 128 pair tiles for remainders);
    // each CTA of a pair loads half of a 256-row W13 block: 128 gate or 128 up rows
    CUtensorMap ta, ta64, tb, tb64;
    if (!make_tmap(&ta, a_perm, k_up, p, R, GEMM_BM) ||
        !make_tmap(&ta64, a_perm, k_up, p, R, GEMM_BM / 2) ||
        !make_tmap(&tb, W->w13, k_up, p, static_cast<uint64_t>(E_) * 2 * I, W13_GROUP) ||
        !make_tmap(&tb64, W->w13, k_up, p, static_cast<uint64_t>(E_) * 2 * I, W13_GROUP / 2))
      return MOE_ERR_CUDA;
    GemmParams P = base_params(status, c.flags);
    P.N = 2 * I; P.K = p; P.bn = 2 * W13_GROUP; P.groups = E_;
    P.row_off = row_off; P.mt_off = mt2_off; P.row_cnt = row_cnt;
    P.out = s_buf; P.ld_out = I; P.out_fmt = exp_f32 ? OUT_TF32 : OUT_F16;
    // the tiles cover each expert's rows up to its 128-row boundary; with zeroed padding
    // rows of A, storing their s (exact zeros) keeps the down GEMM's padding zero too
    P.pad_rows = zero_pad ? 1 : 0;
    P.debug_skip_first_load = (c.flags & MOE_FLAG_TEST_TIMEOUT) ? 1 : 0;
    CUtensorMap to;
    if (!make_tmap(&to, s_buf, exp_f32 ? OP_TF32 : OP_F16, I, R, 32)) return MOE_ERR_CUDA;
    const int tiles = (rows / 256 + E_) * (2 * I / P.bn);
    if (exp_f32) MOE_TRY((launch_pair<OP_TF32, EPI_SWIGLU>(ta, ta64, tb, tb64, to, P, tiles, sms, st)));
    else MOE_TRY((launch_pair<OP_F16, EPI_SWIGLU>(ta, ta64, tb, tb64, to, P, tiles, sms, st)));
  }
  E.mark(5);

  // ---- stage: grouped down GEMM -> y ------------------------------------------------------
  // y: FP16 (FP32 only for FP32 experts), with FP32 sums of squares of the stored values
  // per 128 columns beside it; the per-expert norm and the weighted sum run in FP32
  void* y_buf = base + L.y;
  float* ssq = reinterpret_cast<float*>(base + L.ssq);
  const bool y_f16 = !exp_f32;
  const int y_fmt = y_f16 ? OUT_F16 : OUT_F32;
  const int y_op = y_f16 ? OP_F16 : OP_TF32;
  if (nvf4) {
    CUtensorMap ta, tb, ty;   // ty: y in 32-row x 64-column FP16 boxes for the epilogue
    if (!make_tmap(&ta, s_buf, OP_NVF4, I / 2, R, GEMM_BM) ||
        !make_tmap(&tb, W->w2, OP_NVF4, I / 2, static_cast<uint64_t>(E_) * p, NV_BN) ||
        !make_tmap(&ty, y_buf, OP_F16, p, R, 32))
      return MOE_ERR_CUDA;
    GemmParams P = base_params(status, c.flags);
    P.N = p; P.K = I; P.bn = NV_BN; P.groups = E_;
    P.row_off = row_off; P.mt_off = mt_off; P.row_cnt = row_cnt;
    P.out = y_buf; P.ld_out = p; P.row_ssq = ssq;
    P.sf_a = sf_s; P.sf_b = W->sf2; P.grp_scale = W->gs2; P.out_scale = W->gs_act2;
    // pairs by default once the experts average a full 256-row pair tile
    const bool pair = (c.flags & MOE_FLAG_NVFP4_PAIR) ||
                      (!(c.flags & MOE_FLAG_NVFP4_ONE_CTA) &&
                       static_cast<int64_t>(c.T) * c.top_k >= int64_t(256) * E_);
    if (!pair) {
      const int grid = std::min(sms, max_mt * (p / NV_BN));
      // experts averaging under 128 rows: tiles are mostly padding and the weights stream
      // from HBM; rows stored directly, with a ring a stage deeper than the boxes allow
      if (static_cast<int64_t>(c.T) * c.top_k < int64_t(128) * E_)
        MOE_TRY(launch_step(gemm_nvf4_kernel<NV_EPI_STORE_Y_ROWS>, dim3(grid), dim3(NV_THREADS),
                            nvf4_smem_bytes(), st, ta, tb, ty, P));
      else
        MOE_TRY(launch_step(gemm_nvf4_kernel<NV_EPI_STORE_Y>, dim3(grid), dim3(NV_THREADS),
                            nvf4_smem_bytes(), st, ta, tb, ty, P));
    } else {
      CUtensorMap tb128;      // each CTA of a pair loads 128 of the tile's 256 weight rows
      if (!make_tmap(&tb128, W->w2, OP_NVF4, I / 2, static_cast<uint64_t>(E_) * p, 128))
        return MOE_ERR_CUDA;
      P.mt_off = mt2_off;
      const int clusters = std::min(sms / 2, (R / 256 + E_) * (p / NV_BN));
      MOE_TRY(launch_step(gemm_nvf4_pair_kernel<NV_EPI_STORE_Y>, dim3(2 * clusters),
                          dim3(NV_THREADS), nvf4_pair_smem_bytes(), st, ta, tb128, ty, P));
    }
  } else if (c.flags & MOE_FLAG_WEIGHT_TILES) {
    // weights on M (128 rows of p), up to 256 tokens on N
    CUtensorMap tw, tx;
    if (!make_tmap(&tw, W->w2, k_down, I, static_cast<uint64_t>(E_) * p, 128) ||
        !make_tmap(&tx, s_buf, k_down, I, R, 256))
      return MOE_ERR_CUDA;
    GemmParams P = base_params(status, c.flags);
    P.N = p; P.K = I; P.bn = 128; P.groups = E_;
    P.row_off = row_off; P.mt_off = mt2_off; P.row_cnt = row_cnt;
    P.out = y_buf; P.ld_out = p; P.out_fmt = y_fmt;
    const int max_mt2 = (rows + 255) / 256 + E_;
    const int grid = std::min(sms, max_mt2 * (p / 128));
    if (exp_f32)
      MOE_TRY(launch_step(gemm_swap_kernel<OP_TF32, SWAP_STORE>, dim3(grid), dim3(GEMM_THREADS),
                          swap_smem_bytes(), st, tw, tx, P));
    else
      MOE_TRY(launch_step(gemm_swap_kernel<OP_F16, SWAP_STORE>, dim3(grid), dim3(GEMM_THREADS),
                          swap_smem_bytes(), st, tw, tx, P));
    const size_t n = static_cast<size_t>(R) * (p / 128);
    const int ssq_grid = static_cast<int>(std::min<size_t>((n + MEM_THREADS - 1) / MEM_THREADS, 4096));
    if (y_f16)
      MOE_TRY(launch_step(row_ssq_kernel<true>, dim3(ssq_grid), dim3(MEM_THREADS), 0, st,
                          static_cast<const void*>(y_buf), R, p, ssq));
    else
      MOE_TRY(launch_step(row_ssq_kernel<false>, dim3(ssq_grid), dim3(MEM_THREADS), 0, st,
                          static_cast<const void*>(y_buf), R, p, ssq));
  } else {
    CUtensorMap ta, tb;
    const int bn = bn_for(p);
    GemmParams P = base_params(status, c.flags);
    P.N = p; P.K = I; P.bn = bn; P.groups = E_;
    P.row_off = row_off; P.row_cnt = row_cnt;
    P.out = y_buf; P.ld_out = p; P.out_fmt = y_fmt; P.row_ssq = ssq;
    if (bn == 256) {    // CTA pairs over 256-row tiles (M = 128 pair tiles for remainders)
      CUtensorMap ta64, to;
      if (!make_tmap(&ta, s_buf, k_down, I, R, GEMM_BM) ||
          !make_tmap(&ta64, s_buf, k_down, I, R, GEMM_BM / 2) ||
          !make_tmap(&tb, W->w2, k_down, I, static_cast<uint64_t>(E_) * p, 128) ||
          !make_tmap(&to, y_buf, y_op, p, R, 32))
        return MOE_ERR_CUDA;
      P.mt_off = mt2_off;
      const int tiles = (rows / 256 + E_) * (p / 256);
      if (exp_f32) MOE_TRY((launch_pair<OP_TF32, EPI_STORE>(ta, ta64, tb, tb, to, P, tiles, sms, st)));
      else MOE_TRY((launch_pair<OP_F16, EPI_STORE>(ta, ta64, tb, tb, to, P, tiles, sms, st)));
    } else {
      if (!make_tmap(&ta, s_buf, k_down, I, R, GEMM_BM) ||
          !make_tmap(&tb, W->w2, k_down, I, static_cast<uint64_t>(E_) * p, bn))
        return MOE_ERR_CUDA;
      P.mt_off = mt_off;
      const int grid = std::min(sms, max_mt * (p / bn));
      if (exp_f32) MOE_TRY((launch_gemm<OP_TF32, EPI_STORE>(ta, tb, P, grid, st)));
      else MOE_TRY((launch_gemm<OP_F16, EPI_STORE>(ta, tb, P, grid, st)));
    }
  }
  E.mark(6);

  // ---- stage: per-expert RMSNorm + FP32 weighted sum -------------------------------------
  void* c_buf = base + L.c;
  {
    const int ccols = combine_cols(p);
    const int cgrid = T * (p / ccols), cthreads = combine_threads(ccols);
    const size_t csmem = combine_smem_bytes(ccols, y_f16);
    const unsigned long long tmo = base_params(status, c.flags).timeout_ns;
#define LMOE_COMBINE(CF, YB)                                                                  \
  MOE_TRY(launch_step(combine_kernel<CF, YB>, dim3(cgrid), dim3(cthreads), csmem, st,          \
                      static_cast<const void*>(y_buf), static_cast<const float*>(ssq),         \
                      static_cast<const int*>(inv), static_cast<const int32_t*>(ids),           \
                      static_cast<const float*>(wts), W->g_exp, c_buf, p, ccols, k, E_, c.eps, \
                      status, tmo))
    if (act_f32) { if (y_f16) LMOE_COMBINE(true, true); else LMOE_COMBINE(true, false); }
    else { if (y_f16) LMOE_COMBINE(false, true); else LMOE_COMBINE(false, false); }
#undef LMOE_COMBINE
  }
  E.mark(7);

  // ---- stage: unpooler GEMM -> out ----------------------------------------------------------
  {
    CUtensorMap ta, tb;
    const int bn = bn_for(d);
    if (!make_tmap(&ta, c_buf, k_proj, p, T, GEMM_BM) ||
        !make_tmap(&tb, W->w_unpool, k_proj, p, d, bn))
      return MOE_ERR_CUDA;
    GemmParams P = base_params(status, c.flags);
    P.M = T; P.N = d; P.K = p; P.bn = bn; P.groups = 0;
    P.b_const = 1;           // W_unpool
    P.out = out; P.ld_out = d; P.out_fmt = c.out == MOE_F32 ? OUT_F32 : OUT_BF16;
    if (sp.unpool > 1) {
      P.ksplit = sp.unpool; P.split_stride = size_t(T) * d; P.out = part; P.out_fmt = OUT_F32;
    }
    const int grid = std::min(sms, mtiles * (d / bn) * sp.unpool);
    if (sp.unpool == 1 && bn == 256) {        // CTA pairs
      CUtensorMap tb2, to;
      if (!make_tmap(&tb2, W->w_unpool, k_proj, p, d, 128) ||
          !make_tmap(&to, out, P.out_fmt == OUT_BF16 ? OP_BF16 : OP_TF32, d, T, 32))
        return MOE_ERR_CUDA;
      const int tiles = ((T + 255) / 256) * (d / 256);
      int bnd_clusters = 0;
      if (bnd) {
        std::lock_guard<std::mutex> lk(g_mu);
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) bnd_clusters = g_dev[dev].bnd_clusters;
      }
      if (bnd && bnd_clusters > 0) {          // the boundary's row pass in this kernel
        P.row_ssq = reinterpret_cast<float*>(base + L.bnd_ssq);
        // test hook: this GEMM's tiles then never complete, so the row workers' bounded
        // waits run out as well
        P.debug_skip_first_load = (c.flags & MOE_FLAG_TEST_TIMEOUT) ? 1 : 0;
        P.bnd = *bnd;
        P.bnd.count = reinterpret_cast<int*>(base + L.bnd_cnt);
        if (act_f32)
          MOE_TRY((launch_pair<OP_TF32, EPI_BOUNDARY>(ta, ta, tb2, tb2, to, P, tiles, sms, st, true,
                                                      bnd_clusters)));
        else
          MOE_TRY((launch_pair<OP_F16, EPI_BOUNDARY>(ta, ta, tb2, tb2, to, P, tiles, sms, st, true,
                                                     bnd_clusters)));
        bnd = nullptr;                        // done
      } else if (act_f32) MOE_TRY((launch_pair<OP_TF32, EPI_STORE>(ta, ta, tb2, tb2, to, P, tiles, sms, st)));
      else MOE_TRY((launch_pair<OP_F16, EPI_STORE>(ta, ta, tb2, tb2, to, P, tiles, sms, st)));
    } else if (act_f32) MOE_TRY((launch_gemm<OP_TF32, EPI_STORE>(ta, tb, P, grid, st)));
    else MOE_TRY((launch_gemm<OP_F16, EPI_STORE>(ta, tb, P, grid, st)));
    if (sp.unpool > 1) {
      const size_t n = size_t(T) * d;
      MOE_TRY(launch_step(splitk_reduce_kernel,
                          dim3(static_cast<int>(std::min<size_t>((n / 4 + 255) / 256, 4096))),
                          dim3(256), 0, st, static_cast<const float*>(part), sp.unpool, n, out,
                          static_cast<int>(c.out == MOE_F32 ? OUT_F32 : OUT_BF16)));
    }
  }
  E.mark(8);
  // no fused row pass for this shape (split-K or 128-wide unpooler tiles): the pass
  if (bnd)
    MOE_TRY(launch_boundary_pass(c, bnd->x, out, bnd->g_post, bnd->gate, bnd->g_next, bnd->x_out,
                                 bnd->h_next, st, sms));
  return MOE_OK;
}

// ---- routing without caller-provided scratch ---------------------------------------------
// Some callers cannot hand the library a workspace: code that runs where no allocator is
// reachable (an engine whose memory is fully reserved up front, a plugin host that
// forbids device allocations after start-up, a replayed CUDA graph that must not grow
// its pool).  moe_route_noalloc serves them from this file-scope array instead.  Every
// GPU that loads the library keeps it until the process exits, so it is kept small:
// status word, h32 [T,d] FP32 for T * d <= NOALLOC_MAX_ELEMS, then the router's split-K
// partial logits (small T: more CTAs share the router weights) in NOALLOC_PART_BYTES.
constexpr size_t NOALLOC_MAX_ELEMS = size_t(1) << 21;   // e.g. T = 256 at d = 8192
constexpr size_t NOALLOC_H32_OFF = 256;
constexpr size_t NOALLOC_PART_OFF = NOALLOC_H32_OFF + NOALLOC_MAX_ELEMS * 4;
constexpr size_t NOALLOC_PART_BYTES = size_t(4) << 20;
constexpr size_t NOALLOC_BYTES = NOALLOC_PART_OFF + NOALLOC_PART_BYTES;   // 12 MiB + 256
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

struct NoAllocDev {
  void* ptr = nullptr;
  bool ready = false;
};
NoAllocDev g_noalloc_dev[64];
std::mutex g_noalloc_mu;

// Device address of the array on the current device, looked up once per device.  In host
// code the array's name only stands for it; the kernels must get this address.
moe_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocDev& D = g_noalloc_dev[dev];
  if (!D.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    D.ptr = p;
    D.ready = true;
  }
  *out = D.ptr;
  return MOE_OK;
}

// K slices of the no-workspace router: the workspace path's split, halved until its
// partial logits fit the array's partial region.
int noalloc_router_split(const moe_config_t& c) {
  const size_t Ep = (c.E + 15) / 16 * 16;
  int ks = split_plan(c).router;
  while (ks > 1 && size_t(ks) * c.T * Ep * 4 > NOALLOC_PART_BYTES) ks /= 2;
  return ks;
}

}  // namespace

// =====================================================================================
extern "C" {

size_t moe_workspace_size(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  return ws_layout(*cfg).total;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255)) return MOE_ERR_WORKSPACE;
  clear_status_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<int*>(ws));
  return last_launch();
}

size_t moe_packed_bytes(const moe_config_t* cfg, int which) {
  if (validate(cfg) != MOE_OK) return 0;
  const moe_config_t& c = *cfg;
  const size_t ea = c.act == MOE_F32 ? 4 : 2;
  const size_t ee = c.expert == MOE_F32 ? 4 : 2;
  const bool q = c.expert == MOE_NVFP4;
  switch (which) {
    case 0: return size_t(c.E) * c.d * 4;
    case 1: return q ? size_t(c.E) * 2 * c.I * c.p / 2 : size_t(c.E) * 2 * c.I * c.p * ee;
    case 2: return q ? size_t(c.E) * c.p * c.I / 2 : size_t(c.E) * c.p * c.I * ee;
    case 3: return size_t(c.p) * c.d * ea;
    case 4: return size_t(c.d) * c.p * ea;
    case 5: return q ? size_t(c.E) * 2 * c.I * c.p / 16 : 0;
    case 6: return q ? size_t(c.E) * c.p * c.I / 16 : 0;
    case 7: return q ? size_t(c.E) * 4 : 0;
    case 8: return q ? size_t(c.E) * 4 : 0;
    default: return 0;
  }
}

moe_status_t moe_pack_weights(const moe_config_t* cfg, const moe_canonical_weights_t* src,
                              float* w_router_out, void* w13_out, void* w2_out,
                              void* w_pool_out, void* w_unpool_out, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config_t& c = *cfg;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool act_f32 = c.act == MOE_F32, exp_f32 = c.expert == MOE_F32;
  if (!src) return MOE_ERR_INVALID_ARG;
  const bool nvf4 = c.expert == MOE_NVFP4;
  if (nvf4 && (w13_out || w2_out)) return MOE_ERR_INVALID_ARG;
  const void* need[] = {src->w_router, src->w_pool, src->w_unpool, w_router_out, w_pool_out,
                        w_unpool_out};
  for (const void* p : need)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (!nvf4 && (!src->w_gate || !src->w_up || !w13_out || !aligned16(src->w_gate) ||
                !aligned16(src->w_up) || !aligned16(w13_out)))
    return MOE_ERR_INVALID_ARG;
  if (!nvf4 && (!src->w_down || !w2_out || !aligned16(src->w_down) || !aligned16(w2_out)))
    return MOE_ERR_INVALID_ARG;
  auto copy = [&](const void* s, void* d, size_t bytes, bool tf32) {
    const size_t n16 = bytes / 16;
    const int grid = static_cast<int>(std::min<size_t>((n16 + 255) / 256, 8192));
    if (tf32) convert_copy_kernel<CONV_TF32><<<grid, 256, 0, st>>>(s, d, n16);
    else convert_copy_kernel<CONV_BF16_TO_F16><<<grid, 256, 0, st>>>(s, d, n16);
    return last_launch();
  };
  MOE_TRY(copy(src->w_router, w_router_out, size_t(c.E) * c.d * 4, true));
  const int es = exp_f32 ? 4 : 2;
  const unsigned rows13 = static_cast<unsigned>(c.E) * 2u * c.I;
  if (!nvf4) {
    if (exp_f32)
      pack_w13_kernel<CONV_TF32><<<rows13, 256, 0, st>>>(src->w_gate, src->w_up, w13_out, c.I, c.p, W13_GROUP, es);
    else
      pack_w13_kernel<CONV_BF16_TO_F16><<<rows13, 256, 0, st>>>(src->w_gate, src->w_up, w13_out, c.I, c.p, W13_GROUP, es);
    MOE_TRY(last_launch());
  }
  if (!nvf4) MOE_TRY(copy(src->w_down, w2_out, size_t(c.E) * c.p * c.I * es, exp_f32));
  const size_t ea = act_f32 ? 4 : 2;
  MOE_TRY(copy(src->w_pool, w_pool_out, size_t(c.p) * c.d * ea, act_f32));
  MOE_TRY(copy(src->w_unpool, w_unpool_out, size_t(c.d) * c.p * ea, act_f32));
  return MOE_OK;
}

moe_status_t moe_quantize_nvfp4(const moe_config_t* cfg, const void* w_gate, const void* w_up,
                                const void* w_down, uint8_t* w13_out, uint8_t* sf13_out,
                                float* gs13_out, uint8_t* w2_out, uint8_t* sf2_out,
                                float* gs2_out, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config_t& c = *cfg;
  if (c.expert != MOE_NVFP4) return MOE_ERR_INVALID_ARG;
  const void* need[] = {w_gate, w_up, w_down, w13_out, sf13_out, gs13_out, w2_out, sf2_out,
                        gs2_out};
  for (const void* p : need)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t E = c.E, I = c.I, p = c.p;
  // global scales: the outputs first hold each expert's amax (FP32 bits), then g
  unsigned* a13 = reinterpret_cast<unsigned*>(gs13_out);
  unsigned* a2 = reinterpret_cast<unsigned*>(gs2_out);
  zero_u32_kernel<<<1, 256, 0, st>>>(a13, c.E);
  zero_u32_kernel<<<1, 256, 0, st>>>(a2, c.E);
  MOE_TRY(last_launch());
  const dim3 grid(64, c.E);
  amax_bf16_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w_gate), I * p, I * p, a13);
  amax_bf16_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w_up), I * p, I * p, a13);
  amax_bf16_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w_down), p * I, p * I, a2);
  MOE_TRY(last_launch());
  global_scale_kernel<<<(c.E + 255) / 256, 256, 0, st>>>(a13, gs13_out, c.E);
  global_scale_kernel<<<(c.E + 255) / 256, 256, 0, st>>>(a2, gs2_out, c.E);
  MOE_TRY(last_launch());
  quantize_weight_kernel<<<static_cast<unsigned>(E * 2 * I), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(w_gate), static_cast<const __nv_bfloat16*>(w_up),
      w13_out, sf13_out, gs13_out, static_cast<int>(2 * I), c.p, NV_W13_GROUP);
  MOE_TRY(last_launch());
  quantize_weight_kernel<<<static_cast<unsigned>(E * p), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(w_down), nullptr, w2_out, sf2_out, gs2_out, c.p, c.I, 0);
  return last_launch();
}

moe_status_t moe_route(const moe_config_t* cfg, const moe_weights_t* W, const void* x,
                       int32_t* ids, float* w, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  return run_layer(cfg, W, x, nullptr, nullptr, nullptr, ids, w, true, ws, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream), nullptr, 0);
}

moe_status_t moe_route_noalloc(const moe_config_t* cfg, const moe_weights_t* W, const void* x,
                               int32_t* ids, float* w, moe_stream_t stream) {
  MOE_TRY(validate(cfg));
  const moe_config_t& c = *cfg;
  if (static_cast<size_t>(c.T) * c.d > NOALLOC_MAX_ELEMS) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_weights(c, W, true, true));
  if (!x || !aligned16(x) || !ids || !w) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int sms = 0;
  MOE_TRY(device_ready(&sms));
  void* scratch = nullptr;
  MOE_TRY(noalloc_scratch(&scratch));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  int* status = reinterpret_cast<int*>(base);
  float* h32 = reinterpret_cast<float*>(base + NOALLOC_H32_OFF);
  float* part = reinterpret_cast<float*>(base + NOALLOC_PART_OFF);
  // the array keeps the previous call's contents: the status word must start at zero
  clear_status_kernel<<<1, 32, 0, st>>>(status);
  MOE_TRY(last_launch());
  if (c.act == MOE_F32)
    norm_in_kernel<true><<<c.T, MEM_THREADS, 0, st>>>(x, W->g_in, h32, nullptr, c.d, c.eps, status);
  else
    norm_in_kernel<false><<<c.T, MEM_THREADS, 0, st>>>(x, W->g_in, h32, nullptr, c.d, c.eps, status);
  MOE_TRY(last_launch());
  const int bn = (c.E + 15) / 16 * 16;
  const int ks = noalloc_router_split(c);
  const int bn_split = bn % 128 == 0 ? 128 : bn;   // as in moe_forward's split router
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, h32, OP_TF32, c.d, c.T, GEMM_BM) ||
      !make_tmap(&tb, W->w_router, OP_TF32, c.d, c.E, ks > 1 ? bn_split : bn))
    return MOE_ERR_CUDA;
  GemmParams P = base_params(status, c.flags);
  P.M = c.T; P.N = bn; P.K = c.d; P.bn = bn; P.groups = 0;
  const int mtiles = (c.T + GEMM_BM - 1) / GEMM_BM;
  if (ks > 1) {     // small T: K slices -> partial logits in the array -> sum + top-k
    P.bn = bn_split;
    P.ksplit = ks; P.split_stride = size_t(c.T) * bn;
    P.out = part; P.ld_out = bn; P.out_fmt = OUT_F32;
    MOE_TRY((launch_gemm<OP_TF32, EPI_STORE>(ta, tb, P,
                                             std::min(sms, mtiles * (bn / bn_split) * ks), st)));
    router_reduce_topk_kernel<<<c.T, 256, 0, st>>>(part, ks, c.T, bn, c.E, c.top_k, ids, w);
    return last_launch();
  }
  P.E = c.E; P.top_k = c.top_k; P.ids = ids; P.wts = w;
  return launch_gemm<OP_TF32, EPI_ROUTER>(ta, tb, P, std::min(sms, mtiles), st);
}

moe_status_t moe_read_noalloc_status(moe_stream_t stream, int32_t* detail) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  MOE_TRY(noalloc_scratch(&scratch));
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpy(h, scratch, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  clear_status_kernel<<<1, 32, 0, st>>>(static_cast<int*>(scratch));
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (detail) *detail = h[1];
  return static_cast<moe_status_t>(h[0]);
}

moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* W, const void* x,
                         const int32_t* ids, const float* w, void* out, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  return run_layer(cfg, W, x, ids, w, out, nullptr, nullptr, false, ws, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream), nullptr, 0);
}

moe_status_t moe_boundary(const moe_config_t* cfg, const void* x, const void* y,
                          const float* g_post, const float* gate, const float* g_next,
                          void* x_out, void* h_next, moe_stream_t stream) {
  const moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  const moe_config_t& c = *cfg;
  if (c.T == 0) return MOE_OK;
  MOE_TRY(check_boundary_buffers(c, x, y, g_post, gate, g_next, x_out, h_next, false));
  int sms = 0;
  MOE_TRY(device_ready(&sms));
  return launch_boundary_pass(c, x, y, g_post, gate, g_next, x_out, h_next,
                              reinterpret_cast<cudaStream_t>(stream), sms);
}

moe_status_t moe_forward_boundary(const moe_config_t* cfg, const moe_weights_t* W,
                                  const void* x, const int32_t* ids, const float* w,
                                  const float* g_post, const float* gate, const float* g_next,
                                  void* y, void* x_out, void* h_next, void* ws, size_t ws_bytes,
                                  moe_stream_t stream) {
  const moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  const moe_config_t& c = *cfg;
  if (c.T > 0) MOE_TRY(check_boundary_buffers(c, x, y, g_post, gate, g_next, x_out, h_next, true));
  BoundaryArgs B{};
  B.x = x; B.x_out = x_out; B.h_next = h_next;
  B.g_post = g_post; B.gate = gate; B.g_next = g_next;
  B.eps = c.eps;
  B.x_f32 = c.act == MOE_F32 ? 1 : 0;
  return run_layer(cfg, W, x, ids, w, y, nullptr, nullptr, false, ws, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream), nullptr, 0, &B);
}

moe_status_t moe_forward_profiled(const moe_config_t* cfg, const moe_weights_t* W,
                                  const void* x, const int32_t* ids, const float* w,
                                  void* out, void* ws, size_t ws_bytes, moe_stream_t stream,
                                  moe_event_t* events, int n_events) {
  if (n_events < 0 || (n_events > 0 && !events)) return MOE_ERR_INVALID_ARG;
  return run_layer(cfg, W, x, ids, w, out, nullptr, nullptr, false, ws, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream),
                   reinterpret_cast<cudaEvent_t*>(events), n_events);
}

int moe_num_stages(void) { return STG_COUNT; }

const char* moe_stage_name(int stage) {
  return (stage >= 0 && stage < STG_COUNT) ? kStageNames[stage] : "";
}

int moe_forward_launches(const moe_config_t* cfg, int route_internally) {
  if (validate(cfg) != MOE_OK || cfg->T == 0) return 0;
  // norm, [router], pooler, 4 dispatch kernels (2 for one chunk of pairs), gate/up, down,
  // combine, unpooler, plus one reduction per split-K GEMM
  const SplitPlan sp = split_plan(*cfg);
  // the weight-row down GEMM leaves the row sums of squares to one more kernel
  const int ssq_pass = (cfg->flags & MOE_FLAG_WEIGHT_TILES) && cfg->expert != MOE_NVFP4 ? 1 : 0;
  const int one_chunk = ws_layout(*cfg).nchunks == 1 ? 2 : 0;
  return 10 - one_chunk + (route_internally ? 1 + (sp.router > 1) : 0) + (sp.pool > 1) +
         (sp.unpool > 1) + ssq_pass;
}

int moe_workspace_offsets(const moe_config_t* cfg, size_t* offsets, int n) {
  if (validate(cfg) != MOE_OK || !offsets || n <= 0) return 0;
  const WsLayout L = ws_layout(*cfg);
  const size_t all[18] = {L.h32, L.h16, L.ids, L.wts, L.pooled, L.row_off, L.src, L.inv,
                          L.a_perm, L.s, L.y, L.c, L.sf_u, L.sf_s, L.alpha, L.row_cnt,
                          L.bnd_ssq, L.bnd_cnt};
  const int m = n < 18 ? n : 18;
  for (int i = 0; i < m; ++i) offsets[i] = all[i];
  return m;
}

moe_status_t moe_read_status(void* ws, size_t ws_bytes, moe_stream_t stream, int32_t* detail) {
  if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  clear_status_kernel<<<1, 32, 0, st>>>(static_cast<int*>(ws));
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (detail) *detail = h[1];
  return static_cast<moe_status_t>(h[0]);
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device index check failed";
    default: return "unknown status";
  }
}

}  // extern "C"
