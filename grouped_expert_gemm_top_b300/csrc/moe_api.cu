// Host side of the C ABI declared in include/moe.h: argument validation,
// workspace layout, TMA tensor-map encoding and the launch sequence of every
// call.  Nothing here allocates device memory or synchronises (except
// moe_read_device_status).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "gemm.cuh"
#include "ep.cuh"
#include "gemm_res.cuh"
#include "kernels_misc.cuh"
#include "moe.h"
#include "route.cuh"

namespace {

using moe::GemmArgs;
using moe::GemmCfg;

constexpr int32_t kAbiVersion = 12;
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// ------------------------------------------------------------------ shapes
moe_status check_dims(const moe_dims* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 1 || d->H < 64 || d->E < 1 || d->k < 1 || d->I < 64 || d->I_shared < 0)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->capacity < 0) return MOE_ERR_INVALID_ARG;
  if (d->H % 64 || d->I % 64 || d->I_shared % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->E > moe::kMaxGroups || d->k > d->E || d->k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long S = (long long)d->T * d->k;
  if (S + (long long)d->E * moe::kPadRows >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)d->H * 2 * d->I >= (1LL << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kDwParts = 1;  // column parts of the down data-gradient epilogue (epilogue warps / 4)

struct Layout {
  size_t status, counts, hist, psum_part, route_end, dep_fwd, h, h_sh, fwd_end;
  size_t dep_bwd, dep_bytes;
  size_t poff, dgu, hw, dxs, dwp, dl, dlb, rwp, db_part, dgu_sh, hw_sh, dxs_sh, gu_rc,
      sh_gu_rc, total;
  int sort_blocks;
  long long S, S_pad_max;
  int nNB_I;  // 256-wide column blocks of the intermediate (dgrad-down tiles)
  int nDW;    // dw partials per padded row (column blocks x epilogue column parts)
};

// Split-K of the router weight-gradient GEMM over the tokens: about one wave
// of 128 x 256 tiles on a 148-SM part, splits of a multiple of 64 tokens.  ldE:
// row stride of the dense logit gradient (16-byte multiple for TMA).
struct RwSplit {
  int nsplit, ksplit, ldE;
};
RwSplit rw_split(const moe_dims& d) {
  RwSplit r;
  const int tiles = ((d.E + 127) / 128) * ((d.H + 255) / 256);
  int n = std::max(1, (148 + tiles - 1) / tiles);
  n = std::min(n, (d.T + 63) / 64);
  r.ksplit = ((d.T + n - 1) / n + 63) / 64 * 64;
  r.nsplit = (d.T + r.ksplit - 1) / r.ksplit;
  r.ldE = (d.E + 7) / 8 * 8;
  return r;
}

// bwd: the backward's buffers; recompute: also room for the gate/up
// pre-activations the backward recomputes when the forward did not save them.
Layout make_layout(const moe_dims& d, bool bwd, bool recompute = false) {
  Layout L{};
  L.S = (long long)d.T * d.k;
  L.S_pad_max = L.S + (long long)d.E * (moe::kPadRows - 1);
  L.S_pad_max = (L.S_pad_max + moe::kPadRows - 1) / moe::kPadRows * moe::kPadRows;
  L.sort_blocks = (int)((L.S + moe::kSortChunk - 1) / moe::kSortChunk);
  L.nNB_I = (d.I + 255) / 256;
  L.nDW = L.nNB_I * kDwParts;
  size_t o = 0;
  L.status = o; o += kAlign;
  L.counts = o; o = align_up(o + (size_t)L.sort_blocks * d.E * 4);
  // the router's per-CTA expert counts [E][hist_ld] and probability sums [CTAs][E],
  // sized for the largest cluster (every tile split over kRouteMaxSplits CTAs)
  const size_t route_ctas_max = (size_t)((d.T + moe::kRouteBM - 1) / moe::kRouteBM) * moe::kRouteMaxSplits;
  L.hist = o; o = align_up(o + (size_t)d.E * ((route_ctas_max + 3) / 4 * 4) * 4);
  L.psum_part = o; o = align_up(o + route_ctas_max * d.E * 4);
  L.route_end = o;
  // cross-kernel overlap: one flag per 256-row block of the sorted (or padded)
  // rows, then the consumer's unit counter; forward and backward each have one
  L.dep_bytes = ((size_t)(L.S + 255 * (long long)d.E) / 256 + d.E + 2) * 4;
  L.dep_fwd = o; o = align_up(o + L.dep_bytes);
  L.h = o; o = align_up(o + (size_t)L.S * d.I * 2);
  L.h_sh = o; o = align_up(o + (size_t)d.T * d.I_shared * 2);
  L.fwd_end = o;
  if (bwd) {
    const size_t P = (size_t)L.S_pad_max;
    L.dep_bwd = o; o = align_up(o + L.dep_bytes);
    L.poff = o; o = align_up(o + (size_t)(d.E + 1) * 4);
    L.dgu = o; o = align_up(o + P * 2 * d.I * 2);
    L.hw = o; o = align_up(o + P * d.I * 2);
    L.dxs = o; o = align_up(o + P * d.H * 2);
    L.dwp = o; o = align_up(o + P * L.nDW * 4);
    L.dl = o; o = align_up(o + (size_t)L.S * 4);
    const RwSplit rs = rw_split(d);
    L.dlb = o; o = align_up(o + (size_t)d.T * rs.ldE * 2);
    L.rwp = o; o = align_up(o + (size_t)rs.nsplit * d.E * d.H * 4);
    L.db_part = o; o = align_up(o + (size_t)((d.T + moe::kAuxDlWarps - 1) / moe::kAuxDlWarps) * d.E * 4);
    L.dgu_sh = o; o = align_up(o + (size_t)d.T * 2 * d.I_shared * 2);
    L.hw_sh = o; o = align_up(o + (size_t)d.T * d.I_shared * 2);
    L.dxs_sh = o; o = align_up(o + (size_t)(d.I_shared ? d.T : 0) * d.H * 2);
    if (recompute) {
      L.gu_rc = o; o = align_up(o + (size_t)L.S * 2 * d.I * 2);
      L.sh_gu_rc = o; o = align_up(o + (size_t)d.T * 2 * d.I_shared * 2);
    }
  }
  L.total = o;
  return L;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ------------------------------------------------------------------ device info
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = cache[dev].load();
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    cache[dev].store(v);
  }
  return v;
}

// ------------------------------------------------------------------ tensor maps
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

// bf16 tensor [depth][rows][inner], zero fill outside.  The swizzle follows the
// box's inner extent: 128-byte rows (64 bf16) use the 128B pattern, 64-byte
// rows (32 bf16, the epilogue's store boxes) the 64B pattern.
CUtensorMapSwizzle swizzle_for(uint32_t box_inner) {
  return box_inner * 2 >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth,
              uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, rows, depth};
  const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const cuuint32_t rank = depth > 1 ? 3 : 2;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box_inner),
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 3-D map whose depth is 1 is still built as 3-D (the kernel passes a group coordinate).
bool make_map3(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth,
               uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, rows, depth};
  const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box_inner),
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ kernel accounting
struct Timing {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> pool;
  struct Rec {
    int id;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::atomic<long long> launches[MOE_K_COUNT];
  Timing() {
    for (auto& l : launches) l.store(0);
  }
};

Timing& timing() {
  static Timing t;
  return t;
}

cudaEvent_t pooled_event() {
  Timing& T = timing();
  std::lock_guard<std::mutex> g(T.mu);
  if (!T.pool.empty()) {
    cudaEvent_t e = T.pool.back();
    T.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Counts one launch of `id`; while timing is on, brackets it with events.
struct KernelScope {
  int id;
  cudaStream_t st;
  cudaEvent_t a = nullptr;
  KernelScope(int id_, cudaStream_t st_) : id(id_), st(st_) {
    Timing& T = timing();
    T.launches[id].fetch_add(1);
    if (T.on) {
      a = pooled_event();
      if (a && cudaEventRecord(a, st) != cudaSuccess) a = nullptr;
    }
  }
  ~KernelScope() {
    if (!a) return;
    cudaEvent_t b = pooled_event();
    if (!b || cudaEventRecord(b, st) != cudaSuccess) return;
    Timing& T = timing();
    std::lock_guard<std::mutex> g(T.mu);
    T.recs.push_back({id, a, b});
  }
};

// ------------------------------------------------------------------ GEMM configs
using moe::EPI_DGRAD_SWIGLU;
using moe::EPI_STORE_F32;
using moe::EPI_STORE;
using moe::EPI_SWIGLU;
using moe::KMAJ_GATHER;
using moe::KMAJ_TILE;
using moe::MN_GATHER;
using moe::MN_TILE;
using moe::RAGGED_K;
using moe::RAGGED_M;

// router weight gradient: A = DL [tokens, E] and B = x [tokens, H], both MN-major
using CfgRouterW = GemmCfg<256, 4, MN_TILE, MN_TILE, RAGGED_K, EPI_STORE_F32, false, false>;
// router term of grad_x with the auxiliary loss: DL [tokens, E] (K-major) x W_r [E, H] (MN-major)
using CfgRouterDx = GemmCfg<256, 3, KMAJ_TILE, MN_TILE, RAGGED_M, EPI_STORE, false, false>;
// Every BN=256 GEMM runs as CTA pairs: 256 x 256 tiles by cta_group::2 UMMAs,
// each CTA staging its 128 A rows and half of the B tile (32 KB per stage).
// The ragged-M GEMMs stream K = 768..2048 per tile through 5 stages with 3
// epilogue store buffers (4 KB) per warp; the weight-gradient GEMMs (K = one
// expert's tokens, output-dominated traffic) use 4 stages and 5 buffers.
template <int STAGES, int AL, int BL, int SCH, int EPI, bool B3D, bool SWIGLU_B, int EPI_WARPS = 4,
          int EPI_BUFS = 3>
using PairCfg = GemmCfg<256, STAGES, AL, BL, SCH, EPI, B3D, SWIGLU_B, EPI_WARPS, true, EPI_BUFS>;
using CfgGateUp = PairCfg<5, KMAJ_GATHER, KMAJ_TILE, RAGGED_M, EPI_SWIGLU, true, true>;
// the inference gate/up GEMM (h only): units of two n-blocks that share every
// token-row stage; its epilogue is not hidden behind the next unit's mainloop,
// so 8 warps share it (48 KB a stage: 4 stages and one 2 KB staging block a
// warp fit).  An expert's last <= 128 rows run as narrow units (the weights
// taking the UMMAs' 256-row side).
using CfgGateUpWide = GemmCfg<256, 4, KMAJ_GATHER, KMAJ_TILE, RAGGED_M, EPI_SWIGLU, true, true, 8,
                              true, 1, false, true, true>;
using CfgGateUpShared = PairCfg<5, KMAJ_TILE, KMAJ_TILE, RAGGED_M, EPI_SWIGLU, false, true>;
// the down GEMM as the consumer of the gate/up GEMM's h, units taken as SMs free up
using CfgDownDyn = GemmCfg<256, 5, KMAJ_TILE, KMAJ_TILE, RAGGED_M, EPI_STORE, true, false, 4, true, 3, true>;
using CfgDownShared = PairCfg<5, KMAJ_TILE, KMAJ_TILE, RAGGED_M, EPI_STORE, false, false>;
using CfgDgradDown =
    PairCfg<5, KMAJ_GATHER, MN_TILE, RAGGED_M, EPI_DGRAD_SWIGLU, true, false, 4 * kDwParts>;
using CfgDgradDownShared = PairCfg<5, KMAJ_TILE, MN_TILE, RAGGED_M, EPI_DGRAD_SWIGLU, false, false>;
// the gate/up data gradient as the consumer of the down data gradient's dgu
using CfgDgradGateUpDyn = GemmCfg<256, 5, KMAJ_TILE, MN_TILE, RAGGED_M, EPI_STORE, true, false, 4, true, 3, true>;
using CfgDgradGateUpShared = PairCfg<5, KMAJ_TILE, MN_TILE, RAGGED_M, EPI_STORE, false, false>;
using CfgWgrad = PairCfg<4, MN_TILE, MN_TILE, RAGGED_K, EPI_STORE, false, false, 4, 5>;
// Expert weight gradients: one operand resident in shared memory for experts
// with at most 256 rows (streamed through the same slots for larger ones).
// gate/up: unit = (expert, n-block of H), x rows gathered once into the resident slots,
//          [dg|du]^T streamed per m-block pair;
// down: unit = (expert, 2 m-blocks of H), dout rows gathered once into the resident slots,
//       w h streamed per n-block.
// Their epilogue (a K = 256 tile's output is as large as its operands) takes a
// large share of each tile: 8 epilogue warps, one 2 KB staging block a warp
// (32 columns), which leaves room for 6 streamed stages beside the resident
// slots, a 6-deep ring: the next unit's first two k-blocks are gathered while
// the running unit computes.
using CfgWgradRes = moe::ResCfg<moe::RES_B, MN_TILE, MN_GATHER, 6, 1, 8, 6, 32>;
using CfgWgradDownRes = moe::ResCfg<moe::RES_A, MN_GATHER, MN_TILE, 6, 1, 8, 6, 32>;

// fp32 [depth][rows][inner] output map with 16x32 boxes (64-byte rows).
bool make_out_map3_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t depth) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, rows, depth};
  const cuuint64_t strides[2] = {inner * 4, inner * rows * 4};
  const cuuint32_t box[3] = {16, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 output (store) maps: 64-column x 32-row boxes, 128-byte swizzle.
bool make_out_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows) {
  return make_map(m, base, inner, rows, 1, 64, 32);
}
bool make_out_map3(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth) {
  return make_map3(m, base, inner, rows, depth, 64, 32);
}

// RES: the resident-operand weight-gradient kernel (same parameters).
// pdl: launch with programmatic stream serialisation (the consumer side of a
// cross-kernel overlap: it may start on SMs the previous grid frees).
template <class C, bool RES = false>
moe_status launch_gemm(int kid, const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& D0,
                       const CUtensorMap& D1, const GemmArgs& a, long long tile_bound,
                       cudaStream_t st, bool pdl = false) {
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, GemmArgs);
  if constexpr (RES) kern = moe::res_gemm_kernel<C>;
  else kern = moe::grouped_gemm_kernel<C>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured.fetch_or(bit);
  }
  if constexpr (C::CL == 2) {
    // 2-CTA clusters; as many as can be resident at once (one CTA per SM)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static std::atomic<int> max_clusters[64];
    int mc = max_clusters[dev & 63].load();
    if (mc == 0) {
      cfg.gridDim = dim3(2 * (sm_count() / 2));
      if (cudaOccupancyMaxActiveClusters(&mc, kern, &cfg) != cudaSuccess ||
          mc <= 0)
        mc = sm_count() / 2;
      max_clusters[dev & 63].store(mc);
    }
    const long long clusters = std::min<long long>(mc, (tile_bound + 1) / 2 + 1);
    if (clusters < 1) return MOE_OK;
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    if (pdl) cfg.numAttrs = 2;
    KernelScope ks(kid, st);
    if (cudaLaunchKernelEx(&cfg, kern, A, B, D0, D1, a) != cudaSuccess)
      return MOE_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  } else {
    long long grid = sm_count();
    if (tile_bound < grid) grid = tile_bound;
    if (grid < 1) return MOE_OK;
    KernelScope ks(kid, st);
    moe::grouped_gemm_kernel<C><<<(int)grid, C::THREADS, C::SMEM_BYTES, st>>>(A, B, D0, D1, a);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
}

GemmArgs base_args(int* status) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.status = status;
  return a;
}

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }



moe_status launched(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The router's cluster shape: one cluster per 128-token tile, split over as many
// CTAs (K slices) as fill the SMs in about one wave, at most 8 and at most one
// 64-deep k-block each.
struct RouteSplit {
  int ntiles, splits, ncta, hist_ld;
};
RouteSplit route_split(const moe_dims& d) {
  RouteSplit r;
  r.ntiles = (d.T + moe::kRouteBM - 1) / moe::kRouteBM;
  r.splits = std::max(1, std::min(moe::kRouteMaxSplits, sm_count() / r.ntiles));
  r.splits = std::min(r.splits, d.H / moe::BK);
  r.ncta = r.ntiles * r.splits;
  r.hist_ld = (r.ncta + 3) / 4 * 4;
  return r;
}

template <int BN>
moe_status launch_route_bn(const CUtensorMap& tX, const CUtensorMap& tW, const moe::RouteArgs& a,
                           int ncta, cudaStream_t st) {
  using C = moe::RouteCfg<BN>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(moe::route_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured.fetch_or(bit);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ncta);
  cfg.blockDim = dim3(moe::kRouteThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KernelScope ks(MOE_K_ROUTER, st);
  if (cudaLaunchKernelEx(&cfg, moe::route_kernel<BN>, tX, tW, a) != cudaSuccess) return MOE_ERR_CUDA;
  return launched(cudaGetLastError());
}

// Router GEMM + softmax + top-k (+ per-CTA expert counts when hist is set, +
// per-CTA probability sums when psum is set), one launch.
moe_status launch_route(const moe_dims& d, int gate_mode, const moe_bf16* x,
                        const moe_bf16* w_router, const float* bias, float* logits_out,
                        int32_t* topk_idx, float* topk_w, float* psum, int32_t* hist,
                        const RouteSplit& rs, int* status, cudaStream_t st) {
  int bn = 16;
  while (bn < d.E) bn *= 2;
  CUtensorMap tX, tW;
  if (!make_map(&tX, x, d.H, d.T, 1, 64, moe::kRouteBM)) return MOE_ERR_CUDA;
  if (!make_map(&tW, w_router, d.H, d.E, 1, 64, (uint32_t)bn)) return MOE_ERR_CUDA;
  moe::RouteArgs a;
  std::memset(&a, 0, sizeof(a));
  a.T = d.T; a.H = d.H; a.E = d.E; a.k = d.k; a.gate_mode = gate_mode;
  a.splits = rs.splits;
  a.bias = bias; a.logits_out = logits_out; a.topk_idx = topk_idx; a.topk_w = topk_w;
  a.psum_part = psum; a.hist = hist; a.hist_ld = rs.hist_ld; a.status = status;
  switch (bn) {
    case 16: return launch_route_bn<16>(tX, tW, a, rs.ncta, st);
    case 32: return launch_route_bn<32>(tX, tW, a, rs.ncta, st);
    case 64: return launch_route_bn<64>(tX, tW, a, rs.ncta, st);
    case 128: return launch_route_bn<128>(tX, tW, a, rs.ncta, st);
    default: return launch_route_bn<256>(tX, tW, a, rs.ncta, st);
  }
}

}  // namespace

// =====================================================================================
extern "C" {

int32_t moe_abi_version(void) { return kAbiVersion; }

const char* moe_status_string(int32_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, misalignment or bad enum)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_DEVICE_INDEX: return "device saw an expert id outside [0, E)";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

moe_status moe_workspace_size(const moe_dims* d, int32_t with_backward, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (with_backward < 0 || with_backward > 2) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*d, with_backward != 0, with_backward == 2).total;
  return MOE_OK;
}

moe_status moe_route(const moe_dims* d, int32_t gate_mode, const moe_bf16* x,
                     const moe_bf16* w_router, const float* router_bias, float* logits_out,
                     int32_t* topk_idx, float* topk_w, float* prob_sum, void* workspace,
                     size_t workspace_bytes, void* stream) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (gate_mode != MOE_GATE_SOFTMAX_TOPK && gate_mode != MOE_GATE_BALANCED)
    return MOE_ERR_INVALID_ARG;
  if (!x || !w_router || !topk_idx || !topk_w || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*d, false);
  if (workspace_bytes < L.route_end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const RouteSplit rs = route_split(*d);
  float* psum = prob_sum ? at<float>(workspace, L.psum_part) : nullptr;
  s = launch_route(*d, gate_mode, x, w_router, router_bias, logits_out, topk_idx, topk_w, psum,
                   nullptr, rs, at<int>(workspace, 0), st);
  if (s != MOE_OK) return s;
  if (prob_sum) {  // sum over tokens of the router softmax (auxiliary loss), fixed order
    KernelScope ks(MOE_K_AUX, st);
    moe::prob_sum_kernel<<<(unsigned)cdiv(d->E, 32), 32 * moe::kProbSumWarps, 0, st>>>(
        psum, rs.ncta, d->E, prob_sum);
  }
  return launched(cudaGetLastError());
}

moe_status moe_route_permute(const moe_dims* d, int32_t gate_mode, const moe_bf16* x,
                             const moe_bf16* w_router, const float* router_bias,
                             float* logits_out, int32_t* topk_idx, float* topk_w,
                             float* prob_sum, int32_t* expert_offsets, int32_t* perm_slot,
                             int32_t* slot_perm, void* workspace, size_t workspace_bytes,
                             void* stream) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (gate_mode != MOE_GATE_SOFTMAX_TOPK && gate_mode != MOE_GATE_BALANCED)
    return MOE_ERR_INVALID_ARG;
  if (!x || !w_router || !topk_idx || !topk_w || !expert_offsets || !perm_slot || !slot_perm ||
      !workspace)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*d, false);
  if (workspace_bytes < L.route_end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const RouteSplit rs = route_split(*d);
  int* status = at<int>(workspace, 0);
  int32_t* hist = at<int32_t>(workspace, L.hist);
  float* psum = prob_sum ? at<float>(workspace, L.psum_part) : nullptr;
  s = launch_route(*d, gate_mode, x, w_router, router_bias, logits_out, topk_idx, topk_w, psum,
                   hist, rs, status, st);
  if (s != MOE_OK) return s;
  {
    KernelScope ks(MOE_K_ROUTE_SORT, st);
    moe::route_sort_kernel<<<(unsigned)rs.ncta, moe::kRouteSortThreads, 0, st>>>(
        topk_idx, d->T, d->k, d->E, rs.splits, rs.ncta, hist, rs.hist_ld, expert_offsets,
        perm_slot, slot_perm, d->capacity, status);
  }
  if (prob_sum) {
    KernelScope ks(MOE_K_AUX, st);
    moe::prob_sum_kernel<<<(unsigned)cdiv(d->E, 32), 32 * moe::kProbSumWarps, 0, st>>>(
        psum, rs.ncta, d->E, prob_sum);
  }
  return launched(cudaGetLastError());
}

moe_status moe_aux_loss(const moe_dims* d, const float* prob_sum, const int32_t* expert_offsets,
                        float alpha, float* loss, float* coef, void* stream) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (!prob_sum || !expert_offsets || (!loss && !coef)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KernelScope ks(MOE_K_AUX, st);
  moe::aux_loss_kernel<<<1, moe::kAuxThreads, 0, st>>>(prob_sum, expert_offsets, d->T, d->E, d->k,
                                                        alpha, loss, coef);
  return launched(cudaGetLastError());
}

moe_status moe_permute(const moe_dims* d, const int32_t* topk_idx, int32_t* expert_offsets,
                       int32_t* perm_slot, int32_t* slot_perm, void* workspace,
                       size_t workspace_bytes, void* stream) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (!topk_idx || !expert_offsets || !perm_slot || !slot_perm || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*d, false);
  if (workspace_bytes < L.hist) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* counts = at<int32_t>(workspace, L.counts);
  { KernelScope ks(MOE_K_SORT_HISTOGRAM, st);
  moe::sort_histogram_kernel<<<L.sort_blocks, moe::kSortThreads, 0, st>>>(
      topk_idx, (int)L.S, d->E, counts, at<int>(workspace, 0)); }
  { KernelScope ks(MOE_K_SORT_SCATTER, st);
  moe::sort_scatter_kernel<<<L.sort_blocks, moe::kSortThreads, 0, st>>>(
      topk_idx, (int)L.S, d->E, L.sort_blocks, counts, expert_offsets, perm_slot, slot_perm,
      d->capacity); }
  return launched(cudaGetLastError());
}

// Grouped gate/up GEMM + SwiGLU of the routed experts (A = token rows of x
// gathered through the sort): gu_out [S,2I] and h_out [S,I] are each optional.
// dep_flags (optional): count each finished unit on its 256-row block for a
// consumer GEMM launched next (the down GEMM), and let it launch early.
// Epilogue passes of the gate/up GEMM per 256-row block (each passes once per
// epilogue warp and CTA of the pair): the consumer's dependency target.
bool gate_up_wide(const moe_bf16* gu_out) { return gu_out == nullptr; }
int gate_up_block_passes(const moe_dims& d, const moe_bf16* gu_out) {
  if (gate_up_wide(gu_out)) return (int)(2 * cdiv(d.I, 256)) * CfgGateUpWide::EPI_WARPS * 2;
  return (int)cdiv(d.I, 128) * CfgGateUp::EPI_WARPS * 2;
}

moe_status launch_gate_up(const moe_dims& d, const moe_bf16* x, const int32_t* expert_offsets,
                          const int32_t* perm_slot, const moe_bf16* w_gate_up, moe_bf16* gu_out,
                          __nv_bfloat16* h_out, int* status, cudaStream_t st,
                          int* dep_flags = nullptr) {
  const int H = d.H, E = d.E, I = d.I;
  const long long S = (long long)d.T * d.k;
  CUtensorMap tB;
  if (!make_map3(&tB, w_gate_up, H, 2LL * I, E, 64, 128)) return MOE_ERR_CUDA;
  const CUtensorMap& tA = tB;  // unused: A is gathered
  CUtensorMap tD0 = tB, tD1 = tB;
  const bool wide = gate_up_wide(gu_out);
  // h leaves in 32 x 64-column blocks, or 32 x 32 in the wide GEMM
  if (h_out && !make_map(&tD1, h_out, I, S, 1, wide ? 32 : 64, 32)) return MOE_ERR_CUDA;
  if (gu_out && !make_out_map(&tD0, gu_out, 2LL * I, S)) return MOE_ERR_CUDA;
  GemmArgs a = base_args(status);
  a.N = 2 * I; a.K = H; a.G = E; a.offsets = expert_offsets; a.cap = d.capacity;
  a.gsrc = reinterpret_cast<const __nv_bfloat16*>(x); a.gld = H; a.gperm = perm_slot;
  a.gdiv = d.k; a.gsrc_rows = d.T;
  a.gu_out = reinterpret_cast<__nv_bfloat16*>(gu_out); a.h_out = h_out; a.inter = I;
  a.dep_flags = dep_flags; a.dep_signal = dep_flags ? 1 : 0;
  if (wide)
    return launch_gemm<CfgGateUpWide>(MOE_K_GATE_UP, tA, tB, tD0, tD1, a,
                                      (cdiv(S, moe::BM) + E) * cdiv(I, 256), st);
  return launch_gemm<CfgGateUp>(MOE_K_GATE_UP, tA, tB, tD0, tD1, a,
                                (cdiv(S, moe::BM) + E) * cdiv(I, 128), st);
}

// The shared expert's gate/up GEMM + SwiGLU (one group, every token).
moe_status launch_shared_gate_up(const moe_dims& d, const moe_bf16* x, const moe_bf16* w_sh_gate_up,
                                 moe_bf16* sh_gu_out, __nv_bfloat16* hs_out, int* status,
                                 cudaStream_t st) {
  const int T = d.T, H = d.H, Is = d.I_shared;
  CUtensorMap tA, tB;
  if (!make_map(&tA, x, H, T, 1, 64, 128)) return MOE_ERR_CUDA;
  if (!make_map(&tB, w_sh_gate_up, H, 2LL * Is, 1, 64, 128)) return MOE_ERR_CUDA;
  CUtensorMap tD0 = tA, tD1 = tA;
  if (hs_out && !make_out_map(&tD1, hs_out, Is, T)) return MOE_ERR_CUDA;
  if (sh_gu_out && !make_out_map(&tD0, sh_gu_out, 2LL * Is, T)) return MOE_ERR_CUDA;
  GemmArgs a = base_args(status);
  a.N = 2 * Is; a.K = H; a.G = 1; a.single_rows = T;
  a.gu_out = reinterpret_cast<__nv_bfloat16*>(sh_gu_out); a.h_out = hs_out; a.inter = Is;
  return launch_gemm<CfgGateUpShared>(MOE_K_SHARED_GATE_UP, tA, tB, tD0, tD1, a,
                                      cdiv(T, moe::BM) * cdiv(Is, 128), st);
}

moe_status moe_grouped_mlp_fwd(const moe_dims* d, const moe_bf16* x,
                               const int32_t* expert_offsets, const int32_t* perm_slot,
                               const moe_bf16* w_gate_up, const moe_bf16* w_down,
                               moe_bf16* gu_saved, moe_bf16* y_perm,
                               const moe_bf16* w_sh_gate_up, const moe_bf16* w_sh_down,
                               moe_bf16* sh_gu_saved, moe_bf16* y_shared, void* workspace,
                               size_t workspace_bytes, void* stream) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (!x || !expert_offsets || !perm_slot || !w_gate_up || !w_down || !y_perm || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (d->I_shared > 0 && (!w_sh_gate_up || !w_sh_down || !y_shared)) return MOE_ERR_INVALID_ARG;
  for (const void* p : {(const void*)x, (const void*)w_gate_up, (const void*)w_down,
                        (const void*)gu_saved, (const void*)y_perm, (const void*)w_sh_gate_up,
                        (const void*)w_sh_down, (const void*)sh_gu_saved, (const void*)y_shared,
                        (const void*)workspace})
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*d, false);
  if (workspace_bytes < L.fwd_end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = at<int>(workspace, 0);
  __nv_bfloat16* h = at<__nv_bfloat16>(workspace, L.h);
  const int T = d->T, H = d->H, E = d->E, I = d->I;
  const long long S = L.S;
  // the down GEMM starts on the SMs the gate/up GEMM frees, each unit once the
  // gate/up GEMM has written its 256 rows of h (every n-block, both CTAs, every
  // epilogue warp)
  int32_t* dep = at<int32_t>(workspace, L.dep_fwd);
  if (cudaMemsetAsync(dep, 0, L.dep_bytes, st) != cudaSuccess) return MOE_ERR_CUDA;
  s = launch_gate_up(*d, x, expert_offsets, perm_slot, w_gate_up, gu_saved, h, status, st, dep);
  if (s != MOE_OK) return s;
  {  // down grouped GEMM
    CUtensorMap tA, tB;
    if (!make_map(&tA, h, I, S, 1, 64, 128)) return MOE_ERR_CUDA;
    if (!make_map3(&tB, w_down, I, H, E, 64, 128)) return MOE_ERR_CUDA;
    CUtensorMap tD;
    if (!make_out_map(&tD, y_perm, H, S)) return MOE_ERR_CUDA;
    GemmArgs a = base_args(status);
    a.N = H; a.K = I; a.G = E; a.offsets = expert_offsets; a.cap = d->capacity;
    a.d = reinterpret_cast<__nv_bfloat16*>(y_perm); a.ldd = H;
    a.dep_flags = dep; a.dep_target = gate_up_block_passes(*d, gu_saved);
    a.sched_counter = dep + (L.dep_bytes / 4 - 1);
    s = launch_gemm<CfgDownDyn>(MOE_K_DOWN, tA, tB, tD, tD, a, (cdiv(S, moe::BM) + E) * cdiv(H, 256), st,
                                /*pdl=*/true);
    if (s != MOE_OK) return s;
  }
  if (d->I_shared > 0) {
    const int Is = d->I_shared;
    __nv_bfloat16* hs = at<__nv_bfloat16>(workspace, L.h_sh);
    s = launch_shared_gate_up(*d, x, w_sh_gate_up, sh_gu_saved, hs, status, st);
    if (s != MOE_OK) return s;
    {
      CUtensorMap tA, tB;
      if (!make_map(&tA, hs, Is, T, 1, 64, 128)) return MOE_ERR_CUDA;
      if (!make_map(&tB, w_sh_down, Is, H, 1, 64, 128)) return MOE_ERR_CUDA;
      CUtensorMap tD;
      if (!make_out_map(&tD, y_shared, H, T)) return MOE_ERR_CUDA;
      GemmArgs a = base_args(status);
      a.N = H; a.K = Is; a.G = 1; a.single_rows = T;
      a.d = reinterpret_cast<__nv_bfloat16*>(y_shared); a.ldd = H;
      s = launch_gemm<CfgDownShared>(MOE_K_SHARED_DOWN, tA, tB, tD, tD, a, cdiv(T, moe::BM) * cdiv(H, 256), st);
      if (s != MOE_OK) return s;
    }
  }
  return MOE_OK;
}

moe_status moe_unpermute_combine(const moe_dims* d, const moe_bf16* y_perm,
                                 const int32_t* slot_perm, const float* topk_w,
                                 const moe_bf16* y_shared, moe_bf16* out, void* stream) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (!y_perm || !slot_perm || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out) || !aligned16(y_shared)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int threads = 256;
  const long long blocks = cdiv((long long)d->T * 32, threads);
  KernelScope ks(MOE_K_COMBINE, st);
  auto* yp = reinterpret_cast<const __nv_bfloat16*>(y_perm);
  auto* ys = reinterpret_cast<const __nv_bfloat16*>(y_shared);
  auto* o = reinterpret_cast<__nv_bfloat16*>(out);
  if (d->k <= 8)
    moe::combine_kernel<8><<<(unsigned)blocks, threads, 0, st>>>(yp, slot_perm, topk_w, ys, o, d->T,
                                                                  d->H, d->k, d->T * d->k);
  else
    moe::combine_kernel<32><<<(unsigned)blocks, threads, 0, st>>>(yp, slot_perm, topk_w, ys, o, d->T,
                                                                   d->H, d->k, d->T * d->k);
  return launched(cudaGetLastError());
}

// The backward in two parts.  Experts: the data gradients of both projections
// (per slot dx, per slot dw partials) and the expert weight gradients.
// Router: the logit gradient, grad_x (the slots' dx summed per token, plus the
// router term) and the router's weight and bias gradients.  moe_layer_bwd runs
// both; the expert-parallel backward runs the experts part on the experts'
// rank (its results handed back in receive order: dx_rows_out, dw_rows_out)
// and the router part on the tokens' rank (from dx_sorted_in, dw_sorted_in:
// the slots' dx and dw in the rank's sorted order).
constexpr int kBwdExperts = 1, kBwdRouter = 2;

static moe_status layer_bwd_impl(const moe_dims* d, const moe_bf16* grad_out, const moe_bf16* x,
                                 const moe_bf16* w_router, const int32_t* topk_idx,
                                 const float* topk_w, const int32_t* expert_offsets,
                                 const int32_t* perm_slot, const int32_t* slot_perm,
                                 const moe_bf16* w_gate_up, const moe_bf16* w_down,
                                 const moe_bf16* gu_saved, const moe_bf16* w_sh_gate_up,
                                 const moe_bf16* w_sh_down, const moe_bf16* sh_gu_saved,
                                 moe_bf16* grad_x, moe_bf16* grad_w_router,
                                 float* grad_router_bias, moe_bf16* grad_w_gate_up,
                                 moe_bf16* grad_w_down, moe_bf16* grad_w_sh_gate_up,
                                 moe_bf16* grad_w_sh_down, const float* router_logits,
                                 const float* aux_coef, void* workspace, size_t workspace_bytes,
                                 void* stream, int parts, moe_bf16* dx_rows_out,
                                 float* dw_rows_out, const moe_bf16* dx_sorted_in,
                                 const float* dw_sorted_in) {
  moe_status s = check_dims(d);
  const bool aux = aux_coef != nullptr;
  const bool do_exp = (parts & kBwdExperts) != 0, do_rt = (parts & kBwdRouter) != 0;
  if (aux && !router_logits) return MOE_ERR_INVALID_ARG;
  if (s != MOE_OK) return s;
  if (!topk_w || !expert_offsets || !perm_slot || !slot_perm || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (do_exp && (!grad_out || !x || !w_gate_up || !w_down || !grad_w_gate_up || !grad_w_down))
    return MOE_ERR_INVALID_ARG;
  if (do_rt && (!x || !w_router || !topk_idx || !grad_x || !grad_w_router))
    return MOE_ERR_INVALID_ARG;
  if (!do_exp && (!dx_sorted_in || !dw_sorted_in || !aligned16(dx_sorted_in)))
    return MOE_ERR_INVALID_ARG;
  if (!do_rt && (!dx_rows_out || !dw_rows_out || !aligned16(dx_rows_out)))
    return MOE_ERR_INVALID_ARG;
  if ((!do_exp || !do_rt) && (d->I_shared > 0 || aux)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->I_shared > 0 && (!w_sh_gate_up || !w_sh_down || !grad_w_sh_gate_up || !grad_w_sh_down))
    return MOE_ERR_INVALID_ARG;
  for (const void* p : {(const void*)grad_out, (const void*)x, (const void*)w_router,
                        (const void*)w_gate_up, (const void*)w_down, (const void*)gu_saved,
                        (const void*)w_sh_gate_up, (const void*)w_sh_down,
                        (const void*)sh_gu_saved, (const void*)grad_x,
                        (const void*)grad_w_router, (const void*)grad_w_gate_up,
                        (const void*)grad_w_down, (const void*)grad_w_sh_gate_up,
                        (const void*)grad_w_sh_down, (const void*)workspace})
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  // pre-activations not saved by the forward are recomputed here (activation
  // recompute), into the workspace
  const bool rc_gu = do_exp && gu_saved == nullptr;
  const bool rc_sh = d->I_shared > 0 && sh_gu_saved == nullptr;
  const Layout L = make_layout(*d, true, rc_gu || rc_sh);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = at<int>(workspace, 0);
  const int T = d->T, H = d->H, E = d->E, I = d->I, k = d->k;
  if (rc_gu) {
    moe_bf16* gu = at<moe_bf16>(workspace, L.gu_rc);
    s = launch_gate_up(*d, x, expert_offsets, perm_slot, w_gate_up, gu, nullptr, status, st);
    if (s != MOE_OK) return s;
    gu_saved = gu;
  }
  if (rc_sh) {
    moe_bf16* gu = at<moe_bf16>(workspace, L.sh_gu_rc);
    s = launch_shared_gate_up(*d, x, w_sh_gate_up, gu, nullptr, status, st);
    if (s != MOE_OK) return s;
    sh_gu_saved = gu;
  }
  const long long P = L.S_pad_max;
  int32_t* poff = at<int32_t>(workspace, L.poff);
  __nv_bfloat16* dgu = at<__nv_bfloat16>(workspace, L.dgu);
  __nv_bfloat16* hw = at<__nv_bfloat16>(workspace, L.hw);
  __nv_bfloat16* dxs = at<__nv_bfloat16>(workspace, L.dxs);
  float* dwp = at<float>(workspace, L.dwp);
  float* dl = at<float>(workspace, L.dl);
  const RwSplit rs = rw_split(*d);
  __nv_bfloat16* dlb = at<__nv_bfloat16>(workspace, L.dlb);
  float* rwp = at<float>(workspace, L.rwp);

  const auto* gob = reinterpret_cast<const __nv_bfloat16*>(grad_out);
  const auto* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  // the gate/up data gradient starts on the SMs the down data gradient frees,
  // each unit once its 256 rows of dgu are written
  int32_t* dep = at<int32_t>(workspace, L.dep_bwd);
  if (do_exp && cudaMemsetAsync(dep, 0, L.dep_bytes, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (do_exp) {  // down-projection data gradient + SwiGLU backward (+ dw partials); A = grad_out rows
    CUtensorMap tB;
    if (!make_map3(&tB, w_down, I, H, E, 64, 64)) return MOE_ERR_CUDA;
    const CUtensorMap& tA = tB;  // unused: A is gathered
    GemmArgs a = base_args(status);
    a.N = I; a.K = H; a.G = E; a.offsets = expert_offsets; a.cap = d->capacity; a.padded = 1;
    a.gsrc = gob; a.gld = H; a.gperm = perm_slot; a.gdiv = k; a.gsrc_rows = T;
    a.poff_out = poff;
    a.inter = I; a.gu_saved = reinterpret_cast<const __nv_bfloat16*>(gu_saved);
    a.perm_slot = perm_slot; a.slot_w = topk_w; a.dgu_out = dgu; a.hw_out = hw; a.dw_part = dwp;
    a.dep_flags = dep; a.dep_signal = 1;
    CUtensorMap tD0, tD1;
    if (!make_out_map(&tD0, dgu, 2LL * I, P) || !make_out_map(&tD1, hw, I, P)) return MOE_ERR_CUDA;
    s = launch_gemm<CfgDgradDown>(MOE_K_DGRAD_DOWN, tA, tB, tD0, tD1, a, cdiv(P, moe::BM) * L.nNB_I, st);
    if (s != MOE_OK) return s;
  }
  if (do_exp) {  // gate/up data gradient -> per-slot dx
    CUtensorMap tA, tB;
    if (!make_map(&tA, dgu, 2LL * I, P, 1, 64, 128)) return MOE_ERR_CUDA;
    if (!make_map3(&tB, w_gate_up, H, 2LL * I, E, 64, 64)) return MOE_ERR_CUDA;
    GemmArgs a = base_args(status);
    a.N = H; a.K = 2 * I; a.G = E; a.offsets = expert_offsets; a.cap = d->capacity; a.padded = 1;
    a.d = dxs; a.ldd = H;
    a.dep_flags = dep; a.dep_target = L.nNB_I * CfgDgradDown::EPI_WARPS * 2;
    a.sched_counter = dep + (L.dep_bytes / 4 - 1);
    CUtensorMap tD;
    if (!make_out_map(&tD, dxs, H, P)) return MOE_ERR_CUDA;
    s = launch_gemm<CfgDgradGateUpDyn>(MOE_K_DGRAD_GATE_UP, tA, tB, tD, tD, a,
                                       cdiv(P, moe::BM) * cdiv(H, 256), st, /*pdl=*/true);
    if (s != MOE_OK) return s;
  }
  __nv_bfloat16* dxs_sh = nullptr;
  if (d->I_shared > 0) {
    const int Is = d->I_shared;
    __nv_bfloat16* dgu_sh = at<__nv_bfloat16>(workspace, L.dgu_sh);
    __nv_bfloat16* hw_sh = at<__nv_bfloat16>(workspace, L.hw_sh);
    dxs_sh = at<__nv_bfloat16>(workspace, L.dxs_sh);
    {
      CUtensorMap tA, tB;
      if (!make_map(&tA, grad_out, H, T, 1, 64, 128)) return MOE_ERR_CUDA;
      if (!make_map(&tB, w_sh_down, Is, H, 1, 64, 64)) return MOE_ERR_CUDA;
      GemmArgs a = base_args(status);
      a.N = Is; a.K = H; a.G = 1; a.single_rows = T;
      a.inter = Is; a.gu_saved = reinterpret_cast<const __nv_bfloat16*>(sh_gu_saved);
      a.dgu_out = dgu_sh; a.hw_out = hw_sh;
      CUtensorMap tD0, tD1;
      if (!make_out_map(&tD0, dgu_sh, 2LL * Is, T) || !make_out_map(&tD1, hw_sh, Is, T))
        return MOE_ERR_CUDA;
      s = launch_gemm<CfgDgradDownShared>(MOE_K_SHARED_DGRAD_DOWN, tA, tB, tD0, tD1, a, cdiv(T, moe::BM) * cdiv(Is, 256), st);
      if (s != MOE_OK) return s;
    }
    {
      CUtensorMap tA, tB;
      if (!make_map(&tA, dgu_sh, 2LL * Is, T, 1, 64, 128)) return MOE_ERR_CUDA;
      if (!make_map(&tB, w_sh_gate_up, H, 2LL * Is, 1, 64, 64)) return MOE_ERR_CUDA;
      GemmArgs a = base_args(status);
      a.N = H; a.K = 2 * Is; a.G = 1; a.single_rows = T;
      a.d = dxs_sh; a.ldd = H;
      CUtensorMap tD;
      if (!make_out_map(&tD, dxs_sh, H, T)) return MOE_ERR_CUDA;
      s = launch_gemm<CfgDgradGateUpShared>(MOE_K_SHARED_DGRAD_GATE_UP, tA, tB, tD, tD, a, cdiv(T, moe::BM) * cdiv(H, 256), st);
      if (s != MOE_OK) return s;
    }
  }
  if (!do_rt) {  // experts part only: the slots' dx and dw back in receive order
    KernelScope ks(MOE_K_EP_ROWS_OUT, st);
    moe::ep_rows_out_kernel<<<(unsigned)cdiv((long long)T * 32, 256), 256, 0, st>>>(
        dxs, dwp, L.nDW, poff, expert_offsets, E, slot_perm, T, H, P,
        reinterpret_cast<__nv_bfloat16*>(dx_rows_out), dw_rows_out, status);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  // router part: the slots' dx and dw partials from the experts part above
  // (padded row space), or given in the sorted order (one partial a slot)
  const __nv_bfloat16* dxs_r =
      do_exp ? dxs : reinterpret_cast<const __nv_bfloat16*>(dx_sorted_in);
  const int32_t* poff_r = do_exp ? poff : expert_offsets;
  const float* dwp_r = do_exp ? dwp : dw_sorted_in;
  const int nDW_r = do_exp ? L.nDW : 1;
  const long long P_r = do_exp ? P : L.S;
  float* dbp = at<float>(workspace, L.db_part);
  const int aux_blocks = (int)cdiv((long long)T, moe::kAuxDlWarps);
  if (do_rt && aux) {
    {  // dense logit gradient with the auxiliary loss's term (and its column sums)
      KernelScope ks(MOE_K_AUX, st);
      if (k <= 8)
        moe::aux_dl_kernel<8><<<(unsigned)aux_blocks, 32 * moe::kAuxDlWarps, 0, st>>>(
            router_logits, aux_coef, topk_idx, topk_w, slot_perm, expert_offsets, poff_r, dwp_r,
            nDW_r, (int)P_r, dl, T, E, k, rs.ldE, dlb, dbp);
      else
        moe::aux_dl_kernel<32><<<(unsigned)aux_blocks, 32 * moe::kAuxDlWarps, 0, st>>>(
            router_logits, aux_coef, topk_idx, topk_w, slot_perm, expert_offsets, poff_r, dwp_r,
            nDW_r, (int)P_r, dl, T, E, k, rs.ldE, dlb, dbp);
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
    // the router's term of grad_x, dense over the experts: grad_x = DL W_r (a
    // small GEMM); the gather below adds the slot gradients into it
    CUtensorMap tA, tB, tD;
    if (!make_map(&tA, dlb, rs.ldE, T, 1, 64, 128)) return MOE_ERR_CUDA;
    if (!make_map(&tB, w_router, H, E, 1, 64, 64)) return MOE_ERR_CUDA;
    if (!make_out_map(&tD, grad_x, H, T)) return MOE_ERR_CUDA;
    GemmArgs a = base_args(status);
    a.N = H; a.K = (int)(cdiv(rs.ldE, moe::BK) * moe::BK); a.G = 1; a.single_rows = T;
    a.d = reinterpret_cast<__nv_bfloat16*>(grad_x); a.ldd = H;
    s = launch_gemm<CfgRouterDx>(MOE_K_ROUTER_DX, tA, tB, tD, tD, a,
                                 cdiv(T, moe::BM) * cdiv(H, 256), st);
    if (s != MOE_OK) return s;
  }
  if (do_rt) {  // router backward + per-token gather of the slot gradients
    KernelScope ks(MOE_K_DX_GATHER, st);
    const unsigned blocks = (unsigned)cdiv((long long)T * 32, 256);
    auto* wr = reinterpret_cast<const __nv_bfloat16*>(w_router);
    auto* gx = reinterpret_cast<__nv_bfloat16*>(grad_x);
    if (k <= 8)
      moe::dx_gather_kernel<8><<<blocks, 256, 0, st>>>(dxs_r, topk_idx, topk_w, slot_perm,
                                                       expert_offsets, poff_r, dwp_r, nDW_r, wr,
                                                       dxs_sh, dl, aux ? nullptr : dlb, rs.ldE,
                                                       aux ? 0 : 1, aux ? 1 : 0, gx, T, H, k, E,
                                                       (int)P_r);
    else
      moe::dx_gather_kernel<32><<<blocks, 256, 0, st>>>(dxs_r, topk_idx, topk_w, slot_perm,
                                                        expert_offsets, poff_r, dwp_r, nDW_r, wr,
                                                        dxs_sh, dl, aux ? nullptr : dlb, rs.ldE,
                                                        aux ? 0 : 1, aux ? 1 : 0, gx, T, H, k, E,
                                                        (int)P_r);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (do_rt) {  // router weight gradient: dW_r = DL^T x, split-K over the tokens (fp32 partials) ...
    CUtensorMap tA, tB, tD;
    if (!make_map(&tA, dlb, rs.ldE, T, 1, 64, 64)) return MOE_ERR_CUDA;
    if (!make_map(&tB, x, H, T, 1, 64, 64)) return MOE_ERR_CUDA;
    if (!make_out_map3_f32(&tD, rwp, H, E, rs.nsplit)) return MOE_ERR_CUDA;
    GemmArgs a = base_args(status);
    a.M = E; a.N = H; a.K = T; a.G = rs.nsplit; a.ksplit = rs.ksplit;
    a.d_f32 = rwp; a.ldd = H; a.d_group_stride = (long long)E * H; a.f32_tma = 1;
    s = launch_gemm<CfgRouterW>(MOE_K_ROUTER_WGRAD, tA, tB, tD, tD, a,
                                (long long)rs.nsplit * cdiv(E, moe::BM) * cdiv(H, 256), st);
    if (s != MOE_OK) return s;
  }
  if (do_rt) {  // ... then the ordered sum of the splits (and the bias gradient)
    KernelScope ks(MOE_K_ROUTER_WGRAD_REDUCE, st);
    const long long n4 = (long long)E * H / 4;
    const long long blocks = std::max<long long>(cdiv(n4, 256), cdiv((long long)E * 32, 256));
    moe::router_wgrad_reduce_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        rwp, rs.nsplit, E, H, expert_offsets, perm_slot, dl, aux ? dbp : nullptr, aux_blocks,
        reinterpret_cast<__nv_bfloat16*>(grad_w_router), grad_router_bias);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (do_exp) {  // dW_down[e] = sum over the expert's rows of dout[token]^T (w h)
    CUtensorMap tA, tB;
    if (!make_map(&tB, hw, I, P, 1, 64, 64)) return MOE_ERR_CUDA;
    tA = tB;  // unused: A = grad_out rows, gathered
    GemmArgs a = base_args(status);
    a.M = H; a.N = I; a.G = E; a.offsets = expert_offsets; a.cap = d->capacity; a.padded = 1;
    a.gsrc = gob; a.gld = H; a.gperm = perm_slot; a.gdiv = k; a.gsrc_rows = T;
    a.d = reinterpret_cast<__nv_bfloat16*>(grad_w_down); a.ldd = I;
    a.d_group_stride = (long long)H * I;
    CUtensorMap tD;
    if (!make_map3(&tD, grad_w_down, I, H, E, CfgWgradDownRes::EPI_COLS, 32)) return MOE_ERR_CUDA;
    a.out_l2[0] = 1;  // evict-first: nothing in the layer reads the weight gradients back
    s = launch_gemm<CfgWgradDownRes, true>(MOE_K_WGRAD_DOWN, tA, tB, tD, tD, a,
                                           (long long)E * cdiv(H, 2 * moe::BM) * cdiv(I, 256), st);
    if (s != MOE_OK) return s;
  }
  if (do_exp) {  // dW_gu[e] = sum over the expert's rows of [dg|du]^T x[token]
    CUtensorMap tA, tB;
    if (!make_map(&tA, dgu, 2LL * I, P, 1, 64, 64)) return MOE_ERR_CUDA;
    tB = tA;  // unused: B = x rows, gathered by token
    GemmArgs a = base_args(status);
    a.M = 2 * I; a.N = H; a.G = E; a.offsets = expert_offsets; a.cap = d->capacity; a.padded = 1;
    a.gsrc = xb; a.gld = H; a.gperm = perm_slot; a.gdiv = k; a.gsrc_rows = T;
    a.d = reinterpret_cast<__nv_bfloat16*>(grad_w_gate_up); a.ldd = H;
    a.d_group_stride = 2LL * I * H;
    CUtensorMap tD;
    if (!make_map3(&tD, grad_w_gate_up, H, 2LL * I, E, CfgWgradRes::EPI_COLS, 32)) return MOE_ERR_CUDA;
    a.out_l2[0] = 1;  // evict-first: nothing in the layer reads the weight gradients back
    s = launch_gemm<CfgWgradRes, true>(MOE_K_WGRAD_GATE_UP, tA, tB, tD, tD, a,
                                       (long long)E * cdiv(2 * I, 2 * moe::BM) * cdiv(H, 256), st);
    if (s != MOE_OK) return s;
  }
  if (d->I_shared > 0) {
    const int Is = d->I_shared;
    __nv_bfloat16* dgu_sh = at<__nv_bfloat16>(workspace, L.dgu_sh);
    __nv_bfloat16* hw_sh = at<__nv_bfloat16>(workspace, L.hw_sh);
    {
      CUtensorMap tA, tB;
      if (!make_map(&tA, grad_out, H, T, 1, 64, 64)) return MOE_ERR_CUDA;
      if (!make_map(&tB, hw_sh, Is, T, 1, 64, 64)) return MOE_ERR_CUDA;
      GemmArgs a = base_args(status);
      a.M = H; a.N = Is; a.G = 1; a.single_rows = T;
      a.d = reinterpret_cast<__nv_bfloat16*>(grad_w_sh_down); a.ldd = Is;
      CUtensorMap tD;
      if (!make_out_map3(&tD, grad_w_sh_down, Is, H, 1)) return MOE_ERR_CUDA;
      a.out_l2[0] = 1;  // evict-first: nothing in the layer reads the weight gradients back
      s = launch_gemm<CfgWgrad>(MOE_K_SHARED_WGRAD_DOWN, tA, tB, tD, tD, a, cdiv(H, moe::BM) * cdiv(Is, 256), st);
      if (s != MOE_OK) return s;
    }
    {
      CUtensorMap tA, tB;
      if (!make_map(&tA, dgu_sh, 2LL * Is, T, 1, 64, 64)) return MOE_ERR_CUDA;
      if (!make_map(&tB, x, H, T, 1, 64, 64)) return MOE_ERR_CUDA;
      GemmArgs a = base_args(status);
      a.M = 2 * Is; a.N = H; a.G = 1; a.single_rows = T;
      a.d = reinterpret_cast<__nv_bfloat16*>(grad_w_sh_gate_up); a.ldd = H;
      CUtensorMap tD;
      if (!make_out_map3(&tD, grad_w_sh_gate_up, H, 2LL * Is, 1)) return MOE_ERR_CUDA;
      a.out_l2[0] = 1;  // evict-first: nothing in the layer reads the weight gradients back
      s = launch_gemm<CfgWgrad>(MOE_K_SHARED_WGRAD_GATE_UP, tA, tB, tD, tD, a, cdiv(2 * Is, moe::BM) * cdiv(H, 256), st);
      if (s != MOE_OK) return s;
    }
  }
  return MOE_OK;
}

moe_status moe_layer_bwd(const moe_dims* d, const moe_bf16* grad_out, const moe_bf16* x,
                         const moe_bf16* w_router, const int32_t* topk_idx, const float* topk_w,
                         const int32_t* expert_offsets, const int32_t* perm_slot,
                         const int32_t* slot_perm, const moe_bf16* w_gate_up,
                         const moe_bf16* w_down, const moe_bf16* gu_saved,
                         const moe_bf16* w_sh_gate_up, const moe_bf16* w_sh_down,
                         const moe_bf16* sh_gu_saved, moe_bf16* grad_x, moe_bf16* grad_w_router,
                         float* grad_router_bias, moe_bf16* grad_w_gate_up,
                         moe_bf16* grad_w_down, moe_bf16* grad_w_sh_gate_up,
                         moe_bf16* grad_w_sh_down, const float* router_logits,
                         const float* aux_coef, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return layer_bwd_impl(d, grad_out, x, w_router, topk_idx, topk_w, expert_offsets, perm_slot,
                        slot_perm, w_gate_up, w_down, gu_saved, w_sh_gate_up, w_sh_down,
                        sh_gu_saved, grad_x, grad_w_router, grad_router_bias, grad_w_gate_up,
                        grad_w_down, grad_w_sh_gate_up, grad_w_sh_down, router_logits, aux_coef,
                        workspace, workspace_bytes, stream, kBwdExperts | kBwdRouter, nullptr,
                        nullptr, nullptr, nullptr);
}

moe_status moe_experts_bwd(const moe_dims* d, const moe_bf16* grad_out_rows,
                           const moe_bf16* x_rows, const float* row_w,
                           const int32_t* expert_offsets, const int32_t* perm_slot,
                           const int32_t* slot_perm, const moe_bf16* w_gate_up,
                           const moe_bf16* w_down, const moe_bf16* gu_saved, moe_bf16* dx_rows,
                           float* dw_rows, moe_bf16* grad_w_gate_up, moe_bf16* grad_w_down,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->k != 1 || d->I_shared != 0 || d->capacity != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  return layer_bwd_impl(d, grad_out_rows, x_rows, nullptr, nullptr, row_w, expert_offsets,
                        perm_slot, slot_perm, w_gate_up, w_down, gu_saved, nullptr, nullptr,
                        nullptr, nullptr, nullptr, nullptr, grad_w_gate_up, grad_w_down, nullptr,
                        nullptr, nullptr, nullptr, workspace, workspace_bytes, stream,
                        kBwdExperts, dx_rows, dw_rows, nullptr, nullptr);
}

moe_status moe_router_bwd(const moe_dims* d, const moe_bf16* x, const moe_bf16* w_router,
                          const int32_t* topk_idx, const float* topk_w,
                          const int32_t* expert_offsets, const int32_t* perm_slot,
                          const int32_t* slot_perm, const moe_bf16* dx_sorted,
                          const float* dw_sorted, moe_bf16* grad_x, moe_bf16* grad_w_router,
                          float* grad_router_bias, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->I_shared != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  return layer_bwd_impl(d, nullptr, x, w_router, topk_idx, topk_w, expert_offsets, perm_slot,
                        slot_perm, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, grad_x,
                        grad_w_router, grad_router_bias, nullptr, nullptr, nullptr, nullptr,
                        nullptr, nullptr, workspace, workspace_bytes, stream, kBwdRouter, nullptr,
                        nullptr, dx_sorted, dw_sorted);
}

moe_status moe_gather_scalars(const void* src, int64_t src_n, const int32_t* idx, int32_t n,
                              int32_t div, void* dst, int32_t* device_status, void* stream) {
  if (n < 0 || src_n < 0 || div < 1) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!src || !idx || !dst) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 3u)
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KernelScope ks(MOE_K_GATHER_SCALARS, st);
  moe::gather_scalars_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(
      static_cast<const uint32_t*>(src), (long long)src_n, idx, n, div, static_cast<uint32_t*>(dst),
      device_status);
  return launched(cudaGetLastError());
}

moe_status moe_gather_rows(const moe_bf16* src, int64_t src_rows, int32_t H, const int32_t* idx,
                           int32_t n, int32_t div, moe_bf16* dst, int32_t* device_status,
                           void* stream) {
  if (n < 0 || src_rows < 0 || div < 1) return MOE_ERR_INVALID_ARG;
  if (H < 8 || H % 8) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (n == 0) return MOE_OK;
  if (!src || !idx || !dst) return MOE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KernelScope ks(MOE_K_GATHER_ROWS, st);
  moe::gather_rows_kernel<<<(unsigned)cdiv((long long)n * 32, 256), 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(src), (long long)src_rows, H, idx, n, div,
      reinterpret_cast<__nv_bfloat16*>(dst), device_status);
  return launched(cudaGetLastError());
}

moe_status moe_ep_receive_layout(int32_t n_src, int32_t E_local, const int32_t* counts, int32_t R,
                                 int32_t* local_offsets, int32_t* recv_perm, int32_t* recv_inv,
                                 int32_t* device_status, void* stream) {
  if (n_src < 1 || E_local < 1 || R < 0) return MOE_ERR_INVALID_ARG;
  if (E_local > moe::kEpMaxLocalExperts || (long long)n_src * E_local > moe::kEpMaxCells)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!counts || !local_offsets || (R > 0 && (!recv_perm || !recv_inv))) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long blocks =
      std::max<long long>(1, std::min<long long>(cdiv(R, moe::kEpLayoutThreads), 4LL * sm_count()));
  KernelScope ks(MOE_K_EP_LAYOUT, st);
  moe::ep_recv_layout_kernel<<<(unsigned)blocks, moe::kEpLayoutThreads, 0, st>>>(
      counts, n_src, E_local, R, local_offsets, recv_perm, recv_inv, device_status);
  return launched(cudaGetLastError());
}

int32_t moe_kernel_count(void) { return MOE_K_COUNT; }

const char* moe_kernel_name(int32_t id) {
  static const char* names[MOE_K_COUNT] = {
      "router", "route_sort", "sort_histogram", "sort_scatter", "gate_up",
      "down", "shared_gate_up", "shared_down", "combine", "dgrad_down",
      "dgrad_gate_up", "shared_dgrad_down", "shared_dgrad_gate_up", "dx_gather",
      "router_wgrad", "wgrad_down", "wgrad_gate_up", "shared_wgrad_down",
      "shared_wgrad_gate_up", "router_wgrad_reduce", "aux_loss", "router_dx", "gather_rows",
      "ep_recv_layout", "ep_rows_out", "gather_scalars"};
  return (id >= 0 && id < MOE_K_COUNT) ? names[id] : "unknown";
}

moe_status moe_timing_enable(int32_t on) {
  Timing& T = timing();
  std::lock_guard<std::mutex> g(T.mu);
  T.on = on != 0;
  return MOE_OK;
}

moe_status moe_kernel_stats(int32_t reset, int64_t* launches, double* event_ms) {
  Timing& T = timing();
  std::lock_guard<std::mutex> g(T.mu);
  moe_status st = MOE_OK;
  if (launches)
    for (int i = 0; i < MOE_K_COUNT; ++i) launches[i] = T.launches[i].load();
  if (event_ms) {
    for (int i = 0; i < MOE_K_COUNT; ++i) event_ms[i] = 0.0;
    for (const auto& r : T.recs) {
      float ms = 0.f;
      if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
        st = MOE_ERR_CUDA;
        continue;
      }
      event_ms[r.id] += ms;
    }
  }
  if (reset) {
    for (auto& l : T.launches) l.store(0);
    for (const auto& r : T.recs) {
      T.pool.push_back(r.a);
      T.pool.push_back(r.b);
    }
    T.recs.clear();
  }
  return st;
}

moe_status moe_read_device_status(void* workspace, size_t workspace_bytes, void* stream,
                                  int32_t clear, int32_t* device_status) {
  if (!workspace || !device_status) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < kAlign) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (clear) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  *device_status = v;
  return MOE_OK;
}

}  // extern "C"

// =====================================================================================
// Allocation-free variant of the expert sort (moe_permute) for callers that
// cannot allocate device memory: code running where cudaMalloc is not allowed
// or not wanted (inside a pre-sized memory pool, a plugin whose host owns all
// device allocations, or a program that must not allocate after start-up), so
// they cannot provide the workspace moe_permute needs.
//
// The sort's only scratch is the per-block expert histogram.  Here it lives in
// a file-scope device array of fixed size; every call on a device shares it.
namespace {

// 65536 int32 = 256 KiB per device; holds ceil(T*k / 1024) * E block counts.
constexpr long long kStaticScratchInts = 65536;

static __device__ __align__(256) int32_t g_sort_scratch[kStaticScratchInts];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
// Per device: the context the address was looked up in, and the address.  A
// device reset (or a torn-down and re-created primary context) reloads the
// module, so the array can move; the address is looked up again whenever the
// current context is not the one it was taken in.
struct ScratchSlot {
  unsigned long long ctx_id;
  int32_t* ptr;
};
ScratchSlot g_scratch_slot[kMaxScratchDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0: none, or the CUDA driver
// could not be reached).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_cur || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_sort_scratch on the current device (in host code the
// symbol's name is only a stand-in, not an address).  Looked up once per
// device and context: the first call on a device (or the first after a device
// reset) performs the lookup.
int32_t* static_scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return nullptr;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  ScratchSlot& slot = g_scratch_slot[dev];
  const unsigned long long ctx = current_context_id();
  if (!slot.ptr || ctx == 0 || ctx != slot.ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sort_scratch) != cudaSuccess || !p) return nullptr;
    slot.ptr = static_cast<int32_t*>(p);
    slot.ctx_id = current_context_id();  // the lookup made the device's context current
  }
  return slot.ptr;
}

}  // namespace

extern "C" moe_status moe_permute_static_scratch(const moe_dims* d, const int32_t* topk_idx,
                                                 int32_t* expert_offsets, int32_t* perm_slot,
                                                 int32_t* slot_perm, int32_t* device_status,
                                                 void* stream) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (!topk_idx || !expert_offsets || !perm_slot || !slot_perm) return MOE_ERR_INVALID_ARG;
  const long long S = (long long)d->T * d->k;
  const long long blocks = (S + moe::kSortChunk - 1) / moe::kSortChunk;
  // the block histograms must fit the fixed device array
  if (blocks * d->E > kStaticScratchInts) return MOE_ERR_UNSUPPORTED_SHAPE;
  int32_t* counts = static_scratch_for_current_device();
  if (!counts) return MOE_ERR_CUDA;
  // Nothing in the array needs clearing: pass 1 writes every (block, expert)
  // count that pass 2 reads.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  { KernelScope ks(MOE_K_SORT_HISTOGRAM, st);
  moe::sort_histogram_kernel<<<(unsigned)blocks, moe::kSortThreads, 0, st>>>(
      topk_idx, (int)S, d->E, counts, device_status); }
  { KernelScope ks(MOE_K_SORT_SCATTER, st);
  moe::sort_scatter_kernel<<<(unsigned)blocks, moe::kSortThreads, 0, st>>>(
      topk_idx, (int)S, d->E, (int)blocks, counts, expert_offsets, perm_slot, slot_perm,
      d->capacity); }
  return launched(cudaGetLastError());
}
