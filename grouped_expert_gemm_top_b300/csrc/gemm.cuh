// Persistent, warp-specialised grouped GEMM on the 5th-generation tensor cores.
//
//   D_g = A_g * B_g^T   for every group g (one group per expert),
//
// with bf16 operands staged in shared memory by TMA tiled loads, tcgen05.mma
// accumulating in fp32 in tensor memory, and a fused epilogue that reads TMEM
// with tcgen05.ld.  This is the "sort the tokens by expert, then one grouped
// matrix multiplication, with no copy of the expert parameters" step of the
// grouped_mm expert backend (NeMo AutoModel blog, "专家后端 / Expert backends"
// table): the expert weights are read in place from the fused [E, ...] 3-D
// tensors, and the activations are read from their expert-sorted copy.
//
// Roles (192 threads, one CTA per SM, static round-robin over tiles):
//   warp 0     TMA producer: fills a STAGES-deep ring of (A, B) k-blocks
//   warp 1     TMEM allocator and single-thread UMMA issuer
//   warps 2-5  epilogue: warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31
// Two TMEM accumulators (2 x BN fp32 columns) let the epilogue of tile i run
// while the mainloop of tile i+1 fills the other one.
//
// Schedules:
//   RAGGED_M  groups are row ranges of A/D (forward and data-gradient GEMMs);
//             tile = (group, n-block, m-block), m-block fastest so M-tiles that
//             share a weight tile run on neighbouring CTAs at the same time.
//   RAGGED_K  groups are K ranges (weight-gradient GEMMs): D_g is a full
//             M x N matrix per expert, K = the expert's token rows; an expert
//             with no rows gets an exact zero gradient.  The same schedule with
//             equal K slices (ksplit) gives split-K partial products.
#pragma once
#include <cuda.h>

#include "ptx.cuh"

namespace moe {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kGemmThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kMaxGroups = 256;
constexpr int kEpiSmemBytesDecl = 4 * 3 * 2048;  // epilogue staging (see the epilogue section)

enum LoadMode : int { KMAJ_TILE = 0, MN_TILE = 2 };
enum Sched : int { RAGGED_M = 0, RAGGED_K = 1 };
enum Epi : int { EPI_STORE_F32 = 0, EPI_SWIGLU = 1, EPI_STORE = 2, EPI_DGRAD_SWIGLU = 3 };

struct GemmArgs {
  int M, N, K;           // see Sched: the ragged one is taken from the groups
  int G;                 // number of groups
  const int32_t* offsets;  // [G+1] row offsets (unpadded); nullptr: one group
  int single_rows;       // rows of the one group when offsets == nullptr
  int ksplit;            // RAGGED_K without offsets: group g = K rows [g*ksplit, (g+1)*ksplit)
  int padded;            // 1: groups start on 128-row boundaries of a padded row space
  // EPI_STORE (bf16) / EPI_STORE_F32 (fp32; f32_tma: row stride allows TMA stores)
  __nv_bfloat16* d; float* d_f32; long long ldd; long long d_group_stride; int f32_tma;
  // EPI_SWIGLU (inter = intermediate size I)
  __nv_bfloat16* gu_out; __nv_bfloat16* h_out; int inter;
  // EPI_DGRAD_SWIGLU
  const __nv_bfloat16* gu_saved; const int32_t* perm_slot; const float* slot_w;
  __nv_bfloat16* dgu_out; __nv_bfloat16* hw_out; float* dw_part;
  int* status;
};

template <int BN_, int STAGES_, int AL_, int BL_, int SCH_, int EPI_, bool B3D_, bool SWIGLU_B_>
struct GemmCfg {
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr int AL = AL_;
  static constexpr int BL = BL_;
  static constexpr int SCH = SCH_;
  static constexpr int EPI = EPI_;
  static constexpr bool B3D = B3D_;
  static constexpr bool SWIGLU_B = SWIGLU_B_;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // K-major B is loaded in boxes of at most 128 rows.
  static constexpr int B_BOX_ROWS = BN < 128 ? BN : 128;
  static constexpr int B_NBOX = BN / B_BOX_ROWS;
  static constexpr bool A_MN = (AL == MN_TILE);
  static constexpr bool B_MN = (BL == MN_TILE);
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, A_MN, B_MN);
  static constexpr bool TMA_OUT = true;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + (TMA_OUT ? kEpiSmemBytesDecl : 0) + 1024;  // + alignment slack
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N");
  static_assert(!B_MN || BN % 64 == 0, "MN-major B needs 64-wide groups");
  static_assert(2 * BN <= kTmemCols, "two accumulators must fit TMEM");
  static_assert(SMEM_BYTES <= 227 * 1024 - 8 * 1024, "dynamic + static shared memory per CTA");
};

struct TileInfo {
  int g, mb, nb;
  int row0;        // RAGGED_M: first row of the M-tile in the A/D row space
  int rows_valid;  // RAGGED_M: rows of the group inside this tile (<= 128)
  int kstart;      // RAGGED_K: first K row of the group
  int kblocks;     // number of 64-deep k-blocks
};

struct SmemTables {
  int tile_prefix[kMaxGroups + 1];
  int start[kMaxGroups];   // group start in the (padded or not) row space
  int cnt[kMaxGroups];     // rows of the group
  int off[kMaxGroups];     // unpadded row offset of the group
  int total_tiles;
  int abort_flag;
  uint32_t tmem_base;
};

template <class C>
__device__ __forceinline__ int num_nblocks(const GemmArgs& a) {
  if (C::SWIGLU_B) return (a.inter + C::BN / 2 - 1) / (C::BN / 2);
  return (a.N + C::BN - 1) / C::BN;
}

template <class C>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, const SmemTables& T, int t) {
  TileInfo ti;
  const int nNB = num_nblocks<C>(a);
  if constexpr (C::SCH == RAGGED_M) {
    int lo = 0, hi = a.G - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (T.tile_prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    ti.g = lo;
    const int local = t - T.tile_prefix[lo];
    const int mt = (T.cnt[lo] + BM - 1) / BM;
    ti.nb = local / mt;
    ti.mb = local - ti.nb * mt;
    ti.row0 = T.start[lo] + ti.mb * BM;
    ti.rows_valid = min(BM, T.cnt[lo] - ti.mb * BM);
    ti.kstart = 0;
    ti.kblocks = a.K / BK;
  } else {
    const int nMB = (a.M + BM - 1) / BM;
    const int per = nMB * nNB;
    ti.g = min(t / per, a.G - 1);
    const int local = t - ti.g * per;
    ti.nb = local / nMB;
    ti.mb = local - ti.nb * nMB;
    ti.row0 = ti.mb * BM;
    ti.rows_valid = min(BM, a.M - ti.mb * BM);
    ti.kstart = T.start[ti.g];
    ti.kblocks = (T.cnt[ti.g] + BK - 1) / BK;
  }
  return ti;
}

// ---------------------------------------------------------------- epilogues
// Output path: each epilogue warp owns 32 rows of the tile.  A 32x32 bf16
// block (one 32-column chunk of its rows) is written into a 2 KB shared buffer
// with the 64-byte swizzle (conflict-free 16-byte writes) and stored by one
// TMA bulk-tensor store, so global writes are full, coalesced lines.  Three
// buffers per warp rotate, letting up to three stores be in flight.  A warp
// whose 32 rows are not all inside the group (ragged expert edge) stores its
// valid rows directly instead.
constexpr int kStageBytes = 2048;            // 32 rows x 64 bytes
constexpr int kStagesPerWarp = 3;
constexpr int kEpiSmemBytes = 4 * kStagesPerWarp * kStageBytes;
static_assert(kEpiSmemBytes == kEpiSmemBytesDecl, "epilogue staging size");

struct WarpOut {
  uint32_t buf0;  // this warp's first staging buffer (1024-byte aligned)
  int lane;
  int next;       // next buffer to use
  int inflight;   // committed store groups not yet known to have read their buffer
};

// Write this thread's 32 values (its row of a 32-column chunk) as bf16 into the
// next staging buffer; waits until that buffer's previous store has read it.
__device__ __forceinline__ uint32_t stage_row(WarpOut& w, const float (&v)[32]) {
  if (w.inflight >= kStagesPerWarp) {
    if (w.lane == 0) bulk_wait_read<kStagesPerWarp - 1>();
    __syncwarp();
    w.inflight = kStagesPerWarp - 1;
  }
  const uint32_t buf = w.buf0 + w.next * kStageBytes;
  w.next = (w.next + 1) % kStagesPerWarp;
  const uint32_t row = buf + w.lane * 64;
  const int sw = (w.lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4(row + ((q ^ sw) << 4), pack_bf16x2(v[8 * q + 0], v[8 * q + 1]),
                 pack_bf16x2(v[8 * q + 2], v[8 * q + 3]), pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                 pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
  return buf;
}

// fp32 variant: 16 values (64 bytes) of this thread's row, v[16*half .. 16*half+15].
__device__ __forceinline__ uint32_t stage_row_f32(WarpOut& w, const float (&v)[32], int half) {
  if (w.inflight >= kStagesPerWarp) {
    if (w.lane == 0) bulk_wait_read<kStagesPerWarp - 1>();
    __syncwarp();
    w.inflight = kStagesPerWarp - 1;
  }
  const uint32_t buf = w.buf0 + w.next * kStageBytes;
  w.next = (w.next + 1) % kStagesPerWarp;
  const uint32_t row = buf + w.lane * 64;
  const int sw = (w.lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int b = 16 * half + 4 * q;
    st_shared_v4(row + ((q ^ sw) << 4), __float_as_uint(v[b]), __float_as_uint(v[b + 1]),
                 __float_as_uint(v[b + 2]), __float_as_uint(v[b + 3]));
  }
  return buf;
}

__device__ __forceinline__ void stage_store(WarpOut& w, uint32_t buf, const CUtensorMap* map, int x,
                                            int y, int z, bool three_d) {
  fence_proxy_async_smem();
  __syncwarp();
  if (w.lane == 0) {
    if (three_d) tma_store_3d(map, buf, x, y, z);
    else tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
  __syncwarp();
  ++w.inflight;
}

template <class C>
__device__ __forceinline__ void store_row_chunk_bf16(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    p[q] = w;
  }
}

__device__ __forceinline__ void load_row_chunk_bf16(const __nv_bfloat16* src, float (&v)[32]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = __ldg(p + q);
    v[8 * q + 0] = bf16lo(w.x); v[8 * q + 1] = bf16hi(w.x);
    v[8 * q + 2] = bf16lo(w.y); v[8 * q + 3] = bf16hi(w.y);
    v[8 * q + 4] = bf16lo(w.z); v[8 * q + 5] = bf16hi(w.z);
    v[8 * q + 6] = bf16lo(w.w); v[8 * q + 7] = bf16hi(w.w);
  }
}

// silu(g) = g * sigmoid(g), with CUDA's fast exponential and division intrinsics.
__device__ __forceinline__ float sigmoid_f(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
__device__ __forceinline__ float silu_f(float g) { return g * sigmoid_f(g); }

// fp32 output (split-K router partials).  RAGGED_K: D is the group's (split's)
// M x N slice, map tmD0 3-D [groups][M][N] with 16x32 fp32 boxes.
template <class C>
__device__ void epilogue_store_f32(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                                   int row_in_tile, WarpOut& w, const CUtensorMap* tmD0) {
  const int quad = row_in_tile >> 5;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool warp_full = a.f32_tma && quad * 32 + 32 <= ti.rows_valid;
  const int n0 = ti.nb * C::BN;
  constexpr bool k3 = C::SCH == RAGGED_K;
  float* base = a.d_f32 + (k3 ? (long long)ti.g * a.d_group_stride : 0);
  const long long row = (k3 ? ti.mb * BM : ti.row0) + row_in_tile;
  const int y = (k3 ? ti.mb * BM : ti.row0) + quad * 32;
  float v[32];
#pragma unroll 1
  for (int c = 0; c < (C::BN + 31) / 32; ++c) {
    const int col = n0 + c * 32;
    if (col >= a.N) break;
    if (ti.kblocks > 0) tmem_ld32(tacc + c * 32, v);
    else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
    }
    if (warp_full) {
      stage_store(w, stage_row_f32(w, v, 0), tmD0, col, y, ti.g, k3);
      if (col + 16 < a.N) stage_store(w, stage_row_f32(w, v, 1), tmD0, col + 16, y, ti.g, k3);
    } else if (valid) {
      float* dst = base + row * a.ldd + col;
      for (int i = 0; i < 32 && col + i < a.N; ++i) dst[i] = v[i];
    }
  }
}

// Gate/up epilogue: acc columns [0, BN/2) are gate, [BN/2, BN) up, for the
// intermediate columns n0 .. n0+BN/2-1.  Writes g, u (bf16, for the backward)
// and h = silu(g) * u.  Maps: tmD0 = gu_out [rows, 2I], tmD1 = h_out [rows, I].
template <class C>
__device__ void epilogue_swiglu(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                                int row_in_tile, WarpOut& w, const CUtensorMap* tmD0,
                                const CUtensorMap* tmD1) {
  const int quad = row_in_tile >> 5;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool warp_full = quad * 32 + 32 <= ti.rows_valid;
  const long long r = ti.row0 + row_in_tile;
  const int y = ti.row0 + quad * 32;
  const int I = a.inter;
  constexpr int HALF = C::BN / 2;
  const int n0 = ti.nb * HALF;
  float g[32], u[32];
#pragma unroll 1
  for (int c = 0; c < HALF / 32; ++c) {
    const int j = n0 + c * 32;
    if (j >= I) break;
    tmem_ld32(tacc + c * 32, g);
    tmem_ld32(tacc + HALF + c * 32, u);
    if (warp_full) {
      if (a.gu_out) {
        stage_store(w, stage_row(w, g), tmD0, j, y, 0, false);
        stage_store(w, stage_row(w, u), tmD0, I + j, y, 0, false);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) g[i] = silu_f(g[i]) * u[i];
      stage_store(w, stage_row(w, g), tmD1, j, y, 0, false);
    } else if (valid) {
      if (a.gu_out) {
        store_row_chunk_bf16<C>(a.gu_out + r * (2LL * I) + j, g);
        store_row_chunk_bf16<C>(a.gu_out + r * (2LL * I) + I + j, u);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) g[i] = silu_f(g[i]) * u[i];
      store_row_chunk_bf16<C>(a.h_out + r * (long long)I + j, g);
    }
  }
}

// Plain bf16 output.  RAGGED_M: D rows are the tile's rows (map tmD0 2-D);
// RAGGED_K: D is the group's full M x N matrix (map tmD0 3-D, group = depth).
template <class C>
__device__ void epilogue_store(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                               int row_in_tile, WarpOut& w, const CUtensorMap* tmD0) {
  const int quad = row_in_tile >> 5;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool warp_full = quad * 32 + 32 <= ti.rows_valid;
  const int n0 = ti.nb * C::BN;
  constexpr bool k3 = C::SCH == RAGGED_K;
  const long long row = (k3 ? ti.mb * BM : ti.row0) + row_in_tile;
  const int y = (k3 ? ti.mb * BM : ti.row0) + quad * 32;
  float v[32];
#pragma unroll 1
  for (int c = 0; c < C::BN / 32; ++c) {
    const int col = n0 + c * 32;
    if (col >= a.N) break;
    if (ti.kblocks == 0) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
    } else {
      tmem_ld32(tacc + c * 32, v);
    }
    if (warp_full) {
      stage_store(w, stage_row(w, v), tmD0, col, y, ti.g, k3);
    } else if (valid) {
      __nv_bfloat16* base = a.d + (k3 ? (long long)ti.g * a.d_group_stride : 0);
      store_row_chunk_bf16<C>(base + row * a.ldd + col, v);
    }
  }
}

// Down-projection data gradient with the SwiGLU backward fused in.
// acc = dh_unw = dout[token] * W_down[e]  (columns n0.. of the intermediate)
// From the saved pre-activations (g, u): h = silu(g) u; dw partial = <acc, h>;
// dh = w acc; dg = dh u s (1 + g (1 - s)); du = dh silu(g); hw = w h.
// Maps: tmD0 = dgu_out [rows, 2I], tmD1 = hw_out [rows, I].  In the padded
// layout the rows past the expert's tokens are written as exact zeros.
template <class C>
__device__ void epilogue_dgrad_swiglu(const GemmArgs& a, const SmemTables& T, const TileInfo& ti,
                                      uint32_t tacc, int row_in_tile, WarpOut& w,
                                      const CUtensorMap* tmD0, const CUtensorMap* tmD1) {
  const int quad = row_in_tile >> 5;
  const long long p = ti.row0 + row_in_tile;  // row in the (padded) row space
  const int y = ti.row0 + quad * 32;
  const int I = a.inter;
  const int n0 = ti.nb * C::BN;
  const int nNB = (I + C::BN - 1) / C::BN;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool pad_row = !valid && a.padded;
  const bool warp_full = a.padded || quad * 32 + 32 <= ti.rows_valid;
  long long r = p;  // row of the saved (unpadded) forward tensors
  float wt = 1.f;
  if (valid) {
    if (a.padded) r = T.off[ti.g] + ti.mb * BM + row_in_tile;
    if (a.slot_w) wt = __ldg(a.slot_w + __ldg(a.perm_slot + r));
  }
  float acc[32], g[32], u[32];
  float dwp = 0.f;
#pragma unroll 1
  for (int c = 0; c < C::BN / 32; ++c) {
    const int j = n0 + c * 32;
    if (j >= I) break;
    tmem_ld32(tacc + c * 32, acc);
    if (valid) {
      load_row_chunk_bf16(a.gu_saved + r * (2LL * I) + j, g);
      load_row_chunk_bf16(a.gu_saved + r * (2LL * I) + I + j, u);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float s = sigmoid_f(g[i]);
        const float sl = g[i] * s;
        const float h = sl * u[i];
        dwp = fmaf(acc[i], h, dwp);
        const float dh = wt * acc[i];
        const float dg = dh * u[i] * s * (1.0f + g[i] * (1.0f - s));
        const float du = dh * sl;
        g[i] = dg;
        u[i] = du;
        acc[i] = wt * h;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) g[i] = u[i] = acc[i] = 0.f;
    }
    if (warp_full) {
      stage_store(w, stage_row(w, g), tmD0, j, y, 0, false);
      stage_store(w, stage_row(w, u), tmD0, I + j, y, 0, false);
      stage_store(w, stage_row(w, acc), tmD1, j, y, 0, false);
    } else if (valid || pad_row) {
      store_row_chunk_bf16<C>(a.dgu_out + p * (2LL * I) + j, g);
      store_row_chunk_bf16<C>(a.dgu_out + p * (2LL * I) + I + j, u);
      store_row_chunk_bf16<C>(a.hw_out + p * (long long)I + j, acc);
    }
  }
  if (a.dw_part && (valid || pad_row)) a.dw_part[p * nNB + ti.nb] = dwp;
}

// ---------------------------------------------------------------- the kernel
template <class C>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmD0,
                        const __grid_constant__ CUtensorMap tmD1, const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ SmemTables T;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  volatile int* abort_flag = &T.abort_flag;

  // ---- set-up: barriers, TMEM, group tables
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), 128);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    T.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (C::TMA_OUT) {
      tma_prefetch_desc(&tmD0);
      if constexpr (C::EPI == EPI_SWIGLU || C::EPI == EPI_DGRAD_SWIGLU) tma_prefetch_desc(&tmD1);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&T.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2) {
    // group tables (one warp; G <= 256)
    const int nNB = num_nblocks<C>(a);
    const int nMB = (a.M + BM - 1) / BM;
    int run_tiles = 0, run_rows = 0;
    for (int base = 0; base < a.G; base += 32) {
      const int g = base + lane;
      int cnt = 0, off = 0;
      if (g < a.G) {
        if (a.offsets) {
          off = __ldg(a.offsets + g);
          cnt = __ldg(a.offsets + g + 1) - off;
        } else if (a.ksplit > 0) {
          off = g * a.ksplit;
          cnt = min(a.ksplit, a.K - off);
        } else {
          cnt = a.single_rows;
        }
        if (cnt < 0) cnt = 0;
      }
      const int mt = (cnt + BM - 1) / BM;
      // lanes past the last group contribute nothing (no tiles, no rows)
      const int tiles = (g >= a.G) ? 0 : ((C::SCH == RAGGED_M) ? mt * nNB : nMB * nNB);
      const int rows = a.padded ? mt * BM : cnt;
      int ti = tiles, ro = rows;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, ti, d);
        const int y = __shfl_up_sync(0xffffffffu, ro, d);
        if (lane >= d) { ti += x; ro += y; }
      }
      if (g < a.G) {
        T.tile_prefix[g] = run_tiles + ti - tiles;
        T.start[g] = a.padded ? run_rows + ro - rows : off;
        T.cnt[g] = cnt;
        T.off[g] = off;
      }
      run_tiles += __shfl_sync(0xffffffffu, ti, 31);
      run_rows += __shfl_sync(0xffffffffu, ro, 31);
    }
    if (lane == 0) {
      T.tile_prefix[a.G] = run_tiles;
      T.total_tiles = run_tiles;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = T.tmem_base;
  const int total = T.total_tiles;

  if (warp == 0) {
    // ================= TMA producer =================
    int stage = 0;
    uint32_t phase = 0;
    uint32_t filled = 0, fill_parity = 0;  // per stage: armed at least once, parity of last fill
    for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
      const TileInfo ti = decode_tile<C>(a, T, t);
      const int n0 = C::SWIGLU_B ? ti.nb * (C::BN / 2) : ti.nb * C::BN;
      const int m0 = ti.mb * BM;
      bool ok = true;
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, a.status)) { ok = false; break; }
        const uint32_t fb = smem_u32(&full_bar[stage]);
        const uint32_t sA = smem_base + stage * C::STAGE_BYTES;
        const uint32_t sB = sA + C::A_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
        filled |= 1u << stage;
        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
        __syncwarp();
        const int kc = kb * BK;               // K coordinate inside the group
        const int kr = ti.kstart + kc;        // absolute K coordinate (RAGGED_K)
        const int kx = C::SCH == RAGGED_K ? kr : kc;
        // ---- A
        if constexpr (C::AL == KMAJ_TILE) {
          if (lane == 0) tma_load_2d(sA, &tmA, fb, kx, C::SCH == RAGGED_K ? m0 : ti.row0);
        } else {  // MN_TILE: two 64-wide groups along M, 64 k-rows each
          if (lane == 0) {
            tma_load_2d(sA, &tmA, fb, m0, kr);
            tma_load_2d(sA + 8192, &tmA, fb, m0 + 64, kr);
          }
        }
        // ---- B
        if constexpr (C::BL == KMAJ_TILE) {
          if (lane == 0) {
#pragma unroll
            for (int b = 0; b < C::B_NBOX; ++b) {
              const int nc = C::SWIGLU_B ? (b == 0 ? n0 : a.inter + n0) : n0 + b * C::B_BOX_ROWS;
              const uint32_t dst = sB + b * C::B_BOX_ROWS * 128;
              if constexpr (C::B3D) tma_load_3d(dst, &tmB, fb, kc, nc, ti.g);
              else tma_load_2d(dst, &tmB, fb, kx, nc);
            }
          }
        } else if constexpr (C::BL == MN_TILE) {
          if (lane == 0) {
#pragma unroll
            for (int b = 0; b < C::BN / 64; ++b) {
              if constexpr (C::B3D) tma_load_3d(sB + b * 8192, &tmB, fb, n0 + 64 * b, kc, ti.g);
              else tma_load_2d(sB + b * 8192, &tmB, fb, n0 + 64 * b, kr);
            }
          }
        }
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
    }
    if (*abort_flag) {
      // let copies already in flight land before the CTA can exit (bounded)
      for (int s = 0; s < C::STAGES; ++s) {
        if (!((filled >> s) & 1u)) continue;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full_bar[s]), (fill_parity >> s) & 1u) &&
               globaltimer() - t0 < 20000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ================= UMMA issuer =================
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
      const TileInfo ti = decode_tile<C>(a, T, t);
      if (!mbar_wait(smem_u32(&tempty_bar[acc]), acc_phase ^ 1, abort_flag, a.status)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * C::BN;
      bool ok = true;
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        if (!mbar_wait(smem_u32(&full_bar[stage]), phase, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sA = smem_base + stage * C::STAGE_BYTES;
          const uint32_t sB = sA + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = C::A_MN ? smem_desc_sw128(sA + kk * 2048, 8192, 1024)
                                        : smem_desc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t bd = C::B_MN ? smem_desc_sw128(sB + kk * 2048, 8192, 1024)
                                        : smem_desc_sw128(sB + kk * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&empty_bar[stage]));
        }
        __syncwarp();
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) {
        if (ti.kblocks > 0) umma_commit(smem_u32(&tfull_bar[acc]));
        else mbar_arrive(smem_u32(&tfull_bar[acc]));
      }
      __syncwarp();
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (*abort_flag) {
      // wait (bounded) for UMMAs already issued before TMEM is released
      if (lane == 0) {
        umma_commit(smem_u32(&drain_bar));
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&drain_bar), 0) && globaltimer() - t0 < 20000000ull) {
        }
      }
      __syncwarp();
    }
  } else {
    // ================= epilogue =================
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    WarpOut wo;
    wo.buf0 = smem_base + C::STAGES * C::STAGE_BYTES + quad * (kStagesPerWarp * kStageBytes);
    wo.lane = lane;
    wo.next = 0;
    wo.inflight = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
      const TileInfo ti = decode_tile<C>(a, T, t);
      if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, a.status)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * C::BN;
      if constexpr (C::EPI == EPI_STORE_F32) epilogue_store_f32<C>(a, ti, tacc, row_in_tile, wo, &tmD0);
      else if constexpr (C::EPI == EPI_SWIGLU) epilogue_swiglu<C>(a, ti, tacc, row_in_tile, wo, &tmD0, &tmD1);
      else if constexpr (C::EPI == EPI_STORE) epilogue_store<C>(a, ti, tacc, row_in_tile, wo, &tmD0);
      else epilogue_dgrad_swiglu<C>(a, T, ti, tacc, row_in_tile, wo, &tmD0, &tmD1);
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty_bar[acc]));
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    // every TMA store must have completed before the CTA exits
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace moe
