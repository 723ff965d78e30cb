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
// tensors, and the activations' token rows are gathered through the sort
// inside the kernel (no expert-sorted copy of them is written).
//
// Roles (one CTA per SM, static round-robin over tiles, or units handed out
// as CTAs free up in the consumer of a cross-kernel overlap):
//   warp 0     TMA producer: fills a STAGES-deep ring of (A, B) k-blocks
//   warp 1     TMEM allocator and single-thread UMMA issuer
//   warps 2..  EPI_WARPS epilogue warps: warp w reads TMEM lanes
//              32*(w%4) .. 32*(w%4)+31; with 8 epilogue warps the two warps of
//              a lane quadrant split the tile's columns in halves
//   then 4     gather warps (only when an operand is gathered): copy the
//              token rows of that operand straight from the unsorted matrix
//              into the swizzled stage with 16-byte cp.async (LSU path), so
//              no expert-sorted copy of the activations is ever written
//   last       (dynamic units only) the scheduler warp
// Two TMEM accumulators (2 x BN fp32 columns) let the epilogue of tile i run
// while the mainloop of tile i+1 fills the other one; a WIDE unit takes both
// for two n-blocks that share every A stage (see GemmCfg).
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
constexpr int kTmemCols = 512;
constexpr int kMaxGroups = 256;

// TILE: TMA tile loads.  GATHER: rows (K-major: M rows; MN-major: K rows) are
// token rows of a [tokens, ld] matrix, selected through the expert sort.
enum LoadMode : int { KMAJ_TILE = 0, KMAJ_GATHER = 1, MN_TILE = 2, MN_GATHER = 3 };
enum Sched : int { RAGGED_M = 0, RAGGED_K = 1 };
enum Epi : int { EPI_STORE_F32 = 0, EPI_SWIGLU = 1, EPI_STORE = 2, EPI_DGRAD_SWIGLU = 3 };

struct GemmArgs {
  int M, N, K;           // see Sched: the ragged one is taken from the groups
  int G;                 // number of groups
  const int32_t* offsets;  // [G+1] row offsets (unpadded); nullptr: one group
  int cap;               // > 0: a group (expert) takes only its first cap rows (capacity)
  int single_rows;       // rows of the one group when offsets == nullptr
  int ksplit;            // RAGGED_K without offsets: group g = K rows [g*ksplit, (g+1)*ksplit)
  int padded;            // 1: groups start on 128-row boundaries of a padded row space
  // gathered operand: row i of group g reads gsrc[gperm[off_g + min(i, n_g-1)] / gdiv]
  const __nv_bfloat16* gsrc; long long gld; const int32_t* gperm; int gdiv; int gsrc_rows;
  int32_t* poff_out;     // optional: CTA 0 publishes the group starts (padded offsets) here
  // EPI_STORE (bf16) / EPI_STORE_F32 (fp32; f32_tma: row stride allows TMA stores)
  __nv_bfloat16* d; float* d_f32; long long ldd; long long d_group_stride; int f32_tma;
  // EPI_SWIGLU (inter = intermediate size I)
  __nv_bfloat16* gu_out; __nv_bfloat16* h_out; int inter;
  // EPI_DGRAD_SWIGLU
  const __nv_bfloat16* gu_saved; const int32_t* perm_slot; const float* slot_w;
  __nv_bfloat16* dgu_out; __nv_bfloat16* hw_out; float* dw_part;
  int* status;
  // L2 hint of the stores through output map i (0 none, 1 evict-first, 2 evict-last)
  int out_l2[2];
  // Cross-kernel overlap (CTA-pair RAGGED_M GEMMs).  Producer side
  // (dep_signal): every epilogue warp, once the stores of a unit are complete,
  // adds 1 to dep_flags[pair] (pair = the unit's 256-row block: the group's
  // earlier blocks + its m-block pair), and every CTA lets the next grid
  // launch early.  Consumer side (a DYN config): work units come from the
  // counter *sched_counter in the order CTAs ask for them, and a unit's
  // operand loads wait until dep_flags[pair] >= dep_target.
  int* dep_flags;
  int dep_signal;
  int dep_target;
  int* sched_counter;
};

template <int BN_, int STAGES_, int AL_, int BL_, int SCH_, int EPI_, bool B3D_, bool SWIGLU_B_,
          int EPI_WARPS_ = 4, bool PAIR_ = false, int EPI_BUFS_ = 3, bool DYN_ = false,
          bool WIDE_ = false, bool NARROW_ = false>
struct GemmCfg {
  // WIDE: a unit is two adjacent n-blocks that share every A stage: each stage
  // carries two B tiles, and the two TMEM accumulators (all 512 columns) take
  // one n-block each, so the A operand enters the SM once per 2 x BN columns
  // instead of once per BN.  The accumulators are then not double-buffered
  // across units: the next unit's UMMAs wait until the epilogue has drained
  // both.  (Gate/up GEMM with SwiGLU only.)
  static constexpr bool WIDE = WIDE_;
  static constexpr int NSUB = WIDE ? 2 : 1;  // n-blocks (accumulators) per unit
  // NARROW (wide gate/up GEMM): a pair unit whose odd m-block would hold no
  // rows (an expert's last <= 128 rows) swaps the operands' roles: each CTA
  // stages gate and up rows of the same 128 columns, the UMMAs' 256-row sides,
  // and its half of the token rows, their N side (N = the rows rounded up to
  // 32), so the tensor work follows the tokens instead of a full 256-row
  // tile.  TMEM lanes are then intermediate columns and TMEM columns tokens;
  // the epilogue stores each thread's column of h directly.
  static constexpr bool NARROW = NARROW_;
  // DYN: units handed out dynamically (consumer side of a cross-kernel overlap)
  static constexpr bool DYN = DYN_;
  // PAIR: 2-CTA clusters computing one 256 x BN tile with CTA-pair UMMAs
  // (cta_group::2): each CTA stages its own 128 A rows and only HALF of the B
  // tile, the even CTA issues the UMMAs, and each CTA's TMEM receives its own
  // 128 rows.  Per SM this halves the B bytes pulled from L2 per FLOP.
  static constexpr bool PAIR = PAIR_;
  static constexpr int CL = PAIR ? 2 : 1;
  static constexpr int EPI_WARPS = EPI_WARPS_;
  // staging buffers per epilogue warp = TMA stores it keeps in flight; the
  // weight-gradient GEMMs, whose output is most of their traffic, need more
  static constexpr int EPI_BUFS = EPI_BUFS_;
  // bf16 columns of a staging block: 64 (128-byte rows), or 32 (64-byte rows)
  // for the wide gate/up GEMM with 8 epilogue warps, whose 48 KB stages leave
  // room for one 2 KB block a warp
  static constexpr int EPI_COLS = (WIDE_ && EPI_WARPS_ == 8) ? 32 : 64;
  // one staging buffer: 32 rows x EPI_COLS bf16 columns, or 32 rows x 16 fp32 columns
  static constexpr int EPI_BUF_BYTES = EPI_ == EPI_STORE_F32 ? 2048 : EPI_COLS * 64;
  static constexpr bool A_GATHER = (AL_ == KMAJ_GATHER || AL_ == MN_GATHER);
  static constexpr bool B_GATHER = (BL_ == MN_GATHER);
  static constexpr bool GATHER = A_GATHER || B_GATHER;
  static constexpr int GATHER_WARPS = GATHER ? 4 : 0;
  // DYN: one more warp hands out the units and clears their dependencies
  static constexpr int SCHED_WARP = 2 + EPI_WARPS + GATHER_WARPS;
  static constexpr int THREADS = 64 + 32 * (EPI_WARPS + GATHER_WARPS + (DYN_ ? 1 : 0));
  static constexpr int GATHER_LAG = STAGES_ - 2;  // stages a gather thread keeps in flight
  static_assert(!GATHER || GATHER_LAG >= 1, "gathers need >= 3 stages");
  static_assert(BL_ != KMAJ_GATHER, "B is gathered only MN-major");
  static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "4 or 8 epilogue warps");
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr int AL = AL_;
  static constexpr int BL = BL_;
  static constexpr int SCH = SCH_;
  static constexpr int EPI = EPI_;
  static constexpr bool B3D = B3D_;
  static constexpr bool SWIGLU_B = SWIGLU_B_;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B rows (N extent) staged by this CTA
  static constexpr int B_BYTES = NSUB * B_ROWS * BK * 2;  // NSUB tiles of B_ROWS rows
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // K-major B is loaded in boxes of at most 128 rows.
  static constexpr int B_BOX_ROWS = BN < 128 ? BN : 128;
  static constexpr int B_NBOX = BN / B_BOX_ROWS;
  static constexpr bool A_MN = (AL == MN_TILE || AL == MN_GATHER);
  static constexpr bool B_MN = (BL == MN_TILE || BL == MN_GATHER);
  static constexpr int TMA_BYTES = (A_GATHER ? 0 : A_BYTES) + (B_GATHER ? 0 : B_BYTES);
  // The pair's stages complete on the even CTA's full barriers: the TMA bytes of
  // both CTAs and one arrival per gather warp of both CTAs.
  static constexpr uint32_t FULL_TX = TMA_BYTES * (PAIR ? 2 : 1);
  static constexpr uint32_t FULL_ARRIVALS = 1 + (GATHER ? GATHER_WARPS * (PAIR ? 2 : 1) : 0);
  // one arrival per epilogue warp (of both CTAs with PAIR) frees a TMEM accumulator
  static constexpr uint32_t TEMPTY_ARRIVALS = EPI_WARPS * (PAIR ? 2 : 1);
  static_assert(!PAIR || (BN == 256 && !B_GATHER), "PAIR splits a 256-wide TMA-loaded B tile");
  static_assert(!SWIGLU_B || BN == 256, "the gate/up tile pairs 128 gate with 128 up columns");
  static constexpr uint32_t IDESC = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, A_MN, B_MN);
  static constexpr bool TMA_OUT = true;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + (TMA_OUT ? EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES : 0) + 1024;  // + align
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N");
  static_assert(!B_MN || BN % 64 == 0, "MN-major B needs 64-wide groups");
  static_assert(2 * BN <= kTmemCols, "two accumulators must fit TMEM");
  static_assert(SMEM_BYTES <= 227 * 1024 - 8 * 1024, "dynamic + static shared memory per CTA");
  static_assert(!DYN || (PAIR && !GATHER && SCH_ == RAGGED_M), "dynamic units: CTA-pair TMA GEMMs");
  static_assert(!DYN || STAGES_ + 2 + 2 + 1 < 32, "unit ring deeper than any role's lag");
  static_assert(!WIDE || (PAIR && BL_ == KMAJ_TILE && EPI_ == EPI_SWIGLU && SWIGLU_B_ && !DYN_),
                "wide units: the CTA-pair gate/up GEMM");
  static_assert(!NARROW || (WIDE && AL_ == KMAJ_GATHER && SCH_ == RAGGED_M),
                "narrow units: the wide gate/up GEMM");
};

struct TileInfo {
  int g, mb, nb;
  bool phantom;    // pair slot past the group's last M-tile: loads only, no output
  int row0;        // RAGGED_M: first row of the M-tile in the A/D row space
  int rows_valid;  // RAGGED_M: rows of the group inside this tile (<= 128)
  int narrow;      // NARROW unit: its token columns (rows_valid rounded up to 32;
                   // row0, rows_valid: the pair's, the same in both CTAs); else 0
  int kstart;      // RAGGED_K: first K row of the group
  int kblocks;     // number of 64-deep k-blocks
};

// The unit's token columns when it is a NARROW unit of config C, else 0.
template <class C>
__device__ __forceinline__ int narrow_cols(const TileInfo& ti) {
  if constexpr (C::NARROW) return ti.narrow;
  else return 0;
}

// First row (within the tile) of this CTA's staged token rows: a NARROW unit's
// N side is split between the pair, rank r staging rows [r N/2, (r+1) N/2).
template <class C>
__device__ __forceinline__ int tile_row_base(const TileInfo& ti, int rank) {
  return rank * (narrow_cols<C>(ti) / 2);
}

struct SmemTables {
  int tile_prefix[kMaxGroups + 1];
  int start[kMaxGroups];   // group start in the (padded or not) row space
  int cnt[kMaxGroups];     // rows of the group
  int off[kMaxGroups];     // unpadded row offset of the group
  int total_tiles;
  int abort_flag;
  uint32_t tmem_base;
};

// Group tables (one warp; G <= 256): rows and offsets of every group, its
// start in the (padded or not) row space, and the prefix sums of its work units
// (units(cnt) for a group of cnt rows).  CTA 0 optionally publishes the starts.
template <class UnitsFn>
__device__ __forceinline__ void build_group_tables(const GemmArgs& a, SmemTables& T, int lane,
                                                   UnitsFn units) {
  // every lane's offsets first (G <= 256: up to 8 per lane), so their load
  // latencies overlap instead of adding up chunk by chunk
  constexpr int kChunks = kMaxGroups / 32;
  int pre_off[kChunks], pre_end[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int g = 32 * c + lane;
    pre_off[c] = pre_end[c] = 0;
    if (a.offsets && g < a.G) {
      pre_off[c] = __ldg(a.offsets + g);
      pre_end[c] = __ldg(a.offsets + g + 1);
    }
  }
  int run_tiles = 0, run_rows = 0;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int base = 32 * c;
    if (base >= a.G) break;
    const int g = base + lane;
    int cnt = 0, off = 0;
    if (g < a.G) {
      if (a.offsets) {
        off = pre_off[c];
        cnt = pre_end[c] - off;
        if (a.cap > 0) cnt = min(cnt, a.cap);
      } else if (a.ksplit > 0) {
        off = g * a.ksplit;
        cnt = min(a.ksplit, a.K - off);
      } else {
        cnt = a.single_rows;
      }
      if (cnt < 0) cnt = 0;
    }
    const int mt = (cnt + BM - 1) / BM;
    // lanes past the last group contribute nothing (no units, no rows)
    const int tiles = (g >= a.G) ? 0 : units(cnt);
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
  if (a.poff_out && blockIdx.x == 0) {
    __syncwarp();
    for (int g = lane; g < a.G; g += 32) a.poff_out[g] = T.start[g];
    if (lane == 0) a.poff_out[a.G] = run_rows;
  }
}

// n-blocks of a group's units (WIDE: pairs of BN-column blocks)
template <class C>
__device__ __forceinline__ int num_nblocks(const GemmArgs& a) {
  constexpr int W = C::SWIGLU_B ? C::NSUB * C::BN / 2 : C::NSUB * C::BN;
  return ((C::SWIGLU_B ? a.inter : a.N) + W - 1) / W;
}

// 256-row block of a unit (the group's earlier blocks + its m-block pair): the
// index of the dependency flag between a producer and a consumer GEMM over the
// same groups (both see the same blocks: units = blocks x n-blocks per group).
template <class C>
__device__ __forceinline__ int dep_pair(const GemmArgs& a, const SmemTables& T, int g, int mb) {
  return T.tile_prefix[g] / num_nblocks<C>(a) + (mb >> 1);
}

// ---------------------------------------------------------------- dynamic units
// The leader CTA's producer thread takes unit ids from a global counter and
// publishes them in order to a ring in both CTAs of the pair (own shared
// memory, and the peer's through the cluster); every role of both CTAs reads
// the same sequence from its own ring.  No role lags the producer's thread by
// more than its look-ahead (2 ids), the stage ring (at most STAGES units of one
// k-block), the two accumulators and the unit in hand, so kSchedRing slots are
// never overwritten while a role still has to read them.  An id >= total ends
// every role's loop.
constexpr int kSchedRing = 32;

struct UnitRing {
  int id[kSchedRing];
  uint64_t full[kSchedRing];
  uint64_t dep_ok[kSchedRing];  // this CTA's scheduler: the unit's dependency is met
  int prod_pos;                 // units the producer has started (the scheduler stays near it)
};

__device__ __forceinline__ void ring_publish(UnitRing& R, int pos, int t) {
  const int s = pos % kSchedRing;
  R.id[s] = t;
  mbar_arrive(smem_u32(&R.full[s]));
  st_shared_cluster_u32(mapa_shared(smem_u32(&R.id[s]), 1), (uint32_t)t);
  mbar_arrive_release_cluster(mapa_shared(smem_u32(&R.full[s]), 1));
}

// Next unit id of this role (pos counts its reads); total on abort.
__device__ __forceinline__ int ring_read(UnitRing& R, int& pos, int total, volatile int* abort_flag,
                                        int* status) {
  const int s = pos % kSchedRing;
  const uint32_t par = (uint32_t)(pos / kSchedRing) & 1u;
  ++pos;
  if (!mbar_wait_cluster(smem_u32(&R.full[s]), par, abort_flag, status)) return total;
  return *reinterpret_cast<volatile int*>(&R.id[s]);
}

// A role's walk over its units: static round-robin, or the ring.
template <bool DYN>
struct UnitWalk {
  UnitRing* ring;
  int pos, ustep, total;
  volatile int* abort_flag;
  int* status;
  __device__ __forceinline__ int first(int unit0) {
    if constexpr (DYN) return ring_read(*ring, pos, total, abort_flag, status);
    else return unit0;
  }
  __device__ __forceinline__ int next(int t) {
    if constexpr (DYN) return ring_read(*ring, pos, total, abort_flag, status);
    else return t + ustep;
  }
};

// Work unit t -> tile.  Without PAIR a unit is one tile (m-block fastest).  With
// PAIR a unit is a pair of adjacent m-blocks of one (group, n-block); CTA rank r
// of the cluster takes m-block 2p + r.
template <class C>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, const SmemTables& T, int t,
                                                int rank = 0) {
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
    const int mu = (mt + C::CL - 1) / C::CL;  // units along M
    ti.nb = local / mu;
    ti.mb = (local - ti.nb * mu) * C::CL + rank;
    ti.phantom = ti.mb >= mt;
    ti.row0 = T.start[lo] + ti.mb * BM;
    ti.rows_valid = ti.phantom ? 0 : min(BM, T.cnt[lo] - ti.mb * BM);
    ti.narrow = 0;
    if constexpr (C::NARROW) {
      const int mbe = ti.mb - rank;  // the pair's even m-block
      if (mbe + 1 == mt) {
        ti.mb = mbe;
        ti.phantom = false;
        ti.row0 = T.start[lo] + mbe * BM;
        ti.rows_valid = T.cnt[lo] - mbe * BM;
        ti.narrow = (ti.rows_valid + 31) & ~31;
      }
    }
    ti.kstart = 0;
    ti.kblocks = a.K / BK;
  } else {
    // groups own contiguous unit ranges
    const int nMB = (a.M + BM - 1) / BM;
    const int mu = (nMB + C::CL - 1) / C::CL;
    int lo = 0, hi = a.G - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (T.tile_prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    ti.g = lo;
    const int local = t - T.tile_prefix[lo];
    ti.nb = local / mu;
    ti.mb = (local - ti.nb * mu) * C::CL + rank;
    ti.phantom = ti.mb >= nMB;
    ti.row0 = ti.mb * BM;
    ti.rows_valid = ti.phantom ? 0 : min(BM, a.M - ti.mb * BM);
    ti.narrow = 0;
    ti.kstart = T.start[ti.g];
    ti.kblocks = (T.cnt[ti.g] + BK - 1) / BK;
  }
  return ti;
}

// ---------------------------------------------------------------- epilogues
// Output path: each epilogue warp owns 32 rows of the tile.  bf16 outputs leave
// in blocks of 32 rows x 64 columns (4 KB): the warp writes its rows of a block
// into a shared staging buffer with the 128-byte swizzle (conflict-free 16-byte
// writes) and one TMA bulk-tensor store sends it, so global writes are whole
// 128-byte lines and each store moves 4 KB.  (The fp32 split-K router partials
// use 32 x 16 fp32 blocks of 2 KB with the 64-byte swizzle.)  NB buffers per
// warp rotate, letting up to NB stores be in flight.  A warp whose 32 rows are
// not all inside the group (ragged expert edge) writes its valid rows directly.
template <int NB, int BYTES>
struct WarpOut {
  uint32_t buf0;  // this warp's first staging buffer (1024-byte aligned)
  int lane;
  int next;       // next buffer to use
  int inflight;   // committed stores not yet known to have read their buffer
  int hint[2];        // L2 hint code of the stores through output map 0 / 1
  uint64_t policy[2];
};

// Take the next K staging buffers (the first is returned, the others follow at
// BYTES strides; callers take K consecutive buffers with K dividing NB, so they
// never wrap).  Buffer next+i was last read by the store issued NB-i stores ago,
// so at most NB-K stores may still be pending.
template <int K, int NB, int BYTES>
__device__ __forceinline__ uint32_t stage_acquire(WarpOut<NB, BYTES>& w) {
  static_assert(K <= NB, "staging ring too small");
  if (w.inflight > NB - K) {
    if (w.lane == 0) bulk_wait_read<NB - K>();
    __syncwarp();
    w.inflight = NB - K;
  }
  const uint32_t buf = w.buf0 + w.next * BYTES;
  w.next = (w.next + 1) % NB;
  return buf;
}

// which: the output map (0 or 1) the store goes through (its L2 hint).
template <int NB, int BYTES>
__device__ __forceinline__ void stage_store(WarpOut<NB, BYTES>& w, uint32_t buf,
                                            const CUtensorMap* map, int x, int y, int z,
                                            bool three_d, int which = 0) {
  fence_proxy_async_smem();
  __syncwarp();
  if (w.lane == 0) {
    if (w.hint[which]) {
      if (three_d) tma_store_3d_hint(map, buf, x, y, z, w.policy[which]);
      else tma_store_2d_hint(map, buf, x, y, w.policy[which]);
    } else {
      if (three_d) tma_store_3d(map, buf, x, y, z);
      else tma_store_2d(map, buf, x, y);
    }
    bulk_commit();
  }
  __syncwarp();
  ++w.inflight;
}

// 16-byte piece p (bf16 columns 8p .. 8p+7 of a 64-column block) of this
// thread's row (row = lane), 128-byte swizzle.
__device__ __forceinline__ void put128(uint32_t buf, int lane, int p, uint32_t x0, uint32_t x1,
                                       uint32_t x2, uint32_t x3) {
  st_shared_v4(buf + lane * 128 + ((p ^ (lane & 7)) << 4), x0, x1, x2, x3);
}

__device__ __forceinline__ void st_global_16(__nv_bfloat16* dst, uint32_t x0, uint32_t x1,
                                             uint32_t x2, uint32_t x3) {
  *reinterpret_cast<uint4*>(dst) = make_uint4(x0, x1, x2, x3);
}

// 64-column blocks [g0, g1) of this warp's column part that lie inside N
// (every output width is a multiple of 64).
__device__ __forceinline__ void block_range(int cpart, int nparts, int nblk, int n0, int N, int& g0,
                                            int& g1) {
  g0 = cpart * nblk / nparts;
  g1 = (cpart + 1) * nblk / nparts;
  const int inside = N > n0 ? (N - n0) / 64 : 0;
  if (g1 > inside) g1 = inside;
}

// 2^x and 1/x on the special-function unit (PTX ex2.approx / rcp.approx).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sigmoid of two values with one reciprocal: with d = 1 + e^(-g) = 1 +
// 2^(-g log2 e), 1/d0 = d1 / (d0 d1) and 1/d1 = d0 / (d0 d1).  The forward
// epilogue is bound by the special-function unit (an exponential and a
// reciprocal per element); sharing the reciprocal takes 1.5 operations per
// element instead of 2.  Each exponent is capped at 2^62 so that the product
// stays finite: for g < -43 the sigmoid comes out as about 2^-62 instead of
// e^g (both below 1e-18).  Relative error a few fp32 ulps.
__device__ __forceinline__ float2 sigmoid2_f(float g0, float g1) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float d0 = 1.0f + ex2_approx(fminf(-g0 * kLog2e, 62.0f));
  const float d1 = 1.0f + ex2_approx(fminf(-g1 * kLog2e, 62.0f));
  const float r = rcp_approx(d0 * d1);
  return make_float2(d1 * r, d0 * r);
}

// fp32 output (split-K router partials).  RAGGED_K: D is the group's (split's)
// M x N slice, map tmD0 3-D [groups][M][N] with 16x32 fp32 boxes.
template <class C, class W>
__device__ void epilogue_store_f32(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                                   int row_in_tile, W& w, const CUtensorMap* tmD0, int cpart,
                                   int nparts) {
  const int quad = row_in_tile >> 5;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool warp_full = a.f32_tma && quad * 32 + 32 <= ti.rows_valid;
  const int n0 = ti.nb * C::BN;
  constexpr bool k3 = C::SCH == RAGGED_K;
  float* base = a.d_f32 + (k3 ? (long long)ti.g * a.d_group_stride : 0);
  const long long row = (k3 ? ti.mb * BM : ti.row0) + row_in_tile;
  const int y = (k3 ? ti.mb * BM : ti.row0) + quad * 32;
  float v[32];
  constexpr int NCH = (C::BN + 31) / 32;
#pragma unroll 1
  for (int c = cpart * NCH / nparts; c < (cpart + 1) * NCH / nparts; ++c) {
    const int col = n0 + c * 32;
    if (col >= a.N) break;
    if (ti.kblocks > 0) tmem_ld32(tacc + c * 32, v);
    else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
    }
    if (warp_full) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (half == 1 && col + 16 >= a.N) break;
        const uint32_t buf = stage_acquire<1>(w);
        const uint32_t rowp = buf + w.lane * 64;
        const int sw = (w.lane >> 1) & 3;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = 16 * half + 4 * q;
          st_shared_v4(rowp + ((q ^ sw) << 4), __float_as_uint(v[e]), __float_as_uint(v[e + 1]),
                       __float_as_uint(v[e + 2]), __float_as_uint(v[e + 3]));
        }
        stage_store(w, buf, tmD0, col + 16 * half, y, ti.g, k3);
      }
    } else if (valid) {
      float* dst = base + row * a.ldd + col;
      for (int i = 0; i < 32 && col + i < a.N; ++i) dst[i] = v[i];
    }
  }
}

// Gate/up epilogue: acc columns [0, BN/2) are gate, [BN/2, BN) up, for the
// intermediate columns n0 .. n0+BN/2-1.  Writes g, u (bf16, for the backward;
// skipped when gu_out is null) and h = silu(g) * u (skipped when h_out is
// null).  Maps: tmD0 = gu_out [rows, 2I], tmD1 = h_out [rows, I].
template <class C, class W>
__device__ void epilogue_swiglu(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                                int row_in_tile, W& w, const CUtensorMap* tmD0,
                                const CUtensorMap* tmD1, int cpart, int nparts) {
  const int quad = row_in_tile >> 5;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool warp_full = quad * 32 + 32 <= ti.rows_valid;
  const long long r = ti.row0 + row_in_tile;
  const int y = ti.row0 + quad * 32;
  const int I = a.inter;
  constexpr int HALF = C::BN / 2;
  const int n0 = ti.nb * HALF;
  // (g, u stores need three staging buffers per warp; configs with fewer
  // serve the inference forward, which keeps h only)
  const bool keep_gu = C::EPI_BUFS >= 3 && a.gu_out != nullptr;
  const bool keep_h = a.h_out != nullptr;  // a backward recomputing g, u needs no h
  int g0, g1;
  block_range(cpart, nparts, HALF / 64, n0, I, g0, g1);
#pragma unroll 1
  for (int gi = g0; gi < g1; ++gi) {
    const int j = n0 + gi * 64;
    uint32_t bg = 0, bu = 0, bh = 0;
    if (warp_full) {
      if constexpr (C::EPI_BUFS >= 3) {
        if (keep_gu) {
          bg = stage_acquire<3>(w);
          bu = stage_acquire<1>(w);  // inside the three just made free
        }
      }
      if (keep_h) bh = stage_acquire<1>(w);
    }
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint32_t g[32], u[32];
      tmem_ld32_issue(tacc + gi * 64 + h * 32, g);
      tmem_ld32_issue(tacc + HALF + gi * 64 + h * 32, u);
      tmem_ld_wait2(g, u);
      // each output is formed only when it is kept (the conversions and the
      // special-function work are a large share of this epilogue)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pc = 4 * h + q;  // piece within the 64-column block
        const int col = j + 8 * pc;
        if (keep_gu) {
          uint32_t pg[4], pu[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = 8 * q + 2 * i;
            pg[i] = pack_bf16x2(__uint_as_float(g[e]), __uint_as_float(g[e + 1]));
            pu[i] = pack_bf16x2(__uint_as_float(u[e]), __uint_as_float(u[e + 1]));
          }
          if (warp_full) {
            put128(bg, w.lane, pc, pg[0], pg[1], pg[2], pg[3]);
            put128(bu, w.lane, pc, pu[0], pu[1], pu[2], pu[3]);
          } else if (valid) {
            st_global_16(a.gu_out + r * (2LL * I) + col, pg[0], pg[1], pg[2], pg[3]);
            st_global_16(a.gu_out + r * (2LL * I) + I + col, pu[0], pu[1], pu[2], pu[3]);
          }
        }
        if (keep_h) {
          uint32_t ph[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = 8 * q + 2 * i;
            const float ga = __uint_as_float(g[e]), gb = __uint_as_float(g[e + 1]);
            const float2 sg = sigmoid2_f(ga, gb);
            ph[i] = pack_bf16x2(ga * sg.x * __uint_as_float(u[e]),
                                gb * sg.y * __uint_as_float(u[e + 1]));
          }
          if (warp_full) put128(bh, w.lane, pc, ph[0], ph[1], ph[2], ph[3]);
          else if (valid) st_global_16(a.h_out + r * (long long)I + col, ph[0], ph[1], ph[2], ph[3]);
        }
      }
    }
    if (warp_full) {
      if (keep_gu) {
        stage_store(w, bg, tmD0, j, y, 0, false);
        stage_store(w, bu, tmD0, I + j, y, 0, false);
      }
      if (keep_h) stage_store(w, bh, tmD1, j, y, 0, false, 1);
    }
  }
}

// Gate/up epilogue of the wide inference GEMM with 8 epilogue warps: h only,
// in 32-column blocks staged as 32 rows x 64 bytes (64-byte swizzle, 2 KB)
// and stored through tmD1 = h_out [rows, I] with 32 x 32 boxes.  The two warps
// of a lane quadrant take half of the tile's h columns each.
template <class C, class W>
__device__ void epilogue_swiglu_h32(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                                    int row_in_tile, W& w, const CUtensorMap* tmD1, int cpart,
                                    int nparts) {
  const int quad = row_in_tile >> 5;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool warp_full = quad * 32 + 32 <= ti.rows_valid;
  const long long r = ti.row0 + row_in_tile;
  const int y = ti.row0 + quad * 32;
  const int I = a.inter;
  constexpr int HALF = C::BN / 2;
  constexpr int NBLK = HALF / 32;
  const int n0 = ti.nb * HALF;
  const int b0 = cpart * NBLK / nparts;
  int b1 = (cpart + 1) * NBLK / nparts;
  const int inside = I > n0 ? (I - n0) / 32 : 0;  // I is a multiple of 64
  if (b1 > inside) b1 = inside;
  const int sw = (w.lane >> 1) & 3;
#pragma unroll 1
  for (int bi = b0; bi < b1; ++bi) {
    const int j = n0 + bi * 32;
    uint32_t g[32], u[32];
    tmem_ld32_issue(tacc + bi * 32, g);
    tmem_ld32_issue(tacc + HALF + bi * 32, u);
    tmem_ld_wait2(g, u);
    uint32_t ph[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float ga = __uint_as_float(g[2 * i]), gb = __uint_as_float(g[2 * i + 1]);
      const float2 sg = sigmoid2_f(ga, gb);
      ph[i] = pack_bf16x2(ga * sg.x * __uint_as_float(u[2 * i]),
                          gb * sg.y * __uint_as_float(u[2 * i + 1]));
    }
    if (warp_full) {
      // the buffer is taken after the math, so the wait for the previous
      // store's read of it overlaps the work above
      const uint32_t rowp = stage_acquire<1>(w) + w.lane * 64;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(rowp + ((q ^ sw) << 4), ph[4 * q], ph[4 * q + 1], ph[4 * q + 2], ph[4 * q + 3]);
      stage_store(w, rowp - w.lane * 64, tmD1, j, y, 0, false, 1);
    } else if (valid) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_global_16(a.h_out + r * (long long)I + j + 8 * q, ph[4 * q], ph[4 * q + 1], ph[4 * q + 2],
                     ph[4 * q + 3]);
    }
  }
}

// Plain bf16 output in 32-column blocks staged as 32 rows x 64 bytes (64-byte
// swizzle, 2 KB), for kernels whose shared memory leaves room for no more:
// tmD0 has 32 x 32 boxes (RAGGED_K: 3-D, group = depth).  Rows and columns as
// in epilogue_store.
template <class C, class W>
__device__ void epilogue_store32(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                                 int row_in_tile, W& w, const CUtensorMap* tmD0, int cpart,
                                 int nparts) {
  const int quad = row_in_tile >> 5;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool warp_full = quad * 32 + 32 <= ti.rows_valid;
  const int n0 = ti.nb * C::BN;
  constexpr bool k3 = C::SCH == RAGGED_K;
  const long long row = (k3 ? ti.mb * BM : ti.row0) + row_in_tile;
  const int y = (k3 ? ti.mb * BM : ti.row0) + quad * 32;
  const bool live = ti.kblocks > 0;  // an expert with no rows has an exact zero gradient
  __nv_bfloat16* drow = a.d + (k3 ? (long long)ti.g * a.d_group_stride : 0) + row * a.ldd;
  constexpr int NBLK = C::BN / 32;
  const int b0 = cpart * NBLK / nparts;
  int b1 = (cpart + 1) * NBLK / nparts;
  const int inside = a.N > n0 ? (a.N - n0) / 32 : 0;  // N is a multiple of 64
  if (b1 > inside) b1 = inside;
  const int sw = (w.lane >> 1) & 3;
#pragma unroll 1
  for (int bi = b0; bi < b1; ++bi) {
    const int col = n0 + bi * 32;
    uint32_t v[32];
    if (live) {
      tmem_ld32_issue(tacc + bi * 32, v);
      tmem_ld_wait(v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;
    }
    uint32_t x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    if (warp_full) {
      const uint32_t buf = stage_acquire<1>(w);
      const uint32_t rowp = buf + w.lane * 64;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(rowp + ((q ^ sw) << 4), x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
      stage_store(w, buf, tmD0, col, y, ti.g, k3);
    } else if (valid) {
#pragma unroll
      for (int q = 0; q < 4; ++q) st_global_16(drow + col + 8 * q, x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
  }
}

// Plain bf16 output.  RAGGED_M: D rows are the tile's rows (map tmD0 2-D);
// RAGGED_K: D is the group's full M x N matrix (map tmD0 3-D, group = depth).
template <class C, class W>
__device__ void epilogue_store(const GemmArgs& a, const TileInfo& ti, uint32_t tacc,
                               int row_in_tile, W& w, const CUtensorMap* tmD0, int cpart,
                               int nparts) {
  const int quad = row_in_tile >> 5;
  const bool valid = row_in_tile < ti.rows_valid;
  const bool warp_full = quad * 32 + 32 <= ti.rows_valid;
  const int n0 = ti.nb * C::BN;
  constexpr bool k3 = C::SCH == RAGGED_K;
  const long long row = (k3 ? ti.mb * BM : ti.row0) + row_in_tile;
  const int y = (k3 ? ti.mb * BM : ti.row0) + quad * 32;
  const bool live = ti.kblocks > 0;  // an expert with no rows has an exact zero gradient
  __nv_bfloat16* drow = a.d + (k3 ? (long long)ti.g * a.d_group_stride : 0) + row * a.ldd;
  int g0, g1;
  block_range(cpart, nparts, C::BN / 64, n0, a.N, g0, g1);
#pragma unroll 1
  for (int gi = g0; gi < g1; ++gi) {
    const int col = n0 + gi * 64;
    const uint32_t buf = warp_full ? stage_acquire<1>(w) : 0u;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint32_t v[32];
      if (live) {
        tmem_ld32_issue(tacc + gi * 64 + h * 32, v);
        tmem_ld_wait(v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          x[i] = pack_bf16x2(__uint_as_float(v[8 * q + 2 * i]), __uint_as_float(v[8 * q + 2 * i + 1]));
        const int pc = 4 * h + q;
        if (warp_full) put128(buf, w.lane, pc, x[0], x[1], x[2], x[3]);
        else if (valid) st_global_16(drow + col + 8 * pc, x[0], x[1], x[2], x[3]);
      }
    }
    if (warp_full) stage_store(w, buf, tmD0, col, y, ti.g, k3);
  }
}

// NARROW units: TMEM lane = output column (weight row) of this CTA's 128, TMEM
// column = token t of the pair's rows_valid rows (row0 + t).  Each thread
// stores its column of every token directly: a warp writes 32 consecutive
// bf16 (64 bytes) per token.  The two column parts of a lane quadrant take
// alternate 32-token chunks.
__device__ __forceinline__ void st_bf16_col(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Wide gate/up GEMM: gate in columns [0, narrow), up in [narrow, 2 narrow) of
// accumulator 0; h[row0 + t, j] for j = j0 + lane row (j0 = 128 x the unit's
// first n-block + 128 rank).  Out of line, every argument by value: the
// callers' loop state stays in registers.
__device__ __noinline__ void epilogue_narrow_swiglu(__nv_bfloat16* h_out, int I, int j0,
                                                    long long row0, int rows_valid, int narrow,
                                                    uint32_t tacc, int row_in_tile, int cpart,
                                                    int nparts) {
  const int j = j0 + row_in_tile;
  const bool col_ok = j < I && h_out != nullptr;
  __nv_bfloat16* hcol = h_out + row0 * I + j;
  // the sigmoids of columns 2m and 2m+1 share one reciprocal, as in the
  // other gate/up epilogues (so h is the same bits whichever unit forms it):
  // the pair's two columns are the lanes l and l^1
  const bool odd = (row_in_tile & 1) != 0;
#pragma unroll 1
  for (int c0 = 32 * cpart; c0 < rows_valid; c0 += 32 * nparts) {
    uint32_t g[32], u[32];
    tmem_ld32_issue(tacc + c0, g);
    tmem_ld32_issue(tacc + narrow + c0, u);
    tmem_ld_wait2(g, u);
    const int nt = min(32, rows_valid - c0);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float gv = __uint_as_float(g[i]);
      const float go = __shfl_xor_sync(0xffffffffu, gv, 1);
      const float2 sg = odd ? sigmoid2_f(go, gv) : sigmoid2_f(gv, go);
      if (col_ok && i < nt)
        st_bf16_col(hcol + (long long)(c0 + i) * I, gv * (odd ? sg.y : sg.x) * __uint_as_float(u[i]));
    }
  }
}

// Down-projection data gradient with the SwiGLU backward fused in.
// acc = dh_unw = dout[token] * W_down[e]  (columns n0.. of the intermediate)
// From the saved pre-activations (g, u): h = silu(g) u; dw partial = <acc, h>;
// dh = w acc; dg = dh u s (1 + g (1 - s)); du = dh silu(g); hw = w h.
// Maps: tmD0 = dgu_out [rows, 2I], tmD1 = hw_out [rows, I].  In the padded
// layout the rows past the expert's tokens are written as exact zeros.  The
// saved (g, u) of the next 32 columns are loaded while this half is computed.
template <class C, class W>
__device__ void epilogue_dgrad_swiglu(const GemmArgs& a, const SmemTables& T, const TileInfo& ti,
                                      uint32_t tacc, int row_in_tile, W& w,
                                      const CUtensorMap* tmD0, const CUtensorMap* tmD1, int cpart,
                                      int nparts) {
  const int quad = row_in_tile >> 5;
  const long long p = ti.row0 + row_in_tile;  // row in the (padded) row space
  const int y = ti.row0 + quad * 32;
  const int I = a.inter;
  const int n0 = ti.nb * C::BN;
  const int nNB = (I + C::BN - 1) / C::BN;
  const int npart_cols = nNB * nparts;  // dw partials per row
  const bool valid = row_in_tile < ti.rows_valid;
  const bool pad_row = !valid && a.padded;
  const bool warp_full = a.padded || quad * 32 + 32 <= ti.rows_valid;
  long long r = p;  // row of the saved (unpadded) forward tensors
  float wt = 1.f;
  if (valid) {
    if (a.padded) r = T.off[ti.g] + ti.mb * BM + row_in_tile;
    if (a.slot_w) wt = __ldg(a.slot_w + __ldg(a.perm_slot + r));
  }
  const __nv_bfloat16* gsrc = a.gu_saved + r * (2LL * I);
  int g0, g1;
  block_range(cpart, nparts, C::BN / 64, n0, I, g0, g1);
  float dwp = 0.f;
  uint4 gs[4], us[4];  // saved g, u of the current 32 columns (valid rows)
  auto load_gu = [&](int col, uint4 (&gd)[4], uint4 (&ud)[4]) {
    const uint4* pg = reinterpret_cast<const uint4*>(gsrc + col);
    const uint4* pu = reinterpret_cast<const uint4*>(gsrc + I + col);
#pragma unroll
    for (int q = 0; q < 4; ++q) { gd[q] = __ldg(pg + q); ud[q] = __ldg(pu + q); }
  };
  if (valid && g0 < g1) load_gu(n0 + g0 * 64, gs, us);
#pragma unroll 1
  for (int gi = g0; gi < g1; ++gi) {
    const int j = n0 + gi * 64;
    uint32_t bdg = 0, bdu = 0, bhw = 0;
    if (warp_full) {
      bdg = stage_acquire<3>(w);
      bdu = stage_acquire<1>(w);  // inside the three just made free
      bhw = stage_acquire<1>(w);
    }
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint32_t acc[32];
      tmem_ld32_issue(tacc + gi * 64 + h * 32, acc);
      uint4 gn[4], un[4];
      const int nxt = j + 32 * (h + 1);  // next 32 columns of this warp, if any
      const bool more = valid && (h == 0 || gi + 1 < g1);
      if (more) load_gu(nxt, gn, un);
      tmem_ld_wait(acc);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pdg[4] = {0u, 0u, 0u, 0u}, pdu[4] = {0u, 0u, 0u, 0u}, phw[4] = {0u, 0u, 0u, 0u};
        if (valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t gw = (&gs[q].x)[i], uw = (&us[q].x)[i];
            float dg2[2], du2[2], hw2[2];
            const float2 s2 = sigmoid2_f(bf16lo(gw), bf16hi(gw));
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const float gg = t ? bf16hi(gw) : bf16lo(gw);
              const float uu = t ? bf16hi(uw) : bf16lo(uw);
              const float ac = __uint_as_float(acc[8 * q + 2 * i + t]);
              const float s = t ? s2.y : s2.x;
              const float sl = gg * s;
              const float hh = sl * uu;
              dwp = fmaf(ac, hh, dwp);
              const float dh = wt * ac;
              dg2[t] = dh * uu * s * (1.0f + gg * (1.0f - s));
              du2[t] = dh * sl;
              hw2[t] = wt * hh;
            }
            pdg[i] = pack_bf16x2(dg2[0], dg2[1]);
            pdu[i] = pack_bf16x2(du2[0], du2[1]);
            phw[i] = pack_bf16x2(hw2[0], hw2[1]);
          }
        }
        const int pc = 4 * h + q;
        if (warp_full) {
          put128(bdg, w.lane, pc, pdg[0], pdg[1], pdg[2], pdg[3]);
          put128(bdu, w.lane, pc, pdu[0], pdu[1], pdu[2], pdu[3]);
          put128(bhw, w.lane, pc, phw[0], phw[1], phw[2], phw[3]);
        } else if (valid || pad_row) {
          const int col = j + 8 * pc;
          st_global_16(a.dgu_out + p * (2LL * I) + col, pdg[0], pdg[1], pdg[2], pdg[3]);
          st_global_16(a.dgu_out + p * (2LL * I) + I + col, pdu[0], pdu[1], pdu[2], pdu[3]);
          st_global_16(a.hw_out + p * (long long)I + col, phw[0], phw[1], phw[2], phw[3]);
        }
      }
      if (more) {
#pragma unroll
        for (int q = 0; q < 4; ++q) { gs[q] = gn[q]; us[q] = un[q]; }
      }
    }
    if (warp_full) {
      stage_store(w, bdg, tmD0, j, y, 0, false);
      stage_store(w, bdu, tmD0, I + j, y, 0, false);
      stage_store(w, bhw, tmD1, j, y, 0, false, 1);
    }
  }
  if (a.dw_part && (valid || pad_row)) a.dw_part[p * npart_cols + ti.nb * nparts + cpart] = dwp;
}

// ---------------------------------------------------------------- gather warps
// Source token row for row i of group g (rows past the group's tokens reuse its
// last token: finite values, for the K-side gathers whose padding rows multiply
// zeros; the M-side gathers skip those rows).
__device__ __forceinline__ int gather_row(const GemmArgs& a, const SmemTables& T, int g, int i) {
  const int n = T.cnt[g];
  const int r = T.off[g] + (i < n ? i : n - 1);
  return clampi(__ldg(a.gperm + r) / a.gdiv, 0, a.gsrc_rows - 1);
}

// First tile at or after t0 (stride gridDim.x) that has k-blocks; total if none.
template <class C>
__device__ __forceinline__ int next_work_tile(const GemmArgs& a, const SmemTables& T, int t0,
                                              int total, int rank, int ustep, TileInfo& out) {
  for (int t = t0; t < total; t += ustep) {
    out = decode_tile<C>(a, T, t, rank);
    if (out.kblocks > 0) return t;
  }
  return total;
}

// This warp's copies into a gathered stage are complete (each thread has
// waited for its own and fenced them to the async proxy): one arrival per warp
// on the stage's full barrier; with PAIR the even CTA's, whose thread issues
// the UMMAs.  The copies sit in this SM's shared memory, which the pair UMMA
// reads on this SM, so the arrival needs no cluster-scope release (one would
// also wait for the copies of later stages still in flight).
template <class C>
__device__ __forceinline__ void arrive_full(uint64_t* full_bar, uint32_t stage, int lane, int rank) {
  __syncwarp();
  if (lane == 0) {
    if (C::PAIR && rank != 0) mbar_arrive_remote(mapa_shared(smem_u32(&full_bar[stage]), 0));
    else mbar_arrive(smem_u32(&full_bar[stage]));
  }
}

// The gather warps walk the same (tile, k-block) sequence as the TMA producer.
// Token ids are software-pipelined: the ids of the next stage (or of the next
// tile) are loaded before the current stage's copies are issued, so their
// latency overlaps the copies in flight.
template <class C>
__device__ void gather_role(const GemmArgs& a, const SmemTables& T, uint32_t smem_base,
                           uint64_t* full_bar, uint64_t* empty_bar, volatile int* abort_flag,
                           int gw, int lane, int total, int rank, int unit0, int ustep) {
  constexpr int LAG = C::GATHER_LAG;
  constexpr bool KM = (C::AL == KMAJ_GATHER);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t ring = 0;  // stages with copies issued but not yet signalled (4 bits each, FIFO)
  int rn = 0;
  TileInfo ti, tn;
  int t = next_work_tile<C>(a, T, unit0, total, rank, ustep, ti);
  int src[8], src_n[8];  // K-major: this lane's rows gw*32 + 4*i + (lane >> 3)
  int kid = 0;           // MN-major: k-row gw*16 + (lane & 15) of the current stage
  if (t < total) {
    if constexpr (KM) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        src[i] = gather_row(a, T, ti.g,
                            ti.mb * BM + tile_row_base<C>(ti, rank) + gw * 32 + 4 * i + (lane >> 3));
    } else {
      kid = gather_row(a, T, ti.g, gw * 16 + (lane & 15));
    }
  }
  int kb = 0;
  int t_next = total;
  while (t < total && !*abort_flag) {
    if (kb == 0) {
      t_next = next_work_tile<C>(a, T, t + ustep, total, rank, ustep, tn);
      if constexpr (KM) {
        if (t_next < total) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            src_n[i] = gather_row(a, T, tn.g, tn.mb * BM + tile_row_base<C>(tn, rank) + gw * 32 +
                                                  4 * i + (lane >> 3));
        }
      }
    }
    int kid_n = 0;
    if constexpr (!KM) {
      if (kb + 1 < ti.kblocks) kid_n = gather_row(a, T, ti.g, (kb + 1) * BK + gw * 16 + (lane & 15));
      else if (t_next < total) kid_n = gather_row(a, T, tn.g, gw * 16 + (lane & 15));
    }
    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, a.status)) break;
    const uint32_t sA = smem_base + stage * C::STAGE_BYTES;
    const uint32_t sB = sA + C::A_BYTES;
    if (ti.phantom) {
      // pair slot past the group's last tile: the stage is not read into any output
    } else if constexpr (KM) {
      // rows of the M-tile past the group's rows are not copied: each feeds
      // only its own output row, which is never stored (K-side gathers below
      // keep their finite padding rows, which multiply zeros).  A NARROW unit
      // stages this CTA's half of its token columns, whose other rows are
      // likewise never stored.
      const int c = lane & 7;
      const __nv_bfloat16* col = a.gsrc + kb * BK + c * 8;
      const int rb = tile_row_base<C>(ti, rank);
      const int nvalid = narrow_cols<C>(ti) ? min(narrow_cols<C>(ti) / 2, ti.rows_valid - rb)
                                            : T.cnt[ti.g] - ti.mb * BM;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = gw * 32 + 4 * i + (lane >> 3);
        if (r < nvalid) cp_async_16(sA + r * 128 + ((c ^ (r & 7)) << 4), col + (size_t)src[i] * a.gld);
      }
    } else {
      // MN-major: operand extent X along M/N, X/8 16-byte chunks per k-row
      constexpr int X = C::A_GATHER ? BM : C::BN;
      constexpr int CPR = X / 8;
      constexpr int RPI = 32 / CPR;  // k-rows per warp instruction
      const uint32_t sOp = C::A_GATHER ? sA : sB;
      const int mn0 = C::A_GATHER ? ti.mb * BM : (C::SWIGLU_B ? ti.nb * (C::BN / 2) : ti.nb * C::BN);
      const int cc = lane % CPR;
      const int j = cc >> 3, c = cc & 7;
      const __nv_bfloat16* col = a.gsrc + mn0 + j * 64 + c * 8;
      // extents are multiples of 64: a 64-wide group past the row is not copied
      // (its rows or columns are not stored)
      const bool inside = mn0 + j * 64 < (C::A_GATHER ? a.M : a.N);
#pragma unroll
      for (int q = 0; q < 16 / RPI; ++q) {
        const int rl = q * RPI + lane / CPR;  // 0..15 within this warp's k-rows
        const int r = gw * 16 + rl;
        const int srow = __shfl_sync(0xffffffffu, kid, rl);
        if (inside)
          cp_async_16(sOp + j * 8192 + r * 128 + ((c ^ (r & 7)) << 4), col + (size_t)srow * a.gld);
      }
    }
    cp_async_commit();
    ring |= (uint32_t)stage << (4 * rn);
    ++rn;
    if (rn > LAG) {
      cp_async_wait<LAG>();
      fence_proxy_async_smem();
      arrive_full<C>(full_bar, ring & 15u, lane, rank);
      ring >>= 4;
      --rn;
    }
    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
    // advance to the next (tile, k-block)
    if (++kb == ti.kblocks) {
      kb = 0;
      t = t_next;
      ti = tn;
      if constexpr (KM) {
#pragma unroll
        for (int i = 0; i < 8; ++i) src[i] = src_n[i];
      }
    }
    if constexpr (!KM) kid = kid_n;
  }
  // signal the stages still in flight
  cp_async_wait<0>();
  fence_proxy_async_smem();
  while (rn > 0) {
    arrive_full<C>(full_bar, ring & 15u, lane, rank);
    ring >>= 4;
    --rn;
  }
}

// ---------------------------------------------------------------- wide units
// The UMMA issuer's work for one WIDE unit (CTA-pair leader, warp-uniform
// control; lane 0 issues).  Stage s, k-block kb: the four K=16 steps into
// accumulator `which` (0 or 1), whose B tile is the stage's tile `which`.
template <class C>
__device__ __forceinline__ void wide_issue(uint32_t smem_base, uint32_t tmem_base, int s, int kb,
                                           int which) {
  const uint32_t sA = smem_base + s * C::STAGE_BYTES;
  const uint32_t sB = sA + C::A_BYTES + which * (C::B_ROWS * 128);
#pragma unroll
  for (int kk = 0; kk < BK / 16; ++kk)
    umma_bf16_pair(tmem_base + which * C::BN, smem_desc_sw128(sA + kk * 32, 16, 1024),
                   smem_desc_sw128(sB + kk * 32, 16, 1024), C::IDESC, (kb | kk) != 0 ? 1u : 0u);
}

// Returns false on abort.  stage/phase: the stage ring position (advanced);
// acc_phase: the accumulators' phase (flipped once the unit is issued).
template <class C>
__device__ bool wide_unit(const TileInfo& ti, uint32_t smem_base, uint32_t tmem_base,
                          uint64_t* full_bar, uint64_t* empty_bar, uint64_t* tfull_bar,
                          uint64_t* tempty_bar, int& stage,
                          uint32_t& phase, uint32_t& acc_phase, int lane, volatile int* abort_flag,
                          int* status) {
  static_assert(C::WIDE && C::PAIR, "wide units run on CTA pairs");
  // Stages that may be held while waiting for the next one to fill.  A stage
  // fills only once the producers could claim the stages after it: the gather
  // warps complete stage s after issuing the copies of the next GATHER_LAG
  // stages, so those (STAGES later in the ring than stages before the held
  // ones) must not be held.  Beyond this, wait for accumulator 1.
  constexpr int kMaxHeld = C::STAGES - 1 - (C::A_GATHER ? C::GATHER_LAG : 0);
  static_assert(kMaxHeld >= 0, "stage ring too shallow");
  if (!mbar_wait(smem_u32(&tempty_bar[0]), acc_phase ^ 1, abort_flag, status)) return false;
  tc_fence_after();
  bool acc1 = false;           // accumulator 1 is free
  int held = 0, h_stage = 0, h_kb = 0;  // stages with only their first half issued
  auto flush = [&]() {         // second halves of the held stages, then release them
    if (lane == 0) {
      for (int i = 0; i < held; ++i) {
        const int s = (h_stage + i) % C::STAGES;
        wide_issue<C>(smem_base, tmem_base, s, h_kb + i, 1);
        umma_commit_pair(smem_u32(&empty_bar[s]));
      }
    }
    __syncwarp();
    held = 0;
  };
  for (int kb = 0; kb < ti.kblocks; ++kb) {
    if (!mbar_wait(smem_u32(&full_bar[stage]), phase, abort_flag, status)) return false;
    tc_fence_after();
    if (lane == 0) wide_issue<C>(smem_base, tmem_base, stage, kb, 0);
    __syncwarp();
    if (!acc1) {
      const bool free1 = __shfl_sync(0xffffffffu,
                                     lane == 0 ? (int)mbar_test_wait(smem_u32(&tempty_bar[1]),
                                                                     acc_phase ^ 1)
                                               : 0,
                                     0) != 0;
      if (free1 || held + 1 > kMaxHeld) {
        if (!free1 && !mbar_wait(smem_u32(&tempty_bar[1]), acc_phase ^ 1, abort_flag, status))
          return false;
        tc_fence_after();
        acc1 = true;
        flush();
      } else {
        if (held == 0) { h_stage = stage; h_kb = kb; }
        ++held;
      }
    }
    if (acc1) {
      if (lane == 0) {
        wide_issue<C>(smem_base, tmem_base, stage, kb, 1);
        umma_commit_pair(smem_u32(&empty_bar[stage]));
      }
      __syncwarp();
    }
    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
  }
  if (!acc1) {
    if (!mbar_wait(smem_u32(&tempty_bar[1]), acc_phase ^ 1, abort_flag, status)) return false;
    tc_fence_after();
    flush();
  }
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      if (ti.kblocks > 0) {
        umma_commit_pair(smem_u32(&tfull_bar[b]));
      } else {
        mbar_arrive(smem_u32(&tfull_bar[b]));
        mbar_arrive_remote(mapa_shared(smem_u32(&tfull_bar[b]), 1));
      }
    }
  }
  __syncwarp();
  acc_phase ^= 1;
  return true;
}

// The UMMA issuer's work for one NARROW wide unit: every stage's gate tile
// (B tile 0) and up tile (B tile 1) are the 256-row sides of two pair UMMAs
// with the stage's token rows as their N side, into columns [0, N) and [N, 2N)
// of accumulator 0.  Accumulator 1 is left unwritten: it is handed to the
// epilogue (which stores nothing for it) once free, keeping both barriers'
// phases in step with the other units.  Out of line, every argument by value
// (the issuer's ring position stays in registers): returns the advanced
// position as stage | phase << 16, or -1 on abort.
template <class C>
__device__ __noinline__ int narrow_wide_unit(int kblocks, int nt, uint32_t smem_base,
                                             uint32_t tmem_base, uint32_t full0, uint32_t empty0,
                                             uint32_t tfull0, uint32_t tempty0, int stage,
                                             uint32_t phase, uint32_t acc_phase, int lane,
                                             volatile int* abort_flag, int* status) {
  const uint32_t idesc = idesc_bf16_f32(2 * BM, nt, false, false);
  if (!mbar_wait(tempty0, acc_phase ^ 1, abort_flag, status)) return -1;
  tc_fence_after();
  for (int kb = 0; kb < kblocks; ++kb) {
    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, status)) return -1;
    tc_fence_after();
    if (lane == 0) {
      const uint32_t sA = smem_base + stage * C::STAGE_BYTES;
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint32_t sW = sA + C::A_BYTES + w * (C::B_ROWS * 128);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_bf16_pair(tmem_base + w * nt, smem_desc_sw128(sW + kk * 32, 16, 1024),
                         smem_desc_sw128(sA + kk * 32, 16, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      umma_commit_pair(empty0 + 8 * stage);
    }
    __syncwarp();
    if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
  }
  if (lane == 0) umma_commit_pair(tfull0);
  __syncwarp();
  if (!mbar_wait(tempty0 + 8, acc_phase ^ 1, abort_flag, status)) return -1;
  if (lane == 0) {
    mbar_arrive(tfull0 + 8);
    mbar_arrive_remote(mapa_shared(tfull0 + 8, 1));
  }
  __syncwarp();
  return stage | (int)(phase << 16);
}

// ---------------------------------------------------------------- the kernel
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
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
  __shared__ UnitRing ring;  // DYN only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  volatile int* abort_flag = &T.abort_flag;

  // ---- set-up: barriers, TMEM, group tables
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), C::FULL_ARRIVALS);
      // with PAIR the even CTA's UMMA commit releases the stage in both CTAs
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), C::TEMPTY_ARRIVALS);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    if constexpr (C::DYN) {
      for (int s = 0; s < kSchedRing; ++s) {
        mbar_init(smem_u32(&ring.full[s]), 1);
        mbar_init(smem_u32(&ring.dep_ok[s]), 1);
      }
      ring.prod_pos = 0;
    }
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
  if (warp == 2) {
    const int nNB = num_nblocks<C>(a);
    const int nMB = (a.M + BM - 1) / BM;
    build_group_tables(a, T, lane, [&](int cnt) {
      // work units of this group (tiles, or m-block pairs with CTA pairs)
      const int mt = (cnt + BM - 1) / BM;
      const int mu = ((C::SCH == RAGGED_M ? mt : nMB) + C::CL - 1) / C::CL;
      return mu * nNB;
    });
  }
  __syncthreads();
  // no work (every CTA of a cluster sees the same tables): leave before
  // touching tensor memory or the peer
  if (T.total_tiles == 0) return;
  if (warp == 1) {
    if constexpr (C::PAIR) {
      tmem_alloc_pair(smem_u32(&T.tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&T.tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (C::CL == 2) cluster_sync();  // the peer's barriers are initialised before any remote op
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = T.tmem_base;
  const int total = T.total_tiles;
  const int rank = C::CL == 2 ? (int)cluster_ctarank() : 0;
  const bool leader = rank == 0;  // PAIR: the CTA whose thread issues the pair's UMMAs
  const int unit0 = blockIdx.x / C::CL;
  const int ustep = gridDim.x / C::CL;
  // producer side of a cross-kernel overlap: every CTA is running, so the
  // consumer grid may start on the SMs this grid frees
  if (a.dep_signal && threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ================= TMA producer =================
    int stage = 0;
    uint32_t phase = 0;
    uint32_t filled = 0, fill_parity = 0;  // per stage: armed at least once, parity of last fill
    UnitWalk<C::DYN> uw{&ring, 0, ustep, total, abort_flag, a.status};
    for (int t = uw.first(unit0); t < total && !*abort_flag; t = uw.next(t)) {
      const TileInfo ti = decode_tile<C>(a, T, t, rank);
      if constexpr (C::DYN) {
        // the scheduler warp has seen the unit's dependency met (its acquire,
        // released to this CTA through dep_ok); the proxy fence then orders this
        // thread's tensor loads after it.  This thread takes no other fence: a
        // release here would wait for its own copies in flight.
        const int j = uw.pos - 1;
        if (lane == 0) *reinterpret_cast<volatile int*>(&ring.prod_pos) = uw.pos;
        if (a.dep_flags) {
          if (!mbar_wait(smem_u32(&ring.dep_ok[j % kSchedRing]), (uint32_t)(j / kSchedRing) & 1u,
                         abort_flag, a.status))
            break;
          if (lane == 0) fence_proxy_async_global();
        }
        __syncwarp();
      }
      const int n0 = C::SWIGLU_B ? ti.nb * (C::NSUB * C::BN / 2) : ti.nb * C::BN;
      const int m0 = ti.mb * BM;
      bool ok = true;
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, a.status)) { ok = false; break; }
        const uint32_t fb = smem_u32(&full_bar[stage]);
        const uint32_t fbp = C::PAIR ? mapa_shared(fb, 0) : fb;  // barrier the copies complete on
        const uint32_t sA = smem_base + stage * C::STAGE_BYTES;
        const uint32_t sB = sA + C::A_BYTES;
        if (!C::PAIR || leader) {
          if (lane == 0) mbar_arrive_expect_tx(fb, C::FULL_TX);
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
        }
        __syncwarp();
        const int kc = kb * BK;               // K coordinate inside the group
        const int kr = ti.kstart + kc;        // absolute K coordinate (RAGGED_K)
        const int kx = C::SCH == RAGGED_K ? kr : kc;
        // ---- A
        if constexpr (C::A_GATHER) {
          // A comes from the gather warps
        } else if constexpr (C::AL == KMAJ_TILE) {
          if (lane == 0) {
            if constexpr (C::PAIR) tma_load_2d_pair(sA, &tmA, fbp, kx, C::SCH == RAGGED_K ? m0 : ti.row0);
            else tma_load_2d(sA, &tmA, fb, kx, C::SCH == RAGGED_K ? m0 : ti.row0);
          }
        } else {  // MN_TILE: two 64-wide groups along M, 64 k-rows each
          if (lane == 0) {
            if constexpr (C::PAIR) {
              tma_load_2d_pair(sA, &tmA, fbp, m0, kr);
              tma_load_2d_pair(sA + 8192, &tmA, fbp, m0 + 64, kr);
            } else {
              tma_load_2d(sA, &tmA, fb, m0, kr);
              tma_load_2d(sA + 8192, &tmA, fb, m0 + 64, kr);
            }
          }
        }
        // ---- B
        if constexpr (C::PAIR && C::BL == KMAJ_TILE) {
          // this CTA's half of the B tile: 128 rows (SwiGLU: rank 0 gate, rank 1
          // up); WIDE: the halves of two tiles, the second 128 columns further.
          // A NARROW wide unit: CTA r takes gate rows n0 + 128 r (tile 0) and the
          // up rows of the same columns (tile 1), the UMMAs' 256-row sides.
          if (lane == 0) {
#pragma unroll
            for (int b = 0; b < C::NSUB; ++b) {
              const int nc = C::SWIGLU_B
                                 ? (narrow_cols<C>(ti) ? (b == 0 ? n0 : a.inter + n0) + 128 * rank
                                              : (rank == 0 ? n0 : a.inter + n0) + 128 * b)
                                 : n0 + rank * 128;
              const uint32_t dst = sB + b * (C::B_ROWS * BK * 2);
              if constexpr (C::B3D) tma_load_3d_pair(dst, &tmB, fbp, kc, nc, ti.g);
              else tma_load_2d_pair(dst, &tmB, fbp, kx, nc);
            }
          }
        } else if constexpr (C::PAIR && C::BL == MN_TILE) {
          // this CTA's half: two 64-wide N groups
          if (lane == 0) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              const int nc = n0 + 128 * rank + 64 * b;
              if constexpr (C::B3D) tma_load_3d_pair(sB + b * 8192, &tmB, fbp, nc, kc, ti.g);
              else tma_load_2d_pair(sB + b * 8192, &tmB, fbp, nc, kr);
            }
          }
        } else if constexpr (C::BL == KMAJ_TILE) {
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
    // wait until every stage this CTA filled has been released by all consumers
    // (with PAIR, the even CTA's commits, which arrive remotely in the odd one)
    for (int i = 0; i < C::STAGES && !*abort_flag; ++i) {
      if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, a.status)) break;
      if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
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
    // with PAIR the odd CTA issues nothing: the even CTA's UMMAs cover both
    UnitWalk<C::DYN> uw{&ring, 0, ustep, total, abort_flag, a.status};
    for (int t = (!C::PAIR || leader) ? uw.first(unit0) : total; t < total && !*abort_flag;
         t = uw.next(t)) {
      const TileInfo ti = decode_tile<C>(a, T, t, rank);
      if constexpr (C::WIDE) {
        // The unit takes both accumulators, which the epilogue drains one after
        // the other.  Once accumulator 0 is free its UMMAs start; each stage is
        // held (not released to the producer) until accumulator 1 is free too
        // and the stage's second half has been issued.
        if (narrow_cols<C>(ti)) {
          const int r = narrow_wide_unit<C>(ti.kblocks, narrow_cols<C>(ti), smem_base, tmem_base,
                                            smem_u32(&full_bar[0]), smem_u32(&empty_bar[0]),
                                            smem_u32(&tfull_bar[0]), smem_u32(&tempty_bar[0]),
                                            stage, phase, acc_phase, lane, abort_flag, a.status);
          if (r < 0) break;
          stage = r & 0xFFFF;
          phase = (uint32_t)r >> 16;
          acc_phase ^= 1;
        } else if (!wide_unit<C>(ti, smem_base, tmem_base, full_bar, empty_bar, tfull_bar,
                                 tempty_bar, stage, phase, acc_phase, lane, abort_flag, a.status)) {
          break;
        }
        continue;
      }
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
            if constexpr (C::PAIR) umma_bf16_pair(d_tmem, ad, bd, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
            else umma_bf16(d_tmem, ad, bd, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          if constexpr (C::PAIR) umma_commit_pair(smem_u32(&empty_bar[stage]));
          else umma_commit(smem_u32(&empty_bar[stage]));
        }
        __syncwarp();
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) {
        if constexpr (C::PAIR) {
          if (ti.kblocks > 0) umma_commit_pair(smem_u32(&tfull_bar[acc]));
          else {
            mbar_arrive(smem_u32(&tfull_bar[acc]));
            mbar_arrive_remote(mapa_shared(smem_u32(&tfull_bar[acc]), 1));
          }
        } else {
          if (ti.kblocks > 0) umma_commit(smem_u32(&tfull_bar[acc]));
          else mbar_arrive(smem_u32(&tfull_bar[acc]));
        }
      }
      __syncwarp();
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (*abort_flag && (!C::PAIR || leader)) {
      // wait (bounded) for UMMAs already issued before TMEM is released
      if (lane == 0) {
        if constexpr (C::PAIR) umma_commit_pair(smem_u32(&drain_bar));
        else umma_commit(smem_u32(&drain_bar));
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&drain_bar), 0) && globaltimer() - t0 < 20000000ull) {
        }
      }
      __syncwarp();
    }
  } else if (C::DYN && warp == C::SCHED_WARP) {
    // ================= scheduler (DYN) =================
    // Leader CTA: takes unit ids from the global counter and publishes them to
    // both CTAs' rings, staying a few units ahead of its producer.  Both CTAs:
    // walks its own ring and, per unit, waits until the producer kernel's count
    // for the unit's 256-row block is complete, then clears the unit to this
    // CTA's producer (dep_ok).  No thread of this warp issues copies, so its
    // releases and fences wait for nothing of the data path.
    if (lane == 0) {
      int published = 0;
      bool sent_end = false;
      int pending = leader ? atomicAdd(a.sched_counter, 1) : 0;
      int pos = 0;  // next ring position to clear
      unsigned long long t0 = globaltimer();
      while (!*abort_flag) {
        if (leader && !sent_end &&
            published < *reinterpret_cast<volatile int*>(&ring.prod_pos) + 3) {
          ring_publish(ring, published++, pending);
          if (pending >= total) sent_end = true;
          else pending = atomicAdd(a.sched_counter, 1);
          t0 = globaltimer();
          continue;
        }
        // clear the next published unit
        const int s = pos % kSchedRing;
        const uint32_t par = (uint32_t)(pos / kSchedRing) & 1u;
        if (mbar_test_wait_cluster(smem_u32(&ring.full[s]), par)) {
          const int t = *reinterpret_cast<volatile int*>(&ring.id[s]);
          if (t >= total) break;
          if (a.dep_flags) {
            const TileInfo ti = decode_tile<C>(a, T, t, rank);
            if (!dep_wait(a.dep_flags + dep_pair<C>(a, T, ti.g, ti.mb), a.dep_target, abort_flag,
                          a.status))
              break;
            mbar_arrive(smem_u32(&ring.dep_ok[s]));
          }
          ++pos;
          t0 = globaltimer();
        } else if (globaltimer() - t0 > kWaitLimitNs) {
          *abort_flag = 1;
          record_status(a.status, MOE_DEV_TIMEOUT);
          break;
        }
      }
    }
    __syncwarp();
  } else if (C::GATHER && warp >= 2 + C::EPI_WARPS) {
    // ================= gather warps (LSU cp.async) =================
    gather_role<C>(a, T, smem_base, full_bar, empty_bar, abort_flag, warp - 2 - C::EPI_WARPS,
                   lane, total, rank, unit0, ustep);
  } else {
    // ================= epilogue =================
    const int quad = warp & 3;
    const int epi = warp - 2;                  // 0 .. EPI_WARPS-1
    const int cpart = epi >> 2;                // column part of this warp
    constexpr int nparts = C::EPI_WARPS / 4;
    const int row_in_tile = quad * 32 + lane;
    WarpOut<C::EPI_BUFS, C::EPI_BUF_BYTES> wo;
    wo.buf0 = smem_base + C::STAGES * C::STAGE_BYTES + epi * (C::EPI_BUFS * C::EPI_BUF_BYTES);
    wo.lane = lane;
    wo.next = 0;
    wo.inflight = 0;
    wo.hint[0] = a.out_l2[0];
    wo.hint[1] = a.out_l2[1];
    wo.policy[0] = l2_policy(a.out_l2[0]);
    wo.policy[1] = l2_policy(a.out_l2[1]);
    int acc = 0;
    uint32_t acc_phase = 0;
    UnitWalk<C::DYN> uw{&ring, 0, ustep, total, abort_flag, a.status};
    for (int t = uw.first(unit0); t < total && !*abort_flag; t = uw.next(t)) {
      const TileInfo tu = decode_tile<C>(a, T, t, rank);
      bool ok = true;
      // WIDE: the unit's n-blocks one after the other, accumulator 0 then 1
      for (int sub = 0; sub < C::NSUB; ++sub) {
        TileInfo ti = tu;
        if constexpr (C::WIDE) ti.nb = 2 * tu.nb + sub;
        if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tacc = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * C::BN;
        if (ti.phantom) {
          // pair slot past the group's last tile: nothing to store
        } else if (narrow_cols<C>(ti)) {
          // a NARROW unit: accumulator 0 holds both halves, accumulator 1 nothing
          if constexpr (C::NARROW)
            if (sub == 0)
              epilogue_narrow_swiglu(a.h_out, a.inter, ti.nb * (C::BN / 2) + 128 * rank, ti.row0,
                                     ti.rows_valid, ti.narrow, tacc, row_in_tile, cpart, nparts);
        } else if constexpr (C::EPI == EPI_STORE_F32)
          epilogue_store_f32<C>(a, ti, tacc, row_in_tile, wo, &tmD0, cpart, nparts);
        else if constexpr (C::EPI == EPI_SWIGLU && C::EPI_COLS == 32)
          epilogue_swiglu_h32<C>(a, ti, tacc, row_in_tile, wo, &tmD1, cpart, nparts);
        else if constexpr (C::EPI == EPI_SWIGLU)
          epilogue_swiglu<C>(a, ti, tacc, row_in_tile, wo, &tmD0, &tmD1, cpart, nparts);
        else if constexpr (C::EPI == EPI_STORE)
          epilogue_store<C>(a, ti, tacc, row_in_tile, wo, &tmD0, cpart, nparts);
        else
          epilogue_dgrad_swiglu<C>(a, T, ti, tacc, row_in_tile, wo, &tmD0, &tmD1, cpart, nparts);
        // the accumulator's TMEM has been read: one arrival per warp (PAIR: on the
        // even CTA's barrier, whose thread overwrites both CTAs' accumulators)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (C::PAIR) mbar_arrive_remote(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
          else mbar_arrive(smem_u32(&tempty_bar[acc]));
        }
        if (a.dep_signal) {
          // producer side: once this warp's rows of the unit are in global memory
          // (its direct stores, and its TMA stores complete), count it on the
          // unit's 256-row block
          __threadfence();
          __syncwarp();
          if (lane == 0) {
            bulk_wait_all();
            fence_proxy_async_global();
            red_release_gpu_add(a.dep_flags + dep_pair<C>(a, T, ti.g, ti.mb), 1);
          }
          __syncwarp();
          wo.inflight = 0;
        }
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      if (!ok) break;
    }
    // every TMA store must have completed before the CTA exits
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  if constexpr (C::CL == 2) cluster_sync();  // no CTA leaves while its peer may still write to it
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (C::PAIR) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace moe
