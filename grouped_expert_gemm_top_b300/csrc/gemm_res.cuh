// Weight-gradient GEMM with one operand resident in shared memory.
//
//   D_g[m, n] = sum over the expert's K token rows k of A_g[k, m] B_g[k, n]
//
// (dW_gu[e] = [dg|du]^T x, dW_down[e] = dout^T (w h): both operands are read
// MN-major from row-per-token matrices.)  The streaming weight-gradient GEMM
// re-reads both operands for every 256 x 256 output tile although an expert
// has only K ~ 256 rows, so each SM pulls 128 KB from L2 per 1 us tile and the
// mainloop is bound by that ingress.  Here, for an expert with K <= 256, one
// operand's whole K slice (4 k-blocks x 16 KB per CTA) stays in shared memory
// for a work unit that runs every tile along the other output dimension,
// streaming only the other operand:
//   RES_A: unit = (expert, m-block pair), A resident, tiles = the n-blocks,
//          B streamed;
//   RES_B: unit = (expert, n-block), B resident, tiles = the m-block pairs,
//          A streamed.
// An operand comes by TMA from a row-per-slot matrix, or is gathered by the
// LSU warps straight from the token rows it is a copy of.
// An expert with more rows gets one unit per output tile instead, and the
// resident slots become a ring through which that operand streams.
// The slots form one ring across units (RSLOTS >= 4 k-blocks): with more slots
// than a unit's four k-blocks, the next unit's first blocks land in slots the
// running unit does not use, so they are fetched while it still computes
// instead of after its last UMMA.
//
// CTA pairs as in the streaming kernel (cta_group::2, 256 x 256 tiles): each
// CTA holds its own 128 rows of A and half of the B columns; the even CTA
// issues the UMMAs.  Roles:
//   warp 0      streamed-operand TMA producer (idle when it is gathered)
//   warp 1      TMEM allocator; UMMA issuer in the even CTA
//   warps 2..    epilogue (the streaming kernel's bf16 store epilogue), 4, 8 or 16
//   next 4      gather warps (a gathered operand only)
//   last warp   resident-operand TMA loader (idle when it is gathered):
//               refills the next slot of the ring as soon as the last UMMA
//               reading it has completed
#pragma once
#include "gemm.cuh"

namespace moe {

enum ResMode : int { RES_A = 1, RES_B = 2 };

template <int RES_, int AL_, int BL_, int STAGES_, int EPI_BUFS_, int EPI_WARPS_ = 4,
          int RSLOTS_ = 4, int EPI_COLS_ = 64>
struct ResCfg {
  static constexpr int RES = RES_;
  static constexpr int AL = AL_;  // MN_TILE or (streamed, RES_B) MN_GATHER
  static constexpr int BL = BL_;  // MN_TILE or (streamed, RES_A) MN_GATHER
  static constexpr int BN = 256;
  static constexpr int CL = 2;
  static constexpr bool PAIR = true;
  static constexpr bool SWIGLU_B = false;
  static constexpr int SCH = RAGGED_K;
  static constexpr int EPI = EPI_STORE;
  // 4, 8 or 16 epilogue warps: 1, 2 or 4 per TMEM lane quarter, each on an
  // equal share of the tile's four 64-column groups
  static constexpr int EPI_WARPS = EPI_WARPS_;
  static_assert(EPI_WARPS == 4 || EPI_WARPS == 8 || EPI_WARPS == 16, "epilogue warps per lane quarter");
  static constexpr int EPI_BUFS = EPI_BUFS_;
  // bf16 columns of a staging block: 64 (4 KB, 128-byte rows) or 32 (2 KB,
  // 64-byte rows: half the staging memory, for one more streamed stage)
  static constexpr int EPI_COLS = EPI_COLS_;
  static_assert(EPI_COLS == 64 || EPI_COLS == 32, "staging block width");
  static constexpr int EPI_BUF_BYTES = EPI_COLS * 64;
  static constexpr bool A_GATHER = AL == MN_GATHER;
  static constexpr bool B_GATHER = BL == MN_GATHER;
  static constexpr bool GATHER = A_GATHER || B_GATHER;
  // which operand the gather warps fill: the streamed one, or the resident one
  static constexpr bool STREAM_GATHER = RES == RES_A ? B_GATHER : A_GATHER;
  static constexpr bool RES_GATHER = RES == RES_A ? A_GATHER : B_GATHER;
  static_assert(!(A_GATHER && B_GATHER), "one gathered operand");
  static_assert((AL == MN_TILE || AL == MN_GATHER) && (BL == MN_TILE || BL == MN_GATHER),
                "weight-gradient operands are MN-major");
  static constexpr int GATHER_WARPS = GATHER ? 4 : 0;
  static constexpr int RES_WARP = 2 + EPI_WARPS + GATHER_WARPS;
  static constexpr int THREADS = 32 * (RES_WARP + 1);
  static constexpr int STAGES = STAGES_;
  static constexpr int GATHER_LAG = STAGES - 2;
  static_assert(!GATHER || GATHER_LAG >= 1, "gathers need >= 3 stages");
  static constexpr int BLK = BM * BK * 2;  // one operand's 128 x 64 block of a CTA: 16 KB
  static constexpr int RSLOTS = RSLOTS_;   // resident-operand ring (k-block slots)
  static constexpr int KRES = 4 * BK;      // experts with at most 256 rows stay resident
  // a resident unit's k-blocks fit the ring; the gather signals a slot 2 fills
  // later, so the ring must be deeper than that; slot ids fit 4 bits
  static_assert(RSLOTS >= KRES / BK && RSLOTS <= 16, "resident ring depth");
  static constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN, true, true);
  // the even CTA's full barriers (streamed stages) and rfull barriers (resident
  // slots): both CTAs' TMA bytes, or one arrival per gather warp of both CTAs
  static constexpr uint32_t FULL_TX = STREAM_GATHER ? 0 : 2 * BLK;
  static constexpr uint32_t FULL_ARRIVALS = STREAM_GATHER ? 2 * GATHER_WARPS : 1;
  static constexpr uint32_t RFULL_ARRIVALS = RES_GATHER ? 2 * GATHER_WARPS : 1;
  static constexpr uint32_t TEMPTY_ARRIVALS = 2 * EPI_WARPS;
  static constexpr int SMEM_BYTES =
      (STAGES + RSLOTS) * BLK + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024 - 8 * 1024, "dynamic + static shared memory per CTA");
};

// A work unit: resident (the expert's K fits the slots) or one streamed tile.
struct ResUnit {
  int g, ntiles, kstart, kblocks;
  bool stream;
  int p, nb;  // the resident operand's pair (RES_A) or n-block (RES_B); both for a streamed tile
};

template <class C>
__device__ __forceinline__ int res_nmb(const GemmArgs& a) { return (a.M + BM - 1) / BM; }
template <class C>
__device__ __forceinline__ int res_nnb(const GemmArgs& a) { return (a.N + C::BN - 1) / C::BN; }

// Unit t: tile_prefix runs over the groups in the order `order` (position ->
// group id).
template <class C>
__device__ __forceinline__ ResUnit res_unit(const GemmArgs& a, const SmemTables& T,
                                            const int* order, int t) {
  int lo = 0, hi = a.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (T.tile_prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  ResUnit u;
  const int g = order[lo];
  u.g = g;
  const int local = t - T.tile_prefix[lo];
  const int mu = (res_nmb<C>(a) + 1) / 2;
  u.stream = T.cnt[g] > C::KRES;
  if (u.stream) {  // one tile; m-block pairs fastest
    u.ntiles = 1;
    u.p = local % mu;
    u.nb = local / mu;
  } else {
    u.ntiles = C::RES == RES_A ? res_nnb<C>(a) : mu;
    u.p = local;
    u.nb = local;
  }
  u.kstart = T.start[g];
  u.kblocks = (T.cnt[g] + BK - 1) / BK;
  return u;
}

// Unit order.  Units are dealt to the CTA pairs round-robin.  When some group
// has more rows than the resident slots hold, its units are single tiles whose
// length grows with its rows, so the groups are taken in descending row count
// (ties: lower id): the longest units start first, on different pairs.
// Otherwise the order is the group ids' (tile_prefix as built).  One warp.
template <class C, class UnitsFn>
__device__ void res_order_groups(const GemmArgs& a, SmemTables& T, int* order, int lane,
                                 UnitsFn units) {
  int mx = 0;
  for (int g = lane; g < a.G; g += 32) mx = max(mx, T.cnt[g]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (mx <= C::KRES) {
    for (int g = lane; g < a.G; g += 32) order[g] = g;
    __syncwarp();
    return;
  }
  for (int g = lane; g < a.G; g += 32) {
    const int c = T.cnt[g];
    int r = 0;
    for (int h = 0; h < a.G; ++h) {
      const int ch = T.cnt[h];
      r += (ch > c) || (ch == c && h < g);
    }
    order[r] = g;
  }
  __syncwarp();
  int run = 0;
  for (int b0 = 0; b0 < a.G; b0 += 32) {
    const int i = b0 + lane;
    const int u = i < a.G ? units(T.cnt[order[i]]) : 0;
    int inc = u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += x;
    }
    if (i < a.G) T.tile_prefix[i] = run + inc - u;
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) {
    T.tile_prefix[a.G] = run;
    T.total_tiles = run;
  }
  __syncwarp();
}

template <class C>
__device__ __forceinline__ TileInfo res_tile(const GemmArgs& a, const ResUnit& u, int j, int rank) {
  TileInfo ti;
  const int p = (u.stream || C::RES == RES_A) ? u.p : j;
  ti.g = u.g;
  ti.nb = (u.stream || C::RES == RES_B) ? u.nb : j;
  ti.mb = 2 * p + rank;
  const int nMB = res_nmb<C>(a);
  ti.phantom = ti.mb >= nMB;
  ti.row0 = ti.mb * BM;
  ti.rows_valid = ti.phantom ? 0 : min(BM, a.M - ti.mb * BM);
  ti.kstart = u.kstart;
  ti.kblocks = u.kblocks;
  return ti;
}

// Gather warp gw's 16 k-rows of an MN-major 128-column block (64 k-rows, two
// 64-wide groups, 128-byte swizzle) from the token rows: k-row r of the block
// is token row `kid` of lane r - 16 gw; columns x0 .. x0+127 (a 64-column
// group at or past xlim, possible when the extent is a multiple of 64 but not
// of 128, is not copied: its rows or columns are not stored).
template <class GA>
__device__ __forceinline__ void gather_block(const GA& a, uint32_t dst, int x0, int xlim, int kid,
                                             int gw, int lane) {
  const int cc = lane & 15;
  const int jg = cc >> 3, c = cc & 7;
  const __nv_bfloat16* col = a.gsrc + x0 + jg * 64 + c * 8;
  const bool inside = x0 + jg * 64 < xlim;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int rl = 2 * q + (lane >> 4);  // 0..15 within this warp's k-rows
    const int r = gw * 16 + rl;
    const int srow = __shfl_sync(0xffffffffu, kid, rl);
    if (inside) cp_async_16(dst + jg * 8192 + r * 128 + ((c ^ (r & 7)) << 4), col + (size_t)srow * a.gld);
  }
}

// MN-major block of an operand (two 64-wide groups of 64 k-rows) by TMA, to
// this CTA's shared memory, completing on the even CTA's barrier `barp`.
__device__ __forceinline__ void res_load_block(uint32_t dst, const CUtensorMap* map, uint32_t barp,
                                               int x, int k) {
  tma_load_2d_pair(dst, map, barp, x, k);
  tma_load_2d_pair(dst + 8192, map, barp, x + 64, k);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    res_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD0,
                    const __grid_constant__ CUtensorMap tmD1, const GemmArgs a) {
  (void)tmD1;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::STAGES];
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
  __shared__ __align__(8) uint64_t rfull_bar[C::RSLOTS];
  __shared__ __align__(8) uint64_t rempty_bar[C::RSLOTS];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ SmemTables T;
  __shared__ int order[kMaxGroups];  // unit order: position -> group

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t res_base = smem_base + C::STAGES * C::BLK;
  volatile int* abort_flag = &T.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), C::FULL_ARRIVALS);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int s = 0; s < C::RSLOTS; ++s) {
      mbar_init(smem_u32(&rfull_bar[s]), C::RFULL_ARRIVALS);
      mbar_init(smem_u32(&rempty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), C::TEMPTY_ARRIVALS);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    T.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD0);
  }
  if (warp == 2) {
    const int nMB = res_nmb<C>(a), nNB = res_nnb<C>(a);
    const auto units = [&](int cnt) {
      const int mu = (nMB + 1) / 2;
      if (cnt > C::KRES) return mu * nNB;  // one unit per streamed tile
      return C::RES == RES_A ? mu : nNB;
    };
    build_group_tables(a, T, lane, units);
    res_order_groups<C>(a, T, order, lane, units);
  }
  __syncthreads();
  if (T.total_tiles == 0) return;  // no work: leave before touching tensor memory or the peer
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&T.tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // the peer's barriers are initialised before any remote op
  tc_fence_after();
  const uint32_t tmem_base = T.tmem_base;
  const int total = T.total_tiles;
  const int rank = (int)cluster_ctarank();
  const bool leader = rank == 0;
  const int unit0 = blockIdx.x / 2;
  const int ustep = gridDim.x / 2;

  if (warp == 0) {
    // ================= streamed-operand producer =================
    int stage = 0;
    uint32_t phase = 0;
    uint32_t filled = 0, fill_parity = 0;
    for (int t = unit0; t < total && !*abort_flag && !C::STREAM_GATHER; t += ustep) {
      const ResUnit u = res_unit<C>(a, T, order, t);
      bool ok = true;
      for (int j = 0; j < u.ntiles && ok; ++j) {
        const TileInfo ti = res_tile<C>(a, u, j, rank);
        // the tile after this one (the next of this unit, or the next unit's
        // first): its k-blocks are sent to L2 one tile ahead of their loads
        ResUnit un = u;
        bool has_next = j + 1 < u.ntiles;
        if (!has_next && t + ustep < total) {
          un = res_unit<C>(a, T, order, t + ustep);
          has_next = true;
        }
        const TileInfo tn = has_next ? res_tile<C>(a, un, j + 1 < u.ntiles ? j + 1 : 0, rank) : ti;
        for (int kb = 0; kb < u.kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, a.status)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full_bar[stage]);
          const uint32_t sS = smem_base + stage * C::BLK;
          if (leader) {
            if (lane == 0) mbar_arrive_expect_tx(fb, C::FULL_TX);
            filled |= 1u << stage;
            fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          }
          if (lane == 0) {
            const int kr = u.kstart + kb * BK;
            if constexpr (C::RES == RES_A) res_load_block(sS, &tmB, mapa_shared(fb, 0), ti.nb * C::BN + 128 * rank, kr);
            else res_load_block(sS, &tmA, mapa_shared(fb, 0), ti.mb * BM, kr);
            if (has_next && kb < un.kblocks && !tn.phantom) {
              const int kn = un.kstart + kb * BK;
              const CUtensorMap* m = C::RES == RES_A ? &tmB : &tmA;
              const int xn = C::RES == RES_A ? tn.nb * C::BN + 128 * rank : tn.mb * BM;
              tma_prefetch_l2_2d(m, xn, kn);
              tma_prefetch_l2_2d(m, xn + 64, kn);
            }
          }
          __syncwarp();
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) break;
    }
    if (!C::STREAM_GATHER) {
      for (int i = 0; i < C::STAGES && !*abort_flag; ++i) {
        if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, a.status)) break;
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag) {
        for (int s = 0; s < C::STAGES; ++s) {
          if (!((filled >> s) & 1u)) continue;
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(smem_u32(&full_bar[s]), (fill_parity >> s) & 1u) &&
                 globaltimer() - t0 < 20000000ull) {
          }
        }
      }
    }
  } else if (warp == C::RES_WARP) {
    // ================= resident-operand loader =================
    uint32_t rph = 0;     // per slot: parity bit of its uses so far
    uint32_t armed = 0;   // slots with a load issued (for the abort drain)
    uint32_t arm_par = 0;
    int rbase = 0;        // ring slot of the unit's first k-block
    for (int t = unit0; t < total && !*abort_flag && !C::RES_GATHER; t += ustep) {
      const ResUnit u = res_unit<C>(a, T, order, t);
      bool ok = true;
      for (int kb = 0; kb < u.kblocks; ++kb) {
        const int sl = (rbase + kb) % C::RSLOTS;
        if (!mbar_wait(smem_u32(&rempty_bar[sl]), ((rph >> sl) & 1u) ^ 1u, abort_flag, a.status)) { ok = false; break; }
        const uint32_t rb = smem_u32(&rfull_bar[sl]);
        const uint32_t slot = res_base + sl * C::BLK;
        if (leader) {
          if (lane == 0) mbar_arrive_expect_tx(rb, 2 * C::BLK);
          armed |= 1u << sl;
          arm_par = (arm_par & ~(1u << sl)) | (((rph >> sl) & 1u) << sl);
        }
        if (lane == 0) {
          const int kr = u.kstart + kb * BK;
          if constexpr (C::RES == RES_A) res_load_block(slot, &tmA, mapa_shared(rb, 0), (2 * u.p + rank) * BM, kr);
          else res_load_block(slot, &tmB, mapa_shared(rb, 0), u.nb * C::BN + 128 * rank, kr);
        }
        __syncwarp();
        rph ^= 1u << sl;
      }
      if (!ok) break;
      rbase = (rbase + u.kblocks) % C::RSLOTS;
    }
    if (*abort_flag) {
      for (int s = 0; s < C::RSLOTS; ++s) {
        if (!((armed >> s) & 1u)) continue;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&rfull_bar[s]), (arm_par >> s) & 1u) &&
               globaltimer() - t0 < 20000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ================= UMMA issuer (even CTA) =================
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t rph = 0;  // per slot: parity of the next resident fill
    int rbase = 0;     // ring slot of the unit's first k-block
    bool ok = true;
    for (int t = unit0; t < total && !*abort_flag && leader && ok; t += ustep) {
      const ResUnit u = res_unit<C>(a, T, order, t);
      for (int j = 0; j < u.ntiles && ok; ++j) {
        if (!mbar_wait(smem_u32(&tempty_bar[acc]), acc_phase ^ 1, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::BN;
        const bool last = j == u.ntiles - 1;
        for (int kb = 0; kb < u.kblocks; ++kb) {
          // the resident operand's block kb: in ring slot rbase + kb, filled
          // once per unit (the first tile waits for it) or, streamed, once per
          // k-block
          const int sl = (rbase + kb) % C::RSLOTS;
          if (j == 0) {
            if (!mbar_wait(smem_u32(&rfull_bar[sl]), (rph >> sl) & 1u, abort_flag, a.status)) { ok = false; break; }
            rph ^= 1u << sl;
          }
          if (!mbar_wait(smem_u32(&full_bar[stage]), phase, abort_flag, a.status)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sR = res_base + sl * C::BLK;
            const uint32_t sS = smem_base + stage * C::BLK;
            const uint32_t sA = C::RES == RES_A ? sR : sS;
            const uint32_t sB = C::RES == RES_A ? sS : sR;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16_pair(d_tmem, smem_desc_sw128(sA + kk * 2048, 8192, 1024),
                             smem_desc_sw128(sB + kk * 2048, 8192, 1024), C::IDESC,
                             (kb | kk) != 0 ? 1u : 0u);
            umma_commit_pair(smem_u32(&empty_bar[stage]));
            if (last) umma_commit_pair(smem_u32(&rempty_bar[sl]));
          }
          __syncwarp();
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) {
          if (u.kblocks > 0) umma_commit_pair(smem_u32(&tfull_bar[acc]));
          else {
            mbar_arrive(smem_u32(&tfull_bar[acc]));
            mbar_arrive_remote(mapa_shared(smem_u32(&tfull_bar[acc]), 1));
          }
        }
        __syncwarp();
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      rbase = (rbase + u.kblocks) % C::RSLOTS;
    }
    if (*abort_flag && leader) {
      if (lane == 0) {
        umma_commit_pair(smem_u32(&drain_bar));
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&drain_bar), 0) && globaltimer() - t0 < 20000000ull) {
        }
      }
      __syncwarp();
    }
  } else if (C::GATHER && warp >= 2 + C::EPI_WARPS) {
    // ================= gather warps: an operand from token rows =================
    const int gw = warp - 2 - C::EPI_WARPS;
    const int xlim = C::A_GATHER ? a.M : a.N;
    uint32_t ring = 0;  // slots or stages copied but not yet signalled (4 bits each, FIFO)
    int rn = 0;
    bool ok = true;
    if constexpr (C::STREAM_GATHER) {
      // the streamed operand, stage by stage; a stage is signalled GATHER_LAG stages later
      constexpr int LAG = C::GATHER_LAG;
      int stage = 0;
      uint32_t phase = 0;
      for (int t = unit0; t < total && !*abort_flag && ok; t += ustep) {
        const ResUnit u = res_unit<C>(a, T, order, t);
        for (int j = 0; j < u.ntiles && ok; ++j) {
          const TileInfo ti = res_tile<C>(a, u, j, rank);
          for (int kb = 0; kb < u.kblocks; ++kb) {
            // token row of k-row gw*16 + (lane & 15) of this k-block (loaded before the wait)
            const int kid = gather_row(a, T, u.g, kb * BK + gw * 16 + (lane & 15));
            if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, a.status)) { ok = false; break; }
            // A: this CTA's 128 rows of the tile; B: its half of the 256 columns
            const int x0 = C::A_GATHER ? ti.mb * BM : ti.nb * C::BN + 128 * rank;
            if (!(C::A_GATHER && ti.phantom))
              gather_block(a, smem_base + stage * C::BLK, x0, xlim, kid, gw, lane);
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
          }
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      while (rn > 0) {
        arrive_full<C>(full_bar, ring & 15u, lane, rank);
        ring >>= 4;
        --rn;
      }
    } else {
      // the resident operand, slot by slot along the ring.  Every slot of a
      // unit is signalled before the next unit's first fill; within a
      // streamed unit a slot is signalled 2 slots later.  A fill waits for
      // the last UMMA that read its slot: with a ring deeper than a unit, the
      // next unit's first fills need none of the running unit's slots.
      constexpr int LAG = 2;
      static_assert(C::RSLOTS > LAG, "a slot is signalled before its next fill");
      uint32_t rph = 0;
      int rbase = 0;
      for (int t = unit0; t < total && !*abort_flag && ok; t += ustep) {
        const ResUnit u = res_unit<C>(a, T, order, t);
        // A: the pair's m-block of this CTA; B: this CTA's half of the n-block
        const int x0 = C::A_GATHER ? (2 * u.p + rank) * BM : u.nb * C::BN + 128 * rank;
        for (int kb = 0; kb < u.kblocks; ++kb) {
          const int sl = (rbase + kb) % C::RSLOTS;
          const int kid = gather_row(a, T, u.g, kb * BK + gw * 16 + (lane & 15));
          if (!mbar_wait(smem_u32(&rempty_bar[sl]), ((rph >> sl) & 1u) ^ 1u, abort_flag, a.status)) { ok = false; break; }
          rph ^= 1u << sl;
          gather_block(a, res_base + sl * C::BLK, x0, xlim, kid, gw, lane);
          cp_async_commit();
          ring |= (uint32_t)sl << (4 * rn);
          ++rn;
          if (rn > LAG) {
            cp_async_wait<LAG>();
            fence_proxy_async_smem();
            arrive_full<C>(rfull_bar, ring & 15u, lane, rank);
            ring >>= 4;
            --rn;
          }
        }
        cp_async_wait<0>();
        fence_proxy_async_smem();
        while (rn > 0) {
          arrive_full<C>(rfull_bar, ring & 15u, lane, rank);
          ring >>= 4;
          --rn;
        }
        rbase = (rbase + u.kblocks) % C::RSLOTS;
      }
    }
  } else if (warp >= 2 && warp < 2 + C::EPI_WARPS) {
    // ================= epilogue =================
    const int quad = warp & 3;
    const int epi = warp - 2;
    const int cpart = epi >> 2;  // column part of this warp
    constexpr int nparts = C::EPI_WARPS / 4;
    const int row_in_tile = quad * 32 + lane;
    WarpOut<C::EPI_BUFS, C::EPI_BUF_BYTES> wo;
    wo.buf0 = smem_base + (C::STAGES + C::RSLOTS) * C::BLK + epi * (C::EPI_BUFS * C::EPI_BUF_BYTES);
    wo.lane = lane;
    wo.next = 0;
    wo.inflight = 0;
    wo.hint[0] = a.out_l2[0];
    wo.hint[1] = a.out_l2[1];
    wo.policy[0] = l2_policy(a.out_l2[0]);
    wo.policy[1] = l2_policy(a.out_l2[1]);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = unit0; t < total && !*abort_flag && ok; t += ustep) {
      const ResUnit u = res_unit<C>(a, T, order, t);
      for (int j = 0; j < u.ntiles; ++j) {
        const TileInfo ti = res_tile<C>(a, u, j, rank);
        if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tacc = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * C::BN;
        if (!ti.phantom) {
          if constexpr (C::EPI_COLS == 32) epilogue_store32<C>(a, ti, tacc, row_in_tile, wo, &tmD0, cpart, nparts);
          else epilogue_store<C>(a, ti, tacc, row_in_tile, wo, &tmD0, cpart, nparts);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still read or write it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace moe
