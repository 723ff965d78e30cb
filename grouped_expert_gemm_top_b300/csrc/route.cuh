// The router of the MoE layer in one kernel, and the expert sort in one more.
//
// route_kernel: logits = x W_r^T (+ bias) on the tensor cores, then per token
// the softmax over all E experts, the top-k selection (or the balanced gate)
// and the renormalised weights; optionally the per-CTA expert counts of the
// chosen slots (for the sort) and per-CTA sums of the probabilities (for the
// auxiliary load-balancing loss).  This is the router in front of the
// experts ("原生路由器", NeMo AutoModel blog, note on the routing gate) and
// the first half of "sort the tokens by their assigned expert" (same page,
// expert-backend table, grouped_mm row).
//
// One cluster of `splits` CTAs per 128-token tile.  CTA r of the cluster
// multiplies the tile by its K slice of W_r (TMA tile loads, 4- or 6-stage ring,
// one tcgen05 UMMA stream into a 128 x BN fp32 accumulator in TMEM), then
// copies its accumulator into its own shared memory.  After a cluster
// barrier each CTA owns a slice of the tile's tokens: a warp per token reads
// the `splits` partial rows of that token from the cluster's shared memory
// (distributed shared memory; lane l takes the consecutive experts l*P ..
// l*P+P-1, 16 bytes per load), adds them in CTA order and then the bias, so
// the fp32 logits never leave the chip and no split-K partials go to HBM.
//
// route_sort_kernel: one block per route CTA (its tokens' slots, in slot
// order).  From the route kernel's counts (layout [E][ld], column = CTA) it
// forms every expert's total and the count in earlier CTAs, the expert
// offsets (exclusive scan), and places each slot at offset + earlier CTAs'
// count + its rank among this CTA's slots of the same expert (slot order), so
// the order inside an expert is ascending slot id s = t*k + j.
//
// Both are fixed-order functions of their inputs (no floating-point atomics):
// results are bit-identical run to run.
#pragma once
#include <cuda.h>

#include "kernels_misc.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kRouteBM = 128;                 // tokens per cluster tile
constexpr int kRouteWarps = 16;               // 4 of them drain the accumulator; all run the top-k
constexpr int kRouteThreads = 32 * kRouteWarps;
constexpr int kRouteMaxStages = 6;
constexpr int kRouteMaxSplits = 8;            // portable cluster size

struct RouteArgs {
  int T, H, E, k, gate_mode;
  int splits;               // CTAs per cluster (K slices of the router GEMM)
  const float* bias;        // [E] or null
  float* logits_out;        // [T, E] or null
  int32_t* topk_idx;        // [T, k]
  float* topk_w;            // [T, k]
  float* psum_part;         // [CTAs, E] or null: per CTA, sum over its tokens of p[t, e]
  int32_t* hist;            // [E, hist_ld] or null: per CTA, slots of its tokens routed to e
  int hist_ld;
  int* status;
};

// Tokens [lo, hi) of tile `tile` owned by CTA `r` of `splits` (clipped to T).
__host__ __device__ __forceinline__ void route_cta_tokens(int tile, int r, int splits, int T, int& lo,
                                                          int& hi) {
  lo = tile * kRouteBM + r * kRouteBM / splits;
  hi = tile * kRouteBM + (r + 1) * kRouteBM / splits;
  if (lo > T) lo = T;
  if (hi > T) hi = T;
}

template <int BN>  // UMMA N: E rounded up to a multiple of 16 (<= 256)
struct RouteCfg {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N");
  static constexpr int A_BYTES = kRouteBM * 64 * 2;
  static constexpr int B_BYTES = BN * 64 * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN <= 128 ? 6 : 4;  // as many K blocks in flight as fit
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  // lane l of a top-k warp holds the consecutive experts l*P .. l*P+P-1
  static constexpr int P = BN <= 128 ? 4 : 8;
  // the accumulator copy, fp32 rows padded by 16 bytes (conflict-free 16-byte
  // writes of a row per thread), in the ring's memory once the GEMM is done
  static constexpr int PART_LD = ((BN + 31) / 32) * 32 + 4;
  static constexpr int PART_BYTES = kRouteBM * PART_LD * 4;
  static constexpr int SMEM_BYTES = (RING_BYTES > PART_BYTES ? RING_BYTES : PART_BYTES) + 1024;
  static constexpr uint32_t IDESC = idesc_bf16_f32(kRouteBM, BN, false, false);
  static constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  static_assert(SMEM_BYTES <= 227 * 1024 - 20 * 1024, "dynamic + static shared memory per CTA");
  static_assert(STAGES <= kRouteMaxStages && P * 32 >= BN && P % 4 == 0, "route config");
};

// 16 bytes of a CTA's shared memory in the cluster (address from mapa).  Not
// volatile, so that a token's loads issue together; they are ordered after the
// cluster barrier by their address, which comes from mapa after it.
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr) {
  float4 v;
  asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "r"(cluster_addr));
  return v;
}

template <int BN>
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const RouteArgs a) {
  using C = RouteCfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kRouteMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kRouteMaxStages];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int hist_s[kMaxGroupsRouter];
  __shared__ float psum_s[kRouteWarps][kMaxGroupsRouter];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = &abort_s;
  const int rank = (int)cluster_ctarank();
  const int tile = blockIdx.x / a.splits;
  const int m0 = tile * kRouteBM;
  const int kb_total = a.H / 64;
  const int kb0 = rank * kb_total / a.splits, kb1 = (rank + 1) * kb_total / a.splits;
  const int E = a.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&acc_bar), 1);
    abort_s = 0;
    fence_mbar_init();
  }
  for (int e = threadIdx.x; e < kMaxGroupsRouter; e += kRouteThreads) hist_s[e] = 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  // ---------------- GEMM over this CTA's K slice
  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int stage = 0;
      uint32_t phase = 0, filled = 0, fill_par = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag, a.status)) break;
        const uint32_t fb = smem_u32(&full_bar[stage]);
        const uint32_t sA = sbase + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
        filled |= 1u << stage;
        fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
        tma_load_2d(sA, &tmX, fb, kb * 64, m0);
        tma_load_2d(sA + C::A_BYTES, &tmW, fb, kb * 64, 0);
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag) {
        // let copies in flight land before the shared memory is reused (bounded)
        for (int s = 0; s < C::STAGES; ++s) {
          if (!((filled >> s) & 1u)) continue;
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(smem_u32(&full_bar[s]), (fill_par >> s) & 1u) &&
                 globaltimer() - t0 < 20000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // UMMA issuer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(smem_u32(&full_bar[stage]), phase, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sA = sbase + stage * C::STAGE_BYTES;
        const uint32_t sB = sA + C::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem, smem_desc_sw128(sA + kk * 32, 16, 1024),
                    smem_desc_sw128(sB + kk * 32, 16, 1024), C::IDESC, (kb > kb0 || kk) ? 1u : 0u);
        umma_commit(smem_u32(&empty_bar[stage]));
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
      // the accumulator is complete (or, on abort, every issued UMMA has finished)
      umma_commit(smem_u32(&acc_bar));
      (void)ok;
    }
  }
  __syncwarp();

  // ---------------- accumulator -> this CTA's shared memory (rows = tokens)
  float* part = reinterpret_cast<float*>(smem);
  if (warp < 4) {
    // (warp-uniform from here: the TMEM loads below are .sync.aligned)
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&acc_bar), 0, abort_flag, a.status));
    tc_fence_after();
    fence_proxy_async_smem();
    const int row = warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c = 0; c < (BN + 31) / 32; ++c) {
      float v[32];
      if (ok && kb1 > kb0) {
        tmem_ld32(trow + c * 32, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      const uint32_t dst = smem_u32(part + (size_t)row * C::PART_LD + c * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4(dst + 16 * q, __float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                     __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  cluster_sync();  // every CTA's partial rows are visible to the cluster

  // ---------------- softmax, top-k, weights: a warp per token of this CTA's slice
  int t_lo, t_hi;
  route_cta_tokens(tile, rank, a.splits, a.T, t_lo, t_hi);
  uint32_t part_rank[kRouteMaxSplits];
#pragma unroll
  for (int sp = 0; sp < kRouteMaxSplits; ++sp)
    part_rank[sp] = sp < a.splits ? mapa_shared(smem_u32(part), sp) : 0u;
  constexpr int P = C::P;
  const int e0 = lane * P;  // this lane's first expert
  float pacc[P];
#pragma unroll
  for (int i = 0; i < P; ++i) pacc[i] = 0.f;
  const int k = a.k;

  for (int t = t_lo + warp; t < t_hi; t += kRouteWarps) {
    const int r = t - m0;  // row in the tile
    // logits of this lane's experts: the K slices' partial sums in CTA order
    // (every load issued first), then the bias; -inf past E
    float v[P];
#pragma unroll
    for (int i = 0; i < P; ++i) v[i] = 0.f;
    if (e0 < E) {
      float4 q[kRouteMaxSplits][P / 4];
#pragma unroll
      for (int sp = 0; sp < kRouteMaxSplits; ++sp)
#pragma unroll
        for (int h = 0; h < P / 4; ++h)
          if (sp < a.splits)
            q[sp][h] = ld_dsmem_v4(part_rank[sp] + (uint32_t)((r * C::PART_LD + e0 + 4 * h) * 4));
#pragma unroll
      for (int sp = 0; sp < kRouteMaxSplits; ++sp)
#pragma unroll
        for (int h = 0; h < P / 4; ++h)
          if (sp < a.splits) {
            v[4 * h] += q[sp][h].x;
            v[4 * h + 1] += q[sp][h].y;
            v[4 * h + 2] += q[sp][h].z;
            v[4 * h + 3] += q[sp][h].w;
          }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const int e = e0 + i;
      if (e < E) {
        if (a.bias) v[i] += __ldg(a.bias + e);
        mx = fmaxf(mx, v[i]);
        if (a.logits_out) a.logits_out[(size_t)t * E + e] = v[i];
      } else {
        v[i] = -INFINITY;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < P; ++i)
      if (e0 + i < E) z += expf(v[i] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (a.psum_part) {
#pragma unroll
      for (int i = 0; i < P; ++i)
        if (e0 + i < E) pacc[i] += expf(v[i] - mx) / z;
    }
    int my_e = 0;
    float my_p = 0.f;
    if (a.gate_mode == 1) {
      // balanced gate: lane j's expert is (t k + j) mod E; its logit comes from
      // the lane holding it (the same bits)
      my_e = lane < k ? (int)(((long long)t * k + lane) % E) : 0;
      const int owner = my_e / P, slot = my_e - owner * P;
      float l = 0.f;
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const float x = __shfl_sync(0xffffffffu, v[i], owner);
        if (i == slot) l = x;
      }
      if (lane < k) my_p = expf(l - mx) / z;
    } else {
      // softmax gate: this lane's candidate keys and its best one (ties: lower id)
      uint32_t kl[P];
      uint32_t lbk = 0u, taken = 0u;
      int lbi = 0;
#pragma unroll
      for (int i = 0; i < P; ++i) {
        kl[i] = e0 + i < E ? logit_key(v[i]) : 0u;
        if (kl[i] > lbk) { lbk = kl[i]; lbi = i; }
      }
      for (int j = 0; j < k; ++j) {
        // warp argmax in two single-instruction reductions: the largest key,
        // then the lowest expert id holding it
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, lbk);
        const int bi = (int)__reduce_min_sync(0xffffffffu,
                                              lbk == kmax ? (uint32_t)(e0 + lbi) : 0xffffffffu);
        if (bi / P == lane) {  // the owner drops it and finds its next best
          taken |= 1u << (bi - e0);
          lbk = 0u;
          lbi = 0;
#pragma unroll
          for (int i = 0; i < P; ++i)
            if (!((taken >> i) & 1u) && kl[i] > lbk) { lbk = kl[i]; lbi = i; }
        }
        if (lane == j) {
          my_e = bi;
          my_p = expf(key_logit(kmax) - mx) / z;
        }
      }
    }
    float psel = lane < k ? my_p : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) psel += __shfl_xor_sync(0xffffffffu, psel, o);
    if (lane < k) {
      a.topk_idx[(size_t)t * k + lane] = my_e;
      a.topk_w[(size_t)t * k + lane] = my_p / psel;
      if (a.hist) atomicAdd(&hist_s[my_e], 1);
    }
  }
  if (a.psum_part) {
#pragma unroll
    for (int i = 0; i < P; ++i)
      if (e0 + i < E) psum_s[warp][e0 + i] = pacc[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kRouteThreads) {
    if (a.hist) a.hist[(size_t)e * a.hist_ld + blockIdx.x] = hist_s[e];
    if (a.psum_part) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kRouteWarps; ++w) s += psum_s[w][e];
      a.psum_part[(size_t)blockIdx.x * E + e] = s;
    }
  }
  cluster_sync();  // no CTA leaves while the others may still read its shared memory
}

// ---------------------------------------------------------------- expert sort
constexpr int kRouteSortThreads = 256;

__global__ void __launch_bounds__(kRouteSortThreads)
    route_sort_kernel(const int32_t* __restrict__ topk_idx, int T, int k, int E, int splits,
                      int nblk, const int32_t* __restrict__ hist, int hist_ld,
                      int32_t* __restrict__ expert_offsets, int32_t* __restrict__ perm_slot,
                      int32_t* __restrict__ slot_perm, int cap, int* status) {
  __shared__ int base[kMaxGroupsRouter];   // next sorted row of each expert for this block
  __shared__ int first[kMaxGroupsRouter];  // expert totals, then the experts' first rows
  constexpr int NW = kRouteSortThreads / 32;
  __shared__ int wcount[NW][kMaxGroupsRouter];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  int t0, t1;
  route_cta_tokens(b / splits, b % splits, splits, T, t0, t1);
  const int s0 = t0 * k, s1 = t1 * k;
  // this thread's first slot id, fetched now so that its latency overlaps step 1
  int e_first = (s0 + (int)threadIdx.x < s1) ? __ldg(topk_idx + s0 + threadIdx.x) : -1;

  // 1. per expert: the slots of every block (total) and of the blocks before b;
  //    a warp takes EB experts at a time with all their loads in flight
  constexpr int EB = 16;
  for (int e0 = warp * EB; e0 < E; e0 += NW * EB) {
    int tot[EB], pre[EB];
#pragma unroll
    for (int i = 0; i < EB; ++i) tot[i] = pre[i] = 0;
    for (int j0 = 0; j0 < nblk; j0 += 128) {
      const int j = j0 + 4 * lane;
      int c[EB][4];
#pragma unroll
      for (int i = 0; i < EB; ++i) {
        const int32_t* row = hist + (size_t)(e0 + i) * hist_ld;
        c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0;
        if (e0 + i < E) {
          if (j + 3 < nblk) {
            const int4 q = __ldg(reinterpret_cast<const int4*>(row + j));
            c[i][0] = q.x; c[i][1] = q.y; c[i][2] = q.z; c[i][3] = q.w;
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (j + u < nblk) c[i][u] = __ldg(row + j + u);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < EB; ++i)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          tot[i] += c[i][u];
          pre[i] += (j + u < b) ? c[i][u] : 0;
        }
    }
#pragma unroll
    for (int i = 0; i < EB; ++i) {
      const int t = (int)__reduce_add_sync(0xffffffffu, (unsigned)tot[i]);
      const int p = (int)__reduce_add_sync(0xffffffffu, (unsigned)pre[i]);
      if (lane == 0 && e0 + i < E) {
        first[e0 + i] = t;
        base[e0 + i] = p;
      }
    }
  }
  for (int i = threadIdx.x; i < NW * kMaxGroupsRouter; i += kRouteSortThreads) (&wcount[0][0])[i] = 0;
  __syncthreads();
  // 2. expert offsets: exclusive scan of the totals (one warp, E <= 256)
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 < E; b0 += 32) {
      const int e = b0 + lane;
      const int v = e < E ? first[e] : 0;
      int inc = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += x;
      }
      if (e < E) {
        const int off = run + inc - v;
        base[e] += off;
        first[e] = off;
        if (b == 0) expert_offsets[e] = off;
      }
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (b == 0 && lane == 0) expert_offsets[E] = run;
  }
  __syncthreads();
  // 3. this block's slots, 256 at a time in slot order: rank within the warp
  //    by lane (match_any), warps in order, rounds in order
  for (int sb = s0; sb < s1; sb += kRouteSortThreads) {
    const int s = sb + threadIdx.x;
    int e = sb == s0 ? e_first : (s < s1 ? __ldg(topk_idx + s) : -1);
    if (s < s1 && (e < 0 || e >= E)) {
      record_status(status, MOE_DEV_BAD_INDEX);
      e = -1;
    }
    const unsigned m = __match_any_sync(0xffffffffu, e);
    const bool leader = lane == __ffs(m) - 1;
    if (e >= 0 && leader) wcount[warp][e] = __popc(m);
    __syncthreads();
    for (int ee = threadIdx.x; ee < E; ee += kRouteSortThreads) {
      int run = base[ee];
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const int c = wcount[w][ee];
        wcount[w][ee] = run;
        run += c;
      }
      base[ee] = run;
    }
    __syncthreads();
    if (e >= 0) {
      const int pos = wcount[warp][e] + __popc(m & ((1u << lane) - 1u));
      perm_slot[pos] = s;
      slot_perm[s] = (cap > 0 && pos - first[e] >= cap) ? -1 : pos;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < NW * kMaxGroupsRouter; i += kRouteSortThreads) (&wcount[0][0])[i] = 0;
    __syncthreads();
  }
}

}  // namespace moe
