// Memory-bound kernels of the MoE layer: the expert sort from given ids
// (permutation and expert offsets), the weighted un-permute/combine, the
// backward's router gradient and token gather-sums, and the auxiliary loss.
//
// All of them are written so that every output is a fixed-order function of
// the inputs: no floating-point atomics, so results are bit-identical run to
// run.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace moe {

constexpr int kSortThreads = 256;                     // 8 warps
constexpr int kSortPerLane = 4;                       // slots per lane
constexpr int kSortChunk = kSortThreads * kSortPerLane;  // slots per block
constexpr int kPadRows = 128;      // per-expert row padding of the backward layout

// ---------------------------------------------------------------- router top-k helpers
// The router (route.cuh) takes the k experts of a token by k rounds of a
// warp-wide argmax under the order (logit descending, expert id ascending),
// each lane holding up to kRouterMaxPerLane experts (e = 32 i + lane).
constexpr int kRouterMaxPerLane = 8;  // E <= 256

// Order-preserving 32-bit key of a logit for the warp argmax (logit
// descending; an equal key goes to the lower expert id): a larger value gives
// a larger key and -0 ties with +0; NaN (outside the
// contract: logits are finite) gets 1, below every number; 0 marks a slot
// that is not a candidate (past E, or already taken).
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) return 1u;
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

constexpr int kMaxGroupsRouter = 256;  // E <= 256

// ---------------------------------------------------------------- expert sort
// Pass 1: per-block expert histogram of the slots s = t*k + j.
__global__ void sort_histogram_kernel(const int32_t* __restrict__ topk_idx, int S, int E,
                                      int32_t* __restrict__ block_counts, int* status) {
  __shared__ int hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  int ids[kSortPerLane];
  const int s0 = blockIdx.x * kSortChunk;
#pragma unroll
  for (int i = 0; i < kSortPerLane; ++i) {
    const int s = s0 + i * kSortThreads + threadIdx.x;
    ids[i] = s < S ? __ldg(topk_idx + s) : -2;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kSortPerLane; ++i) {
    const int e = ids[i];
    if (e == -2) continue;
    if (e < 0 || e >= E) { record_status(status, MOE_DEV_BAD_INDEX); continue; }
    atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) block_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// Pass 2: global offsets + stable scatter.  Warp w of block b owns the
// contiguous slots [b*C + w*C/8, b*C + (w+1)*C/8), held in registers, walked
// 32 at a time in order; lanes holding the same expert are ranked by lane id
// (match_any), so the sorted order within an expert is ascending slot id.
// Expert capacity cap > 0: a slot whose rank inside its expert is cap or more
// is dropped; it keeps its sorted row (perm_slot is the full sort) but its
// slot_perm entry is -1.
__global__ void sort_scatter_kernel(const int32_t* __restrict__ topk_idx, int S, int E,
                                    int num_blocks, const int32_t* __restrict__ block_counts,
                                    int32_t* __restrict__ expert_offsets,
                                    int32_t* __restrict__ perm_slot,
                                    int32_t* __restrict__ slot_perm, int cap) {
  __shared__ int base[256];
  __shared__ int total[256];
  __shared__ int wcount[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w0 = blockIdx.x * kSortChunk + warp * (kSortChunk / 8);
  int ids[kSortPerLane];
#pragma unroll
  for (int i = 0; i < kSortPerLane; ++i) {
    const int s = w0 + i * 32 + lane;
    int e = s < S ? __ldg(topk_idx + s) : -1;
    ids[i] = (e >= E || e < 0) ? -1 : e;
  }
  // expert totals and this block's start inside each expert
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int tot = 0, before = 0;
#pragma unroll 8
    for (int b = 0; b < num_blocks; ++b) {
      const int c = __ldg(block_counts + (size_t)b * E + e);
      before += (b < (int)blockIdx.x) ? c : 0;
      tot += c;
    }
    total[e] = tot;
    base[e] = before;
  }
  for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) (&wcount[0][0])[i] = 0;
  __syncthreads();
  // exclusive scan of the totals (one warp, E <= 256)
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 < E; b0 += 32) {
      const int e = b0 + lane;
      const int v = e < E ? total[e] : 0;
      int inc = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += x;
      }
      if (e < E) {
        const int off = run + inc - v;
        base[e] += off;
        total[e] = off;  // from here on: the expert's first sorted row
        if (blockIdx.x == 0) expert_offsets[e] = off;
      }
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (blockIdx.x == 0 && lane == 0) expert_offsets[E] = run;
  }
  // per-warp counts
#pragma unroll
  for (int i = 0; i < kSortPerLane; ++i) {
    const int e = ids[i];
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(m) - 1) wcount[warp][e] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  // warp bases: block base + counts of the earlier warps
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = base[e];
    for (int w = 0; w < 8; ++w) {
      const int c = wcount[w][e];
      wcount[w][e] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kSortPerLane; ++i) {
    const int e = ids[i];
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int pos = wcount[warp][e] + __popc(m & ((1u << lane) - 1u));
      const int s = w0 + i * 32 + lane;
      perm_slot[pos] = s;
      slot_perm[s] = (cap > 0 && pos - total[e] >= cap) ? -1 : pos;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) wcount[warp][e] += __popc(m);
    __syncwarp();
  }
}

// ---------------------------------------------------------------- combine
// out[t] = sum_j w[t,j] * y_perm[slot_perm[t*k+j]] (+ y_shared[t]); fp32 sum in
// j order, one bf16 rounding.  One warp per token; the k row indices and
// weights sit in registers so each lane has k independent 16-byte loads in
// flight per chunk.
template <int KMAX>
__global__ void combine_kernel(const __nv_bfloat16* __restrict__ y_perm,
                               const int32_t* __restrict__ slot_perm,
                               const float* __restrict__ topk_w,
                               const __nv_bfloat16* __restrict__ y_shared,
                               __nv_bfloat16* __restrict__ out, int T, int H, int k, int S) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int row_l = -1;  // -1: slot dropped by the expert capacity (no row, adds nothing)
  float w_l = 0.f;
  if (lane < k) {
    const int r = __ldg(slot_perm + (size_t)t * k + lane);
    row_l = r < 0 ? -1 : min(r, S - 1);
    w_l = r < 0 ? 0.f : __ldg(topk_w + (size_t)t * k + lane);
  }
  int rows[KMAX];
  float ws[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    rows[j] = __shfl_sync(0xffffffffu, row_l, j);
    ws[j] = __shfl_sync(0xffffffffu, w_l, j);
  }
  for (int c = lane; c < H / 8; c += 32) {
    uint4 v[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k)
        v[j] = rows[j] < 0 ? make_uint4(0u, 0u, 0u, 0u)
                           : ld_stream_v4(reinterpret_cast<const uint4*>(y_perm + (size_t)rows[j] * H) + c);
    uint4 vs = make_uint4(0, 0, 0, 0);
    if (y_shared) vs = __ldg(reinterpret_cast<const uint4*>(y_shared + (size_t)t * H) + c);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        const float w = ws[j];
        acc[0] = fmaf(w, bf16lo(v[j].x), acc[0]); acc[1] = fmaf(w, bf16hi(v[j].x), acc[1]);
        acc[2] = fmaf(w, bf16lo(v[j].y), acc[2]); acc[3] = fmaf(w, bf16hi(v[j].y), acc[3]);
        acc[4] = fmaf(w, bf16lo(v[j].z), acc[4]); acc[5] = fmaf(w, bf16hi(v[j].z), acc[5]);
        acc[6] = fmaf(w, bf16lo(v[j].w), acc[6]); acc[7] = fmaf(w, bf16hi(v[j].w), acc[7]);
      }
    }
    if (y_shared) {
      acc[0] += bf16lo(vs.x); acc[1] += bf16hi(vs.x); acc[2] += bf16lo(vs.y); acc[3] += bf16hi(vs.y);
      acc[4] += bf16lo(vs.z); acc[5] += bf16hi(vs.z); acc[6] += bf16lo(vs.w); acc[7] += bf16hi(vs.w);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]); o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]); o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + (size_t)t * H)[c] = o;
  }
}

// ---------------------------------------------------------------- backward helpers
// Padded per-expert layout: expert e's rows start at poff[e], a multiple of
// 128, and occupy ceil(n_e / 128) * 128 rows; the rows past its n_e tokens are
// zero in every sorted copy, so weight-gradient GEMMs can run whole 64-row
// k-blocks.

// Router backward fused with the per-token gradient gather, one warp per token.
// Router: dw_j = sum of the down-projection partials of slot j; the renormalised
// top-k weights are a softmax over the chosen logits, so
// dlogit_j = w_j (dw_j - sum_i w_i dw_i) (every other logit gets zero); dl is
// written per slot for the router weight gradient.
// dx[t] = sum_j dx_slot[p(t,j)] + sum_j dlogit_j W_r[e_j] (+ dx_shared[t]).
// With accumulate set, dx[t] already holds a term (the dense router term of the
// auxiliary loss) and the sum is added to it.
template <int KMAX>
__global__ void dx_gather_kernel(const __nv_bfloat16* __restrict__ dx_slot,
                                 const int32_t* __restrict__ topk_idx,
                                 const float* __restrict__ topk_w,
                                 const int32_t* __restrict__ slot_perm,
                                 const int32_t* __restrict__ expert_offsets,
                                 const int32_t* __restrict__ poff, const float* __restrict__ dw_part,
                                 int nNB, const __nv_bfloat16* __restrict__ w_router,
                                 const __nv_bfloat16* __restrict__ dx_shared,
                                 float* __restrict__ dl_out, __nv_bfloat16* __restrict__ dl_dense,
                                 int ldE, int router_term, int accumulate,
                                 __nv_bfloat16* __restrict__ dx, int T, int H, int k, int E, int P) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int row_l = -1, e_l = 0;  // row -1: slot dropped by the expert capacity (dw = 0, no dx)
  float dw_l = 0.f, w_l = 0.f;
  if (lane < k) {
    const int s = t * k + lane;
    e_l = clampi(__ldg(topk_idx + s), 0, E - 1);
    const int sp = __ldg(slot_perm + s);
    if (sp >= 0) {
      row_l = clampi(sp - __ldg(expert_offsets + e_l) + __ldg(poff + e_l), 0, P - 1);
      for (int b = 0; b < nNB; ++b) dw_l += __ldg(dw_part + (size_t)row_l * nNB + b);
    }
    w_l = __ldg(topk_w + s);
  }
  float dot = w_l * dw_l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  const float dl_l = w_l * (dw_l - dot);
  if (lane < k) dl_out[(size_t)t * k + lane] = dl_l;
  int rows[KMAX], es[KMAX];
  float dls[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    rows[j] = __shfl_sync(0xffffffffu, row_l, j);
    es[j] = __shfl_sync(0xffffffffu, e_l, j);
    dls[j] = __shfl_sync(0xffffffffu, dl_l, j);
  }
  if (dl_dense) {  // row t of the dense [T, ldE] logit gradient (zero off the selected experts)
    for (int e = lane; e < ldE; e += 32) {
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k && es[j] == e) v = dls[j];
      dl_dense[(size_t)t * ldE + e] = __float2bfloat16_rn(v);
    }
  }
  // slot rows in chunks of up to 8 (k <= 8: one chunk); per chunk, every slot's
  // gradient in j order, then every router term in j order; the shared expert
  // last.  Chunks keep k up to 32 within the register file.
  constexpr int CH = KMAX < 8 ? KMAX : 8;
  for (int c = lane; c < H / 8; c += 32) {
    uint4 vs = make_uint4(0, 0, 0, 0);
    if (dx_shared) vs = __ldg(reinterpret_cast<const uint4*>(dx_shared + (size_t)t * H) + c);
    const uint4 va = accumulate ? reinterpret_cast<const uint4*>(dx + (size_t)t * H)[c]
                                : make_uint4(0u, 0u, 0u, 0u);
    float acc[8] = {bf16lo(va.x), bf16hi(va.x), bf16lo(va.y), bf16hi(va.y),
                    bf16lo(va.z), bf16hi(va.z), bf16lo(va.w), bf16hi(va.w)};
#pragma unroll
    for (int j0 = 0; j0 < KMAX; j0 += CH) {
      if (j0 < k) {  // warp-uniform
        uint4 v[CH], r[CH];
#pragma unroll
        for (int jj = 0; jj < CH; ++jj) {
          const int j = j0 + jj;
          v[jj] = (j < k && rows[j] >= 0)
                      ? ld_stream_v4(reinterpret_cast<const uint4*>(dx_slot + (size_t)rows[j] * H) + c)
                      : make_uint4(0u, 0u, 0u, 0u);
          r[jj] = (j < k && router_term)
                      ? __ldg(reinterpret_cast<const uint4*>(w_router + (size_t)es[j] * H) + c)
                      : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int jj = 0; jj < CH; ++jj) {
          if (j0 + jj < k) {
            acc[0] += bf16lo(v[jj].x); acc[1] += bf16hi(v[jj].x); acc[2] += bf16lo(v[jj].y);
            acc[3] += bf16hi(v[jj].y); acc[4] += bf16lo(v[jj].z); acc[5] += bf16hi(v[jj].z);
            acc[6] += bf16lo(v[jj].w); acc[7] += bf16hi(v[jj].w);
          }
        }
#pragma unroll
        for (int jj = 0; jj < CH; ++jj) {
          if (j0 + jj < k) {
            const float d = dls[j0 + jj];
            acc[0] = fmaf(d, bf16lo(r[jj].x), acc[0]); acc[1] = fmaf(d, bf16hi(r[jj].x), acc[1]);
            acc[2] = fmaf(d, bf16lo(r[jj].y), acc[2]); acc[3] = fmaf(d, bf16hi(r[jj].y), acc[3]);
            acc[4] = fmaf(d, bf16lo(r[jj].z), acc[4]); acc[5] = fmaf(d, bf16hi(r[jj].z), acc[5]);
            acc[6] = fmaf(d, bf16lo(r[jj].w), acc[6]); acc[7] = fmaf(d, bf16hi(r[jj].w), acc[7]);
          }
        }
      }
    }
    if (dx_shared) {
      acc[0] += bf16lo(vs.x); acc[1] += bf16hi(vs.x); acc[2] += bf16lo(vs.y); acc[3] += bf16hi(vs.y);
      acc[4] += bf16lo(vs.z); acc[5] += bf16hi(vs.z); acc[6] += bf16lo(vs.w); acc[7] += bf16hi(vs.w);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]); o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]); o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(dx + (size_t)t * H)[c] = o;
  }
}

// Router weight gradient, second step.  The first is a split-K tensor-core
// GEMM dW_r = DL^T x over the tokens, where DL [T, E] is the logit gradient
// (zero off each token's selected experts: the renormalised top-k weights are
// a softmax over the selected logits) in bf16; it leaves one fp32 partial
// [E, H] per token split.  Here the splits are added in order and rounded to
// bf16 (thread = 4 consecutive elements of dW_r, up to 16 splits' loads in
// flight at once); the first E warps of the grid also form db[e] = sum of the
// fp32 dl over expert e's rows (sorted order, lane-strided partial sums, then a
// fixed butterfly; with the auxiliary loss the dense per-block partials).
__global__ void router_wgrad_reduce_kernel(const float* __restrict__ part, int nsplit, int E, int H,
                                           const int32_t* __restrict__ expert_offsets,
                                           const int32_t* __restrict__ perm_slot,
                                           const float* __restrict__ dl,
                                           const float* __restrict__ db_part, int db_nblk,
                                           __nv_bfloat16* __restrict__ dw_router,
                                           float* __restrict__ dbias) {
  const long long n4 = (long long)E * H / 4;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n4) {
    const float4* p = reinterpret_cast<const float4*>(part) + i;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g0 = 0; g0 < nsplit; g0 += 16) {
      float4 u[16];
#pragma unroll
      for (int g = 0; g < 16; ++g)
        if (g0 + g < nsplit) u[g] = __ldg(p + (size_t)(g0 + g) * n4);
#pragma unroll
      for (int g = 0; g < 16; ++g)
        if (g0 + g < nsplit) { o.x += u[g].x; o.y += u[g].y; o.z += u[g].z; o.w += u[g].w; }
    }
    uint2 w;
    w.x = pack_bf16x2(o.x, o.y);
    w.y = pack_bf16x2(o.z, o.w);
    reinterpret_cast<uint2*>(dw_router)[i] = w;
  }
  const int gw = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (dbias && gw < E) {
    // db[e]: the routed rows' dl or, with the auxiliary loss (dense logit
    // gradient), the per-block column sums of every token's
    const int e = gw;
    float b = 0.f;
    if (db_part) {
      for (int blk = lane; blk < db_nblk; blk += 32) b += __ldg(db_part + (size_t)blk * E + e);
    } else {
      const int r0 = __ldg(expert_offsets + e), r1 = __ldg(expert_offsets + e + 1);
      for (int r = r0 + lane; r < r1; r += 32) b += __ldg(dl + __ldg(perm_slot + r));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
    if (lane == 0) dbias[e] = b;
  }
}

// ---------------------------------------------------------------- auxiliary load-balancing loss
// Switch-Transformer form (the load-balancing auxiliary loss named on the
// pages): L_aux = alpha E sum_e f_e P_e with f_e = count_e / (T k) the fraction
// of slots routed to e and P_e = (1/T) sum_t p[t, e].  The counts pass no
// gradient, so dL_aux/dp[t, e] = c_e = alpha E f_e / T.

// prob_sum[e] = sum over the top-k kernel's blocks of their sums of p[t, e].
// Block = 32 experts (lane = expert, coalesced rows); warp w sums the partial
// rows w, w + 32, ... in order, then a fixed tree over the 32 warps.
constexpr int kProbSumWarps = 32;
__global__ void __launch_bounds__(32 * kProbSumWarps)
prob_sum_kernel(const float* __restrict__ psum_part, int nblk, int E, float* __restrict__ prob_sum) {
  __shared__ float part[kProbSumWarps][33];
  const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (e < E) {
#pragma unroll 4
    for (int b = wi; b < nblk; b += kProbSumWarps) s += __ldg(psum_part + (size_t)b * E + e);
  }
  part[wi][lane] = s;
  __syncthreads();
  for (int w = kProbSumWarps / 2; w > 0; w >>= 1) {
    if (wi < w) part[wi][lane] += part[wi + w][lane];
    __syncthreads();
  }
  if (wi == 0 && e < E) prob_sum[e] = part[0][lane];
}

// One block: coef[e] = alpha E f_e / T and loss = sum_e alpha E f_e prob_sum[e] / T
// (per-thread partial sums over e, then a fixed tree over the block).
constexpr int kAuxThreads = 256;
__global__ void aux_loss_kernel(const float* __restrict__ prob_sum,
                                const int32_t* __restrict__ expert_offsets, int T, int E, int k,
                                float alpha, float* __restrict__ loss, float* __restrict__ coef) {
  __shared__ float part[kAuxThreads];
  float acc = 0.f;
  for (int e = threadIdx.x; e < E; e += kAuxThreads) {
    const float f = (float)(__ldg(expert_offsets + e + 1) - __ldg(expert_offsets + e)) /
                    ((float)T * (float)k);
    const float c = alpha * (float)E * f / (float)T;
    if (coef) coef[e] = c;
    acc += c * __ldg(prob_sum + e);
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = kAuxThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0 && loss) *loss = part[0];
}

// The dense logit gradient with the auxiliary loss, one warp per token:
//   p = softmax(logits[t]); s = sum_e c_e p_e;
//   DL[t, e] = dl_main[t, e] + p_e (c_e - s)
// where dl_main is the top-k weights' gradient on the token's selected experts
// and zero elsewhere: dl_j = w_j (dw_j - sum_i w_i dw_i), dw_j the sum of slot
// j's down-projection partials (the same arithmetic as the per-token gather,
// which is why the router term of grad_x can be formed before that gather);
// dl is written per slot (fp32), DL once in bf16 ([T, ldE], zero padding), and
// each block (8 tokens) writes its fp32 column sums (warp order) for the bias
// gradient.
constexpr int kAuxDlWarps = 8;
template <int KMAX>
__global__ void aux_dl_kernel(const float* __restrict__ logits, const float* __restrict__ coef,
                              const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                              const int32_t* __restrict__ slot_perm,
                              const int32_t* __restrict__ expert_offsets,
                              const int32_t* __restrict__ poff, const float* __restrict__ dw_part,
                              int nNB, int P, float* __restrict__ dl_out, int T, int E, int k,
                              int ldE, __nv_bfloat16* __restrict__ dl_dense,
                              float* __restrict__ db_part) {
  __shared__ float rows[kAuxDlWarps][kMaxGroupsRouter];
  const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAuxDlWarps + wi;
  float lv[kRouterMaxPerLane];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kRouterMaxPerLane; ++i) {
    const int e = i * 32 + lane;
    lv[i] = (t < T && e < E) ? __ldg(logits + (size_t)t * E + e) : -INFINITY;
    mx = fmaxf(mx, lv[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < kRouterMaxPerLane; ++i) {
    lv[i] = (t < T && i * 32 + lane < E) ? expf(lv[i] - mx) : 0.f;
    z += lv[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kRouterMaxPerLane; ++i) {
    const int e = i * 32 + lane;
    lv[i] = t < T ? lv[i] / z : 0.f;
    if (e < E) s += __ldg(coef + e) * lv[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  int sel_e = -1;
  float dw_l = 0.f, w_l = 0.f;
  if (t < T && lane < k) {
    const int sl = t * k + lane;
    sel_e = clampi(__ldg(topk_idx + sl), 0, E - 1);
    const int sp = __ldg(slot_perm + sl);  // -1: dropped by the expert capacity, dw = 0
    if (sp >= 0) {
      const int row = clampi(sp - __ldg(expert_offsets + sel_e) + __ldg(poff + sel_e), 0, P - 1);
      for (int b = 0; b < nNB; ++b) dw_l += __ldg(dw_part + (size_t)row * nNB + b);
    }
    w_l = __ldg(topk_w + sl);
  }
  float dot = w_l * dw_l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  const float sel_d = w_l * (dw_l - dot);
  if (t < T && lane < k) dl_out[(size_t)t * k + lane] = sel_d;
  int es[KMAX];
  float ds[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    es[j] = __shfl_sync(0xffffffffu, sel_e, j);
    ds[j] = __shfl_sync(0xffffffffu, sel_d, j);
  }
#pragma unroll
  for (int i = 0; i < kRouterMaxPerLane; ++i) {
    if (i * 32 >= ldE) break;  // warp-uniform
    const int e = i * 32 + lane;
    float main_d = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k && es[j] == e) main_d = ds[j];
    const float v = (e < E && t < T) ? main_d + lv[i] * (__ldg(coef + (e < E ? e : 0)) - s) : 0.f;
    if (e < E) rows[wi][e] = v;
    if (t < T && e < ldE) dl_dense[(size_t)t * ldE + e] = __float2bfloat16_rn(v);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kAuxDlWarps; ++w) acc += rows[w][e];
    db_part[(size_t)blockIdx.x * E + e] = acc;
  }
}

}  // namespace moe
