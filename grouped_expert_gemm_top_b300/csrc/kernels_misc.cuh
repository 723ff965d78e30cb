// Memory-bound kernels of the MoE layer: the router's softmax/top-k, the
// expert sort (permutation and expert offsets), the weighted
// un-permute/combine, and the backward's router gradient and token
// gather-sums.
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

// ---------------------------------------------------------------- router top-k
// One warp per token.  logits[e] = sum of the split-K partial products (in
// split order) + bias[e]; p = softmax over all E; the k experts are taken by k
// rounds of a warp-wide argmax under the order (logit descending, expert id
// ascending); w_j = p[e_j] / sum_j p[e_j].  The balanced gate takes
// e_j = (t*k + j) mod E instead of the argmax rounds.  Reductions use a fixed
// butterfly order, so results are bit-identical run to run.
constexpr int kRouterMaxPerLane = 8;  // E <= 256
constexpr int kMaxSplitsRouter = 8;   // split-K slices of the router GEMM

__device__ __forceinline__ bool topk_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__global__ void router_topk_kernel(const float* __restrict__ partial, int splits,
                                   const float* __restrict__ bias, float* __restrict__ logits_out,
                                   int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                   int T, int E, int k, int gate_mode) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float v[kRouterMaxPerLane];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kRouterMaxPerLane; ++i) {
    const int e = i * 32 + lane;
    v[i] = -INFINITY;
    if (e < E) {
      float part[kMaxSplitsRouter];
#pragma unroll
      for (int sp = 0; sp < kMaxSplitsRouter; ++sp)
        part[sp] = sp < splits ? __ldg(partial + ((size_t)sp * T + t) * E + e) : 0.f;
      float l = 0.f;
#pragma unroll
      for (int sp = 0; sp < kMaxSplitsRouter; ++sp)
        if (sp < splits) l += part[sp];
      if (bias) l += __ldg(bias + e);
      v[i] = l;
      mx = fmaxf(mx, l);
      if (logits_out) logits_out[(size_t)t * E + e] = l;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < kRouterMaxPerLane; ++i)
    if (i * 32 + lane < E) z += expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  uint32_t taken = 0;
  int my_e = 0;
  float my_p = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv;
    int bi;
    if (gate_mode == 1) {
      bi = (int)(((long long)t * k + j) % E);
      float mine = 0.f;
#pragma unroll
      for (int i = 0; i < kRouterMaxPerLane; ++i)
        if (i == (bi >> 5)) mine = v[i];
      bv = __shfl_sync(0xffffffffu, mine, bi & 31);
    } else {
      bv = -INFINITY;
      bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kRouterMaxPerLane; ++i) {
        const int e = i * 32 + lane;
        if (e < E && !((taken >> i) & 1u) && topk_before(v[i], e, bv, bi)) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (topk_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (bi == 0x7fffffff) bi = j;  // only with NaN logits: stay in range
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    const float p = expf(bv - mx) / z;
    if (lane == j) { my_e = bi; my_p = p; }
  }
  float psum = lane < k ? my_p : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = my_e;
    topk_w[(size_t)t * k + lane] = my_p / psum;
  }
}

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
__global__ void sort_scatter_kernel(const int32_t* __restrict__ topk_idx, int S, int E,
                                    int num_blocks, const int32_t* __restrict__ block_counts,
                                    int32_t* __restrict__ expert_offsets,
                                    int32_t* __restrict__ perm_slot,
                                    int32_t* __restrict__ slot_perm) {
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
      slot_perm[s] = pos;
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
  int row_l = 0;
  float w_l = 0.f;
  if (lane < k) {
    row_l = clampi(__ldg(slot_perm + (size_t)t * k + lane), 0, S - 1);
    w_l = __ldg(topk_w + (size_t)t * k + lane);
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
      if (j < k) v[j] = __ldg(reinterpret_cast<const uint4*>(y_perm + (size_t)rows[j] * H) + c);
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

// Padded sorted copy of the tokens for the gate/up weight gradient: row p of
// expert e's padded block [poff[e], poff[e+1]) holds x[token of sorted row
// offsets[e] + (p - poff[e])], or zeros past the expert's tokens.  One warp
// per row, grid-stride; rows at or past poff[E] are not touched.
__global__ void sorted_rows_padded_kernel(const int32_t* __restrict__ poff,
                                          const int32_t* __restrict__ expert_offsets,
                                          const int32_t* __restrict__ perm_slot, int E, int k,
                                          int H, int T, const __nv_bfloat16* __restrict__ x,
                                          __nv_bfloat16* __restrict__ x_sorted) {
  __shared__ int sp[257];
  __shared__ int so[257];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    sp[e] = __ldg(poff + e);
    so[e] = __ldg(expert_offsets + e);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long p = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < sp[E];
       p += nwarps) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sp[mid] <= p) lo = mid; else hi = mid - 1;
    }
    const int i = (int)(p - sp[lo]);
    uint4* dst = reinterpret_cast<uint4*>(x_sorted + (size_t)p * H);
    if (i < so[lo + 1] - so[lo]) {
      const int tok = clampi(__ldg(perm_slot + so[lo] + i) / k, 0, T - 1);
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)tok * H);
      for (int c = lane; c < H / 8; c += 32) dst[c] = __ldg(src + c);
    } else {
      for (int c = lane; c < H / 8; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

// Router backward fused with the per-token gradient gather, one warp per token.
// Router: dw_j = sum of the down-projection partials of slot j; the renormalised
// top-k weights are a softmax over the chosen logits, so
// dlogit_j = w_j (dw_j - sum_i w_i dw_i) (every other logit gets zero); dl is
// written per slot for the router weight gradient.
// dx[t] = sum_j dx_slot[p(t,j)] + sum_j dlogit_j W_r[e_j] (+ dx_shared[t]).
template <int KMAX>
__global__ void dx_gather_kernel(const __nv_bfloat16* __restrict__ dx_slot,
                                 const int32_t* __restrict__ topk_idx,
                                 const float* __restrict__ topk_w,
                                 const int32_t* __restrict__ slot_perm,
                                 const int32_t* __restrict__ expert_offsets,
                                 const int32_t* __restrict__ poff, const float* __restrict__ dw_part,
                                 int nNB, const __nv_bfloat16* __restrict__ w_router,
                                 const __nv_bfloat16* __restrict__ dx_shared,
                                 float* __restrict__ dl_out, __nv_bfloat16* __restrict__ dx, int T,
                                 int H, int k, int E, int P) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int row_l = 0, e_l = 0;
  float dw_l = 0.f, w_l = 0.f;
  if (lane < k) {
    const int s = t * k + lane;
    e_l = clampi(__ldg(topk_idx + s), 0, E - 1);
    row_l = clampi(__ldg(slot_perm + s) - __ldg(expert_offsets + e_l) + __ldg(poff + e_l), 0, P - 1);
    for (int b = 0; b < nNB; ++b) dw_l += __ldg(dw_part + (size_t)row_l * nNB + b);
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
  for (int c = lane; c < H / 8; c += 32) {
    uint4 v[KMAX], r[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        v[j] = __ldg(reinterpret_cast<const uint4*>(dx_slot + (size_t)rows[j] * H) + c);
        r[j] = __ldg(reinterpret_cast<const uint4*>(w_router + (size_t)es[j] * H) + c);
      }
    }
    uint4 vs = make_uint4(0, 0, 0, 0);
    if (dx_shared) vs = __ldg(reinterpret_cast<const uint4*>(dx_shared + (size_t)t * H) + c);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        acc[0] += bf16lo(v[j].x); acc[1] += bf16hi(v[j].x); acc[2] += bf16lo(v[j].y);
        acc[3] += bf16hi(v[j].y); acc[4] += bf16lo(v[j].z); acc[5] += bf16hi(v[j].z);
        acc[6] += bf16lo(v[j].w); acc[7] += bf16hi(v[j].w);
      }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        const float d = dls[j];
        acc[0] = fmaf(d, bf16lo(r[j].x), acc[0]); acc[1] = fmaf(d, bf16hi(r[j].x), acc[1]);
        acc[2] = fmaf(d, bf16lo(r[j].y), acc[2]); acc[3] = fmaf(d, bf16hi(r[j].y), acc[3]);
        acc[4] = fmaf(d, bf16lo(r[j].z), acc[4]); acc[5] = fmaf(d, bf16hi(r[j].z), acc[5]);
        acc[6] = fmaf(d, bf16lo(r[j].w), acc[6]); acc[7] = fmaf(d, bf16hi(r[j].w), acc[7]);
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

// dW_r[e, :] = sum over the rows of expert e (sorted order) of dl[slot] * x[token, :];
// db[e] = sum of those dl.  Block = (expert, 256-column chunk); the expert's
// rows are taken 32 at a time (lane j loads row j's slot and dl), 4 warps take
// every 4th batch, and the 4 partials are added in warp order.
__global__ void router_wgrad_kernel(const __nv_bfloat16* __restrict__ x,
                                    const int32_t* __restrict__ expert_offsets,
                                    const int32_t* __restrict__ perm_slot,
                                    const float* __restrict__ dl, int H, int k,
                                    __nv_bfloat16* __restrict__ dw_router,
                                    float* __restrict__ dbias) {
  __shared__ float part[4][256];
  __shared__ float bpart[4];
  const int e = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 256 + lane * 8;  // 8 columns per lane
  const bool col_ok = c0 < H;
  const int r0 = __ldg(expert_offsets + e), r1 = __ldg(expert_offsets + e + 1);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  float bsum = 0.f;
  for (int rb = r0 + warp * 32; rb < r1; rb += 4 * 32) {
    int tok_l = 0;
    float d_l = 0.f;
    if (rb + lane < r1) {
      const int s = __ldg(perm_slot + rb + lane);
      tok_l = s / k;
      d_l = __ldg(dl + s);
    }
    const int nb = min(32, r1 - rb);
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
      const int tok = __shfl_sync(0xffffffffu, tok_l, j);
      const float d = __shfl_sync(0xffffffffu, d_l, j);
      if (j < nb) {
        bsum += d;
        if (col_ok) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * H + c0));
          acc[0] = fmaf(d, bf16lo(v.x), acc[0]); acc[1] = fmaf(d, bf16hi(v.x), acc[1]);
          acc[2] = fmaf(d, bf16lo(v.y), acc[2]); acc[3] = fmaf(d, bf16hi(v.y), acc[3]);
          acc[4] = fmaf(d, bf16lo(v.z), acc[4]); acc[5] = fmaf(d, bf16hi(v.z), acc[5]);
          acc[6] = fmaf(d, bf16lo(v.w), acc[6]); acc[7] = fmaf(d, bf16hi(v.w), acc[7]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[warp][lane * 8 + i] = acc[i];
  if (lane == 0) bpart[warp] = bsum;
  __syncthreads();
  if (warp == 0) {
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      o[i] = ((part[0][lane * 8 + i] + part[1][lane * 8 + i]) + part[2][lane * 8 + i]) +
             part[3][lane * 8 + i];
    if (col_ok) {
      uint4 v;
      v.x = pack_bf16x2(o[0], o[1]); v.y = pack_bf16x2(o[2], o[3]);
      v.z = pack_bf16x2(o[4], o[5]); v.w = pack_bf16x2(o[6], o[7]);
      *reinterpret_cast<uint4*>(dw_router + (size_t)e * H + c0) = v;
    }
    if (dbias && blockIdx.x == 0 && lane == 0)
      dbias[e] = ((bpart[0] + bpart[1]) + bpart[2]) + bpart[3];
  }
}

}  // namespace moe
