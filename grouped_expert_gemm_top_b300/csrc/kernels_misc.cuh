// Memory-bound kernels of the MoE layer: the router's softmax/top-k, the
// expert sort (permutation and expert offsets), the sorted token copies, the
// weighted un-permute/combine, and the small backward kernels (padded row
// tables, router gradient, token gather-sums).
//
// All of them are written so that every output is a fixed-order function of
// the inputs: no floating-point atomics, so results are bit-identical run to
// run.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace moe {

constexpr int kSortChunk = 2048;   // slots per block in the expert sort
constexpr int kSortThreads = 256;  // 8 warps x 256 slots
constexpr int kPadRows = 128;      // per-expert row padding of the backward layout

// ---------------------------------------------------------------- router top-k
// One warp per token.  logits[e] = sum of the split-K partial products (in
// split order) + bias[e]; p = softmax over all E; the k experts are taken by k
// rounds of a warp-wide argmax under the order (logit descending, expert id
// ascending); w_j = p[e_j] / sum_j p[e_j].  The balanced gate takes
// e_j = (t*k + j) mod E instead of the argmax rounds.  Reductions use a fixed
// butterfly order, so results are bit-identical run to run.
constexpr int kRouterMaxPerLane = 8;  // E <= 256

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
      float l = 0.f;
      for (int sp = 0; sp < splits; ++sp) l += __ldg(partial + ((size_t)sp * T + t) * E + e);
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

// ---------------------------------------------------------------- sorted token copies
// x_sorted[r, :] = x[perm_slot[r] / k, :] for the S sorted rows (one warp per row).
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                   const int32_t* __restrict__ perm_slot, int k, int S, int H,
                                   int T, __nv_bfloat16* __restrict__ x_sorted) {
  const long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= S) return;
  const int t = clampi(__ldg(perm_slot + r) / k, 0, T - 1);
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(x_sorted + (size_t)r * H);
  for (int c = lane; c < H / 8; c += 32) dst[c] = __ldg(src + c);
}

// Backward copies in the padded per-expert layout: for padded row p with token
// row_tok[p] (-1 = padding), a_sorted[p] = a[token] and b_sorted[p] = b[token],
// padding rows are zero.  Rows at or past poff[E] are not touched.
__global__ void gather_rows_padded_kernel(const int32_t* __restrict__ row_tok,
                                          const int32_t* __restrict__ poff, int E, int P, int H,
                                          int T, const __nv_bfloat16* __restrict__ a,
                                          __nv_bfloat16* __restrict__ a_sorted,
                                          const __nv_bfloat16* __restrict__ b,
                                          __nv_bfloat16* __restrict__ b_sorted) {
  const long long p = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (p >= P || p >= __ldg(poff + E)) return;
  const int tok = __ldg(row_tok + p);
  uint4* da = reinterpret_cast<uint4*>(a_sorted + (size_t)p * H);
  uint4* db = reinterpret_cast<uint4*>(b_sorted + (size_t)p * H);
  if (tok < 0 || tok >= T) {
    for (int c = lane; c < H / 8; c += 32) {
      da[c] = make_uint4(0, 0, 0, 0);
      db[c] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const uint4* sa = reinterpret_cast<const uint4*>(a + (size_t)tok * H);
  const uint4* sb = reinterpret_cast<const uint4*>(b + (size_t)tok * H);
  for (int c = lane; c < H / 8; c += 32) {
    da[c] = __ldg(sa + c);
    db[c] = __ldg(sb + c);
  }
}

// ---------------------------------------------------------------- expert sort
// Pass 1: per-block expert histogram of the slots s = t*k + j.
__global__ void sort_histogram_kernel(const int32_t* __restrict__ topk_idx, int S, int E,
                                      int32_t* __restrict__ block_counts, int* status) {
  __shared__ int hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int s0 = blockIdx.x * kSortChunk;
  const int s1 = min(S, s0 + kSortChunk);
  for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
    const int e = __ldg(topk_idx + s);
    if (e < 0 || e >= E) { record_status(status, MOE_DEV_BAD_INDEX); continue; }
    atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) block_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// Pass 2: global offsets + stable scatter.  Each warp walks its 256 slots in
// order, 32 at a time; lanes holding the same expert are ranked by lane id
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
  // expert totals and this block's start inside each expert
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int tot = 0, before = 0;
    for (int b = 0; b < num_blocks; ++b) {
      const int c = __ldg(block_counts + (size_t)b * E + e);
      if (b < (int)blockIdx.x) before += c;
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
  const int w0 = blockIdx.x * kSortChunk + warp * (kSortChunk / 8);
  const int w1 = min(S, w0 + kSortChunk / 8);
  for (int g = w0; g < w1; g += 32) {
    const int s = g + lane;
    int e = (s < w1) ? __ldg(topk_idx + s) : -1;
    if (e >= E) e = -1;
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
  for (int g = w0; g < w1; g += 32) {
    const int s = g + lane;
    int e = (s < w1) ? __ldg(topk_idx + s) : -1;
    if (e >= E) e = -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int rank = __popc(m & ((1u << lane) - 1u));
      const int pos = wcount[warp][e] + rank;
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
// j order, one bf16 rounding.  One warp per token, 16-byte loads.
__global__ void combine_kernel(const __nv_bfloat16* __restrict__ y_perm,
                               const int32_t* __restrict__ slot_perm,
                               const float* __restrict__ topk_w,
                               const __nv_bfloat16* __restrict__ y_shared,
                               __nv_bfloat16* __restrict__ out, int T, int H, int k, int S) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const int t = warp;
  int row_l = 0;
  float w_l = 0.f;
  if (lane < k) {
    row_l = clampi(__ldg(slot_perm + (size_t)t * k + lane), 0, S - 1);
    w_l = __ldg(topk_w + (size_t)t * k + lane);
  }
  const int nchunk = H / 8;
  for (int c = lane; c < nchunk; c += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, row_l, j);
      const float w = __shfl_sync(0xffffffffu, w_l, j);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(y_perm + (size_t)row * H) + c);
      acc[0] = fmaf(w, bf16lo(v.x), acc[0]); acc[1] = fmaf(w, bf16hi(v.x), acc[1]);
      acc[2] = fmaf(w, bf16lo(v.y), acc[2]); acc[3] = fmaf(w, bf16hi(v.y), acc[3]);
      acc[4] = fmaf(w, bf16lo(v.z), acc[4]); acc[5] = fmaf(w, bf16hi(v.z), acc[5]);
      acc[6] = fmaf(w, bf16lo(v.w), acc[6]); acc[7] = fmaf(w, bf16hi(v.w), acc[7]);
    }
    if (y_shared) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(y_shared + (size_t)t * H) + c);
      acc[0] += bf16lo(v.x); acc[1] += bf16hi(v.x); acc[2] += bf16lo(v.y); acc[3] += bf16hi(v.y);
      acc[4] += bf16lo(v.z); acc[5] += bf16hi(v.z); acc[6] += bf16lo(v.w); acc[7] += bf16hi(v.w);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]); o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]); o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + (size_t)t * H)[c] = o;
  }
}

// ---------------------------------------------------------------- backward helpers
// Padded offsets: every expert's rows start on a 128-row boundary.
__global__ void pad_offsets_kernel(const int32_t* __restrict__ expert_offsets, int E,
                                   int32_t* __restrict__ poff) {
  const int lane = threadIdx.x;
  int run = 0;
  for (int b0 = 0; b0 < E; b0 += 32) {
    const int e = b0 + lane;
    int v = 0;
    if (e < E) {
      const int n = __ldg(expert_offsets + e + 1) - __ldg(expert_offsets + e);
      v = ((n + kPadRows - 1) / kPadRows) * kPadRows;
    }
    int inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += x;
    }
    if (e < E) poff[e] = run + inc - v;
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) poff[E] = run;
}

// For every row p of the padded layout: the token it reads (-1 for padding rows).
__global__ void padded_row_tokens_kernel(const int32_t* __restrict__ expert_offsets,
                                         const int32_t* __restrict__ poff,
                                         const int32_t* __restrict__ perm_slot, int E, int k,
                                         int S_pad_max, int32_t* __restrict__ row_tok) {
  __shared__ int sp[257];
  __shared__ int so[257];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    sp[e] = poff[e];
    so[e] = expert_offsets[e];
  }
  __syncthreads();
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= S_pad_max) return;
  int tok = -1;
  if (p < sp[E]) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sp[mid] <= p) lo = mid; else hi = mid - 1;
    }
    const int i = p - sp[lo];
    if (i < so[lo + 1] - so[lo]) tok = __ldg(perm_slot + so[lo] + i) / k;
  }
  row_tok[p] = tok;
}

// Router backward, one thread per token.  dw[j] = sum of the down-projection
// partials; the renormalised top-k weights are a softmax over the chosen
// logits, so dlogit[j] = w_j (dw_j - sum_i w_i dw_i) and every other logit
// gets zero.  Output dl per slot (fp32).
__global__ void router_backward_kernel(const int32_t* __restrict__ topk_idx,
                                       const float* __restrict__ topk_w,
                                       const int32_t* __restrict__ slot_perm,
                                       const int32_t* __restrict__ expert_offsets,
                                       const int32_t* __restrict__ poff,
                                       const float* __restrict__ dw_part, int nNB, int T, int k,
                                       int E, int P, float* __restrict__ dl) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float dw[32], w[32];
  float dot = 0.f;
  for (int j = 0; j < k; ++j) {
    const int s = t * k + j;
    const int e = clampi(__ldg(topk_idx + s), 0, E - 1);
    const int p = clampi(__ldg(slot_perm + s) - __ldg(expert_offsets + e) + __ldg(poff + e), 0, P - 1);
    float sum = 0.f;
    for (int b = 0; b < nNB; ++b) sum += __ldg(dw_part + (size_t)p * nNB + b);
    dw[j] = sum;
    w[j] = __ldg(topk_w + s);
    dot = fmaf(w[j], sum, dot);
  }
  for (int j = 0; j < k; ++j) dl[(size_t)t * k + j] = w[j] * (dw[j] - dot);
}

// dx[t] = sum_j dx_slot[p(t,j)] + sum_j dl[t,j] W_r[e_j] (+ dx_shared[t]).  One warp per token.
__global__ void dx_gather_kernel(const __nv_bfloat16* __restrict__ dx_slot,
                                 const int32_t* __restrict__ topk_idx,
                                 const int32_t* __restrict__ slot_perm,
                                 const int32_t* __restrict__ expert_offsets,
                                 const int32_t* __restrict__ poff, const float* __restrict__ dl,
                                 const __nv_bfloat16* __restrict__ w_router,
                                 const __nv_bfloat16* __restrict__ dx_shared,
                                 __nv_bfloat16* __restrict__ dx, int T, int H, int k, int E,
                                 int P) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const int t = warp;
  int row_l = 0, e_l = 0;
  float dl_l = 0.f;
  if (lane < k) {
    const int s = t * k + lane;
    e_l = clampi(__ldg(topk_idx + s), 0, E - 1);
    row_l = clampi(__ldg(slot_perm + s) - __ldg(expert_offsets + e_l) + __ldg(poff + e_l), 0, P - 1);
    dl_l = __ldg(dl + s);
  }
  for (int c = lane; c < H / 8; c += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, row_l, j);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(dx_slot + (size_t)row * H) + c);
      acc[0] += bf16lo(v.x); acc[1] += bf16hi(v.x); acc[2] += bf16lo(v.y); acc[3] += bf16hi(v.y);
      acc[4] += bf16lo(v.z); acc[5] += bf16hi(v.z); acc[6] += bf16lo(v.w); acc[7] += bf16hi(v.w);
    }
    for (int j = 0; j < k; ++j) {
      const int e = __shfl_sync(0xffffffffu, e_l, j);
      const float d = __shfl_sync(0xffffffffu, dl_l, j);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(w_router + (size_t)e * H) + c);
      acc[0] = fmaf(d, bf16lo(v.x), acc[0]); acc[1] = fmaf(d, bf16hi(v.x), acc[1]);
      acc[2] = fmaf(d, bf16lo(v.y), acc[2]); acc[3] = fmaf(d, bf16hi(v.y), acc[3]);
      acc[4] = fmaf(d, bf16lo(v.z), acc[4]); acc[5] = fmaf(d, bf16hi(v.z), acc[5]);
      acc[6] = fmaf(d, bf16lo(v.w), acc[6]); acc[7] = fmaf(d, bf16hi(v.w), acc[7]);
    }
    if (dx_shared) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(dx_shared + (size_t)t * H) + c);
      acc[0] += bf16lo(v.x); acc[1] += bf16hi(v.x); acc[2] += bf16lo(v.y); acc[3] += bf16hi(v.y);
      acc[4] += bf16lo(v.z); acc[5] += bf16hi(v.z); acc[6] += bf16lo(v.w); acc[7] += bf16hi(v.w);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]); o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]); o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(dx + (size_t)t * H)[c] = o;
  }
}

// dW_r[e, :] = sum over the rows of expert e (sorted order) of dl[slot] * x[token, :];
// db[e] = sum of those dl.  Block = (expert, 256-column chunk), 4 warps split the
// rows round-robin and their partials are added in warp order.
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
  const int r0 = __ldg(expert_offsets + e), r1 = __ldg(expert_offsets + e + 1);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  float bsum = 0.f;
  for (int r = r0 + warp; r < r1; r += 4) {
    const int s = __ldg(perm_slot + r);
    const float d = __ldg(dl + s);
    bsum += d;
    if (c0 < H) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(s / k) * H + c0));
      acc[0] = fmaf(d, bf16lo(v.x), acc[0]); acc[1] = fmaf(d, bf16hi(v.x), acc[1]);
      acc[2] = fmaf(d, bf16lo(v.y), acc[2]); acc[3] = fmaf(d, bf16hi(v.y), acc[3]);
      acc[4] = fmaf(d, bf16lo(v.z), acc[4]); acc[5] = fmaf(d, bf16hi(v.z), acc[5]);
      acc[6] = fmaf(d, bf16lo(v.w), acc[6]); acc[7] = fmaf(d, bf16hi(v.w), acc[7]);
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
    if (c0 < H) {
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
