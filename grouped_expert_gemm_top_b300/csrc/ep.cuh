// Expert-parallel dispatch / combine helpers (NeMo AutoModel blog, "专家并行与
// DeepEP": every rank holds 1/ep of the experts, split along the expert
// dimension, and trains on its own tokens; DeepEP dispatches the tokens to the
// experts' ranks and combines the results back).
//
// The exchange itself is the caller's collective (all-to-all over a process
// group).  These kernels lay the data out around it:
//   gather_rows_kernel      dst[i] = src[idx[i] / div]: a source's token rows in
//                           its expert-sorted order (the send buffer, rank-major
//                           because every rank's experts are contiguous), or
//                           the expert outputs put back in receive order.
//   ep_recv_layout_kernel   the receiving rank's grouping: its buffer holds the
//                           sources' blocks in source order, each in expert
//                           order; the one grouped GEMM over its local experts
//                           takes the rows expert by expert, within an expert
//                           source by source (so the rows of an expert are in
//                           global slot order, as on one rank).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace moe {

// One warp per row, 16-byte copies (H a multiple of 8).  Row indices outside
// [0, src_rows) are recorded as MOE_DEV_BAD_INDEX and give a zero row.
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ src, long long src_rows, int H,
                                   const int32_t* __restrict__ idx, int n, int div,
                                   __nv_bfloat16* __restrict__ dst, int* status) {
  const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= n) return;
  const long long r = (long long)__ldg(idx + i) / div;
  const bool ok = r >= 0 && r < src_rows;
  if (!ok && lane == 0) record_status(status, MOE_DEV_BAD_INDEX);
  const uint4* s = reinterpret_cast<const uint4*>(src + (ok ? r : 0) * (long long)H);
  uint4* d = reinterpret_cast<uint4*>(dst + i * (long long)H);
  for (int c = lane; c < H / 8; c += 32) d[c] = ok ? __ldg(s + c) : make_uint4(0u, 0u, 0u, 0u);
}

// dst[i] = src[idx[i] / div] for 4-byte elements (a source's routing weights
// in its sorted order).  Indices outside [0, src_n) give 0 and MOE_DEV_BAD_INDEX.
__global__ void gather_scalars_kernel(const uint32_t* __restrict__ src, long long src_n,
                                      const int32_t* __restrict__ idx, int n, int div,
                                      uint32_t* __restrict__ dst, int* status) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const long long r = (long long)__ldg(idx + i) / div;
  const bool ok = r >= 0 && r < src_n;
  if (!ok) record_status(status, MOE_DEV_BAD_INDEX);
  dst[i] = ok ? __ldg(src + r) : 0u;
}

// The expert side of the expert-parallel backward hands its results back in
// receive order: received row i sits at grouped row g = slot_perm[i] of local
// expert e (offsets[e] <= g < offsets[e+1]), i.e. at row poff[e] + g -
// offsets[e] of the padded row space the backward GEMMs use.  A warp per row
// copies that row of the per-slot dx and sums its dw partials in column-part
// order (the order the one-GPU router backward sums them in).
__global__ void ep_rows_out_kernel(const __nv_bfloat16* __restrict__ dxs,
                                   const float* __restrict__ dwp, int nDW,
                                   const int32_t* __restrict__ poff,
                                   const int32_t* __restrict__ offsets, int E,
                                   const int32_t* __restrict__ slot_perm, int R, int H,
                                   long long P, __nv_bfloat16* __restrict__ dx_rows,
                                   float* __restrict__ dw_rows, int* status) {
  const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= R) return;
  long long p = -1;
  if (lane == 0) {
    const int g = __ldg(slot_perm + i);
    if (g >= 0 && g < __ldg(offsets + E)) {
      int lo = 0, hi = E - 1;  // the last expert whose first row is <= g
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(offsets + mid) <= g) lo = mid; else hi = mid - 1;
      }
      p = (long long)__ldg(poff + lo) + g - __ldg(offsets + lo);
      if (p >= P) p = -1;
    }
    if (p < 0) record_status(status, MOE_DEV_BAD_INDEX);
  }
  p = __shfl_sync(0xffffffffu, p, 0);
  const uint4* s = reinterpret_cast<const uint4*>(dxs + (p < 0 ? 0 : p) * (long long)H);
  uint4* d = reinterpret_cast<uint4*>(dx_rows + i * (long long)H);
  for (int c = lane; c < H / 8; c += 32) d[c] = p < 0 ? make_uint4(0u, 0u, 0u, 0u) : ld_stream_v4(s + c);
  if (lane == 0) {
    float dw = 0.f;
    if (p >= 0)
      for (int b = 0; b < nDW; ++b) dw += __ldg(dwp + p * nDW + b);
    dw_rows[i] = dw;
  }
}

constexpr int kEpLayoutThreads = 256;
constexpr int kEpMaxCells = 4096;     // sources x local experts
constexpr int kEpMaxLocalExperts = 256;

// counts [n_src][E_loc]: rows source s sends for local expert e.  Every block
// forms, in shared memory, the receive start seg[s][e] (source-major prefix)
// and the grouped start grp[s][e] = local_offsets[e] + rows of expert e from
// earlier sources; then each thread places receive rows r (grid-stride):
// (s, e) = the last cell whose receive start is <= r, g = grp + (r - seg);
// recv_perm[g] = r, recv_inv[r] = g.  Block 0 writes local_offsets [E_loc+1].
__global__ void __launch_bounds__(kEpLayoutThreads)
    ep_recv_layout_kernel(const int32_t* __restrict__ counts, int n_src, int E_loc, int R,
                          int32_t* __restrict__ local_offsets, int32_t* __restrict__ recv_perm,
                          int32_t* __restrict__ recv_inv, int* status) {
  __shared__ int seg[kEpMaxCells];
  __shared__ int grp[kEpMaxCells];
  __shared__ int eoff[kEpMaxLocalExperts + 1];
  const int cells = n_src * E_loc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int c = threadIdx.x; c < cells; c += kEpLayoutThreads) seg[c] = __ldg(counts + c);
  __syncthreads();
  if (warp == 0) {
    // receive starts: exclusive scan of the counts in source-major order
    int run = 0;
    for (int c0 = 0; c0 < cells; c0 += 32) {
      const int c = c0 + lane;
      const int v = c < cells ? seg[c] : 0;
      int inc = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += x;
      }
      if (c < cells) grp[c] = v;  // keep the count
      __syncwarp();
      if (c < cells) seg[c] = run + inc - v;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0 && run != R) record_status(status, MOE_DEV_BAD_INDEX);
  }
  __syncthreads();
  if (warp == 1) {
    // expert totals, then their exclusive scan: the local expert offsets
    int run = 0;
    for (int e0 = 0; e0 < E_loc; e0 += 32) {
      const int e = e0 + lane;
      int v = 0;
      if (e < E_loc)
        for (int s = 0; s < n_src; ++s) v += grp[s * E_loc + e];
      int inc = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += x;
      }
      if (e < E_loc) eoff[e] = run + inc - v;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) eoff[E_loc] = run;
  }
  __syncthreads();
  // grouped starts: expert start + rows of the same expert from earlier sources
  for (int e = threadIdx.x; e < E_loc; e += kEpLayoutThreads) {
    int run = eoff[e];
    for (int s = 0; s < n_src; ++s) {
      const int c = grp[s * E_loc + e];
      grp[s * E_loc + e] = run;
      run += c;
    }
    if (blockIdx.x == 0) local_offsets[e] = eoff[e];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) local_offsets[E_loc] = eoff[E_loc];
  __syncthreads();
  for (int r = blockIdx.x * kEpLayoutThreads + threadIdx.x; r < R;
       r += gridDim.x * kEpLayoutThreads) {
    int lo = 0, hi = cells - 1;  // last cell with seg <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seg[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int g = grp[lo] + (r - seg[lo]);
    if (g < 0 || g >= R) {
      record_status(status, MOE_DEV_BAD_INDEX);
      continue;
    }
    recv_perm[g] = r;
    recv_inv[r] = g;
  }
}

}  // namespace moe
