// attn_varlen_plan: the work tiles of a ragged batch, longest first, for the varlen forward.
//
// "flash-attention-3" (ai.thesatyajit.com), "Five schedulers": a varlen persistent scheduler for
// ragged batches and a longest-processing-time-first order for causal work; "What is actually in
// the box": the scheduler's metadata is computed once so that a serving loop can reuse it.
//
// A work tile is (sequence b, query head h, query block m): rows m*R .. m*R+R-1 of sequence b,
// R = 128 * (Q tiles per CTA). Its cost is the number of 128-key tiles its longest Q tile visits.
// One CTA on the stream:
//   1. tiles per sequence, ceil(Nq_b / R), and their exclusive prefix over b;
//   2. a histogram of tile costs in shared memory;
//   3. start offsets of the cost bins, largest cost first;
//   4. each tile written at its bin's next slot (warp-aggregated atomics, so the order within a
//      bin depends on timing; outputs do not depend on the order).
// The plan also records B, H, R, the mask and the packed row totals; the forward checks them.
// Offsets that are not non-decreasing, exceed the totals, or give more tiles than the plan holds
// make an empty plan marked invalid (the forward then reports it through the status word).
#include <cstdint>

#include <cuda_runtime.h>

#include "launch.h"
#include "varlen.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int kCostBins = 4096;   // costs from 4095 up share the last bin

// Work tile e (natural order: sequence, then head, then query block) -> (b, h, m).
__device__ __forceinline__ void tile_of(long long e, const int* prefix, int B, int H, int& b, int& h, int& m) {
  int lo = 0, hi = B - 1;   // last b with H * prefix[b] <= e
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)H * prefix[mid] <= e) lo = mid;
    else hi = mid - 1;
  }
  b = lo;
  const int tb = prefix[b + 1] - prefix[b];
  const long long local = e - (long long)H * prefix[b];
  h = (int)(local / tb);
  m = (int)(local % tb);
}

__device__ __forceinline__ int tile_cost(const int* cu_q, const int* cu_k, int b, int m, int R, bool causal) {
  const int nq = cu_q[b + 1] - cu_q[b], nk = cu_k[b + 1] - cu_k[b];
  int cost = 0;
  for (int pos0 = m * R; pos0 < m * R + R; pos0 += 128) {
    const int c = gb300::varlen_kv_tiles(pos0, nq, nk, causal);
    cost = c > cost ? c : cost;
  }
  return cost;
}

__global__ void __launch_bounds__(kThreads) varlen_plan_kernel(const int* cu_q, const int* cu_k, int B, int H, int R,
                                                               bool causal, int total_q, int total_k, int capacity,
                                                               int* plan) {
  __shared__ int bins[kCostBins];
  __shared__ int scan[kThreads];
  __shared__ int carry, bad;
  const int tid = threadIdx.x, lane = tid & 31;
  int* prefix = plan + gb300::kPlanHeaderWords;   // [B + 1]
  int2* tiles = reinterpret_cast<int2*>(plan + gb300::plan_tiles_offset(B));
  if (tid == 0) {
    carry = 0;
    bad = (cu_q[0] != 0 || cu_k[0] != 0 || cu_q[B] > total_q || cu_k[B] > total_k) ? 1 : 0;
  }
  for (int i = tid; i < kCostBins; i += kThreads) bins[i] = 0;
  __syncthreads();
  // 1. tiles per sequence and their prefix, kThreads sequences at a time
  for (int b0 = 0; b0 < B; b0 += kThreads) {
    const int b = b0 + tid;
    int tb = 0;
    if (b < B) {
      const int nq = cu_q[b + 1] - cu_q[b], nk = cu_k[b + 1] - cu_k[b];
      if (nq < 0 || nk < 0 || (nq + R - 1) / R > 0xFFFF) atomicExch(&bad, 1);
      tb = nq > 0 ? (nq + R - 1) / R : 0;
    }
    scan[tid] = tb;
    __syncthreads();
    for (int off = 1; off < kThreads; off <<= 1) {
      const int v = tid >= off ? scan[tid - off] : 0;
      __syncthreads();
      scan[tid] += v;
      __syncthreads();
    }
    if (b < B) prefix[b] = carry + scan[tid] - tb;
    __syncthreads();
    if (tid == kThreads - 1) carry += scan[tid];
    __syncthreads();
  }
  const long long n_tiles = (long long)carry * H;
  if (tid == 0) {
    prefix[B] = carry;
    if (n_tiles > capacity || H > 0x7FFF) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      plan[0] = 0;
      plan[1] = -1;   // matches no launch: the forward reports the plan as invalid
    }
    return;
  }
  // 2. histogram of costs
  for (long long e = tid; e < n_tiles; e += kThreads) {
    int b, h, m;
    tile_of(e, prefix, B, H, b, h, m);
    const int c = tile_cost(cu_q, cu_k, b, m, R, causal);
    atomicAdd(&bins[c < kCostBins ? c : kCostBins - 1], 1);
  }
  __syncthreads();
  // 3. bin starts, largest cost first: thread t owns bins kCostBins-1-4t .. kCostBins-4-4t
  constexpr int PER = kCostBins / kThreads;
  int own = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) own += bins[kCostBins - 1 - (tid * PER + i)];
  scan[tid] = own;
  __syncthreads();
  for (int off = 1; off < kThreads; off <<= 1) {
    const int v = tid >= off ? scan[tid - off] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  int run = scan[tid] - own;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int bin = kCostBins - 1 - (tid * PER + i);
    const int cnt = bins[bin];
    bins[bin] = run;   // each bin is read and rewritten by its one owner thread
    run += cnt;
  }
  __syncthreads();
  // 4. scatter
  for (long long e0 = 0; e0 < n_tiles; e0 += kThreads) {
    const long long e = e0 + tid;
    const bool active = e < n_tiles;
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (active) {
      int b, h, m;
      tile_of(e, prefix, B, H, b, h, m);
      const int c = tile_cost(cu_q, cu_k, b, m, R, causal);
      const int bin = c < kCostBins ? c : kCostBins - 1;
      const unsigned peers = __match_any_sync(act, bin);
      const int leader = __ffs(peers) - 1;
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int base = 0;
      if (lane == leader) base = atomicAdd(&bins[bin], __popc(peers));
      base = __shfl_sync(peers, base, leader);
      tiles[base + rank] = make_int2(b, (h << 16) | m);
    }
  }
  __syncthreads();
  if (tid == 0) {
    plan[0] = (int)n_tiles;
    plan[1] = B;
    plan[2] = H;
    plan[3] = R;
    plan[4] = causal ? 1 : 0;
    plan[5] = gb300::plan_tiles_offset(B);
    plan[6] = total_q;
    plan[7] = total_k;
  }
}

}  // namespace

namespace gb300 {

cudaError_t launch_varlen_plan(const int* cu_q, const int* cu_k, int B, int H, int rows_per_tile, bool causal,
                               int total_q, int total_k, int capacity, int* plan, cudaStream_t stream) {
  varlen_plan_kernel<<<1, kThreads, 0, stream>>>(cu_q, cu_k, B, H, rows_per_tile, causal, total_q, total_k, capacity,
                                                 plan);
  return cudaGetLastError();
}

}  // namespace gb300
