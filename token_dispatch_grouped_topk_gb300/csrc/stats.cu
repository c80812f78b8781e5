// Layer statistics of one routing: the route, message and tile counts the
// pages use to account for a layer's traffic and GEMM efficiency.
//
// "SGLang、NCCL 与 MoE EP", §5.3: a token's payload goes once to each distinct
// destination rank among its routes (D_t of them, §2.3.2), so the exchange
// moves sum_t D_t messages; routes whose expert lives on another logical rank
// than the token are the cross-rank routes (160 of the 224 in the traced
// scenario).  "SGLang Expert Compute Backend", §5.4: the M-row fill rate of a
// grouped GEMM is the valid rows over the rows its M-blocks cover; here the
// blocks are the 128-row blocks the GEMM tile list holds (sum_e ceil(c_e/128))
// against the E * ceil(R/128) blocks a capacity-dense launch would cover.
//
// One thread per token: its K routes give D_t (distinct ranks among the valid
// ids, K <= 32 compares) and its cross-rank routes; block sums are added to
// 64-bit counters.  Block 0 also walks the experts' counts.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kStatsThreads = 256;

__device__ __forceinline__ int token_rank(const int32_t* offsets, int W, int per, int t) {
  if (offsets == nullptr) return min(t / per, W - 1);
  int lo = 0, hi = W - 1;  // largest r with offsets[r] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename IdT>
__global__ void __launch_bounds__(kStatsThreads)
    layer_stats_kernel(const IdT* __restrict__ topk_idx, const int32_t* __restrict__ counts,
                       int T, int K, int E, int L, int R, const int32_t* __restrict__ rank_offsets,
                       unsigned long long* __restrict__ stats) {
  __shared__ unsigned long long s_sum[3];  // valid routes, messages, cross-rank routes
  if (threadIdx.x < 3) s_sum[threadIdx.x] = 0;
  __syncthreads();
  const int W = E / L;
  const int per = (T + W - 1) / W > 0 ? (T + W - 1) / W : 1;
  const int t = blockIdx.x * kStatsThreads + threadIdx.x;
  int valid = 0, msgs = 0, cross = 0;
  if (t < T) {
    const int src = token_rank(rank_offsets, W, per, t);
    int ranks[32];
    for (int k = 0; k < K; ++k) {
      const int64_t id = static_cast<int64_t>(topk_idx[static_cast<int64_t>(t) * K + k]);
      if (id < 0 || id >= E) continue;
      const int r = static_cast<int>(id) / L;
      ++valid;
      cross += r != src;
      bool seen = false;
      for (int j = 0; j < msgs; ++j) seen |= ranks[j] == r;
      if (!seen) ranks[msgs++] = r;
    }
  }
  atomicAdd(&s_sum[0], static_cast<unsigned long long>(valid));
  atomicAdd(&s_sum[1], static_cast<unsigned long long>(msgs));
  atomicAdd(&s_sum[2], static_cast<unsigned long long>(cross));
  __syncthreads();
  if (threadIdx.x < 3) atomicAdd(&stats[threadIdx.x == 0 ? 0 : threadIdx.x + 1], s_sum[threadIdx.x]);
  if (blockIdx.x == 0) {
    // per-expert part: kept routes, 128-row blocks, active experts, busiest count
    unsigned long long kept = 0, blocks = 0, active = 0;
    int busiest = 0;
    for (int e = threadIdx.x; e < E; e += kStatsThreads) {
      const int c = max(0, min(counts[e], R));
      kept += c;
      blocks += (c + 127) / 128;
      active += c > 0;
      busiest = max(busiest, c);
    }
    atomicAdd(&stats[1], kept);
    atomicAdd(&stats[4], blocks);
    atomicAdd(&stats[5], active);
    atomicMax(&stats[6], static_cast<unsigned long long>(busiest));
  }
}

}  // namespace

cudaError_t launch_layer_stats(const void* topk_idx, int idx_bits, const int32_t* counts, int T,
                               int K, int E, int L, int R, const int32_t* rank_offsets,
                               unsigned long long* stats, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(stats, 0, kLayerStats * sizeof(unsigned long long), s);
  if (err != cudaSuccess) return err;
  const int blocks = std::max(1, (T + kStatsThreads - 1) / kStatsThreads);
  if (idx_bits == 32)
    layer_stats_kernel<int32_t><<<blocks, kStatsThreads, 0, s>>>(
        static_cast<const int32_t*>(topk_idx), counts, T, K, E, L, R, rank_offsets, stats);
  else
    layer_stats_kernel<int64_t><<<blocks, kStatsThreads, 0, s>>>(
        static_cast<const int64_t*>(topk_idx), counts, T, K, E, L, R, rank_offsets, stats);
  return cudaGetLastError();
}

}  // namespace moe
