// Expert parallelism across ranks: the send plan, the routes-per-message
// offsets, the return pack and the source's result map.
//
// "SGLang、NCCL 与 MoE EP", §2.3.2: a token sends one payload to each distinct
// destination rank among its routes (the unit of deduplication is (source
// rank, token row, destination rank)); the message header keeps the original
// token and the route list.  §2.3.4: the destination writes one expert input
// per route.  §3.2 (合对): the destination sends every route's expert output
// back into that route's result slot at the source rank, which multiplies by
// the router weight and sums into the token's row.
//
// On each rank the data path is:
//   source     ep_dedup_kernel   the route owning each (token, destination)
//              dispatch kernels   one payload row per message, packed by
//                                 destination rank in ascending token order
//              ep_header_kernel  per message the destination-local expert id
//                                 of each top-k position (-1 elsewhere); per
//                                 route its message and its position in it
//   -- all-to-all of payload rows and route lists --
//   destination the layer's own dispatch / expert compute on the received rows
//              ep_offsets_*      exclusive prefix of routes per received row
//              ep_return_kernel  one row per route: the expert output, or zeros
//                                and flag 0 for a route dropped by capacity
//   -- all-to-all of the returned rows back --
//   source     ep_offsets_*      the same prefix over the sent messages
//              ep_result_kernel  route (t, k) -> its returned row, or -1
//              combine           (moe_combine_packed) as on one GPU
// Rows arrive at a destination grouped by source rank in ascending token order,
// so its per-expert slots follow ascending global route id: the slots, capacity
// drops and results are those of the one-GPU layer on all ranks' tokens.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kEpThreads = 256;
constexpr int kScanRows = 1024;  // rows per block of the offsets scan (4 per thread)

template <typename IdT>
__device__ __forceinline__ int route_dest(const IdT* idx, int E, int L, int64_t i) {
  const int64_t id = static_cast<int64_t>(idx[i]);
  return (id >= 0 && id < E) ? static_cast<int>(id / L) : -1;
}

// dest[t, k] = destination rank of route (t, k) if it is the token's first
// route to that rank (the one that owns the message), else -1.
template <typename IdT>
__global__ void __launch_bounds__(kEpThreads)
    ep_dedup_kernel(const IdT* __restrict__ topk_idx, int T, int K, int E, int L,
                    int32_t* __restrict__ dest) {
  const int t = blockIdx.x * kEpThreads + threadIdx.x;
  if (t >= T) return;
  const int64_t row = static_cast<int64_t>(t) * K;
  for (int k = 0; k < K; ++k) {
    const int d = route_dest(topk_idx, E, L, row + k);
    bool owner = d >= 0;
    for (int j = 0; j < k && owner; ++j) owner = route_dest(topk_idx, E, L, row + j) != d;
    dest[row + k] = owner ? d : -1;
  }
}

// From the message row msg[t, k] of each owning route: the message's route
// list send_ids[u, :] (destination-local expert id of every top-k position
// that goes to the same rank, -1 elsewhere), and for every route its message
// route_msg[t, k] and its position route_pos[t, k] among the message's routes.
template <typename IdT>
__global__ void __launch_bounds__(kEpThreads)
    ep_header_kernel(const IdT* __restrict__ topk_idx, const int32_t* __restrict__ msg, int T,
                     int K, int E, int L, int32_t* __restrict__ send_ids,
                     int32_t* __restrict__ route_msg, int32_t* __restrict__ route_pos,
                     int32_t* dev_status) {
  const int t = blockIdx.x * kEpThreads + threadIdx.x;
  if (t >= T) return;
  const int64_t row = static_cast<int64_t>(t) * K;
  for (int k = 0; k < K; ++k) {
    const int d = route_dest(topk_idx, E, L, row + k);
    if (d < 0) {
      const int64_t id = static_cast<int64_t>(topk_idx[row + k]);
      if (id != -1) atomicOr(dev_status, kDevBadExpertId);   // reported, route ignored
      route_msg[row + k] = -1;
      route_pos[row + k] = -1;
      continue;
    }
    int owner = k, pos = 0;
    for (int j = k - 1; j >= 0; --j) {
      if (route_dest(topk_idx, E, L, row + j) == d) {
        owner = j;
        ++pos;
      }
    }
    const int u = msg[row + owner];
    route_msg[row + k] = u;
    route_pos[row + k] = u >= 0 ? pos : -1;
    if (owner == k && u >= 0) {
      int32_t* ids = send_ids + static_cast<int64_t>(u) * K;
      for (int j = 0; j < K; ++j) {
        const int dj = route_dest(topk_idx, E, L, row + j);
        ids[j] = dj == d ? static_cast<int>(static_cast<int64_t>(topk_idx[row + j]) % L) : -1;
      }
    }
  }
}

__device__ __forceinline__ int routes_of_row(const int32_t* ids, int K, int64_t j) {
  int n = 0;
  for (int k = 0; k < K; ++k) n += ids[j * K + k] >= 0;
  return n;
}

// Offsets scan, phase 1: routes of each block of kScanRows rows.
__global__ void __launch_bounds__(kEpThreads)
    ep_offsets_sum_kernel(const int32_t* __restrict__ ids, int64_t S, int K,
                          int32_t* __restrict__ block_sums) {
  __shared__ int s_warp[kEpThreads / 32];
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kScanRows;
  int n = 0;
  for (int i = threadIdx.x; i < kScanRows; i += kEpThreads)
    if (j0 + i < S) n += routes_of_row(ids, K, j0 + i);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    int tot = 0;
    for (int w = 0; w < kEpThreads / 32; ++w) tot += s_warp[w];
    block_sums[blockIdx.x] = tot;
  }
}

// Phase 2: exclusive prefix of the block sums (one block, in chunks).
__global__ void __launch_bounds__(kEpThreads)
    ep_offsets_blocks_kernel(int32_t* __restrict__ block_sums, int nb) {
  __shared__ int s_warp[kEpThreads / 32];
  __shared__ int s_carry;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int b0 = 0; b0 < nb; b0 += kEpThreads) {
    const int b = b0 + threadIdx.x;
    const int v = b < nb ? block_sums[b] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = s_carry;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    if (b < nb) block_sums[b] = before + incl - v;
    __syncthreads();
    if (threadIdx.x == kEpThreads - 1) s_carry = before + incl;
    __syncthreads();
  }
}

// Phase 3: offsets[j] = routes of rows before j; offsets[S] = all routes.
__global__ void __launch_bounds__(kEpThreads)
    ep_offsets_write_kernel(const int32_t* __restrict__ ids, int64_t S, int K,
                            const int32_t* __restrict__ block_prefix,
                            int32_t* __restrict__ offsets) {
  __shared__ int s_warp[kEpThreads / 32];
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kScanRows;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // each thread owns 4 consecutive rows
  constexpr int kPer = kScanRows / kEpThreads;
  int n[kPer];
  int mine = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int64_t j = j0 + threadIdx.x * kPer + i;
    n[i] = j < S ? routes_of_row(ids, K, j) : 0;
    mine += n[i];
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int run = block_prefix[blockIdx.x] + incl - mine;
  for (int w = 0; w < warp; ++w) run += s_warp[w];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int64_t j = j0 + threadIdx.x * kPer + i;
    if (j < S) offsets[j] = run;
    run += n[i];
    if (j == S - 1) offsets[S] = run;
  }
}

// One warp per received row: each of its routes (top-k positions with a local
// id) gets one returned row at offsets[j] + position: the expert output if the
// layer kept the route (src_map >= 0), zeros and flag 0 if capacity dropped it.
__global__ void __launch_bounds__(kEpThreads)
    ep_return_kernel(const uint4* __restrict__ out, int64_t out_rows,
                     const int32_t* __restrict__ src_map, const int32_t* __restrict__ ids,
                     const int32_t* __restrict__ offsets, int64_t S, int K, int H,
                     uint4* __restrict__ ret, int32_t* __restrict__ flag) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * (kEpThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= S) return;
  const int nvec = H / 8;
  int p = 0;
  for (int k = 0; k < K; ++k) {
    if (ids[j * K + k] < 0) continue;
    const int64_t dst = offsets[j] + p;
    ++p;
    const int q = src_map[j * K + k];
    const bool kept = q >= 0 && q < out_rows;
    if (lane == 0) flag[dst] = kept ? 1 : 0;
    uint4* drow = ret + dst * nvec;
    if (kept) {
      const uint4* srow = out + static_cast<int64_t>(q) * nvec;
      for (int v = lane; v < nvec; v += 32) drow[v] = ld_stream(srow + v);
    } else {
      for (int v = lane; v < nvec; v += 32) drow[v] = make_uint4(0, 0, 0, 0);
    }
  }
}

// result_map[t, k] = the returned row of route (t, k) if its destination kept
// it, else -1 (also for routes with no destination).
__global__ void __launch_bounds__(kEpThreads)
    ep_result_kernel(const int32_t* __restrict__ route_msg, const int32_t* __restrict__ route_pos,
                     const int32_t* __restrict__ offsets, const int32_t* __restrict__ flag,
                     int64_t n_ret, int64_t n, int32_t* __restrict__ result_map) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kEpThreads + threadIdx.x;
  if (i >= n) return;
  const int u = route_msg[i];
  int r = -1;
  if (u >= 0) {
    const int64_t row = static_cast<int64_t>(offsets[u]) + route_pos[i];
    if (row >= 0 && row < n_ret && flag[row]) r = static_cast<int>(row);
  }
  result_map[i] = r;
}

template <typename IdT>
cudaError_t ep_pack_impl(const void* x, const IdT* topk_idx, int T, int H, int K, int E, int L,
                         void* send_x, int32_t* send_ids, int32_t* send_counts,
                         int32_t* route_msg, int32_t* route_pos, int32_t* dev_status,
                         int32_t* dest, int32_t* msg, int32_t* hist, int sm_count,
                         cudaStream_t s) {
  const int W = E / L;
  const int blocks = std::max(1, (T + kEpThreads - 1) / kEpThreads);
  cudaError_t err;
  if (T > 0) {
    ep_dedup_kernel<IdT><<<blocks, kEpThreads, 0, s>>>(topk_idx, T, K, E, L, dest);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  // one payload per message: a dispatch whose experts are the destination
  // ranks, capacity T, packed rows (messages to rank d back to back)
  const int64_t rows = std::max<int64_t>(1, static_cast<int64_t>(T) * std::min(K, W));
  err = launch_dispatch(x, dest, 32, T, H, K, W, RowLayout{T > 0 ? T : 1, 1, rows}, send_x,
                        send_counts, msg, dev_status, hist, sm_count, s);
  if (err != cudaSuccess || T == 0) return err;
  ep_header_kernel<IdT><<<blocks, kEpThreads, 0, s>>>(topk_idx, msg, T, K, E, L, send_ids,
                                                      route_msg, route_pos, dev_status);
  return cudaGetLastError();
}

}  // namespace

size_t ep_offsets_scratch_ints(int64_t S) { return static_cast<size_t>((S + kScanRows - 1) / kScanRows) + 1; }

cudaError_t launch_ep_pack(const void* x, const void* topk_idx, int idx_bits, int T, int H, int K,
                           int E, int L, void* send_x, int32_t* send_ids, int32_t* send_counts,
                           int32_t* route_msg, int32_t* route_pos, int32_t* dev_status,
                           int32_t* dest, int32_t* msg, int32_t* hist, int sm_count,
                           cudaStream_t s) {
  if (idx_bits == 32)
    return ep_pack_impl(x, static_cast<const int32_t*>(topk_idx), T, H, K, E, L, send_x, send_ids,
                        send_counts, route_msg, route_pos, dev_status, dest, msg, hist, sm_count, s);
  return ep_pack_impl(x, static_cast<const int64_t*>(topk_idx), T, H, K, E, L, send_x, send_ids,
                      send_counts, route_msg, route_pos, dev_status, dest, msg, hist, sm_count, s);
}

cudaError_t launch_ep_offsets(const int32_t* ids, int64_t S, int K, int32_t* offsets,
                              int32_t* scratch, cudaStream_t s) {
  if (S == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t), s);
  const int nb = static_cast<int>((S + kScanRows - 1) / kScanRows);
  ep_offsets_sum_kernel<<<nb, kEpThreads, 0, s>>>(ids, S, K, scratch);
  ep_offsets_blocks_kernel<<<1, kEpThreads, 0, s>>>(scratch, nb);
  ep_offsets_write_kernel<<<nb, kEpThreads, 0, s>>>(ids, S, K, scratch, offsets);
  return cudaGetLastError();
}

cudaError_t launch_ep_return(const void* out, int64_t out_rows, const int32_t* src_map,
                             const int32_t* ids, const int32_t* offsets, int64_t S, int K, int H,
                             void* ret, int32_t* flag, cudaStream_t s) {
  if (S == 0) return cudaSuccess;
  const int64_t warps = kEpThreads / 32;
  const int blocks = static_cast<int>((S + warps - 1) / warps);
  ep_return_kernel<<<blocks, kEpThreads, 0, s>>>(static_cast<const uint4*>(out), out_rows, src_map,
                                                 ids, offsets, S, K, H, static_cast<uint4*>(ret),
                                                 flag);
  return cudaGetLastError();
}

cudaError_t launch_ep_result(const int32_t* route_msg, const int32_t* route_pos,
                             const int32_t* offsets, const int32_t* flag, int64_t n_ret, int T,
                             int K, int32_t* result_map, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(T) * K;
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>((n + kEpThreads - 1) / kEpThreads);
  ep_result_kernel<<<blocks, kEpThreads, 0, s>>>(route_msg, route_pos, offsets, flag, n_ret, n,
                                                 result_map);
  return cudaGetLastError();
}

}  // namespace moe
