// Dispatch: route validation, per-expert counting, slot assignment and the
// payload scatter into the expert-major receive buffer.
//
// "SGLang、NCCL 与 MoE EP", §2.3.4: every route to expert e takes a row s from
// e's counter, the payload is written to recv[e, s, :] and the flat row
// q = e*R + s is recorded for combine (§2.3.6).  On one GPU the per-expert
// counter is replaced by a deterministic three-kernel scheme so the slot of a
// route is its rank among e's routes in ascending route id:
//   1. route_hist    -- each block counts its routes per expert (warp match +
//                       shared-memory atomics; integer sums are order-free);
//   2. route_scan    -- one block per expert: exclusive scan of the block
//                       counts, counts[e] = min(total, R), drops reported;
//   3. route_scatter -- each block re-derives the in-block rank of its routes
//                       (warp match + per-warp counts), writes src_map and
//                       copies each token row once from x to its K rows of
//                       recv with 16-byte vector accesses.
// The row of slot s of expert e is e*R + s (padded layout) or base_e + s with
// base_e the prefix of the clamped counts (packed layout, §2.6 of "SGLang
// Expert Compute Backend": the valid rows of all experts back to back).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// Lane `lane` of global warp `gw` holds route (t, k) with
// t = gw * (32/K) + lane / K and k = lane % K.
struct RouteLane {
  int t, k, e;  // e = expert id, or -1 for padding / invalid id / idle lane
  bool active;  // the lane maps to a real route (t < T)
};

// Router ids are int64 or int32 (IdT); -1 marks a padding route.
template <typename IdT>
__device__ __forceinline__ RouteLane load_route(const IdT* __restrict__ topk_idx, int T, int K,
                                                int E, int gw, int lane, int32_t* dev_status) {
  const int tpw = 32 / K;
  RouteLane r;
  r.t = gw * tpw + lane / K;
  r.k = lane % K;
  r.active = (lane < tpw * K) && (r.t < T);
  r.e = -1;
  if (r.active) {
    const int64_t id = static_cast<int64_t>(topk_idx[static_cast<int64_t>(r.t) * K + r.k]);
    if (id >= 0 && id < E) {
      r.e = static_cast<int>(id);
    } else if (id != -1 && dev_status != nullptr) {
      atomicOr(dev_status, kDevBadExpertId);
    }
  }
  return r;
}

template <typename IdT>
__global__ void __launch_bounds__(kDispatchWarps * 32)
    route_hist_kernel(const IdT* __restrict__ topk_idx, int T, int K, int E, int nblocks,
                      int32_t* __restrict__ hist, int32_t* dev_status) {
  extern __shared__ int s_hist[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RouteLane r =
      load_route(topk_idx, T, K, E, blockIdx.x * kDispatchWarps + warp, lane, dev_status);
  const unsigned peers = __match_any_sync(0xffffffffu, r.e);
  if (r.e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[r.e], __popc(peers));
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    hist[static_cast<size_t>(e) * nblocks + blockIdx.x] = s_hist[e];
}

constexpr int kScanThreads = 512;

__global__ void __launch_bounds__(kScanThreads)
    route_scan_kernel(int32_t* __restrict__ hist, int nblocks, int R, int32_t* __restrict__ counts,
                      int32_t* dev_status) {
  __shared__ int s_warp[kScanThreads / 32];
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* h = hist + static_cast<size_t>(e) * nblocks;
  const int per = (nblocks + kScanThreads - 1) / kScanThreads;
  const int b0 = threadIdx.x * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (b0 + i < nblocks) local += h[b0 + i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = lane < kScanThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane < kScanThreads / 32) s_warp[lane] = v;
  }
  __syncthreads();
  int run = (warp > 0 ? s_warp[warp - 1] : 0) + incl - local;
  for (int i = 0; i < per; ++i) {
    if (b0 + i < nblocks) {
      const int v = h[b0 + i];
      h[b0 + i] = run;
      run += v;
    }
  }
  if (threadIdx.x == 0) {
    const int total = s_warp[kScanThreads / 32 - 1];
    counts[e] = min(total, R);
    if (total > R) {
      atomicAdd(dev_status + 1, total - R);
      atomicOr(dev_status, kDevCapacityDropped);
    }
  }
}

// Single-pass slot bases for small route counts (T*K <= kSinglePassRoutes):
// instead of the histogram and scan kernels, every block counts in shared
// memory, straight from topk_idx, the routes to each expert before its own
// first route (s_prev) and in all (s_tot).  The slots are then the ones the
// scanned histograms give.  Block (0, 0) writes counts[e] = min(s_tot[e], R)
// and both status words (bad-id bit, drop bit and count), so the launch needs
// no status reset either.  With the packed layout the row bases are the
// prefix of the clamped totals (s_rows).  Every thread of the block calls it.
template <typename IdT>
__device__ void single_pass_bases(const IdT* __restrict__ topk_idx, int T, int K, int E,
                                  RowLayout rl, int* s_prev, int* s_tot, int* s_rows,
                                  int32_t* __restrict__ counts, int32_t* dev_status) {
  __shared__ int s_dropped;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_prev[e] = s_tot[e] = 0;
  if (threadIdx.x == 0) s_dropped = 0;
  __syncthreads();
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kDispatchWarps * (32 / K) * K;
  const int64_t n = static_cast<int64_t>(T) * K;
  int bad = 0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t id = static_cast<int64_t>(topk_idx[i]);
    if (id >= 0 && id < E) {
      atomicAdd(&s_tot[id], 1);
      if (i < first) atomicAdd(&s_prev[id], 1);
    } else if (id != -1) {
      bad = 1;
    }
  }
  bad = __syncthreads_or(bad);
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    int dropped = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      counts[e] = min(s_tot[e], rl.R);
      dropped += max(s_tot[e] - rl.R, 0);
    }
    if (dropped) atomicAdd(&s_dropped, dropped);
    __syncthreads();
    if (threadIdx.x == 0) {
      dev_status[0] = (bad ? kDevBadExpertId : 0) | (s_dropped > 0 ? kDevCapacityDropped : 0);
      dev_status[1] = s_dropped;
    }
  }
  if (rl.packed) expert_prefix(s_tot, E, rl.R, 1, 1, s_rows, nullptr);
  __syncthreads();
}

template <typename IdT, bool kSingle, int kPreload>
__global__ void __launch_bounds__(kDispatchWarps * 32)
    route_scatter_kernel(const uint4* __restrict__ x, const IdT* __restrict__ topk_idx, int T,
                         int H, int K, int E, RowLayout rl, int nblocks,
                         const int32_t* __restrict__ base, int32_t* __restrict__ counts,
                         uint4* __restrict__ recv, int32_t* __restrict__ src_map,
                         int32_t* dev_status, int vec_per_slice) {
  extern __shared__ int smem[];
  int* s_cnt = smem;                           // [kDispatchWarps][E]
  int* s_dest = smem + kDispatchWarps * E;     // [kDispatchWarps][32]
  int* s_rows = s_dest + kDispatchWarps * 32;  // [E + 1] packed row bases
  int* s_prev = s_rows + E + 1;                // single pass: [E] routes before this block
  int* s_tot = s_prev + E;                     //              [E] all routes
  for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) s_cnt[i] = 0;
  if (kSingle)
    single_pass_bases(topk_idx, T, K, E, rl, s_prev, s_tot, s_rows, counts, dev_status);
  else if (rl.packed)
    expert_prefix(counts, E, rl.R, 1, 1, s_rows, nullptr);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kDispatchWarps + warp;
  const RouteLane r = load_route(topk_idx, T, K, E, gw, lane, nullptr);
  const unsigned peers = __match_any_sync(0xffffffffu, r.e);
  const int lane_rank = __popc(peers & ((1u << lane) - 1u));
  if (r.e >= 0 && lane == __ffs(peers) - 1) s_cnt[warp * E + r.e] = __popc(peers);
  __syncthreads();
  int q = -1;
  if (r.e >= 0) {
    int s = (kSingle ? s_prev[r.e] : base[static_cast<size_t>(r.e) * nblocks + blockIdx.x]) +
            lane_rank;
    for (int w = 0; w < warp; ++w) s += s_cnt[w * E + r.e];
    if (s < rl.R) q = (rl.packed ? s_rows[r.e] : r.e * rl.R) + s;
  }
  if (blockIdx.y == 0 && r.active) src_map[static_cast<int64_t>(r.t) * K + r.k] = q;
  s_dest[warp * 32 + lane] = q;
  __syncwarp();

  // Payload: each token row is read once (this block's slice of it) and
  // written to every kept destination row.
  const int tpw = 32 / K;
  const int nvec = H / 8;
  const int v0 = blockIdx.y * vec_per_slice;
  const int v1 = min(nvec, v0 + vec_per_slice);
  const int* wdest = s_dest + warp * 32;
  // When the warp's tokens' slices fit in kPreload (8 or 16) 16-byte vectors
  // per lane (U per token; the slices are short when there are few tokens, as
  // at decode and prefill), every load is issued before the first store: one
  // memory round trip per warp instead of one per token (prefill -5 %, and
  // -3 % more with the 8-deep form, which needs 64 registers against 128).
  // It is a kernel of its own: its registers would cut the resident warps of
  // the loop below (48 registers).
  if constexpr (kPreload > 0) {
    const int U = (vec_per_slice + 31) / 32;
    uint4 a[kPreload];
#pragma unroll
    for (int i = 0; i < kPreload; ++i) {
      const int tt = i / U, u = i - (i / U) * U;
      const int t = gw * tpw + tt;
      const int v = v0 + lane + 32 * u;
      if (tt < tpw && t < T && v < v1) a[i] = ld_stream(x + static_cast<size_t>(t) * nvec + v);
    }
#pragma unroll
    for (int i = 0; i < kPreload; ++i) {
      const int tt = i / U, u = i - (i / U) * U;
      const int t = gw * tpw + tt;
      const int v = v0 + lane + 32 * u;
      if (tt >= tpw || t >= T || v >= v1) continue;
      const int* dq = wdest + tt * K;
      for (int k = 0; k < K; ++k) {
        const int qq = dq[k];
        if (qq >= 0) recv[static_cast<size_t>(qq) * nvec + v] = a[i];
      }
    }
  } else {
    for (int tt = 0; tt < tpw; ++tt) {
      const int t = gw * tpw + tt;
      if (t >= T) break;
      const int* dq = wdest + tt * K;
      bool any = false;
      for (int k = 0; k < K; ++k) any |= dq[k] >= 0;
      if (!any) continue;
      const uint4* src = x + static_cast<size_t>(t) * nvec;
      // eight 16-byte vectors per lane in flight (four left the large layer's
      // scatter 6 % slower)
      for (int v = v0 + lane; v < v1; v += 32 * 8) {
        uint4 a[8];
  #pragma unroll
        for (int u = 0; u < 8; ++u)
          if (v + 32 * u < v1) a[u] = ld_stream(src + v + 32 * u);
        for (int k = 0; k < K; ++k) {
          const int qq = dq[k];
          if (qq < 0) continue;
          uint4* dst = recv + static_cast<size_t>(qq) * nvec;
  #pragma unroll
          for (int u = 0; u < 8; ++u)
            if (v + 32 * u < v1) dst[v + 32 * u] = a[u];
        }
      }
    }
  }
}

// One 128-element group per half-warp (8 BF16 per lane): the group amax by a
// 4-step shuffle, then the lane's 8 e4m3 codes and the group's scale.  Every
// lane of the warp calls it (the shuffles); `on` marks lanes with a group.
__device__ __forceinline__ void quantize_group(const uint4& v, bool on, uint2* codes,
                                               float* scale) {
  float f[8];
  float amax = 0.f;
  if (on) {
    bf16x8_to_f32(v, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  *codes = make_uint2(0u, 0u);
  *scale = 0.f;
  if (!on) return;
  float mult;
  fp8_group_scale(amax, &mult, scale);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lo |= static_cast<uint32_t>(pack_e4m3x2(__fmul_rn(f[2 * i], mult), __fmul_rn(f[2 * i + 1], mult)))
          << (16 * i);
    hi |= static_cast<uint32_t>(pack_e4m3x2(__fmul_rn(f[4 + 2 * i], mult), __fmul_rn(f[5 + 2 * i], mult)))
          << (16 * i);
  }
  *codes = make_uint2(lo, hi);
}

// The FP8 scatter issues all of a warp's loads before its first conversion
// (kPreload = 8 or 16 loads per lane, one per half-warp group pair and token)
// when each lane needs at most eight, or at most sixteen and the grid fits on
// the GPU in one wave.  The 8-deep form costs no registers over the loop
// (64): decode 15.0 -> 12.9 us, prefill 52.9 -> 42.7 us.  The 16-deep form
// takes 127 registers, which with more blocks than one wave cost more
// resident warps than the loads gain; kPreload = 0 is the loop over tokens.
//
// Dispatch fused with the per-token FP8 quantisation ("SGLang Expert Compute
// Backend", §4.4: quantise while packing instead of materialising BF16 rows).
// Every route of a token carries the same row, and the quantisation is per row
// and per 128-group, so each token row is quantised once and its e4m3 codes and
// fp32 scales are written to every kept destination row; the BF16 receive
// buffer is never formed.  Rank derivation is the one of route_scatter_kernel.
// Each block takes a slice of whole 128-groups of its tokens' rows.
template <typename IdT, bool kSingle, int kPreload>
__global__ void __launch_bounds__(kDispatchWarps * 32)
    route_scatter_fp8_kernel(const uint4* __restrict__ x, const IdT* __restrict__ topk_idx,
                             int T, int H, int K, int E, RowLayout rl, int nblocks,
                             const int32_t* __restrict__ base, int32_t* __restrict__ counts,
                             uint2* __restrict__ xq, float* __restrict__ xs,
                             int32_t* __restrict__ src_map, int32_t* dev_status,
                             int groups_per_slice) {
  extern __shared__ int smem[];
  int* s_cnt = smem;                                               // [kDispatchWarps][E]
  int* s_dest = smem + kDispatchWarps * E;                         // [kDispatchWarps][32]
  int* s_rows = s_dest + kDispatchWarps * 32;                       // [E + 1] packed row bases
  int* s_prev = s_rows + E + 1;                                    // single pass: [E]
  int* s_tot = s_prev + E;                                         //              [E]
  float* s_sc = reinterpret_cast<float*>(s_tot + E);  // [warps][tpw or 1][groups_per_slice]
  for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) s_cnt[i] = 0;
  if (kSingle)
    single_pass_bases(topk_idx, T, K, E, rl, s_prev, s_tot, s_rows, counts, dev_status);
  else if (rl.packed)
    expert_prefix(counts, E, rl.R, 1, 1, s_rows, nullptr);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int gw = blockIdx.x * kDispatchWarps + warp;
  const RouteLane r = load_route(topk_idx, T, K, E, gw, lane, nullptr);
  const unsigned peers = __match_any_sync(0xffffffffu, r.e);
  const int lane_rank = __popc(peers & ((1u << lane) - 1u));
  if (r.e >= 0 && lane == __ffs(peers) - 1) s_cnt[warp * E + r.e] = __popc(peers);
  __syncthreads();
  int q = -1;
  if (r.e >= 0) {
    int sl = (kSingle ? s_prev[r.e] : base[static_cast<size_t>(r.e) * nblocks + blockIdx.x]) +
             lane_rank;
    for (int w = 0; w < warp; ++w) sl += s_cnt[w * E + r.e];
    if (sl < rl.R) q = (rl.packed ? s_rows[r.e] : r.e * rl.R) + sl;
  }
  if (blockIdx.y == 0 && r.active) src_map[static_cast<int64_t>(r.t) * K + r.k] = q;
  s_dest[warp * 32 + lane] = q;
  __syncwarp();

  const int tpw = 32 / K;
  const int G = H / kGroup;
  const int g0 = blockIdx.y * groups_per_slice;
  const int g1 = min(G, g0 + groups_per_slice);
  const int* wdest = s_dest + warp * 32;
  if constexpr (kPreload > 0) {
    // Scales staged per token: [tpw][groups_per_slice].  Load i is token
    // i / U's group pair i % U (U pairs per half-warp per token).
    float* wsc = s_sc + warp * tpw * groups_per_slice;
    const int U = (groups_per_slice + 1) / 2;
    const unsigned kept = __ballot_sync(0xffffffffu, q >= 0);
    const unsigned kmask = K >= 32 ? 0xffffffffu : ((1u << K) - 1u);
    uint4 v[kPreload];
#pragma unroll
    for (int i = 0; i < kPreload; ++i) {
      const int tt = i / U, u = i - (i / U) * U;
      const int t = gw * tpw + tt;
      const int g = g0 + 2 * u + half;
      if (tt < tpw && t < T && g < g1 && ((kept >> (tt * K)) & kmask))
        v[i] = ld_stream(x + static_cast<size_t>(t) * (H / 8) + g * 16 + hl);
    }
#pragma unroll
    for (int i = 0; i < kPreload; ++i) {
      const int tt = i / U, u = i - (i / U) * U;
      if (tt >= tpw) continue;   // the same for the whole warp
      const int t = gw * tpw + tt;
      const int g = g0 + 2 * u + half;
      const bool on = t < T && g < g1 && ((kept >> (tt * K)) & kmask);
      uint2 codes;
      float scale;
      quantize_group(v[i], on, &codes, &scale);
      if (on) {
        const int* dq = wdest + tt * K;
        for (int k = 0; k < K; ++k) {
          const int qq = dq[k];
          if (qq >= 0) xq[static_cast<size_t>(qq) * (H / 8) + g * 16 + hl] = codes;
        }
        if (hl == 0) wsc[tt * groups_per_slice + (g - g0)] = scale;
      }
    }
    __syncwarp();
    // scales: lane i takes (route, group) pairs i, i + 32, ...
    const int ng = g1 - g0;
    for (int i = lane; i < tpw * K * ng; i += 32) {
      const int rt = i / ng, g = i - (i / ng) * ng;
      const int qq = wdest[rt];
      if (qq >= 0) xs[static_cast<size_t>(qq) * G + g0 + g] = wsc[(rt / K) * groups_per_slice + g];
    }
  } else {
    float* wsc = s_sc + warp * groups_per_slice;
    for (int tt = 0; tt < tpw; ++tt) {
      const int t = gw * tpw + tt;
      if (t >= T) break;
      const int* dq = wdest + tt * K;
      bool any = false;
      for (int k = 0; k < K; ++k) any |= dq[k] >= 0;
      if (!any) continue;
      const uint4* src = x + static_cast<size_t>(t) * (H / 8);
      // eight groups per pass: half-warp `half` takes groups gg + 2u + half
      for (int gg = g0; gg < g1; gg += 8) {
        uint4 v[4];
  #pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int g = gg + 2 * u + half;
          if (g < g1) v[u] = ld_stream(src + g * 16 + hl);
        }
  #pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int g = gg + 2 * u + half;
          const bool on = g < g1;
          uint2 codes;
          float scale;
          quantize_group(v[u], on, &codes, &scale);
          if (on) {
            for (int k = 0; k < K; ++k) {
              const int qq = dq[k];
              if (qq >= 0) xq[static_cast<size_t>(qq) * (H / 8) + g * 16 + hl] = codes;
            }
            if (hl == 0) wsc[g - g0] = scale;
          }
        }
      }
      __syncwarp();
      for (int k = 0; k < K; ++k) {
        const int qq = dq[k];
        if (qq < 0) continue;
        for (int g = g0 + lane; g < g1; g += 32) xs[static_cast<size_t>(qq) * G + g] = wsc[g - g0];
      }
      __syncwarp();
    }
  }
}

// Per-source fixed-slot dispatch ("DeepEP 架构与实现笔记", §9.5): expert e's
// R = W * mt rows are W ranges of mt slots, one per source rank, and route
// (t, k) of source rank r goes to slot r * mt + p, p its position among r's
// routes to e in ascending route id.  A slot follows from the source's own
// routes alone, so each block takes one source rank's tokens (blockIdx.x = r,
// blockIdx.y = column slice) and walks them in chunks of kDispatchWarps *
// (32 / K) tokens, with running per-expert positions in shared memory: no
// histogram or scan across blocks.  Routes whose position reaches mt are
// dropped.  Each (y = 0) block adds its clamped positions to counts[e] (the
// per-expert valid rows, zeroed by the launcher) and writes its column of
// seg_counts [E, W].
//
// kFp8: the same slots, with the quantisation fused as in route_scatter_fp8_kernel:
// each token row is quantised once (a half-warp per 128-group of the block's
// column slice of `slice` groups) and its e4m3 codes and scales are written to
// xq/xs at every kept slot; otherwise `slice` counts 16-byte vectors of BF16.
// kShort: at most eight tokens per warp and one 16-byte vector per lane and
// token (a slice of at most two groups, or 32 vectors); every token's load is
// then issued before the first store.  A separate instantiation: its eight
// preloaded vectors would double the loop form's registers.
template <typename IdT, bool kFp8, bool kShort>
__global__ void __launch_bounds__(kDispatchWarps * 32)
    route_source_slots_kernel(const uint4* __restrict__ x, const IdT* __restrict__ topk_idx,
                              int T, int H, int K, int E, int W, int mt,
                              const int32_t* __restrict__ rank_offsets, uint4* __restrict__ recv,
                              uint2* __restrict__ xq, float* __restrict__ xs,
                              int32_t* __restrict__ counts, int32_t* __restrict__ seg_counts,
                              int32_t* __restrict__ src_map, int32_t* dev_status, int slice) {
  extern __shared__ int smem[];
  int* s_cnt = smem;                        // [kDispatchWarps][E] routes per warp of a chunk
  int* s_dest = smem + kDispatchWarps * E;  // [kDispatchWarps][32]
  int* s_pos = s_dest + kDispatchWarps * 32;  // [E] next position of this source per expert
  float* s_sc = reinterpret_cast<float*>(s_pos + E);   // FP8: [kDispatchWarps][slice] scales
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tpw = 32 / K;
  const int per = (T + W - 1) / W;
  // this source rank's tokens, clamped to [0, T] whatever the offsets say
  const int t0 = max(0, min(T, rank_offsets ? rank_offsets[r] : r * per));
  const int t1 = max(t0, min(T, rank_offsets ? rank_offsets[r + 1] : (r + 1) * per));
  const int64_t R = static_cast<int64_t>(W) * mt;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_pos[e] = 0;
  const int nvec = H / 8;
  const int v0 = blockIdx.y * slice;
  const int v1 = min(nvec, v0 + slice);
  const int G = H / kGroup;
  const int g0 = blockIdx.y * slice;
  const int g1 = min(G, g0 + slice);
  const int half = lane >> 4, hl = lane & 15;
  int bad = 0;
  for (int c0 = t0; c0 < t1; c0 += kDispatchWarps * tpw) {
    for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();
    const int t = c0 + warp * tpw + lane / K;
    const int k = lane % K;
    const bool active = lane < tpw * K && t < t1;
    int e = -1;
    if (active) {
      const int64_t id = static_cast<int64_t>(topk_idx[static_cast<int64_t>(t) * K + k]);
      if (id >= 0 && id < E) e = static_cast<int>(id);
      else if (id != -1) bad = 1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int lane_rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = e >= 0 && lane == __ffs(peers) - 1;
    if (leader) s_cnt[warp * E + e] = __popc(peers);
    __syncthreads();
    int q = -1;
    if (e >= 0) {
      int p = s_pos[e] + lane_rank;
      for (int w = 0; w < warp; ++w) p += s_cnt[w * E + e];
      if (p < mt) q = static_cast<int>(e * R + static_cast<int64_t>(r) * mt + p);
    }
    if (blockIdx.y == 0 && active) src_map[static_cast<int64_t>(t) * K + k] = q;
    s_dest[warp * 32 + lane] = q;
    __syncthreads();
    if (leader) atomicAdd(&s_pos[e], __popc(peers));   // positions for the next chunk
    // payload: this warp's tokens, this block's column slice
    const int* wdest = s_dest + warp * 32;
    const int tbase = c0 + warp * tpw;
    if constexpr (kShort) {
      const unsigned kept = __ballot_sync(0xffffffffu, q >= 0);
      const unsigned kmask = K >= 32 ? 0xffffffffu : ((1u << K) - 1u);
      const int unit = kFp8 ? (g0 + half) * 16 + hl : v0 + lane;   // vector of the row
      const bool has = kFp8 ? g0 + half < g1 : v0 + lane < v1;
      uint4 a[8];
#pragma unroll
      for (int tt = 0; tt < 8; ++tt)
        if (tt < tpw && tbase + tt < t1 && has && ((kept >> (tt * K)) & kmask))
          a[tt] = ld_stream(x + static_cast<size_t>(tbase + tt) * nvec + unit);
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        if (tt >= tpw || tbase + tt >= t1) break;   // the same for the whole warp
        if (!((kept >> (tt * K)) & kmask)) continue;
        const int* dq = wdest + tt * K;
        if constexpr (kFp8) {
          uint2 codes;
          float scale;
          quantize_group(a[tt], has, &codes, &scale);
          if (has) {
            const int g = g0 + half;
            for (int kk = 0; kk < K; ++kk) {
              const int qq = dq[kk];
              if (qq < 0) continue;
              xq[static_cast<size_t>(qq) * (H / 8) + unit] = codes;
              if (hl == 0) xs[static_cast<size_t>(qq) * G + g] = scale;
            }
          }
        } else if (has) {
          for (int kk = 0; kk < K; ++kk) {
            const int qq = dq[kk];
            if (qq >= 0) recv[static_cast<size_t>(qq) * nvec + unit] = a[tt];
          }
        }
      }
    } else {
      for (int tt = 0; tt < tpw; ++tt) {
        const int tok = c0 + warp * tpw + tt;
        if (tok >= t1) break;
        const int* dq = wdest + tt * K;
        bool any = false;
        for (int kk = 0; kk < K; ++kk) any |= dq[kk] >= 0;
        if (!any) continue;
        const uint4* src = x + static_cast<size_t>(tok) * nvec;
        if constexpr (kFp8) {
          float* wsc = s_sc + warp * slice;
          // eight groups per pass: half-warp `half` takes groups gg + 2u + half
          for (int gg = g0; gg < g1; gg += 8) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int g = gg + 2 * u + half;
              if (g < g1) v[u] = ld_stream(src + g * 16 + hl);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int g = gg + 2 * u + half;
              const bool on = g < g1;
              uint2 codes;
              float scale;
              quantize_group(v[u], on, &codes, &scale);
              if (on) {
                for (int kk = 0; kk < K; ++kk) {
                  const int qq = dq[kk];
                  if (qq >= 0) xq[static_cast<size_t>(qq) * (H / 8) + g * 16 + hl] = codes;
                }
                if (hl == 0) wsc[g - g0] = scale;
              }
            }
          }
          __syncwarp();
          for (int kk = 0; kk < K; ++kk) {
            const int qq = dq[kk];
            if (qq < 0) continue;
            for (int g = g0 + lane; g < g1; g += 32) xs[static_cast<size_t>(qq) * G + g] = wsc[g - g0];
          }
          __syncwarp();
        } else {
          for (int v = v0 + lane; v < v1; v += 32 * 8) {
            uint4 a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              if (v + 32 * u < v1) a[u] = ld_stream(src + v + 32 * u);
            for (int kk = 0; kk < K; ++kk) {
              const int qq = dq[kk];
              if (qq < 0) continue;
              uint4* dst = recv + static_cast<size_t>(qq) * nvec;
#pragma unroll
              for (int u = 0; u < 8; ++u)
                if (v + 32 * u < v1) dst[v + 32 * u] = a[u];
            }
          }
        }
      }
    }
  }
  bad = __syncthreads_or(bad);
  if (blockIdx.y != 0) return;
  int dropped = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int n = s_pos[e];
    const int kept = min(n, mt);
    seg_counts[static_cast<size_t>(e) * W + r] = kept;
    if (kept) atomicAdd(&counts[e], kept);
    dropped += n - kept;
  }
  if (dropped) {
    atomicAdd(dev_status + 1, dropped);
    atomicOr(dev_status, kDevCapacityDropped);
  }
  if (bad && threadIdx.x == 0) atomicOr(dev_status, kDevBadExpertId);
}

}  // namespace

namespace {

// Column slices per token row when there are too few tokens to keep enough
// warps in flight; a slice keeps at least `min_units` units.
int row_slices(int nblocks, int units, int min_units, int sm_count) {
  const int target_warps = sm_count * 48;
  int hsplit = (target_warps + nblocks * kDispatchWarps - 1) / (nblocks * kDispatchWarps);
  return max(1, min(hsplit, units / min_units));
}

// Dynamic shared memory above the 48 KB default needs an opt-in per kernel.
template <typename Kernel>
cudaError_t allow_smem(Kernel k, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

bool single_pass(int T, int K) {
  return T > 0 && static_cast<int64_t>(T) * K <= kSinglePassRoutes;
}

template <typename IdT>
cudaError_t dispatch_impl(const void* x, const IdT* topk_idx, int T, int H, int K, int E,
                          RowLayout rl, void* recv, int32_t* counts, int32_t* src_map,
                          int32_t* dev_status, int32_t* hist, int sm_count, cudaStream_t s) {
  const int R = rl.R;
  const int nblocks = dispatch_blocks(T, K);
  const int nvec = H / 8;
  const bool one = single_pass(T, K);
  cudaError_t err;
  if (!one) {
    err = cudaMemsetAsync(dev_status, 0, 2 * sizeof(int32_t), s);
    if (err != cudaSuccess) return err;
    if (nblocks > 0) {
      route_hist_kernel<IdT><<<nblocks, kDispatchWarps * 32, E * sizeof(int), s>>>(
          topk_idx, T, K, E, nblocks, hist, dev_status);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    route_scan_kernel<<<E, kScanThreads, 0, s>>>(hist, nblocks, R, counts, dev_status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (nblocks == 0) return cudaSuccess;
  }
  int hsplit = row_slices(nblocks, nvec, 32, sm_count);
  const int vec_per_slice = (nvec + hsplit - 1) / hsplit;
  hsplit = (nvec + vec_per_slice - 1) / vec_per_slice;
  const size_t smem = (kDispatchWarps * E + kDispatchWarps * 32 + 3 * E + 1) * sizeof(int);
  const dim3 grid(nblocks, hsplit);
  const int need = (vec_per_slice + 31) / 32 * (32 / K);
  const int depth = need <= 8 ? 8 : (need <= 16 ? 16 : 0);
  auto kernel = one ? (depth == 8 ? route_scatter_kernel<IdT, true, 8>
                       : depth == 16 ? route_scatter_kernel<IdT, true, 16> : route_scatter_kernel<IdT, true, 0>)
                    : (depth == 8 ? route_scatter_kernel<IdT, false, 8>
                       : depth == 16 ? route_scatter_kernel<IdT, false, 16> : route_scatter_kernel<IdT, false, 0>);
  if ((err = allow_smem(kernel, smem)) != cudaSuccess) return err;
  kernel<<<grid, kDispatchWarps * 32, smem, s>>>(static_cast<const uint4*>(x), topk_idx, T, H, K, E,
                                                 rl, nblocks, hist, counts, static_cast<uint4*>(recv),
                                                 src_map, dev_status, vec_per_slice);
  return cudaGetLastError();
}
}  // namespace

namespace {
// xq == nullptr: BF16 rows into recv; else e4m3 codes and scales into xq/xs.
template <typename IdT>
cudaError_t source_slots_impl(const void* x, const IdT* topk_idx, int T, int H, int K, int E,
                              int W, int mt, const int32_t* rank_offsets, void* recv,
                              uint8_t* xq, float* xs, int32_t* counts, int32_t* seg_counts,
                              int32_t* src_map, int32_t* dev_status, int sm_count,
                              cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(dev_status, 0, 2 * sizeof(int32_t), s);
  if (err == cudaSuccess) err = cudaMemsetAsync(counts, 0, E * sizeof(int32_t), s);
  if (err != cudaSuccess) return err;
  const bool fp8 = xq != nullptr;
  // column slices: 16-byte BF16 vectors (at least 32), or whole 128-groups (at least two)
  const int units = fp8 ? H / kGroup : H / 8;
  int hsplit = row_slices(W, units, fp8 ? 2 : 32, sm_count);
  const int per_slice = (units + hsplit - 1) / hsplit;
  hsplit = (units + per_slice - 1) / per_slice;
  const size_t smem = (kDispatchWarps * E + kDispatchWarps * 32 + E) * sizeof(int) +
                      (fp8 ? kDispatchWarps * per_slice * sizeof(float) : 0);
  const bool short_slice = 32 / K <= 8 && per_slice <= (fp8 ? 2 : 32);
  auto kernel = fp8 ? (short_slice ? route_source_slots_kernel<IdT, true, true>
                                   : route_source_slots_kernel<IdT, true, false>)
                    : (short_slice ? route_source_slots_kernel<IdT, false, true>
                                   : route_source_slots_kernel<IdT, false, false>);
  if ((err = allow_smem(kernel, smem)) != cudaSuccess) return err;
  kernel<<<dim3(W, hsplit), kDispatchWarps * 32, smem, s>>>(
      static_cast<const uint4*>(x), topk_idx, T, H, K, E, W, mt, rank_offsets,
      static_cast<uint4*>(recv), reinterpret_cast<uint2*>(xq), xs, counts, seg_counts, src_map,
      dev_status, per_slice);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_dispatch_source_slots(const void* x, const void* topk_idx, int idx_bits, int T,
                                         int H, int K, int E, int W, int mt,
                                         const int32_t* rank_offsets, void* recv, uint8_t* xq,
                                         float* xs, int32_t* counts, int32_t* seg_counts,
                                         int32_t* src_map, int32_t* dev_status, int sm_count,
                                         cudaStream_t s) {
  if (idx_bits == 32)
    return source_slots_impl(x, static_cast<const int32_t*>(topk_idx), T, H, K, E, W, mt,
                             rank_offsets, recv, xq, xs, counts, seg_counts, src_map, dev_status,
                             sm_count, s);
  return source_slots_impl(x, static_cast<const int64_t*>(topk_idx), T, H, K, E, W, mt,
                           rank_offsets, recv, xq, xs, counts, seg_counts, src_map, dev_status,
                           sm_count, s);
}

cudaError_t launch_dispatch(const void* x, const void* topk_idx, int idx_bits, int T, int H, int K,
                            int E, RowLayout rl, void* recv, int32_t* counts, int32_t* src_map,
                            int32_t* dev_status, int32_t* hist, int sm_count, cudaStream_t s) {
  if (idx_bits == 32)
    return dispatch_impl(x, static_cast<const int32_t*>(topk_idx), T, H, K, E, rl, recv, counts,
                         src_map, dev_status, hist, sm_count, s);
  return dispatch_impl(x, static_cast<const int64_t*>(topk_idx), T, H, K, E, rl, recv, counts,
                       src_map, dev_status, hist, sm_count, s);
}

}  // namespace moe

namespace moe {

namespace {
template <typename IdT>
cudaError_t dispatch_quant_impl(const void* x, const IdT* topk_idx, int T, int H, int K, int E,
                                RowLayout rl, uint8_t* xq, float* xs, int32_t* counts,
                                int32_t* src_map, int32_t* dev_status, int32_t* hist,
                                int sm_count, cudaStream_t s) {
  const int nblocks = dispatch_blocks(T, K);
  const bool one = single_pass(T, K);
  cudaError_t err;
  if (!one) {
    err = cudaMemsetAsync(dev_status, 0, 2 * sizeof(int32_t), s);
    if (err != cudaSuccess) return err;
    if (nblocks > 0) {
      route_hist_kernel<IdT><<<nblocks, kDispatchWarps * 32, E * sizeof(int), s>>>(
          topk_idx, T, K, E, nblocks, hist, dev_status);
      if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    route_scan_kernel<<<E, kScanThreads, 0, s>>>(hist, nblocks, rl.R, counts, dev_status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (nblocks == 0) return cudaSuccess;
  }
  // Slices of two or more whole 128-groups when there are too few tokens to
  // fill the GPU (one-group slices would leave a half-warp idle).
  const int G = H / kGroup;
  int hsplit = row_slices(nblocks, G, 2, sm_count);
  const int gps = (G + hsplit - 1) / hsplit;
  hsplit = (G + gps - 1) / gps;
  const int need = (gps + 1) / 2 * (32 / K);   // loads per lane to preload a warp's slices
  const bool one_wave = static_cast<long long>(nblocks) * hsplit <= sm_count;
  const int depth = need <= 8 ? 8 : (need <= 16 && one_wave ? 16 : 0);
  const bool pre = depth > 0;
  const size_t smem = (kDispatchWarps * E + kDispatchWarps * 32 + 3 * E + 1) * sizeof(int) +
                      kDispatchWarps * (pre ? 32 / K : 1) * gps * sizeof(float);
  const dim3 grid(nblocks, hsplit);
  auto kernel = one ? (depth == 16 ? route_scatter_fp8_kernel<IdT, true, 16>
                       : depth == 8 ? route_scatter_fp8_kernel<IdT, true, 8>
                                    : route_scatter_fp8_kernel<IdT, true, 0>)
                    : (depth == 16 ? route_scatter_fp8_kernel<IdT, false, 16>
                       : depth == 8 ? route_scatter_fp8_kernel<IdT, false, 8>
                                    : route_scatter_fp8_kernel<IdT, false, 0>);
  if ((err = allow_smem(kernel, smem)) != cudaSuccess) return err;
  kernel<<<grid, kDispatchWarps * 32, smem, s>>>(
      static_cast<const uint4*>(x), topk_idx, T, H, K, E, rl, nblocks, hist, counts,
      reinterpret_cast<uint2*>(xq), xs, src_map, dev_status, gps);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_dispatch_quant(const void* x, const void* topk_idx, int idx_bits, int T, int H,
                                  int K, int E, RowLayout rl, uint8_t* xq, float* xs,
                                  int32_t* counts, int32_t* src_map, int32_t* dev_status,
                                  int32_t* hist, int sm_count, cudaStream_t s) {
  if (idx_bits == 32)
    return dispatch_quant_impl(x, static_cast<const int32_t*>(topk_idx), T, H, K, E, rl, xq, xs,
                               counts, src_map, dev_status, hist, sm_count, s);
  return dispatch_quant_impl(x, static_cast<const int64_t*>(topk_idx), T, H, K, E, rl, xq, xs,
                             counts, src_map, dev_status, hist, sm_count, s);
}

}  // namespace moe
