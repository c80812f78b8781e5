// Combine: the weighted gather back into token order.
//
// "SGLang、NCCL 与 MoE EP", §3.2 (合对): the output of route (t, k), found at
// flat row q = src_map[t, k] of the expert-major output, is multiplied by its
// router weight topk_w[t, k] exactly once and summed into y[t]; §1.1: the
// weight multiplies the expert output, never its input.  "DeepEP 架构与实现笔记",
// §9.6: the weighted reduce happens inside the combine kernel.
//
// One warp per token (and column slice): the kept routes' rows are gathered
// with 16-byte loads, eight routes in flight per lane, and accumulated in fp32
// in ascending k -- acc = acc + w * v, product and sum each rounded to fp32 --
// then rounded to BF16 (nearest even).  Routes with q = -1 are skipped.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const uint4* __restrict__ out, const int32_t* __restrict__ src_map,
                   const float* __restrict__ topk_w, int T, int H, int K, int64_t rows,
                   uint4* __restrict__ y, int vec_per_slice) {
  __shared__ int s_q[kCombineWarps][32];
  __shared__ float s_w[kCombineWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kCombineWarps + warp;
  if (t >= T) return;
  int q = -1;
  float w = 0.f;
  if (lane < K) {
    q = src_map[static_cast<int64_t>(t) * K + lane];
    w = topk_w[static_cast<int64_t>(t) * K + lane];
    if (q >= rows) q = -1;  // not a row of the output buffer: treated as no route
  }
  // Compact the kept routes, keeping ascending k.
  const unsigned kept = __ballot_sync(0xffffffffu, q >= 0);
  const int nk = __popc(kept);
  if (q >= 0) {
    const int pos = __popc(kept & ((1u << lane) - 1u));
    s_q[warp][pos] = q;
    s_w[warp][pos] = w;
  }
  __syncwarp();
  const int nvec = H / 8;
  const int v0 = blockIdx.y * vec_per_slice;
  const int v1 = min(nvec, v0 + vec_per_slice);
  uint4* dst = y + static_cast<size_t>(t) * nvec;
  for (int v = v0 + lane; v < v1; v += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int k0 = 0; k0 < nk; k0 += 8) {
      uint4 raw[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (k0 + j < nk) raw[j] = ld_stream(out + static_cast<size_t>(s_q[warp][k0 + j]) * nvec + v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (k0 + j < nk) {
          const float wk = s_w[warp][k0 + j];
          float f[8];
          bf16x8_to_f32(raw[j], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(wk, f[i]));
        }
      }
    }
    uint4 o;
    o.x = pack_bf16x2_rn(acc[0], acc[1]);
    o.y = pack_bf16x2_rn(acc[2], acc[3]);
    o.z = pack_bf16x2_rn(acc[4], acc[5]);
    o.w = pack_bf16x2_rn(acc[6], acc[7]);
    dst[v] = o;
  }
}

}  // namespace

cudaError_t launch_combine(const void* out, const int32_t* src_map, const float* topk_w, int T,
                           int H, int K, int64_t rows, void* y, int sm_count, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int nblocks = (T + kCombineWarps - 1) / kCombineWarps;
  const int nvec = H / 8;
  const int target_warps = sm_count * 48;
  int hsplit = (target_warps + nblocks * kCombineWarps - 1) / (nblocks * kCombineWarps);
  hsplit = max(1, min(hsplit, nvec / 32));
  const int vec_per_slice = (nvec + hsplit - 1) / hsplit;
  hsplit = (nvec + vec_per_slice - 1) / vec_per_slice;
  combine_kernel<<<dim3(nblocks, hsplit), kCombineWarps * 32, 0, s>>>(
      static_cast<const uint4*>(out), src_map, topk_w, T, H, K, rows, static_cast<uint4*>(y),
      vec_per_slice);
  return cudaGetLastError();
}

}  // namespace moe
