// Per-token FP8 quantisation of the valid receive rows.
//
// "SGLang、NCCL 与 MoE EP", §2.3.5: after receive, the valid rows of recv
// [L, M, H] are quantised to FP8 with one fp32 scale per row per 128 hidden
// elements; rows past counts[e] are never touched.  The rule is the one of
// "DeepEP 架构与实现笔记", §11: amax = max(max|v|, 1e-4), codes =
// e4m3(v * (448 / amax)), scale = amax / 448, computed here in fp32 with IEEE
// division and a round-to-nearest-even, saturating e4m3 conversion.
//
// Work is split into row blocks of 8 valid rows of one expert, one row per
// warp: at decode-sized layers (tens of rows per expert) blocks of 32 rows left
// most SMs idle and each warp walking four rows one load round trip after
// another (8-row blocks: decode 29 -> 15 us, prefill -11 %, large -1 %).
// A persistent grid walks the row blocks; each warp takes whole rows, each
// half-warp one 128-element group (16 lanes x 8 BF16 = one 16-byte load per
// lane), so the group amax is a 4-step shuffle reduction.  Scales are staged in shared
// memory and written row-major ([rows, H/128], as on the pages), the block's
// rows as one contiguous run.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace moe {
namespace {

constexpr int kQuantWarps = 8;
constexpr int kRowsPerBlock = 8;

// kPack (per-source slots only): the slot rows already hold e4m3 codes `pq` and
// scales `ps` (the dispatch quantised them); each packed row copies its slot's.
template <bool kPack>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_kernel(const uint4* __restrict__ recv, const int32_t* __restrict__ counts, int E,
                    RowLayout rl, int H, uint2* __restrict__ xq, float* __restrict__ xs,
                    const uint4* __restrict__ pq, const float* __restrict__ ps) {
  extern __shared__ int smem[];
  int* s_start = smem;               // [E + 1] prefix of row blocks
  int* s_cnt = smem + E + 1;         // [E]
  int* s_rows = smem + 2 * E + 1;    // [E + 1] packed row bases
  const int G = H / kGroup;
  float* s_scale = reinterpret_cast<float*>(smem + 3 * E + 2);  // [G][kRowsPerBlock]
  int* s_rp = reinterpret_cast<int*>(s_scale + G * kRowsPerBlock);  // per-source: [W + 1]
  const int R = rl.R;
  // Per-source slots: expert e's valid rows are packed to rows [0, c_e) of its
  // range of xq/xs, in slot order; s_rp holds the current expert's prefix of
  // valid rows over its source ranges.
  const int W = rl.seg ? R / rl.seg : 0;
  if (rl.seg) source_slot_totals(rl.seg_counts, E, R, rl.seg, s_cnt);
  expert_prefix(rl.seg ? s_cnt : counts, E, R, kRowsPerBlock, 1, s_start, s_cnt);
  if (rl.packed) expert_prefix(counts, E, R, 1, 1, s_rows, nullptr);
  const int nvec = H / 8;
  const int total = s_start[E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  int rp_e = -1;
  for (int b = blockIdx.x; b < total; b += gridDim.x) {
    const int e = find_expert(s_start, E, b);
    if (rl.seg && e != rp_e) {   // the same for the whole block
      if (warp == 0) {
        int carry = 0;
        if (lane == 0) s_rp[0] = 0;
        for (int r0 = 0; r0 < W; r0 += 32) {
          const int r = r0 + lane;
          int v = r < W ? min(max(rl.seg_counts[static_cast<size_t>(e) * W + r], 0), rl.seg) : 0;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
          }
          if (r < W) s_rp[r + 1] = carry + v;
          carry += __shfl_sync(0xffffffffu, v, 31);
        }
      }
      __syncthreads();
      rp_e = e;
    }
    const int row0 = (b - s_start[e]) * kRowsPerBlock;
    const int64_t base = (rl.packed ? static_cast<int64_t>(s_rows[e]) : static_cast<int64_t>(e) * R) + row0;
    // rows of the block: valid rows of e, and never past the buffer
    const int nrows = static_cast<int>(
        min(static_cast<int64_t>(min(kRowsPerBlock, s_cnt[e] - row0)), rl.rows - base));
    if (nrows <= 0) continue;
    for (int r = warp; r < nrows; r += kQuantWarps) {
      const size_t row = static_cast<size_t>(base) + r;
      size_t src_row = row;
      if (rl.seg) {
        // packed row j of e comes from source range q: s_rp[q] <= j < s_rp[q + 1]
        const int j = row0 + r;
        int lo = 0, hi = W - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_rp[mid] <= j) lo = mid; else hi = mid - 1;
        }
        const int slot = lo * rl.seg + (j - s_rp[lo]);
        src_row = static_cast<size_t>(e) * R + slot;
        if (lane == 0) rl.slot_of[row] = slot;
      }
      if constexpr (kPack) {
        const uint4* csrc = pq + src_row * (H / 16);
        uint4* cdst = reinterpret_cast<uint4*>(xq) + row * (H / 16);
        for (int i = lane; i < H / 16; i += 32) cdst[i] = ld_stream(csrc + i);
        for (int g = lane; g < G; g += 32) s_scale[g * kRowsPerBlock + r] = ps[src_row * G + g];
        continue;
      }
      const uint4* src = recv + src_row * nvec;
      uint2* dst = xq + row * (H / 8);
      // Four pairs of groups per pass: every lane has four 16-byte loads in
      // flight before the reductions.  (Sixteen per pass, a 4096-wide row in
      // one round trip, halved the resident blocks and was slower at every
      // layer shape: decode 14.1 vs 12.8 us, large 0.62 vs 0.47 ms.)
      for (int g0 = 0; g0 < G; g0 += 8) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int g = g0 + 2 * u + half;
          if (g < G) v[u] = ld_stream(src + g * 16 + hl);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int g = g0 + 2 * u + half;
          const bool on = g < G;
          float f[8];
          float amax = 0.f;
          if (on) {
            bf16x8_to_f32(v[u], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
          }
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          if (on) {
            float mult, scale;
            fp8_group_scale(amax, &mult, &scale);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              lo |= static_cast<uint32_t>(pack_e4m3x2(__fmul_rn(f[2 * i], mult),
                                                      __fmul_rn(f[2 * i + 1], mult)))
                    << (16 * i);
              hi |= static_cast<uint32_t>(pack_e4m3x2(__fmul_rn(f[4 + 2 * i], mult),
                                                      __fmul_rn(f[5 + 2 * i], mult)))
                    << (16 * i);
            }
            dst[g * 16 + hl] = make_uint2(lo, hi);
            if (hl == 0) s_scale[g * kRowsPerBlock + r] = scale;
          }
        }
      }
    }
    __syncthreads();
    // scales are stored row-major [rows, G]: the block's rows are one contiguous run
    for (int i = threadIdx.x; i < G * nrows; i += blockDim.x) {
      const int r = i / G, g = i % G;
      xs[static_cast<size_t>(base) * G + i] = s_scale[g * kRowsPerBlock + r];
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_quantize(const void* recv, const int32_t* counts, int E, RowLayout rl, int H,
                            uint8_t* xq, float* xs, int sm_count, cudaStream_t s,
                            const uint8_t* pq, const float* ps) {
  const int R = rl.R;
  const int G = H / kGroup;
  const size_t smem = (3 * E + 2) * sizeof(int) + G * kRowsPerBlock * sizeof(float) +
                      (rl.seg ? (R / rl.seg + 1) * sizeof(int) : 0);
  // Upper bound of row blocks; the kernel walks the true count read from device memory.
  const long long max_blocks = static_cast<long long>(E) * ((R + kRowsPerBlock - 1) / kRowsPerBlock);
  const int grid = static_cast<int>(std::min<long long>(max_blocks, sm_count * 8LL));
  if (grid <= 0) return cudaSuccess;
  auto kernel = pq != nullptr ? quantize_kernel<true> : quantize_kernel<false>;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  kernel<<<grid, kQuantWarps * 32, smem, s>>>(static_cast<const uint4*>(recv), counts, E, rl, H,
                                              reinterpret_cast<uint2*>(xq), xs,
                                              reinterpret_cast<const uint4*>(pq), ps);
  return cudaGetLastError();
}

}  // namespace moe
