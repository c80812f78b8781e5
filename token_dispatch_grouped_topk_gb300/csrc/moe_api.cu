// The C ABI of include/moe.h: argument validation, workspace carving and the
// launch sequence of each call.  No call allocates, synchronises or reads
// device memory on the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_info_mu;
DeviceInfo g_info[kMaxDevices];
bool g_info_ok[kMaxDevices];

constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

const DeviceInfo* current_device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_info_mu);
  if (!g_info_ok[dev]) {
    DeviceInfo d{};
    int smem = 0;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return nullptr;
    d.smem_optin = static_cast<size_t>(smem);
    g_info[dev] = d;
    g_info_ok[dev] = true;
  }
  return &g_info[dev];
}

namespace {

// The kernels are built for sm_103a only.
moe_status check_device(const DeviceInfo** out) {
  const DeviceInfo* d = current_device_info();
  if (d == nullptr) return MOE_ERR_CUDA;
  if (d->cc_major != 10 || d->cc_minor != 3) return MOE_ERR_UNSUPPORTED;
  *out = d;
  return MOE_OK;
}

bool valid_hidden(int H) { return H > 0 && H % 128 == 0 && H <= 16384; }
bool valid_experts(int E, int R) {
  return E >= 1 && E <= 1024 && R >= 1 && static_cast<int64_t>(E) * R <= (int64_t{1} << 30);
}

struct ComputeWorkspace {
  size_t xq, xs, zq, zs, sync, sync_ints, slot, total;
};

bool valid_rows(int64_t rows) { return rows >= 1 && rows <= (int64_t{1} << 30); }

// FP8 activations and their scales, Z and its scales, for `rows` buffer rows.
ComputeWorkspace compute_workspace_rows(int64_t rows_i, int H, int I) {
  ComputeWorkspace w{};
  const size_t rows = static_cast<size_t>(rows_i);
  size_t off = 0;
  w.xq = off;
  off = align_up(off + rows * H, 256);
  w.xs = off;
  off = align_up(off + rows * (H / 128) * sizeof(float), 256);
  w.zq = off;
  off = align_up(off + rows * I, 256);
  w.zs = off;
  off = align_up(off + rows * (I / 128) * sizeof(float), 256);
  // Scratch of the fused GEMM launch: a tile ticket and one completion count
  // per 128-row block (at most ceil(rows / 128) plus one partial block for each
  // of up to 1024 experts).
  w.sync = off;
  w.sync_ints = 1 + (rows + 127) / 128 + 1024;
  off = align_up(off + w.sync_ints * sizeof(int), 256);
  // Per-source slot layout: the slot row of each packed row (int32 per row).
  w.slot = off;
  off = align_up(off + rows * sizeof(int32_t), 256);
  w.total = off;
  return w;
}
ComputeWorkspace compute_workspace(int E, int R, int H, int I) {
  return compute_workspace_rows(static_cast<int64_t>(E) * R, H, I);
}

moe_status from_cuda(cudaError_t e);

// Both GEMMs, as one launch or as the gate/up launch then the down launch
// (MOE_GEMM_ONE_LAUNCH / MOE_GEMM_TWO_LAUNCHES, else by the tile count).
cudaError_t run_gemms(const uint8_t* xq, const float* xs, const int32_t* counts, int E, RowLayout rl,
                      int H, int I, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                      const float* w2_scale, uint8_t* zq, float* zs, void* out, int* sync,
                      size_t sync_ints, int32_t* dev_status, int sm_count, cudaStream_t s,
                      int flags) {
  const int inter = (flags & MOE_W13_INTERLEAVED) ? 1 : 0;
  const bool one = (flags & MOE_GEMM_ONE_LAUNCH)     ? true
                   : (flags & MOE_GEMM_TWO_LAUNCHES) ? false
                                                     : gemm_prefer_one_launch(E, rl, I, sm_count);
  // MOE_GEMM_MAX_CTAS(n): the persistent grids take at most n SMs
  const int cap = (flags >> 16) & 0x7FFF;
  const int grid = cap > 0 ? std::min(cap, sm_count) : sm_count;
  if (one)
    return launch_gemm_gateup_down(xq, xs, counts, E, rl, H, I, w13, w13_scale, w2, w2_scale, zq,
                                   zs, out, sync, sync_ints, dev_status, grid, s, inter);
  cudaError_t err = launch_gemm_gateup(xq, xs, counts, E, rl, H, I, w13, w13_scale, zq, zs,
                                       dev_status, grid, s, inter);
  if (err != cudaSuccess) return err;
  return launch_gemm_down(zq, zs, counts, E, rl, H, I, w2, w2_scale, out, dev_status, grid, s);
}

bool valid_gemm_flags(int flags) {
  const int known = MOE_W13_INTERLEAVED | MOE_GEMM_ONE_LAUNCH | MOE_GEMM_TWO_LAUNCHES |
                    MOE_GEMM_MAX_CTAS(0x7FFF);
  return (flags & ~known) == 0 &&
         !((flags & MOE_GEMM_ONE_LAUNCH) && (flags & MOE_GEMM_TWO_LAUNCHES));
}


// The expert compute on a carved workspace: quantisation (or, with pq/ps, the
// packing of per-source FP8 slots), then both GEMMs.
moe_status expert_compute_impl(const void* recv, const int32_t* counts, int E, RowLayout rl, int H,
                               int I, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                               const float* w2_scale, void* out, int32_t* dev_status, void* workspace,
                               const ComputeWorkspace& w, int sm_count, cudaStream_t s,
                               int flags = 0, const uint8_t* pq = nullptr,
                               const float* ps = nullptr) {
  auto* ws = static_cast<uint8_t*>(workspace);
  uint8_t* xq = ws + w.xq;
  float* xs = reinterpret_cast<float*>(ws + w.xs);
  uint8_t* zq = ws + w.zq;
  float* zs = reinterpret_cast<float*>(ws + w.zs);
  int* sync = reinterpret_cast<int*>(ws + w.sync);
  cudaError_t err = launch_quantize(recv, counts, E, rl, H, xq, xs, sm_count, s, pq, ps);
  if (err == cudaSuccess)
    err = run_gemms(xq, xs, counts, E, rl, H, I, w13, w13_scale, w2, w2_scale, zq, zs, out, sync,
                    w.sync_ints, dev_status, sm_count, s, flags);
  return from_cuda(err);
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return 1; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
  }
  return "MOE_ERR_UNKNOWN";
}

size_t moe_dispatch_workspace_size(int T, int K, int E) {
  if (T < 0 || K < 1 || K > 32 || E < 1) return 0;
  const size_t nb = static_cast<size_t>(dispatch_blocks64(T, K));
  return align_up(std::max<size_t>(nb * E * sizeof(int32_t), 1), 256);
}

moe_status moe_dispatch_ex(const void* x, const void* topk_idx, int idx_bits, const float* topk_w,
                           int T, int H, int K, int E, int R, int64_t rows, void* recv,
                           int32_t* counts, int32_t* src_map, int32_t* dev_status,
                           void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  (void)topk_w;  // router weights stay at the source; combine reads them
  if (T < 0 || !valid_hidden(H) || !valid_experts(E, R) || K < 1 || K > 32 || K > E)
    return MOE_ERR_INVALID_ARG;
  if (idx_bits != 32 && idx_bits != 64) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || dev_status == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || topk_idx == nullptr || recv == nullptr || src_map == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(x) || !aligned16(recv))) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * K > (int64_t{1} << 31) - 1) return MOE_ERR_INVALID_ARG;
  RowLayout rl = padded_rows(E, R);
  if (rows != 0) {
    // packed: every kept route must have a row, at most min(T*K, E*R) of them
    const int64_t need_rows =
        std::min<int64_t>(static_cast<int64_t>(T) * K, static_cast<int64_t>(E) * R);
    if (!valid_rows(rows) || rows < need_rows) return MOE_ERR_INVALID_ARG;
    rl = RowLayout{R, 1, rows};
  }
  const size_t need = moe_dispatch_workspace_size(T, K, E);
  if (workspace == nullptr || workspace_bytes < need) return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_dispatch(x, topk_idx, idx_bits, T, H, K, E, rl, recv, counts, src_map,
                                   dev_status, static_cast<int32_t*>(workspace), dev->sm_count,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch(const void* x, const int64_t* topk_idx, const float* topk_w, int T, int H,
                        int K, int E, int R, void* recv, int32_t* counts, int32_t* src_map,
                        int32_t* dev_status, void* workspace, size_t workspace_bytes,
                        moe_stream_t stream) {
  return moe_dispatch_ex(x, topk_idx, 64, topk_w, T, H, K, E, R, 0, recv, counts, src_map,
                         dev_status, workspace, workspace_bytes, stream);
}

moe_status moe_dispatch_packed(const void* x, const int64_t* topk_idx, const float* topk_w, int T,
                               int H, int K, int E, int R, int64_t rows, void* recv,
                               int32_t* counts, int32_t* src_map, int32_t* dev_status,
                               void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (rows == 0) return MOE_ERR_INVALID_ARG;
  return moe_dispatch_ex(x, topk_idx, 64, topk_w, T, H, K, E, R, rows, recv, counts, src_map,
                         dev_status, workspace, workspace_bytes, stream);
}

namespace {
// Host checks and launch of the per-source fixed-slot dispatch: BF16 rows into
// recv, or (fp8) e4m3 codes and scales into xq/xs.
moe_status source_slots_dispatch(bool fp8, const void* x, const void* topk_idx, int idx_bits,
                                 int T, int H, int K, int E, int L, int max_tokens,
                                 const int32_t* rank_offsets, void* recv, uint8_t* xq, float* xs,
                                 int32_t* counts, int32_t* seg_counts, int32_t* src_map,
                                 int32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || !valid_hidden(H) || K < 1 || K > 32 || L < 1 || E % L != 0 || K > E ||
      max_tokens < 1)
    return MOE_ERR_INVALID_ARG;
  const int W = E / L;
  if (!valid_experts(E, static_cast<int>(std::min<int64_t>(int64_t{W} * max_tokens, INT32_MAX))) ||
      int64_t{W} * max_tokens > (int64_t{1} << 30))
    return MOE_ERR_INVALID_ARG;
  if (idx_bits != 32 && idx_bits != 64) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || seg_counts == nullptr || dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || topk_idx == nullptr || src_map == nullptr ||
                (fp8 ? (xq == nullptr || xs == nullptr) : recv == nullptr)))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(x) || (!fp8 && !aligned16(recv)) ||
                (fp8 && (reinterpret_cast<uintptr_t>(xq) & 7u) != 0)))
    return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * K > (int64_t{1} << 31) - 1) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_dispatch_source_slots(
      x, topk_idx, idx_bits, T, H, K, E, W, max_tokens, rank_offsets, fp8 ? nullptr : recv,
      fp8 ? xq : nullptr, fp8 ? xs : nullptr, counts, seg_counts, src_map, dev_status,
      dev->sm_count, reinterpret_cast<cudaStream_t>(stream)));
}

// Host checks of the per-source expert compute; then the quantisation (recv
// BF16) or the packing (xq/xs e4m3 slots) and both GEMMs on the packed rows.
moe_status source_slots_compute(const void* recv, const uint8_t* xq_slots, const float* xs_slots,
                                const int32_t* seg_counts, int E, int L, int max_tokens, int H,
                                int I, const uint8_t* w13, const float* w13_scale,
                                const uint8_t* w2, const float* w2_scale, void* out,
                                int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                int flags, moe_stream_t stream) {
  if (L < 1 || E % L != 0 || max_tokens < 1 || !valid_hidden(H) || !valid_hidden(I))
    return MOE_ERR_INVALID_ARG;
  const int64_t R64 = int64_t{E / L} * max_tokens;
  if (R64 > (int64_t{1} << 30) || !valid_experts(E, static_cast<int>(R64)))
    return MOE_ERR_INVALID_ARG;
  const int R = static_cast<int>(R64);
  if (!valid_gemm_flags(flags)) return MOE_ERR_INVALID_ARG;
  const bool fp8 = recv == nullptr;
  if ((fp8 && (xq_slots == nullptr || xs_slots == nullptr)) || seg_counts == nullptr ||
      w13 == nullptr || w13_scale == nullptr || w2 == nullptr || w2_scale == nullptr ||
      out == nullptr || dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if ((!fp8 && !aligned16(recv)) || (fp8 && !aligned16(xq_slots)) || !aligned16(w13) ||
      !aligned16(w2) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  const ComputeWorkspace w = compute_workspace(E, R, H, I);
  if (workspace == nullptr || workspace_bytes < w.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  // the tile list and the stored rows come from seg_counts
  int32_t* slot_of = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + w.slot);
  return expert_compute_impl(recv, seg_counts, E,
                             source_slot_rows(E, R, max_tokens, seg_counts, slot_of), H, I, w13,
                             w13_scale, w2, w2_scale, out, dev_status, workspace, w,
                             dev->sm_count, reinterpret_cast<cudaStream_t>(stream), flags,
                             fp8 ? xq_slots : nullptr, fp8 ? xs_slots : nullptr);
}
}  // namespace

moe_status moe_dispatch_source_slots(const void* x, const void* topk_idx, int idx_bits,
                                     const float* topk_w, int T, int H, int K, int E, int L,
                                     int max_tokens, const int32_t* rank_offsets, void* recv,
                                     int32_t* counts, int32_t* seg_counts, int32_t* src_map,
                                     int32_t* dev_status, moe_stream_t stream) {
  (void)topk_w;
  return source_slots_dispatch(false, x, topk_idx, idx_bits, T, H, K, E, L, max_tokens,
                               rank_offsets, recv, nullptr, nullptr, counts, seg_counts, src_map,
                               dev_status, stream);
}

moe_status moe_dispatch_quant_source_slots(const void* x, const void* topk_idx, int idx_bits,
                                           const float* topk_w, int T, int H, int K, int E,
                                           int L, int max_tokens, const int32_t* rank_offsets,
                                           uint8_t* xq, float* xs, int32_t* counts,
                                           int32_t* seg_counts, int32_t* src_map,
                                           int32_t* dev_status, moe_stream_t stream) {
  (void)topk_w;
  return source_slots_dispatch(true, x, topk_idx, idx_bits, T, H, K, E, L, max_tokens,
                               rank_offsets, nullptr, xq, xs, counts, seg_counts, src_map,
                               dev_status, stream);
}

moe_status moe_expert_compute_source_slots(const void* recv, const int32_t* counts,
                                           const int32_t* seg_counts, int E, int L,
                                           int max_tokens, int H, int I, const uint8_t* w13,
                                           const float* w13_scale, const uint8_t* w2,
                                           const float* w2_scale, void* out, int32_t* dev_status,
                                           void* workspace, size_t workspace_bytes, int flags,
                                           moe_stream_t stream) {
  (void)counts;  // the tile list follows seg_counts
  if (recv == nullptr) return MOE_ERR_INVALID_ARG;
  return source_slots_compute(recv, nullptr, nullptr, seg_counts, E, L, max_tokens, H, I, w13,
                              w13_scale, w2, w2_scale, out, dev_status, workspace,
                              workspace_bytes, flags, stream);
}

moe_status moe_gemm_source_slots(const uint8_t* xq, const float* xs, const int32_t* seg_counts,
                                 int E, int L, int max_tokens, int H, int I, const uint8_t* w13,
                                 const float* w13_scale, const uint8_t* w2,
                                 const float* w2_scale, void* out, int32_t* dev_status,
                                 void* workspace, size_t workspace_bytes, int flags,
                                 moe_stream_t stream) {
  return source_slots_compute(nullptr, xq, xs, seg_counts, E, L, max_tokens, H, I, w13, w13_scale,
                              w2, w2_scale, out, dev_status, workspace, workspace_bytes, flags,
                              stream);
}

moe_status moe_dispatch_quant_ex(const void* x, const void* topk_idx, int idx_bits,
                                 const float* topk_w, int T, int H, int K, int E, int R,
                                 int64_t rows, uint8_t* xq, float* xs, int32_t* counts,
                                 int32_t* src_map, int32_t* dev_status, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream) {
  (void)topk_w;
  if (T < 0 || !valid_hidden(H) || !valid_experts(E, R) || K < 1 || K > 32 || K > E)
    return MOE_ERR_INVALID_ARG;
  if (idx_bits != 32 && idx_bits != 64) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || dev_status == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || topk_idx == nullptr || xq == nullptr || xs == nullptr ||
                src_map == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(x) || (reinterpret_cast<uintptr_t>(xq) & 7u) != 0))
    return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * K > (int64_t{1} << 31) - 1) return MOE_ERR_INVALID_ARG;
  RowLayout rl = padded_rows(E, R);
  if (rows != 0) {
    const int64_t need_rows =
        std::min<int64_t>(static_cast<int64_t>(T) * K, static_cast<int64_t>(E) * R);
    if (!valid_rows(rows) || rows < need_rows) return MOE_ERR_INVALID_ARG;
    rl = RowLayout{R, 1, rows};
  }
  const size_t need = moe_dispatch_workspace_size(T, K, E);
  if (workspace == nullptr || workspace_bytes < need) return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_dispatch_quant(x, topk_idx, idx_bits, T, H, K, E, rl, xq, xs, counts,
                                         src_map, dev_status, static_cast<int32_t*>(workspace),
                                         dev->sm_count, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_quant(const void* x, const int64_t* topk_idx, const float* topk_w, int T,
                              int H, int K, int E, int R, uint8_t* xq, float* xs, int32_t* counts,
                              int32_t* src_map, int32_t* dev_status, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream) {
  return moe_dispatch_quant_ex(x, topk_idx, 64, topk_w, T, H, K, E, R, 0, xq, xs, counts, src_map,
                               dev_status, workspace, workspace_bytes, stream);
}

size_t moe_expert_compute_workspace_size(int E, int R, int H, int I) {
  if (!valid_experts(E, R) || !valid_hidden(H) || !valid_hidden(I)) return 0;
  return compute_workspace(E, R, H, I).total;
}

moe_status moe_quantize_fp8(const void* recv, const int32_t* counts, int E, int R, int H,
                            uint8_t* xq, float* xs, moe_stream_t stream) {
  if (!valid_experts(E, R) || !valid_hidden(H)) return MOE_ERR_INVALID_ARG;
  if (recv == nullptr || counts == nullptr || xq == nullptr || xs == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(recv) || (reinterpret_cast<uintptr_t>(xq) & 7u) != 0) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_quantize(recv, counts, E, padded_rows(E, R), H, xq, xs, dev->sm_count,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_gateup_silu(const uint8_t* xq, const float* xs, const int32_t* counts, int E,
                                int R, int H, int I, const uint8_t* w13, const float* w13_scale,
                                uint8_t* zq, float* zs, int32_t* dev_status, moe_stream_t stream) {
  if (!valid_experts(E, R) || !valid_hidden(H) || !valid_hidden(I)) return MOE_ERR_INVALID_ARG;
  if (xq == nullptr || xs == nullptr || counts == nullptr || w13 == nullptr ||
      w13_scale == nullptr || zq == nullptr || zs == nullptr || dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(w13) || !aligned16(zq)) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_gemm_gateup(xq, xs, counts, E, padded_rows(E, R), H, I, w13, w13_scale,
                                      zq, zs, dev_status, dev->sm_count,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_gemm_down(const uint8_t* zq, const float* zs, const int32_t* counts, int E, int R,
                         int H, int I, const uint8_t* w2, const float* w2_scale, void* out,
                         int32_t* dev_status, moe_stream_t stream) {
  if (!valid_experts(E, R) || !valid_hidden(H) || !valid_hidden(I)) return MOE_ERR_INVALID_ARG;
  if (zq == nullptr || zs == nullptr || counts == nullptr || w2 == nullptr ||
      w2_scale == nullptr || out == nullptr || dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(zq) || !aligned16(w2) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_gemm_down(zq, zs, counts, E, padded_rows(E, R), H, I, w2, w2_scale, out,
                                    dev_status, dev->sm_count,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_gemm_gateup_down_sync_size(int E, int R, int64_t rows) {
  if (!valid_experts(E, R) || (rows != 0 && !valid_rows(rows))) return 0;
  const RowLayout rl = rows == 0 ? padded_rows(E, R) : RowLayout{R, 1, rows};
  return gemm_sync_ints(E, rl) * sizeof(int);
}

moe_status moe_gemm_gateup_down(const uint8_t* xq, const float* xs, const int32_t* counts, int E,
                                int R, int64_t rows, int H, int I, const uint8_t* w13,
                                const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                uint8_t* zq, float* zs, void* out, int32_t* dev_status, void* sync,
                                size_t sync_bytes, int flags, moe_stream_t stream) {
  if (!valid_experts(E, R) || !valid_hidden(H) || !valid_hidden(I)) return MOE_ERR_INVALID_ARG;
  if (!valid_gemm_flags(flags)) return MOE_ERR_INVALID_ARG;
  if (rows != 0 && !valid_rows(rows)) return MOE_ERR_INVALID_ARG;
  if (xq == nullptr || xs == nullptr || counts == nullptr || w13 == nullptr ||
      w13_scale == nullptr || w2 == nullptr || w2_scale == nullptr || zq == nullptr ||
      zs == nullptr || out == nullptr || dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(w13) || !aligned16(w2) || !aligned16(zq) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  const RowLayout rl = rows == 0 ? padded_rows(E, R) : RowLayout{R, 1, rows};
  const size_t need = gemm_sync_ints(E, rl);
  if (sync == nullptr || sync_bytes < need * sizeof(int) ||
      (reinterpret_cast<uintptr_t>(sync) & 3u) != 0)
    return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(run_gemms(xq, xs, counts, E, rl, H, I, w13, w13_scale, w2, w2_scale, zq, zs,
                             out, static_cast<int*>(sync), sync_bytes / sizeof(int), dev_status,
                             dev->sm_count, reinterpret_cast<cudaStream_t>(stream), flags));
}

moe_status moe_expert_compute(const void* recv, const int32_t* counts, int E, int R, int H, int I,
                              const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                              const float* w2_scale, void* out, int32_t* dev_status,
                              void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (!valid_experts(E, R) || !valid_hidden(H) || !valid_hidden(I)) return MOE_ERR_INVALID_ARG;
  if (recv == nullptr || counts == nullptr || w13 == nullptr || w13_scale == nullptr ||
      w2 == nullptr || w2_scale == nullptr || out == nullptr || dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(recv) || !aligned16(w13) || !aligned16(w2) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  const ComputeWorkspace w = compute_workspace(E, R, H, I);
  if (workspace == nullptr || workspace_bytes < w.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return expert_compute_impl(recv, counts, E, padded_rows(E, R), H, I, w13, w13_scale, w2,
                             w2_scale, out, dev_status, workspace, w, dev->sm_count,
                             reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_expert_compute_packed_workspace_size(int64_t rows, int H, int I) {
  if (!valid_rows(rows) || !valid_hidden(H) || !valid_hidden(I)) return 0;
  return compute_workspace_rows(rows, H, I).total;
}

moe_status moe_expert_compute_packed(const void* recv, const int32_t* counts, int E, int R,
                                     int64_t rows, int H, int I, const uint8_t* w13,
                                     const float* w13_scale, const uint8_t* w2,
                                     const float* w2_scale, void* out, int32_t* dev_status,
                                     void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (!valid_experts(E, R) || !valid_rows(rows) || !valid_hidden(H) || !valid_hidden(I))
    return MOE_ERR_INVALID_ARG;
  if (recv == nullptr || counts == nullptr || w13 == nullptr || w13_scale == nullptr ||
      w2 == nullptr || w2_scale == nullptr || out == nullptr || dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(recv) || !aligned16(w13) || !aligned16(w2) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  const ComputeWorkspace w = compute_workspace_rows(rows, H, I);
  if (workspace == nullptr || workspace_bytes < w.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return expert_compute_impl(recv, counts, E, RowLayout{R, 1, rows}, H, I, w13, w13_scale, w2,
                             w2_scale, out, dev_status, workspace, w, dev->sm_count,
                             reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_expert_compute_ex_workspace_size(int E, int R, int64_t rows, int H, int I) {
  if (rows == 0) return moe_expert_compute_workspace_size(E, R, H, I);
  return moe_expert_compute_packed_workspace_size(rows, H, I);
}

int moe_expert_compute_gemm_launches(int E, int R, int64_t rows, int I, int flags) {
  if (!valid_hidden(I) || !valid_gemm_flags(flags)) return MOE_ERR_INVALID_ARG;
  if (rows == 0 ? !valid_experts(E, R) : (!valid_experts(E, R) || !valid_rows(rows)))
    return MOE_ERR_INVALID_ARG;
  if (flags & MOE_GEMM_ONE_LAUNCH) return 1;
  if (flags & MOE_GEMM_TWO_LAUNCHES) return 2;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  const RowLayout rl = rows == 0 ? padded_rows(E, R) : RowLayout{R, 1, rows};
  return gemm_prefer_one_launch(E, rl, I, dev->sm_count) ? 1 : 2;
}

int moe_expert_compute_workspace_layout(int E, int R, int64_t rows, int H, int I,
                                        size_t* offsets) {
  if (offsets == nullptr || !valid_hidden(H) || !valid_hidden(I)) return MOE_ERR_INVALID_ARG;
  if (rows == 0 ? !valid_experts(E, R) : !valid_rows(rows)) return MOE_ERR_INVALID_ARG;
  const ComputeWorkspace w =
      compute_workspace_rows(rows == 0 ? static_cast<int64_t>(E) * R : rows, H, I);
  offsets[0] = w.xq;
  offsets[1] = w.xs;
  offsets[2] = w.zq;
  offsets[3] = w.zs;
  offsets[4] = w.sync;
  offsets[5] = w.sync_ints * sizeof(int);
  offsets[6] = w.total;
  return MOE_OK;
}

moe_status moe_expert_compute_ex(const void* recv, const int32_t* counts, int E, int R, int64_t rows,
                                 int H, int I, const uint8_t* w13, const float* w13_scale,
                                 const uint8_t* w2, const float* w2_scale, void* out,
                                 int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                 int flags, moe_stream_t stream) {
  if (!valid_experts(E, R) || !valid_hidden(H) || !valid_hidden(I)) return MOE_ERR_INVALID_ARG;
  if (!valid_gemm_flags(flags)) return MOE_ERR_INVALID_ARG;
  if (rows != 0 && !valid_rows(rows)) return MOE_ERR_INVALID_ARG;
  if (recv == nullptr || counts == nullptr || w13 == nullptr || w13_scale == nullptr ||
      w2 == nullptr || w2_scale == nullptr || out == nullptr || dev_status == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(recv) || !aligned16(w13) || !aligned16(w2) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  const RowLayout rl = rows == 0 ? padded_rows(E, R) : RowLayout{R, 1, rows};
  const ComputeWorkspace w = compute_workspace_rows(rl.rows, H, I);
  if (workspace == nullptr || workspace_bytes < w.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return expert_compute_impl(recv, counts, E, rl, H, I, w13, w13_scale, w2, w2_scale, out,
                             dev_status, workspace, w, dev->sm_count,
                             reinterpret_cast<cudaStream_t>(stream), flags);
}

moe_status moe_layer_stats(const void* topk_idx, int idx_bits, const int32_t* counts, int T, int K,
                           int E, int L, int R, const int32_t* rank_offsets, uint64_t* stats,
                           moe_stream_t stream) {
  if (T < 0 || K < 1 || K > 32 || E < 1 || E > 1024 || R < 1 || L < 1 || E % L != 0)
    return MOE_ERR_INVALID_ARG;
  if (idx_bits != 32 && idx_bits != 64) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || stats == nullptr || (T > 0 && topk_idx == nullptr))
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(stats) & 7u) != 0) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * K > (int64_t{1} << 31) - 1) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_layer_stats(topk_idx, idx_bits, counts, T, K, E, L, R, rank_offsets,
                                      reinterpret_cast<unsigned long long*>(stats),
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_ep_pack_workspace_size(int T, int K, int E, int L) {
  if (T < 0 || K < 1 || K > 32 || L < 1 || E < 1 || E % L != 0) return 0;
  const size_t tk = align_up(static_cast<size_t>(T) * K * sizeof(int32_t) + 1, 256);
  return 2 * tk + moe_dispatch_workspace_size(T, K, E / L);
}

moe_status moe_ep_pack(const void* x, const void* topk_idx, int idx_bits, int T, int H, int K,
                       int E, int L, void* send_x, int32_t* send_ids, int32_t* send_counts,
                       int32_t* route_msg, int32_t* route_pos, int32_t* dev_status,
                       void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (T < 0 || !valid_hidden(H) || K < 1 || K > 32 || L < 1 || E < 1 || E > 1024 || E % L != 0 ||
      K > E)
    return MOE_ERR_INVALID_ARG;
  if (idx_bits != 32 && idx_bits != 64) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * K > (int64_t{1} << 30)) return MOE_ERR_INVALID_ARG;
  if (send_counts == nullptr || dev_status == nullptr) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (x == nullptr || topk_idx == nullptr || send_x == nullptr || send_ids == nullptr ||
                route_msg == nullptr || route_pos == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(x) || !aligned16(send_x))) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_ep_pack_workspace_size(T, K, E, L);
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  const size_t tk = align_up(static_cast<size_t>(T) * K * sizeof(int32_t) + 1, 256);
  auto* ws = static_cast<uint8_t*>(workspace);
  return from_cuda(launch_ep_pack(x, topk_idx, idx_bits, T, H, K, E, L, send_x, send_ids,
                                  send_counts, route_msg, route_pos, dev_status,
                                  reinterpret_cast<int32_t*>(ws), reinterpret_cast<int32_t*>(ws + tk),
                                  reinterpret_cast<int32_t*>(ws + 2 * tk), dev->sm_count,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_ep_offsets_workspace_size(int64_t S) {
  if (S < 0) return 0;
  return align_up(ep_offsets_scratch_ints(S) * sizeof(int32_t), 256);
}

moe_status moe_ep_route_offsets(const int32_t* ids, int64_t S, int K, int32_t* offsets,
                                void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (S < 0 || S > (int64_t{1} << 30) || K < 1 || K > 32) return MOE_ERR_INVALID_ARG;
  if (offsets == nullptr || (S > 0 && ids == nullptr)) return MOE_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < moe_ep_offsets_workspace_size(S))
    return MOE_ERR_WORKSPACE;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_ep_offsets(ids, S, K, offsets, static_cast<int32_t*>(workspace),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_ep_return(const void* out, int64_t out_rows, const int32_t* src_map,
                         const int32_t* ids, const int32_t* offsets, int64_t S, int K, int H,
                         void* ret, int32_t* flag, moe_stream_t stream) {
  if (S < 0 || S > (int64_t{1} << 30) || K < 1 || K > 32 || !valid_hidden(H) || out_rows < 0)
    return MOE_ERR_INVALID_ARG;
  if (S > 0 && (out == nullptr || src_map == nullptr || ids == nullptr || offsets == nullptr ||
                ret == nullptr || flag == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (S > 0 && (!aligned16(out) || !aligned16(ret))) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_ep_return(out, out_rows, src_map, ids, offsets, S, K, H, ret, flag,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_ep_result_map(const int32_t* route_msg, const int32_t* route_pos,
                             const int32_t* offsets, const int32_t* flag, int64_t n_ret, int T,
                             int K, int32_t* result_map, moe_stream_t stream) {
  if (T < 0 || K < 1 || K > 32 || n_ret < 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (route_msg == nullptr || route_pos == nullptr || offsets == nullptr ||
                result_map == nullptr || (n_ret > 0 && flag == nullptr)))
    return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_ep_result(route_msg, route_pos, offsets, flag, n_ret, T, K, result_map,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const void* out, const int32_t* src_map, const float* topk_w, int T, int H,
                       int K, int E, int R, void* y, moe_stream_t stream) {
  if (T < 0 || !valid_hidden(H) || !valid_experts(E, R) || K < 1 || K > 32 || K > E)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (out == nullptr || src_map == nullptr || topk_w == nullptr || y == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(out) || !aligned16(y))) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_combine(out, src_map, topk_w, T, H, K, static_cast<int64_t>(E) * R, y,
                                  dev->sm_count,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_packed(const void* out, int64_t rows, const int32_t* src_map,
                              const float* topk_w, int T, int H, int K, void* y,
                              moe_stream_t stream) {
  if (T < 0 || !valid_hidden(H) || !valid_rows(rows) || K < 1 || K > 32) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (out == nullptr || src_map == nullptr || topk_w == nullptr || y == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned16(out) || !aligned16(y))) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if (moe_status st = check_device(&dev); st != MOE_OK) return st;
  return from_cuda(launch_combine(out, src_map, topk_w, T, H, K, rows, y, dev->sm_count,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
