// Internal launch wrappers of the sm_103a kernels (host side).  The C ABI in
// include/moe.h validates arguments and then calls these.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

struct DeviceInfo {
  int sm_count;
  int cc_major;
  int cc_minor;
  size_t smem_optin;
};
// Cached properties of the current device; nullptr if the query fails.
const DeviceInfo* current_device_info();

// Where expert e's rows live in the buffers indexed by slot (recv, xq/xs,
// zq/zs, out): padded, rows [e*R, e*R + R) with capacity rows between
// experts; packed, rows [base_e, base_e + c_e) with base_e the prefix of the
// clamped counts c_e = min(counts[e], R), so the valid rows are contiguous
// ("SGLang Expert Compute Backend", §2.6, compact storage).  `rows` is the
// row count of those buffers: E*R when padded, at least the largest possible
// sum of counts when packed.  Per-source fixed slots ("DeepEP 架构与实现笔记",
// §9.5; padded only): expert e's R rows are R / seg ranges of seg rows, one
// per source rank, and row m is valid iff m % seg < seg_counts[e * (R / seg) +
// m / seg]; the rows an expert's tiles cover run to its last valid row.
struct RowLayout {
  int R;
  int packed;
  int64_t rows;
  int seg = 0;                          // rows per source range, 0: not segmented
  const int32_t* seg_counts = nullptr;  // [E, R / seg] valid rows per range
  // Segmented: the quantisation packs each expert's valid rows to the front
  // of its range of xq/xs (row j of expert e at e*R + j) and records their
  // slot rows in slot_of[e*R + j]; the GEMMs run on the packed rows and the
  // down GEMM stores row j at its slot row e*R + slot_of[e*R + j].
  int32_t* slot_of = nullptr;
};
inline RowLayout padded_rows(int E, int R) { return RowLayout{R, 0, static_cast<int64_t>(E) * R}; }
inline RowLayout source_slot_rows(int E, int R, int seg, const int32_t* seg_counts,
                                  int32_t* slot_of) {
  return RowLayout{R, 0, static_cast<int64_t>(E) * R, seg, seg_counts, slot_of};
}

// ----- dispatch (route validation, histogram, scan, stable scatter)
constexpr int kDispatchWarps = 8;
inline int dispatch_tokens_per_warp(int K) { return 32 / K; }
inline int dispatch_tokens_per_block(int K) { return kDispatchWarps * (32 / K); }
// Blocks of the routing kernels; computed in 64 bits so T near INT_MAX cannot
// overflow (callers bound T * K below 2^31, so the result fits an int).
inline int64_t dispatch_blocks64(int64_t T, int K) {
  const int64_t tpb = dispatch_tokens_per_block(K);
  return (T + tpb - 1) / tpb;
}
inline int dispatch_blocks(int T, int K) { return static_cast<int>(dispatch_blocks64(T, K)); }
// Up to this many routes (T * K) the dispatch runs as one kernel: every block
// counts the routes before its own straight from topk_idx instead of the
// histogram and scan kernels (same slots, counts and status).
constexpr int kSinglePassRoutes = 4096;
// topk_idx holds int64 ids (idx_bits = 64) or int32 ids (idx_bits = 32).
cudaError_t launch_dispatch(const void* x, const void* topk_idx, int idx_bits, int T, int H, int K,
                            int E, RowLayout rl, void* recv, int32_t* counts, int32_t* src_map,
                            int32_t* dev_status, int32_t* hist, int sm_count, cudaStream_t s);

// ----- per-source fixed-slot dispatch: recv [E, W * mt, H] BF16, or (recv
// null) the e4m3 codes xq [E, W * mt, H] and scales xs [E, W * mt, H / 128] of
// each token row quantised once; counts [E] valid rows per expert, seg_counts
// [E, W] per (expert, source rank); rank_offsets [W + 1] token offsets of the
// source ranks, or null for ceil(T / W) each
cudaError_t launch_dispatch_source_slots(const void* x, const void* topk_idx, int idx_bits, int T,
                                         int H, int K, int E, int W, int mt,
                                         const int32_t* rank_offsets, void* recv, uint8_t* xq,
                                         float* xs, int32_t* counts, int32_t* seg_counts,
                                         int32_t* src_map, int32_t* dev_status, int sm_count,
                                         cudaStream_t s);

// ----- dispatch fused with the per-token FP8 quantisation: xq e4m3 and xs
// (row layout rl, int32 or int64 ids) instead of the BF16 receive buffer
cudaError_t launch_dispatch_quant(const void* x, const void* topk_idx, int idx_bits, int T, int H,
                                  int K, int E, RowLayout rl, uint8_t* xq, float* xs,
                                  int32_t* counts, int32_t* src_map, int32_t* dev_status,
                                  int32_t* hist, int sm_count, cudaStream_t s);

// ----- per-token FP8 quantisation of the valid rows; xs is [E, R, H/128].
// With pq/ps (per-source slots only) the slot rows already hold e4m3 codes and
// scales, which are packed instead of quantised.
cudaError_t launch_quantize(const void* recv, const int32_t* counts, int E, RowLayout rl, int H,
                            uint8_t* xq, float* xs, int sm_count, cudaStream_t s,
                            const uint8_t* pq = nullptr, const float* ps = nullptr);

// ----- grouped block-scaled FP8 GEMMs on tcgen05
// w13_interleaved: W13 output rows alternate gate and up (2j gate, 2j+1 up)
// instead of the first I rows gate and the last I up.
cudaError_t launch_gemm_gateup(const uint8_t* xq, const float* xs, const int32_t* counts, int E,
                               RowLayout rl, int H, int I, const uint8_t* w13,
                               const float* w13_scale, uint8_t* zq, float* zs,
                               int32_t* dev_status, int sm_count, cudaStream_t s,
                               int w13_interleaved = 0);
cudaError_t launch_gemm_down(const uint8_t* zq, const float* zs, const int32_t* counts, int E,
                             RowLayout rl, int H, int I, const uint8_t* w2, const float* w2_scale,
                             void* out, int32_t* dev_status, int sm_count, cudaStream_t s);
// Both GEMMs in one persistent launch: a down tile starts as soon as the
// gate/up tiles of its 128-row block have written their Z rows.  `sync` holds
// gemm_sync_ints(E, rl) ints of device scratch (zeroed by the launch).  With
// H % 256 != 0 it runs the two launches above instead.
size_t gemm_sync_ints(int E, RowLayout rl);
// Whether moe_expert_compute runs both GEMMs as one launch (true) or as the
// gate/up launch followed by the down launch, from the largest possible tile
// count of the layout.
bool gemm_prefer_one_launch(int E, RowLayout rl, int I, int sm_count);
cudaError_t launch_gemm_gateup_down(const uint8_t* xq, const float* xs, const int32_t* counts,
                                    int E, RowLayout rl, int H, int I, const uint8_t* w13,
                                    const float* w13_scale, const uint8_t* w2,
                                    const float* w2_scale, uint8_t* zq, float* zs, void* out,
                                    int* sync, size_t sync_ints, int32_t* dev_status,
                                    int sm_count, cudaStream_t s, int w13_interleaved);

// ----- weighted combine
// rows = the number of rows of `out` (E * R padded, the buffer's rows packed);
// a src_map entry outside [0, rows) is treated like -1.
cudaError_t launch_combine(const void* out, const int32_t* src_map, const float* topk_w, int T,
                           int H, int K, int64_t rows, void* y, int sm_count, cudaStream_t s);

// ----- expert parallelism across ranks (ep.cu)
// Send plan of one source rank: send_x [T * min(K, W), H] one payload row per
// (token, destination rank), packed by destination in ascending token order;
// send_ids [same rows, K] the destination-local expert id of each top-k
// position (-1 elsewhere); send_counts [W]; route_msg / route_pos [T, K] the
// message of each route and its position among the message's routes.  dest,
// msg [T, K] int32 and hist (dispatch workspace) are scratch.
cudaError_t launch_ep_pack(const void* x, const void* topk_idx, int idx_bits, int T, int H, int K,
                           int E, int L, void* send_x, int32_t* send_ids, int32_t* send_counts,
                           int32_t* route_msg, int32_t* route_pos, int32_t* dev_status,
                           int32_t* dest, int32_t* msg, int32_t* hist, int sm_count,
                           cudaStream_t s);
// offsets [S + 1]: exclusive prefix over rows of ids [S, K] of their valid
// (>= 0) entries; scratch of ep_offsets_scratch_ints(S) ints.
size_t ep_offsets_scratch_ints(int64_t S);
cudaError_t launch_ep_offsets(const int32_t* ids, int64_t S, int K, int32_t* offsets,
                              int32_t* scratch, cudaStream_t s);
// One returned row per route of the received rows (expert output or zeros),
// at offsets[j] + position; flag 1 where the layer kept the route.
cudaError_t launch_ep_return(const void* out, int64_t out_rows, const int32_t* src_map,
                             const int32_t* ids, const int32_t* offsets, int64_t S, int K, int H,
                             void* ret, int32_t* flag, cudaStream_t s);
// result_map [T, K]: the returned row of each route at the source, or -1.
cudaError_t launch_ep_result(const int32_t* route_msg, const int32_t* route_pos,
                             const int32_t* offsets, const int32_t* flag, int64_t n_ret, int T,
                             int K, int32_t* result_map, cudaStream_t s);

// ----- layer statistics of one routing (kLayerStats 64-bit counters):
// [0] valid routes, [1] kept routes, [2] messages (sum over tokens of the
// distinct destination ranks), [3] cross-rank routes, [4] 128-row blocks of
// the GEMM tile list, [5] active experts, [6] the busiest expert's kept rows
constexpr int kLayerStats = 7;
cudaError_t launch_layer_stats(const void* topk_idx, int idx_bits, const int32_t* counts, int T,
                               int K, int E, int L, int R, const int32_t* rank_offsets,
                               unsigned long long* stats, cudaStream_t s);

}  // namespace moe
