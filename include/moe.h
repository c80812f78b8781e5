/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed-MoE library.
 *
 * One MoE layer's routed branch on one GPU, in three calls:
 *
 *   moe_dispatch        x, topk_idx            -> recv [E,R,H], counts [E], src_map [T,K]
 *   moe_expert_compute  recv, counts, weights  -> out  [E,R,H]
 *   moe_combine         out, src_map, topk_w   -> y    [T,H]
 *
 * plus the same three calls for a packed layout without capacity gaps
 * (moe_*_packed, below) and a dispatch fused with the FP8 quantisation.
 *
 * The steps follow "SGLang、NCCL 与 MoE EP" (Level 1 §1.1: the routed output
 * is the weighted sum of the expert outputs; §2.3: receive, compact and the
 * source map; §3.2: dispatch, compute, combine of one token) and "SGLang
 * Expert Compute Backend" (§1.1 gated-SiLU expert; §3.5-3.7 block-wise FP8
 * GEMMs writing each output back at its original slot).  The pages' multi-rank
 * EP layout is modelled inside one GPU: global expert g belongs to logical rank
 * g / L as local expert g % L, and the all-to-all exchange becomes the
 * in-memory scatter of moe_dispatch and gather of moe_combine.
 *
 * Conventions for every call:
 *  - Pointers marked "device" are CUDA device memory owned by the caller; the
 *    library never allocates, frees or retains them.  Tensors are contiguous
 *    and row-major.  BF16 tensors are passed as void* (IEEE bfloat16, 2 bytes).
 *    FP8 tensors are e4m3 (OCP "float8_e4m3fn") codes, one byte each.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream): no host synchronisation, no allocation, no host reads of
 *    device data.  Every call other than moe_dispatch_noalloc can be
 *    captured into a CUDA graph; nothing is stated here either way about
 *    capturing moe_dispatch_noalloc.
 *  - Host-detectable errors (null pointers, bad sizes, workspace too small,
 *    unsupported device) return a negative moe_status before anything is
 *    launched.  MOE_ERR_CUDA means a CUDA runtime call failed; the CUDA error
 *    is left for the caller's cudaGetLastError().
 *  - Data-dependent problems are reported in a caller-owned device status
 *    word `dev_status` (int32[2]): dev_status[0] holds MOE_DEV_* bits and
 *    dev_status[1] the number of routes dropped for capacity.  moe_dispatch
 *    resets both words; moe_expert_compute only ORs bits into dev_status[0].
 *    Read it after your own synchronisation.
 *  - Sizes: 0 <= T, 1 <= K <= min(E, 32), E <= 1024, 1 <= R, H and I
 *    multiples of 128, H <= 16384, I <= 16384.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* null pointer, negative or inconsistent size */
  MOE_ERR_UNSUPPORTED = -2, /* device is not sm_103, or a size outside the limits above */
  MOE_ERR_WORKSPACE = -3,   /* workspace pointer null or smaller than *_workspace_size() */
  MOE_ERR_CUDA = -4         /* a CUDA runtime call failed (see cudaGetLastError) */
} moe_status;

/* Bits of dev_status[0]. */
#define MOE_DEV_BAD_EXPERT_ID 1    /* a topk_idx entry outside [-1, E): that route was ignored */
#define MOE_DEV_CAPACITY_DROPPED 2 /* some expert had more than R routes; dev_status[1] = how many dropped */
#define MOE_DEV_TIMEOUT 4          /* a bounded device-side wait expired; that kernel's outputs are invalid */

/* Version of this ABI (incremented on any signature change). */
int moe_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* ---------------------------------------------------------------------------
 * Dispatch -- "SGLang、NCCL 与 MoE EP", §2.3.1 (source tensors), §2.3.4
 * (receive and compact: recv[e, s, :] = payload, s from expert e's counter),
 * §2.3.6 (expert_counters and the source map, flat row q = e*R + s).
 *
 *   x         device, BF16 [T, H]      token activations (read once per token)
 *   topk_idx  device, int64 [T, K]     global expert ids; -1 = padding route
 *   topk_w    device, fp32 [T, K]      accepted for interface fidelity, not read
 *                                      (the pages keep router weights at the source)
 *   recv      device, BF16 [E, R, H]   out: rows [0, counts[e]) of expert e hold the
 *                                      payload of its routes; other rows untouched
 *   counts    device, int32 [E]        out: kept routes per expert (= min(routes, R))
 *   src_map   device, int32 [T, K]     out: q = e*R + s of route (t, k), or -1 for a
 *                                      padding, invalid or dropped route
 *   dev_status device, int32 [2]       out: reset, then MOE_DEV_* bits and drop count
 *   workspace device, >= moe_dispatch_workspace_size(T, K, E) bytes, 256-byte aligned;
 *                                      scratch, contents need not be initialised
 *
 * Slot order: the slot of a route within its expert is its rank among that
 * expert's routes in ascending route id i = t*K + k (deterministic; any order
 * would be a valid compact prefix, the pages leave it to atomic arrival order).
 * Routes past capacity R are dropped in that order.  T == 0 is legal: counts
 * are zeroed and nothing else is written.
 * ------------------------------------------------------------------------- */
size_t moe_dispatch_workspace_size(int T, int K, int E);
moe_status moe_dispatch(const void* x, const int64_t* topk_idx, const float* topk_w, int T, int H,
                        int K, int E, int R, void* recv, int32_t* counts, int32_t* src_map,
                        int32_t* dev_status, void* workspace, size_t workspace_bytes,
                        moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_dispatch_noalloc -- the pages have no counterpart; this is a convenience
 * of this library.  The same dispatch as moe_dispatch, for callers that cannot
 * allocate device memory: serving runtimes that reserve all device memory at
 * start-up and forbid allocation afterwards, hosts (plain C programs, other
 * language runtimes) that link this library without handing it an allocator,
 * and latency-critical loops that cannot afford cudaMalloc's implicit device
 * synchronisation.  It calls no allocating routine of CUDA or any library.
 *
 * Arguments and outputs are those of moe_dispatch, minus the workspace: the
 * scratch is a 1 MiB array inside the library (held by every GPU that loads
 * the library until the process exits), which limits the problem to
 * moe_dispatch_workspace_size(T, K, E) <= 1 MiB, i.e. E * ceil(T / (8*(32/K)))
 * <= 262144; larger problems return MOE_ERR_WORKSPACE without launching.
 * The first call on a device (and the first after a cudaDeviceReset) looks up
 * the array's device address with that device current and caches it per
 * device and context; make that first call before any stream capture.  Every
 * call shares the one array, and nothing in it needs to start at zero (each
 * call writes every entry it reads); calls whose kernels overlap on the GPU
 * (different streams without ordering) race on it and must not be issued.
 * ------------------------------------------------------------------------- */
moe_status moe_dispatch_noalloc(const void* x, const int64_t* topk_idx, const float* topk_w, int T,
                                int H, int K, int E, int R, void* recv, int32_t* counts,
                                int32_t* src_map, int32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_dispatch_quant -- dispatch fused with the per-token FP8 quantisation,
 * the "quantise while packing" candidate of "SGLang Expert Compute Backend",
 * §4.4.  Every kept route's row is written to the receive layout already as
 * e4m3 codes plus fp32 scales; the BF16 receive buffer is never formed.  Each
 * token row is quantised once (the rule of moe_quantize_fp8, which is per row,
 * so all K copies are identical).  Outputs equal moe_quantize_fp8 applied to
 * moe_dispatch's recv, bit for bit; counts, src_map and dev_status are those of
 * moe_dispatch.  Feed xq/xs to moe_gemm_gateup_silu.
 *
 *   xq  device, e4m3 [E, R, H]       out: rows [0, counts[e]) written
 *   xs  device, fp32 [E, R, H/128]   out: scales of those rows
 *   other arguments and the workspace as for moe_dispatch
 * ------------------------------------------------------------------------- */
moe_status moe_dispatch_quant(const void* x, const int64_t* topk_idx, const float* topk_w, int T,
                              int H, int K, int E, int R, uint8_t* xq, float* xs, int32_t* counts,
                              int32_t* src_map, int32_t* dev_status, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_dispatch_quant_ex -- the general fused dispatch: moe_dispatch_quant is
 * its int64, padded case.  idx_bits (32 or 64) and rows (0: padded layout,
 * xq [E, R, H] / xs [E, R, H/128]; > 0: packed layout, xq [rows, H] / xs
 * [rows, H/128], rows as for moe_dispatch_packed) as for moe_dispatch_ex.
 * Outputs equal moe_quantize_fp8's on moe_dispatch_ex's receive rows, bit for
 * bit, with the src_map, counts and status of moe_dispatch_ex.
 * ------------------------------------------------------------------------- */
moe_status moe_dispatch_quant_ex(const void* x, const void* topk_idx, int idx_bits,
                                 const float* topk_w, int T, int H, int K, int E, int R,
                                 int64_t rows, uint8_t* xq, float* xs, int32_t* counts,
                                 int32_t* src_map, int32_t* dev_status, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Expert compute -- per-token FP8 quantisation of the valid receive rows
 * ("SGLang、NCCL 与 MoE EP", §2.3.5; rule of "DeepEP 架构与实现笔记", §11), then
 * the gated-SiLU expert of "SGLang Expert Compute Backend", §1.1 and §3.5-3.7:
 * G = block-scaled FP8 GEMM of x with W13 (first I output columns gate, last
 * I up), Z = SiLU(gate) * up re-quantised per row per 128, out = block-scaled
 * FP8 GEMM of Z with W2, written at the original slot (e, s).  When the
 * gate/up tiles fill only a few waves of CTAs (decode-sized layers) both GEMMs
 * run in one launch (see moe_gemm_gateup_down: the down tiles of a 128-row
 * block start once that block's Z is written); otherwise as two launches,
 * which measured faster there.
 *
 *   recv       device, BF16 [E, R, H]          rows >= counts[e] are never read
 *   counts     device, int32 [E]               valid rows per expert (values > R act as R)
 *   w13        device, e4m3 [E, 2I, H]         gate/up weights, output-major
 *   w13_scale  device, fp32 [E, 2I/128, H/128] one scale per 128x128 block
 *   w2         device, e4m3 [E, H, I]          down weights, output-major
 *   w2_scale   device, fp32 [E, H/128, I/128]
 *   out        device, BF16 [E, R, H]          out: rows [0, counts[e]); others untouched
 *   dev_status device, int32 [2]               MOE_DEV_TIMEOUT may be ORed in
 *   workspace  device, >= moe_expert_compute_workspace_size(E, R, H, I) bytes,
 *              256-byte aligned; holds the FP8 activations and their scales, Z
 *              and its scales, and the GEMM launch's tile ticket and block
 *              counts; not shared with another call in flight
 *
 * Router weights never enter this call ("SGLang、NCCL 与 MoE EP", §1.1: the
 * weight multiplies the expert output, not its input).
 * ------------------------------------------------------------------------- */
size_t moe_expert_compute_workspace_size(int E, int R, int H, int I);
moe_status moe_expert_compute(const void* recv, const int32_t* counts, int E, int R, int H, int I,
                              const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                              const float* w2_scale, void* out, int32_t* dev_status,
                              void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Combine -- "SGLang、NCCL 与 MoE EP", §3.2 (合对): each route's expert output
 * is multiplied by its router weight exactly once and summed into the token's
 * own row; "DeepEP 架构与实现笔记", §9.6: the weighted reduce is done inside the
 * combine kernel.
 *
 *   out      device, BF16 [E, R, H]   expert outputs at flat rows q
 *   src_map  device, int32 [T, K]     from moe_dispatch; -1 entries are skipped
 *   topk_w   device, fp32 [T, K]      router weights
 *   y        device, BF16 [T, H]      out: y[t] = bf16( sum over k ascending of
 *                                     w[t,k] * out[q] ), accumulated in fp32 from 0,
 *                                     each product and each sum rounded to fp32;
 *                                     a token with no kept route gets zeros
 * ------------------------------------------------------------------------- */
moe_status moe_combine(const void* out, const int32_t* src_map, const float* topk_w, int T, int H,
                       int K, int E, int R, void* y, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * The three steps inside moe_expert_compute, exposed for testing and
 * profiling.  Scales are stored row-major per row, [E, R, G] (G = H/128 or
 * I/128), the pages' layout.
 *
 * moe_quantize_fp8 -- "DeepEP 架构与实现笔记", §11: per valid row and 128-group,
 *   amax = max(max|v|, 1e-4); xq = e4m3_rn_satfinite(v * (448/amax)); xs = amax/448,
 *   all in fp32.  xq device e4m3 [E, R, H]; xs device fp32 [E, R, H/128].
 * moe_gemm_gateup_silu -- "SGLang Expert Compute Backend", §3.5-3.6: G from xq/xs
 *   and W13, Z = SiLU(G[:, :I]) * G[:, I:], quantised like moe_quantize_fp8.
 *   zq device e4m3 [E, R, I]; zs device fp32 [E, R, I/128].
 * moe_gemm_down -- the same page, §3.6-3.7: out = block-scaled GEMM of zq/zs
 *   with W2, BF16 [E, R, H], rows [0, counts[e]) only.
 * Only rows < counts[e] are read or written in every step.  Activations must
 * be finite: a NaN or infinity in a 128-group gives unspecified codes and
 * scale for that group (never a fault).
 * ------------------------------------------------------------------------- */
moe_status moe_quantize_fp8(const void* recv, const int32_t* counts, int E, int R, int H,
                            uint8_t* xq, float* xs, moe_stream_t stream);
moe_status moe_gemm_gateup_silu(const uint8_t* xq, const float* xs, const int32_t* counts, int E,
                                int R, int H, int I, const uint8_t* w13, const float* w13_scale,
                                uint8_t* zq, float* zs, int32_t* dev_status, moe_stream_t stream);
moe_status moe_gemm_down(const uint8_t* zq, const float* zs, const int32_t* counts, int E, int R,
                         int H, int I, const uint8_t* w2, const float* w2_scale, void* out,
                         int32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_gemm_gateup_down -- moe_gemm_gateup_silu followed by moe_gemm_down, in
 * one persistent launch where that is the faster form, else as those two
 * launches (the MOE_GEMM_* flags of moe_expert_compute_ex; MOE_GEMM_ONE_LAUNCH
 * always takes the one launch).  The arithmetic is that of "SGLang Expert
 * Compute Backend", §3.5-3.7.  The scheduling of the one launch applies the
 * tile events of "XTuner Domino EP" (HyperParallel-MoE section, from whole
 * collectives to destination tile events): a task waits on a per-tile counter
 * reaching its threshold rather than on the whole preceding operator.  Here a
 * down tile of a 128-row block starts once every gate/up tile of that block
 * has written its Z rows.  Results are bit-identical to the two calls.
 *
 *   xq, xs     as for moe_gemm_gateup_silu, in the layout given by rows:
 *              rows = 0 padded [E, R, ...], rows > 0 packed [rows, ...]
 *              (see "Packed layout" below)
 *   zq, zs     device scratch for Z, [E, R, I] / [E, R, I/128] or [rows, ...]
 *   out        device BF16, [E, R, H] or [rows, H]; valid rows only
 *   sync       device scratch of moe_gemm_gateup_down_sync_size(E, R, rows)
 *              bytes, 4-byte aligned, overwritten (zeroed) by the call;
 *              not shared with another call in flight
 *   flags      MOE_W13_INTERLEAVED, MOE_GEMM_ONE_LAUNCH, MOE_GEMM_TWO_LAUNCHES
 *              (see moe_expert_compute_ex)
 * Returns MOE_ERR_INVALID_ARG for bad sizes, pointers or flags,
 * MOE_ERR_WORKSPACE if sync is too small.  Waits between tiles are bounded:
 * one that runs out raises MOE_DEV_TIMEOUT in dev_status.  moe_expert_compute
 * and its variants run these GEMMs, in the same form, after their quantisation.
 * ------------------------------------------------------------------------- */
size_t moe_gemm_gateup_down_sync_size(int E, int R, int64_t rows);
moe_status moe_gemm_gateup_down(const uint8_t* xq, const float* xs, const int32_t* counts, int E,
                                int R, int64_t rows, int H, int I, const uint8_t* w13,
                                const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                uint8_t* zq, float* zs, void* out, int32_t* dev_status, void* sync,
                                size_t sync_bytes, int flags, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Packed layout -- "SGLang Expert Compute Backend", §2.6 (compact storage):
 * the valid rows of all experts are stored back to back, expert e's rows at
 * [base_e, base_e + c_e) with c_e = min(counts[e], R) and base_e the sum of
 * c_j over j < e (the page's example: counts [70, 12] -> expert 1 starts at row
 * 70, 82 rows in all), instead of one capacity block of R rows per expert.
 * Routing, slots, capacity drops and all arithmetic are those of the padded
 * calls above; only the row of slot s of expert e changes from e*R + s to
 * base_e + s, so src_map holds base_e + s.  The receive-side buffers need
 * `rows` rows instead of E*R; the bases are derived on the device from counts.
 *
 * moe_dispatch_packed      as moe_dispatch, with recv device BF16 [rows, H];
 *                          rows >= min(T*K, E*R) (room for every kept route),
 *                          rows <= 2^30, else MOE_ERR_INVALID_ARG.
 * moe_expert_compute_packed  as moe_expert_compute, with recv and out device
 *                          BF16 [rows, H] in the packed layout (counts, E and R
 *                          as given to moe_dispatch_packed) and a workspace of
 *                          moe_expert_compute_packed_workspace_size(rows, H, I)
 *                          bytes.  Rows at or past `rows` are never touched, even
 *                          if counts claim more.
 * moe_combine_packed       as moe_combine, with out device BF16 [rows, H]; a
 *                          src_map entry outside [0, rows) counts as no route.
 * ------------------------------------------------------------------------- */
moe_status moe_dispatch_packed(const void* x, const int64_t* topk_idx, const float* topk_w, int T,
                               int H, int K, int E, int R, int64_t rows, void* recv,
                               int32_t* counts, int32_t* src_map, int32_t* dev_status,
                               void* workspace, size_t workspace_bytes, moe_stream_t stream);
size_t moe_expert_compute_packed_workspace_size(int64_t rows, int H, int I);
moe_status moe_expert_compute_packed(const void* recv, const int32_t* counts, int E, int R,
                                     int64_t rows, int H, int I, const uint8_t* w13,
                                     const float* w13_scale, const uint8_t* w2,
                                     const float* w2_scale, void* out, int32_t* dev_status,
                                     void* workspace, size_t workspace_bytes, moe_stream_t stream);
moe_status moe_combine_packed(const void* out, int64_t rows, const int32_t* src_map,
                              const float* topk_w, int T, int H, int K, void* y,
                              moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Per-source fixed slots -- the low-latency receive layout of "DeepEP 架构与实现笔记",
 * §9.5: the receive buffer is [L, W*max_tokens, H] per rank and every source
 * rank owns a fixed range of max_tokens slots inside every expert, so a route's
 * row follows from its source rank and its position among that source's routes
 * to the expert, with no layout agreed across ranks first (no global count or
 * scan).  The cost, as the page says: a larger buffer whose padding rows lie
 * between the source ranges, which the expert GEMM must skip.  On one GPU the
 * W = E / L logical ranks' experts share one buffer:
 *
 * moe_dispatch_source_slots
 *   x, topk_idx, idx_bits, topk_w, T, H, K as for moe_dispatch_ex
 *   L            local experts per logical rank (E % L == 0, W = E / L ranks)
 *   max_tokens   slots per source range (the page's max tokens per rank)
 *   rank_offsets device, int32 [W + 1]: source rank r's tokens are
 *                [rank_offsets[r], rank_offsets[r+1]), or NULL for
 *                ceil(T / W) tokens per rank (the last ones fewer)
 *   recv         device, BF16 [E, W*max_tokens, H]: route (t, k) of source rank
 *                r to expert e, the p-th of r's routes to e in ascending route
 *                id, lands at row r*max_tokens + p of expert e; other rows
 *                untouched
 *   counts       device, int32 [E]: valid rows per expert (the page's masked_m)
 *   seg_counts   device, int32 [E, W]: valid rows of each (expert, source) range
 *   src_map      device, int32 [T, K]: q = e*W*max_tokens + r*max_tokens + p, or -1
 *   dev_status   as for moe_dispatch; a route with p >= max_tokens is dropped
 *                (MOE_DEV_CAPACITY_DROPPED, counted in dev_status[1])
 * No workspace: each source rank's slots are computed by its own blocks.
 *
 * moe_expert_compute_source_slots -- moe_expert_compute on that layout: the
 *   quantisation packs expert e's valid rows together (in slot order, inside
 *   the workspace), so the GEMM tiles cover valid rows only (the page's masked
 *   expert compute); the down GEMM stores each row at its slot, and the rows
 *   between source ranges are never written.
 *   recv/out device BF16 [E, W*max_tokens, H]; counts may be NULL (not read);
 *   seg_counts from moe_dispatch_source_slots; workspace of
 *   moe_expert_compute_workspace_size(E, W*max_tokens, H, I) bytes; flags as
 *   for moe_expert_compute_ex.  Output rows equal those of the padded layout
 *   for the same routes, bit for bit.  Combine with moe_combine(out, src_map,
 *   topk_w, T, H, K, E, W*max_tokens, y).
 *
 * The same layout with the quantisation fused into the dispatch ("SGLang
 * Expert Compute Backend", §4.4), as moe_dispatch_quant_ex does for the padded
 * and packed layouts:
 * moe_dispatch_quant_source_slots -- the slots, counts, seg_counts, src_map and
 *   status of moe_dispatch_source_slots; each token row is quantised once (the
 *   rule of moe_quantize_fp8) and its codes and scales are written to every
 *   kept slot: xq device e4m3 [E, W*max_tokens, H] (8-byte aligned), xs device
 *   fp32 [E, W*max_tokens, H/128]; other rows untouched.
 * moe_gemm_source_slots -- both GEMMs on those slots: each expert's valid rows
 *   are packed inside the workspace (no quantisation: the codes and scales are
 *   copied), then the GEMMs of moe_expert_compute_source_slots run with the
 *   same workspace size, flags and output.  xq 16-byte aligned (else
 *   MOE_ERR_INVALID_ARG); xs and seg_counts as written by
 *   moe_dispatch_quant_source_slots.  Outputs equal
 *   moe_expert_compute_source_slots' on the BF16 slots of the same routes, bit
 *   for bit.
 * ------------------------------------------------------------------------- */
moe_status moe_dispatch_source_slots(const void* x, const void* topk_idx, int idx_bits,
                                     const float* topk_w, int T, int H, int K, int E, int L,
                                     int max_tokens, const int32_t* rank_offsets, void* recv,
                                     int32_t* counts, int32_t* seg_counts, int32_t* src_map,
                                     int32_t* dev_status, moe_stream_t stream);
moe_status moe_expert_compute_source_slots(const void* recv, const int32_t* counts,
                                           const int32_t* seg_counts, int E, int L,
                                           int max_tokens, int H, int I, const uint8_t* w13,
                                           const float* w13_scale, const uint8_t* w2,
                                           const float* w2_scale, void* out, int32_t* dev_status,
                                           void* workspace, size_t workspace_bytes, int flags,
                                           moe_stream_t stream);
moe_status moe_dispatch_quant_source_slots(const void* x, const void* topk_idx, int idx_bits,
                                           const float* topk_w, int T, int H, int K, int E,
                                           int L, int max_tokens, const int32_t* rank_offsets,
                                           uint8_t* xq, float* xs, int32_t* counts,
                                           int32_t* seg_counts, int32_t* src_map,
                                           int32_t* dev_status, moe_stream_t stream);
moe_status moe_gemm_source_slots(const uint8_t* xq, const float* xs, const int32_t* seg_counts,
                                 int E, int L, int max_tokens, int H, int I, const uint8_t* w13,
                                 const float* w13_scale, const uint8_t* w2,
                                 const float* w2_scale, void* out, int32_t* dev_status,
                                 void* workspace, size_t workspace_bytes, int flags,
                                 moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_dispatch_ex -- the general dispatch: moe_dispatch and moe_dispatch_packed
 * are its two common cases.
 *   topk_idx   device, [T, K] router ids, int32 (idx_bits = 32) or int64
 *              (idx_bits = 64); -1 marks a padding route, ids outside [-1, E)
 *              are reported as MOE_DEV_BAD_EXPERT_ID and ignored
 *   rows       0: padded layout, recv [E, R, H];  > 0: packed layout, recv
 *              [rows, H] with the conditions of moe_dispatch_packed
 * Everything else as moe_dispatch.  MOE_ERR_INVALID_ARG for idx_bits other
 * than 32 or 64.
 * ------------------------------------------------------------------------- */
moe_status moe_dispatch_ex(const void* x, const void* topk_idx, int idx_bits, const float* topk_w,
                           int T, int H, int K, int E, int R, int64_t rows, void* recv,
                           int32_t* counts, int32_t* src_map, int32_t* dev_status,
                           void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_expert_compute_ex -- the general expert compute: moe_expert_compute and
 * moe_expert_compute_packed are its flags = 0 cases.
 *   rows   0: padded layout, recv/out [E, R, H];  > 0: packed layout [rows, H]
 *   flags  MOE_W13_INTERLEAVED: W13 output rows alternate gate and up (row 2j
 *          is gate feature j, row 2j+1 up feature j; the scale blocks are the
 *          128x128 blocks of this layout): the expert of "XTuner Domino EP"
 *          (section on the complete runtime path), whose SiLU takes the even
 *          output columns of the first GEMM and multiplies by the odd ones.
 *          Default: the first I rows gate, the last I up ("SGLang Expert
 *          Compute Backend", §3.6).
 *          MOE_GEMM_ONE_LAUNCH / MOE_GEMM_TWO_LAUNCHES: force the GEMMs' launch
 *          form (see below); at most one of them.  MOE_GEMM_MAX_CTAS(n): cap
 *          the GEMMs' grid at n SMs.
 * Workspace: moe_expert_compute_ex_workspace_size(E, R, rows, H, I) bytes.
 * MOE_ERR_INVALID_ARG for unknown flag bits.
 * ------------------------------------------------------------------------- */
#define MOE_W13_INTERLEAVED 1
/* How the two GEMMs are launched (results are bit-identical either way): by
 * default one launch (moe_gemm_gateup_down) when the gate/up tiles fill only a
 * few waves of CTAs, else the gate/up launch followed by the down launch.
 * These flags force one form or the other. */
#define MOE_GEMM_ONE_LAUNCH 2
#define MOE_GEMM_TWO_LAUNCHES 4
/* At most n CTAs (SMs) for the GEMMs' persistent grids, 1 <= n <= 32767; the
 * default (n = 0) takes one CTA per SM.  Leaves SMs to kernels of other
 * streams, e.g. the other micro-batch's dispatch and combine in a two-batch
 * overlap ("SGLang、NCCL 与 MoE EP", §2.4).  Combine with | into flags. */
#define MOE_GEMM_MAX_CTAS(n) ((int)(((unsigned)(n) & 0x7FFFu) << 16))
size_t moe_expert_compute_ex_workspace_size(int E, int R, int64_t rows, int H, int I);
moe_status moe_expert_compute_ex(const void* recv, const int32_t* counts, int E, int R, int64_t rows,
                                 int H, int I, const uint8_t* w13, const float* w13_scale,
                                 const uint8_t* w2, const float* w2_scale, void* out,
                                 int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                 int flags, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_layer_stats -- the counts the pages account a layer by, for one routing:
 * "SGLang、NCCL 与 MoE EP", §5.3 (each token sends one payload per distinct
 * destination rank, D_t of them, §2.3.2; routes to an expert on another logical
 * rank than the token's are cross-rank) and "SGLang Expert Compute Backend",
 * §5.4 (M-row fill of the grouped GEMM's blocks).
 *
 *   topk_idx     device, [T, K] int32 (idx_bits = 32) or int64 router ids;
 *                ids outside [0, E) do not count as routes
 *   counts       device, int32 [E]: kept rows per expert (moe_dispatch's output)
 *   L            local experts per logical rank (E % L == 0); expert g lives on
 *                rank g / L
 *   rank_offsets device, int32 [E/L + 1]: token t comes from the rank r with
 *                rank_offsets[r] <= t < rank_offsets[r+1] (tokens concatenated
 *                in rank order), or NULL: ceil(T / (E/L)) tokens per rank
 *   stats        device, uint64 [7], 8-byte aligned, overwritten:
 *                [0] valid routes  [1] kept routes (dropped = [0] - [1])
 *                [2] messages, sum over tokens of D_t  [3] cross-rank routes
 *                [4] 128-row blocks of the GEMM tile list, sum_e ceil(c_e/128)
 *                    (M-row fill = [1] / (128 * [4]); a capacity-dense launch
 *                    covers E * ceil(R/128) blocks)
 *                [5] active experts  [6] the busiest expert's kept rows
 * Asynchronous on `stream` like the other calls.
 * ------------------------------------------------------------------------- */
moe_status moe_layer_stats(const void* topk_idx, int idx_bits, const int32_t* counts, int T, int K,
                           int E, int L, int R, const int32_t* rank_offsets, uint64_t* stats,
                           moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_expert_compute_gemm_launches -- how many launches the GEMMs of
 * moe_expert_compute_ex take on this device for these sizes and flags: 1 (both
 * GEMMs in one launch) or 2 (gate/up, then down); rows as for
 * moe_expert_compute_ex.  A negative moe_status for bad arguments or an
 * unsupported device.  Host only.
 * ------------------------------------------------------------------------- */
int moe_expert_compute_gemm_launches(int E, int R, int64_t rows, int I, int flags);

/* ---------------------------------------------------------------------------
 * moe_expert_compute_workspace_layout -- where moe_expert_compute_ex (and so
 * moe_expert_compute and moe_expert_compute_packed) keeps its intermediate
 * tensors inside the workspace, for callers that want to read them (FP8
 * activations, Z) or to run moe_dispatch_quant + moe_gemm_gateup_down on the
 * same workspace.  rows = 0: padded layout (E*R rows), else the packed row
 * count.  Writes 7 byte counts to offsets:
 *   [0] xq   e4m3 [rows, H]          [1] xs  fp32 [rows, H/128]
 *   [2] zq   e4m3 [rows, I]          [3] zs  fp32 [rows, I/128]
 *   [4] the GEMM launch's sync scratch, [5] its size in bytes
 *   [6] the workspace size (= moe_expert_compute_ex_workspace_size)
 * Every offset is a multiple of 256.  Returns MOE_ERR_INVALID_ARG for bad
 * sizes or a null offsets pointer.  Host only; touches no device memory.
 * ------------------------------------------------------------------------- */
int moe_expert_compute_workspace_layout(int E, int R, int64_t rows, int H, int I,
                                        size_t* offsets);

/* ---------------------------------------------------------------------------
 * Expert parallelism across ranks (one GPU each, W = E / L ranks, rank r holding
 * experts [r*L, r*L + L)) -- "SGLang、NCCL 与 MoE EP": §2.3.2 (a token sends one
 * payload to each distinct destination rank among its routes, with a header
 * carrying its route list), §2.3.4 (the destination writes one expert input per
 * route) and §3.2 (合对: every route's expert output goes back into that route's
 * result slot at the source, which applies the router weight and sums).  The
 * exchanges themselves are the caller's all-to-all (e.g. NCCL through
 * torch.distributed); these calls are each rank's data path around them:
 *
 * source      moe_ep_pack           -> send_x, send_ids, send_counts per rank
 *             (all-to-all of send_counts, then of send_x rows and send_ids rows)
 * destination moe_dispatch_ex(recv_x, recv_ids as int32 ids, E = L, R) and
 *             moe_expert_compute on the received rows; moe_ep_route_offsets on
 *             recv_ids; moe_ep_return -> one returned row per route
 *             (all-to-all of the returned rows and flags back)
 * source      moe_ep_route_offsets on send_ids; moe_ep_result_map;
 *             moe_combine_packed(returned rows, result_map, topk_w) -> y
 * Rows reach a destination grouped by source rank in ascending token order, so
 * with tokens numbered rank after rank the slots, capacity drops and y equal
 * those of moe_dispatch / moe_expert_compute / moe_combine on all ranks' tokens
 * on one GPU, bit for bit.
 *
 * moe_ep_pack
 *   x, topk_idx, idx_bits, T, H, K as for moe_dispatch_ex (global expert ids)
 *   send_x      device BF16 [T*min(K, W), H]: one row per (token, destination
 *               rank), rows for rank d back to back (d ascending), tokens
 *               ascending; send_counts device int32 [W]: rows for each rank
 *   send_ids    device int32 [T*min(K, W), K]: row u's destination-local
 *               expert id (global id % L) at each top-k position routed to
 *               that rank, -1 at the others
 *   route_msg, route_pos  device int32 [T, K]: the send row carrying route
 *               (t, k) and its position among that row's routes (-1 if none)
 *   dev_status  as for moe_dispatch (bad ids reported and ignored)
 *   workspace   moe_ep_pack_workspace_size(T, K, E, L) bytes, 256-byte aligned
 * moe_ep_route_offsets  offsets device int32 [S + 1]: offsets[j] = number of
 *               entries >= 0 in rows [0, j) of ids [S, K]; offsets[S] = all;
 *               workspace moe_ep_offsets_workspace_size(S) bytes
 * moe_ep_return  for each row j of ids [S, K] (the received send_ids) and each
 *               of its routes in k order: ret row offsets[j] + position = out
 *               row src_map[j, k] (the local layer's output and source map), or
 *               zeros with flag 0 if src_map is -1 (dropped for capacity).
 *               ret device BF16 [offsets[S], H]; flag device int32 [offsets[S]]
 * moe_ep_result_map  result_map device int32 [T, K]: for route (t, k) with
 *               message u = route_msg and position p, offsets[u] + p (offsets of
 *               the source's send_ids) if that returned row's flag is 1, else -1
 * ------------------------------------------------------------------------- */
size_t moe_ep_pack_workspace_size(int T, int K, int E, int L);
moe_status moe_ep_pack(const void* x, const void* topk_idx, int idx_bits, int T, int H, int K,
                       int E, int L, void* send_x, int32_t* send_ids, int32_t* send_counts,
                       int32_t* route_msg, int32_t* route_pos, int32_t* dev_status,
                       void* workspace, size_t workspace_bytes, moe_stream_t stream);
size_t moe_ep_offsets_workspace_size(int64_t S);
moe_status moe_ep_route_offsets(const int32_t* ids, int64_t S, int K, int32_t* offsets,
                                void* workspace, size_t workspace_bytes, moe_stream_t stream);
moe_status moe_ep_return(const void* out, int64_t out_rows, const int32_t* src_map,
                         const int32_t* ids, const int32_t* offsets, int64_t S, int K, int H,
                         void* ret, int32_t* flag, moe_stream_t stream);
moe_status moe_ep_result_map(const int32_t* route_msg, const int32_t* route_pos,
                             const int32_t* offsets, const int32_t* flag, int64_t n_ret, int T,
                             int K, int32_t* result_map, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_selftest_bounded_wait -- exercises the device-side failure path: the
 * kernels' two bounded waits run on things nothing completes, at the same
 * time (an mbarrier wait, and the acquire wait on a global completion counter
 * used by moe_gemm_gateup_down's down tiles).  After the wait limit (about
 * 2 s) each sets MOE_DEV_TIMEOUT in dev_status[0] and its bit in dev_status[1]
 * (1: mbarrier, 2: counter); the kernel returns normally.  dev_status is
 * int32[2], zeroed by the caller.  For tests of failure handling; no GPU fault
 * is involved.
 * ------------------------------------------------------------------------- */
moe_status moe_selftest_bounded_wait(int32_t* dev_status, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
