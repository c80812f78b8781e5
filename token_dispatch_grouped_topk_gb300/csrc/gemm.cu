// Grouped block-scaled FP8 GEMMs of the gated-SiLU expert on tcgen05.
//
// "SGLang Expert Compute Backend", §3.5: activations carry one fp32 scale per
// row per 128 K-elements, weights (stored [E, N, K]) one per 128x128 block, and
//   G[m, n] = sum_g  sx[m, g] * sw[n/128, g] * sum_{k in g} xq[m, k] * wq[n, k].
// §2.4: each expert's valid rows are tiled on their own; only tiles that hold
// valid rows are scheduled.  §3.6: the gate/up output's first I columns are
// gate and the last I up; Z = SiLU(gate) * up is re-quantised per row per 128
// for the down GEMM, whose output is written back at the original slot (§3.7).
//
// Design (one CTA per SM, persistent):
//  - tiles are 128 rows x BN columns of one expert; the tile list is derived on
//    the device from counts (prefix of ceil(count/128) per expert, times the
//    N slices per block).  The one-GEMM launch forms walk it with a stride of
//    gridDim.x; the two-GEMM form takes tiles from a ticket.  Within an expert the
//    walk is M-block major: the N slices of one 128-row block are adjacent,
//    so a block's activation rows are fetched once while the CTAs running at
//    the same time share the expert's weight slices in L2.  (Measured on
//    real FP8 activations at the large layer: the N-slice-major walk re-read
//    activation blocks once per slice and moved 25 GB per gate/up launch
//    against 20 GB, 12% slower.);
//  - warp 0 (one thread) streams A and B tiles with TMA (128-byte swizzle) into
//    a 4-stage shared-memory ring guarded by full/empty mbarriers;
//  - warp 1 (one thread) issues tcgen05.mma kind::f8f6f4 (M=128, N=BN, K=32,
//    fp32 accumulate) -- one 128-wide K group per TMEM buffer, two buffers, so
//    the tensor core fills one while the epilogue drains the other;
//  - warp 2 owns the TMEM allocation;
//  - warps 4-11 promote each K group's partial product: acc += sx * sw * P in
//    registers (the fp32 scales are not of a form the hardware block-scaled
//    MMA accepts).  Warp w reads TMEM lanes 32*(w%4).. (its lane quarter) and
//    one half of the tile's columns: 128 accumulators per thread, filled by
//    64-column TMEM loads (a load takes ~150 clocks, so 8 KB per warp must be
//    in flight for eight warps to drain 128x256 fp32 per K group in time) and
//    updated with packed two-lane fp32 FMAs.  The
//    register file is re-split per warpgroup (setmaxnreg): the producer/MMA
//    warpgroup drops to 40 registers, the two epilogue warpgroups rise to 232.
//    After the last K group they run the fused epilogue: SiLU(gate) * up and
//    the per-row FP8 requantisation of Z for the gate/up GEMM; for the down
//    GEMM BF16 rows staged through shared memory so each store instruction
//    writes 64-byte row segments.  Only rows below counts[e] are stored.
//  - one kernel serves three launch forms: the gate/up GEMM alone, the down
//    GEMM alone, or both ("XTuner Domino EP", HyperParallel-MoE section: a
//    task starts when the per-tile event counter it depends on reaches its
//    threshold, not when the whole preceding operator ends).  In the fused
//    form the tile list is every gate/up tile followed by every down tile;
//    the producer takes tiles in list order from a global ticket, so a tile
//    only ever waits for tiles already held by running CTAs, and passes each
//    to the MMA and epilogue warps through a small shared-memory ring.  Each
//    epilogue warp of a gate/up tile, after storing its 32 rows x 64 columns
//    of Z, adds one to its block's count (release); the producer publishes a
//    down tile of that block only after the count reaches 8 x the gate/up
//    tiles per block (acquire, bounded), then loads Z with TMA; the epilogue
//    reads Z's scales after taking the tile from the ring.  The down GEMM of
//    the first blocks so runs under the last gate/up wave instead of after it;
//  - the epilogue takes its next tile, and requests that tile's first scales,
//    before the current tile's tail whenever the tile is already published.
// Every wait is bounded; on expiry the kernel raises MOE_DEV_TIMEOUT in the
// status word, drains its own copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kStages = 4;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
// What one launch computes: the gate/up GEMM, the down GEMM, or both, with
// each down tile starting once the gate/up tiles of its 128-row block are done.
constexpr int kModeGateUp = 0;
constexpr int kModeDown = 1;
constexpr int kModeFused = 2;
// Fused launches hand tiles from the producer to the MMA and epilogue warps
// through a ring of this many slots.
constexpr int kTileSlots = 8;
// Register split: launched at kLaunchRegs per thread (the __launch_bounds__
// maximum for 384 threads); warpgroup 0 (producer, MMA, TMEM owner) gives
// back to kCtrlRegs, warpgroups 1-2 (epilogue) take kEpiRegs.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 40;
constexpr int kEpiRegs = 232;
static_assert(4 * kCtrlRegs + 8 * kEpiRegs == 12 * kLaunchRegs, "register split must fit the launch");
// Output staging (Z codes of gate/up tiles, BF16 rows of down tiles): per
// epilogue warp 32 rows x 64 bytes, rows padded to 80 bytes.
constexpr int kStageRowBytes = 80;
constexpr int kStageWarpBytes = 32 * kStageRowBytes;
constexpr int kMaxExperts = 1024;

struct GemmArgs {
  const int32_t* counts;
  const float* xs;         // [rows, H/128]: scales of the gate/up GEMM's activations
  const float* w13_scale;  // [E, 2I/128, H/128]
  const float* w2_scale;   // [E, H/128, I/128]
  uint8_t* zq;             // [rows, I]: written by gate/up tiles, read by down tiles
  float* zs;               // [rows, I/128]
  __nv_bfloat16* out;      // [rows, H]
  int* sched;              // fused: [0] tile ticket, [1 + b] epilogue warps done on block b
  int E, R, I, H;
  int nt_gu, nt_dn;        // N slices per 128-row block of each GEMM
  int packed;              // row layout of xq/xs, zq/zs and out (see RowLayout)
  int inter;               // W13 rows interleaved (2j gate, 2j+1 up) instead of the
                           // first I gate and the last I up
  long long rows;          // their row count
  int seg;                 // per-source slots: rows per source range (0: none)
  const int32_t* seg_counts;  // [E, R / seg] valid rows per range
  const int32_t* slot_of;  // per-source slots: slot row of each packed row (down stores)
  int32_t* dev_status;
};

// Tensor maps: activation boxes of 128, 64 and 32 rows and the weights, for
// the gate/up GEMM ([0]: xq, W13) and the down GEMM ([1]: zq, W2).
struct GemmMaps {
  CUtensorMap a[2][3];
  CUtensorMap b[2];
};

struct Control {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t tile_full[kTileSlots];
  uint64_t tile_empty[kTileSlots];
  uint64_t drain;
  uint64_t amax_bar;
  uint32_t tmem_base;
  int abort;
  int tile_slot[kTileSlots];
  int blk_start[kMaxExperts + 1];  // prefix of ceil(count / 128): expert e's first block
  // Padded layout: clamped count of expert e.  Packed layout: prefix of the
  // clamped counts (expert e's first row), cnt[E] = their sum.
  int cnt[kMaxExperts + 1];
  float amax[2][2][kBM];  // [tile parity][column half][row]
};

template <int BN, int kMode>
struct Layout {
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kOutStage = kEpiWarps * kStageWarpBytes;
  static constexpr size_t kSmem =
      1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(Control) + kOutStage;
};

// 227 KB of dynamic shared memory per block on sm_103.
static_assert(Layout<256, kModeGateUp>::kSmem <= 232448 &&
                  Layout<256, kModeDown>::kSmem <= 232448 &&
                  Layout<128, kModeDown>::kSmem <= 232448 &&
                  Layout<256, kModeFused>::kSmem <= 232448,
              "GEMM shared memory exceeds the per-block limit");

struct Tile {
  bool gu;   // a gate/up tile (else a down tile)
  int blk;   // 128-row block over all experts
  int e, m_blk, n_blk, rows;
  int base;  // buffer row of the tile's first row
};

// Tile t -> (GEMM, block, expert, N slice).  Each GEMM's tiles are M-block
// major (the N slices of one block adjacent); a fused launch lists all gate/up
// tiles before all down tiles.
template <int kMode>
__device__ __forceinline__ Tile decode_tile(const Control* ctl, const GemmArgs& a, int t) {
  Tile r;
  const int gu_tiles = kMode == kModeFused ? ctl->blk_start[a.E] * a.nt_gu : 0;
  r.gu = kMode == kModeGateUp || (kMode == kModeFused && t < gu_tiles);
  const int local = r.gu ? t : t - gu_tiles;
  const int nt = r.gu ? a.nt_gu : a.nt_dn;
  r.blk = local / nt;
  r.n_blk = local - r.blk * nt;
  r.e = find_expert(ctl->blk_start, a.E, r.blk);
  r.m_blk = r.blk - ctl->blk_start[r.e];
  const int count = a.packed ? ctl->cnt[r.e + 1] - ctl->cnt[r.e] : ctl->cnt[r.e];
  r.base = (a.packed ? ctl->cnt[r.e] : r.e * a.R) + r.m_blk * kBM;
  r.rows = min(kBM, count - r.m_blk * kBM);
  return r;
}

// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  int dummy = 0;
  mbar_wait(bar, parity, &dummy);
}

// Generic-proxy writes of Z (epilogue stores) and async-proxy reads of Z (the
// down tiles' TMA loads) are ordered on both sides with a proxy fence.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void red_add_release_gpu(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Scales written by this launch (Z's, in a fused launch) are read through L2.
__device__ __forceinline__ float ld_scale(const float* p, bool coherent) {
  return coherent ? __ldcg(p) : __ldg(p);
}

// Per-tile state of one epilogue thread: the tile, where its scales and TMEM
// columns are, and the scales of its first two K groups (requested ahead).
struct EpiTile {
  int t;  // tile index, -1: none left
  Tile tl;
  int nkb;
  bool in_cap, coherent;
  long long grow;  // buffer row of this thread
  const float* asc;
  const float* wsc0;
  const float* wsc1;
  uint32_t col0, col1;  // TMEM columns of this thread's two 64-column chunks
  float sa1, w01, w11, sa2, w02, w12;
};

// Tile `it` of this CTA for an epilogue warp.  Fused launches read it from the
// ring: with `wait` the warp waits (bounded) for the slot, without it takes the
// slot only if it is already published.  Returns 1 with *t set (-1: no tiles
// left), 0 if not yet published, -1 if the wait gave up.
__device__ __forceinline__ int epi_claim(Control* ctl, int it, bool fused, int total, bool wait,
                                         volatile int* abort, int lane, int* t) {
  if (!fused) {
    const int v = blockIdx.x + it * gridDim.x;
    *t = v < total ? v : -1;
    return 1;
  }
  const int slot = it % kTileSlots;
  const uint32_t par = (it / kTileSlots) & 1;
  const bool got = wait ? mbar_wait(&ctl->tile_full[slot], par, abort)
                        : mbar_try_wait(&ctl->tile_full[slot], par);
  if (!__all_sync(0xffffffffu, got)) return wait ? -1 : 0;
  *t = ctl->tile_slot[slot];
  __syncwarp();
  if (lane == 0) mbar_arrive(&ctl->tile_empty[slot]);
  return 1;
}

// Decodes p->t and requests the scales of its first two K groups.
template <int BN, int kMode>
__device__ __forceinline__ void epi_prepare(EpiTile* p, const Control* ctl, const GemmArgs& args,
                                            int row, int ch) {
  constexpr int kCols = BN / 2;
  const Tile tl = decode_tile<kMode>(ctl, args, p->t);
  p->tl = tl;
  const int nkb = (tl.gu ? args.H : args.I) / kBK;
  p->nkb = nkb;
  // A fused down tile reads Z's scales, written by other CTAs of this launch:
  // the producer published the tile only after acquiring its block's
  // completion, and the loads go through L2.
  p->coherent = kMode == kModeFused && !tl.gu;
  const int m = tl.m_blk * kBM + row;
  p->grow = static_cast<long long>(tl.base) + row;
  // Scales are read for rows inside the expert's capacity (padded) or the
  // buffer (packed); rows past the count are promoted but never stored.
  p->in_cap = args.packed ? p->grow < args.rows : m < args.R;
  p->asc = (tl.gu ? args.xs : args.zs) + (p->in_cap ? p->grow : 0) * nkb;
  // gate/up: gate columns [64ch, 64ch+64) and up columns [128+64ch, ..+64);
  // down:    columns [kCols*ch, kCols*ch + kCols), inside one 128-column
  //          weight-scale block.
  //          Interleaved gate/up: columns [128ch, 128ch+128), 64 (gate, up)
  //          pairs inside one 128-row weight-scale block.
  if (tl.gu && args.inter) {
    const int nb = 2 * args.I / 128;
    p->wsc0 = args.w13_scale + (static_cast<size_t>(tl.e) * nb + 2 * tl.n_blk + ch) * nkb;
    p->wsc1 = p->wsc0;
    p->col0 = static_cast<uint32_t>(ch * 128);
    p->col1 = p->col0 + 64;
  } else if (tl.gu) {
    const int nb = 2 * args.I / 128;
    p->wsc0 = args.w13_scale + (static_cast<size_t>(tl.e) * nb + tl.n_blk) * nkb;
    p->wsc1 = args.w13_scale + (static_cast<size_t>(tl.e) * nb + args.I / 128 + tl.n_blk) * nkb;
    p->col0 = static_cast<uint32_t>(ch * 64);
    p->col1 = p->col0 + 128;
  } else {
    const int nb = args.H / 128;
    const int cb = (tl.n_blk * BN + ch * kCols) / 128;
    p->wsc0 = args.w2_scale + (static_cast<size_t>(tl.e) * nb + cb) * nkb;
    p->wsc1 = p->wsc0;
    p->col0 = static_cast<uint32_t>(ch * kCols);
    p->col1 = p->col0 + 64;
  }
  p->sa1 = p->in_cap ? ld_scale(p->asc, p->coherent) : 0.f;
  p->w01 = __ldg(p->wsc0);
  p->w11 = __ldg(p->wsc1);
  p->sa2 = p->w02 = p->w12 = 0.f;
  if (nkb > 1) {
    p->sa2 = p->in_cap ? ld_scale(p->asc + 1, p->coherent) : 0.f;
    p->w02 = __ldg(p->wsc0 + 1);
    p->w12 = __ldg(p->wsc1 + 1);
  }
}

template <int BN, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  using L = Layout<BN, kMode>;
  constexpr bool kFused = kMode == kModeFused;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Control* ctl = reinterpret_cast<Control*>(smem + kStages * L::kStageBytes);
  uint8_t* out_stage = smem + kStages * L::kStageBytes + sizeof(Control);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->tfull[i], 1);
      mbar_init(&ctl->tempty[i], kEpiThreads / 32);
    }
    for (int i = 0; i < kTileSlots; ++i) {
      mbar_init(&ctl->tile_full[i], 1);
      mbar_init(&ctl->tile_empty[i], 1 + kEpiWarps);   // the MMA thread + each epilogue warp
    }
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->amax_bar, kEpiThreads);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < 4) {
    const int g = kMode == kModeDown ? 1 : 0;
    tma_prefetch_desc(lane < 3 ? &maps.a[g][lane] : &maps.b[g]);
    if (kFused) tma_prefetch_desc(lane < 3 ? &maps.a[1][lane] : &maps.b[1]);
  }
  if (warp == 2) {
    tmem_alloc(&ctl->tmem_base, L::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  // Block prefix per expert (ends with __syncthreads, which also publishes the
  // barrier initialisation and the TMEM address).
  // per-source slots: each expert's tiles cover its packed valid rows
  if (args.seg) source_slot_totals(args.seg_counts, args.E, args.R, args.seg, ctl->cnt);
  expert_prefix(args.seg ? ctl->cnt : args.counts, args.E, args.R, kBM, 1, ctl->blk_start,
                ctl->cnt);
  if (args.packed) expert_prefix(args.counts, args.E, args.R, 1, 1, ctl->cnt, nullptr);
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int nblk = ctl->blk_start[args.E];
  const int total = nblk * ((kMode == kModeDown ? 0 : args.nt_gu) +
                            (kMode == kModeGateUp ? 0 : args.nt_dn));
  const int done_target = kEpiWarps * args.nt_gu;   // fused: signals that complete a block's Z
  volatile int* abort_flag = &ctl->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    warpgroup_reg_dealloc<kCtrlRegs>();
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      for (int it = 0;; ++it) {
        int t;
        if (kFused) {
          // Tiles are taken in list order by whichever CTAs are running, so
          // every gate/up tile a down tile waits for is held by a running CTA
          // that never waits on anything else first.
          const int slot = it % kTileSlots;
          if (!mbar_wait(&ctl->tile_empty[slot], ((it / kTileSlots) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          t = atomicAdd(args.sched, 1);
          if (t >= total) t = -1;
          // A down tile is published only once the gate/up tiles of its block
          // are done (acquire): the MMA and epilogue warps that take it from
          // the ring are then ordered after Z's stores.
          if (t >= 0) {
            const Tile dt = decode_tile<kMode>(ctl, args, t);
            if (!dt.gu) {
              if (!wait_count(args.sched + 1 + dt.blk, done_target, abort_flag)) {
                ok = false;
                break;
              }
              fence_proxy_async_global();
            }
          }
          ctl->tile_slot[slot] = t;
          mbar_arrive(&ctl->tile_full[slot]);
        } else {
          t = blockIdx.x + it * gridDim.x;
          if (t >= total) t = -1;
        }
        if (t < 0) break;
        const Tile tl = decode_tile<kMode>(ctl, args, t);
        const int g = tl.gu ? 0 : 1;
        const int nkb = (tl.gu ? args.H : args.I) / kBK;
        const int a_row = tl.base;
        int b_row0, b_row1;
        if (tl.gu && args.inter) {         // 256 consecutive interleaved rows
          b_row0 = tl.e * 2 * args.I + tl.n_blk * 256;
          b_row1 = b_row0 + 128;
        } else if (tl.gu) {
          b_row0 = tl.e * 2 * args.I + tl.n_blk * 128;
          b_row1 = b_row0 + args.I;
        } else {
          b_row0 = tl.e * args.H + tl.n_blk * BN;
          b_row1 = b_row0 + 128;
        }
        // Only the tile's valid activation rows are fetched (32, 64 or 128):
        // the rest of the A tile keeps stale bytes, which reach only output
        // rows that are never stored.
        const int a_box = tl.rows <= 32 ? 32 : (tl.rows <= 64 ? 64 : kBM);
        const CUtensorMap* ma = &maps.a[g][a_box == kBM ? 0 : (a_box == 64 ? 1 : 2)];
        const CUtensorMap* mb = &maps.b[g];
        for (int kb = 0; kb < nkb; ++kb) {
          const int stage = issued % kStages;
          const uint32_t phase = (issued / kStages) & 1;
          if (!mbar_wait(&ctl->empty[stage], phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * L::kStageBytes;
          uint8_t* sb = sa + L::kABytes;
          mbar_arrive_expect_tx(&ctl->full[stage], L::kBBytes + a_box * kBK);
          tma_load_2d(sa, ma, &ctl->full[stage], kb * kBK, a_row);
          tma_load_2d(sb, mb, &ctl->full[stage], kb * kBK, b_row0);
          if (BN == 256) tma_load_2d(sb + 128 * kBK, mb, &ctl->full[stage], kb * kBK, b_row1);
          ++issued;
        }
        if (!ok) break;
      }
      if (!ok) *abort_flag = 1;
      // No copy may land after the block exits: wait for the last loads.
      for (int i = 0; i < min(issued, kStages); ++i) {
        const int n = issued - 1 - i;
        drain_wait(&ctl->full[n % kStages], (n / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    warpgroup_reg_dealloc<kCtrlRegs>();
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, BN);
      int consumed = 0, kcount = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int t;
        if (kFused) {
          const int slot = it % kTileSlots;
          if (!mbar_wait(&ctl->tile_full[slot], (it / kTileSlots) & 1, abort_flag)) {
            ok = false;
            break;
          }
          t = ctl->tile_slot[slot];
          mbar_arrive(&ctl->tile_empty[slot]);
        } else {
          t = blockIdx.x + it * gridDim.x;
          if (t >= total) t = -1;
        }
        if (t < 0) break;
        const int gu_tiles = kFused ? nblk * args.nt_gu : 0;
        const bool gu = kMode == kModeGateUp || (kFused && t < gu_tiles);
        const int nkb = (gu ? args.H : args.I) / kBK;
        for (int kb = 0; kb < nkb; ++kb) {
          const int stage = consumed % kStages;
          const uint32_t phase = (consumed / kStages) & 1;
          const int acc = kcount & 1;
          const uint32_t acc_phase = (kcount >> 1) & 1;
          if (!mbar_wait(&ctl->tempty[acc], acc_phase ^ 1, abort_flag) ||
              !mbar_wait(&ctl->full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * L::kStageBytes);
          const uint64_t adesc = smem_desc_kmajor_sw128(sa);
          const uint64_t bdesc = smem_desc_kmajor_sw128(sa + L::kABytes);
          const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k)  // 32 e4m3 = 32 bytes = 2 descriptor units
            mma_e4m3(d, adesc + 2 * k, bdesc + 2 * k, kIdesc, k > 0 ? 1u : 0u);
          mma_commit(&ctl->empty[stage]);
          mma_commit(&ctl->tfull[acc]);
          ++consumed;
          ++kcount;
        }
      }
      if (!ok) *abort_flag = 1;
      if (kcount > 0) {
        mma_commit(&ctl->drain);
        drain_wait(&ctl->drain, 0);
      }
    }
  } else if (warp < kEpiWarp0) {
    warpgroup_reg_dealloc<kCtrlRegs>();   // warps 2-3: TMEM owner and spare
  } else {
    // ------------------------------------------------------------ epilogue
    warpgroup_reg_alloc<kEpiRegs>();
    constexpr int kCols = BN / 2;   // columns of the tile this thread owns
    constexpr int kPairs = kCols / 2;
    const int ew = warp - kEpiWarp0;
    const int lq = warp & 3;        // TMEM lane quarter accessible to this warp
    const int ch = ew >> 2;         // which half of the tile's columns
    const int row = lq * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(lq * 32) << 16);
    int kcount = 0, gu_iter = 0;
    bool ok = true;
    EpiTile cur;
    cur.t = -1;
    {
      int t = -1;
      if (epi_claim(ctl, 0, kFused, total, true, abort_flag, lane, &t) < 0) ok = false;
      cur.t = t;
      if (ok && t >= 0) epi_prepare<BN, kMode>(&cur, ctl, args, row, ch);
    }
    for (int it = 0; ok && cur.t >= 0; ++it) {
      const Tile tl = cur.tl;
      const long long grow = cur.grow;   // buffer row of this thread
      uint64_t acc2[kPairs];
#pragma unroll
      for (int i = 0; i < kPairs; ++i) acc2[i] = 0;
      // Scales of K groups kb+1 and kb+2 are in flight while group kb is promoted.
      float sa1 = cur.sa1, w01 = cur.w01, w11 = cur.w11;
      float sa2 = cur.sa2, w02 = cur.w02, w12 = cur.w12;
      const int nkb = cur.nkb;
      for (int kb = 0; kb < nkb; ++kb) {
        const float s0 = sa1 * w01;
        const float s1 = sa1 * w11;
        sa1 = sa2;
        w01 = w02;
        w11 = w12;
        if (kb + 2 < nkb) {
          sa2 = cur.in_cap ? ld_scale(cur.asc + kb + 2, cur.coherent) : 0.f;
          w02 = __ldg(cur.wsc0 + kb + 2);
          w12 = __ldg(cur.wsc1 + kb + 2);
        }
        const int acc = kcount & 1;
        const uint32_t acc_phase = (kcount >> 1) & 1;
        if (!mbar_wait(&ctl->tfull[acc], acc_phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = t_lane + static_cast<uint32_t>(acc * BN);
        const uint64_t s0x2 = f32x2_pack(s0, s0);
        const uint64_t s1x2 = f32x2_pack(s1, s1);
        // Chunk j of 64 columns (one TMEM load, 8 KB per warp in flight):
        // gate/up j = 0 gate, j = 1 up; down j = 0 .. kCols/64-1, all with
        // the one scale of their 128-column block.
        uint32_t buf[64];
#pragma unroll
        for (int j = 0; j < kCols / 64; ++j) {
          const uint32_t col = j ? cur.col1 : cur.col0;
          const uint64_t sx2 = (tl.gu && j) ? s1x2 : s0x2;
          if constexpr (kMode == kModeDown)
            tmem_load64_sync_2x32(base + col, buf);
          else
            tmem_load64_sync(base + col, buf);
#pragma unroll
          for (int i = 0; i < 32; ++i) ffma2_acc(acc2[32 * j + i], sx2, buf[2 * i], buf[2 * i + 1]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->tempty[acc]);
        ++kcount;
      }
      if (!ok) break;
      // The next tile is taken, and its first scales requested, before this
      // tile's tail when it is already published, so their latency is hidden
      // behind the tail.  Otherwise (its block may be waiting for this very
      // tile's Z) it is taken after the tail.
      EpiTile nxt;
      nxt.t = -1;
      int t_next = -1;
      const bool early = epi_claim(ctl, it + 1, kFused, total, false, abort_flag, lane, &t_next) > 0;
      if (early) {
        nxt.t = t_next;
        if (t_next >= 0) epi_prepare<BN, kMode>(&nxt, ctl, args, row, ch);
      }
      // rows stored: inside the tile's valid range and the buffer; bit r of
      // vmask is the warp's row r
      const bool valid = row < tl.rows && grow < args.rows;
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
      if (kMode != kModeDown && tl.gu) {
        // Z = SiLU(gate) * up on this thread's 64 columns (written over the
        // gate half of acc2), then the row amax over the tile's 128 Z columns
        // shared with the partner warp holding the other half.  SiLU uses the
        // fast exponential and division intrinsics: their few-ulp error is far
        // below the fp32 accumulation's, and the IEEE forms cost 7-17 % of the
        // launch at the decode and prefill shapes.  For g -> -inf the quotient
        // tends to 0, as SiLU does.
        float amax = 0.f;
        if (args.inter) {
          // pair p holds (gate, up) of feature 64ch + p; Z of features 2i and
          // 2i+1 go to acc2[i] (written after both pairs are read)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float g0 = f32x2_lo(acc2[2 * i]), u0 = f32x2_hi(acc2[2 * i]);
            const float g1 = f32x2_lo(acc2[2 * i + 1]), u1 = f32x2_hi(acc2[2 * i + 1]);
            const float z0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            const float z1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
            acc2[i] = f32x2_pack(z0, z1);
            amax = fmaxf(amax, fmaxf(fabsf(z0), fabsf(z1)));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float g0 = f32x2_lo(acc2[i]), g1 = f32x2_hi(acc2[i]);
            const float u0 = f32x2_lo(acc2[32 + i]), u1 = f32x2_hi(acc2[32 + i]);
            const float z0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            const float z1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
            acc2[i] = f32x2_pack(z0, z1);
            amax = fmaxf(amax, fmaxf(fabsf(z0), fabsf(z1)));
          }
        }
        const int par = gu_iter & 1;
        ++gu_iter;
        ctl->amax[par][ch][row] = amax;
        mbar_arrive(&ctl->amax_bar);
        if (!mbar_wait(&ctl->amax_bar, par, abort_flag)) {
          ok = false;
          break;
        }
        amax = fmaxf(ctl->amax[par][0][row], ctl->amax[par][1][row]);
        float mult, scale;
        fp8_group_scale(amax, &mult, &scale);
        {
          // The warp's 32 rows x 64 Z bytes go through its shared-memory stage,
          // so each store instruction writes 8 rows x 64 bytes.
          uint8_t* stage = out_stage + ew * kStageWarpBytes;
          uint4* srow = reinterpret_cast<uint4*>(stage + lane * kStageRowBytes);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint64_t za = acc2[8 * j + 2 * i], zb = acc2[8 * j + 2 * i + 1];
              w[i] = static_cast<uint32_t>(pack_e4m3x2(__fmul_rn(f32x2_lo(za), mult),
                                                       __fmul_rn(f32x2_hi(za), mult))) |
                     (static_cast<uint32_t>(pack_e4m3x2(__fmul_rn(f32x2_lo(zb), mult),
                                                        __fmul_rn(f32x2_hi(zb), mult)))
                      << 16);
            }
            srow[j] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
          const long long grow0 = static_cast<long long>(tl.base) + lq * 32;  // warp's first row
          const int c = lane & 3;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = 8 * i + (lane >> 2);
            if ((vmask >> r) & 1u) {
              const uint4 v = *reinterpret_cast<const uint4*>(stage + r * kStageRowBytes + 16 * c);
              *reinterpret_cast<uint4*>(args.zq + (grow0 + r) * args.I + tl.n_blk * 128 + ch * 64 +
                                        16 * c) = v;
            }
          }
          __syncwarp();
        }
        if (valid) {
          if (ch == 0)
            args.zs[grow * (args.I / 128) + tl.n_blk] = scale;
        }
        if (kFused) {
          // Publish this warp's part of the block's Z (32 rows x 64 columns
          // and their scales) to the down tiles of other CTAs.
          fence_proxy_async_global();
          __threadfence();
          __syncwarp();
          if (lane == 0) red_add_release_gpu(args.sched + 1 + tl.blk, 1);
        }
      } else if (kMode != kModeGateUp) {
        // BF16 rows through a per-warp shared-memory stage: each round the
        // 32 threads deposit 32 columns of their rows, then the warp writes
        // 8 rows x 64 bytes per store instruction.
        uint8_t* stage = out_stage + ew * kStageWarpBytes;
        const long long grow0 = static_cast<long long>(tl.base) + lq * 32;  // warp's first row
        __nv_bfloat16* gbase = args.out + grow0 * args.H + tl.n_blk * BN + ch * kCols;
        // lane -> (row 8i + lane/4, 16-byte chunk lane%4) of each store instruction i
        const int c = lane & 3;
        const uint32_t goff = static_cast<uint32_t>((lane >> 2) * args.H + 8 * c);
        const uint32_t sidx = static_cast<uint32_t>((lane >> 2) * kStageRowBytes + 16 * c);
        const uint32_t gstep = static_cast<uint32_t>(8 * args.H);
        // per-source slots: packed row -> its slot row, as an offset from the
        // packed row of this lane's store rows 8i + lane/4
        long long soff[4] = {0, 0, 0, 0};
        if (args.seg) {
          const long long mine = valid ? static_cast<long long>(args.slot_of[grow]) -
                                             (static_cast<long long>(tl.m_blk) * kBM + row)
                                       : 0;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            soff[i] = __shfl_sync(0xffffffffu, mine, 8 * i + (lane >> 2)) * args.H;
        }
#pragma unroll
        for (int r = 0; r < kCols / 32; ++r) {
          uint4* srow = reinterpret_cast<uint4*>(stage + lane * kStageRowBytes);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int p = 16 * r + 4 * j;
            uint4 o;
            o.x = pack_bf16x2_rn(f32x2_lo(acc2[p + 0]), f32x2_hi(acc2[p + 0]));
            o.y = pack_bf16x2_rn(f32x2_lo(acc2[p + 1]), f32x2_hi(acc2[p + 1]));
            o.z = pack_bf16x2_rn(f32x2_lo(acc2[p + 2]), f32x2_hi(acc2[p + 2]));
            o.w = pack_bf16x2_rn(f32x2_lo(acc2[p + 3]), f32x2_hi(acc2[p + 3]));
            srow[j] = o;
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if ((vmask >> (8 * i + (lane >> 2))) & 1u) {
              const uint4 v = *reinterpret_cast<const uint4*>(stage + sidx + i * 8 * kStageRowBytes);
              *reinterpret_cast<uint4*>(gbase + soff[i] + goff + i * gstep + 32 * r) = v;
            }
          }
          __syncwarp();
        }
      }
      if (!early) {
        if (epi_claim(ctl, it + 1, kFused, total, true, abort_flag, lane, &t_next) < 0) {
          ok = false;
          break;
        }
        nxt.t = t_next;
        if (t_next >= 0) epi_prepare<BN, kMode>(&nxt, ctl, args, row, ch);
      }
      cur = nxt;
    }
    if (!ok) *abort_flag = 1;
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0 && ctl->abort) atomicOr(args.dev_status, kDevTimeout);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2D map over a row-major byte matrix [rows, cols] with boxes of 128 bytes x
// box_rows and the 128-byte swizzle the MMA descriptors expect.
cudaError_t make_map_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                        uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                         box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Activation maps with 128-, 64- and 32-row boxes.
cudaError_t make_activation_maps(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  cudaError_t err = make_map_u8(&m[0], base, cols, rows, kBM);
  if (err == cudaSuccess) err = make_map_u8(&m[1], base, cols, rows, 64);
  if (err == cudaSuccess) err = make_map_u8(&m[2], base, cols, rows, 32);
  return err;
}

template <int BN, int kMode>
cudaError_t launch_impl(const GemmMaps& maps, const GemmArgs& a, long long max_tiles, int sm_count,
                        cudaStream_t s) {
  using L = Layout<BN, kMode>;
  // The setmaxnreg split assumes the kernel was compiled to exactly
  // kLaunchRegs registers per thread; any other count could leave the
  // epilogue's register increase waiting forever, so refuse to launch.
  static const int compiled_regs = [] {
    cudaFuncAttributes attr{};
    return cudaFuncGetAttributes(&attr, grouped_gemm_kernel<BN, kMode>) == cudaSuccess
               ? attr.numRegs
               : -1;
  }();
  if (compiled_regs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  const int grid = static_cast<int>(std::min<long long>(max_tiles, sm_count));
  if (grid <= 0) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<BN, kMode>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::kSmem));
  if (err != cudaSuccess) return err;
  grouped_gemm_kernel<BN, kMode><<<grid, kThreads, L::kSmem, s>>>(maps, a);
  return cudaGetLastError();
}

// Upper bound on the 128-row blocks of a launch: every expert's count is
// clamped to R, and in the packed layout the blocks also fit in ceil(rows/128)
// plus one partial block per expert.
long long max_blocks(int E, RowLayout rl) {
  const long long padded = static_cast<long long>(E) * ((rl.R + kBM - 1) / kBM);
  return rl.packed ? std::min<long long>(padded, (rl.rows + kBM - 1) / kBM + E) : padded;
}

GemmArgs common_args(const int32_t* counts, int E, RowLayout rl, int H, int I,
                     int32_t* dev_status) {
  GemmArgs a{};
  a.counts = counts;
  a.E = E;
  a.R = rl.R;
  a.I = I;
  a.H = H;
  a.nt_gu = I / 128;
  a.nt_dn = H % 256 == 0 ? H / 256 : H / 128;
  a.packed = rl.packed;
  a.rows = rl.rows;
  a.seg = rl.seg;
  a.seg_counts = rl.seg_counts;
  a.slot_of = rl.slot_of;
  a.dev_status = dev_status;
  return a;
}

cudaError_t gateup_maps(GemmMaps* m, const uint8_t* xq, int E, RowLayout rl, int H, int I,
                        const uint8_t* w13) {
  cudaError_t err = make_activation_maps(m->a[0], xq, H, static_cast<uint64_t>(rl.rows));
  if (err == cudaSuccess)
    err = make_map_u8(&m->b[0], w13, H, static_cast<uint64_t>(E) * 2 * I, kBM);
  return err;
}

cudaError_t down_maps(GemmMaps* m, const uint8_t* zq, int E, RowLayout rl, int H, int I,
                      const uint8_t* w2) {
  cudaError_t err = make_activation_maps(m->a[1], zq, I, static_cast<uint64_t>(rl.rows));
  if (err == cudaSuccess) err = make_map_u8(&m->b[1], w2, I, static_cast<uint64_t>(E) * H, kBM);
  return err;
}

}  // namespace

cudaError_t launch_gemm_gateup(const uint8_t* xq, const float* xs, const int32_t* counts, int E,
                               RowLayout rl, int H, int I, const uint8_t* w13,
                               const float* w13_scale, uint8_t* zq, float* zs,
                               int32_t* dev_status, int sm_count, cudaStream_t s,
                               int w13_interleaved) {
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  GemmMaps maps{};
  cudaError_t err = gateup_maps(&maps, xq, E, rl, H, I, w13);
  if (err != cudaSuccess) return err;
  GemmArgs a = common_args(counts, E, rl, H, I, dev_status);
  a.xs = xs;
  a.w13_scale = w13_scale;
  a.zq = zq;
  a.zs = zs;
  a.inter = w13_interleaved ? 1 : 0;
  return launch_impl<256, kModeGateUp>(maps, a, max_blocks(E, rl) * a.nt_gu, sm_count, s);
}

cudaError_t launch_gemm_down(const uint8_t* zq, const float* zs, const int32_t* counts, int E,
                             RowLayout rl, int H, int I, const uint8_t* w2, const float* w2_scale,
                             void* out, int32_t* dev_status, int sm_count, cudaStream_t s) {
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  GemmMaps maps{};
  cudaError_t err = down_maps(&maps, zq, E, rl, H, I, w2);
  if (err != cudaSuccess) return err;
  GemmArgs a = common_args(counts, E, rl, H, I, dev_status);
  a.zq = const_cast<uint8_t*>(zq);
  a.zs = const_cast<float*>(zs);
  a.w2_scale = w2_scale;
  a.out = static_cast<__nv_bfloat16*>(out);
  const long long tiles = max_blocks(E, rl) * a.nt_dn;
  if (H % 256 == 0) return launch_impl<256, kModeDown>(maps, a, tiles, sm_count, s);
  return launch_impl<128, kModeDown>(maps, a, tiles, sm_count, s);
}

bool gemm_prefer_one_launch(int E, RowLayout rl, int I, int sm_count) {
  // Measured on the three layer shapes (same process, interleaved): with the
  // gate/up tiles spanning ~5 waves of CTAs (decode) the one launch is 3-5 %
  // faster, the down tiles of finished blocks filling the last wave; with
  // 100+ waves (prefill, large) the two launches are 6-8 % faster.
  return max_blocks(E, rl) * (I / 128) <= 16LL * sm_count;
}

size_t gemm_sync_ints(int E, RowLayout rl) {
  return 1 + static_cast<size_t>(max_blocks(E, rl));
}

cudaError_t launch_gemm_gateup_down(const uint8_t* xq, const float* xs, const int32_t* counts,
                                    int E, RowLayout rl, int H, int I, const uint8_t* w13,
                                    const float* w13_scale, const uint8_t* w2,
                                    const float* w2_scale, uint8_t* zq, float* zs, void* out,
                                    int* sync, size_t sync_ints, int32_t* dev_status,
                                    int sm_count, cudaStream_t s, int w13_interleaved) {
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  // The fused kernel runs 256-column down tiles only.
  if (H % 256 != 0) {
    cudaError_t err = launch_gemm_gateup(xq, xs, counts, E, rl, H, I, w13, w13_scale, zq, zs,
                                         dev_status, sm_count, s, w13_interleaved);
    if (err != cudaSuccess) return err;
    return launch_gemm_down(zq, zs, counts, E, rl, H, I, w2, w2_scale, out, dev_status,
                            sm_count, s);
  }
  const size_t need = gemm_sync_ints(E, rl);
  if (sync == nullptr || sync_ints < need) return cudaErrorInvalidValue;
  GemmMaps maps{};
  cudaError_t err = gateup_maps(&maps, xq, E, rl, H, I, w13);
  if (err == cudaSuccess) err = down_maps(&maps, zq, E, rl, H, I, w2);
  if (err != cudaSuccess) return err;
  GemmArgs a = common_args(counts, E, rl, H, I, dev_status);
  a.xs = xs;
  a.w13_scale = w13_scale;
  a.w2_scale = w2_scale;
  a.zq = zq;
  a.zs = zs;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.sched = sync;
  a.inter = w13_interleaved ? 1 : 0;
  // Tile ticket and per-block completion counts start at zero every launch.
  err = cudaMemsetAsync(sync, 0, need * sizeof(int), s);
  if (err != cudaSuccess) return err;
  return launch_impl<256, kModeFused>(maps, a, max_blocks(E, rl) * (a.nt_gu + a.nt_dn), sm_count,
                                      s);
}

}  // namespace moe
