// Implicit-GEMM convolutions on CTA pairs: tcgen05.mma with .cta_group::2 (M = 256 over two SMs).
//
// Same computations as conv_tc.cu (mode 0: the causal 3x3x3 convolution with its cache frames,
// binding.cpp `Decoder::conv`; mode 1: the four 2x2 phase convolutions of the upsampler,
// `Decoder::up`), for output-channel blocks of 256. Why a second kernel: with one CTA per tile,
// an M128 x N256 x K16 MMA reads 12 KB of operands from shared memory while the TMA unit writes
// the next 12 KB, which is more shared-memory traffic per SM than the SM can serve. On a CTA pair
// (a cluster of 2 on two SMs) each SM holds its own 128 output rows of A and HALF of B (128 of the
// 256 weight rows); one thread of the even CTA issues the M256 x N256 MMAs that read both SMs'
// halves, and each SM's TMEM receives its 128 rows.
//
// Operand traffic. A CTA's 128 output pixels are one frame x 8 rows x 16 columns, stored in shared
// memory column-major (row m = h + 8 w: the activation tensor map lists H before W). One TMA box of
// 8 rows x 18 columns (the tile plus a column on each side) then holds the A operand of all three
// horizontal taps of a kernel row: tap dw starts 8 * (dw + 1) rows = 1024 bytes further, a whole
// 128-byte-swizzle atom, so the plain descriptor addresses it. The box is loaded once per (kernel
// row, K block) instead of once per tap, which cuts the bytes per MMA from 32 KB (A + B per K
// block) to about 22 KB. A and B have separate rings; MMA order per accumulator is kernel row,
// K block, horizontal tap, K step.
//
// Pair protocol (all waits bounded):
//   full_a[s], full_b[s]  in the even CTA: both CTAs' TMA bytes for the stage (the odd CTA's loads
//                         complete on the even CTA's barrier directly)
//   empty_a[s], empty_b[s] both CTAs: the MMAs reading the stage are done (multicast commit)
//   tmem_full[a]          both CTAs: accumulator a holds a finished tile (multicast commit)
//   tmem_empty[a]         in the even CTA: both CTAs' epilogues drained accumulator a (8 warps)
// Items: (N block, phase, pair of pixel tiles); the even CTA computes the first tile, the odd CTA
// the second (a missing second tile loads zeros and stores nothing). Both tiles of a pair use the
// same weights, so in mode 1 a pair never mixes phases. Items go to the CTA pairs in snake order
// (round r: pair c takes item r * P + c, or r * P + P - 1 - c on odd rounds), which evens out
// items of different cost (the first frames of a chunk without history skip taps). When the last
// round holds at most P / 2 items, each of them is scheduled as two halves of 128 output channels
// (M256 x N128 MMAs, 64 weight rows per SM) on twice as many pairs: that round would otherwise
// leave most pairs idle (the C=1024 stage's 240 items over 76 pairs). A half computes the same
// output elements with the same sequence of K steps as the whole item, so the split changes no
// result.
//
// Modes (run time) and kinds (compile time, Cfg below). Mode 0 is the causal 3x3x3 conv, 1 the
// phase convs, 2 the causal 3x1x1 time conv with one output frame per CTA (the time upsample call
// has a kernel of its own, time_up_tc2.cu), and 3 the 1x1x1 conv of a channel-changing shortcut.
// Kind 0 is the plain kernel on 8 x 16 tiles. Kind 1 adds the GroupNorm + SiLU operand prologue
// and takes tall 10 x 18 boxes, one box holding a tap column's three kernel rows. Kind 2 is the
// phase convs with one tall box per K block. Kind 3 is kind 1 on 16 x 8 tiles, with 18 x 10 boxes
// stored row by row.
//
// MMA issue. One thread issues every MMA of the pair, and its issue rate, not the tensor pipe, was
// the limit: with a wait, a fence and a stage release per tap inside a run-time loop, each MMA
// took ~160 cycles to issue against 128 to execute (M256 x N256 x K16), whatever N was. Each A box
// is therefore issued as one straight-line burst (9 taps of a tall box, 3 of a plain mode-0 box,
// 2 of a phase box, two consecutive 1-tap boxes in modes 2 and 3) whose descriptors differ by
// constants; the B ring is used 9 or 8 stages deep so that no burst wraps it. The halves of the
// last round, whose N128 MMAs are short, take their B stages in groups of 3 (2 in phase mode) that
// land on one barrier and are released by one commit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "tma_host.h"
#include "conv_tc.h"

namespace wan {

namespace {

constexpr int kBlockK = 64;
constexpr int kTileH = 8, kTileW = 16;  // output pixels of one CTA: 8 rows x 16 columns
constexpr int kBoxW = kTileW + 2;       // input columns of one A box (one halo column per side)
constexpr int kABytes = kTileH * kBoxW * 128;  // 144 rows x 64 bf16 = 18 KB
constexpr int kBBytes = 128 * 128;             // this CTA's 128 weight rows x 64 bf16
constexpr int kN = 256;                 // output channels per item (both halves)
constexpr int kTmemCols = 512;          // 2 accumulators x 256 columns
constexpr uint32_t kShiftDesc = (kTileH * 128) >> 4;  // one column of the box, in descriptor units
constexpr int kCoefBytes = kBlockK * 16;                // GroupNorm coefficients of one A stage
constexpr int kTallRows = kTileH + 2;                   // rows of a tall A box (one halo row per side)
constexpr int kPhaseRows = kTileH + 1;                  // rows of a phase box (taps u = 0, 1)

static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
// Stage rings and shared memory. The plain kernel: producer, MMA issuer, 4 epilogue warps. With
// the GroupNorm + SiLU operand prologue: 8 more warps that normalise each A box in place between
// its arrival and the MMAs.
// Kernel kinds: 0 plain, 1 with the GroupNorm + SiLU operand prologue (mode 0), 2 the phase
// convolutions of mode 1 with one tall A box per K block, 3 kind 1 on tiles of 16 rows x 8
// columns (boxes stored row by row; chosen where it pads the frame less, e.g. 176 x 312).
template <int kKind>
struct Cfg {
  static constexpr bool kNorm = kKind == 1 || kKind == 3;
  static constexpr bool kPhase = kKind == 2;
  // Tile orientation. kWFast: the tile is 16 rows x 8 columns and its boxes land in shared memory
  // row by row (the tensor map lists W before H), TMEM row m = w + 8 h; otherwise 8 rows x 16
  // columns, column by column, m = h + 8 w. Either way an 8-row swizzle atom is 8 consecutive
  // pixels along the fast dimension.
  static constexpr bool kWFast = kKind == 3;
  static constexpr int kTH = kWFast ? 16 : kTileH, kTW = kWFast ? 8 : kTileW;
  // The norm kernel's tall box: the tile plus one halo pixel on each side in both dimensions;
  // kSlow = its pixels along the fast dimension (the stride, in 128-byte rows, from one line of
  // the box to the next, and the descriptors' 8-row group stride).
  static constexpr int kBoxRowsH = kTH + 2, kBoxColsW = kTW + 2;
  static constexpr int kSlow = kWFast ? kBoxColsW : kBoxRowsH;
  static constexpr int kThreads = kNorm ? 448 : 192;  // + 8 prologue warps
  // kNorm: one tall A box per (kernel frame, 64 channels), 10 x 18 pixels, serves all 9 taps of
  // that frame (the plain kernel loads one 8 x 18 box per kernel row, for its 3 taps), so every
  // pixel is normalised once per box instead of three times.
  // kPhase: one 9 x 18 box per 64 channels serves the 4 taps (u, v) of a phase, at row offsets
  // u + 9 v (the plain kernel loads one 8 x 18 box per tap row u, for its 2 taps).
  static constexpr int kABox = kNorm ? kBoxRowsH * kBoxColsW * 128 : kPhase ? kPhaseRows * kBoxW * 128 : kABytes;
  static constexpr int kAStride = (kABox + 1023) / 1024 * 1024;
  static constexpr int kAStages = kNorm ? 3 : 4;
  static constexpr int kBStages = kPhase ? 8 : 9;  // 4-tap boxes: two per ring
  static constexpr int kBOffset = kAStages * kAStride;
  // kNorm: each A stage's 64 channels of coefficients (16 bytes each) arrive with the box.
  static constexpr int kCoefOffset = kBOffset + kBStages * kBBytes;
  static constexpr int kBarOffset = kCoefOffset + (kNorm ? kAStages * kCoefBytes : 0);
  static constexpr int kSmemTotal = kBarOffset + 512 + 1024;
};
static_assert(Cfg<0>::kSmemTotal <= 232448 && Cfg<1>::kSmemTotal <= 232448 && Cfg<2>::kSmemTotal <= 232448 &&
                  Cfg<3>::kSmemTotal <= 232448,
              "shared memory per CTA");
static_assert(Cfg<1>::kABox == Cfg<3>::kABox && Cfg<3>::kBoxRowsH == 18 && Cfg<3>::kBoxColsW == 10,
              "both orientations of the norm kernel use 180-pixel tall boxes");

struct Conv2Args {
  int N, T, H, W, Cin, Cout;
  int tiles_h, tiles_w;
  int px_tiles, px_pairs;
  int n_blks, phases, items;
  // Scheduling units: item i < split0 is one unit, items from split0 on are two (their halves of
  // 128 output channels); units = split0 + 2 (items - split0).
  int units, split0;
  int kb_per_tap, mode, has_cache;
  const wan_bf16* bias;
  const wan_bf16* residual;
  wan_bf16* y;
  unsigned* err;
  // GroupNorm statistics of y (null: none): one record per (frame, group, pixel tile, epilogue
  // warp): st_rec = float-float (sum d, sum d^2) over the warp's valid pixels x the group's
  // cg = 2^st_lg channels, d = y - s as stored (bf16); st_meta = (s, count), s the group's first
  // channel at the warp's first valid pixel (all zero for a warp without valid pixels). st_hdr:
  // the buffer's header, which receives the records per (frame, group) (st_parts) so that their
  // reader needs no knowledge of this launch's tiles.
  float4* st_rec;
  float2* st_meta;
  int* st_hdr;
  int st_cg, st_lg, st_parts;
  // Operand prologue (the kNorm kernel): per (frame n*T + t, input channel) the GroupNorm + SiLU
  // coefficients (S_hi, S_lo, B_hi, B_lo), blocked layout (coef_blocked_index), applied to every
  // A box read from `a` (not the cache).
  const float4* coef;
  const wan_bf16* a;  // the conv input itself (the prologue's rare exact path reads it again)
  // Optional, with the prologue: the new history [N, 2, H, W, Cin] (never the cache being read).
  // The tiles of frames T - 2 and T - 1 store their own normalised pixels there (frame
  // t - T + 2 of cache_out) from the box of their current frame, so no pass over x rewrites them.
  wan_bf16* cache_out;
  // Mode 2 (time upsample): y has y_frames frames per n of Cout / 2 channels; conv output frame
  // t, channel half i goes to frame y_frame0 + 2 t + i.
  int y_frames, y_frame0;
};

struct PTile {
  int n, t0, h0, w0, ph, nb;
  bool valid;
};

// item -> N block (fastest), phase, pixel pair; `which` picks the pair's first or second tile.
// Pixel tiles are numbered frame-fastest, so concurrently running pairs share input frames in L2.
template <int kKind>
__device__ __forceinline__ PTile decode_pair(const Conv2Args& a, int item, int which) {
  PTile t;
  t.nb = item % a.n_blks;
  item /= a.n_blks;
  t.ph = item % a.phases;
  item /= a.phases;
  int px = 2 * item + which;
  t.valid = px < a.px_tiles;
  if (!t.valid) px = 2 * item;
  t.t0 = px % a.T;
  px /= a.T;
  t.w0 = (px % a.tiles_w) * Cfg<kKind>::kTW;
  px /= a.tiles_w;
  t.h0 = (px % a.tiles_h) * Cfg<kKind>::kTH;
  t.n = px / a.tiles_h;
  return t;
}

// Snake order of scheduling units over the CTA pairs; -1 once this pair has no unit in round r.
__device__ __forceinline__ int item_of(const Conv2Args& a, int r, int cluster, int nclusters) {
  const int base = r * nclusters;
  if (base >= a.units) return -1;
  const int unit = base + ((r & 1) ? nclusters - 1 - cluster : cluster);
  return unit < a.units ? unit : -2;  // -2: nothing in this (last) round
}

// Unit -> item, and which 128-channel half of the item's N block it computes (-1: all 256).
__device__ __forceinline__ int unit_item(const Conv2Args& a, int unit, int& sub) {
  if (unit < a.split0) {
    sub = -1;
    return unit;
  }
  sub = (unit - a.split0) & 1;
  return a.split0 + ((unit - a.split0) >> 1);
}

// Kernel row `row` of the tap grid: its frame and row offsets, and the input column of the A
// box's first column relative to the tile. Mode 0: 9 rows (dt, dh) of 3 horizontal taps; mode 1:
// for phase (pa, pb) the 2 rows u of 2 taps v, reading input (h + pa - 1 + u, w + pb - 1 + v);
// mode 2 (3x1x1 time conv): 3 rows dt of one tap; mode 3 (1x1x1): one row of one tap.
__device__ __forceinline__ void row_offsets(const Conv2Args& a, int row, int ph, int& dt, int& dh, int& dw0) {
  if (a.mode == 0) {
    dt = row / 3 - 2;
    dh = row % 3 - 1;
    dw0 = -1;
  } else if (a.mode >= 2) {  // the current pixel of frame t + dt: mode 2 dt = -2..0, mode 3 dt = 0
    dt = a.mode == 2 ? row - 2 : 0;
    dh = 0;
    dw0 = 0;
  } else {
    dt = 0;
    dh = (ph >> 1) - 1 + row;
    dw0 = (ph & 1) - 1;
  }
}

// A kernel row is skipped only when it reads nothing but zeros for BOTH tiles of the pair
// (frames before a chunk that has no history; a missing second tile counts as zeros).
__device__ __forceinline__ bool skip_pair(const Conv2Args& a, const PTile& p0, const PTile& p1, int dt) {
  if (a.has_cache) return false;
  const bool z0 = p0.t0 + dt < 0;
  const bool z1 = !p1.valid || (p1.t0 + dt < 0);
  return z0 && z1;
}

// Float-float sums of 8 values over the 32 lanes of a warp as a reduce-scatter: three halving
// exchanges (xor 4, 2, 1) leave lane l with value l & 7 summed over its 8-lane set, two butterfly
// steps (xor 8, 16) add the 4 sets. 18 shuffles for 8 totals.
__device__ __forceinline__ void st_reduce8(const float (&vh)[8], const float (&vl)[8], int lane, float& H, float& L) {
  const bool b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
  float hh[4], hl[4], eh[2], el[2];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    hh[j] = b2 ? vh[j + 4] : vh[j];
    hl[j] = b2 ? vl[j + 4] : vl[j];
    const float oh = __shfl_xor_sync(0xffffffffu, b2 ? vh[j] : vh[j + 4], 4);
    const float ol = __shfl_xor_sync(0xffffffffu, b2 ? vl[j] : vl[j + 4], 4);
    ff_add(hh[j], hl[j], oh, ol);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    eh[j] = b1 ? hh[j + 2] : hh[j];
    el[j] = b1 ? hl[j + 2] : hl[j];
    const float oh = __shfl_xor_sync(0xffffffffu, b1 ? hh[j] : hh[j + 2], 2);
    const float ol = __shfl_xor_sync(0xffffffffu, b1 ? hl[j] : hl[j + 2], 2);
    ff_add(eh[j], el[j], oh, ol);
  }
  H = b0 ? eh[1] : eh[0];
  L = b0 ? el[1] : el[0];
  {
    const float oh = __shfl_xor_sync(0xffffffffu, b0 ? eh[0] : eh[1], 1);
    const float ol = __shfl_xor_sync(0xffffffffu, b0 ? el[0] : el[1], 1);
    ff_add(H, L, oh, ol);
  }
#pragma unroll
  for (int off = 8; off < 32; off <<= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, H, off), ol = __shfl_xor_sync(0xffffffffu, L, off);
    ff_add(H, L, oh, ol);
  }
}

// The MMAs of one A box whose kTaps taps read the consecutive B stages starting at full_b[0] /
// empty_b[0] (no wrap of the ring inside the box): straight-line code whose descriptors differ by
// constants, with each tap's wait, fence and stage release in place. A probe of the tensor pipe
// (one issuing thread, M256 x N128 pair MMAs) measured that per-tap wait, fence and commit inside
// a run-time loop cost ~120 cycles of issue per MMA against ~86 in straight-line code.
// kGroup > 1 (the 128-channel halves of the last round, whose MMAs are short): the B stages of
// kGroup consecutive taps land on the first one's barrier and are released together, so one
// wait and one commit serve kGroup taps.
// kTallR > 0: a tall box of kTallR-row columns whose tap j = kTapW dh + dw starts at row dh + kTallR dw
// (8-row groups kTallR * 128 bytes apart); kTallR = 0: a plain box, tap j one column (1024 bytes) on.
// kRowMajor: the box is stored row by row with kTallR pixels per row, so tap j starts at row
// kTallR dh + dw (8-row groups one box row apart).
template <int kTaps, int kTallR, int kTapW, int kGroup, bool kRowMajor = false>
__device__ __forceinline__ bool mma_box(uint32_t d_tmem, uint32_t a_box, uint32_t b_stage, uint64_t* full_b,
                                        uint64_t* empty_b, uint32_t phb, uint32_t idesc, bool first, unsigned* err) {
  static_assert(kTaps % kGroup == 0, "whole groups of taps");
  const uint64_t a0 = kTallR ? smem_desc_sw128(a_box, kTallR * 128) : smem_desc_sw128(a_box);
  const uint64_t b0 = smem_desc_sw128(b_stage);
#pragma unroll
  for (int j = 0; j < kTaps; ++j) {
    if (j % kGroup == 0) {
      if (!mbar_wait_cluster(&full_b[j], phb, err, kDevErrTimeoutMma)) return false;
      tc_fence_after();
    }
    const uint64_t aj =
        a0 + (kTallR ? (uint64_t)((kRowMajor ? (j / kTapW) * kTallR + j % kTapW : (j % kTapW) * kTallR + j / kTapW) * 8)
                     : (uint64_t)j * kShiftDesc);
    const uint64_t bj = b0 + (uint64_t)j * (kBBytes >> 4);
#pragma unroll
    for (int k = 0; k < kBlockK / 16; ++k)
      mma_bf16_pair(d_tmem, aj + 2 * k, bj + 2 * k, idesc, (first && j == 0 && k == 0) ? 0u : 1u);
    if (j % kGroup == kGroup - 1) mma_commit_pair(&empty_b[j - (kGroup - 1)], 0x3);
  }
  return true;
}

// Two consecutive boxes of one tap each (modes 2 and 3: consecutive K blocks of one kernel row):
// A stages 0, 1 and B stages 0, 1 from the given ones, in straight-line code.
__device__ __forceinline__ bool mma_two_boxes(uint32_t d_tmem, uint32_t a_box, uint32_t a_stride, uint32_t b_stage,
                                              uint64_t* full_a, uint64_t* empty_a, uint64_t* full_b,
                                              uint64_t* empty_b, uint32_t pha, uint32_t phb, uint32_t idesc,
                                              bool first, unsigned* err) {
  const uint64_t a0 = smem_desc_sw128(a_box), b0 = smem_desc_sw128(b_stage);
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    if (!mbar_wait_cluster(&full_a[g], pha, err, kDevErrTimeoutMma)) return false;
    if (!mbar_wait_cluster(&full_b[g], phb, err, kDevErrTimeoutMma)) return false;
    tc_fence_after();
    const uint64_t ag = a0 + (uint64_t)g * (a_stride >> 4), bg = b0 + (uint64_t)g * (kBBytes >> 4);
#pragma unroll
    for (int k = 0; k < kBlockK / 16; ++k)
      mma_bf16_pair(d_tmem, ag + 2 * k, bg + 2 * k, idesc, (first && g == 0 && k == 0) ? 0u : 1u);
    mma_commit_pair(&empty_b[g], 0x3);
    mma_commit_pair(&empty_a[g], 0x3);
  }
  return true;
}

template <int kKind>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kKind>::kThreads, 1)
    conv_tc2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_cache,
                    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_w64,
                    const Conv2Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr bool kNorm = Cfg<kKind>::kNorm, kPhase = Cfg<kKind>::kPhase;
  constexpr int kAStages = Cfg<kKind>::kAStages, kBStages = Cfg<kKind>::kBStages;
  constexpr int kBOffset = Cfg<kKind>::kBOffset, kAStride = Cfg<kKind>::kAStride, kABox = Cfg<kKind>::kABox;
  uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + Cfg<kKind>::kBarOffset);
  uint64_t* empty_a = full_a + kAStages;
  uint64_t* full_b = empty_a + kAStages;
  uint64_t* empty_b = full_b + kBStages;
  uint64_t* tmem_full = empty_b + kBStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* mma_done = tmem_empty + 2;
  uint64_t* ready_a = mma_done + 1;  // kNorm: both CTAs' prologue warps are done with stage s (leader)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ready_a + kAStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  // A boxes per K slice of an item, and taps (B stages) per A box: kernel rows of 3 (mode 0) or 2
  // (mode 1) taps; with the prologue, kernel frames of 9 taps. The boxes go in the order (group of
  // rows_in rows, K slice, row in the group): mode 0 takes a kernel frame's 3 rows per K slice, so
  // the taps are added in the order (dt, K slice, dh, dw), the prologue kernel's order too, and
  // the two kernels give the same bits.
  const int rows = kNorm ? 3 : kPhase ? 1 : (args.mode == 0 ? 9 : args.mode == 1 ? 2 : args.mode == 2 ? 3 : 1);
  const int taps_per_row = kNorm ? 9 : kPhase ? 4 : (args.mode == 0 ? 3 : args.mode == 1 ? 2 : 1);
  const int rows_in = (!kNorm && args.mode == 0) ? 3 : 1;
  // B stages in use: 8 for boxes of 2 taps (mode 1) and of 1 tap (modes 2, 3), so that no box,
  // and no pair of 1-tap boxes, wraps the ring.
  const int b_ring = taps_per_row <= 2 ? kBStages - 1 : kBStages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&full_a[s], 1);
      // with the prologue, an A stage is free once the pair's MMAs (one commit) and this CTA's 8
      // prologue warps (which may still copy the box's pixels to the new history) are done with it
      mbar_init(&empty_a[s], kNorm ? 9 : 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_b[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(mma_done, 1);
    if (blockIdx.x == 0 && args.st_hdr) *args.st_hdr = args.st_parts;  // the statistics' record count
    if (kNorm)
      for (int s = 0; s < kAStages; ++s) mbar_init(&ready_a[s], 16);  // 8 prologue warps per CTA
    fence_mbarrier_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_cache);
    prefetch_tensormap(&tm_w);
    if (args.split0 < args.items) prefetch_tensormap(&tm_w64);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);  // one warp in each CTA of the pair, collectively
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anyone arrives on them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    const uint64_t w_policy = l2_policy_evict_last();
    int sa = 0, sb = 0;
    uint32_t pha = 0, phb = 0;
    uint32_t armed_a = 0, parity_a = 0, armed_b = 0, parity_b = 0;  // stages the even CTA armed
    uint32_t fresh_b = 0xffffffffu;  // B group heads not yet used by a half (see below)
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int unit = item_of(args, r, cluster, nclusters);
      if (unit == -1) break;
      if (unit < 0) continue;
      int sub;
      const int item = unit_item(args, unit, sub);
      const PTile me = decode_pair<kKind>(args, item, (int)rank);
      const PTile p0 = decode_pair<kKind>(args, item, 0), p1 = decode_pair<kKind>(args, item, 1);
      // This CTA's weight rows: half of the N block, or half of the unit's 128-channel half.
      const int brow = me.nb * kN + (sub < 0 ? (int)rank * 128 : sub * 128 + (int)rank * 64);
      const CUtensorMap* wmap = sub < 0 ? &tm_w : &tm_w64;
      const uint32_t b_tx = sub < 0 ? 2 * kBBytes : kBBytes;
      for (int rg = 0; ok && rg < rows; rg += rows_in) {
        for (int kb = 0; ok && kb < args.kb_per_tap; ++kb) {
          for (int row = rg; ok && row < rg + rows_in; ++row) {
            int dt, dh, dw0;
            if (kNorm) {  // kernel frame row: the tall box starts one row above and left of the tile
              dt = row - 2;
              dh = -1;
              dw0 = -1;
            } else {
              row_offsets(args, row, me.ph, dt, dh, dw0);
            }
            if (skip_pair(args, p0, p1, dt)) continue;
            const int hh = me.h0 + dh, ww = me.w0 + dw0;
            int tau = me.t0 + dt;
            if (!me.valid) tau = args.T + 8;  // out of range: the TMA unit fills zeros
            if (!mbar_wait_cluster(&empty_a[sa], pha ^ 1, args.err, kDevErrTimeoutProducer)) {
              ok = false;
              break;
            }
            uint8_t* a_dst = smem + sa * kAStride;
            if (kNorm) {
              // Each CTA's box lands on its own barrier, with the 64 channels' coefficients of its
              // frame (any in-range frame for boxes the prologue leaves alone): its prologue warps
              // wait for both.
              mbar_arrive_expect_tx(&full_a[sa], kABox + kCoefBytes);
              const int fc = min(max(tau, 0), args.T - 1);
              bulk_load(smem + Cfg<kKind>::kCoefOffset + sa * kCoefBytes,
                        args.coef + ((size_t)me.n * args.T + fc) * args.Cin + kb * kBlockK, kCoefBytes, &full_a[sa]);
              armed_a |= 1u << sa;
              parity_a = (parity_a & ~(1u << sa)) | (pha << sa);
              // the tensor map lists the box's fast dimension first: (c, h, w) or, kWFast, (c, w, h)
              const int d1 = Cfg<kKind>::kWFast ? ww : hh, d2 = Cfg<kKind>::kWFast ? hh : ww;
              if (tau < 0 && args.has_cache)
                tma_load_5d(a_dst, &tm_cache, &full_a[sa], kb * kBlockK, d1, d2, tau + 2, me.n);
              else
                tma_load_5d(a_dst, &tm_a, &full_a[sa], kb * kBlockK, d1, d2, tau, me.n);
            } else {
              if (leader) {
                mbar_arrive_expect_tx(&full_a[sa], 2 * kABox);  // both CTAs' bytes land on it
                armed_a |= 1u << sa;
                parity_a = (parity_a & ~(1u << sa)) | (pha << sa);
              }
              const uint32_t bar_a = mapa_shared(smem_u32(&full_a[sa]), 0);
              if (tau < 0 && args.has_cache)
                tma_load_5d_pair(a_dst, &tm_cache, bar_a, kb * kBlockK, hh, ww, tau + 2, me.n);
              else
                tma_load_5d_pair(a_dst, &tm_a, bar_a, kb * kBlockK, hh, ww, tau, me.n);
            }
            if (++sa == kAStages) {
              sa = 0;
              pha ^= 1;
            }
            // A half's B stages go in groups of bg (the MMA issuer's mma_box): the group's bytes land
            // on its first stage's barrier, whose release covers the group. The first time a group's
            // stages are used this way, the full-item MMAs before may still read any of them: all
            // their releases are waited for then.
            const int bg = sub < 0 ? 1 : (taps_per_row % 3 == 0 ? 3 : taps_per_row == 4 ? 4 : taps_per_row == 2 ? 2 : 1);
            int head = sb;
            for (int j = 0; j < taps_per_row; ++j) {
              if (j % bg == 0) {
                head = sb;
                const int ng = (bg > 1 && ((fresh_b >> sb) & 1u)) ? bg : 1;
                for (int g = 0; g < ng; ++g) {
                  if (!mbar_wait_cluster(&empty_b[sb + g], phb ^ 1, args.err, kDevErrTimeoutProducer)) {
                    ok = false;
                    break;
                  }
                }
                if (!ok) break;
                if (bg > 1) fresh_b &= ~(1u << sb);
                if (leader) {
                  mbar_arrive_expect_tx(&full_b[sb], (uint32_t)bg * b_tx);
                  armed_b |= 1u << sb;
                  parity_b = (parity_b & ~(1u << sb)) | (phb << sb);
                }
              }
              const int tap = row * taps_per_row + j;
              tma_load_3d_pair(smem + kBOffset + sb * kBBytes, wmap, mapa_shared(smem_u32(&full_b[head]), 0),
                               tap * args.Cin + kb * kBlockK, brow, me.ph, w_policy);
              if (++sb == b_ring) {
                sb = 0;
                phb ^= 1;
              }
            }
          }
        }
      }
    }
    // Drain: every load counted on this CTA's full barriers has landed (the even CTA's B barriers
    // count both CTAs' weights; with the prologue each CTA's A barriers count its own boxes).
    for (int s = 0; s < kAStages; ++s)
      if (armed_a & (1u << s)) mbar_wait(&full_a[s], (parity_a >> s) & 1, args.err, kDevErrTimeoutDrain);
    for (int s = 0; s < kBStages; ++s)
      if (armed_b & (1u << s)) mbar_wait(&full_b[s], (parity_b >> s) & 1, args.err, kDevErrTimeoutDrain);
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc_full = idesc_bf16_f32(256, kN), idesc_half = idesc_bf16_f32(256, kN / 2);
    const uint32_t a_base = smem_u32(smem), b_base = smem_u32(smem + kBOffset);
    int sa = 0, sb = 0;
    uint32_t pha = 0, phb = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int unit = item_of(args, r, cluster, nclusters);
      if (unit == -1) break;
      if (unit < 0) continue;
      int sub;
      const int item = unit_item(args, unit, sub);
      const uint32_t idesc = sub < 0 ? idesc_full : idesc_half;  // a half: the first 128 columns
      const PTile p0 = decode_pair<kKind>(args, item, 0), p1 = decode_pair<kKind>(args, item, 1);
      if (!mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1, args.err, kDevErrTimeoutMma)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kN;
      bool first = true;
      for (int rg = 0; ok && rg < rows; rg += rows_in) {
        for (int kb = 0; ok && kb < args.kb_per_tap; ++kb) {
          for (int row = rg; ok && row < rg + rows_in; ++row) {
            if (!args.has_cache) {  // without history some rows read only zeros for both tiles
              int dt, dh, dw0;
              if (kNorm)
                dt = row - 2;
              else
                row_offsets(args, row, p0.ph, dt, dh, dw0);
              if (skip_pair(args, p0, p1, dt)) continue;
            }
            if (!kNorm && taps_per_row == 1 && rows_in == 1 && (kb & 1) == 0 && kb + 1 < args.kb_per_tap &&
                (sa & 1) == 0 && (sb & 1) == 0) {
              // K blocks kb and kb + 1 of this kernel row in one burst (the loop's kb++ skips kb + 1).
              ok = mma_two_boxes(d_tmem, a_base + sa * kAStride, kAStride, b_base + sb * kBBytes, full_a + sa,
                                 empty_a + sa, full_b + sb, empty_b + sb, pha, phb, idesc, first, args.err);
              first = false;
              if ((sa += 2) == kAStages) {
                sa = 0;
                pha ^= 1;
              }
              if ((sb += 2) == b_ring) {
                sb = 0;
                phb ^= 1;
              }
              ++kb;
              continue;
            }
            if (!mbar_wait_cluster(kNorm ? &ready_a[sa] : &full_a[sa], pha, args.err, kDevErrTimeoutMma)) {
              ok = false;
              break;
            }
            const uint32_t a_box = a_base + sa * kAStride;
            // Boxes of 9 taps (tall), 3 taps (mode 0) or 2 taps (mode 1, an 8-stage ring) never wrap
            // the B ring: one straight-line burst each. Boxes of 1 tap (modes 2, 3) take the loop.
            static_assert(kBStages == (kPhase ? 8 : 9), "whole boxes of 3, 4 and 9 taps");
            // Halves (sub >= 0) take their B stages in groups (mma_box); the producer arms them so.
            if (kNorm && sb == 0) {
              constexpr int kS = Cfg<kKind>::kSlow;
              constexpr bool kR = Cfg<kKind>::kWFast;
              ok = sub >= 0 ? mma_box<9, kS, 3, 3, kR>(d_tmem, a_box, b_base, full_b, empty_b, phb, idesc, first, args.err)
                            : mma_box<9, kS, 3, 1, kR>(d_tmem, a_box, b_base, full_b, empty_b, phb, idesc, first, args.err);
              sb = kBStages;
            } else if (kPhase && sb % 4 == 0) {
              const uint32_t bs = b_base + sb * kBBytes;
              ok = sub >= 0 ? mma_box<4, kPhaseRows, 2, 4>(d_tmem, a_box, bs, full_b + sb, empty_b + sb, phb, idesc, first, args.err)
                            : mma_box<4, kPhaseRows, 2, 1>(d_tmem, a_box, bs, full_b + sb, empty_b + sb, phb, idesc, first, args.err);
              sb += 4;
            } else if (!kNorm && !kPhase && taps_per_row == 3 && sb % 3 == 0) {
              const uint32_t bs = b_base + sb * kBBytes;
              ok = sub >= 0 ? mma_box<3, 0, 3, 3>(d_tmem, a_box, bs, full_b + sb, empty_b + sb, phb, idesc, first, args.err)
                            : mma_box<3, 0, 3, 1>(d_tmem, a_box, bs, full_b + sb, empty_b + sb, phb, idesc, first, args.err);
              sb += 3;
            } else if (!kNorm && !kPhase && taps_per_row == 2 && sb % 2 == 0) {
              const uint32_t bs = b_base + sb * kBBytes;
              ok = sub >= 0 ? mma_box<2, 0, 2, 2>(d_tmem, a_box, bs, full_b + sb, empty_b + sb, phb, idesc, first, args.err)
                            : mma_box<2, 0, 2, 1>(d_tmem, a_box, bs, full_b + sb, empty_b + sb, phb, idesc, first, args.err);
              sb += 2;
            } else {
              const uint64_t a_desc = smem_desc_sw128(a_box);
              for (int j = 0; j < taps_per_row; ++j) {
                if (!mbar_wait_cluster(&full_b[sb], phb, args.err, kDevErrTimeoutMma)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint64_t aj = kNorm    ? smem_desc_sw128(a_box + (Cfg<kKind>::kWFast ? (j / 3) * Cfg<kKind>::kSlow + j % 3
                                                                                    : (j % 3) * Cfg<kKind>::kSlow + j / 3) * 128,
                                                               Cfg<kKind>::kSlow * 128)
                                    : kPhase ? smem_desc_sw128(a_box + ((j % 2) * kPhaseRows + j / 2) * 128, kPhaseRows * 128)
                                             : a_desc + j * kShiftDesc;
                const uint64_t b_desc = smem_desc_sw128(b_base + sb * kBBytes);
  #pragma unroll
                for (int k = 0; k < kBlockK / 16; ++k)
                  mma_bf16_pair(d_tmem, aj + 2 * k, b_desc + 2 * k, idesc, (first && j == 0 && k == 0) ? 0u : 1u);
                mma_commit_pair(&empty_b[sb], 0x3);
                if (++sb == b_ring) {
                  sb = 0;
                  phb ^= 1;
                }
              }
            }
            if (sb == b_ring) {
              sb = 0;
              phb ^= 1;
            }
            first = false;
            if (!ok) break;
            mma_commit_pair(&empty_a[sa], 0x3);
            if (++sa == kAStages) {
              sa = 0;
              pha ^= 1;
            }
          }
        }
      }
      if (!ok) break;
      mma_commit_pair(&tmem_full[acc], 0x3);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    mma_commit_pair(mma_done, 0x1);
    mbar_wait(mma_done, 0, args.err, kDevErrTimeoutDrain);
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue (both CTAs, own 128 rows)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int Ho = args.mode == 1 ? 2 * args.H : args.H;
    const int Wo = args.mode == 1 ? 2 * args.W : args.W;
    const int Cy = args.mode == 2 ? args.Cout / 2 : args.Cout;  // channels of a y pixel
    const bool vec8 = (args.Cout % 8) == 0;
    const uint32_t leader_empty0 = mapa_shared(smem_u32(&tmem_empty[0]), 0);
    const uint32_t leader_empty1 = mapa_shared(smem_u32(&tmem_empty[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int r = 0;; ++r) {
      const int unit = item_of(args, r, cluster, nclusters);
      if (unit == -1) break;
      if (unit < 0) continue;
      int sub;
      const int item = unit_item(args, unit, sub);
      const PTile t = decode_pair<kKind>(args, item, (int)rank);
      const int ncols = sub < 0 ? kN : kN / 2;                  // accumulator columns of the unit
      const int cbase = t.nb * kN + (sub > 0 ? kN / 2 : 0);     // its first output channel
      if (!mbar_wait_cluster(&tmem_full[acc], acc_phase, args.err, kDevErrTimeoutEpilogue)) break;
      tc_fence_after();
      // TMEM row = h + 8 w, or w + 8 h for the 16 x 8 tiles
      const int hh = t.h0 + (Cfg<kKind>::kWFast ? row / 8 : row & 7), ww = t.w0 + (Cfg<kKind>::kWFast ? row & 7 : row / 8);
      const int tt = t.t0;
      const bool valid = t.valid && hh < args.H && ww < args.W;
      size_t pix;
      wan_bf16* yrow;
      if (args.mode == 1) {
        pix = (((size_t)t.n * args.T + tt) * Ho + (2 * hh + (t.ph >> 1))) * Wo + (2 * ww + (t.ph & 1));
        yrow = args.y + pix * args.Cout;
      } else if (args.mode == 2) {  // channel half i of this N block -> frame y_frame0 + 2 t + i
        const int half = t.nb * kN / Cy;
        pix = (((size_t)t.n * args.y_frames + args.y_frame0 + 2 * tt + half) * Ho + hh) * Wo + ww;
        yrow = args.y + pix * Cy - (size_t)half * Cy;  // + col lands on channel col - half * Cy
      } else {
        pix = (((size_t)t.n * args.T + tt) * Ho + hh) * Wo + ww;
        yrow = args.y + pix * args.Cout;
      }
      const wan_bf16* rrow = args.residual ? args.residual + pix * args.Cout : nullptr;
      const uint32_t taddr = tmem_base + (uint32_t)(acc * kN) + ((uint32_t)(quarter * 32) << 16);
      // GroupNorm statistics of this tile's output (optional): per group, each lane adds d and d^2
      // over the group's channels as float-float pairs (TwoSum, Fast2Sum; even and odd channels
      // in the two halves of packed fp32x2), the warp totals 4 groups at once (float-float
      // reduce-scatter) and writes one record per group.
      const bool stats = args.st_rec != nullptr && t.valid;
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
      const int src = vmask ? __ffs(vmask) - 1 : 0;
      const int cg = args.st_cg, lg = args.st_lg;
      const size_t rec_stride = (size_t)args.tiles_h * args.tiles_w * 4;  // between groups
      const size_t rec0 = ((((size_t)t.n * args.T + tt) * (args.Cout >> lg) + (size_t)(cbase >> lg)) *
                               (size_t)args.tiles_h * args.tiles_w +
                           (size_t)(t.h0 / Cfg<kKind>::kTH) * args.tiles_w + t.w0 / Cfg<kKind>::kTW) * 4 + quarter;
      float wh[8], wl[8], shw[4];  // the window's 4 groups: (sum d, sum d^2) as float-float, shifts
#pragma unroll
      for (int k = 0; k < 8; ++k) wh[k] = wl[k] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) shw[k] = 0.f;
      float sh = 0.f;
      float2 h1 = make_float2(0.f, 0.f), l1 = h1, h2 = h1, l2 = h1;
      // The TMEM load of the next 16 columns is in flight while this chunk is processed.
      uint32_t rn[16];
      __syncwarp();
      tmem_ld16_issue(taddr, rn);
      tmem_ld16_wait(rn);
#pragma unroll 1
      for (int c0 = 0; c0 < ncols; c0 += 16) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(rn[i]);
        if (c0 + 16 < ncols) {
          __syncwarp();
          tmem_ld16_issue(taddr + c0 + 16, rn);
        }
        uint32_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // the chunk as stored (valid lanes)
        const int col = cbase + c0;
        if (valid && col < args.Cout) {
          if (args.bias) {
            if (vec8 && col + 16 <= args.Cout) {  // 16 bias values in two 16-byte loads
              const uint4 b0 = __ldg(reinterpret_cast<const uint4*>(args.bias + col));
              const uint4 b1 = __ldg(reinterpret_cast<const uint4*>(args.bias + col + 8));
              const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[2 * i] += bf16lo_to_f32(bw[i]);
                v[2 * i + 1] += bf16hi_to_f32(bw[i]);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (col + i < args.Cout) v[i] += __uint_as_float(((uint32_t)args.bias[col + i]) << 16);
            }
          }
          if (vec8 && col + 16 <= args.Cout) {
            if (rrow) {
              const uint4 r0 = *reinterpret_cast<const uint4*>(rrow + col);
              const uint4 r1 = *reinterpret_cast<const uint4*>(rrow + col + 8);
              const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[2 * i] += bf16lo_to_f32(rw[i]);
                v[2 * i + 1] += bf16hi_to_f32(rw[i]);
              }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            *reinterpret_cast<uint4*>(yrow + col) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(yrow + col + 8) = make_uint4(o[4], o[5], o[6], o[7]);
          } else {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              if (col + i < args.Cout) {
                float a0 = v[i], a1 = v[i + 1];
                if (rrow) {
                  const uint32_t rw = *reinterpret_cast<const uint32_t*>(rrow + col + i);
                  a0 += bf16lo_to_f32(rw);
                  a1 += bf16hi_to_f32(rw);
                }
                *reinterpret_cast<uint32_t*>(yrow + col + i) = pack_bf16x2(a0, a1);
              }
            }
          }
        }
        if (stats) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int ch = c0 + 4 * j;  // channel within the N block (the same for the whole warp)
            if ((ch & (cg - 1)) == 0) sh = __shfl_sync(0xffffffffu, bf16lo_to_f32(o[2 * j]), src);
            const float2 nsh = make_float2(-sh, -sh);
            const float2 d01 = __fadd2_rn(make_float2(bf16lo_to_f32(o[2 * j]), bf16hi_to_f32(o[2 * j])), nsh);
            const float2 d23 = __fadd2_rn(make_float2(bf16lo_to_f32(o[2 * j + 1]), bf16hi_to_f32(o[2 * j + 1])), nsh);
            if (valid) {
              two_sum2(h1, l1, d01);
              two_sum2(h1, l1, d23);
              fast_two_sum2(h2, l2, __fmul2_rn(d01, d01));
              fast_two_sum2(h2, l2, __fmul2_rn(d23, d23));
            }
            if (((ch + 4) & (cg - 1)) == 0) {  // the group ends: even + odd halves into its slot
              float a1h = h1.x, a1l = l1.x, a2h = h2.x, a2l = l2.x;
              ff_add(a1h, a1l, h1.y, l1.y);
              ff_add(a2h, a2l, h2.y, l2.y);
              const int slot = (ch >> lg) & 3;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if (slot == k) {
                  wh[2 * k] = a1h;
                  wl[2 * k] = a1l;
                  wh[2 * k + 1] = a2h;
                  wl[2 * k + 1] = a2l;
                  shw[k] = sh;
                }
              }
              h1 = l1 = h2 = l2 = make_float2(0.f, 0.f);
            }
          }
          if (((c0 + 16) & (4 * cg - 1)) == 0) {  // 4 groups complete: lane 2k (k < 4) writes group k
            float H, L;
            st_reduce8(wh, wl, lane, H, L);
            const float H2 = __shfl_down_sync(0xffffffffu, H, 1), L2 = __shfl_down_sync(0xffffffffu, L, 1);
            const int k = lane >> 1;
            const float sk = k == 0 ? shw[0] : k == 1 ? shw[1] : k == 2 ? shw[2] : shw[3];
            if (lane < 8 && !(lane & 1)) {
              const size_t idx = rec0 + (size_t)(((c0 + 16) >> lg) - 4 + k) * rec_stride;
              __stcg(args.st_rec + idx, make_float4(H, L, H2, L2));
              __stcg(args.st_meta + idx, make_float2(sk, (float)(__popc(vmask) << lg)));
            }
          }
        }
        if (c0 + 16 < ncols) tmem_ld16_wait(rn);
      }
      // This warp is done with the accumulator: one arrival per warp on the even CTA's barrier.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(acc == 0 ? leader_empty0 : leader_empty1);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  } else if (kNorm && warp >= 6) {
    // ------------------------------------------------------------ operand prologue (both CTAs)
    // Each tall A box of x is replaced in place by silu(x S + B) with its frame's coefficients,
    // the arithmetic of the norm's own apply pass (so the MMAs see exactly the bf16 values it
    // would have written). Boxes of the cache (already normalised) and rows of zero padding are
    // left as loaded. Thread t of the 256 owns the 16-byte chunk jl = t % 8 (channels 8 jl ..
    // 8 jl + 7 of the box's 64) of rows r0 + 32 i, r0 = t / 8, of the box's 180 rows
    // (row = h + 10 c for the 8 x 16 tiles' 10 x 18 boxes, c the column; row = c + 10 h for the
    // 16 x 8 tiles' 18 x 10 boxes); the swizzle puts the chunk at jl ^ (row % 8) = jl ^ (r0 % 8).
    constexpr int kRows = Cfg<kKind>::kBoxRowsH * Cfg<kKind>::kBoxColsW;
    constexpr int kSl = Cfg<kKind>::kSlow;
    constexpr bool kWF = Cfg<kKind>::kWFast;
    const int pt = (int)threadIdx.x - 192;
    const int jl = pt & 7, r0 = pt >> 3;
    const uint32_t chunk_off = (uint32_t)r0 * 128 + ((uint32_t)(jl ^ (r0 & 7)) << 4);
    const uint32_t ready0 = mapa_shared(smem_u32(&ready_a[0]), 0);
    const float4* coef_sm = reinterpret_cast<const float4*>(smem + Cfg<kKind>::kCoefOffset) + jl;  // blocked
    int sa = 0;
    uint32_t pha = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int unit = item_of(args, r, cluster, nclusters);
      if (unit == -1) break;
      if (unit < 0) continue;
      int sub;
      const int item = unit_item(args, unit, sub);
      const PTile me = decode_pair<kKind>(args, item, (int)rank);
      const PTile p0 = decode_pair<kKind>(args, item, 0), p1 = decode_pair<kKind>(args, item, 1);
      for (int row = 0; ok && row < rows; ++row) {
        const int dt = row - 2;
        if (skip_pair(args, p0, p1, dt)) continue;
        const int tau = me.t0 + dt;
        const bool xf = me.valid && tau >= 0;  // this box holds x
        // this box's tile pixels are the new history (once per pixel: the current frame's box of
        // the first N block, not the second half of a split item)
        const bool wcache = args.cache_out && xf && dt == 0 && tau >= args.T - 2 && me.nb == 0 && sub <= 0;
        for (int kb = 0; kb < args.kb_per_tap; ++kb) {
          if (!mbar_wait(&full_a[sa], pha, args.err, kDevErrTimeoutPrologue)) {
            ok = false;
            break;
          }
          if (xf) {
            const GnCoef8 k8 = gn_coef8_blocked(coef_sm + sa * (kCoefBytes / 16));
            uint8_t* box = smem + sa * kAStride + chunk_off;
            // Branch-free fast formula for all chunks (their exp/reciprocal chains interleave),
            // then the rare chunk with a z < -80 again through gn_silu8: per chunk the same
            // choice as the norm's own pass.
            unsigned slow = 0;
#pragma unroll
            for (int i = 0; i < 6; ++i) {
              const int rr = r0 + 32 * i;
              const int hh = me.h0 - 1 + (kWF ? rr / kSl : rr % kSl), ww = me.w0 - 1 + (kWF ? rr % kSl : rr / kSl);
              if (rr < kRows && hh >= 0 && hh < args.H && ww >= 0 && ww < args.W) {
                bool sl;
                uint4* q = reinterpret_cast<uint4*>(box + i * 4096);
                *q = gn_silu8_fast(*q, k8, &sl);
                slow |= (unsigned)sl << i;
              }
            }
            if (slow) {  // x of those chunks again from global memory (the box now holds results)
              const wan_bf16* src = args.a + (size_t)kb * kBlockK + 8 * jl;
#pragma unroll 1
              for (int i = 0; i < 6; ++i) {
                if ((slow >> i) & 1) {
                  const int rr = r0 + 32 * i;
                  const int hh = me.h0 - 1 + (kWF ? rr / kSl : rr % kSl), ww = me.w0 - 1 + (kWF ? rr % kSl : rr / kSl);
                  const size_t px = (((size_t)me.n * args.T + tau) * args.H + hh) * args.W + ww;
                  const uint4 xv = *reinterpret_cast<const uint4*>(src + px * args.Cin);
                  *reinterpret_cast<uint4*>(box + i * 4096) = gn_silu8(xv, k8);
                }
              }
            }
            fence_proxy_async_smem();  // the MMAs read the box through the async proxy
          }
          __syncwarp();
          // Hand the box to the MMA issuer in the even CTA: what it hands over is this CTA's own
          // shared memory, complete with a release at CTA scope.
          if (lane == 0) {
            if (leader)
              mbar_arrive(&ready_a[sa]);
            else
              mbar_arrive_remote_cta(ready0 + 8u * (uint32_t)sa);
          }
          if (wcache) {  // while the MMAs run: the tile's own pixels of the box to the new history
            const uint8_t* box = smem + sa * kAStride + chunk_off;
            wan_bf16* dst = args.cache_out + ((size_t)me.n * 2 + (tau - args.T + 2)) * args.H * args.W * args.Cin +
                            (size_t)kb * kBlockK + 8 * jl;
#pragma unroll
            for (int i = 0; i < 6; ++i) {
              const int rr = r0 + 32 * i, rh = kWF ? rr / kSl : rr % kSl, rc = kWF ? rr % kSl : rr / kSl;
              const int hh = me.h0 - 1 + rh, ww = me.w0 - 1 + rc;
              if (rr < kRows && rh >= 1 && rh <= Cfg<kKind>::kTH && rc >= 1 && rc <= Cfg<kKind>::kTW && hh < args.H &&
                  ww < args.W)
                __stcs(reinterpret_cast<int4*>(dst + ((size_t)hh * args.W + ww) * args.Cin),
                       *reinterpret_cast<const int4*>(box + i * 4096));  // streamed: L2 keeps the conv's operands
            }
            __syncwarp();
          }
          if (lane == 0) mbar_arrive(&empty_a[sa]);  // this warp is done reading the stage
          if (++sa == kAStages) {
            sa = 0;
            pha ^= 1;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or arrivals may still touch it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// Activations [N, T, H, W, C] addressed as (c, h, w, t, n): H is listed before W, so a box of
// 8 rows x 18 columns lands in shared memory column by column (row m = h + 8 w).
// T frames per n are mapped; consecutive n are n_frames frames apart (n_frames >= T).
bool map_act_hw(CUtensorMap* m, const void* base, int C, int W, int H, int T, int N, int box_h = kTileH,
                int n_frames = 0) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  if (n_frames < T) n_frames = T;
  const cuuint64_t dims[5] = {(cuuint64_t)C, (cuuint64_t)H, (cuuint64_t)W, (cuuint64_t)T, (cuuint64_t)N};
  const cuuint64_t e = 2;
  const cuuint64_t strides[4] = {(cuuint64_t)W * C * e, C * e, (cuuint64_t)H * W * C * e,
                                 (cuuint64_t)n_frames * H * W * C * e};
  const cuuint32_t box[5] = {(cuuint32_t)kBlockK, (cuuint32_t)box_h, (cuuint32_t)kBoxW, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same activations addressed as (c, w, h, t, n) for the 16 x 8 tiles: a box of 18 rows x 10
// columns lands in shared memory row by row (row m = w + 10 h).
bool map_act_wh(CUtensorMap* m, const void* base, int C, int W, int H, int T, int N, int n_frames = 0) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  if (n_frames < T) n_frames = T;
  const cuuint64_t dims[5] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)N};
  const cuuint64_t e = 2;
  const cuuint64_t strides[4] = {C * e, (cuuint64_t)W * C * e, (cuuint64_t)H * W * C * e,
                                 (cuuint64_t)n_frames * H * W * C * e};
  const cuuint32_t box[5] = {(cuuint32_t)kBlockK, (cuuint32_t)Cfg<3>::kBoxColsW, (cuuint32_t)Cfg<3>::kBoxRowsH, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weights [P][Cout][K] addressed as (k, cout, p); a box is 64 K x `rows` output channels.
bool map_w_half(CUtensorMap* m, const void* base, int K, int Cout, int P, int rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)Cout, (cuuint64_t)P};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * Cout * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Persistent grid: as many CTA pairs as the GPU can hold at once (not every SM can be paired:
// a pair lives in one GPC), so no pair waits for a second wave.
template <int kKind>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tc, const CUtensorMap& tw, const CUtensorMap& tw64,
                        Conv2Args args, int sms, cudaStream_t stream) {
  constexpr int kSmem = Cfg<kKind>::kSmemTotal, kThr = Cfg<kKind>::kThreads;
  cudaError_t e = cudaFuncSetAttribute(conv_tc2_kernel<kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  int clusters = resident_pairs(reinterpret_cast<const void*>(conv_tc2_kernel<kKind>), kThr, kSmem, sms);
  // A last round of at most half the pairs' worth of items runs as twice as many 128-channel
  // halves (with the epilogue statistics only while a half holds whole windows of 4 groups).
  const int rem = args.items % clusters;
  args.split0 = args.items;
  args.units = args.items;
  if (rem > 0 && 2 * rem <= clusters && (args.st_rec == nullptr || 4 * args.st_cg <= kN / 2)) {
    args.split0 = args.items - rem;
    args.units = args.items + rem;
  }
  if (clusters > args.units) clusters = args.units;
  conv_tc2_kernel<kKind><<<2 * clusters, kThr, kSmem, stream>>>(ta, tc, tw, tw64, args);
  return cudaGetLastError();
}

}  // namespace

bool conv_pair_supported(int Cout) { return Cout >= 256; }

bool conv_gn_stats_supported(int Cout, int groups) {
  if (groups <= 0 || Cout % 256 != 0 || Cout % groups != 0) return false;
  const int cg = Cout / groups;  // a power of two from 4 to 64: 4 groups tile a 256-channel block
  return cg >= 4 && cg <= 64 && (cg & (cg - 1)) == 0;
}

void conv_gn_stats_records(int H, int W, int* q_a, int* q_b) {
  *q_a = cdiv(H, kTileH) * cdiv(W, kTileW) * 4;      // 8 x 16 tiles, 4 epilogue warps each
  *q_b = cdiv(H, Cfg<3>::kTH) * cdiv(W, Cfg<3>::kTW) * 4;  // 16 x 8 tiles
}

size_t conv_gn_stats_bytes(int N, int T, int H, int W, int Cout, int groups) {
  (void)Cout;
  int q_a, q_b;
  conv_gn_stats_records(H, W, &q_a, &q_b);
  return kGnStatsHeader + (size_t)N * T * groups * std::max(q_a, q_b) * (sizeof(float4) + sizeof(float2));
}

cudaError_t conv_pair_launch(int mode, const wan_bf16* a, const wan_bf16* cache_in, const wan_bf16* w,
                             const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                             int Cin, int Cout, int sms, unsigned* err, cudaStream_t stream, void* st_buf,
                             int st_groups, const float4* coef, int a_frames, int y_frames, int y_frame0,
                             wan_bf16* cache_out) {
  if (mode < 0 || mode > 3) return cudaErrorInvalidValue;
  if (mode == 2 && (Cout % (2 * kN) != 0 || residual != nullptr)) return cudaErrorInvalidValue;
  if (mode == 3 && cache_in) return cudaErrorInvalidValue;
  Conv2Args args{};
  args.N = N;
  args.T = T;
  args.H = H;
  args.W = W;
  args.Cin = Cin;
  args.Cout = Cout;
  // The norm kernel takes 16 x 8 tiles where they cover the frame with fewer tiles than 8 x 16 ones
  // (176 x 312: 429 tiles against 440, whose last column is half padding). Every output element
  // gets the same K steps in the same order either way.
  const bool wfast = coef != nullptr && mode == 0 &&
                     (long long)cdiv(H, Cfg<3>::kTH) * cdiv(W, Cfg<3>::kTW) < (long long)cdiv(H, kTileH) * cdiv(W, kTileW);
  args.tiles_h = cdiv(H, wfast ? Cfg<3>::kTH : kTileH);
  args.tiles_w = cdiv(W, wfast ? Cfg<3>::kTW : kTileW);
  args.px_tiles = N * T * args.tiles_h * args.tiles_w;
  args.px_pairs = cdiv(args.px_tiles, 2);
  args.n_blks = cdiv(Cout, kN);
  args.phases = mode == 1 ? 4 : 1;
  args.items = args.px_pairs * args.phases * args.n_blks;
  args.kb_per_tap = Cin / kBlockK;
  args.mode = mode;
  args.has_cache = cache_in != nullptr;
  args.bias = bias;
  args.residual = residual;
  args.y = y;
  args.err = err;
  args.y_frames = y_frames;
  args.y_frame0 = y_frame0;
  if (st_buf) {
    if (mode != 0 || !conv_gn_stats_supported(Cout, st_groups)) return cudaErrorInvalidValue;
    args.st_parts = args.tiles_h * args.tiles_w * 4;
    args.st_hdr = reinterpret_cast<int*>(st_buf);
    args.st_rec = reinterpret_cast<float4*>(static_cast<char*>(st_buf) + kGnStatsHeader);
    args.st_meta = reinterpret_cast<float2*>(args.st_rec + (size_t)N * T * st_groups * args.st_parts);
    args.st_cg = Cout / st_groups;
    while ((1 << args.st_lg) < args.st_cg) ++args.st_lg;
  }
  CUtensorMap ta, tc, tw, tw64;
  const int box_h = coef ? kTallRows : mode == 1 ? kPhaseRows : kTileH;  // tall boxes: prologue and phase kernels
  if (wfast ? !map_act_wh(&ta, a, Cin, W, H, T, N, a_frames) : !map_act_hw(&ta, a, Cin, W, H, T, N, box_h, a_frames))
    return cudaErrorInvalidValue;
  if (cache_in) {
    if (wfast ? !map_act_wh(&tc, cache_in, Cin, W, H, 2, N) : !map_act_hw(&tc, cache_in, Cin, W, H, 2, N, box_h))
      return cudaErrorInvalidValue;
  } else {
    tc = ta;
  }
  const int taps = mode == 0 ? 27 : mode == 1 ? 4 : mode == 2 ? 3 : 1;
  if (!map_w_half(&tw, w, taps * Cin, Cout, args.phases, 128)) return cudaErrorInvalidValue;
  if (!map_w_half(&tw64, w, taps * Cin, Cout, args.phases, 64)) return cudaErrorInvalidValue;
  if (cache_out && (!coef || cache_out == cache_in)) return cudaErrorInvalidValue;
  if (coef) {
    if (mode != 0) return cudaErrorInvalidValue;
    args.coef = coef;
    args.a = a;
    args.cache_out = cache_out;
    return wfast ? launch_pair<3>(ta, tc, tw, tw64, args, sms, stream) : launch_pair<1>(ta, tc, tw, tw64, args, sms, stream);
  }
  if (mode == 1) return launch_pair<2>(ta, tc, tw, tw64, args, sms, stream);
  return launch_pair<0>(ta, tc, tw, tw64, args, sms, stream);
}

}  // namespace wan
