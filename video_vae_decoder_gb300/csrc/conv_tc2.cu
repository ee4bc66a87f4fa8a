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
// items of different cost (the first frames of a chunk without history skip taps).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "conv_tc.h"

namespace wan {

namespace {

constexpr int kThreads = 192;           // producer, MMA issuer, 4 epilogue warps
constexpr int kBlockK = 64;
constexpr int kTileH = 8, kTileW = 16;  // output pixels of one CTA: 8 rows x 16 columns
constexpr int kBoxW = kTileW + 2;       // input columns of one A box (one halo column per side)
constexpr int kABytes = kTileH * kBoxW * 128;  // 144 rows x 64 bf16 = 18 KB
constexpr int kBBytes = 128 * 128;             // this CTA's 128 weight rows x 64 bf16
constexpr int kAStages = 4;
constexpr int kBStages = 9;
constexpr int kBOffset = kAStages * kABytes;
constexpr int kBarOffset = kBOffset + kBStages * kBBytes;
constexpr int kSmemTotal = kBarOffset + 512 + 1024;
constexpr int kN = 256;                 // output channels per item (both halves)
constexpr int kTmemCols = 512;          // 2 accumulators x 256 columns
constexpr uint32_t kShiftDesc = (kTileH * 128) >> 4;  // one column of the box, in descriptor units

static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
static_assert(kSmemTotal <= 232448, "shared memory per CTA");

struct Conv2Args {
  int N, T, H, W, Cin, Cout;
  int tiles_h, tiles_w;
  int px_tiles, px_pairs;
  int n_blks, phases, items;
  int kb_per_tap, mode, has_cache;
  const wan_bf16* bias;
  const wan_bf16* residual;
  wan_bf16* y;
  unsigned* err;
};

struct PTile {
  int n, t0, h0, w0, ph, nb;
  bool valid;
};

// item -> N block (fastest), phase, pixel pair; `which` picks the pair's first or second tile.
// Pixel tiles are numbered frame-fastest, so concurrently running pairs share input frames in L2.
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
  t.w0 = (px % a.tiles_w) * kTileW;
  px /= a.tiles_w;
  t.h0 = (px % a.tiles_h) * kTileH;
  t.n = px / a.tiles_h;
  return t;
}

// Snake order of items over the CTA pairs; -1 once this pair has no item in round r.
__device__ __forceinline__ int item_of(const Conv2Args& a, int r, int cluster, int nclusters) {
  const int base = r * nclusters;
  if (base >= a.items) return -1;
  const int item = base + ((r & 1) ? nclusters - 1 - cluster : cluster);
  return item < a.items ? item : -2;  // -2: nothing in this (last) round
}

// Kernel row `row` of the tap grid: its frame and row offsets, and the input column of the A
// box's first column relative to the tile. Mode 0: 9 rows (dt, dh) of 3 horizontal taps; mode 1:
// for phase (pa, pb) the 2 rows u of 2 taps v, reading input (h + pa - 1 + u, w + pb - 1 + v).
__device__ __forceinline__ void row_offsets(const Conv2Args& a, int row, int ph, int& dt, int& dh, int& dw0) {
  if (a.mode == 0) {
    dt = row / 3 - 2;
    dh = row % 3 - 1;
    dw0 = -1;
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    conv_tc2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_cache,
                    const __grid_constant__ CUtensorMap tm_w, const Conv2Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty_a = full_a + kAStages;
  uint64_t* full_b = empty_a + kAStages;
  uint64_t* empty_b = full_b + kBStages;
  uint64_t* tmem_full = empty_b + kBStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* mma_done = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int rows = args.mode == 0 ? 9 : 2;     // kernel rows
  const int taps_per_row = args.mode == 0 ? 3 : 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&empty_a[s], 1);
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
    fence_mbarrier_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_cache);
    prefetch_tensormap(&tm_w);
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
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = item_of(args, r, cluster, nclusters);
      if (item == -1) break;
      if (item < 0) continue;
      const PTile me = decode_pair(args, item, (int)rank);
      const PTile p0 = decode_pair(args, item, 0), p1 = decode_pair(args, item, 1);
      const int brow = me.nb * kN + (int)rank * 128;
      for (int row = 0; ok && row < rows; ++row) {
        int dt, dh, dw0;
        row_offsets(args, row, me.ph, dt, dh, dw0);
        if (skip_pair(args, p0, p1, dt)) continue;
        const int hh = me.h0 + dh, ww = me.w0 + dw0;
        int tau = me.t0 + dt;
        if (!me.valid) tau = args.T + 8;  // out of range: the TMA unit fills zeros
        for (int kb = 0; ok && kb < args.kb_per_tap; ++kb) {
          if (!mbar_wait_cluster(&empty_a[sa], pha ^ 1, args.err, kDevErrTimeoutProducer)) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(&full_a[sa], 2 * kABytes);  // both CTAs' bytes land on it
            armed_a |= 1u << sa;
            parity_a = (parity_a & ~(1u << sa)) | (pha << sa);
          }
          const uint32_t bar_a = mapa_shared(smem_u32(&full_a[sa]), 0);
          uint8_t* a_dst = smem + sa * kABytes;
          if (tau < 0 && args.has_cache)
            tma_load_5d_pair(a_dst, &tm_cache, bar_a, kb * kBlockK, hh, ww, tau + 2, me.n);
          else
            tma_load_5d_pair(a_dst, &tm_a, bar_a, kb * kBlockK, hh, ww, tau, me.n);
          if (++sa == kAStages) {
            sa = 0;
            pha ^= 1;
          }
          for (int j = 0; j < taps_per_row; ++j) {
            if (!mbar_wait_cluster(&empty_b[sb], phb ^ 1, args.err, kDevErrTimeoutProducer)) {
              ok = false;
              break;
            }
            if (leader) {
              mbar_arrive_expect_tx(&full_b[sb], 2 * kBBytes);
              armed_b |= 1u << sb;
              parity_b = (parity_b & ~(1u << sb)) | (phb << sb);
            }
            const int tap = row * taps_per_row + j;
            tma_load_3d_pair(smem + kBOffset + sb * kBBytes, &tm_w, mapa_shared(smem_u32(&full_b[sb]), 0),
                             tap * args.Cin + kb * kBlockK, brow, me.ph, w_policy);
            if (++sb == kBStages) {
              sb = 0;
              phb ^= 1;
            }
          }
        }
      }
    }
    // Drain (even CTA): both CTAs' loads counted on its full barriers have landed.
    for (int s = 0; s < kAStages; ++s)
      if (armed_a & (1u << s)) mbar_wait(&full_a[s], (parity_a >> s) & 1, args.err, kDevErrTimeoutDrain);
    for (int s = 0; s < kBStages; ++s)
      if (armed_b & (1u << s)) mbar_wait(&full_b[s], (parity_b >> s) & 1, args.err, kDevErrTimeoutDrain);
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16_f32(256, kN);
    const uint32_t a_base = smem_u32(smem), b_base = smem_u32(smem + kBOffset);
    int sa = 0, sb = 0;
    uint32_t pha = 0, phb = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = item_of(args, r, cluster, nclusters);
      if (item == -1) break;
      if (item < 0) continue;
      const PTile p0 = decode_pair(args, item, 0), p1 = decode_pair(args, item, 1);
      if (!mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1, args.err, kDevErrTimeoutMma)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kN;
      bool first = true;
      for (int row = 0; ok && row < rows; ++row) {
        if (!args.has_cache) {  // without history some rows read only zeros for both tiles
          int dt, dh, dw0;
          row_offsets(args, row, p0.ph, dt, dh, dw0);
          if (skip_pair(args, p0, p1, dt)) continue;
        }
        for (int kb = 0; ok && kb < args.kb_per_tap; ++kb) {
          if (!mbar_wait_cluster(&full_a[sa], pha, args.err, kDevErrTimeoutMma)) {
            ok = false;
            break;
          }
          const uint64_t a_desc = smem_desc_sw128(a_base + sa * kABytes);
          for (int j = 0; j < taps_per_row; ++j) {
            if (!mbar_wait_cluster(&full_b[sb], phb, args.err, kDevErrTimeoutMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t aj = a_desc + j * kShiftDesc;
            const uint64_t b_desc = smem_desc_sw128(b_base + sb * kBBytes);
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k)
              mma_bf16_pair(d_tmem, aj + 2 * k, b_desc + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
            first = false;
            mma_commit_pair(&empty_b[sb], 0x3);
            if (++sb == kBStages) {
              sb = 0;
              phb ^= 1;
            }
          }
          if (!ok) break;
          mma_commit_pair(&empty_a[sa], 0x3);
          if (++sa == kAStages) {
            sa = 0;
            pha ^= 1;
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
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs, own 128 rows)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int Ho = args.mode == 0 ? args.H : 2 * args.H;
    const int Wo = args.mode == 0 ? args.W : 2 * args.W;
    const bool vec8 = (args.Cout % 8) == 0;
    const uint32_t leader_empty0 = mapa_shared(smem_u32(&tmem_empty[0]), 0);
    const uint32_t leader_empty1 = mapa_shared(smem_u32(&tmem_empty[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int r = 0;; ++r) {
      const int item = item_of(args, r, cluster, nclusters);
      if (item == -1) break;
      if (item < 0) continue;
      const PTile t = decode_pair(args, item, (int)rank);
      if (!mbar_wait_cluster(&tmem_full[acc], acc_phase, args.err, kDevErrTimeoutEpilogue)) break;
      tc_fence_after();
      const int hh = t.h0 + (row & (kTileH - 1)), ww = t.w0 + row / kTileH;  // TMEM row = h + 8 w
      const int tt = t.t0;
      const bool valid = t.valid && hh < args.H && ww < args.W;
      size_t pix;
      if (args.mode == 0)
        pix = (((size_t)t.n * args.T + tt) * Ho + hh) * Wo + ww;
      else
        pix = (((size_t)t.n * args.T + tt) * Ho + (2 * hh + (t.ph >> 1))) * Wo + (2 * ww + (t.ph & 1));
      wan_bf16* yrow = args.y + pix * args.Cout;
      const wan_bf16* rrow = args.residual ? args.residual + pix * args.Cout : nullptr;
      const uint32_t taddr = tmem_base + (uint32_t)(acc * kN) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < kN; c0 += 16) {
        float v[16];
        __syncwarp();
        tmem_ld16(taddr + c0, v);
        const int col = t.nb * kN + c0;
        if (valid && col < args.Cout) {
          if (args.bias) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (col + i < args.Cout) v[i] += __uint_as_float(((uint32_t)args.bias[col + i]) << 16);
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
            uint32_t o[8];
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
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or arrivals may still touch it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn2() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Activations [N, T, H, W, C] addressed as (c, h, w, t, n): H is listed before W, so a box of
// 8 rows x 18 columns lands in shared memory column by column (row m = h + 8 w).
bool map_act_hw(CUtensorMap* m, const void* base, int C, int W, int H, int T, int N) {
  auto fn = encode_fn2();
  if (!fn) return false;
  const cuuint64_t dims[5] = {(cuuint64_t)C, (cuuint64_t)H, (cuuint64_t)W, (cuuint64_t)T, (cuuint64_t)N};
  const cuuint64_t e = 2;
  const cuuint64_t strides[4] = {(cuuint64_t)W * C * e, C * e, (cuuint64_t)H * W * C * e, (cuuint64_t)T * H * W * C * e};
  const cuuint32_t box[5] = {(cuuint32_t)kBlockK, (cuuint32_t)kTileH, (cuuint32_t)kBoxW, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_w_half(CUtensorMap* m, const void* base, int K, int Cout, int P) {
  auto fn = encode_fn2();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)Cout, (cuuint64_t)P};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * Cout * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBlockK, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool conv_pair_supported(int Cout) { return Cout >= 256; }

cudaError_t conv_pair_launch(int mode, const wan_bf16* a, const wan_bf16* cache_in, const wan_bf16* w,
                             const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                             int Cin, int Cout, int sms, unsigned* err, cudaStream_t stream) {
  Conv2Args args{};
  args.N = N;
  args.T = T;
  args.H = H;
  args.W = W;
  args.Cin = Cin;
  args.Cout = Cout;
  args.tiles_h = cdiv(H, kTileH);
  args.tiles_w = cdiv(W, kTileW);
  args.px_tiles = N * T * args.tiles_h * args.tiles_w;
  args.px_pairs = cdiv(args.px_tiles, 2);
  args.n_blks = cdiv(Cout, kN);
  args.phases = mode == 0 ? 1 : 4;
  args.items = args.px_pairs * args.phases * args.n_blks;
  args.kb_per_tap = Cin / kBlockK;
  args.mode = mode;
  args.has_cache = cache_in != nullptr;
  args.bias = bias;
  args.residual = residual;
  args.y = y;
  args.err = err;
  CUtensorMap ta, tc, tw;
  if (!map_act_hw(&ta, a, Cin, W, H, T, N)) return cudaErrorInvalidValue;
  if (cache_in) {
    if (!map_act_hw(&tc, cache_in, Cin, W, H, 2, N)) return cudaErrorInvalidValue;
  } else {
    tc = ta;
  }
  if (!map_w_half(&tw, w, (mode == 0 ? 27 : 4) * Cin, Cout, args.phases)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(conv_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
  if (e != cudaSuccess) return e;
  // Persistent grid: as many CTA pairs as the GPU can hold at once (not every SM can be paired:
  // a pair lives in one GPC), so no pair waits for a second wave.
  static int max_clusters[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && max_clusters[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemTotal;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, conv_tc2_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sms / 2;
    }
    max_clusters[dev] = n;
  }
  int clusters = (dev >= 0 && dev < 64) ? max_clusters[dev] : sms / 2;
  if (clusters > args.items) clusters = args.items;
  if (clusters < 1) clusters = 1;
  conv_tc2_kernel<<<2 * clusters, kThreads, kSmemTotal, stream>>>(ta, tc, tw, args);
  return cudaGetLastError();
}

}  // namespace wan
