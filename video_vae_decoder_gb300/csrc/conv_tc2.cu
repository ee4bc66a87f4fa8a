// Implicit-GEMM convolutions on CTA pairs: tcgen05.mma with .cta_group::2 (M = 256 over two SMs).
//
// Same computations as conv_tc.cu (mode 0: the causal 3x3x3 convolution with its cache frames,
// binding.cpp `Decoder::conv`; mode 1: the four 2x2 phase convolutions of the upsampler,
// `Decoder::up`), for output-channel blocks of 256. Why a second kernel: with one CTA per tile,
// an M128 x N256 x K16 MMA reads 12 KB of operands from shared memory while the TMA unit writes
// the next 12 KB, which is more shared-memory traffic per SM than the SM can serve, so the tensor
// pipe idled about 40% of the time. On a CTA pair (a cluster of 2 on two SMs) each SM holds its own
// 128 output rows of A and HALF of B (128 of the 256 weight rows); one thread of the even CTA
// issues the M256 x N256 MMAs that read both SMs' halves, and each SM's TMEM receives its 128
// rows. Each SM then moves 8 KB per K16 step instead of 12.
//
// Pair protocol (all waits bounded):
//   full[s]       in the even CTA: both CTAs' TMA bytes for stage s (A: each CTA's pixel block,
//                 B: each CTA's weight half); the odd CTA's loads complete on it directly
//   empty[s]      both CTAs: the MMAs reading stage s are done (multicast tcgen05.commit)
//   tmem_full[a]  both CTAs: accumulator a holds a finished tile (multicast commit)
//   tmem_empty[a] in the even CTA: both CTAs' epilogues drained accumulator a (8 warp arrivals)
// Tiles: an item is (N block, phase, pair of pixel blocks); the even CTA computes the first pixel
// block, the odd CTA the second (a missing second block loads zeros and stores nothing). Both
// blocks of a pair use the same weights, so in mode 1 a pair never mixes phases.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "conv_tc.h"

namespace wan {

namespace {

constexpr int kThreads = 192;
constexpr int kBlockK = 64;
constexpr int kABytes = 128 * 128;      // 128 rows x 64 bf16
constexpr int kBBytes = 128 * 128;      // this CTA's 128 weight rows x 64 bf16
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStages = 6;
constexpr int kBarOffset = kStages * kStageBytes;
constexpr int kSmemTotal = kBarOffset + 512 + 1024;
constexpr int kN = 256;                 // output channels per item (both halves)
constexpr int kTmemCols = 512;          // 2 accumulators x 256 columns

struct Conv2Args {
  int N, T, H, W, Cin, Cout;
  int TT, TH, TW;
  int tiles_t, tiles_h, tiles_w;
  int px_tiles, px_pairs;
  int n_blks, phases, items;
  int kb_per_tap, taps, mode, has_cache;
  const wan_bf16* bias;
  const wan_bf16* residual;
  wan_bf16* y;
  unsigned* err;
};

struct PTile {
  int n, t0, h0, w0, ph, nb;
  bool valid;
};

// item -> N block (fastest), phase, pixel pair; `which` picks the pair's first or second block.
__device__ __forceinline__ PTile decode_pair(const Conv2Args& a, int item, int which) {
  PTile t;
  t.nb = item % a.n_blks;
  item /= a.n_blks;
  t.ph = item % a.phases;
  item /= a.phases;
  int px = 2 * item + which;
  t.valid = px < a.px_tiles;
  if (!t.valid) px = 2 * item;
  t.t0 = (px % a.tiles_t) * a.TT;
  px /= a.tiles_t;
  t.w0 = (px % a.tiles_w) * a.TW;
  px /= a.tiles_w;
  t.h0 = (px % a.tiles_h) * a.TH;
  t.n = px / a.tiles_h;
  return t;
}

__device__ __forceinline__ void tap_offsets2(const Conv2Args& a, int tap, int ph, int& dt, int& dh, int& dw) {
  if (a.mode == 0) {
    dt = tap / 9 - 2;
    dh = (tap / 3) % 3 - 1;
    dw = tap % 3 - 1;
  } else {
    const int pa = ph >> 1, pb = ph & 1, u = tap >> 1, v = tap & 1;
    dt = 0;
    dh = pa - 1 + u;
    dw = pb - 1 + v;
  }
}

// A k-step is skipped only when it reads nothing but zeros for BOTH blocks of the pair (frames
// before a chunk that has no history; a missing second block counts as zeros).
__device__ __forceinline__ bool skip_pair(const Conv2Args& a, const PTile& p0, const PTile& p1, int dt) {
  if (a.has_cache) return false;
  const bool z0 = p0.t0 + a.TT - 1 + dt < 0;
  const bool z1 = !p1.valid || (p1.t0 + a.TT - 1 + dt < 0);
  return z0 && z1;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    conv_tc2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_cache,
                    const __grid_constant__ CUtensorMap tm_w, const Conv2Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* mma_done = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
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
  const int num_k = args.taps * args.kb_per_tap;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    const uint64_t w_policy = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    uint32_t bar_addr[kStages];  // the even CTA's full barriers, shared::cluster addresses
#pragma unroll
    for (int s2 = 0; s2 < kStages; ++s2) bar_addr[s2] = mapa_shared(smem_u32(&full[s2]), 0);
    const int box_bytes = args.TH * args.TW * 128;
    for (int item = cluster; ok && item < args.items; item += nclusters) {
      const PTile me = decode_pair(args, item, (int)rank);
      const PTile p0 = decode_pair(args, item, 0), p1 = decode_pair(args, item, 1);
      const int brow = me.nb * kN + (int)rank * 128;
      for (int tap = 0; ok && tap < args.taps; ++tap) {
        int dt, dh, dw;
        tap_offsets2(args, tap, me.ph, dt, dh, dw);
        if (skip_pair(args, p0, p1, dt)) continue;
        const int hh = me.h0 + dh, ww = me.w0 + dw;
        for (int kb = 0; kb < args.kb_per_tap; ++kb) {
          if (!mbar_wait_cluster(&empty[stage], phase ^ 1, args.err, kDevErrTimeoutProducer)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = smem + stage * kStageBytes;
          uint8_t* b_dst = a_dst + kABytes;
          const uint32_t bar = bar_addr[stage];
          if (leader) {
            mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);  // both CTAs' bytes land on it
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          for (int i = 0; i < args.TT; ++i) {
            int tau = me.t0 + i + dt;
            if (!me.valid) tau = args.T + 8;  // out of range: the TMA unit fills zeros
            if (tau < 0 && args.has_cache)
              tma_load_5d_pair(a_dst + i * box_bytes, &tm_cache, bar, kb * kBlockK, ww, hh, tau + 2, me.n);
            else
              tma_load_5d_pair(a_dst + i * box_bytes, &tm_a, bar, kb * kBlockK, ww, hh, tau, me.n);
          }
          tma_load_3d_pair(b_dst, &tm_w, bar, tap * args.Cin + kb * kBlockK, brow, me.ph, w_policy);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    // Drain (even CTA): both CTAs' loads counted on its full barriers have landed.
    for (int s = 0; s < kStages; ++s)
      if (armed & (1u << s)) mbar_wait(&full[s], (armed_parity >> s) & 1, args.err, kDevErrTimeoutDrain);
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16_f32(256, kN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int item = cluster; ok && item < args.items; item += nclusters) {
      const PTile p0 = decode_pair(args, item, 0), p1 = decode_pair(args, item, 1);
      if (!mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1, args.err, kDevErrTimeoutMma)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kN;
      bool first = true;
      for (int tap = 0; ok && tap < args.taps; ++tap) {
        if (!args.has_cache) {  // without history some taps read only zeros for both blocks
          int dt, dh, dw;
          tap_offsets2(args, tap, p0.ph, dt, dh, dw);
          if (skip_pair(args, p0, p1, dt)) continue;
        }
        for (int kb = 0; kb < args.kb_per_tap; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase, args.err, kDevErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kStageBytes);
          const uint64_t a_desc = smem_desc_sw128(a_addr);
          const uint64_t b_desc = smem_desc_sw128(a_addr + kABytes);
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k)
            mma_bf16_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
          first = false;
          mma_commit_pair(&empty[stage], 0x3);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
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
    for (int item = cluster; item < args.items; item += nclusters) {
      const PTile t = decode_pair(args, item, (int)rank);
      if (!mbar_wait_cluster(&tmem_full[acc], acc_phase, args.err, kDevErrTimeoutEpilogue)) break;
      tc_fence_after();
      const int per_frame = args.TH * args.TW;
      const int it = row / per_frame;
      const int ih = (row / args.TW) % args.TH;
      const int iw = row % args.TW;
      const int tt = t.t0 + it, hh = t.h0 + ih, ww = t.w0 + iw;
      const bool valid = t.valid && tt < args.T && hh < args.H && ww < args.W;
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

bool map_act(CUtensorMap* m, const void* base, int C, int W, int H, int T, int N, int box_w, int box_h) {
  auto fn = encode_fn2();
  if (!fn) return false;
  const cuuint64_t dims[5] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)N};
  const cuuint64_t e = 2;
  const cuuint64_t strides[4] = {C * e, (cuuint64_t)W * C * e, (cuuint64_t)H * W * C * e, (cuuint64_t)T * H * W * C * e};
  const cuuint32_t box[5] = {(cuuint32_t)kBlockK, (cuuint32_t)box_w, (cuuint32_t)box_h, 1, 1};
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
                             int Cin, int Cout, int TT, int TH, int TW, int sms, unsigned* err, cudaStream_t stream) {
  Conv2Args args{};
  args.N = N;
  args.T = T;
  args.H = H;
  args.W = W;
  args.Cin = Cin;
  args.Cout = Cout;
  args.TT = TT;
  args.TH = TH;
  args.TW = TW;
  args.tiles_t = cdiv(T, TT);
  args.tiles_h = cdiv(H, TH);
  args.tiles_w = cdiv(W, TW);
  args.px_tiles = N * args.tiles_t * args.tiles_h * args.tiles_w;
  args.px_pairs = cdiv(args.px_tiles, 2);
  args.n_blks = cdiv(Cout, kN);
  args.phases = mode == 0 ? 1 : 4;
  args.items = args.px_pairs * args.phases * args.n_blks;
  args.kb_per_tap = Cin / kBlockK;
  args.taps = mode == 0 ? 27 : 4;
  args.mode = mode;
  args.has_cache = cache_in != nullptr;
  args.bias = bias;
  args.residual = residual;
  args.y = y;
  args.err = err;
  CUtensorMap ta, tc, tw;
  if (!map_act(&ta, a, Cin, W, H, T, N, TW, TH)) return cudaErrorInvalidValue;
  if (cache_in) {
    if (!map_act(&tc, cache_in, Cin, W, H, 2, N, TW, TH)) return cudaErrorInvalidValue;
  } else {
    tc = ta;
  }
  if (!map_w_half(&tw, w, args.taps * Cin, Cout, args.phases)) return cudaErrorInvalidValue;
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
