// The causal 3x1x1 time upsample on CTA pairs, two output frames per item.
//
// What it computes (binding.cpp, `Decoder::up`, `time_upsample`): conv output frame t of the
// chunk is c[t] = sum_{kt} W_kt x[t + kt - 2] + bias over 2C output channels (frames before the
// chunk from the cache, else zeros); its channel half i is frame y_frame0 + 2 t + i of y. The
// general pair kernel (conv_tc2.cu, mode 2) computes one output frame per CTA and loads, for each
// of its 3 taps, a box of the input frame and a stage of the tap's weights: every MMA then streams
// both operands through shared memory and the SM's shared-memory bandwidth, not the tensor pipe,
// bounds it. Here a CTA computes output frames t and t + 1 of its 128-pixel tile into two
// accumulators (the whole of TMEM): per 64-channel K block it loads the four input frames
// t - 2 .. t + 1 once (one 64 KB stage) and the three taps' weights once (one 48 KB stage), and
// issues 24 MMAs, taps kt into accumulator 0 reading frame kt and into accumulator 1 reading frame
// kt + 1. Per K16 step and SM that is 4 KB of A and 4 KB of B read by the tensor core per MMA
// and 4.7 KB written by the TMA unit, against 8 KB written for one output frame at a time.
// Eight epilogue warps drain each accumulator, four lane quarters by two column halves. When the
// last round holds at most half as many items as there are pairs, its items run as single-frame
// units, each on its own pair (one accumulator, half the MMAs).
//
// Pair protocol (all waits bounded), as conv_tc2.cu: the odd CTA's loads complete on the even
// CTA's full barriers; MMAs are issued by one thread of the even CTA; stage releases and the
// accumulators' completion are multicast commits; both CTAs' epilogues hand the accumulators back
// to the even CTA. Each output element gets the K steps of its taps in a fixed order (K block,
// tap, K step), whatever the tile and the chunking, so chunked and unchunked calls agree bit for bit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "tma_host.h"
#include "conv_tc.h"

namespace wan {

namespace {

constexpr int kTuTileH = 8, kTuTileW = 16;   // a CTA's 128 output pixels: 8 rows x 16 columns
constexpr int kTuFrameBytes = 128 * 128;     // one input frame of the tile x 64 channels (16 KB)
constexpr int kTuAStage = 4 * kTuFrameBytes; // input frames t - 2 .. t + 1 of one K block (64 KB)
constexpr int kTuAStages = 2;
constexpr int kTuTapBytes = 128 * 128;       // this CTA's 128 weight rows x 64 channels of one tap
constexpr int kTuBStage = 3 * kTuTapBytes;   // the three taps of one K block (48 KB)
constexpr int kTuBStages = 2;
constexpr int kTuN = 256;                    // output channels per item (both CTAs' halves of B)
constexpr int kTuBOffset = kTuAStages * kTuAStage;
constexpr int kTuBarOffset = kTuBOffset + kTuBStages * kTuBStage;
constexpr int kTuSmem = kTuBarOffset + 256 + 1024;  // + barriers, + 1024-byte alignment slack
constexpr int kTuThreads = 576;              // producer, MMA issuer, 8 epilogue warps per accumulator
static_assert(kTuSmem <= 232448, "shared memory per CTA");
static_assert(kTuAStage % 1024 == 0 && kTuBStage % 1024 == 0, "stages keep the 1024-byte swizzle alignment");

struct TuArgs {
  int N, nf, H, W, C;            // input frames of the chunk (nf), channels C; output channels 2 C
  int tiles_w, tiles, tile_pairs, frame_pairs, n_blks, items;
  // Scheduling units: item i < split0 is one unit (both output frames), items from split0 on are
  // two (one output frame each): units = split0 + 2 (items - split0).
  int units, split0;
  int has_cache;
  int y_frames, y_frame0;        // y: [N, y_frames, H, W, C]
  const wan_bf16* bias;          // [2 C] or null
  wan_bf16* y;
  unsigned* err;
};

struct TuItem {
  int n, f0, h0, w0, nb;  // batch item, first output frame (f0, f0 + 1), tile origin, N block
  bool valid, second;     // this CTA's tile exists; output frame f0 + 1 exists
};

// item -> N block (fastest), tile pair, frame pair, batch item; `which` picks the pair's tile.
__device__ __forceinline__ TuItem tu_decode(const TuArgs& a, int item, int which) {
  TuItem it;
  it.nb = item % a.n_blks;
  item /= a.n_blks;
  int tile = 2 * (item % a.tile_pairs) + which;
  item /= a.tile_pairs;
  const int fp = item % a.frame_pairs;
  it.n = item / a.frame_pairs;
  it.valid = tile < a.tiles;
  if (!it.valid) tile = a.tiles - 1;  // loads as usual, stores nothing
  it.h0 = (tile / a.tiles_w) * kTuTileH;
  it.w0 = (tile % a.tiles_w) * kTuTileW;
  it.f0 = 2 * fp;
  it.second = it.f0 + 1 < a.nf;
  return it;
}

// Snake order of units over the CTA pairs; -1 once this pair has no unit in round r.
__device__ __forceinline__ int tu_unit_of(const TuArgs& a, int r, int cluster, int nclusters) {
  const int base = r * nclusters;
  if (base >= a.units) return -1;
  const int unit = base + ((r & 1) ? nclusters - 1 - cluster : cluster);
  return unit < a.units ? unit : -2;
}

// Unit -> item, and which of its output frames the unit computes (-1: both).
__device__ __forceinline__ int tu_unit_item(const TuArgs& a, int unit, int& sub) {
  if (unit < a.split0) {
    sub = -1;
    return unit;
  }
  sub = (unit - a.split0) & 1;
  return a.split0 + ((unit - a.split0) >> 1);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTuThreads, 1)
    time_up_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_cache,
                   const __grid_constant__ CUtensorMap tm_w, const TuArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + kTuBarOffset);
  uint64_t* empty_a = full_a + kTuAStages;
  uint64_t* full_b = empty_a + kTuAStages;
  uint64_t* empty_b = full_b + kTuBStages;
  uint64_t* tmem_full = empty_b + kTuBStages;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* mma_done = tmem_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int kblocks = args.C / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTuAStages; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&empty_a[s], 1);
    }
    for (int s = 0; s < kTuBStages; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_b[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 32);  // 16 epilogue warps in each CTA of the pair
    mbar_init(mma_done, 1);
    fence_mbarrier_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_cache);
    prefetch_tensormap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);  // both accumulators: 2 x 256 columns
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
    const uint32_t full_a0 = mapa_shared(smem_u32(&full_a[0]), 0), full_b0 = mapa_shared(smem_u32(&full_b[0]), 0);
    int sa = 0, sb = 0;
    uint32_t pha = 0, phb = 0;
    uint32_t armed = 0, parity = 0;  // stages whose barriers the even CTA armed: A in bits 0-1, B in 2-3
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int unit = tu_unit_of(args, r, cluster, nclusters);
      if (unit == -1) break;
      if (unit < 0) continue;
      int sub;
      const TuItem me = tu_decode(args, tu_unit_item(args, unit, sub), (int)rank);
      const int brow = me.nb * kTuN + (int)rank * 128;
      for (int kb = 0; ok && kb < kblocks; ++kb) {
        // the three taps' weights of this K block
        if (!mbar_wait_cluster(&empty_b[sb], phb ^ 1, args.err, kDevErrTimeoutProducer)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_arrive_expect_tx(&full_b[sb], 2 * kTuBStage);  // both CTAs' bytes land on it
          armed |= 4u << sb;
          parity = (parity & ~(4u << sb)) | (phb << (2 + sb));
        }
        for (int kt = 0; kt < 3; ++kt)
          tma_load_3d_pair(smem + kTuBOffset + sb * kTuBStage + kt * kTuTapBytes, &tm_w, full_b0 + 8u * (uint32_t)sb,
                           kt * args.C + kb * 64, brow, 0, w_policy);
        if (++sb == kTuBStages) {
          sb = 0;
          phb ^= 1;
        }
        // input frames f0 - 2 .. f0 + 1 of the tile (frames before the chunk from the cache, or
        // zeros; frames past the chunk's end, read only by a missing second output, zeros)
        if (!mbar_wait_cluster(&empty_a[sa], pha ^ 1, args.err, kDevErrTimeoutProducer)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_arrive_expect_tx(&full_a[sa], 2 * kTuAStage);
          armed |= 1u << sa;
          parity = (parity & ~(1u << sa)) | (pha << sa);
        }
        for (int j = 0; j < 4; ++j) {
          const int tau = me.f0 - 2 + j;
          uint8_t* dst = smem + sa * kTuAStage + j * kTuFrameBytes;
          if (tau < 0 && args.has_cache)
            tma_load_5d_pair(dst, &tm_cache, full_a0 + 8u * (uint32_t)sa, kb * 64, me.h0, me.w0, tau + 2, me.n);
          else
            tma_load_5d_pair(dst, &tm_x, full_a0 + 8u * (uint32_t)sa, kb * 64, me.h0, me.w0, tau, me.n);
        }
        if (++sa == kTuAStages) {
          sa = 0;
          pha ^= 1;
        }
      }
    }
    // Drain: every load counted on the even CTA's full barriers has landed.
    if (leader) {
      for (int s = 0; s < kTuAStages; ++s)
        if (armed & (1u << s)) mbar_wait(&full_a[s], (parity >> s) & 1, args.err, kDevErrTimeoutDrain);
      for (int s = 0; s < kTuBStages; ++s)
        if (armed & (4u << s)) mbar_wait(&full_b[s], (parity >> (2 + s)) & 1, args.err, kDevErrTimeoutDrain);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16_f32(256, kTuN);
    const uint32_t a_base = smem_u32(smem), b_base = smem_u32(smem + kTuBOffset);
    int sa = 0, sb = 0;
    uint32_t pha = 0, phb = 0, acc_phase = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int unit = tu_unit_of(args, r, cluster, nclusters);
      if (unit == -1) break;
      if (unit < 0) continue;
      int sub;
      const int item = tu_unit_item(args, unit, sub);
      // the second output frame exists for both tiles of the pair or for neither (same frames); a
      // unit of one frame accumulates frame f0 + sub into accumulator 0 from frames sub .. sub + 2
      const bool second = sub < 0 && tu_decode(args, item, 0).second;
      const uint32_t first_off = sub > 0 ? (uint32_t)(kTuFrameBytes >> 4) : 0u;
      if (!mbar_wait_cluster(tmem_empty, acc_phase ^ 1, args.err, kDevErrTimeoutMma)) break;
      tc_fence_after();
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_cluster(&full_b[sb], phb, args.err, kDevErrTimeoutMma) ||
            !mbar_wait_cluster(&full_a[sa], pha, args.err, kDevErrTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t a0 = smem_desc_sw128(a_base + sa * kTuAStage), b0 = smem_desc_sw128(b_base + sb * kTuBStage);
#pragma unroll
        for (int kt = 0; kt < 3; ++kt) {
          const uint64_t bk = b0 + (uint64_t)kt * (kTuTapBytes >> 4);
          const uint64_t af = a0 + first_off + (uint64_t)kt * (kTuFrameBytes >> 4);  // frame f0 - 2 + kt (+ sub)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_pair(tmem_base, af + 2 * k, bk + 2 * k, idesc, (kb == 0 && kt == 0 && k == 0) ? 0u : 1u);
          if (second) {
            const uint64_t ag = af + (uint64_t)(kTuFrameBytes >> 4);  // frame f0 - 1 + kt
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_pair(tmem_base + kTuN, ag + 2 * k, bk + 2 * k, idesc, (kb == 0 && kt == 0 && k == 0) ? 0u : 1u);
          }
        }
        mma_commit_pair(&empty_a[sa], 0x3);
        mma_commit_pair(&empty_b[sb], 0x3);
        if (++sa == kTuAStages) {
          sa = 0;
          pha ^= 1;
        }
        if (++sb == kTuBStages) {
          sb = 0;
          phb ^= 1;
        }
      }
      if (!ok) break;
      mma_commit_pair(tmem_full, 0x3);
      acc_phase ^= 1;
    }
    mma_commit_pair(mma_done, 0x1);
    mbar_wait(mma_done, 0, args.err, kDevErrTimeoutDrain);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs, own 128 rows)
    // Warps 2-9 drain accumulator 0 and warps 10-17 accumulator 1, each warp 128 of its 256 columns
    // for the TMEM lanes of quarter warp % 4, so an item's two output frames are written at once.
    const int quarter = warp & 3, row = quarter * 32 + lane, o = (warp - 2) / 8;
    const int col0 = (((warp - 2) >> 2) & 1) * (kTuN / 2);
    const uint32_t leader_empty = mapa_shared(smem_u32(tmem_empty), 0);
    uint32_t acc_phase = 0;
    for (int r = 0;; ++r) {
      const int unit = tu_unit_of(args, r, cluster, nclusters);
      if (unit == -1) break;
      if (unit < 0) continue;
      int sub;
      const TuItem t = tu_decode(args, tu_unit_item(args, unit, sub), (int)rank);
      // accumulator o holds output frame f0 + o of a whole unit; a unit of one frame has it in
      // accumulator 0 (accumulator 1's warps only hand the accumulators back)
      const int frame = sub < 0 ? t.f0 + o : t.f0 + sub;
      const bool writes = sub < 0 ? (o == 0 || t.second) : (o == 0 && (sub == 0 || t.second));
      const int hh = t.h0 + (row & 7), ww = t.w0 + row / 8;  // TMEM row = h + 8 w
      const bool valid = t.valid && hh < args.H && ww < args.W;
      const int half = t.nb * kTuN / args.C;  // the N block's channel half: output frame 2 t + half
      const int cy = t.nb * kTuN - half * args.C;
      if (!mbar_wait_cluster(tmem_full, acc_phase, args.err, kDevErrTimeoutEpilogue)) break;
      tc_fence_after();
      if (writes) {
        const int fy = args.y_frame0 + 2 * frame + half;
        wan_bf16* yrow = args.y + ((((size_t)t.n * args.y_frames + fy) * args.H + hh) * args.W + ww) * args.C + cy;
        const uint32_t taddr =
            tmem_base + (uint32_t)((sub < 0 ? o : 0) * kTuN + col0) + ((uint32_t)(quarter * 32) << 16);
        uint32_t rn[16];
        __syncwarp();
        tmem_ld16_issue(taddr, rn);
        tmem_ld16_wait(rn);
#pragma unroll 1
        for (int c0 = 0; c0 < kTuN / 2; c0 += 16) {
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(rn[i]);
          if (c0 + 16 < kTuN / 2) {
            __syncwarp();
            tmem_ld16_issue(taddr + c0 + 16, rn);
          }
          if (valid) {
            if (args.bias) {
              const uint4 b0 = __ldg(reinterpret_cast<const uint4*>(args.bias + t.nb * kTuN + col0 + c0));
              const uint4 b1 = __ldg(reinterpret_cast<const uint4*>(args.bias + t.nb * kTuN + col0 + c0 + 8));
              const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[2 * i] += bf16lo_to_f32(bw[i]);
                v[2 * i + 1] += bf16hi_to_f32(bw[i]);
              }
            }
            uint32_t ov[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) ov[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            *reinterpret_cast<uint4*>(yrow + col0 + c0) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
            *reinterpret_cast<uint4*>(yrow + col0 + c0 + 8) = make_uint4(ov[4], ov[5], ov[6], ov[7]);
          }
          if (c0 + 16 < kTuN / 2) tmem_ld16_wait(rn);
        }
      }
      // This warp is done with both accumulators: one arrival per warp on the even CTA's barrier.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(leader_empty);
      acc_phase ^= 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or arrivals may still touch it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, 512);
}

// Activations [N, ., H, W, C] addressed as (c, h, w, t, n) with `frames` frames mapped per n
// (n_frames apart): a box of 64 channels x 8 rows x 16 columns of one frame lands column by column
// (row m = h + 8 w). Coordinates outside the map read zeros.
bool tu_map_act(CUtensorMap* m, const void* base, int C, int W, int H, int frames, int N, int n_frames) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[5] = {(cuuint64_t)C, (cuuint64_t)H, (cuuint64_t)W, (cuuint64_t)frames, (cuuint64_t)N};
  const cuuint64_t e = 2;
  const cuuint64_t strides[4] = {(cuuint64_t)W * C * e, C * e, (cuuint64_t)H * W * C * e,
                                 (cuuint64_t)n_frames * H * W * C * e};
  const cuuint32_t box[5] = {64, (cuuint32_t)kTuTileH, (cuuint32_t)kTuTileW, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weights [2 C][3 C] (output channel, tap * C + input channel) as (k, cout): boxes of 64 K x 128 rows.
bool tu_map_w(CUtensorMap* m, const void* base, int K, int Cout) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)Cout, 1};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * Cout * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool time_up_supported(int C) { return C >= 256 && C % 256 == 0; }

cudaError_t time_up_launch(const wan_bf16* x, const wan_bf16* cache_in, const wan_bf16* w, const wan_bf16* bias,
                           wan_bf16* y, int N, int nf, int H, int W, int C, int a_frames, int y_frames, int y_frame0,
                           int sms, unsigned* err, cudaStream_t stream) {
  if (!time_up_supported(C) || nf <= 0 || a_frames < nf) return cudaErrorInvalidValue;
  TuArgs args{};
  args.N = N;
  args.nf = nf;
  args.H = H;
  args.W = W;
  args.C = C;
  args.tiles_w = cdiv(W, kTuTileW);
  args.tiles = cdiv(H, kTuTileH) * args.tiles_w;
  args.tile_pairs = cdiv(args.tiles, 2);
  args.frame_pairs = cdiv(nf, 2);
  args.n_blks = 2 * C / kTuN;
  const long long items = (long long)N * args.frame_pairs * args.tile_pairs * args.n_blks;
  if (items >= (1LL << 31)) return cudaErrorInvalidValue;
  args.items = (int)items;
  args.has_cache = cache_in != nullptr;
  args.y_frames = y_frames;
  args.y_frame0 = y_frame0;
  args.bias = bias;
  args.y = y;
  args.err = err;
  CUtensorMap tx, tc, tw;
  if (!tu_map_act(&tx, x, C, W, H, nf, N, a_frames)) return cudaErrorInvalidValue;
  if (cache_in) {
    if (!tu_map_act(&tc, cache_in, C, W, H, 2, N, 2)) return cudaErrorInvalidValue;
  } else {
    tc = tx;
  }
  if (!tu_map_w(&tw, w, 3 * C, 2 * C)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(time_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTuSmem);
  if (e != cudaSuccess) return e;
  int clusters = resident_pairs(reinterpret_cast<const void*>(time_up_kernel), kTuThreads, kTuSmem, sms);
  // A last round of at most half the pairs' worth of items runs as twice as many units of one
  // output frame each (half the MMAs).
  const int rem = args.items % clusters;
  args.split0 = args.items;
  args.units = args.items;
  if (rem > 0 && 2 * rem <= clusters) {
    args.split0 = args.items - rem;
    args.units = args.items + rem;
  }
  if (clusters > args.units) clusters = args.units;
  if (clusters < 1) clusters = 1;
  time_up_kernel<<<2 * clusters, kTuThreads, kTuSmem, stream>>>(tx, tc, tw, args);
  return cudaGetLastError();
}

}  // namespace wan
