// Implicit-GEMM convolutions on the sm_103a tensor cores (tcgen05.mma, accumulators in TMEM,
// operands staged by TMA), for
//   mode 0: the causal 3x3x3 convolution of the video decoder (binding.cpp, `Decoder::conv`):
//           the input frames of output frame t are t-2, t-1, t; frames before the chunk come
//           from the carried two-frame cache (or are zero), H and W are zero-padded by one;
//   mode 1: the four 2x2 phase convolutions of the nearest-x2 upsampler (binding.cpp,
//           `Decoder::up`), each output written to its parity position of the 2H x 2W frame.
//
// GEMM view: rows m = output pixels (a TT x TH x TW block of frames x rows x columns, 128 rows),
// columns n = output channels (BN per tile), reduction k = (tap, input channel). For every tap
// the A tile is the same pixel block shifted by the tap's offset: one TMA box per frame
// [64 channels x TW x TH] from the 5-D channels-last tensor, out-of-range pixels and frames
// zero-filled by the TMA unit (this is the zero padding, and the zero history of a first
// chunk). The B tile is [BN rows x 64 k] of the weights viewed as [Cout][taps * Cin].
// Both tiles land in shared memory in the 128-byte-swizzled K-major layout that tcgen05 reads.
//
// One persistent CTA per SM, three roles:
//   warp 0      TMA producer: fills a STAGES-deep ring of (A, B) stages;
//   warp 1      MMA issuer: one thread issues 4 x (M128 x N x K16) MMAs per stage into one of
//               two TMEM accumulators, and releases stages with tcgen05.commit;
//   warps 2..5  epilogue: TMEM -> registers, + bias + residual in fp32, one rounding to bf16,
//               stores; the other accumulator keeps the tensor cores busy meanwhile.
// Every reduction runs in the same tap order for every output, independent of the tile's
// position and of how the video was chunked, so chunked and unchunked runs give equal bits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "tma_host.h"
#include "conv_tc.h"

namespace wan {

namespace {

constexpr int kThreads = 192;
constexpr int kBlockK = 64;            // channels per k-step: one 128-byte swizzle row
constexpr int kTileM = 128;
constexpr int kABytes = kTileM * 128;  // 16 KB

struct ConvArgs {
  int N, T, H, W, Cin, Cout;
  int TT, TH, TW;
  int tiles_t, tiles_h, tiles_w;
  int n_blks, phases, num_tiles;
  int kb_per_tap, taps, mode, has_cache;
  const wan_bf16* bias;
  const wan_bf16* residual;
  wan_bf16* y;
  unsigned* err;
};

struct Tile {
  int n, t0, h0, w0, ph, nb;
};

// Tile order: N block fastest, then phase, then the frame block, then the pixel block. Tiles of
// the same pixels in neighbouring frames run side by side, so the input frames they share (an
// output frame reads frames t-2..t) are fetched from HBM about once and then hit in L2.
__device__ __forceinline__ Tile decode_tile(const ConvArgs& a, int idx) {
  Tile t;
  t.nb = idx % a.n_blks;
  idx /= a.n_blks;
  t.ph = idx % a.phases;
  idx /= a.phases;
  t.t0 = (idx % a.tiles_t) * a.TT;
  idx /= a.tiles_t;
  t.w0 = (idx % a.tiles_w) * a.TW;
  idx /= a.tiles_w;
  t.h0 = (idx % a.tiles_h) * a.TH;
  t.n = idx / a.tiles_h;
  return t;
}

// Offsets of tap `tap` of phase `ph`: (dt, dh, dw).
__device__ __forceinline__ void tap_offsets(const ConvArgs& a, int tap, int ph, int& dt, int& dh,
                                            int& dw) {
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

// A k-step whose every frame lies before a chunk that has no history reads only zeros.
__device__ __forceinline__ bool skip_step(const ConvArgs& a, const Tile& t, int dt) {
  return !a.has_cache && (t.t0 + a.TT - 1 + dt < 0);
}

template <int BN, int STAGES>
struct Smem {
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kTotal = kBarOffset + 256 + 1024;  // barriers + alignment slack
  static constexpr int kTmemCols = (2 * BN) < 32 ? 32 : 2 * BN;
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    conv_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_cache,
                   const __grid_constant__ CUtensorMap tm_w, const ConvArgs args) {
  using S = Smem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOffset);
  uint64_t* empty = full + STAGES;
  uint64_t* tmem_full = empty + STAGES;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* mma_done = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], 128);
    }
    mbar_init(mma_done, 1);
    fence_mbarrier_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_cache);
    prefetch_tensormap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_k = args.taps * args.kb_per_tap;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    const uint64_t w_policy = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;  // per-stage: ever armed, parity of the last arming
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
      const Tile t = decode_tile(args, tile);
      for (int ks = 0; ks < num_k; ++ks) {
        const int tap = ks / args.kb_per_tap;
        const int kb = ks - tap * args.kb_per_tap;
        int dt, dh, dw;
        tap_offsets(args, tap, t.ph, dt, dh, dw);
        if (skip_step(args, t, dt)) continue;
        if (!mbar_wait(&empty[stage], phase ^ 1, args.err, kDevErrTimeoutProducer)) {
          ok = false;
          break;
        }
        uint8_t* a_dst = smem + stage * S::kStageBytes;
        uint8_t* b_dst = a_dst + kABytes;
        mbar_arrive_expect_tx(&full[stage], kABytes + S::kBBytes);
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        const int box_bytes = args.TH * args.TW * 128;
        for (int i = 0; i < args.TT; ++i) {
          const int tau = t.t0 + i + dt;
          if (tau < 0 && args.has_cache)
            tma_load_5d(a_dst + i * box_bytes, &tm_cache, &full[stage], kb * kBlockK, t.w0 + dw,
                        t.h0 + dh, tau + 2, t.n);
          else
            tma_load_5d(a_dst + i * box_bytes, &tm_a, &full[stage], kb * kBlockK, t.w0 + dw, t.h0 + dh,
                        tau, t.n);
        }
        tma_load_3d(b_dst, &tm_w, &full[stage], tap * args.Cin + kb * kBlockK, t.nb * BN, t.ph, w_policy);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // Drain: every load this thread issued has landed before the CTA may exit.
    for (int s = 0; s < STAGES; ++s)
      if (armed & (1u << s)) mbar_wait(&full[s], (armed_parity >> s) & 1, args.err, kDevErrTimeoutDrain);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kTileM, BN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
      const Tile t = decode_tile(args, tile);
      if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1, args.err, kDevErrTimeoutMma)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      bool first = true;
      for (int ks = 0; ks < num_k; ++ks) {
        const int tap = ks / args.kb_per_tap;
        int dt, dh, dw;
        tap_offsets(args, tap, t.ph, dt, dh, dw);
        if (skip_step(args, t, dt)) continue;
        if (!mbar_wait(&full[stage], phase, args.err, kDevErrTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + stage * S::kStageBytes);
        const uint64_t a_desc = smem_desc_sw128(a_addr);
        const uint64_t b_desc = smem_desc_sw128(a_addr + kABytes);
#pragma unroll
        for (int k = 0; k < kBlockK / 16; ++k)  // +32 bytes along K per step (encoded >> 4)
          mma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
        first = false;
        mma_commit(&empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      mma_commit(&tmem_full[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    // All MMAs of this thread complete before TMEM is released.
    mma_commit(mma_done);
    mbar_wait(mma_done, 0, args.err, kDevErrTimeoutDrain);
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const int Ho = args.mode == 0 ? args.H : 2 * args.H;
    const int Wo = args.mode == 0 ? args.W : 2 * args.W;
    const bool vec8 = (args.Cout % 8) == 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x) {
      const Tile t = decode_tile(args, tile);
      if (!mbar_wait(&tmem_full[acc], acc_phase, args.err, kDevErrTimeoutEpilogue)) break;
      tc_fence_after();
      const int per_frame = args.TH * args.TW;
      const int it = row / per_frame;
      const int ih = (row / args.TW) % args.TH;
      const int iw = row % args.TW;
      const int tt = t.t0 + it, hh = t.h0 + ih, ww = t.w0 + iw;
      const bool valid = tt < args.T && hh < args.H && ww < args.W;
      size_t pix;
      if (args.mode == 0)
        pix = (((size_t)t.n * args.T + tt) * Ho + hh) * Wo + ww;
      else
        pix = (((size_t)t.n * args.T + tt) * Ho + (2 * hh + (t.ph >> 1))) * Wo + (2 * ww + (t.ph & 1));
      wan_bf16* yrow = args.y + pix * args.Cout;
      const wan_bf16* rrow = args.residual ? args.residual + pix * args.Cout : nullptr;
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        __syncwarp();
        tmem_ld16(taddr + c0, v);
        const int col = t.nb * BN + c0;
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
      tc_fence_before();
      mbar_arrive(&tmem_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, S::kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
bool make_map_5d(CUtensorMap* m, const void* base, int C, int W, int H, int T, int N, int box_w,
                 int box_h) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[5] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)N};
  const cuuint64_t e = 2;
  const cuuint64_t strides[4] = {C * e, (cuuint64_t)W * C * e, (cuuint64_t)H * W * C * e,
                                 (cuuint64_t)T * H * W * C * e};
  const cuuint32_t box[5] = {(cuuint32_t)kBlockK, (cuuint32_t)box_w, (cuuint32_t)box_h, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_w(CUtensorMap* m, const void* base, int K, int Cout, int P, int BN) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)Cout, (cuuint64_t)P};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * Cout * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)BN, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Pixel-block shape of the 128-row M tile with the least padding for this frame size.
void choose_tile(int T, int H, int W, int& TT, int& TH, int& TW) {
  double best = 1e30;
  for (int tt = 1; tt <= 2; ++tt) {
    for (int tw = 8; tw <= 128; tw *= 2) {
      const int rows = kTileM / tt;
      if (rows % tw) continue;
      const int th = rows / tw;
      if (th < 1) continue;
      const double vol = (double)cdiv(T, tt) * tt * cdiv(H, th) * th * cdiv(W, tw) * tw;
      const double score = vol * (1.0 + 1e-3 * (tt - 1)) * (1.0 - 1e-6 * tw);
      if (score < best) {
        best = score;
        TT = tt;
        TH = th;
        TW = tw;
      }
    }
  }
}

template <int BN, int STAGES>
cudaError_t launch_bn(const CUtensorMap& ta, const CUtensorMap& tc, const CUtensorMap& tw, const ConvArgs& a,
                      int sms, cudaStream_t s) {
  using S = Smem<BN, STAGES>;
  const cudaError_t e = cudaFuncSetAttribute(conv_tc_kernel<BN, STAGES>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
  if (e != cudaSuccess) return e;
  const int grid = a.num_tiles < sms ? a.num_tiles : sms;
  conv_tc_kernel<BN, STAGES><<<grid, kThreads, S::kTotal, s>>>(ta, tc, tw, a);
  return cudaGetLastError();
}

int pick_bn(int Cout) {
  if (Cout > 128) return 256;
  if (Cout > 64) return 128;
  if (Cout > 32) return 64;
  if (Cout > 16) return 32;
  return 16;
}

}  // namespace

size_t conv_workspace() { return 0; }

cudaError_t conv_launch(int mode, const wan_bf16* a, const wan_bf16* cache_in, const wan_bf16* w,
                        const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T, int H,
                        int W, int Cin, int Cout, int sms, unsigned* err, cudaStream_t stream, void* st_buf,
                        int st_groups) {
  if (conv_pair_supported(Cout))
    return conv_pair_launch(mode, a, cache_in, w, bias, residual, y, N, T, H, W, Cin, Cout, sms, err, stream, st_buf,
                            st_groups);
  if (st_buf) return cudaErrorInvalidValue;  // output statistics come from the CTA-pair kernel only
  ConvArgs args{};
  args.N = N;
  args.T = T;
  args.H = H;
  args.W = W;
  args.Cin = Cin;
  args.Cout = Cout;
  choose_tile(T, H, W, args.TT, args.TH, args.TW);
  args.tiles_t = cdiv(T, args.TT);
  args.tiles_h = cdiv(H, args.TH);
  args.tiles_w = cdiv(W, args.TW);
  const int BN = pick_bn(Cout);
  args.n_blks = cdiv(Cout, BN);
  args.phases = mode == 0 ? 1 : 4;
  args.num_tiles = N * args.tiles_t * args.tiles_h * args.tiles_w * args.phases * args.n_blks;
  args.kb_per_tap = Cin / kBlockK;
  args.taps = mode == 0 ? 27 : 4;
  args.mode = mode;
  args.has_cache = cache_in != nullptr;
  args.bias = bias;
  args.residual = residual;
  args.y = y;
  args.err = err;

  CUtensorMap ta, tc, tw;
  if (!make_map_5d(&ta, a, Cin, W, H, T, N, args.TW, args.TH)) return cudaErrorInvalidValue;
  if (cache_in) {
    if (!make_map_5d(&tc, cache_in, Cin, W, H, 2, N, args.TW, args.TH)) return cudaErrorInvalidValue;
  } else {
    tc = ta;
  }
  if (!make_map_w(&tw, w, args.taps * Cin, Cout, args.phases, BN)) return cudaErrorInvalidValue;

  switch (BN) {
    case 256: return launch_bn<256, 4>(ta, tc, tw, args, sms, stream);
    case 128: return launch_bn<128, 6>(ta, tc, tw, args, sms, stream);
    case 64: return launch_bn<64, 8>(ta, tc, tw, args, sms, stream);
    case 32: return launch_bn<32, 8>(ta, tc, tw, args, sms, stream);
    default: return launch_bn<16, 8>(ta, tc, tw, args, sms, stream);
  }
}

// ---------------------------------------------------------------------------------------------
// Temporal cache update: cache_out[n, j] = P[n, T + j] for j = 0, 1, where P = [cache_in; a].
// ---------------------------------------------------------------------------------------------
__global__ void cache_frame_kernel(const wan_bf16* __restrict__ a, const wan_bf16* __restrict__ cache_in,
                                   wan_bf16* __restrict__ cache_out, int T, size_t frame_vecs, int j) {
  const int n = blockIdx.y;
  const int src = T + j;  // index into P
  const uint4* from;
  if (src >= 2)
    from = reinterpret_cast<const uint4*>(a) + ((size_t)n * T + (src - 2)) * frame_vecs;
  else
    from = cache_in ? reinterpret_cast<const uint4*>(cache_in) + ((size_t)n * 2 + src) * frame_vecs : nullptr;
  uint4* to = reinterpret_cast<uint4*>(cache_out) + ((size_t)n * 2 + j) * frame_vecs;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < frame_vecs; i += (size_t)gridDim.x * blockDim.x)
    to[i] = from ? from[i] : make_uint4(0, 0, 0, 0);
}

cudaError_t cache_update_launch(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out, int N, int T,
                                int H, int W, int C, int sms, cudaStream_t stream) {
  const size_t frame_vecs = (size_t)H * W * C / 8;
  int blocks = (int)((frame_vecs + 255) / 256);
  const int cap = 2 * sms;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  // Frame 0 first: when T == 1 and cache_out aliases cache_in, frame 0 reads cache_in[1],
  // which the frame-1 launch then overwrites.
  for (int j = 0; j < 2; ++j) {
    cache_frame_kernel<<<dim3(blocks, N), 256, 0, stream>>>(a, cache_in, cache_out, T, frame_vecs, j);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---------------------------------------------------------------------------------------------
// Phase weights of the nearest-x2 upsampler: fp32 sums of the source taps (r outer, c inner,
// starting from zero), rounded once to bf16.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ bool phase_src(int a, int u, int r) {
  const int dy = a + r - 1;
  const int iy = dy < 0 ? -1 : dy / 2;
  return iy == u + a - 1;
}

__global__ void phase_weights_kernel(const wan_bf16* __restrict__ w3, wan_bf16* __restrict__ wp, int Cin,
                                     int Cout) {
  const size_t per_phase = (size_t)Cout * 4 * Cin;
  const size_t total = 4 * per_phase;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int ci = (int)(i % Cin);
    size_t r_ = i / Cin;
    const int v = (int)(r_ % 2);
    r_ /= 2;
    const int u = (int)(r_ % 2);
    r_ /= 2;
    const int co = (int)(r_ % Cout);
    const int p = (int)(r_ / Cout);
    const int pa = p >> 1, pb = p & 1;
    float s = 0.0f;
    for (int r = 0; r < 3; ++r) {
      if (!phase_src(pa, u, r)) continue;
      for (int c = 0; c < 3; ++c) {
        if (!phase_src(pb, v, c)) continue;
        const uint32_t bits = w3[(((size_t)co * 3 + r) * 3 + c) * Cin + ci];
        s = __fadd_rn(s, __uint_as_float(bits << 16));
      }
    }
    uint16_t out;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(out) : "f"(s));
    wp[i] = out;
  }
}

// The same transform for Cin % 8 == 0, 8 channels per thread (16-byte loads and stores, 32-bit
// index arithmetic); the sums of each element run in the same order.
__global__ void phase_weights_vec_kernel(const wan_bf16* __restrict__ w3, wan_bf16* __restrict__ wp, int Cin,
                                         int Cout, int total_vec) {
  const int cv = Cin / 8;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total_vec; i += gridDim.x * blockDim.x) {
    const int c8 = i % cv;
    int r_ = i / cv;
    const int v = r_ & 1;
    r_ >>= 1;
    const int u = r_ & 1;
    r_ >>= 1;
    const int co = r_ % Cout;
    const int p = r_ / Cout;
    const int pa = p >> 1, pb = p & 1;
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < 3; ++r) {
      if (!phase_src(pa, u, r)) continue;
      for (int c = 0; c < 3; ++c) {
        if (!phase_src(pb, v, c)) continue;
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(w3 + (((size_t)co * 3 + r) * 3 + c) * Cin) + c8);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          s[2 * k] = __fadd_rn(s[2 * k], bf16lo_to_f32(qw[k]));
          s[2 * k + 1] = __fadd_rn(s[2 * k + 1], bf16hi_to_f32(qw[k]));
        }
      }
    }
    reinterpret_cast<uint4*>(wp)[i] =
        make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7]));
  }
}

cudaError_t phase_weights_launch(const wan_bf16* w3, wan_bf16* wp, int Cin, int Cout, int sms,
                                 cudaStream_t stream) {
  if (Cin % 8 == 0 && (long long)2 * Cout * Cin < (1LL << 31)) {
    const int total_vec = 2 * Cout * Cin;  // 16 Cout Cin / 8
    int blocks = cdiv(total_vec, 256);
    if (blocks > 8 * sms) blocks = 8 * sms;
    phase_weights_vec_kernel<<<blocks, 256, 0, stream>>>(w3, wp, Cin, Cout, total_vec);
    return cudaGetLastError();
  }
  const size_t total = (size_t)16 * Cout * Cin;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 8 * sms) blocks = 8 * sms;
  phase_weights_kernel<<<blocks, 256, 0, stream>>>(w3, wp, Cin, Cout);
  return cudaGetLastError();
}

// The channel-changing block's shortcut bias folded into the second conv's (binding.cpp,
// prepare()): out = b2 + b_shortcut rounded once to bf16. The sum of two bf16 values is exact in
// fp64; it reaches fp32 rounded to odd (truncate, then set the last bit if anything was lost),
// from which round-to-nearest-even to bf16 gives the correctly rounded result (Boldo and
// Melquiond's round-to-odd: 24 bits >= 8 + 2).
__global__ void fold_bias_kernel(const wan_bf16* __restrict__ b2, const wan_bf16* __restrict__ bsc,
                                 wan_bf16* __restrict__ out, int C) {
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < C; c += gridDim.x * blockDim.x) {
    const double v = (double)__uint_as_float(((uint32_t)b2[c]) << 16) + (double)__uint_as_float(((uint32_t)bsc[c]) << 16);
    float r = __double2float_rz(v);
    if ((double)r != v) r = __uint_as_float(__float_as_uint(r) | 1u);
    out[c] = (wan_bf16)(pack_bf16x2(r, 0.f) & 0xFFFFu);
  }
}

cudaError_t fold_bias_launch(const wan_bf16* b2, const wan_bf16* bsc, wan_bf16* out, int C, cudaStream_t stream) {
  fold_bias_kernel<<<cdiv(C, 256), 256, 0, stream>>>(b2, bsc, out, C);
  return cudaGetLastError();
}

}  // namespace wan
