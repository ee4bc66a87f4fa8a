// The causal 3x3x3 convolution with its spatial taps through Winograd F(2x2, 3x3), fp16 operands.
//
// Source: FastVideo, binding.cpp: `prepare()` (the Winograd weights G g G^T of the up blocks, each
// of the components keeping the causal 3-tap temporal convolution; fp32 sums), `Decoder::conv`
// (only the spatial 3x3 convolutions use Winograd: the padded input is transformed once, every
// component is a convolution of its own, and an epilogue applies the output transform with bias
// and residual). The transforms are Lavin and Gray's ("Fast Algorithms for Convolutional Neural
// Networks", 2016): for a 2x2 output tile, its 4x4 input tile d and the 3x3 kernel g,
//     Y = A^T [ (G g G^T) . (B^T d B) ] A.
// The pages use F(4x4, 3x3) with bf16 operands; that misses the direct conv's accuracy by 15x, and
// F(4x4) with fp16 operands by about 2x, while F(2x2) with fp16 operands has the direct conv's
// error (relative L2 within 5%): the variant built here. A component's products are the 3 temporal
// taps x Cin channels of a GEMM, 16 components per 2x2 outputs against 36 products of the direct
// conv (0.44 of its tensor work), paid for by moving the transformed input (4x the input, fp16) and
// the component products (16 fp32 per 2x2 outputs) through HBM, which pays where the channels are
// many (Cin = Cout = 1024 at 44 x 78).
//
// Three kernels on the caller's stream:
//   wino_input_kernel   V[xy][n, tau, tile][ci] = fp16(B^T d B) for every frame tau of the padded
//                       input P = [cache (2 frames, or zeros); silu(x S + B) or x] and tile; the
//                       GroupNorm + SiLU is the one every other path uses (gn_silu8), so the frames
//                       a chunk hands on in its cache are the bits this kernel used.
//   wino_gemm_kernel    per component xy (tcgen05 kind::f16 on CTA pairs, M256 x N256 x K16):
//                       M[xy][n, t, tile][co] = sum_{kt, ci} U[xy][co][kt, ci] V[xy][n, t + kt, tile][ci]
//                       in fp32; the temporal tap kt is a row offset of kt * tiles into V.
//   wino_output_kernel  Y = A^T M A (+ bias + residual), rounded once to bf16.
// Every sum runs in a fixed order that depends on neither the tile nor the chunking of the frames,
// so chunked and unchunked calls give the same bits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "conv_tc.h"
#include "tma_host.h"
#include "winograd.h"

namespace wan {

namespace {

constexpr int kWK = 64;                   // K per stage: 64 fp16 = one 128-byte swizzled row
constexpr int kWStages = 6;               // (A + B) stages per CTA; MMA bursts of 3 never wrap
constexpr int kWA = 128 * 128;            // this CTA's 128 rows of V x 64 channels
constexpr int kWB = 128 * 128;            // this CTA's 128 of the 256 weight rows x 64 channels
constexpr int kWStage = kWA + kWB;
constexpr int kWBarOff = kWStages * kWStage;
constexpr int kWSmem = kWBarOff + 256 + 1024;
constexpr int kWThreads = 192;            // producer, MMA issuer, 4 epilogue warps
constexpr int kWN = 256;                  // output channels per item
constexpr int kWBurst = 3;                // stages per straight-line MMA burst
static_assert(kWStages % kWBurst == 0 && kWStage % 1024 == 0, "bursts never wrap; 1024-byte stages");
static_assert(kWSmem <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Instruction descriptor of kind::f16 with fp16 A and B (K-major), fp32 D, shape M x N (the bf16
// descriptor with the A and B formats 0 = f16).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------------------------------------
// Weight transform: one thread per (component xy, co, kt, 8 input channels).
// ------------------------------------------------------------------------------------------------
__global__ void wino_weights_kernel(const wan_bf16* __restrict__ w, uint16_t* __restrict__ u, int Cin, int Cout,
                                    long long total) {
  // G = [[1, 0, 0], [1/2, 1/2, 1/2], [1/2, -1/2, 1/2], [0, 0, 1]]
  const float G[4][3] = {{1.f, 0.f, 0.f}, {0.5f, 0.5f, 0.5f}, {0.5f, -0.5f, 0.5f}, {0.f, 0.f, 1.f}};
  const int cv = Cin / 8;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    long long r = idx;
    const int v = (int)(r % cv);
    r /= cv;
    const int kt = (int)(r % 3);
    r /= 3;
    const int co = (int)(r % Cout);
    const int xy = (int)(r / Cout);
    const int x = xy >> 2, y = xy & 3;
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // sum over the spatial taps with a non-zero coefficient, rows outer, columns inner, from zero
    for (int rr = 0; rr < 3; ++rr)
      for (int cc = 0; cc < 3; ++cc) {
        const float k = G[x][rr] * G[y][cc];
        if (k == 0.f) continue;
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(
            w + ((((size_t)co * 3 + kt) * 3 + rr) * 3 + cc) * Cin + (size_t)v * 8));
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // k * w is exact (k is 1, 1/2 or 1/4 with a sign)
          s[2 * i] = __fadd_rn(s[2 * i], __fmul_rn(k, bf16lo_to_f32(qw[i])));
          s[2 * i + 1] = __fadd_rn(s[2 * i + 1], __fmul_rn(k, bf16hi_to_f32(qw[i])));
        }
      }
    const uint4 o = make_uint4(pack_f16x2(s[0], s[1]), pack_f16x2(s[2], s[3]), pack_f16x2(s[4], s[5]),
                               pack_f16x2(s[6], s[7]));
    *reinterpret_cast<uint4*>(u + (((size_t)xy * Cout + co) * 3 + kt) * Cin + (size_t)v * 8) = o;
  }
}

// ------------------------------------------------------------------------------------------------
// Input transform. A CTA takes a block of kInTileRows x kInTileCols tiles of one frame and 64
// channels: it stages the pixels they read (their rows and columns plus one halo row and column on
// each side, zeros outside the frame) in shared memory, each pixel loaded and normalised once, then
// transforms the tiles from there with 4 channels per thread.
// ------------------------------------------------------------------------------------------------
constexpr int kInTileRows = 4;
constexpr int kInTileCols = 40;
constexpr int kInRows = 2 * kInTileRows + 2;  // pixel rows staged per CTA
constexpr int kInCols = 2 * kInTileCols + 2;  // pixel columns staged per CTA (at most)
constexpr int kInThreads = 256;
constexpr int kInLoads = 4;  // 16-byte loads in flight per thread while staging

struct WinoInArgs {
  const wan_bf16* x;       // [N, T, H, W, C]
  const float4* coef;      // blocked GroupNorm coefficients per (n T + t, c), or null
  const wan_bf16* cache;   // [N, 2, H, W, C] or null (zeros)
  uint16_t* v;             // [16][N (T + 2) tiles][C] fp16
  wan_bf16* cache_out;     // [N, 2, H, W, C] or null: the new history, from the staged pixels
  int N, T, H, W, C, Ht, Wt, tiles, col_groups;
  long long rows;          // N (T + 2) tiles
};

__global__ void __launch_bounds__(kInThreads) wino_input_kernel(const WinoInArgs a) {
  extern __shared__ __align__(16) uint8_t sm_in[];  // [kInRows][cols][64 channels] bf16
  const int slice = blockIdx.x;                     // 64 channels
  const int i0 = (blockIdx.y / a.col_groups) * kInTileRows;  // first tile row
  const int j0 = (blockIdx.y % a.col_groups) * kInTileCols;  // first tile column
  const int ncols = min(kInTileCols, a.Wt - j0);
  const int cols = 2 * ncols + 2;                   // staged pixel columns
  const int nrows = min(kInTileRows, a.Ht - i0);
  const int ft = blockIdx.z;                        // n (T + 2) + tau
  const int tau = ft % (a.T + 2), n = ft / (a.T + 2);
  const wan_bf16* src = nullptr;
  const float4* cf = nullptr;
  // frames T - 2 and T - 1 of the input are the new history: each CTA stores the pixels of its own
  // tiles (not the halo) of its 64 channels
  const bool wcache = a.cache_out && tau >= 2 && tau - 2 >= a.T - 2;
  wan_bf16* cdst = wcache ? a.cache_out + ((size_t)n * 2 + (tau - a.T)) * a.H * a.W * a.C + slice * 64 : nullptr;
  if (tau < 2) {
    if (a.cache) src = a.cache + ((size_t)n * 2 + tau) * a.H * a.W * a.C;
  } else {
    const int f = n * a.T + tau - 2;
    src = a.x + (size_t)f * a.H * a.W * a.C;
    if (a.coef) cf = a.coef + (size_t)f * a.C + slice * 64;
  }
  // 1. pixel rows 2 i0 - 1 .. 2 i0 + 2 kInTileRows, columns 2 j0 - 1 .. 2 (j0 + ncols): 8 threads
  // per pixel.
  {
    const int v = threadIdx.x & 7;
    GnCoef8 k8;
    if (cf) k8 = gn_coef8_blocked(cf + v);  // the blocked layout: channels 8 v .. 8 v + 7 of the slice
    const int npx = kInRows * cols;
    constexpr int kStride = kInThreads / 8;
    for (int p0 = threadIdx.x >> 3; p0 < npx; p0 += kStride * kInLoads) {
      uint4 q[kInLoads];
      bool in[kInLoads];
#pragma unroll
      for (int u = 0; u < kInLoads; ++u) {  // kInLoads loads in flight before any is used
        const int p = p0 + u * kStride;
        const int r = p / cols, c = p - r * cols;
        const int hh = 2 * i0 - 1 + r, ww = 2 * j0 - 1 + c;
        in[u] = p < npx && src && hh >= 0 && hh < a.H && ww >= 0 && ww < a.W;
        q[u] = in[u] ? __ldg(reinterpret_cast<const uint4*>(src + ((size_t)hh * a.W + ww) * a.C + slice * 64) + v)
                     : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kInLoads; ++u) {
        const int p = p0 + u * kStride;
        if (cf && in[u]) q[u] = gn_silu8(q[u], k8);
        if (p < npx) *reinterpret_cast<uint4*>(sm_in + (size_t)p * 128 + v * 16) = q[u];
        if (wcache && in[u]) {
          const int r = p / cols, c = p - r * cols;
          if (r >= 1 && r <= 2 * nrows && c >= 1 && c <= 2 * ncols)
            *reinterpret_cast<uint4*>(cdst + ((size_t)(2 * i0 - 1 + r) * a.W + (2 * j0 - 1 + c)) * a.C + v * 8) = q[u];
        }
      }
    }
  }
  __syncthreads();
  // 2. V = B^T d B per channel, B^T = [[1, 0, -1, 0], [0, 1, 1, 0], [0, -1, 1, 0], [0, 1, 0, -1]]:
  // rows first (s = B^T d), then columns (V = s B), in fp32, rounded once to fp16.
  const int work = nrows * ncols * 16;
  for (int idx = threadIdx.x; idx < work; idx += kInThreads) {
    const int q = idx & 15;  // channels 4 q .. 4 q + 3 of the slice
    const int t = idx >> 4;
    const int il = t / ncols, tj = t - il * ncols;  // tile (i0 + il, j0 + tj)
    float2 e[4][4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint2 wv = *reinterpret_cast<const uint2*>(sm_in + ((size_t)(2 * il + r) * cols + 2 * tj + c) * 128 +
                                                         q * 8);
        e[r][c][0] = unpack2(wv.x);
        e[r][c][1] = unpack2(wv.y);
      }
    // Two channels per packed fp32x2 operation (sub2 = an FMA by -1: the same rounding as a - b).
    uint32_t out[16][2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      float2 sr[4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        sr[0][c] = sub2(e[0][c][w], e[2][c][w]);
        sr[1][c] = __fadd2_rn(e[1][c][w], e[2][c][w]);
        sr[2][c] = sub2(e[2][c][w], e[1][c][w]);
        sr[3][c] = sub2(e[1][c][w], e[3][c][w]);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float2 o0 = sub2(sr[x][0], sr[x][2]), o1 = __fadd2_rn(sr[x][1], sr[x][2]);
        const float2 o2 = sub2(sr[x][2], sr[x][1]), o3 = sub2(sr[x][1], sr[x][3]);
        out[4 * x + 0][w] = pack_f16x2(o0.x, o0.y);
        out[4 * x + 1][w] = pack_f16x2(o1.x, o1.y);
        out[4 * x + 2][w] = pack_f16x2(o2.x, o2.y);
        out[4 * x + 3][w] = pack_f16x2(o3.x, o3.y);
      }
    }
    const size_t row = (size_t)ft * a.tiles + (size_t)(i0 + il) * a.Wt + j0 + tj;
#pragma unroll
    for (int xy = 0; xy < 16; ++xy)
      *reinterpret_cast<uint2*>(a.v + ((size_t)xy * a.rows + row) * a.C + slice * 64 + q * 4) =
          make_uint2(out[xy][0], out[xy][1]);
  }
}

// ------------------------------------------------------------------------------------------------
// Component GEMMs on CTA pairs.
// ------------------------------------------------------------------------------------------------
struct WinoGemmArgs {
  int tiles;           // 2x2 output tiles per frame
  int rows_in_per_n;   // rows of V per batch item: (T + 2) tiles
  int rows_out_per_n;  // output rows per batch item: T tiles
  int mpairs_per_n;    // pair tiles (256 rows) per batch item
  int n_mpairs, n_blks, items, kb, Cin, Cout;
  long long mrows;     // N T tiles: rows of one component of M
  float* mbuf;         // [16][mrows][Cout] fp32
  unsigned* err;
};

struct WItem {
  int xy, nb, n, mloc;  // component, N block, batch item, first local output row of the pair tile
};

// item -> (component, pair tile, N block), N block fastest: pairs that run together share the rows
// of V they read, and a component's weights stay in L2 while its items run.
__device__ __forceinline__ WItem wdecode(const WinoGemmArgs& a, int item) {
  WItem w;
  w.nb = item % a.n_blks;
  item /= a.n_blks;
  const int mp = item % a.n_mpairs;
  w.xy = item / a.n_mpairs;
  w.n = mp / a.mpairs_per_n;
  w.mloc = (mp % a.mpairs_per_n) * 256;
  return w;
}

// The MMAs of kWBurst consecutive stages in straight-line code, each stage's wait and release in
// place (a barrier wait per stage inside a run-time loop costs the tensor pipe issue cycles).
__device__ __forceinline__ bool wino_burst(uint32_t d_tmem, uint32_t stage0, uint64_t* full, uint64_t* empty,
                                           uint32_t ph, uint32_t idesc, bool first, unsigned* err) {
#pragma unroll
  for (int j = 0; j < kWBurst; ++j) {
    if (!mbar_wait_cluster(&full[j], ph, err, kDevErrTimeoutMma)) return false;
    tc_fence_after();
    const uint64_t ad = smem_desc_sw128(stage0 + j * kWStage), bd = smem_desc_sw128(stage0 + j * kWStage + kWA);
#pragma unroll
    for (int k = 0; k < kWK / 16; ++k)
      mma_bf16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (first && j == 0 && k == 0) ? 0u : 1u);
    mma_commit_pair(&empty[j], 0x3);
  }
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kWThreads, 1)
    wino_gemm_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_u,
                     const WinoGemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWBarOff);
  uint64_t* empty = full + kWStages;
  uint64_t* tmem_full = empty + kWStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* mma_done = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int stages_per_item = 3 * args.kb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(mma_done, 1);
    fence_mbarrier_init();
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_u);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);  // two accumulators of 256 columns
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    const uint64_t policy = l2_policy_evict_last();
    int s = 0;
    uint32_t ph = 0, armed = 0, parity = 0;
    bool ok = true;
    for (int item = cluster; ok && item < args.items; item += nclusters) {
      const WItem it = wdecode(args, item);
      const int arow = it.n * args.rows_in_per_n + it.mloc + (int)rank * 128;
      const int brow = it.nb * kWN + (int)rank * 128;
      for (int kt = 0; ok && kt < 3; ++kt) {
        for (int kb = 0; kb < args.kb; ++kb) {
          if (!mbar_wait_cluster(&empty[s], ph ^ 1, args.err, kDevErrTimeoutProducer)) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(&full[s], 2 * kWStage);  // both CTAs' A and B land on it
            armed |= 1u << s;
            parity = (parity & ~(1u << s)) | (ph << s);
          }
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
          uint8_t* dst = smem + s * kWStage;
          tma_load_3d_pair(dst, &tm_v, bar, kb * kWK, arow + kt * args.tiles, it.xy, policy);
          tma_load_3d_pair(dst + kWA, &tm_u, bar, kt * args.Cin + kb * kWK, brow, it.xy, policy);
          if (++s == kWStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
    }
    for (int q = 0; q < kWStages; ++q)
      if (armed & (1u << q)) mbar_wait(&full[q], (parity >> q) & 1, args.err, kDevErrTimeoutDrain);
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_f16_f32(256, kWN);
    const uint32_t base = smem_u32(smem);
    int s = 0, acc = 0;
    uint32_t ph = 0, acc_phase = 0;
    bool ok = true;
    for (int item = cluster; ok && item < args.items; item += nclusters) {
      if (!mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1, args.err, kDevErrTimeoutMma)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kWN;
      for (int g = 0; ok && g < stages_per_item; g += kWBurst) {
        ok = wino_burst(d_tmem, base + s * kWStage, full + s, empty + s, ph, idesc, g == 0, args.err);
        if ((s += kWBurst) == kWStages) {
          s = 0;
          ph ^= 1;
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
    const uint32_t leader_empty0 = mapa_shared(smem_u32(&tmem_empty[0]), 0);
    const uint32_t leader_empty1 = mapa_shared(smem_u32(&tmem_empty[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int item = cluster; item < args.items; item += nclusters) {
      const WItem it = wdecode(args, item);
      if (!mbar_wait_cluster(&tmem_full[acc], acc_phase, args.err, kDevErrTimeoutEpilogue)) break;
      tc_fence_after();
      const int mloc = it.mloc + (int)rank * 128 + row;
      const bool valid = mloc < args.rows_out_per_n;
      float* dst = args.mbuf + ((size_t)it.xy * args.mrows + (size_t)it.n * args.rows_out_per_n + mloc) * args.Cout +
                   (size_t)it.nb * kWN;
      const uint32_t taddr = tmem_base + (uint32_t)(acc * kWN) + ((uint32_t)(quarter * 32) << 16);
      uint32_t rn[16];
      __syncwarp();
      tmem_ld16_issue(taddr, rn);
      tmem_ld16_wait(rn);
#pragma unroll 1
      for (int c0 = 0; c0 < kWN; c0 += 16) {
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = rn[i];
        if (c0 + 16 < kWN) {
          __syncwarp();
          tmem_ld16_issue(taddr + c0 + 16, rn);
        }
        if (valid) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<uint4*>(dst + c0 + i) = make_uint4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
        if (c0 + 16 < kWN) tmem_ld16_wait(rn);
      }
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
  if (warp == 1) tmem_dealloc_pair(tmem_base, 512);
}

// ------------------------------------------------------------------------------------------------
// Output transform: one thread per (n, t, tile, 4 output channels).
// ------------------------------------------------------------------------------------------------
struct WinoOutArgs {
  const float* mbuf;        // [16][mrows][Cout]
  const wan_bf16* bias;     // [Cout] or null
  const wan_bf16* residual; // [N, T, H, W, Cout] or null
  wan_bf16* y;
  int H, W, Cout, Wt, tiles;
  long long mrows, total;   // mrows = N T tiles; total = mrows Cout / 4
  // GroupNorm statistics of y (optional): per (frame, group, tile) the float-float sums of d and
  // d^2 of d = y - s over the tile's pixels and the group's 2^st_lg channels (st_rec), and (s,
  // count) (st_meta), s the group's first channel at the tile's first pixel; st_hdr receives the
  // records per (frame, group), the tile count.
  float4* st_rec;
  float2* st_meta;
  int* st_hdr;
  int st_lg, st_groups;
};

// kStats: the launch writes the GroupNorm statistics of y (a.st_rec set). The plain instance fits
// three CTAs per SM in 80 registers; the statistics instance takes two, in 115 registers: held to
// 80 it spilled 150 bytes a thread and ran 12 us slower at [1, 4, 44, 78, 1024], against 1.5 us
// for the lower occupancy.
template <bool kStats>
__global__ void __launch_bounds__(256, kStats ? 2 : 3) wino_output_kernel(const WinoOutArgs a) {
  const int cq = a.Cout / 4;
  const int lane = threadIdx.x & 31;
  if (kStats && blockIdx.x == 0 && threadIdx.x == 0) *a.st_hdr = a.tiles;
  // A warp's 32 threads take 32 consecutive channel quads of one tile (cq is a multiple of 32 and
  // so is every index the loop visits), so a group's quads are neighbouring lanes of one warp.
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < a.total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int q = (int)(idx % cq);
    const long long m = idx / cq;  // (n T + t) tiles + tile
    const int tile = (int)(m % a.tiles);
    const long long f = m / a.tiles;
    const int ti = tile / a.Wt, tj = tile - ti * a.Wt;
    float4 M[16];
#pragma unroll
    for (int xy = 0; xy < 16; ++xy)
      M[xy] = __ldcs(reinterpret_cast<const float4*>(a.mbuf + ((size_t)xy * a.mrows + m) * a.Cout) + q);
    // the residual of the tile's 4 pixels, loaded with the products rather than after them
    uint2 res[2][2];
#pragma unroll
    for (int pa = 0; pa < 2; ++pa)
#pragma unroll
      for (int pb = 0; pb < 2; ++pb) {
        const int hh = 2 * ti + pa, ww = 2 * tj + pb;
        res[pa][pb] = (a.residual && hh < a.H && ww < a.W)
                          ? *reinterpret_cast<const uint2*>(a.residual + (((size_t)f * a.H + hh) * a.W + ww) * a.Cout +
                                                            (size_t)q * 4)
                          : make_uint2(0u, 0u);
      }
    // A^T = [[1, 1, 1, 0], [0, 1, -1, -1]]: z = A^T M (rows), then Y = z A (columns).
    float4 z[2][4];
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const float4 m0 = M[y], m1 = M[4 + y], m2 = M[8 + y], m3 = M[12 + y];
      z[0][y] = make_float4((m0.x + m1.x) + m2.x, (m0.y + m1.y) + m2.y, (m0.z + m1.z) + m2.z, (m0.w + m1.w) + m2.w);
      z[1][y] = make_float4((m1.x - m2.x) - m3.x, (m1.y - m2.y) - m3.y, (m1.z - m2.z) - m3.z, (m1.w - m2.w) - m3.w);
    }
    float bv[4] = {0.f, 0.f, 0.f, 0.f};
    if (a.bias) {
      const uint2 b = __ldg(reinterpret_cast<const uint2*>(a.bias) + q);
      bv[0] = bf16lo_to_f32(b.x);
      bv[1] = bf16hi_to_f32(b.x);
      bv[2] = bf16lo_to_f32(b.y);
      bv[3] = bf16hi_to_f32(b.y);
    }
    // GroupNorm statistics of the stored values (kStats): each lane sums d and d^2 over its 4
    // channels of the tile's pixels in fp32 as it stores them (a sum of at most 16 deviations of
    // bf16 values, exact unless they lie about 12 binades apart); sh is the group's first channel
    // at the tile's first pixel, which every tile has.
    const int lpg = kStats ? (1 << a.st_lg) >> 2 : 1;  // lanes per group
    const int first = lane & ~(lpg - 1);
    float sh = 0.f, s1 = 0.f, s2 = 0.f;
    int npx = 0;
#pragma unroll
    for (int pa = 0; pa < 2; ++pa) {
      const int hh = 2 * ti + pa;
      if (hh >= a.H) continue;
#pragma unroll
      for (int pb = 0; pb < 2; ++pb) {
        const int ww = 2 * tj + pb;
        if (ww >= a.W) continue;
        const float4 z0 = z[pa][0], z1 = z[pa][1], z2 = z[pa][2], z3 = z[pa][3];
        float v[4];
        if (pb == 0) {
          v[0] = (z0.x + z1.x) + z2.x;
          v[1] = (z0.y + z1.y) + z2.y;
          v[2] = (z0.z + z1.z) + z2.z;
          v[3] = (z0.w + z1.w) + z2.w;
        } else {
          v[0] = (z1.x - z2.x) - z3.x;
          v[1] = (z1.y - z2.y) - z3.y;
          v[2] = (z1.z - z2.z) - z3.z;
          v[3] = (z1.w - z2.w) - z3.w;
        }
        const size_t px = ((size_t)f * a.H + hh) * a.W + ww;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] += bv[i];
        if (a.residual) {
          const uint2 r = res[pa][pb];
          v[0] += bf16lo_to_f32(r.x);
          v[1] += bf16hi_to_f32(r.x);
          v[2] += bf16lo_to_f32(r.y);
          v[3] += bf16hi_to_f32(r.y);
        }
        const uint2 o = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        *reinterpret_cast<uint2*>(a.y + px * a.Cout + (size_t)q * 4) = o;
        if (kStats) {
          if (pa == 0 && pb == 0) sh = __shfl_sync(0xffffffffu, bf16lo_to_f32(o.x), first);
          ++npx;
          const float d[4] = {bf16lo_to_f32(o.x) - sh, bf16hi_to_f32(o.x) - sh, bf16lo_to_f32(o.y) - sh,
                              bf16hi_to_f32(o.y) - sh};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            s1 += d[k];
            s2 = fmaf(d[k], d[k], s2);
          }
        }
      }
    }
    if (kStats) {
      // The group's lanes add their sums as float-float pairs in a fixed butterfly order; the
      // group's first lane writes the record.
      float h1 = s1, l1 = 0.f, h2 = s2, l2 = 0.f;
      for (int off = 1; off < lpg; off <<= 1) {
        const float oh1 = __shfl_xor_sync(0xffffffffu, h1, off), ol1 = __shfl_xor_sync(0xffffffffu, l1, off);
        const float oh2 = __shfl_xor_sync(0xffffffffu, h2, off), ol2 = __shfl_xor_sync(0xffffffffu, l2, off);
        ff_add(h1, l1, oh1, ol1);
        ff_add(h2, l2, oh2, ol2);
      }
      if (lane == first) {
        const int g = (4 * q) >> a.st_lg;
        const size_t rec = ((size_t)f * a.st_groups + g) * a.tiles + tile;
        __stcg(a.st_rec + rec, make_float4(h1, l1, h2, l2));
        __stcg(a.st_meta + rec, make_float2(sh, (float)(npx << a.st_lg)));
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
// A [P][rows][K] fp16 tensor addressed as (k, row, p); a box is 64 K x 128 rows, 128-byte swizzle.
bool map_f16_3d(CUtensorMap* m, const void* base, long long K, long long rows, int P) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)P};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)(K * rows * 2)};
  const cuuint32_t box[3] = {(cuuint32_t)kWK, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t a256(size_t b) { return (b + 255) & ~(size_t)255; }

struct WinoPlan {
  int Ht, Wt, tiles;
  long long rows_in, mrows;
  size_t v_bytes, m_bytes;
};

WinoPlan wplan(int N, int T, int H, int W, int Cin, int Cout) {
  WinoPlan p;
  p.Ht = (H + 1) / 2;
  p.Wt = (W + 1) / 2;
  p.tiles = p.Ht * p.Wt;
  p.rows_in = (long long)N * (T + 2) * p.tiles;
  p.mrows = (long long)N * T * p.tiles;
  p.v_bytes = a256((size_t)16 * p.rows_in * Cin * 2);
  p.m_bytes = a256((size_t)16 * p.mrows * Cout * 4);
  return p;
}

int grid_for(long long work, int sms, int per_sm) {
  const long long g = (work + 255) / 256;
  return (int)(g < (long long)sms * per_sm ? (g > 0 ? g : 1) : (long long)sms * per_sm);
}

}  // namespace

bool wino_supported(int Cin, int Cout) { return Cin > 0 && Cout > 0 && Cin % 64 == 0 && Cout % kWN == 0; }

bool wino_gn_stats_supported(int Cout, int groups) {
  if (groups <= 0 || Cout <= 0 || Cout % kWN != 0 || Cout % groups != 0) return false;
  const int cg = Cout / groups;  // a group's quads are 1 .. 16 neighbouring lanes of a warp
  return cg >= 4 && cg <= 64 && (cg & (cg - 1)) == 0;
}

int wino_gn_stats_records(int H, int W) { return ((H + 1) / 2) * ((W + 1) / 2); }

size_t wino_gn_stats_bytes(int N, int T, int H, int W, int groups) {
  return kGnStatsHeader + (size_t)N * T * groups * wino_gn_stats_records(H, W) * (sizeof(float4) + sizeof(float2));
}

size_t wino_workspace(int N, int T, int H, int W, int Cin, int Cout) {
  const WinoPlan p = wplan(N, T, H, W, Cin, Cout);
  return p.v_bytes + p.m_bytes;
}

cudaError_t wino_weights_launch(const wan_bf16* w, uint16_t* u, int Cin, int Cout, int sms, cudaStream_t s) {
  if (Cin % 8 != 0) return cudaErrorInvalidValue;
  const long long total = (long long)16 * Cout * 3 * (Cin / 8);
  wino_weights_kernel<<<grid_for(total, sms, 8), 256, 0, s>>>(w, u, Cin, Cout, total);
  return cudaGetLastError();
}

cudaError_t wino_conv_launch(const wan_bf16* a, const float4* coef, const wan_bf16* cache_in, const uint16_t* u,
                             const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                             int Cin, int Cout, void* ws, int sms, unsigned* err, cudaStream_t s,
                             wan_bf16* cache_out, void* st_buf, int st_groups) {
  if (!wino_supported(Cin, Cout) || (cache_out && cache_out == cache_in)) return cudaErrorInvalidValue;
  if (st_buf && !wino_gn_stats_supported(Cout, st_groups)) return cudaErrorInvalidValue;
  const WinoPlan p = wplan(N, T, H, W, Cin, Cout);
  uint16_t* v = static_cast<uint16_t*>(ws);
  float* mbuf = reinterpret_cast<float*>(static_cast<char*>(ws) + p.v_bytes);

  WinoInArgs ia;
  ia.x = a;
  ia.coef = coef;
  ia.cache = cache_in;
  ia.v = v;
  ia.cache_out = cache_out;
  ia.N = N;
  ia.T = T;
  ia.H = H;
  ia.W = W;
  ia.C = Cin;
  ia.Ht = p.Ht;
  ia.Wt = p.Wt;
  ia.tiles = p.tiles;
  ia.col_groups = cdiv(p.Wt, kInTileCols);
  ia.rows = p.rows_in;
  const size_t in_smem = (size_t)kInRows * std::min(kInCols, 2 * p.Wt + 2) * 128;
  const long long ygrid = (long long)cdiv(p.Ht, kInTileRows) * ia.col_groups;
  if ((long long)N * (T + 2) > 65535 || ygrid > 65535) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(wino_input_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)in_smem);
  if (e != cudaSuccess) return e;
  wino_input_kernel<<<dim3(Cin / 64, (unsigned)ygrid, N * (T + 2)), kInThreads, in_smem, s>>>(ia);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  WinoGemmArgs ga;
  ga.tiles = p.tiles;
  ga.rows_in_per_n = (T + 2) * p.tiles;
  ga.rows_out_per_n = T * p.tiles;
  ga.mpairs_per_n = cdiv(ga.rows_out_per_n, 256);
  ga.n_mpairs = N * ga.mpairs_per_n;
  ga.n_blks = Cout / kWN;
  ga.items = 16 * ga.n_mpairs * ga.n_blks;
  ga.kb = Cin / kWK;
  ga.Cin = Cin;
  ga.Cout = Cout;
  ga.mrows = p.mrows;
  ga.mbuf = mbuf;
  ga.err = err;
  CUtensorMap tv, tu;
  if (!map_f16_3d(&tv, v, Cin, p.rows_in, 16)) return cudaErrorInvalidValue;
  if (!map_f16_3d(&tu, u, 3LL * Cin, Cout, 16)) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(wino_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
  if (e != cudaSuccess) return e;
  int clusters = resident_pairs(reinterpret_cast<const void*>(wino_gemm_kernel), kWThreads, kWSmem, sms);
  if (clusters > ga.items) clusters = ga.items;
  if (clusters < 1) clusters = 1;
  wino_gemm_kernel<<<2 * clusters, kWThreads, kWSmem, s>>>(tv, tu, ga);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  WinoOutArgs oa;
  oa.mbuf = mbuf;
  oa.bias = bias;
  oa.residual = residual;
  oa.y = y;
  oa.H = H;
  oa.W = W;
  oa.Cout = Cout;
  oa.Wt = p.Wt;
  oa.tiles = p.tiles;
  oa.mrows = p.mrows;
  oa.total = p.mrows * (Cout / 4);
  oa.st_rec = nullptr;
  oa.st_meta = nullptr;
  oa.st_hdr = nullptr;
  oa.st_lg = 0;
  oa.st_groups = 0;
  if (st_buf) {
    oa.st_hdr = static_cast<int*>(st_buf);
    oa.st_rec = reinterpret_cast<float4*>(static_cast<char*>(st_buf) + kGnStatsHeader);
    oa.st_meta = reinterpret_cast<float2*>(oa.st_rec + (size_t)N * T * st_groups * p.tiles);
    oa.st_groups = st_groups;
    while ((1 << oa.st_lg) < Cout / st_groups) ++oa.st_lg;
  }
  if (st_buf)
    wino_output_kernel<true><<<grid_for(oa.total, sms, 8), 256, 0, s>>>(oa);
  else
    wino_output_kernel<false><<<grid_for(oa.total, sms, 8), 256, 0, s>>>(oa);
  return cudaGetLastError();
}

}  // namespace wan
