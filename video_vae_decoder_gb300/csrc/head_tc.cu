// Causal 3x3x3 convolution to 12 output channels (the decoder's output head), on tcgen05.
//
// Source of the idea: FastVideo wan22_vae_decode/solution/binding.cpp, `prepare()` (the head's
// nine spatial taps become output channels of a temporal-only convolution:
// W'[(i*3+j)*12 + c, ci, kt] = W[c, ci, kt, i, j], padded from 108 to 112 rows) and
// `Decoder::output_head` (a stencil then sums the nine shifted copies). A 12-column GEMM would
// leave almost all of a tensor-core tile idle; the transform gives it 112 columns.
//
// GB300 design (one kernel, no intermediate tensor):
//   * GEMM per (image row r, output frame t): G[p, n] = sum_{kt, ci} W'[n, kt*Cin + ci]
//     * x[t + kt - 2, r, p, ci] for the 128 pixels p of a column strip. W' (112 x 3*Cin bf16,
//     168 KB at Cin = 256) is built once per CTA straight into shared memory in the 128-byte
//     swizzled K-major layout and stays resident; only x streams through a 3-stage TMA ring.
//   * Each CTA owns (batch item, pair of output frames t and t+1, 128-pixel column strip, band
//     of image rows) and walks the rows of its band. A pair shares the input frames t-1 and t,
//     so 4 input rows feed 2 output rows; the two accumulators (2 x 112 TMEM columns) are
//     double-buffered so the epilogue of row r overlaps the MMAs of row r+1.
//   * The epilogue applies the 3x3 stencil: out[h, w, c] = sum_{i,j} G[h+i-1, w+j-1, (i,j,c)].
//     The column shift j is a warp shuffle (with the lanes at warp edges exchanged through
//     shared memory); the row shift i is carried in registers: G of row r adds its i=2 part to
//     output row r-1 (then complete and stored), its i=1 part to row r, its i=0 part to row r+1.
//   * Strips overlap by two pixels (each strip's first and last pixel lack a neighbour), bands
//     by one image row on each side (the rows just outside a band feed its edge outputs).
// Reduction order per output is fixed (taps, then the 9 stencil terms), independent of the
// band/strip/pair placement and of chunking along T.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "conv_tc.h"

namespace wan {

namespace {

constexpr int kCout = 12;
constexpr int kNP = 112;                 // 9 * 12 = 108 columns, padded to a multiple of 16
constexpr int kStripW = 128;             // pixels per strip (the MMA's M)
constexpr int kStripOut = kStripW - 2;   // outputs per strip
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kABytes = kStripW * 128;   // one 64-channel slice of one image row strip
constexpr int kBBlockBytes = kNP * 128;  // one 64-wide K block of W'
constexpr int kMaxKB = 12;               // 3 frames x (Cin <= 256) / 64
constexpr int kBOffset = kStages * kABytes;
constexpr int kBarOffset = kBOffset + kMaxKB * kBBlockBytes;
constexpr int kXchgOffset = kBarOffset + 256;
constexpr int kXchgBytes = 2 * 4 * 2 * 2 * 3 * kCout * 4;  // [parity][quarter][frame][side][i][c]
constexpr int kSmemTotal = kXchgOffset + kXchgBytes + 1024;
constexpr int kTmemCols = 512;           // 2 buffers x 2 frames x 112 columns = 448

struct HeadArgs {
  int N, T, H, W, Cin;
  int kb_per_frame;          // Cin / 64
  int pairs, strips, bands, band_rows, items;
  int has_cache;
  const wan_bf16* w;         // [12, 3, 3, 3, Cin]
  const wan_bf16* bias;      // [12] or null
  const wan_bf16* residual;  // [N, T, H, W, 12] or null
  wan_bf16* y;               // [N, T, H, W, 12]
  unsigned* err;
};

struct Item {
  int n, t, w0, h0, h1;
};

__device__ __forceinline__ Item decode_item(const HeadArgs& a, int idx) {
  Item it;
  const int pair = idx % a.pairs;
  idx /= a.pairs;
  const int band = idx % a.bands;
  idx /= a.bands;
  const int strip = idx % a.strips;
  it.n = idx / a.strips;
  it.t = 2 * pair;
  it.w0 = strip * kStripOut - 1;
  it.h0 = band * a.band_rows;
  it.h1 = min(a.H, it.h0 + a.band_rows);
  return it;
}

// Rows of G this item computes: the band plus one row on each side (inside the frame).
__device__ __forceinline__ int row_first(const Item& it) { return max(it.h0 - 1, 0); }
__device__ __forceinline__ int row_last(const HeadArgs& a, const Item& it) { return min(it.h1, a.H - 1); }

// Input frames of one row step: tau in [t-2, t+1] (t+1 only when frame t+1 exists); frames
// before the chunk without a cache read zeros and are skipped.
__device__ __forceinline__ int tau_first(const HeadArgs& a, const Item& it) {
  return a.has_cache ? it.t - 2 : max(it.t - 2, 0);
}
__device__ __forceinline__ int tau_last(const HeadArgs& a, const Item& it) {
  return it.t + 1 < a.T ? it.t + 1 : it.t;
}

// 32 lanes x 4 columns
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// G columns of tap row i for this lane's pixel: g[j*12 + c] = G[p, (i*3 + j)*12 + c].
__device__ __forceinline__ void load_tap_row(uint32_t taddr, int i, float (&g)[36]) {
  float a[16], b[16], c[4];
  tmem_ld16(taddr + i * 36, a);
  tmem_ld16(taddr + i * 36 + 16, b);
  tmem_ld4(taddr + i * 36 + 32, c);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    g[k] = a[k];
    g[16 + k] = b[k];
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) g[32 + k] = c[k];
}

__global__ void __launch_bounds__(kThreads, 1)
    head_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_cache,
                   const HeadArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* mma_done = tmem_empty + 2;
  uint64_t* xbar = mma_done + 1;  // edge-exchange barrier of the 128 epilogue threads
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 1);
  float* xchg = reinterpret_cast<float*>(smem + kXchgOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = 3 * args.kb_per_frame;

  // W' -> shared memory, 128-byte swizzle (16-byte chunk j of row n stored at chunk j ^ (n & 7)).
  {
    const int chunks = KB * kNP * 8;
    for (int q = threadIdx.x; q < chunks; q += blockDim.x) {
      const int jc = q & 7;
      const int n = (q >> 3) % kNP;
      const int kb = (q >> 3) / kNP;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < 9 * kCout) {
        const int c = n % kCout, ij = n / kCout, i = ij / 3, j = ij % 3;
        const int k = kb * 64 + jc * 8;
        const int kt = k / args.Cin, ci = k % args.Cin;
        v = *reinterpret_cast<const uint4*>(args.w + ((((size_t)c * 3 + kt) * 3 + i) * 3 + j) * args.Cin + ci);
      }
      *reinterpret_cast<uint4*>(smem + kBOffset + kb * kBBlockBytes + n * 128 + ((jc ^ (n & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], 128);
    }
    mbar_init(mma_done, 1);
    mbar_init(xbar, 128);
    fence_mbarrier_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_cache);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < args.items; item += gridDim.x) {
      const Item it = decode_item(args, item);
      const int r1 = row_last(args, it);
      for (int r = row_first(it); ok && r <= r1; ++r) {
        for (int tau = tau_first(args, it); tau <= tau_last(args, it); ++tau) {
          for (int kb = 0; kb < args.kb_per_frame; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, args.err, kDevErrTimeoutProducer)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], kABytes);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            uint8_t* dst = smem + stage * kABytes;
            if (tau < 0)
              tma_load_5d(dst, &tm_cache, &full[stage], kb * 64, it.w0, r, tau + 2, it.n);
            else
              tma_load_5d(dst, &tm_a, &full[stage], kb * 64, it.w0, r, tau, it.n);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
        }
      }
    }
    for (int s = 0; s < kStages; ++s)
      if (armed & (1u << s)) mbar_wait(&full[s], (armed_parity >> s) & 1, args.err, kDevErrTimeoutDrain);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(128, kNP);
    const uint32_t b_base = smem_u32(smem + kBOffset);
    int stage = 0;
    uint32_t phase = 0;
    int buf = 0;
    uint32_t buf_phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < args.items; item += gridDim.x) {
      const Item it = decode_item(args, item);
      const bool second = it.t + 1 < args.T;
      const int r1 = row_last(args, it);
      for (int r = row_first(it); ok && r <= r1; ++r) {
        if (!mbar_wait(&tmem_empty[buf], buf_phase ^ 1, args.err, kDevErrTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * 2 * kNP;  // frame t
        const uint32_t d1 = d0 + kNP;                   // frame t + 1
        bool first0 = true, first1 = true;
        for (int tau = tau_first(args, it); ok && tau <= tau_last(args, it); ++tau) {
          const int kt0 = tau - it.t + 2;  // tap of this input frame for output frame t
          const int kt1 = tau - it.t + 1;  // ... and for output frame t + 1
          for (int kb = 0; kb < args.kb_per_frame; ++kb) {
            if (!mbar_wait(&full[stage], phase, args.err, kDevErrTimeoutMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a_desc = smem_desc_sw128(smem_u32(smem + stage * kABytes));
            if (kt0 >= 0 && kt0 <= 2) {
              const uint64_t b_desc = smem_desc_sw128(b_base + (kt0 * args.kb_per_frame + kb) * kBBlockBytes);
#pragma unroll
              for (int k = 0; k < 4; ++k) mma_bf16(d0, a_desc + 2 * k, b_desc + 2 * k, idesc, (first0 && k == 0) ? 0u : 1u);
              first0 = false;
            }
            if (second && kt1 >= 0 && kt1 <= 2) {
              const uint64_t b_desc = smem_desc_sw128(b_base + (kt1 * args.kb_per_frame + kb) * kBBlockBytes);
#pragma unroll
              for (int k = 0; k < 4; ++k) mma_bf16(d1, a_desc + 2 * k, b_desc + 2 * k, idesc, (first1 && k == 0) ? 0u : 1u);
              first1 = false;
            }
            mma_commit(&empty[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        if (!ok) break;
        mma_commit(&tmem_full[buf]);
        if (++buf == 2) {
          buf = 0;
          buf_phase ^= 1;
        }
      }
    }
    mma_commit(mma_done);
    mbar_wait(mma_done, 0, args.err, kDevErrTimeoutDrain);
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- stencil epilogue
    const int quarter = warp & 3;
    const int q = quarter * 32 + lane;  // pixel index within the strip
    float bias[kCout];
#pragma unroll
    for (int c = 0; c < kCout; ++c) bias[c] = args.bias ? __uint_as_float(((uint32_t)args.bias[c]) << 16) : 0.f;
    int buf = 0;
    uint32_t buf_phase = 0;
    int parity = 0;
    uint32_t xphase = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < args.items; item += gridDim.x) {
      const Item it = decode_item(args, item);
      const int nframes = it.t + 1 < args.T ? 2 : 1;
      const int wcol = it.w0 + q;
      const bool col_ok = q >= 1 && q <= kStripW - 2 && wcol >= 0 && wcol < args.W;
      // Partial outputs carried across rows: prev = row r-1, cur = row r (per frame).
      float prev[2][kCout], cur[2][kCout];
#pragma unroll
      for (int f = 0; f < 2; ++f)
#pragma unroll
        for (int c = 0; c < kCout; ++c) prev[f][c] = cur[f][c] = 0.f;
      const int r0 = row_first(it), r1 = row_last(args, it);
      for (int r = r0; r <= r1; ++r) {
        if (!mbar_wait(&tmem_full[buf], buf_phase, args.err, kDevErrTimeoutEpilogue)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float next[2][kCout];
#pragma unroll
        for (int f = 0; f < 2; ++f)
#pragma unroll
          for (int c = 0; c < kCout; ++c) next[f][c] = 0.f;
        float* xw = xchg + ((parity * 4 + quarter) * 2) * 2 * 3 * kCout;  // [frame][side][i][c]
#pragma unroll
        for (int f = 0; f < 2; ++f) {
          if (f >= nframes) break;
          const uint32_t taddr = tmem_base + (uint32_t)(buf * 2 * kNP + f * kNP) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            float g[36];
            __syncwarp();
            load_tap_row(taddr, i, g);
            float s[kCout];
#pragma unroll
            for (int c = 0; c < kCout; ++c) {
              const float left = __shfl_up_sync(0xffffffffu, g[c], 1);        // G[p-1, (i,0,c)]
              const float right = __shfl_down_sync(0xffffffffu, g[24 + c], 1);  // G[p+1, (i,2,c)]
              s[c] = ((lane > 0 ? left : 0.f) + g[12 + c]) + (lane < 31 ? right : 0.f);
            }
            // Warp-edge lanes publish what the neighbouring warp's edge lane is missing.
            if (lane == 31) {
#pragma unroll
              for (int c = 0; c < kCout; ++c) xw[((f * 2 + 0) * 3 + i) * kCout + c] = g[c];
            }
            if (lane == 0) {
#pragma unroll
              for (int c = 0; c < kCout; ++c) xw[((f * 2 + 1) * 3 + i) * kCout + c] = g[24 + c];
            }
#pragma unroll
            for (int c = 0; c < kCout; ++c) {
              if (i == 2) prev[f][c] += s[c];
              else if (i == 1) cur[f][c] += s[c];
              else next[f][c] = s[c];
            }
          }
        }
        // TMEM buffer free for the next row's MMAs.
        tc_fence_before();
        mbar_arrive(&tmem_empty[buf]);
        if (++buf == 2) {
          buf = 0;
          buf_phase ^= 1;
        }
        mbar_arrive(xbar);  // publishes this thread's edge values (release) ...
        if (!mbar_wait(xbar, xphase, args.err, kDevErrTimeoutEpilogue)) {  // ... and sees the others'
          ok = false;
          break;
        }
        xphase ^= 1;
        // Edge fix-ups: lane 0 adds G[p-1, (i,0,c)] from the previous quarter's lane 31,
        // lane 31 adds G[p+1, (i,2,c)] from the next quarter's lane 0.
        if ((lane == 0 && quarter > 0) || (lane == 31 && quarter < 3)) {
          const int nq = lane == 0 ? quarter - 1 : quarter + 1;
          const int side = lane == 0 ? 0 : 1;
          const float* xn = xchg + ((parity * 4 + nq) * 2) * 2 * 3 * kCout;
#pragma unroll
          for (int f = 0; f < 2; ++f) {
            if (f >= nframes) break;
#pragma unroll
            for (int c = 0; c < kCout; ++c) {
              prev[f][c] += xn[((f * 2 + side) * 3 + 2) * kCout + c];
              cur[f][c] += xn[((f * 2 + side) * 3 + 1) * kCout + c];
              next[f][c] += xn[((f * 2 + side) * 3 + 0) * kCout + c];
            }
          }
        }
        parity ^= 1;
        // Output row r-1 is complete.
        const int ho = r - 1;
        if (col_ok && ho >= it.h0 && ho < it.h1) {
#pragma unroll
          for (int f = 0; f < 2; ++f) {
            if (f >= nframes) break;
            const size_t pix = (((size_t)it.n * args.T + it.t + f) * args.H + ho) * args.W + wcol;
            float o[kCout];
#pragma unroll
            for (int c = 0; c < kCout; ++c) o[c] = prev[f][c] + bias[c];
            if (args.residual) {
              const uint2* rp = reinterpret_cast<const uint2*>(args.residual + pix * kCout);
#pragma unroll
              for (int k = 0; k < 3; ++k) {
                const uint2 rv = rp[k];
                o[4 * k] += bf16lo_to_f32(rv.x);
                o[4 * k + 1] += bf16hi_to_f32(rv.x);
                o[4 * k + 2] += bf16lo_to_f32(rv.y);
                o[4 * k + 3] += bf16hi_to_f32(rv.y);
              }
            }
            uint2* yp = reinterpret_cast<uint2*>(args.y + pix * kCout);
#pragma unroll
            for (int k = 0; k < 3; ++k)
              yp[k] = make_uint2(pack_bf16x2(o[4 * k], o[4 * k + 1]), pack_bf16x2(o[4 * k + 2], o[4 * k + 3]));
          }
        }
#pragma unroll
        for (int f = 0; f < 2; ++f)
#pragma unroll
          for (int c = 0; c < kCout; ++c) {
            prev[f][c] = cur[f][c];
            cur[f][c] = next[f][c];
          }
      }
      if (!ok) break;
      // The last computed row was the frame's last row: its output row (r1) has no row below.
      if (r1 == args.H - 1 && col_ok && r1 >= it.h0 && r1 < it.h1) {
#pragma unroll
        for (int f = 0; f < 2; ++f) {
          if (f >= nframes) break;
          const size_t pix = (((size_t)it.n * args.T + it.t + f) * args.H + r1) * args.W + wcol;
          float o[kCout];
#pragma unroll
          for (int c = 0; c < kCout; ++c) o[c] = prev[f][c] + bias[c];
          if (args.residual) {
            const uint2* rp = reinterpret_cast<const uint2*>(args.residual + pix * kCout);
#pragma unroll
            for (int k = 0; k < 3; ++k) {
              const uint2 rv = rp[k];
              o[4 * k] += bf16lo_to_f32(rv.x);
              o[4 * k + 1] += bf16hi_to_f32(rv.x);
              o[4 * k + 2] += bf16lo_to_f32(rv.y);
              o[4 * k + 3] += bf16hi_to_f32(rv.y);
            }
          }
          uint2* yp = reinterpret_cast<uint2*>(args.y + pix * kCout);
#pragma unroll
          for (int k = 0; k < 3; ++k)
            yp[k] = make_uint2(pack_bf16x2(o[4 * k], o[4 * k + 1]), pack_bf16x2(o[4 * k + 2], o[4 * k + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_head() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_row_map(CUtensorMap* m, const void* base, int C, int W, int H, int T, int N) {
  auto fn = encode_fn_head();
  if (!fn) return false;
  const cuuint64_t dims[5] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)N};
  const cuuint64_t e = 2;
  const cuuint64_t strides[4] = {C * e, (cuuint64_t)W * C * e, (cuuint64_t)H * W * C * e,
                                 (cuuint64_t)T * H * W * C * e};
  const cuuint32_t box[5] = {64, (cuuint32_t)kStripW, 1, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool head_supported(int Cin, int Cout) { return Cout == kCout && Cin % 64 == 0 && Cin <= 256; }

cudaError_t head_launch(const wan_bf16* a, const wan_bf16* cache_in, const wan_bf16* w, const wan_bf16* bias,
                        const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W, int Cin, int sms,
                        unsigned* err, cudaStream_t stream) {
  HeadArgs args{};
  args.N = N;
  args.T = T;
  args.H = H;
  args.W = W;
  args.Cin = Cin;
  args.kb_per_frame = Cin / 64;
  args.pairs = cdiv(T, 2);
  args.strips = cdiv(W, kStripOut);
  args.has_cache = cache_in != nullptr;
  args.w = w;
  args.bias = bias;
  args.residual = residual;
  args.y = y;
  args.err = err;
  // Rows per band: the fewest rounds over the SMs, counting the two halo rows of every band.
  const long long base = (long long)N * args.pairs * args.strips;
  long long best_cost = -1;
  int best_bands = 1;
  for (int bands = 1; bands <= H && bands <= 256; ++bands) {
    const int rows = cdiv(H, bands);
    const int nb = cdiv(H, rows);
    const long long items = base * nb;
    const long long rounds = (items + sms - 1) / sms;
    const long long cost = rounds * (rows + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_bands = nb;
    }
  }
  args.band_rows = cdiv(H, best_bands);
  args.bands = cdiv(H, args.band_rows);
  args.items = (int)(base * args.bands);

  CUtensorMap ta, tc;
  if (!make_row_map(&ta, a, Cin, W, H, T, N)) return cudaErrorInvalidValue;
  if (cache_in) {
    if (!make_row_map(&tc, cache_in, Cin, W, H, 2, N)) return cudaErrorInvalidValue;
  } else {
    tc = ta;
  }
  cudaError_t e = cudaFuncSetAttribute(head_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
  if (e != cudaSuccess) return e;
  const int grid = args.items < sms ? args.items : sms;
  head_tc_kernel<<<grid, kThreads, kSmemTotal, stream>>>(ta, tc, args);
  return cudaGetLastError();
}

}  // namespace wan
