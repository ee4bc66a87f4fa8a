// GroupNorm + SiLU over bf16 NDHWC video tensors, statistics per (frame, group).
//
// Method (WanGP, shared/kernels/group_norm_silu.py: module docstring, `_sums_kernel`,
// `_group_stats`, `_apply_kernel`): FP32 arithmetic whose sums carry their rounding errors
// (two-sum), partials combined in a fixed order, population variance with eps inside the root,
// then z * sigmoid(z) rounded once to bf16.
//
// GB300 layout of the work: ONE cooperative, persistent kernel in three phases separated by
// two grid barriers (bounded waits; a barrier that times out records an error and the kernel
// winds down):
//   A  statistics: work items are (frame, pixel span of ~64 KB), dealt round-robin to the CTAs.
//      x streams through shared memory: each CTA keeps six 16 KB pieces in flight with bulk async
//      copies (cp.async.bulk, completion on an mbarrier). Every thread owns one 16-byte
//      vector of 8 channels (so its groups are fixed) and accumulates, per channel, sum(d) and
//      sum(d^2) of d = x - s, where s is one value of the channel's group in the frame (its
//      first pixel). Both sums are fp32 pairs (hi, lo): sum(d) with Knuth's TwoSum, sum(d^2)
//      (non-negative terms) with Dekker's Fast2Sum, two channels per packed fp32x2 instruction.
//      The CTA merges its threads' pairs per group (float-float adds, fixed order) and writes
//      one partial per (frame, span, group).
//   B  finalize: one warp per (frame, group) adds the span partials as float-float pairs in a
//      fixed order (lane-strided, then a butterfly), gets in fp64 mean = s + S1/L and the variance
//      S2/L - (S1/L)^2, and writes per channel the scale S = gamma/sqrt(var + eps) and shift
//      B = beta - mean*S, each as an fp32 (hi, lo) pair.
//   C  apply, newest items first (their x is still in L2), read with plain 16-byte loads
//      (eight in flight per thread); the frame's coefficients reach shared memory with one bulk
//      copy per CTA. z = (x*S_hi + B_hi) + (x*S_lo + B_lo) (two FMAs: z is accurate to fp32
//      rounding even where x*S and B nearly cancel), then z * sigmoid(z) = z / (1 + e^-z)
//      (z e^z / (1 + e^z) for vectors holding a z < -80, whose result may be subnormal), rounded
//      once to bf16.
// x is read from HBM once (phase A); phase C re-reads it mostly from L2 and writes y. The
// pages' second, centred pass over x is replaced by the shifted one-pass sums: the shift is a
// value of the group itself, so the subtraction in the variance loses only the few bits of
// (mean - s)^2 / var, against the ~45 bits the error-free sums carry.
// Statistics depend only on the frame (the span partition depends on H, W and C alone), so a
// frame gets the same bits whether the video comes in one call or in chunks.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "gn_silu.h"

namespace wan {

namespace {

constexpr int kThreads = 256;

struct GnPartial {  // one (frame, span, group): float-float sums of d and d^2
  float s1_hi, s1_lo, s2_hi, s2_lo;
};

// a - b on float2 in one packed instruction: b * (-1) + a with one rounding equals the rounded
// difference (there is no packed subtract).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.f, -1.f), a); }

// Knuth TwoSum: s + e == a + b exactly (round-to-nearest, no overflow). Packed on float2.
__device__ __forceinline__ void two_sum2(float2& hi, float2& lo, float2 x) {
  const float2 s = __fadd2_rn(hi, x);
  const float2 bb = sub2(s, hi);
  const float2 e1 = sub2(hi, sub2(s, bb));  // hi - (s - bb)
  const float2 e2 = sub2(x, bb);            // x - bb
  lo = __fadd2_rn(lo, __fadd2_rn(e1, e2));
  hi = s;
}

// Dekker Fast2Sum for non-negative running sums: exact when hi >= x, and otherwise off by at
// most the rounding of the smaller (earlier) partial sum.
__device__ __forceinline__ void fast_two_sum2(float2& hi, float2& lo, float2 x) {
  const float2 s = __fadd2_rn(hi, x);
  lo = __fadd2_rn(lo, sub2(x, sub2(s, hi)));
  hi = s;
}

// Float-float addition (hi, lo) += (bhi, blo), result renormalised.
__device__ __forceinline__ void ff_add(float& hi, float& lo, float bhi, float blo) {
  const float s = __fadd_rn(hi, bhi);
  const float bb = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(bhi, bb));
  const float t = __fadd_rn(e, __fadd_rn(lo, blo));
  hi = __fadd_rn(s, t);
  lo = __fsub_rn(t, __fsub_rn(hi, s));
}

__device__ __forceinline__ void stg_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float2 unpack2(uint32_t w) {
  return make_float2(bf16lo_to_f32(w), bf16hi_to_f32(w));
}

__device__ __forceinline__ float bf16_at(const wan_bf16* p) { return __uint_as_float(((uint32_t)*p) << 16); }

__device__ __forceinline__ float ex2_approx(float x) {  // subnormal results kept
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ex2_approx_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx_ftz(float x) {  // used on [1, 5.6e34]
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// SiLU of two values for z >= -80: z / (1 + e^-z), with e^-z = 2^(-z log2 e) <= 2^116 (no overflow;
// it underflows to 0 for large z, where the result is z) and 1 + e^-z <= 5.6e34, whose reciprocal
// is a normal fp32 number (no flush). For z << 0, 1 + e^-z rounds to e^-z and the quotient to
// z e^z with fp32 relative precision.
__device__ __forceinline__ float2 silu2_fast(float2 z) {
  const float2 m = __fmul2_rn(z, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  const float2 u = __fadd2_rn(make_float2(ex2_approx_ftz(m.x), ex2_approx_ftz(m.y)), make_float2(1.f, 1.f));
  return __fmul2_rn(z, make_float2(rcp_approx_ftz(u.x), rcp_approx_ftz(u.y)));
}

// z * sigmoid(z): t = e^-|z| (never overflows), sigmoid = 1/(1+t) or t/(1+t). Used for vectors
// holding a z < -80, whose result may be subnormal.
__device__ __forceinline__ float silu_exact_range(float z) {
  const float t = ex2_approx(fminf(z, -z) * 1.4426950408889634f);
  const float r = rcp_approx_ftz(1.0f + t);
  return z < 0.f ? (z * t) * r : z * r;
}

// Grid-wide barrier for a cooperative launch (all CTAs co-resident). `ctr` counts arrivals
// over the whole call (cleared before the launch); barrier k waits for k * gridDim.x arrivals.
// The wait is bounded: on timeout it records kDevErrTimeoutGrid and returns false everywhere.
__device__ bool grid_barrier(unsigned* ctr, unsigned target, unsigned* err, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    int ok = 1;
    const long long start = clock64();
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if (clock64() - start > kWaitCycles) {
        atomicOr(err, kDevErrTimeoutGrid);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

constexpr int kSlots = 3;          // 32 KB pieces of x in flight per CTA
constexpr int kVecPerThread = 8;   // 16-byte vectors per thread per piece
constexpr int kPiecesPerSpan = 2;  // a statistics partial covers 2 pieces (about 64 KB)
constexpr int kApplyUnroll = 8;    // 16-byte loads in flight per thread in the apply phase
constexpr int kFinBatch = 8;       // partials in flight per lane in the finalize

struct GnArgs {
  const wan_bf16* x;
  wan_bf16* y;
  const float* gamma;
  const float* beta;
  GnPartial* part;  // [F][G][spans]
  float4* coef;     // [F][C]: (S_hi, S_lo, B_hi, B_lo)
  unsigned* bar;    // grid-barrier arrival counter, zero at launch
  unsigned* err;
  int P, C, G, F, piece_px, spans, items;
  float eps;
  double inv_len;   // 1 / (H * W * C / G)
};

// Pixel range [q0, q1) of piece j of statistics item `item` (empty past the end of a frame).
__device__ __forceinline__ void piece_range(const GnArgs& a, int item, int j, int& f, int& q0, int& q1) {
  f = item / a.spans;
  const int piece = (item - f * a.spans) * kPiecesPerSpan + j;
  q0 = min(a.P, piece * a.piece_px);
  q1 = min(a.P, q0 + a.piece_px);
}

__global__ void __launch_bounds__(kThreads) gn_silu_kernel(const GnArgs a) {
  extern __shared__ __align__(128) uint8_t gsm[];
  uint8_t* slots = gsm;                                                  // kSlots x piece bytes
  const int vpp = a.C >> 3;
  const int ppi = blockDim.x / vpp;
  const int piece_bytes = a.piece_px * a.C * 2;
  float* red = reinterpret_cast<float*>(gsm + kSlots * piece_bytes);   // [blockDim][slots][4]
  float* s_shift = red + (size_t)blockDim.x * (a.C / a.G >= 8 ? 1 : 8 / (a.C / a.G)) * 4;  // [G]
  float4* s_coef = reinterpret_cast<float4*>(slots);  // [C], phase C only (the slots are idle then)
  __shared__ uint64_t full[kSlots];
  __shared__ uint64_t cbar;
  __shared__ int s_flag;
  const int tid = threadIdx.x;
  const int j = tid % vpp;
  const int lp = tid / vpp;
  const bool active = lp < ppi;
  const int cg = a.C / a.G;
  const int nslot = cg >= 8 ? 1 : 8 / cg;
  const int cnt = (a.items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // items of this CTA

  // The CTA's stream of pieces: its statistics items (item = blockIdx + k * grid), kPiecesPerSpan
  // pieces each; piece n is piece n % kPiecesPerSpan of the (n / kPiecesPerSpan)-th item.
  auto issue = [&](int n) {  // thread 0: start loading piece n of the stream
    if (n >= cnt * kPiecesPerSpan) return;
    const int k = n / kPiecesPerSpan, jj = n - k * kPiecesPerSpan;
    uint64_t* bar = &full[n % kSlots];
    int f, q0, q1;
    piece_range(a, blockIdx.x + k * gridDim.x, jj, f, q0, q1);
    const uint32_t bytes = (uint32_t)(q1 - q0) * a.C * 2;
    if (bytes) {
      mbar_arrive_expect_tx(bar, bytes);
      bulk_load(slots + (n % kSlots) * piece_bytes, a.x + ((size_t)f * a.P + q0) * a.C, bytes, bar);
    } else {
      mbar_arrive(bar);
    }
  };
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) mbar_init(&full[s], 1);
    fence_mbarrier_init();
    for (int n = 0; n < kSlots; ++n) issue(n);
  }
  __syncthreads();
  int n = 0;  // next piece of the stream to consume

  // Waits for piece n (all threads), bounded; the failure is made CTA-uniform by the caller.
  auto wait_piece = [&](int nn) -> bool {
    return mbar_wait(&full[nn % kSlots], (uint32_t)((nn / kSlots) & 1), a.err, kDevErrTimeoutGrid);
  };

  // ---------------------------------------------------------------- A: statistics
  for (int k = 0; k < cnt; ++k) {
    const int item = blockIdx.x + k * gridDim.x;
    const int f = item / a.spans, span = item - f * a.spans;
    // The group shifts (each group's first value in the frame), loaded once per CTA: a
    // per-thread load would send every thread of the grid to the same few L2 lines.
    const wan_bf16* xf = a.x + (size_t)f * a.P * a.C;
    for (int g = tid; g < a.G; g += blockDim.x) s_shift[g] = bf16_at(xf + (size_t)g * cg);
    __syncthreads();
    float2 s1h[4], s1l[4], s2h[4], s2l[4], sh[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      s1h[w] = s1l[w] = s2h[w] = s2l[w] = make_float2(0.f, 0.f);
      const int c0 = 8 * j + 2 * w;
      sh[w] = active ? make_float2(s_shift[c0 / cg], s_shift[(c0 + 1) / cg]) : make_float2(0.f, 0.f);
    }
    for (int pj = 0; pj < kPiecesPerSpan; ++pj, ++n) {
      const bool ok = wait_piece(n);
      int f2, q0, q1;
      piece_range(a, item, pj, f2, q0, q1);
      if (ok && active) {
        const uint8_t* src = slots + (n % kSlots) * piece_bytes + (size_t)j * 16;
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
          const int pl = lp + i * ppi;
          if (q0 + pl >= q1) break;
          const uint4 v = *reinterpret_cast<const uint4*>(src + (size_t)pl * vpp * 16);
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float2 d = sub2(unpack2(wv[w]), sh[w]);
            two_sum2(s1h[w], s1l[w], d);
            fast_two_sum2(s2h[w], s2l[w], __fmul2_rn(d, d));
          }
        }
      }
      if (__syncthreads_or(!ok)) return;  // every thread is done with the slot
      if (tid == 0) issue(n + kSlots);
    }
    (void)span;
    // Fold this thread's 8 channel partials by group slot (channels of a group are consecutive:
    // a vector holds 8/cg groups when cg < 8, else part of one group).
    float* mine = red + (size_t)tid * nslot * 4;
    for (int q = 0; q < nslot; ++q) {
      float ah = 0.f, al = 0.f, bh = 0.f, bl = 0.f;
      if (active) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if ((cg >= 8 ? 0 : c / cg) != q) continue;
          const int w = c >> 1;
          ff_add(ah, al, (c & 1) ? s1h[w].y : s1h[w].x, (c & 1) ? s1l[w].y : s1l[w].x);
          ff_add(bh, bl, (c & 1) ? s2h[w].y : s2h[w].x, (c & 1) ? s2l[w].y : s2l[w].x);
        }
      }
      mine[q * 4 + 0] = ah;
      mine[q * 4 + 1] = al;
      mine[q * 4 + 2] = bh;
      mine[q * 4 + 3] = bl;
    }
    __syncthreads();
    // One thread per group adds the contributions of the threads holding it, in thread order.
    for (int g = tid; g < a.G; g += blockDim.x) {
      float ah = 0.f, al = 0.f, bh = 0.f, bl = 0.f;
      const int c_first = g * cg, c_last = c_first + cg - 1;
      const int q = cg >= 8 ? 0 : (c_first % 8) / cg;
      for (int jj = c_first / 8; jj <= c_last / 8; ++jj)
        for (int l = 0; l < ppi; ++l) {
          const float* r = red + ((size_t)(l * vpp + jj) * nslot + q) * 4;
          ff_add(ah, al, r[0], r[1]);
          ff_add(bh, bl, r[2], r[3]);
        }
      GnPartial out;
      out.s1_hi = ah;
      out.s1_lo = al;
      out.s2_hi = bh;
      out.s2_lo = bl;
      a.part[((size_t)f * a.G + g) * a.spans + span] = out;
    }
    __syncthreads();  // red is reused by the next item
  }
  if (!grid_barrier(a.bar, gridDim.x, a.err, &s_flag)) return;

  // ---------------------------------------------------------------- B: finalize per (frame, group)
  {
    const int warps = blockDim.x >> 5, warp = tid >> 5, lane = tid & 31;
    // pair p -> CTA p % grid, warp (p / grid) % warps: the few pairs spread over many SMs.
    for (int pr = warp * gridDim.x + blockIdx.x; pr < a.F * a.G; pr += gridDim.x * warps) {
      const int f = pr / a.G, g = pr - f * a.G;
      // Float-float sums (fp64 issue is scarce on this GPU): lane-strided, then a butterfly.
      // The float-float add is commutative bit for bit (TwoSum's error term is unique), so every
      // lane ends with the same bits.
      // A lane adds spans lane, lane + 32, ... in order, loading kFinBatch of them at a time.
      float h1 = 0.f, l1 = 0.f, h2 = 0.f, l2 = 0.f;
      const float4* src = reinterpret_cast<const float4*>(a.part) + ((size_t)f * a.G + g) * a.spans;
      for (int sp0 = 0; sp0 < a.spans; sp0 += 32 * kFinBatch) {
        float4 q[kFinBatch];
#pragma unroll
        for (int i = 0; i < kFinBatch; ++i) {
          const int sp = sp0 + lane + 32 * i;
          q[i] = sp < a.spans ? __ldcg(src + sp) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kFinBatch; ++i) {  // adding (0, 0) to a normalised pair changes nothing
          ff_add(h1, l1, q[i].x, q[i].y);
          ff_add(h2, l2, q[i].z, q[i].w);
        }
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float oh1 = __shfl_xor_sync(0xffffffffu, h1, off), ol1 = __shfl_xor_sync(0xffffffffu, l1, off);
        const float oh2 = __shfl_xor_sync(0xffffffffu, h2, off), ol2 = __shfl_xor_sync(0xffffffffu, l2, off);
        ff_add(h1, l1, oh1, ol1);
        ff_add(h2, l2, oh2, ol2);
      }
      const double s1 = (double)h1 + (double)l1, s2 = (double)h2 + (double)l2;
      // fp64 division and square root are slow on this GPU: 1/L comes from the host and
      // 1/sqrt(v) is an fp32 estimate refined by two Newton steps r <- r (3 - v r^2) / 2 in fp64
      // (relative error 2^-22 -> 2^-44 -> below fp64 rounding).
      const double m1 = s1 * a.inv_len;
      const double mean = (double)bf16_at(a.x + (size_t)f * a.P * a.C + (size_t)g * cg) + m1;
      const double v = fmax(s2 * a.inv_len - m1 * m1, 0.0) + (double)a.eps;
      double rstd;
      if (v > 1e-30 && v < 1e30) {
        rstd = (double)rsqrtf((float)v);
        rstd = rstd * (1.5 - 0.5 * v * rstd * rstd);
        rstd = rstd * (1.5 - 0.5 * v * rstd * rstd);
      } else {
        rstd = 1.0 / sqrt(v);
      }
      for (int kk = lane; kk < cg; kk += 32) {
        const int c = g * cg + kk;
        const double S = (double)a.gamma[c] * rstd;
        const double B = (double)a.beta[c] - mean * S;
        const float shi = (float)S, bhi = (float)B;
        a.coef[(size_t)f * a.C + c] = make_float4(shi, (float)(S - (double)shi), bhi, (float)(B - (double)bhi));
      }
    }
  }
  if (!grid_barrier(a.bar, 2 * gridDim.x, a.err, &s_flag)) return;

  // ---------------------------------------------------------------- C: apply, newest spans first
  // The frame's coefficients reach shared memory with one bulk copy per CTA (a per-thread load
  // would send every thread of the grid to the same few L2 lines).
  if (tid == 0) {
    mbar_init(&cbar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  int fcur = -1;
  uint32_t cphase = 0;
  float2 shi[4], slo[4], bhi[4], blo[4];
  for (int k = 0; k < cnt; ++k) {
    const int item = a.items - 1 - (int)(blockIdx.x + k * gridDim.x);  // newest spans first
    const int f = item / a.spans;
    if (f != fcur) {
      __syncthreads();  // the previous frame's coefficients have been read
      if (tid == 0) {
        // Written by other CTAs with ordinary stores (ordered before the grid barrier); the copy
        // reads them through the async proxy.
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_expect_tx(&cbar, (uint32_t)a.C * 16u);
        bulk_load(s_coef, a.coef + (size_t)f * a.C, (uint32_t)a.C * 16u, &cbar);
      }
      const bool okc = mbar_wait(&cbar, cphase, a.err, kDevErrTimeoutGrid);
      cphase ^= 1;
      if (__syncthreads_or(!okc)) return;
      fcur = f;
      const float4* cf = s_coef + 8 * j;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float4 u = cf[2 * w], v = cf[2 * w + 1];
        shi[w] = make_float2(u.x, v.x);
        slo[w] = make_float2(u.y, v.y);
        bhi[w] = make_float2(u.z, v.z);
        blo[w] = make_float2(u.w, v.w);
      }
    }
    // x comes back from L2 (phase A read it from HBM moments ago) with plain 16-byte loads,
    // kApplyUnroll in flight per thread, and no CTA-wide synchronisation.
    const int span = item - f * a.spans;
    const int q0 = min(a.P, span * kPiecesPerSpan * a.piece_px);
    const int q1 = min(a.P, q0 + kPiecesPerSpan * a.piece_px);
    if (active) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)f * a.P * a.C) + j;
      char* dst = reinterpret_cast<char*>(a.y + (size_t)f * a.P * a.C) + (size_t)j * 16;
      for (int p = q0 + lp; p < q1; p += ppi * kApplyUnroll) {
        uint4 v[kApplyUnroll];
#pragma unroll
        for (int u = 0; u < kApplyUnroll; ++u) {
          const int pp = p + u * ppi;
          v[u] = pp < q1 ? __ldg(src + (size_t)pp * vpp) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kApplyUnroll; ++u) {
          const int pp = p + u * ppi;
          if (pp >= q1) break;
          uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          float2 z[4];
          float zmin = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float2 xv = unpack2(wv[w]);
            z[w] = __fadd2_rn(__ffma2_rn(xv, shi[w], bhi[w]), __ffma2_rn(xv, slo[w], blo[w]));
            zmin = fminf(zmin, fminf(z[w].x, z[w].y));
          }
          if (zmin >= -80.f) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float2 o = silu2_fast(z[w]);
              wv[w] = pack_bf16x2(o.x, o.y);
            }
          } else {
#pragma unroll
            for (int w = 0; w < 4; ++w) wv[w] = pack_bf16x2(silu_exact_range(z[w].x), silu_exact_range(z[w].y));
          }
          stg_v4(dst + (size_t)pp * vpp * 16, make_uint4(wv[0], wv[1], wv[2], wv[3]));
        }
      }
    }
  }
}

struct GnPlan {
  int P, F, threads, ppi, piece_px, spans, items, slots;
  size_t part_bytes, coef_bytes, smem;
};

GnPlan plan(int N, int T, int H, int W, int C, int G) {
  GnPlan pl;
  pl.P = H * W;
  pl.F = N * T;
  const int vpp = C / 8;
  pl.threads = (kThreads / vpp) * vpp;  // C <= 2048: vpp <= 256
  pl.ppi = pl.threads / vpp;
  // Pieces and spans depend on the frame's geometry only, never on the number of frames in the
  // call: a frame's statistics are summed in the same order in any chunking of the video.
  pl.piece_px = kVecPerThread * pl.ppi;
  const int pieces = cdiv(pl.P, pl.piece_px);
  pl.spans = cdiv(pieces, kPiecesPerSpan);
  pl.items = pl.F * pl.spans;
  const int cg = C / G;
  pl.slots = cg >= 8 ? 1 : 8 / cg;
  pl.part_bytes = (size_t)pl.F * pl.spans * G * sizeof(GnPartial);
  pl.coef_bytes = (size_t)pl.F * C * sizeof(float4);
  pl.smem = (size_t)kSlots * pl.piece_px * C * 2 + (size_t)pl.threads * pl.slots * 4 * sizeof(float) +
            (size_t)G * sizeof(float);
  return pl;
}

inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t gn_silu_workspace(int N, int T, int H, int W, int C, int G, int sms) {
  (void)sms;
  const GnPlan pl = plan(N, T, H, W, C, G);
  return align256(pl.part_bytes) + align256(pl.coef_bytes) + 256;
}

bool gn_silu_supported(int C, int G) {
  if (C <= 0 || G <= 0 || C % G != 0 || C % 8 != 0) return false;
  if (C > 2048) return false;
  const int cg = C / G;
  return (cg % 8 == 0) || (8 % cg == 0);
}

cudaError_t gn_silu_launch(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta,
                           int N, int T, int H, int W, int C, int G, float eps, void* ws, int sms,
                           cudaStream_t stream) {
  const GnPlan pl = plan(N, T, H, W, C, G);
  char* base = reinterpret_cast<char*>(ws);
  GnArgs a;
  a.x = x;
  a.y = y;
  a.gamma = gamma;
  a.beta = beta;
  a.part = reinterpret_cast<GnPartial*>(base);
  a.coef = reinterpret_cast<float4*>(base + align256(pl.part_bytes));
  a.bar = reinterpret_cast<unsigned*>(base + align256(pl.part_bytes) + align256(pl.coef_bytes));
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidValue;
  a.P = pl.P;
  a.C = C;
  a.G = G;
  a.F = pl.F;
  a.piece_px = pl.piece_px;
  a.spans = pl.spans;
  a.items = pl.items;
  a.eps = eps;
  a.inv_len = 1.0 / ((double)pl.P * (C / G));
  // Persistent grid: every CTA resident at once (the cooperative launch checks it).
  cudaError_t e = cudaFuncSetAttribute(gn_silu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gn_silu_kernel, pl.threads, pl.smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // As many CTAs as fit, then evened out so every CTA gets the same number of items (a CTA with
  // fewer items would only wait at the grid barriers).
  const int items = pl.items;
  int grid = per_sm * sms;
  if (grid > items) grid = items;
  const int rounds = cdiv(items, grid);
  grid = cdiv(items, rounds);
  // The barrier counter is the one scratch word that must start at zero.
  e = cudaMemsetAsync(a.bar, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  void* args[] = {&a};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(gn_silu_kernel), dim3(grid), dim3(pl.threads),
                                     args, pl.smem, stream);
}

}  // namespace wan
