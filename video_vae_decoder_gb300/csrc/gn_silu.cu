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
//   A  statistics: work items are (frame, pixel span of ~64 KB). Every thread owns one 16-byte
//      vector of 8 channels (so its groups are fixed) and accumulates, per channel, sum(d) and
//      sum(d^2) of d = x - s, where s is one value of the channel's group in the frame (its
//      first pixel). Both sums are fp32 pairs (hi, lo): sum(d) with Knuth's TwoSum, sum(d^2)
//      (non-negative terms) with Dekker's Fast2Sum, two channels per packed fp32x2 instruction.
//      The CTA merges its threads' pairs per group (float-float adds, fixed order) and writes
//      one partial per (frame, span, group).
//   B  finalize: one warp per (frame, group) adds the span partials in fp64 in a fixed order
//      (lane-strided, then a butterfly), gets mean = s + S1/L and the population variance
//      S2/L - (S1/L)^2, and writes per channel the scale S = gamma/sqrt(var + eps) and shift
//      B = beta - mean*S, each as an fp32 (hi, lo) pair.
//   C  apply: z = (x*S_hi + B_hi) + (x*S_lo + B_lo) (two FMAs: z is accurate to fp32 rounding
//      even where x*S and B nearly cancel), then z * sigmoid(z) with sigmoid = 1/(1+e^-z) for
//      z >= 0 and e^z/(1+e^z) for z < 0, rounded once to bf16. Items run in the reverse order
//      of phase A, so the most recently read spans (still in L2) are read again first.
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

// Knuth TwoSum: s + e == a + b exactly (round-to-nearest, no overflow). Packed on float2.
__device__ __forceinline__ void two_sum2(float2& hi, float2& lo, float2 x) {
  const float2 s = __fadd2_rn(hi, x);
  const float2 bb = __fadd2_rn(s, make_float2(-hi.x, -hi.y));
  const float2 t1 = __fadd2_rn(s, make_float2(-bb.x, -bb.y));   // s - bb
  const float2 e1 = __fadd2_rn(hi, make_float2(-t1.x, -t1.y));  // hi - (s - bb)
  const float2 e2 = __fadd2_rn(x, make_float2(-bb.x, -bb.y));   // x - bb
  lo = __fadd2_rn(lo, __fadd2_rn(e1, e2));
  hi = s;
}

// Dekker Fast2Sum for non-negative running sums: exact when hi >= x, and otherwise off by at
// most the rounding of the smaller (earlier) partial sum.
__device__ __forceinline__ void fast_two_sum2(float2& hi, float2& lo, float2 x) {
  const float2 s = __fadd2_rn(hi, x);
  const float2 z = __fadd2_rn(s, make_float2(-hi.x, -hi.y));
  lo = __fadd2_rn(lo, __fadd2_rn(x, make_float2(-z.x, -z.y)));
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

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void stg_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float2 unpack2(uint32_t w) {
  return make_float2(bf16lo_to_f32(w), bf16hi_to_f32(w));
}

__device__ __forceinline__ float bf16_at(const wan_bf16* p) { return __uint_as_float(((uint32_t)*p) << 16); }

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// z * sigmoid(z): t = e^-|z| (never overflows), sigmoid = 1/(1+t) or t/(1+t).
__device__ __forceinline__ float silu_f32(float z) {
  const float t = ex2_approx(-fabsf(z) * 1.4426950408889634f);
  const float r = rcp_approx(1.0f + t);
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

struct GnArgs {
  const wan_bf16* x;
  wan_bf16* y;
  const float* gamma;
  const float* beta;
  GnPartial* part;  // [F][spans][G]
  float4* coef;     // [F][C]: (S_hi, S_lo, B_hi, B_lo)
  unsigned* bar;    // grid-barrier arrival counter, zero at launch
  unsigned* err;
  int P, C, G, F, span_px, spans;
  float eps;
  double inv_len;   // 1 / (H * W * C / G)
};

__global__ void __launch_bounds__(kThreads) gn_silu_kernel(const GnArgs a) {
  extern __shared__ float red[];  // [blockDim][slots][4] float-float partial sums
  __shared__ int s_flag;
  const int vpp = a.C >> 3;
  const int ppi = blockDim.x / vpp;
  const int tid = threadIdx.x;
  const int j = tid % vpp;
  const int lp = tid / vpp;
  const bool active = lp < ppi;
  const int cg = a.C / a.G;
  const int slots = cg >= 8 ? 1 : 8 / cg;
  const int items = a.F * a.spans;
  const size_t pstride = (size_t)a.C * 2;
  constexpr int U = 4;

  // ---------------------------------------------------------------- A: statistics
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int f = item / a.spans, span = item - f * a.spans;
    const int p0 = span * a.span_px, p1 = min(a.P, p0 + a.span_px);
    const wan_bf16* xf = a.x + (size_t)f * a.P * a.C;
    float2 s1h[4], s1l[4], s2h[4], s2l[4], sh[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      s1h[w] = s1l[w] = s2h[w] = s2l[w] = make_float2(0.f, 0.f);
      const int c0 = 8 * j + 2 * w;
      sh[w] = active ? make_float2(bf16_at(xf + (c0 / cg) * cg), bf16_at(xf + ((c0 + 1) / cg) * cg))
                     : make_float2(0.f, 0.f);
    }
    if (active) {
      const char* base = reinterpret_cast<const char*>(xf) + (size_t)j * 16;
      int p = p0 + lp;
      for (; p + (U - 1) * ppi < p1; p += U * ppi) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = ldg_nc_v4(base + (size_t)(p + u * ppi) * pstride);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float2 d = __fadd2_rn(unpack2(wv[w]), make_float2(-sh[w].x, -sh[w].y));
            two_sum2(s1h[w], s1l[w], d);
            fast_two_sum2(s2h[w], s2l[w], __fmul2_rn(d, d));
          }
        }
      }
      for (; p < p1; p += ppi) {
        const uint4 v = ldg_nc_v4(base + (size_t)p * pstride);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 d = __fadd2_rn(unpack2(wv[w]), make_float2(-sh[w].x, -sh[w].y));
          two_sum2(s1h[w], s1l[w], d);
          fast_two_sum2(s2h[w], s2l[w], __fmul2_rn(d, d));
        }
      }
    }
    // Fold this thread's 8 channel partials by group slot (channels of a group are consecutive:
    // a vector holds 8/cg groups when cg < 8, else part of one group).
    float* mine = red + (size_t)tid * slots * 4;
    for (int q = 0; q < slots; ++q) {
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
          const float* r = red + ((size_t)(l * vpp + jj) * slots + q) * 4;
          ff_add(ah, al, r[0], r[1]);
          ff_add(bh, bl, r[2], r[3]);
        }
      GnPartial out;
      out.s1_hi = ah;
      out.s1_lo = al;
      out.s2_hi = bh;
      out.s2_lo = bl;
      a.part[((size_t)f * a.spans + span) * a.G + g] = out;
    }
    __syncthreads();  // red is reused by the next item
  }
  if (!grid_barrier(a.bar, gridDim.x, a.err, &s_flag)) return;

  // ---------------------------------------------------------------- B: finalize per (frame, group)
  {
    const int warps = blockDim.x >> 5, warp = tid >> 5, lane = tid & 31;
    for (int pr = blockIdx.x * warps + warp; pr < a.F * a.G; pr += gridDim.x * warps) {
      const int f = pr / a.G, g = pr - f * a.G;
      double s1 = 0.0, s2 = 0.0;
      for (int s = lane; s < a.spans; s += 32) {
        const GnPartial q = a.part[((size_t)f * a.spans + s) * a.G + g];
        s1 += (double)q.s1_hi + (double)q.s1_lo;
        s2 += (double)q.s2_hi + (double)q.s2_lo;
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {  // fixed butterfly; addition commutes, so every
        s1 += __shfl_xor_sync(0xffffffffu, s1, off);  // lane ends with the same bits
        s2 += __shfl_xor_sync(0xffffffffu, s2, off);
      }
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
      for (int k = lane; k < cg; k += 32) {
        const int c = g * cg + k;
        const double S = (double)a.gamma[c] * rstd;
        const double B = (double)a.beta[c] - mean * S;
        const float shi = (float)S, bhi = (float)B;
        a.coef[(size_t)f * a.C + c] = make_float4(shi, (float)(S - (double)shi), bhi, (float)(B - (double)bhi));
      }
    }
  }
  if (!grid_barrier(a.bar, 2 * gridDim.x, a.err, &s_flag)) return;

  // ---------------------------------------------------------------- C: apply, newest spans first
  if (!active) return;
  for (int k = blockIdx.x; k < items; k += gridDim.x) {
    const int item = items - 1 - k;
    const int f = item / a.spans, span = item - f * a.spans;
    const int p0 = span * a.span_px, p1 = min(a.P, p0 + a.span_px);
    float2 shi[4], slo[4], bhi[4], blo[4];
    const float4* cf = a.coef + (size_t)f * a.C + 8 * j;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 u = cf[2 * w], v = cf[2 * w + 1];
      shi[w] = make_float2(u.x, v.x);
      slo[w] = make_float2(u.y, v.y);
      bhi[w] = make_float2(u.z, v.z);
      blo[w] = make_float2(u.w, v.w);
    }
    const size_t frame_off = (size_t)f * a.P * a.C;
    const char* xb = reinterpret_cast<const char*>(a.x + frame_off) + (size_t)j * 16;
    char* yb = reinterpret_cast<char*>(a.y + frame_off) + (size_t)j * 16;
    for (int p = p0 + lp; p < p1; p += U * ppi) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (p + u * ppi < p1) v[u] = ldg_nc_v4(xb + (size_t)(p + u * ppi) * pstride);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (p + u * ppi >= p1) break;
        uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 xv = unpack2(wv[w]);
          const float2 z = __fadd2_rn(__ffma2_rn(xv, shi[w], bhi[w]), __ffma2_rn(xv, slo[w], blo[w]));
          wv[w] = pack_bf16x2(silu_f32(z.x), silu_f32(z.y));
        }
        stg_v4(yb + (size_t)(p + u * ppi) * pstride, make_uint4(wv[0], wv[1], wv[2], wv[3]));
      }
    }
  }
}

struct GnPlan {
  int P, F, threads, ppi, span_px, spans, slots;
  size_t part_bytes, coef_bytes, smem;
};

GnPlan plan(int N, int T, int H, int W, int C, int G) {
  GnPlan pl;
  pl.P = H * W;
  pl.F = N * T;
  const int vpp = C / 8;
  pl.threads = (kThreads / vpp) * vpp;  // C <= 2048: vpp <= 256
  pl.ppi = pl.threads / vpp;
  // Spans depend on the frame's geometry only (about 64 KB of x each), never on the number of
  // frames in the call: a frame's statistics are summed in the same order in any chunking.
  int span_px = (65536 / (C * 2)) / pl.ppi * pl.ppi;
  if (span_px < pl.ppi) span_px = pl.ppi;
  const int whole = cdiv(pl.P, pl.ppi) * pl.ppi;
  if (span_px > whole) span_px = whole;
  pl.span_px = span_px;
  pl.spans = cdiv(pl.P, span_px);
  const int cg = C / G;
  pl.slots = cg >= 8 ? 1 : 8 / cg;
  pl.part_bytes = (size_t)pl.F * pl.spans * G * sizeof(GnPartial);
  pl.coef_bytes = (size_t)pl.F * C * sizeof(float4);
  pl.smem = (size_t)pl.threads * pl.slots * 4 * sizeof(float);
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
  a.span_px = pl.span_px;
  a.spans = pl.spans;
  a.eps = eps;
  a.inv_len = 1.0 / ((double)pl.P * (C / G));
  // Persistent grid: every CTA resident at once (the cooperative launch checks it).
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gn_silu_kernel, pl.threads, pl.smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = per_sm * sms;
  const int items = pl.F * pl.spans;
  if (grid > items) grid = items;
  // The barrier counter is the one scratch word that must start at zero.
  e = cudaMemsetAsync(a.bar, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  void* args[] = {&a};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(gn_silu_kernel), dim3(grid), dim3(pl.threads),
                                     args, pl.smem, stream);
}

}  // namespace wan
