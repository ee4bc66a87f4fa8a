// GroupNorm + SiLU over bf16 NDHWC video tensors, statistics per (frame, group).
//
// Method (WanGP, shared/kernels/group_norm_silu.py: module docstring, `_sums_kernel`,
// `_group_stats`, `_apply_kernel`): FP32 arithmetic whose sums carry their rounding errors
// (two-sum), partials combined in a fixed order, population variance with eps inside the root,
// then z * sigmoid(z) rounded once to bf16.
//
// GB300 layout of the work (three launches):
//   gn_stats     one CTA per (frame, pixel span). Every thread owns one 16-byte vector of 8
//                channels for the whole span (so its groups are fixed) and accumulates, per
//                channel, sum(d) and sum(d^2) of d = x - s, where s is the first value of the
//                channel's group in the span. Both sums are fp32 pairs (hi, lo): sum(d) with
//                Knuth's TwoSum, sum(d^2) (non-negative terms) with Dekker's Fast2Sum. Packed
//                fp32x2 instructions carry two channels per instruction. The CTA merges its
//                threads' pairs per group (float-float adds, fixed order) and writes one
//                partial (count, shift, S1, S2) per group.
//   gn_finalize  one warp per (frame, group): merges the span partials with the pairwise
//                mean/variance update of Chan, Golub and LeVeque (1979) in fp64, in span order,
//                then per channel writes scale S = gamma/sqrt(var+eps) and shift
//                B = beta - mean*S, each as an fp32 (hi, lo) pair.
//   gn_apply     z = (x*S_hi + B_hi) + (x*S_lo + B_lo) with two FMAs (the hi/lo pairs make z
//                accurate to fp32 rounding even where x*S and B nearly cancel), then
//                z * sigmoid(z) with sigmoid = 1/(1+e^-z) for z >= 0 and e^z/(1+e^z) for z < 0,
//                rounded once to bf16 (round to nearest even).
// The one-pass statistics with a per-span shift replace the pages' second (centred) pass over
// x: on GB300 a statistics pass is bounded by HBM and by fp32 issue, so reading x once for both
// moments is the cheaper exact route; the merge is exact up to fp64 rounding.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "gn_silu.h"

namespace wan {

namespace {

struct GnPartial {  // one (frame, span, group)
  float s1_hi, s1_lo, s2_hi, s2_lo;
  float shift;
  int count;
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

// ----------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gn_stats_kernel(const wan_bf16* __restrict__ x,
                                                       GnPartial* __restrict__ part, int P, int C,
                                                       int G, int span_px, int spans) {
  extern __shared__ float red[];  // [blockDim][slots][4] float-float partial sums
  const int f = blockIdx.y;
  const int span = blockIdx.x;
  const int vpp = C >> 3;
  const int ppi = blockDim.x / vpp;
  const int tid = threadIdx.x;
  const int j = tid % vpp;
  const int lp = tid / vpp;
  const bool active = lp < ppi;
  const int cg = C / G;
  const int p0 = span * span_px;
  const int p1 = min(P, p0 + span_px);
  const size_t frame_off = (size_t)f * P * C;

  float2 s1h[4], s1l[4], s2h[4], s2l[4], sh[4];
  if (active && p0 < p1) {
    const wan_bf16* first = x + frame_off + (size_t)p0 * C;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int c0 = 8 * j + 2 * w;
      sh[w] = make_float2(bf16_at(first + (c0 / cg) * cg), bf16_at(first + ((c0 + 1) / cg) * cg));
    }
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    s1h[w] = s1l[w] = s2h[w] = s2l[w] = make_float2(0.f, 0.f);
  }
  if (active) {
    const char* base = reinterpret_cast<const char*>(x + frame_off) + (size_t)j * 16;
    const size_t pstride = (size_t)C * 2;
    int p = p0 + lp;
    constexpr int U = 4;
    for (; p + (U - 1) * ppi < p1; p += U * ppi) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = ldg_nc_v4(base + (size_t)(p + u * ppi) * pstride);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 xv = unpack2(wv[w]);
          const float2 d = __fadd2_rn(xv, make_float2(-sh[w].x, -sh[w].y));
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
        const float2 xv = unpack2(wv[w]);
        const float2 d = __fadd2_rn(xv, make_float2(-sh[w].x, -sh[w].y));
        two_sum2(s1h[w], s1l[w], d);
        fast_two_sum2(s2h[w], s2l[w], __fmul2_rn(d, d));
      }
    }
  }
  // Fold this thread's 8 channel partials by group. Channels of one group inside the vector
  // are consecutive; a vector holds 8/cg groups (cg < 8) or part of one group (cg >= 8).
  // red layout: per thread, per vector-group slot q (0 .. slots-1), four floats.
  const int slots = cg >= 8 ? 1 : 8 / cg;
  float* mine = red + (size_t)tid * slots * 4;
  for (int q = 0; q < slots; ++q) {
    float a_hi = 0.f, a_lo = 0.f, b_hi = 0.f, b_lo = 0.f;
    if (active) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int q_of_c = cg >= 8 ? 0 : c / cg;
        if (q_of_c != q) continue;
        const int w = c >> 1;
        const float h1 = (c & 1) ? s1h[w].y : s1h[w].x;
        const float l1 = (c & 1) ? s1l[w].y : s1l[w].x;
        const float h2 = (c & 1) ? s2h[w].y : s2h[w].x;
        const float l2 = (c & 1) ? s2l[w].y : s2l[w].x;
        ff_add(a_hi, a_lo, h1, l1);
        ff_add(b_hi, b_lo, h2, l2);
      }
    }
    mine[q * 4 + 0] = a_hi;
    mine[q * 4 + 1] = a_lo;
    mine[q * 4 + 2] = b_hi;
    mine[q * 4 + 3] = b_lo;
  }
  __syncthreads();
  // One thread per group sums the contributions of the threads holding it, in thread order.
  for (int g = tid; g < G; g += blockDim.x) {
    float a_hi = 0.f, a_lo = 0.f, b_hi = 0.f, b_lo = 0.f;
    const int c_first = g * cg;
    const int c_last = c_first + cg - 1;
    for (int jj = c_first / 8; jj <= c_last / 8; ++jj) {
      const int q = cg >= 8 ? 0 : (c_first % 8) / cg;
      for (int l = 0; l < ppi; ++l) {
        const float* r = red + ((size_t)(l * vpp + jj) * slots + q) * 4;
        ff_add(a_hi, a_lo, r[0], r[1]);
        ff_add(b_hi, b_lo, r[2], r[3]);
      }
    }
    GnPartial out;
    out.s1_hi = a_hi;
    out.s1_lo = a_lo;
    out.s2_hi = b_hi;
    out.s2_lo = b_lo;
    out.shift = p0 < p1 ? bf16_at(x + frame_off + (size_t)p0 * C + c_first) : 0.f;
    out.count = (p1 > p0 ? (p1 - p0) : 0) * cg;
    part[((size_t)f * spans + span) * G + g] = out;
  }
}

// Chan-Golub-LeVeque pairwise merge of (n, mean, M2) summaries in fp64.
struct Moments {
  double n, mean, m2;
};
__device__ __forceinline__ Moments merge(Moments a, Moments b) {
  if (b.n == 0.0) return a;
  if (a.n == 0.0) return b;
  const double n = a.n + b.n;
  const double delta = b.mean - a.mean;
  Moments r;
  r.n = n;
  r.mean = a.mean + delta * (b.n / n);
  r.m2 = a.m2 + b.m2 + delta * delta * (a.n * b.n / n);
  return r;
}

__global__ void __launch_bounds__(32) gn_finalize_kernel(const GnPartial* __restrict__ part,
                                                         const float* __restrict__ gamma,
                                                         const float* __restrict__ beta,
                                                         float4* __restrict__ coef, int C, int G,
                                                         int spans, float eps) {
  const int g = blockIdx.x;
  const int f = blockIdx.y;
  const int lane = threadIdx.x;
  const int cg = C / G;
  Moments acc = {0.0, 0.0, 0.0};
  for (int s = lane; s < spans; s += 32) {
    const GnPartial p = part[((size_t)f * spans + s) * G + g];
    if (p.count == 0) continue;
    const double n = (double)p.count;
    const double s1 = (double)p.s1_hi + (double)p.s1_lo;
    const double s2 = (double)p.s2_hi + (double)p.s2_lo;
    Moments m;
    m.n = n;
    m.mean = (double)p.shift + s1 / n;
    m.m2 = fmax(s2 - s1 * (s1 / n), 0.0);
    acc = merge(acc, m);
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {  // fixed butterfly order: deterministic
    Moments o;
    o.n = __shfl_xor_sync(0xffffffffu, acc.n, off);
    o.mean = __shfl_xor_sync(0xffffffffu, acc.mean, off);
    o.m2 = __shfl_xor_sync(0xffffffffu, acc.m2, off);
    acc = (lane & off) ? merge(o, acc) : merge(acc, o);
  }
  const double var = fmax(acc.m2 / acc.n, 0.0);
  const double rstd = 1.0 / sqrt(var + (double)eps);
  for (int k = lane; k < cg; k += 32) {
    const int c = g * cg + k;
    const double S = (double)gamma[c] * rstd;
    const double B = (double)beta[c] - acc.mean * S;
    const float sh = (float)S;
    const float bh = (float)B;
    coef[(size_t)f * C + c] = make_float4(sh, (float)(S - (double)sh), bh, (float)(B - (double)bh));
  }
}

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

__global__ void __launch_bounds__(256) gn_apply_kernel(const wan_bf16* __restrict__ x,
                                                       wan_bf16* __restrict__ y,
                                                       const float4* __restrict__ coef, int P,
                                                       int C, int span_px) {
  const int f = blockIdx.y;
  const int span = blockIdx.x;
  const int vpp = C >> 3;
  const int ppi = blockDim.x / vpp;
  const int tid = threadIdx.x;
  const int j = tid % vpp;
  const int lp = tid / vpp;
  if (lp >= ppi) return;
  const int p0 = span * span_px;
  const int p1 = min(P, p0 + span_px);
  float2 shi[4], slo[4], bhi[4], blo[4];
  const float4* cf = coef + (size_t)f * C + 8 * j;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 a = cf[2 * w], b = cf[2 * w + 1];
    shi[w] = make_float2(a.x, b.x);
    slo[w] = make_float2(a.y, b.y);
    bhi[w] = make_float2(a.z, b.z);
    blo[w] = make_float2(a.w, b.w);
  }
  const size_t frame_off = (size_t)f * P * C;
  const char* xb = reinterpret_cast<const char*>(x + frame_off) + (size_t)j * 16;
  char* yb = reinterpret_cast<char*>(y + frame_off) + (size_t)j * 16;
  const size_t pstride = (size_t)C * 2;
  int p = p0 + lp;
  constexpr int U = 4;
  for (; p < p1; p += U * ppi) {
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

struct GnPlan {
  int P, F, threads, ppi, span_px, spans;
  size_t part_bytes, coef_bytes;
};

GnPlan plan(int N, int T, int H, int W, int C, int G, int sms) {
  GnPlan pl;
  pl.P = H * W;
  pl.F = N * T;
  const int vpp = C / 8;
  pl.threads = (256 / vpp) * vpp;  // C <= 2048: vpp <= 256
  pl.ppi = pl.threads / vpp;
  // Spans per frame depend on the frame's geometry only (about 64 KB of x each), never on the
  // number of frames in the call: the statistics of a frame are then summed in the same order
  // whether the video comes in one call or in chunks, which keeps chunked runs bit-identical.
  (void)sms;
  const int px_bytes = C * 2;
  int span_px = (65536 / px_bytes) / pl.ppi * pl.ppi;
  if (span_px < pl.ppi) span_px = pl.ppi;
  const int whole = cdiv(pl.P, pl.ppi) * pl.ppi;
  if (span_px > whole) span_px = whole;
  pl.span_px = span_px;
  pl.spans = cdiv(pl.P, span_px);
  pl.part_bytes = (size_t)pl.F * pl.spans * G * sizeof(GnPartial);
  pl.coef_bytes = (size_t)pl.F * C * sizeof(float4);
  return pl;
}

inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t gn_silu_workspace(int N, int T, int H, int W, int C, int G, int sms) {
  const GnPlan pl = plan(N, T, H, W, C, G, sms);
  return align256(pl.part_bytes) + align256(pl.coef_bytes);
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
  const GnPlan pl = plan(N, T, H, W, C, G, sms);
  GnPartial* part = reinterpret_cast<GnPartial*>(ws);
  float4* coef = reinterpret_cast<float4*>(reinterpret_cast<char*>(ws) + align256(pl.part_bytes));
  const int cg = C / G;
  const size_t red_bytes = (size_t)pl.threads * (cg >= 8 ? 1 : 8 / cg) * 4 * sizeof(float);
  gn_stats_kernel<<<dim3(pl.spans, pl.F), pl.threads, red_bytes, stream>>>(x, part, pl.P, C, G,
                                                                          pl.span_px, pl.spans);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  gn_finalize_kernel<<<dim3(G, pl.F), 32, 0, stream>>>(part, gamma, beta, coef, C, G, pl.spans, eps);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  gn_apply_kernel<<<dim3(pl.spans, pl.F), pl.threads, 0, stream>>>(x, y, coef, pl.P, C, pl.span_px);
  return cudaGetLastError();
}

}  // namespace wan
