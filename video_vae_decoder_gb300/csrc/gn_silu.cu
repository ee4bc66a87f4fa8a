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
//      x streams through shared memory: each CTA keeps three 32 KB pieces in flight with bulk async
//      copies (cp.async.bulk, completion on an mbarrier). Every thread owns one 16-byte
//      vector of 8 channels (so its groups are fixed) and accumulates, per channel, sum(d) and
//      sum(d^2) of d = x - s, where s is one value of the channel's group in the frame (its
//      first pixel). A thread first sums its run of up to 8 pixels of a piece in plain fp32
//      (d^2 by FMA), then adds each run sum into fp32 pairs (hi, lo): sum(d) with Knuth's
//      TwoSum, sum(d^2) (non-negative terms) with Dekker's Fast2Sum, two channels per packed
//      fp32x2 instruction. A run sum is exact unless the run mixes values about 12 binades apart.
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

#include <algorithm>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "conv_tc.h"
#include "gn_silu.h"
#include "winograd.h"

namespace wan {

namespace {

constexpr int kThreads = 256;

struct GnPartial {  // one (frame, span, group): float-float sums of d and d^2
  float s1_hi, s1_lo, s2_hi, s2_lo;
};

__device__ __forceinline__ void stg_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float bf16_at(const wan_bf16* p) { return __uint_as_float(((uint32_t)*p) << 16); }

// Grid-wide barrier for a cooperative launch (all CTAs co-resident). `ctr` counts arrivals
// over the whole call (cleared before the launch); barrier k waits for k * gridDim.x arrivals.
// The wait is bounded by `limit` SM cycles: on timeout it records kDevErrTimeoutGrid and returns
// false everywhere.
__device__ bool grid_barrier(unsigned* ctr, unsigned target, unsigned* err, int* s_flag, long long limit) {
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
      if (clock64() - start > limit) {
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
constexpr int kFinBatchSpans = 16; // the same for the span partials (one round of loads up to 512 spans)

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
  int cthreads;     // compute threads of a CTA (a multiple of C / 8); one more warp loads x
  float eps;
  double inv_len;   // 1 / (H * W * C / G)
  // Whole-clip statistics: 0 per frame; T: per (n, group) over the T frames of each n (F = N T).
  int clip_T;
  // Bound of the grid-barrier waits in SM cycles, and arrivals the first barrier waits for beyond
  // the grid's own: kWaitCycles and 0, except in the self-test of the timeout path, which sets a
  // short bound and a target the grid cannot reach.
  long long wait_cycles;
  unsigned bar_extra;
  int apply;  // 0: stop after the coefficients (phase B), the caller applies them elsewhere
  // 1: coefficients in the blocked layout (coef_blocked_index), for readers that take 8
  // consecutive channels per thread with 8 threads side by side (apply == 0 only).
  int coef_blocked;
};

// Pixel range [q0, q1) of piece j of statistics item `item` (empty past the end of a frame).
__device__ __forceinline__ void piece_range(const GnArgs& a, int item, int j, int& f, int& q0, int& q1) {
  f = item / a.spans;
  const int piece = (item - f * a.spans) * kPiecesPerSpan + j;
  q0 = min(a.P, piece * a.piece_px);
  q1 = min(a.P, q0 + a.piece_px);
}

// OR of `v` over the `nthreads` threads (a multiple of 32) that use named barrier `id`; the barrier
// also orders their shared-memory accesses like __syncthreads does.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kThreads + 32, 2) gn_silu_kernel(const GnArgs a) {
  extern __shared__ __align__(128) uint8_t gsm[];
  uint8_t* slots = gsm;                                                  // kSlots x piece bytes
  const int vpp = a.C >> 3;
  const int ct = a.cthreads;        // compute threads (a multiple of vpp); the last warp loads x
  const int cw = (ct + 31) >> 5;    // compute warps
  const int ppi = ct / vpp;
  const int piece_bytes = a.piece_px * a.C * 2;
  const int cg = a.C / a.G;
  const int nslot = cg >= 8 ? 1 : 8 / cg;
  float* red = reinterpret_cast<float*>(gsm + kSlots * piece_bytes);   // [2][32 cw][nslot][4]
  float4* s_coef = reinterpret_cast<float4*>(slots);  // [C], phase C only (the slots are idle then)
  __shared__ uint64_t full[kSlots], empty[kSlots];
  __shared__ uint64_t cbar;
  __shared__ int s_flag;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int j = tid % vpp;
  const int lp = tid / vpp;
  const bool active = lp < ppi;
  const int cnt = (a.items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // items of this CTA

  // The CTA's stream of pieces: its statistics items (item = blockIdx + k * grid), kPiecesPerSpan
  // pieces each; piece n is piece n % kPiecesPerSpan of the (n / kPiecesPerSpan)-th item. One
  // thread of the last warp issues them into kSlots slots; each compute warp releases a slot on
  // `empty` once it has read it, so warps never wait for one another while streaming.
  auto issue = [&](int n) {
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
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], cw);
    }
    fence_mbarrier_init();
    s_flag = 0;
  }
  __syncthreads();

  // ---------------------------------------------------------------- A: statistics
  if (warp == cw) {
    if (lane == 0) {
      const int npieces = cnt * kPiecesPerSpan;
      for (int n = 0; n < npieces; ++n) {
        if (n >= kSlots &&
            !mbar_wait(&empty[n % kSlots], (uint32_t)(((n / kSlots) - 1) & 1), a.err, kDevErrTimeoutGrid))
          break;  // the compute warps time out on the pieces that never come
        issue(n);
      }
    }
  } else if (cnt > 0) {
    int n = 0, buf = 0;  // next piece of the stream; reduction buffer of this item
    bool fail = false;
    for (int k = 0; k < cnt; ++k) {
      const int item = blockIdx.x + k * gridDim.x;
      const int f = item / a.spans, span = item - f * a.spans;
      // Each group's shift: its first value in the frame (a 2-byte load per group and thread; the
      // warp's loads fall in the frame's first pixel).
      const wan_bf16* xf = a.x + (size_t)f * a.P * a.C;
      float2 s1h[4], s1l[4], s2h[4], s2l[4], sh[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        s1h[w] = s1l[w] = s2h[w] = s2l[w] = make_float2(0.f, 0.f);
        const int c0 = 8 * j + 2 * w;
        sh[w] = active ? make_float2(bf16_at(xf + (size_t)(c0 / cg) * cg), bf16_at(xf + (size_t)((c0 + 1) / cg) * cg))
                       : make_float2(0.f, 0.f);
      }
      for (int pj = 0; pj < kPiecesPerSpan; ++pj, ++n) {
        const bool ok = !fail && mbar_wait(&full[n % kSlots], (uint32_t)((n / kSlots) & 1), a.err, kDevErrTimeoutGrid);
        fail = !ok;
        int f2, q0, q1;
        piece_range(a, item, pj, f2, q0, q1);
        if (ok && active) {
          // This thread's run of up to kVecPerThread pixels of the piece: plain fp32 sums of d
          // and d^2 over the run, then one error-free addition of each run sum into the span's
          // float-float accumulators. The deviations of nearby bf16 values carry few bits, so a
          // run sum is exact unless the run mixes values more than about 12 binades apart.
          const uint8_t* src = slots + (n % kSlots) * piece_bytes + (size_t)j * 16;
          float2 rs[4], rq[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) rs[w] = rq[w] = make_float2(0.f, 0.f);
          if (q1 - q0 == a.piece_px) {  // a whole piece: all loads first
            uint4 v[kVecPerThread];
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i)
              v[i] = *reinterpret_cast<const uint4*>(src + (size_t)(lp + i * ppi) * vpp * 16);
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i) {
              const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const float2 d = sub2(unpack2(wv[w]), sh[w]);
                rs[w] = __fadd2_rn(rs[w], d);
                rq[w] = __ffma2_rn(d, d, rq[w]);
              }
            }
          } else {
            for (int i = 0; i < kVecPerThread; ++i) {
              const int pl = lp + i * ppi;
              if (q0 + pl >= q1) break;
              const uint4 v = *reinterpret_cast<const uint4*>(src + (size_t)pl * vpp * 16);
              const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const float2 d = sub2(unpack2(wv[w]), sh[w]);
                rs[w] = __fadd2_rn(rs[w], d);
                rq[w] = __ffma2_rn(d, d, rq[w]);
              }
            }
          }
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            two_sum2(s1h[w], s1l[w], rs[w]);
            fast_two_sum2(s2h[w], s2l[w], rq[w]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[n % kSlots]);  // this warp is done with the slot
      }
      // Fold this thread's 8 channel partials by group slot (channels of a group are consecutive:
      // a vector holds 8/cg groups when cg < 8, else part of one group).
      float* rb = red + (size_t)buf * 32 * cw * nslot * 4;
      float* mine = rb + (size_t)tid * nslot * 4;
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
      // The compute warps only (the loading warp runs ahead on its own): the buffer is complete,
      // and whether any warp gave up a wait, so that all leave the loop at the same item.
      if (bar_red_or(1, 32 * cw, fail)) {
        fail = true;
        break;
      }
      // One thread per group adds the contributions of the threads holding it, in thread order.
      for (int g = tid; g < a.G; g += 32 * cw) {
        float ah = 0.f, al = 0.f, bh = 0.f, bl = 0.f;
        const int c_first = g * cg, c_last = c_first + cg - 1;
        const int q = cg >= 8 ? 0 : (c_first % 8) / cg;
        for (int jj = c_first / 8; jj <= c_last / 8; ++jj)
          for (int l = 0; l < ppi; ++l) {
            const float* r = rb + ((size_t)(l * vpp + jj) * nslot + q) * 4;
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
      buf ^= 1;  // the next item fills the other buffer; the one after waits for its barrier
    }
    if (fail && tid == 0) s_flag = 1;
  }
  __syncthreads();
  if (s_flag) return;  // a wait gave up (recorded in the error word): no coefficients from here
  if (!grid_barrier(a.bar, gridDim.x + a.bar_extra, a.err, &s_flag, a.wait_cycles)) return;

  // ---------------------------------------------------------------- B: finalize per (frame, group)
  {
    const int warps = blockDim.x >> 5, warp = tid >> 5, lane = tid & 31;
    // pair p -> CTA p % grid, warp (p / grid) % warps: the few pairs spread over many SMs.
    const int pairs = a.clip_T ? (a.F / a.clip_T) * a.G : a.F * a.G;
    for (int pr = warp * gridDim.x + blockIdx.x; pr < pairs; pr += gridDim.x * warps) {
      if (a.clip_T) {
        // Whole clip: each frame's span partials merged as below (fixed order), then moved exactly
        // from the frame's own shift s_t to frame 0's shift s, in float-float (dl = s_t - s by
        // TwoSum, n dl by an FMA product error):
        //   sum (x - s) = S1_t + n dl,  sum (x - s)^2 = S2_t + dl (2 S1_t + n dl),
        // and added in frame order. n = H W C/G per frame.
        const int nn = pr / a.G, g = pr - nn * a.G;
        const int f0 = nn * a.clip_T;
        const float s = bf16_at(a.x + (size_t)f0 * a.P * a.C + (size_t)g * cg);
        const float nf = (float)a.P * (float)cg;
        float h1 = 0.f, l1 = 0.f, h2 = 0.f, l2 = 0.f;
        for (int t = 0; t < a.clip_T; ++t) {
          const int f = f0 + t;
          const float4* src = reinterpret_cast<const float4*>(a.part) + ((size_t)f * a.G + g) * a.spans;
          float fh1 = 0.f, fl1 = 0.f, fh2 = 0.f, fl2 = 0.f;
          for (int sp0 = 0; sp0 < a.spans; sp0 += 32 * kFinBatch) {
            float4 q[kFinBatch];
#pragma unroll
            for (int i = 0; i < kFinBatch; ++i) {
              const int sp = sp0 + lane + 32 * i;
              q[i] = sp < a.spans ? __ldcg(src + sp) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < kFinBatch; ++i) {
              ff_add(fh1, fl1, q[i].x, q[i].y);
              ff_add(fh2, fl2, q[i].z, q[i].w);
            }
          }
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float oh1 = __shfl_xor_sync(0xffffffffu, fh1, off), ol1 = __shfl_xor_sync(0xffffffffu, fl1, off);
            const float oh2 = __shfl_xor_sync(0xffffffffu, fh2, off), ol2 = __shfl_xor_sync(0xffffffffu, fl2, off);
            ff_add(fh1, fl1, oh1, ol1);
            ff_add(fh2, fl2, oh2, ol2);
          }
          float dh = bf16_at(a.x + (size_t)f * a.P * a.C + (size_t)g * cg), dlo = 0.f;
          ff_add(dh, dlo, -s, 0.f);  // s_t - s exactly
          const float ph = nf * dh, pl = fmaf(nf, dh, -ph) + nf * dlo;
          ff_add(h1, l1, fh1, fl1);
          ff_add(h1, l1, ph, pl);
          float uh = 2.f * fh1, ul = 2.f * fl1;  // 2 S1_t + n dl
          ff_add(uh, ul, ph, pl);
          const float vh = dh * uh, vl = fmaf(dh, uh, -vh) + fmaf(dh, ul, dlo * uh);
          ff_add(h2, l2, fh2, fl2);
          ff_add(h2, l2, vh, vl);
        }
        const double s1 = (double)h1 + (double)l1;
        const double s2 = (double)h2 + (double)l2;
        const double m1 = s1 * a.inv_len;
        const double mean = (double)s + m1;
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
          const float4 cf = make_float4(shi, (float)(S - (double)shi), bhi, (float)(B - (double)bhi));
          for (int t = 0; t < a.clip_T; ++t)
            a.coef[(size_t)(f0 + t) * a.C + (a.coef_blocked ? coef_blocked_index(c) : c)] = cf;
        }
        continue;
      }
      const int f = pr / a.G, g = pr - f * a.G;
      // The lane's gamma and beta (and below, the group's shift) are loaded with the partials, not
      // after them: the finalize is a chain of round trips to L2, one of them instead of three.
      const float gam0 = lane < cg ? __ldg(a.gamma + g * cg + lane) : 0.f;
      const float bet0 = lane < cg ? __ldg(a.beta + g * cg + lane) : 0.f;
      // Float-float sums (fp64 issue is scarce on this GPU): lane-strided, then a butterfly.
      // The float-float add is commutative bit for bit (TwoSum's error term is unique), so every
      // lane ends with the same bits.
      // A lane adds items lane, lane + 32, ... in order, loading kFinBatch of them at a time.
      float h1 = 0.f, l1 = 0.f, h2 = 0.f, l2 = 0.f;
      const float4* src = reinterpret_cast<const float4*>(a.part) + ((size_t)f * a.G + g) * a.spans;
      const float sh = bf16_at(a.x + (size_t)f * a.P * a.C + (size_t)g * cg);
      for (int sp0 = 0; sp0 < a.spans; sp0 += 32 * kFinBatchSpans) {
        float4 q[kFinBatchSpans];
#pragma unroll
        for (int i = 0; i < kFinBatchSpans; ++i) {
          const int sp = sp0 + lane + 32 * i;
          q[i] = sp < a.spans ? __ldcg(src + sp) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kFinBatchSpans; ++i) {  // adding (0, 0) to a normalised pair changes nothing
          ff_add(h1, l1, q[i].x, q[i].y);
          ff_add(h2, l2, q[i].z, q[i].w);
        }
      }
      const double shift = (double)sh;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float oh1 = __shfl_xor_sync(0xffffffffu, h1, off), ol1 = __shfl_xor_sync(0xffffffffu, l1, off);
        const float oh2 = __shfl_xor_sync(0xffffffffu, h2, off), ol2 = __shfl_xor_sync(0xffffffffu, l2, off);
        ff_add(h1, l1, oh1, ol1);
        ff_add(h2, l2, oh2, ol2);
      }
      const double s1 = (double)h1 + (double)l1;
      const double s2 = (double)h2 + (double)l2;
      // fp64 division and square root are slow on this GPU: 1/L comes from the host and
      // 1/sqrt(v) is an fp32 estimate refined by two Newton steps r <- r (3 - v r^2) / 2 in fp64
      // (relative error 2^-22 -> 2^-44 -> below fp64 rounding).
      const double m1 = s1 * a.inv_len;
      const double mean = shift + m1;
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
        const double S = (double)(kk == lane ? gam0 : a.gamma[c]) * rstd;
        const double B = (double)(kk == lane ? bet0 : a.beta[c]) - mean * S;
        const float shi = (float)S, bhi = (float)B;
        a.coef[(size_t)f * a.C + (a.coef_blocked ? coef_blocked_index(c) : c)] =
            make_float4(shi, (float)(S - (double)shi), bhi, (float)(B - (double)bhi));
      }
    }
  }
  if (!a.apply) return;  // coefficients only
  if (!grid_barrier(a.bar, 2 * gridDim.x, a.err, &s_flag, a.wait_cycles)) return;

  // ---------------------------------------------------------------- C: apply, newest spans first
  // The coefficients reach shared memory with bulk copies (a per-thread load would send every
  // thread of the grid to the same few L2 lines): those of every frame at once when they fit the
  // idle slots (a CTA's successive spans usually lie in different frames), else the frame's as
  // the frame changes.
  const bool all_coef = (size_t)a.F * a.C * 16 <= (size_t)kSlots * piece_bytes;
  if (tid == 0) {
    mbar_init(&cbar, 1);
    fence_mbarrier_init();
    if (all_coef) {
      // Written by other CTAs with ordinary stores (ordered before the grid barrier); the copy
      // reads them through the async proxy.
      asm volatile("fence.proxy.async.global;" ::: "memory");
      mbar_arrive_expect_tx(&cbar, (uint32_t)a.F * a.C * 16u);
      bulk_load(s_coef, a.coef, (uint32_t)a.F * a.C * 16u, &cbar);
    }
  }
  __syncthreads();
  int fcur = -1;
  uint32_t cphase = 0;
  if (all_coef) {
    const bool okc = mbar_wait(&cbar, cphase, a.err, kDevErrTimeoutGrid);
    cphase ^= 1;
    if (__syncthreads_or(!okc)) return;
  }
  GnCoef8 k8;
  for (int k = 0; k < cnt; ++k) {
    const int item = a.items - 1 - (int)(blockIdx.x + k * gridDim.x);  // newest spans first
    const int f = item / a.spans;
    if (f != fcur && all_coef) {
      fcur = f;
      k8 = gn_coef8(s_coef + (size_t)f * a.C + 8 * j);
    } else if (f != fcur) {
      __syncthreads();  // the previous frame's coefficients have been read
      if (tid == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_expect_tx(&cbar, (uint32_t)a.C * 16u);
        bulk_load(s_coef, a.coef + (size_t)f * a.C, (uint32_t)a.C * 16u, &cbar);
      }
      const bool okc = mbar_wait(&cbar, cphase, a.err, kDevErrTimeoutGrid);
      cphase ^= 1;
      if (__syncthreads_or(!okc)) return;
      fcur = f;
      k8 = gn_coef8(s_coef + 8 * j);
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
          stg_v4(dst + (size_t)pp * vpp * 16, gn_silu8(v[u], k8));
        }
      }
    }
  }
}

// Coefficients from the statistics a conv emitted with its output (the pair conv's epilogue or the
// Winograd output transform; the same record layout): one CTA per (frame, group). Its threads take
// the group's records q = t, t + 256, ... in order, each moved exactly to record 0's shift s in
// float-float (dl = s_q - s by TwoSum, n dl by an FMA product error):
//   sum (x - s) = S1_q + n dl,  sum (x - s)^2 = S2_q + dl (2 S1_q + n dl),
// then the threads' pairs are added in a fixed order (warp butterflies, then the warps in turn)
// and the mean, variance and coefficients follow as in the norm's own finalize.
constexpr int kStatThreads = 256;
constexpr int kStatBatch = 8;  // records in flight per thread

__global__ void __launch_bounds__(kStatThreads) gn_coef_from_stats_kernel(const char* __restrict__ stats, int q_max,
                                                                          int q_a, int q_b, int q_c,
                                                                          const float* __restrict__ gamma,
                                                                          const float* __restrict__ beta, float4* coef,
                                                                          int F, int C, int G, double inv_len, float eps,
                                                                          int blocked, unsigned* err) {
  __shared__ float red[kStatThreads / 32][4];
  const int q = __ldcg(reinterpret_cast<const int*>(stats));
  if (q <= 0 || q > q_max || (q != q_a && q != q_b && q != q_c)) {  // not statistics of these sizes
    if (threadIdx.x == 0) atomicOr(err, kDevErrBadStats);
    return;
  }
  const int pr = blockIdx.x, f = pr / G, g = pr - f * G, cg = C / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float4* rec = reinterpret_cast<const float4*>(stats + kGnStatsHeader) + (size_t)pr * q;
  const float2* meta = reinterpret_cast<const float2*>(stats + kGnStatsHeader + (size_t)F * G * q * sizeof(float4)) +
                       (size_t)pr * q;
  const float gam0 = lane < cg ? __ldg(gamma + g * cg + lane) : 0.f;
  const float bet0 = lane < cg ? __ldg(beta + g * cg + lane) : 0.f;
  const float s = __ldcg(meta).x;
  float h1 = 0.f, l1 = 0.f, h2 = 0.f, l2 = 0.f;
  for (int q0 = 0; q0 < q; q0 += kStatThreads * kStatBatch) {
    float4 r[kStatBatch];
    float2 m[kStatBatch];
#pragma unroll
    for (int i = 0; i < kStatBatch; ++i) {
      const int k = q0 + (int)threadIdx.x + kStatThreads * i;
      r[i] = k < q ? __ldcg(rec + k) : make_float4(0.f, 0.f, 0.f, 0.f);
      m[i] = k < q ? __ldcg(meta + k) : make_float2(s, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kStatBatch; ++i) {
      float dh = m[i].x, dlo = 0.f;
      ff_add(dh, dlo, -s, 0.f);  // s_q - s exactly
      const float n = m[i].y;
      const float ph = n * dh, pl = fmaf(n, dh, -ph) + n * dlo;  // n dl (n < 2^24)
      ff_add(h1, l1, r[i].x, r[i].y);
      ff_add(h1, l1, ph, pl);
      float uh = 2.f * r[i].x, ul = 2.f * r[i].y;  // 2 S1_q + n dl
      ff_add(uh, ul, ph, pl);
      const float vh = dh * uh, vl = fmaf(dh, uh, -vh) + fmaf(dh, ul, dlo * uh);
      ff_add(h2, l2, r[i].z, r[i].w);
      ff_add(h2, l2, vh, vl);
    }
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float oh1 = __shfl_xor_sync(0xffffffffu, h1, off), ol1 = __shfl_xor_sync(0xffffffffu, l1, off);
    const float oh2 = __shfl_xor_sync(0xffffffffu, h2, off), ol2 = __shfl_xor_sync(0xffffffffu, l2, off);
    ff_add(h1, l1, oh1, ol1);
    ff_add(h2, l2, oh2, ol2);
  }
  if (lane == 0) {
    red[warp][0] = h1;
    red[warp][1] = l1;
    red[warp][2] = h2;
    red[warp][3] = l2;
  }
  __syncthreads();
  if (warp != 0) return;
  h1 = red[0][0], l1 = red[0][1], h2 = red[0][2], l2 = red[0][3];
  for (int w = 1; w < kStatThreads / 32; ++w) {
    ff_add(h1, l1, red[w][0], red[w][1]);
    ff_add(h2, l2, red[w][2], red[w][3]);
  }
  const double s1 = (double)h1 + (double)l1;
  const double s2 = (double)h2 + (double)l2;
  const double m1 = s1 * inv_len;
  const double mean = (double)s + m1;
  const double v = fmax(s2 * inv_len - m1 * m1, 0.0) + (double)eps;
  double rstd;
  if (v > 1e-30 && v < 1e30) {  // an fp32 estimate refined by two Newton steps in fp64
    rstd = (double)rsqrtf((float)v);
    rstd = rstd * (1.5 - 0.5 * v * rstd * rstd);
    rstd = rstd * (1.5 - 0.5 * v * rstd * rstd);
  } else {
    rstd = 1.0 / sqrt(v);
  }
  for (int kk = lane; kk < cg; kk += 32) {
    const int c = g * cg + kk;
    const double S = (double)(kk == lane ? gam0 : gamma[c]) * rstd;
    const double B = (double)(kk == lane ? bet0 : beta[c]) - mean * S;
    const float shi = (float)S, bhi = (float)B;
    coef[(size_t)f * C + (blocked ? coef_blocked_index(c) : c)] =
        make_float4(shi, (float)(S - (double)shi), bhi, (float)(B - (double)bhi));
  }
}

// The apply pass alone, on frames [t_lo, T) of every n, with the coefficients a coefficients-only
// call left in `coef` ([N*T][C], blocked layout): y[n, o + t - t_lo] (y has To frames per n)
// = silu(x[n, t] S + B). Items are (frame, run of px_per_item pixels); a thread owns one
// 16-byte channel vector and walks the run's pixels with kApplyUnroll loads in flight.
__global__ void __launch_bounds__(kThreads) gn_apply_frames_kernel(const wan_bf16* __restrict__ x,
                                                                   const float4* __restrict__ coef,
                                                                   wan_bf16* __restrict__ y, int T, int t_lo,
                                                                   int To, int o, int P, int C, int px_per_item,
                                                                   int items_per_frame, int items) {
  const int vpp = C >> 3, ppi = blockDim.x / vpp;
  const int j = threadIdx.x % vpp, lp = threadIdx.x / vpp;
  if (lp >= ppi) return;
  const int nt = T - t_lo;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int fi = item / items_per_frame, n = fi / nt, t = t_lo + fi % nt;
    const int q0 = (item - fi * items_per_frame) * px_per_item, q1 = min(P, q0 + px_per_item);
    const GnCoef8 k8 = gn_coef8_blocked(coef + (size_t)(n * T + t) * C + 8 * (j & ~7) + (j & 7));
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(n * T + t) * P * C) + j;
    char* dst = reinterpret_cast<char*>(y + (size_t)(n * To + o + t - t_lo) * P * C) + (size_t)j * 16;
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
        stg_v4(dst + (size_t)pp * vpp * 16, gn_silu8(v[u], k8));
      }
    }
  }
}

struct GnPlan {
  int P, F, threads, ppi, piece_px, spans, items, slots, launch_threads;
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
  const int cw = (pl.threads + 31) / 32;
  pl.smem = (size_t)kSlots * pl.piece_px * C * 2 + (size_t)2 * 32 * cw * pl.slots * 4 * sizeof(float);
  pl.launch_threads = 32 * (cw + 1);
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

const float4* gn_silu_coef(const void* ws, int N, int T, int H, int W, int C, int G) {
  const GnPlan pl = plan(N, T, H, W, C, G);
  return reinterpret_cast<const float4*>(reinterpret_cast<const char*>(ws) + align256(pl.part_bytes));
}

cudaError_t gn_apply_frames_launch(const wan_bf16* x, const float4* coef, wan_bf16* y, int N, int T, int H, int W,
                                   int C, int t_lo, int To, int o, int sms, cudaStream_t stream) {
  if (t_lo < 0 || t_lo >= T || o < 0 || o + (T - t_lo) > To || C % 8 != 0 || C > 2048) return cudaErrorInvalidValue;
  const int P = H * W, vpp = C / 8, threads = (kThreads / vpp) * vpp;
  const int px_per_item = max(1, 65536 / (C * 2));  // about 64 KB of x per item
  const int items_per_frame = cdiv(P, px_per_item);
  const long long items = (long long)N * (T - t_lo) * items_per_frame;
  if (items >= (1LL << 31)) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(items, (long long)sms * 8);
  gn_apply_frames_kernel<<<grid, threads, 0, stream>>>(x, coef, y, T, t_lo, To, o, P, C, px_per_item,
                                                       items_per_frame, (int)items);
  return cudaGetLastError();
}

cudaError_t gn_coef_from_stats_launch(const void* stats, size_t stats_bytes, const float* gamma, const float* beta,
                                      int N, int T, int H, int W, int C, int G, float eps, float4* coef, bool blocked,
                                      unsigned* err, cudaStream_t stream) {
  if (!stats || !coef || !err || G <= 0 || C % G != 0) return cudaErrorInvalidValue;
  const long long F = (long long)N * T;
  const long long pairs = F * G;
  if (pairs >= (1LL << 31) || stats_bytes < kGnStatsHeader) return cudaErrorInvalidValue;
  int q_a, q_b;  // the record counts of the two tilings the pair conv may have used
  conv_gn_stats_records(H, W, &q_a, &q_b);
  const int q_c = wino_gn_stats_records(H, W);  // and of the Winograd output transform
  const long long q_max = (long long)((stats_bytes - kGnStatsHeader) / ((size_t)pairs * (sizeof(float4) + sizeof(float2))));
  gn_coef_from_stats_kernel<<<(unsigned)pairs, kStatThreads, 0, stream>>>(
      static_cast<const char*>(stats), (int)std::min<long long>(q_max, 1 << 30), q_a, q_b, q_c, gamma, beta, coef, (int)F, C,
      G, 1.0 / ((double)H * W * (C / G)), eps, blocked ? 1 : 0, err);
  return cudaGetLastError();
}

cudaError_t gn_silu_launch(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta,
                           int N, int T, int H, int W, int C, int G, float eps, void* ws, int sms,
                           cudaStream_t stream, bool apply, float4* coef_out,
                           bool whole_clip, long long wait_cycles, unsigned bar_extra) {
  const GnPlan pl = plan(N, T, H, W, C, G);
  char* base = reinterpret_cast<char*>(ws);
  GnArgs a;
  a.x = x;
  a.y = y;
  a.gamma = gamma;
  a.beta = beta;
  a.part = reinterpret_cast<GnPartial*>(base);
  a.coef = coef_out ? coef_out : reinterpret_cast<float4*>(base + align256(pl.part_bytes));
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
  a.cthreads = pl.threads;
  a.eps = eps;
  a.clip_T = whole_clip ? T : 0;
  a.inv_len = 1.0 / ((double)pl.P * (C / G) * (whole_clip ? T : 1));
  a.wait_cycles = wait_cycles > 0 ? wait_cycles : kWaitCycles;
  a.bar_extra = bar_extra;
  a.apply = apply ? 1 : 0;
  a.coef_blocked = (!apply && C % 64 == 0) ? 1 : 0;
  // Persistent grid: every CTA resident at once (the cooperative launch checks it).
  cudaError_t e = cudaFuncSetAttribute(gn_silu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gn_silu_kernel, pl.launch_threads, pl.smem);
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
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(gn_silu_kernel), dim3(grid), dim3(pl.launch_threads),
                                     args, pl.smem, stream);
}

}  // namespace wan
