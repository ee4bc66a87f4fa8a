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
//     * x[t + kt - 2, r, p, ci] for the 128 pixels p of a column strip. The kernel runs on CTA
//     pairs (clusters of 2, tcgen05 .cta_group::2): each CTA owns one strip (M = 256 over the
//     pair) and keeps HALF of W' (56 of its 112 rows, 84 KB at Cin = 256) resident in shared
//     memory in the 128-byte swizzled K-major layout, built once straight from the weights. That
//     leaves room for an 8-deep TMA ring of input strips (one resident copy of all of W' would
//     leave room for 3, and the MMAs would wait on load latency). One thread of the even CTA
//     issues the M256 x N112 MMAs; the odd CTA's loads complete on the even CTA's barriers.
//   * Each pair owns (batch item, 4 output frames t .. t+3, two neighbouring 128-pixel strips,
//     band of image rows) and walks the rows of its band. Per row it loads the 6 input frames
//     t-2 .. t+3 once (1.5 input rows per output row instead of 3), and each input frame feeds the
//     accumulators of the output frames that use it (4 x 112 of the 512 TMEM columns, one barrier
//     pair per output frame), so one frame's epilogue runs while the MMAs of the others go on.
//     Two epilogue warpgroups take two frames each; a frame's epilogue applies the 3x3 stencil and
//     carries two partial output rows from one image row to the next.
// Reduction order per output is fixed (taps, then the 9 stencil terms), independent of the
// band/strip/pair placement and of chunking along T.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "tma_host.h"
#include "conv_tc.h"

namespace wan {

namespace {

constexpr int kCout = 12;
constexpr int kNP = 112;                 // 9 * 12 = 108 columns, padded to a multiple of 16
constexpr int kStripW = 128;             // pixels per strip (the MMA's M)
constexpr int kStripOut = kStripW - 2;   // outputs per strip
constexpr int kStages = 8;
constexpr int kThreads = 320;            // producer, MMA issuer, 2 epilogue warpgroups
constexpr int kABytes = kStripW * 128;   // one 64-channel slice of one image row strip
constexpr int kBRows = kNP / 2;            // W' rows held by each CTA of a pair
constexpr int kBBlockBytes = kBRows * 128;  // this CTA's rows of one 64-wide K block of W'
constexpr int kMaxKB = 12;               // 3 frames x (Cin <= 256) / 64
constexpr int kBOffset = kStages * kABytes;
constexpr int kBarOffset = kBOffset + kMaxKB * kBBlockBytes;
constexpr int kXchgOffset = kBarOffset + 256;
constexpr int kFrames = 4;               // output frames per item (4 x 112 of 512 TMEM columns)
constexpr int kFramesPerGroup = kFrames / 2;  // frames of an item per epilogue warpgroup
constexpr int kXchgBytes = 2 * 2 * 4 * 2 * 3 * kCout * 4;  // [group][parity][quarter][side][i][c]
constexpr int kSmemTotal = kXchgOffset + kXchgBytes + 1024;
constexpr int kTmemCols = 512;           // 4 frames x 112 columns = 448

struct HeadArgs {
  int N, T, H, W, Cin;
  int kb_per_frame;          // Cin / 64
  int quads, strips, strip_pairs, bands, band_rows, items;
  int order;                 // item order over the CTA pairs: 0 snake, 1 rotating (see item_of)
  int has_cache;
  const wan_bf16* w;         // [12, 3, 3, 3, Cin]
  const wan_bf16* bias;      // [12] or null
  const wan_bf16* residual;  // [N, T, H, W, 12] or null
  wan_bf16* y;               // [N, T, H, W, 12]
  unsigned* err;
};

struct Item {
  int n, t, w0, h0, h1;
  bool valid;  // false for the odd CTA of a pair when the strip count is odd
};

// item -> frame pair (fastest), band, pair of strips, batch item; `which` picks the strip of the
// pair (the even CTA takes the first).
__device__ __forceinline__ Item decode_item(const HeadArgs& a, int idx, int which) {
  Item it;
  const int quad = idx % a.quads;
  idx /= a.quads;
  const int band = idx % a.bands;
  idx /= a.bands;
  int strip = 2 * (idx % a.strip_pairs) + which;
  it.n = idx / a.strip_pairs;
  it.valid = strip < a.strips;
  if (!it.valid) strip = a.strips + 1;  // entirely right of the frame: its loads read zeros
  it.t = kFrames * quad;
  it.w0 = strip * kStripOut - 1;
  it.h0 = band * a.band_rows;
  it.h1 = min(a.H, it.h0 + a.band_rows);
  return it;
}

// Items of round r go to the P CTA pairs as a permutation of items r * P .. r * P + P - 1 (so the
// items running together share input frames in L2): snake order (pair c takes r * P + c, or
// r * P + P - 1 - c on odd rounds) or rotating order (r * P + (c + r) % P). The frame quad is the
// fastest index of an item and the quads differ in cost (the first quad of a chunk without
// history has fewer taps), so which order spreads them evenly depends on P; the launcher picks
// the better one. -1: no item left; -2: none in this last round.
__device__ __forceinline__ int item_of(const HeadArgs& a, int r, int cluster, int nclusters) {
  const int base = r * nclusters;
  if (base >= a.items) return -1;
  const int off = a.order ? (cluster + r) % nclusters : ((r & 1) ? nclusters - 1 - cluster : cluster);
  const int item = base + off;
  return item < a.items ? item : -2;
}

// Rows of G this item computes: the band plus one row on each side (inside the frame).
__device__ __forceinline__ int row_first(const Item& it) { return max(it.h0 - 1, 0); }
__device__ __forceinline__ int row_last(const HeadArgs& a, const Item& it) { return min(it.h1, a.H - 1); }

// Input frames of one row step: tau in [t-2, t+3] (up to the chunk's last frame); frames before
// the chunk without a cache read zeros and are skipped.
__device__ __forceinline__ int tau_first(const HeadArgs& a, const Item& it) {
  return a.has_cache ? it.t - 2 : max(it.t - 2, 0);
}
__device__ __forceinline__ int tau_last(const HeadArgs& a, const Item& it) {
  return min(it.t + kFrames - 1, a.T - 1);
}

// G columns of tap row i for this lane's pixel: g[j*12 + c] = G[p, (i*3 + j)*12 + c].
__device__ __forceinline__ void load_tap_row(uint32_t taddr, int i, float (&g)[36]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(g);
  const uint32_t a = taddr + i * 36;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(a));
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(a + 16));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35])
               : "r"(a + 32));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// One output pixel: 12 channels + bias (+ residual), rounded once to bf16, 24 bytes stored.
__device__ __forceinline__ void store_row(const HeadArgs& args, const float (&acc)[kCout], size_t pix) {
  float o[kCout];
#pragma unroll
  for (int c = 0; c < kCout; ++c) o[c] = acc[c] + (args.bias ? __uint_as_float(((uint32_t)args.bias[c]) << 16) : 0.f);
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

// Input frame U (tau = t - 2 + U) of an image row of an item of 4 output frames whose input frames
// t-2+U0 .. t+3 are present (U0 = 0: all of them; U0 = 2: the first quad of a chunk without
// history, whose frames before t read zeros and are skipped): it is tap kt = U - o of the output
// frames o in [max(U-2, 0), min(U, 3)], frame o is first written in the row at U = max(o, U0) (its
// accumulator released by the epilogue first), and frame U-2 sees its last input. Every burst
// size, frame, weight tap and barrier is a compile-time constant, so the issuing thread spends no
// time between bursts on bookkeeping: with run-time bookkeeping between input frames the tensor
// pipe idled 28% of the time (62.6 cycles per M256 x N112 MMA inside the bursts, 86.7 overall).
template <int KBPF, int U, int U0>
__device__ __forceinline__ bool head_full_tau(uint32_t tmem_base, uint32_t a_stage0, uint64_t b_desc0, uint64_t* full,
                                              uint64_t* empty, uint64_t* tmem_full, uint64_t* tmem_empty, int& grp,
                                              uint32_t& phase, uint32_t rc, unsigned* err) {
  constexpr uint32_t idesc = idesc_bf16_f32(256, kNP);
  constexpr uint64_t kBStep = kBBlockBytes >> 4;  // descriptor units between K blocks of W'
  constexpr int kGroups = kStages / KBPF;
  constexpr int o_lo = U - 2 > 0 ? U - 2 : 0, o_hi = U < kFrames - 1 ? U : kFrames - 1;
  if (!mbar_wait_cluster(&full[grp], phase, err, kDevErrTimeoutMma)) return false;
#pragma unroll
  for (int o = o_lo; o <= o_hi; ++o) {
    if ((o > U0 ? o : U0) == U) {  // first written in this row here
      if (!mbar_wait_cluster(&tmem_empty[o], (rc & 1) ^ 1, err, kDevErrTimeoutMma)) return false;
    }
  }
  tc_fence_after();
  const uint64_t a0 = smem_desc_sw128(a_stage0 + (uint32_t)(grp * KBPF * kABytes));
#pragma unroll
  for (int o = o_lo; o <= o_hi; ++o) {
    const int kt = U - o;
#pragma unroll
    for (int kb = 0; kb < KBPF; ++kb)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16_pair(tmem_base + o * kNP, a0 + (uint64_t)kb * (kABytes >> 4) + 2 * k,
                      b_desc0 + (uint64_t)(kt * KBPF + kb) * kBStep + 2 * k, idesc,
                      ((o > U0 ? o : U0) == U && kb == 0 && k == 0) ? 0u : 1u);
  }
  mma_commit_pair(&empty[grp], 0x3);
  if (++grp == kGroups) {
    grp = 0;
    phase ^= 1;
  }
  if (U >= 2) mma_commit_pair(&tmem_full[U - 2], 0x3);
  return true;
}

template <int KBPF>  // Cin / 64
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    head_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_cache,
                   const HeadArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;       // per output frame of the item
  uint64_t* tmem_empty = tmem_full + kFrames;  // per output frame, in the even CTA
  uint64_t* mma_done = tmem_empty + kFrames;
  uint64_t* xbar = mma_done + 1;  // edge-exchange barriers, one per epilogue warpgroup (128 threads)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 2);
  float* xchg = reinterpret_cast<float*>(smem + kXchgOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = 3 * KBPF;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  // W' -> shared memory, 128-byte swizzle (16-byte chunk j of row n stored at chunk j ^ (n & 7)).
  {
    const int chunks = KB * kBRows * 8;
    for (int q = threadIdx.x; q < chunks; q += blockDim.x) {
      const int jc = q & 7;
      const int nl = (q >> 3) % kBRows;  // row within this CTA's half
      const int kb = (q >> 3) / kBRows;
      const int n = (int)rank * kBRows + nl;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < 9 * kCout) {
        const int c = n % kCout, ij = n / kCout, i = ij / 3, j = ij % 3;
        const int k = kb * 64 + jc * 8;
        const int kt = k / args.Cin, ci = k % args.Cin;
        v = *reinterpret_cast<const uint4*>(args.w + ((((size_t)c * 3 + kt) * 3 + i) * 3 + j) * args.Cin + ci);
      }
      *reinterpret_cast<uint4*>(smem + kBOffset + kb * kBBlockBytes + nl * 128 + ((jc ^ (nl & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kFrames; ++s) {
      mbar_init(&tmem_full[s], 1);
      mbar_init(&tmem_empty[s], 8);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(mma_done, 1);
    mbar_init(&xbar[0], 128);
    mbar_init(&xbar[1], 128);
    fence_mbarrier_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_cache);
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

  // The ring holds kGroups groups of KBPF stages, one group per input frame tau: the KBPF tiles of
  // a tau are produced, waited for and released together (one barrier, one wait, one commit).
  constexpr int kGroups = kStages / KBPF;
  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    int grp = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int item = item_of(args, round, cluster, nclusters);
      if (item == -1) break;
      if (item < 0) continue;
      const Item it = decode_item(args, item, (int)rank);
      const int r1 = row_last(args, it);
      for (int r = row_first(it); ok && r <= r1; ++r) {
        for (int tau = tau_first(args, it); tau <= tau_last(args, it); ++tau) {
          if (!mbar_wait_cluster(&empty[grp], phase ^ 1, args.err, kDevErrTimeoutProducer)) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(&full[grp], 2 * KBPF * kABytes);  // both CTAs' tiles of this tau
            armed |= 1u << grp;
            armed_parity = (armed_parity & ~(1u << grp)) | (phase << grp);
          }
          const uint32_t bar = mapa_shared(smem_u32(&full[grp]), 0);  // the even CTA's barrier
#pragma unroll
          for (int kb = 0; kb < KBPF; ++kb) {
            uint8_t* dst = smem + (grp * KBPF + kb) * kABytes;
            if (tau < 0)
              tma_load_5d_pair(dst, &tm_cache, bar, kb * 64, it.w0, r, tau + 2, it.n);
            else
              tma_load_5d_pair(dst, &tm_a, bar, kb * 64, it.w0, r, tau, it.n);
          }
          // The ring holds only the next input frame; the one after it is pulled into L2 now so
          // that its loads, issued once a group frees up, do not wait for HBM.
          {
            int pr = r, pt = tau + 2;
            if (pt > tau_last(args, it)) {
              pt = tau_first(args, it) + (pt - tau_last(args, it) - 1);
              ++pr;
            }
            if (pr <= r1 && pt >= 0)
#pragma unroll
              for (int kb = 0; kb < KBPF; ++kb) tma_prefetch_5d(&tm_a, kb * 64, it.w0, pr, pt, it.n);
          }
          if (++grp == kGroups) {
            grp = 0;
            phase ^= 1;
          }
        }
      }
    }
    for (int s = 0; s < kStages; ++s)
      if (armed & (1u << s)) mbar_wait(&full[s], (armed_parity >> s) & 1, args.err, kDevErrTimeoutDrain);
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    // Per row: input frames tau ascending. The KBPF tiles of one input frame are waited for
    // together; then, for each output frame o the input frame is a tap of (kt = tau - (t+o) + 2
    // in 0..2), the 4 * KBPF MMAs into o's accumulator go out back to back with all descriptors
    // known in advance: the tensor pipe stays full only while MMAs follow each other directly,
    // so no address arithmetic or branch sits between two of them. Per accumulator the order
    // is tau, then K block, then K step. Frame o is complete after tau = t+o, and is first
    // written in a row only after the epilogue released it for that row.
    constexpr uint32_t idesc = idesc_bf16_f32(256, kNP);
    constexpr uint32_t kBStep = kBBlockBytes >> 4;  // descriptor units between K blocks of W'
    const uint32_t b_base = smem_u32(smem + kBOffset);
    int grp = 0;
    uint32_t phase = 0;
    uint32_t rc = 0;  // rows processed so far (parity of the per-frame TMEM barriers)
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int item = item_of(args, round, cluster, nclusters);
      if (item == -1) break;
      if (item < 0) continue;
      const Item it = decode_item(args, item, 0);
      const int nfr = min(kFrames, args.T - it.t);
      const int r1 = row_last(args, it);
      // Items of 4 output frames with all 6 input frames of a row (full) or with the last 4 (the
      // first quad of a chunk without history) take the compile-time rows below; a short last
      // quad takes the loop.
      const bool full_rows = nfr == kFrames && tau_first(args, it) == it.t - 2 && tau_last(args, it) == it.t + 3;
      const bool first_rows = nfr == kFrames && tau_first(args, it) == it.t && it.t == 0 && !args.has_cache &&
                              tau_last(args, it) == it.t + 3;
      for (int r = row_first(it); ok && r <= r1; ++r, ++rc) {
        if (first_rows) {
          const uint32_t a_stage0 = smem_u32(smem);
          const uint64_t bd = smem_desc_sw128(b_base);
          ok = head_full_tau<KBPF, 2, 2>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                         args.err) &&
               head_full_tau<KBPF, 3, 2>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                         args.err) &&
               head_full_tau<KBPF, 4, 2>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                         args.err) &&
               head_full_tau<KBPF, 5, 2>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                         args.err);
          continue;
        }
        if (full_rows) {
          const uint32_t a_stage0 = smem_u32(smem);
          const uint64_t bd = smem_desc_sw128(b_base);
          ok = head_full_tau<KBPF, 0, 0>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                      args.err) &&
               head_full_tau<KBPF, 1, 0>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                      args.err) &&
               head_full_tau<KBPF, 2, 0>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                      args.err) &&
               head_full_tau<KBPF, 3, 0>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                      args.err) &&
               head_full_tau<KBPF, 4, 0>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                      args.err) &&
               head_full_tau<KBPF, 5, 0>(tmem_base, a_stage0, bd, full, empty, tmem_full, tmem_empty, grp, phase, rc,
                                      args.err);
          continue;
        }
        uint32_t fresh = (1u << nfr) - 1;  // frames not yet written in this row
        for (int tau = tau_first(args, it); ok && tau <= tau_last(args, it); ++tau) {
          if (!mbar_wait_cluster(&full[grp], phase, args.err, kDevErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint64_t a_desc[KBPF];
#pragma unroll
          for (int kb = 0; kb < KBPF; ++kb) a_desc[kb] = smem_desc_sw128(smem_u32(smem + (grp * KBPF + kb) * kABytes));
          const int o_lo = max(tau - it.t, 0), o_hi = min(tau - it.t + 2, nfr - 1);
          // Frames written for the first time in this row wait until the epilogue released their
          // accumulator; then every MMA of this input frame goes out in one straight-line burst.
          uint32_t acc0[3];  // accumulate flag of each frame's first MMA (0: first write in the row)
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            const int o = o_lo + i;
            acc0[i] = 1u;
            if (o > o_hi || !((fresh >> o) & 1u)) continue;
            if (!mbar_wait_cluster(&tmem_empty[o], (rc & 1) ^ 1, args.err, kDevErrTimeoutMma)) ok = false;
            fresh &= ~(1u << o);
            acc0[i] = 0u;
          }
          if (!ok) break;
          tc_fence_after();
          const uint32_t d0 = tmem_base + o_lo * kNP;
          // W' block of kernel tap kt = tau - (t + o) + 2: one frame further is one tap lower.
          const uint64_t b0 = smem_desc_sw128(b_base + (tau - it.t - o_lo + 2) * KBPF * kBBlockBytes);
          constexpr uint64_t kTapDesc = (uint64_t)(KBPF * kBBlockBytes) >> 4;
          auto burst = [&](int i) {
#pragma unroll
            for (int kb = 0; kb < KBPF; ++kb)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16_pair(d0 + i * kNP, a_desc[kb] + 2 * k, b0 - i * kTapDesc + kb * kBStep + 2 * k, idesc,
                              (kb == 0 && k == 0) ? acc0[i] : 1u);
          };
          switch (o_hi - o_lo) {
            case 0:
              burst(0);
              break;
            case 1:
              burst(0);
              burst(1);
              break;
            default:
              burst(0);
              burst(1);
              burst(2);
              break;
          }
          if (!ok) break;
          mma_commit_pair(&empty[grp], 0x3);
          if (++grp == kGroups) {
            grp = 0;
            phase ^= 1;
          }
          const int done = tau - it.t;  // frame t+done has seen its last input (kt = 2)
          if (done >= 0 && done < nfr) mma_commit_pair(&tmem_full[done], 0x3);
        }
      }
    }
    mma_commit_pair(mma_done, 0x1);
    mbar_wait(mma_done, 0, args.err, kDevErrTimeoutDrain);
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- stencil epilogue
    // Two warpgroups; group g owns frames 2g and 2g+1 of every item. A warp may read only its
    // TMEM lane quarter (warp index mod 4), so each group covers the 128 pixels once.
    const int group = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int q = quarter * 32 + lane;  // pixel index within the strip
    uint64_t* gbar = &xbar[group];
    float* gx = xchg + group * (2 * 4 * 2 * 3 * kCout);
    uint32_t rc = 0;
    int parity = 0;
    uint32_t xphase = 0;
    bool ok = true;
    uint32_t leader_empty[kFramesPerGroup];
#pragma unroll
    for (int k = 0; k < kFramesPerGroup; ++k)
      leader_empty[k] = mapa_shared(smem_u32(&tmem_empty[group * kFramesPerGroup + k]), 0);
    for (int round = 0; ok; ++round) {
      const int item = item_of(args, round, cluster, nclusters);
      if (item == -1) break;
      if (item < 0) continue;
      const Item it = decode_item(args, item, (int)rank);
      const int nfr = min(kFrames, args.T - it.t);
      const int wcol = it.w0 + q;
      const bool col_ok = it.valid && q >= 1 && q <= kStripW - 2 && wcol >= 0 && wcol < args.W;
      // Partial outputs carried across rows: prev = row r-1, cur = row r (per frame of the group).
      float prev[kFramesPerGroup][kCout], cur[kFramesPerGroup][kCout];
#pragma unroll
      for (int k = 0; k < kFramesPerGroup; ++k)
#pragma unroll
        for (int c = 0; c < kCout; ++c) prev[k][c] = cur[k][c] = 0.f;
      const int r0 = row_first(it), r1 = row_last(args, it);
      for (int r = r0; r <= r1; ++r, ++rc) {
        const int ho = r - 1;  // output row completed by this row's G
#pragma unroll
        for (int k = 0; k < kFramesPerGroup; ++k) {
          const int f = group * kFramesPerGroup + k;
          if (f >= nfr) break;
          if (!mbar_wait_cluster(&tmem_full[f], rc & 1, args.err, kDevErrTimeoutEpilogue)) {
            ok = false;
            break;
          }
          tc_fence_after();
          float next[kCout];
          float* xw = gx + (parity * 4 + quarter) * 2 * 3 * kCout;  // [side][i][c]
          const uint32_t taddr = tmem_base + (uint32_t)(f * kNP) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            float g[36];
            __syncwarp();
            load_tap_row(taddr, i, g);
            float sv[kCout];
#pragma unroll
            for (int c = 0; c < kCout; ++c) {
              const float left = __shfl_up_sync(0xffffffffu, g[c], 1);        // G[p-1, (i,0,c)]
              const float right = __shfl_down_sync(0xffffffffu, g[24 + c], 1);  // G[p+1, (i,2,c)]
              sv[c] = ((lane > 0 ? left : 0.f) + g[12 + c]) + (lane < 31 ? right : 0.f);
            }
            // Warp-edge lanes publish what the neighbouring warp's edge lane is missing.
            if (lane == 31) {
#pragma unroll
              for (int c = 0; c < kCout; ++c) xw[(0 * 3 + i) * kCout + c] = g[c];
            }
            if (lane == 0) {
#pragma unroll
              for (int c = 0; c < kCout; ++c) xw[(1 * 3 + i) * kCout + c] = g[24 + c];
            }
#pragma unroll
            for (int c = 0; c < kCout; ++c) {
              if (i == 2) prev[k][c] += sv[c];
              else if (i == 1) cur[k][c] += sv[c];
              else next[c] = sv[c];
            }
          }
          // Frame f's accumulator is free for the next row: one arrival per warp, even CTA.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(leader_empty[k]);
          mbar_arrive(gbar);  // publishes this thread's edge values (release) ...
          if (!mbar_wait(gbar, xphase, args.err, kDevErrTimeoutEpilogue)) {  // ... and sees the others'
            ok = false;
            break;
          }
          xphase ^= 1;
          // Edge fix-ups: lane 0 adds G[p-1, (i,0,c)] from the previous quarter's lane 31,
          // lane 31 adds G[p+1, (i,2,c)] from the next quarter's lane 0.
          if ((lane == 0 && quarter > 0) || (lane == 31 && quarter < 3)) {
            const int nq = lane == 0 ? quarter - 1 : quarter + 1;
            const int side = lane == 0 ? 0 : 1;
            const float* xn = gx + (parity * 4 + nq) * 2 * 3 * kCout;
#pragma unroll
            for (int c = 0; c < kCout; ++c) {
              prev[k][c] += xn[(side * 3 + 2) * kCout + c];
              cur[k][c] += xn[(side * 3 + 1) * kCout + c];
              next[c] += xn[(side * 3 + 0) * kCout + c];
            }
          }
          parity ^= 1;
          if (col_ok && ho >= it.h0 && ho < it.h1)
            store_row(args, prev[k], (((size_t)it.n * args.T + it.t + f) * args.H + ho) * args.W + wcol);
#pragma unroll
          for (int c = 0; c < kCout; ++c) {
            prev[k][c] = cur[k][c];
            cur[k][c] = next[c];
          }
        }
        if (!ok) break;
      }
      if (!ok) break;
      // The last computed row was the frame's last row: its output row (r1) has no row below.
      if (r1 == args.H - 1 && col_ok && r1 >= it.h0 && r1 < it.h1) {
#pragma unroll
        for (int k = 0; k < kFramesPerGroup; ++k) {
          const int f = group * kFramesPerGroup + k;
          if (f >= nfr) break;
          store_row(args, prev[k], (((size_t)it.n * args.T + it.t + f) * args.H + r1) * args.W + wcol);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or arrivals may still touch it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

bool make_row_map(CUtensorMap* m, const void* base, int C, int W, int H, int T, int N) {
  auto fn = tensor_map_encoder();
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
  args.quads = cdiv(T, kFrames);
  args.strips = cdiv(W, kStripOut);
  args.strip_pairs = cdiv(args.strips, 2);
  args.has_cache = cache_in != nullptr;
  args.w = w;
  args.bias = bias;
  args.residual = residual;
  args.y = y;
  args.err = err;
  void (*kern)(const CUtensorMap, const CUtensorMap, const HeadArgs) = nullptr;
  switch (args.kb_per_frame) {
    case 1: kern = head_tc_kernel<1>; break;
    case 2: kern = head_tc_kernel<2>; break;
    case 3: kern = head_tc_kernel<3>; break;
    case 4: kern = head_tc_kernel<4>; break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
  if (e != cudaSuccess) return e;
  // CTA pairs the GPU can hold at once (a pair lives in one GPC).
  int slots = resident_pairs(reinterpret_cast<const void*>(kern), kThreads, kSmemTotal, sms);
  constexpr int kMaxSlots = 512;  // the per-pair load table below lives on the stack
  slots = std::max(1, std::min(slots, kMaxSlots));
  // Rows per band and item order. First the fewest rounds over the CTA pairs, counting the two halo
  // rows of a band; then, among band counts within 10% of that, the schedule whose busiest pair
  // has the least work, counting a quad's real taps (frames before a chunk without history have
  // none) and a band's real rows.
  const long long base = (long long)N * args.quads * args.strip_pairs;
  auto rounds_cost = [&](int bands) {
    const int rows = cdiv(H, bands);
    const long long items = base * cdiv(H, rows);
    return ((items + slots - 1) / slots) * (rows + 2);
  };
  long long min_cost = -1;
  for (int bands = 1; bands <= H && bands <= 256; ++bands) {
    const long long c = rounds_cost(bands);
    if (min_cost < 0 || c < min_cost) min_cost = c;
  }
  int quad_taps[64];
  for (int q = 0; q < args.quads && q < 64; ++q) {
    quad_taps[q] = 0;
    for (int o = 0; o < kFrames && kFrames * q + o < T; ++o)
      quad_taps[q] += args.has_cache ? 3 : std::min(3, kFrames * q + o + 1);
  }
  long long best_max = -1;
  int best_bands = 1, best_order = 0;
  long long load[kMaxSlots];
  for (int bands = 1; bands <= H && bands <= 256; ++bands) {
    if (rounds_cost(bands) * 10 > min_cost * 11) continue;
    const int rows = cdiv(H, bands);
    const int nb = cdiv(H, rows);
    const long long items = base * nb;
    for (int order = 0; order < 2; ++order) {
      std::fill(load, load + slots, 0LL);
      for (long long r = 0; r * slots < items; ++r)
        for (int c = 0; c < slots; ++c) {
          const long long off = order ? (c + r) % slots : ((r & 1) ? slots - 1 - c : c);
          const long long it = r * slots + off;
          if (it >= items) continue;
          const int q = (int)(it % args.quads), band = (int)((it / args.quads) % nb);
          const int h0 = band * rows, h1 = std::min(H, h0 + rows);
          const int nrows = std::min(h1, H - 1) - std::max(h0 - 1, 0) + 1;
          load[c] += (long long)nrows * (q < 64 ? quad_taps[q] : 3 * kFrames);
        }
      const long long mx = *std::max_element(load, load + slots);
      if (best_max < 0 || mx < best_max) {
        best_max = mx;
        best_bands = nb;
        best_order = order;
      }
    }
  }
  args.band_rows = cdiv(H, best_bands);
  args.bands = cdiv(H, args.band_rows);
  args.items = (int)(base * args.bands);
  args.order = best_order;

  CUtensorMap ta, tc;
  if (!make_row_map(&ta, a, Cin, W, H, T, N)) return cudaErrorInvalidValue;
  if (cache_in) {
    if (!make_row_map(&tc, cache_in, Cin, W, H, 2, N)) return cudaErrorInvalidValue;
  } else {
    tc = ta;
  }
  const int clusters = args.items < slots ? args.items : slots;
  kern<<<2 * clusters, kThreads, kSmemTotal, stream>>>(ta, tc, args);
  return cudaGetLastError();
}

}  // namespace wan
