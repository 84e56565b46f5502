// dq_gemm for wide m on the 5th-generation tensor cores (tcgen05), where the
// tile is a dense contraction: INT4 g128 at verify widths, BF16 and FP8-E4M3
// from m = 32 up.
//
// Source: "降低每個 Token 的生成成本" (Making each token cheaper), section
// "推測式解碼" (speculative decoding): verifying gamma + 1 positions per
// sequence multiplies the rows of the weight-only GEMM, and with INT4 weights
// the verify step turns compute-bound; sections "格式" (Formats) and "量化省下
// 什麼": weight-only INT4 and FP8 dequantise to 16-bit before the matrix
// arithmetic, FP8 with one fp32 scale per output channel.
//
// One CTA computes D[128 weight rows][N tokens] (N <= 256, a multiple of 16)
// over its k range (all of k, or one split of it), in 64-wide k slabs:
//  * warp 0 streams the weights with TMA. BF16: the 128 x 64 tile straight
//    into a 128-byte-swizzled K-major A slot. INT4: the packed codes of the
//    CTA's eight 16-row tiles (half of each 1 KB group block) and their group
//    scales into a ring of code slots. FP8: 128 x 128 code tiles (two slabs,
//    whole 128-byte rows) into a ring of code slots. Weights are constants: they are requested before the
//    wait on the preceding kernel;
//  * warp 1 streams the activation slab x[N tokens][64 k] with TMA as one
//    128-byte-swizzled box (rows past the ends arrive as zeros) into a ring of
//    about 128 KB (4 to 16 slabs deep, by N);
//  * warps 2-9 dequantise each code slab into the A slot, in two groups of
//    four taking alternate slabs: INT4 two 16-row tiles per warp,
//    deq = RN((q - z) * s) (the exact bf16 subtraction, then one rounded bf16
//    multiply; zero points prefetched a group ahead); FP8 eight codes per
//    16-byte row chunk, converted exactly to bf16 (the scale is applied to
//    the fp32 result);
//  * one thread each of warps 10 and 11 issues tcgen05.mma (M 128, N, K 16,
//    bf16 in, fp32 accumulate in tensor memory) for the even and the odd
//    slabs, into two accumulators, once both operands of a slab are in place,
//    and commits the slab's MMAs to the "empty" mbarriers of both slots;
//  * warps 2-9 read the accumulators back with tcgen05.ld (two warps per
//    32-lane quarter, splitting its columns), add them and write bf16 y, or with k
//    split, fp32 partials that the last-arriving CTA of the tile sums in
//    split order (deterministic).
// Every wait is bounded; tensor memory is released on every path.
#include "dqd_device.cuh"
#include "dqd_internal.h"
#include "rope_device.cuh"
#include "tcgen05.cuh"

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <type_traits>

namespace dqd {
namespace {

__device__ unsigned int g_tc_error;

constexpr int kRows = 128;    // weight rows per CTA (MMA M)
constexpr int kMaxN = 256;    // tokens per CTA at most (MMA N)
constexpr int kSlabK = 64;    // k per slab: one 128-byte swizzle row of bf16
constexpr int kABytes = kRows * kSlabK * 2;   // 16 KB
constexpr int kMaxASlots = 12;
constexpr int kMaxTSlots = 6;                 // A stages in tensor memory (64 columns each)
constexpr int kMaxBSlots = 16;
constexpr int kMaxCSlots = 12;
constexpr int kI4Codes = 8 * 512;             // INT4: 8 tiles x half a group block
constexpr int kI4Scales = 8 * 32;             // INT4: group scales of the 8 tiles
constexpr int kDeqWarps = 8;
constexpr int kDeq0 = 2;                      // first dequantising warp
constexpr int kMmaWarp = kDeq0 + kDeqWarps;  // first MMA-issuing warp
constexpr int kMmaWarps = 2;                  // MMA issuers: even and odd slabs
constexpr int kThreads = (kMmaWarp + kMmaWarps) * 32;
constexpr int kTmemCols = 512;                // all of an SM's tensor memory: one CTA per SM
constexpr int kAccCols = 256;                 // column offset of the odd slabs' accumulator
constexpr int kRingBytes = 222 * 1024;        // all rings
constexpr int kSmem = kRingBytes + 1024;      // + alignment slack
static_assert(kSmem + 1024 <= 227 * 1024, "shared memory");
static_assert(256 * kRows * 2 <= kRingBytes, "the fused RoPE epilogue stages up to 256 tokens x 128 rows of bf16 in the rings");

// Code slot bytes per weight type (INT4: codes + scales of one 64-k slab;
// FP8: a 128 x 128 code tile, two slabs, so that every row is one full
// 128-byte line; BF16 has none: its weight tiles land straight in the A slots).
// With A in tensor memory a code slot holds a 128-k stage: FP8 unchanged
// (a 128 x 128 tile), INT4 whole group blocks (both halves) and their scales.
__host__ __device__ constexpr int code_slot(int wt, bool atm = false) {
  return wt == kINT4 ? (atm ? 2 : 1) * kI4Codes + kI4Scales : (wt == kFP8 ? kRows * 2 * kSlabK : 0);
}

// Ring depths for N tokens per CTA: the activation ring gets about 64 KB
// (3 to 16 slabs: activations come from L2, where every CTA asks for the same
// lines at about the same time; 64 KB instead of 32 KB measured 4-12% faster
// at N = 64..128 and equal elsewhere); BF16 weight tiles take the rest
// (they stream from HBM, so they need the depth). Dequantised weights get up
// to eight A slots (the dequantise -> MMA -> release round trip spans the A
// ring), keeping room for a few code slots, and the code ring the rest.
//
// Both the A and the activation ring hold an even number of slots. The two
// MMA issuers take alternate slabs, so with an even ring each slot is only
// ever used by one issuer, which waits on its "full" barrier use after use.
// With an odd ring a slot alternates between the issuers, and the one running
// ahead can wait for use u + 1 of a slot whose use u has not landed yet: the
// barrier is then two phases behind, its parity matches, and the wait passes
// on stale data. It then commits early and the slot is refilled under copies
// still in flight. (A randomised model of the protocol shows such passes for
// every odd ring size and none for even ones.)
struct Rings {
  int nas, nbs, ncs;
};
// Tensor-memory columns of each accumulator when A lives in tensor memory
// (N tokens, rounded up to the 32-column reads of the epilogue).
__host__ __device__ constexpr int tc_acc_cols(int ntok) {
  return (ntok + 31) & ~31;
}
__host__ __device__ inline Rings rings(int wt, int ntok, bool atm = false) {
  const int bslot = ntok * kSlabK * 2;
  Rings r;
  if (atm) {
    // A in tensor memory, in stages of two slabs (128 k): the two
    // accumulators take the first columns, every A stage 64 columns (128 rows
    // x 128 k of bf16) of the rest; shared memory holds activation stages
    // (two slabs each, about 64 KB) and code slots (one stage each, the
    // rest). Every ring holds an even number of stages: the two issuers take
    // alternate stages, and so do the two dequantising groups, so each code
    // slot always serves the same group.
    r.nas = min(kMaxTSlots, (kTmemCols - 2 * tc_acc_cols(ntok)) / 64) & ~1;
    r.nbs = (min(kMaxBSlots, max(2, (64 * 1024) / (2 * bslot))) + 1) & ~1;
    r.ncs = min(kMaxCSlots, (kRingBytes - r.nbs * 2 * bslot) / code_slot(wt, true)) & ~1;
    return r;
  }
  r.nbs = (min(kMaxBSlots, max(3, (64 * 1024) / bslot)) + 1) & ~1;
  // keep room for four A slots and two code slots
  if (r.nbs > 2 && r.nbs * bslot + 4 * kABytes + 2 * code_slot(wt) > kRingBytes) r.nbs -= 2;
  const int rest = kRingBytes - r.nbs * bslot;
  if (wt == kBF16) {
    r.nas = min(kMaxASlots, rest / kABytes) & ~1;
    r.ncs = 0;
  } else {
    // INT4: even slot counts, so that slab i's slots (i % n) always serve the
    // same one of the two dequantising groups (which take alternate slabs)
    // and every waiter sees each phase of its slots' barriers. FP8 code
    // slots hold a slab pair, one slab for each group.
    const int min_codes = wt == kINT4 ? 8 : 3;  // at least ~32-48 KB of weights in flight
    r.nas = max(4, min(8, (rest - min_codes * code_slot(wt)) / kABytes)) & ~1;
    r.ncs = min(kMaxCSlots, (rest - r.nas * kABytes) / code_slot(wt));
    if (wt == kINT4) r.ncs &= ~1;
  }
  return r;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// 5-D tiled TMA load (the INT4 code blocks, reordered on the way in).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1, int c2,
                                            int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ void sts128(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// Named barrier over the dequantising / epilogue warps only.
__device__ __forceinline__ void deq_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDeqWarps * 32) : "memory");
}

struct TcArgs {
  const uint8_t* wz;     // INT4 packed zeros
  const float* wscale;   // FP8 per-row scales
  uint16_t* y;
  unsigned* counters;    // split-K tickets (splits > 1)
  float* part;           // split-K fp32 partials [split][m][n]
  int64_t m, n, k;
  int ntok;              // N: tokens per CTA
  int splits;
  int slabs_per_split;   // INT4 and FP8: even (splits fall on groups / code slots)
};

__device__ __forceinline__ float4 ldcg4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

// Last-arriving CTA of a split-K tile: y = bf16(sum of the split partials in
// split order) over the tile's rows [r0, r0 + rows) and tokens [m0, m0 + toks).
// Each thread keeps four outputs' partial loads of up to four splits in flight.
// ROPE: the four consecutive rows of a unit are two rotation pairs, stored
// through rope_store instead of y (n is a multiple of 128 there).
template <bool ROPE>
__device__ __forceinline__ bool reduce_splits(const TcArgs& a, int64_t r0, int rows, int64_t m0, int toks, int tid,
                                              int nthreads, const typename EpiOf<ROPE>::type& epi) {
  bool bad = false;
  const int64_t plane = a.m * a.n;
  const float* part = a.part;
  if ((a.n & 3) == 0) {
    const int per_tok = rows >> 2;  // rows is a multiple of 4 here
    const int units = per_tok * toks;
    for (int u0 = tid; u0 < units; u0 += 4 * nthreads) {
      float4 acc[4];
      int64_t off[4];
      bool live[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int u = u0 + q * nthreads;
        live[q] = u < units;
        off[q] = live[q] ? (m0 + u / per_tok) * a.n + r0 + 4 * (u % per_tok) : 0;
        acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int sp = 0; sp < a.splits; sp += 4) {
        float4 v[4][4];
#pragma unroll
        for (int d = 0; d < 4; ++d)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            v[d][q] = (live[q] && sp + d < a.splits) ? ldcg4(part + (sp + d) * plane + off[q])
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int d = 0; d < 4; ++d)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (sp + d < a.splits) {
              acc[q].x += v[d][q].x;
              acc[q].y += v[d][q].y;
              acc[q].z += v[d][q].z;
              acc[q].w += v[d][q].w;
            }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (live[q] && a.wscale) {
          const float4 sc = *reinterpret_cast<const float4*>(a.wscale + r0 + 4 * ((u0 + q * nthreads) % per_tok));
          acc[q].x *= sc.x;
          acc[q].y *= sc.y;
          acc[q].z *= sc.z;
          acc[q].w *= sc.w;
        }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (live[q]) {
          if constexpr (ROPE) {
            const int64_t mm = off[q] / a.n, nn = off[q] % a.n;
            const float b0 = bf16_round(acc[q].x), b1 = bf16_round(acc[q].y);
            const float b2 = bf16_round(acc[q].z), b3 = bf16_round(acc[q].w);
            bad |= rope_store(epi, mm, nn, b0, b1);
            bad |= rope_store(epi, mm, nn + 1, b1, b0);
            bad |= rope_store(epi, mm, nn + 2, b2, b3);
            bad |= rope_store(epi, mm, nn + 3, b3, b2);
          } else {
            uint2 o;
            o.x = pack_bf16x2(acc[q].x, acc[q].y);
            o.y = pack_bf16x2(acc[q].z, acc[q].w);
            *reinterpret_cast<uint2*>(a.y + off[q]) = o;
          }
        }
    }
  } else if constexpr (!ROPE) {
    const int units = rows * toks;
    for (int u = tid; u < units; u += nthreads) {
      const int64_t off = (m0 + u / rows) * a.n + r0 + u % rows;
      float acc = 0.f;
      for (int sp = 0; sp < a.splits; ++sp) acc += __ldcg(part + sp * plane + off);
      a.y[off] = f32_to_bf16(a.wscale ? acc * a.wscale[r0 + u % rows] : acc);
    }
  }
  return bad;
}

// ATM: A (the dequantised weights) in tensor memory, written by the
// dequantising warps with tcgen05.st (FP8, N <= 128); otherwise in shared memory.
template <int WT, bool ROPE, bool ATM>
__global__ void __launch_bounds__(kThreads, 1)
    dq_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                      const __grid_constant__ CUtensorMap tms, const TcArgs a,
                      const __grid_constant__ typename EpiOf<ROPE>::type epi) {
  constexpr int CSLOT = code_slot(WT, ATM);
  extern __shared__ uint8_t smem_raw[];
  constexpr int kMaxA = kMaxASlots > kMaxTSlots ? kMaxASlots : kMaxTSlots;
  __shared__ __align__(8) uint64_t bars[2 * kMaxCSlots + 2 * kMaxA + 2 * kMaxBSlots + 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int last_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Rings R = rings(WT, a.ntok, ATM);
  const uint32_t bslot_bytes = (uint32_t)a.ntok * kSlabK * 2;
  const int nbs = R.nbs, nas = R.nas, ncs = R.ncs;
  // tensor memory: accumulators at columns 0 and acc_off; with ATM the A
  // slots from column a_tcol on
  const uint32_t acc_off = ATM ? (uint32_t)tc_acc_cols(a.ntok) : (uint32_t)kAccCols;
  const uint32_t a_tcol = 2 * acc_off;
  const uint32_t aring = (smem_addr(smem_raw) + 1023u) & ~1023u;  // the ring memory (A slots first unless ATM)
  const uint32_t bring = aring + (ATM ? 0 : nas) * kABytes;
  const uint32_t bstage = (ATM ? 2 : 1) * bslot_bytes;  // activation bytes per stage (see SK below)
  const uint32_t cring = bring + nbs * bstage;
  const uint32_t cfull = smem_addr(&bars[0]), cempty = cfull + 8 * kMaxCSlots;
  const uint32_t afull = cempty + 8 * kMaxCSlots, aempty = afull + 8 * kMaxA;
  const uint32_t bfull = aempty + 8 * kMaxA, bempty = bfull + 8 * kMaxBSlots;
  const uint32_t done = bempty + 8 * kMaxBSlots;
  // blockIdx.x walks the token chunks fastest, so the CTAs that use the same
  // weight tile run together and share it through L2.
  const int64_t tile0 = (int64_t)blockIdx.y * 8;  // first 16-row tile
  const int64_t row0 = tile0 * 16;
  const int64_t ntiles = (a.n + 15) / 16;
  const int64_t m0 = (int64_t)blockIdx.x * a.ntok;
  const int nslabs = (int)((a.k + kSlabK - 1) / kSlabK);
  const int jb = (int)blockIdx.z * a.slabs_per_split;
  const int nl = min(nslabs - jb, a.slabs_per_split);  // slabs of this CTA (>= 1)
  // Pipeline stages: one slab, or with ATM two (128 k: one FP8 code slot).
  // An odd last slab (only in the last split: FP8 splits hold whole code
  // slots) is paired with a slab beyond k, which every copy fills with zeros.
  constexpr int SK = ATM ? 2 : 1;
  const int nu = (nl + SK - 1) / SK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < ncs; ++i) {
      mbar_init(cfull + 8 * i, 1);
      // INT4: one group of four warps per slot; FP8: both groups
      // one arrival per dequantising warp (lane 0, after __syncwarp): an FP8
      // code slot serves both groups, an INT4 one a single group
      mbar_init(cempty + 8 * i, (WT == kFP8 && !ATM) ? kDeqWarps : kDeqWarps / 2);
    }
    for (int i = 0; i < nas; ++i) {
      mbar_init(afull + 8 * i, WT == kBF16 ? 1 : kDeqWarps / 2);
      mbar_init(aempty + 8 * i, 1);
    }
    for (int i = 0; i < nbs; ++i) {
      mbar_init(bfull + 8 * i, 1);
      mbar_init(bempty + 8 * i, 1);
    }
    mbar_init(done, nu >= 2 ? kMmaWarps : 1);  // one commit per issuer that has stages
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(&tmem_base_sh), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  bool ok = true;

  // Slot cursors: slot index and the parity of its current use; a slot's
  // "empty" barrier is waited on with the opposite parity (its previous use).
  if (warp == 0) {
    // ---------------- weights (constants) ----------------
    if (lane == 0) {
      allow_dependent_launch();
      int cs = 0;
      uint32_t ph = 0;
      const int NSL = WT == kBF16 ? nas : ncs;
      const uint32_t empty = WT == kBF16 ? aempty : cempty, full = WT == kBF16 ? afull : cfull;
      const int step = (WT == kFP8 || ATM) ? 2 : 1;  // slabs per weight slot
      for (int i = 0, slot_i = 0; i < nl; i += step, ++slot_i) {
        const int j = jb + i;
        if (slot_i >= NSL && !mbar_wait(empty + 8 * cs, ph ^ 1u)) {
          atomicOr(&g_tc_error, kErrWaitTimeout);
          break;
        }
        const uint32_t fb = full + 8 * cs;
        if constexpr (WT == kBF16) {
          mbar_arrive_expect_tx(fb, kABytes);
          tma_load_2d(aring + cs * kABytes, &tmw, fb, j * kSlabK, (int)row0);
        } else if constexpr (WT == kFP8) {
          mbar_arrive_expect_tx(fb, CSLOT);  // slabs j, j + 1 (j even)
          tma_load_2d(cring + cs * CSLOT, &tmw, fb, j * kSlabK, (int)row0);
        } else if constexpr (ATM) {
          // a whole group (slabs j, j + 1; j even): both halves of the eight
          // tiles' blocks in one 5-D box that puts 16-byte chunk t of row r0 at
          // t * 128 + r0 * 16 (see the tensor map), then their scales
          const uint32_t dst = cring + cs * CSLOT;
          mbar_arrive_expect_tx(fb, CSLOT);
          tma_load_5d(dst, &tmw, fb, 0, 0, 0, j, (int)tile0);
          tma_load_2d(dst + 2 * kI4Codes, &tms, fb, (j >> 1) * 8, (int)tile0);
        } else {
          const uint32_t dst = cring + cs * CSLOT;
          mbar_arrive_expect_tx(fb, CSLOT);
          tma_load_2d(dst, &tmw, fb, j * 128, (int)tile0);
          tma_load_2d(dst + kI4Codes, &tms, fb, (j >> 1) * 8, (int)tile0);
        }
        if (++cs == NSL) {
          cs = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- activations ----------------
    if (lane == 0) {
      grid_dependency_wait();
      allow_dependent_launch();
      int s = 0;
      uint32_t ph = 0;
      for (int u = 0; u < nu; ++u) {
        if (u >= nbs && !mbar_wait(bempty + 8 * s, ph ^ 1u)) {
          atomicOr(&g_tc_error, kErrWaitTimeout);
          break;
        }
        mbar_arrive_expect_tx(bfull + 8 * s, bstage);
#pragma unroll
        for (int h = 0; h < SK; ++h)
          tma_load_2d(bring + s * bstage + h * bslot_bytes, &tmx, bfull + 8 * s, (jb + SK * u + h) * kSlabK, (int)m0);
        if (++s == nbs) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp < kMmaWarp) {
    grid_dependency_wait();
    allow_dependent_launch();
    // Two groups of four warps take alternate slabs (group 0 the even ones),
    // so that two slabs are dequantised at once and each warp has twice the
    // independent work between its barrier round trips. Slot cursors advance
    // by two slabs per iteration.
    const int grp = (warp - kDeq0) >> 2, gw = (warp - kDeq0) & 3;
    int cs = grp, s = grp;
    uint32_t cph = 0, sph = 0;
    auto advance = [&]() {
      if ((cs += 2) >= ncs) {
        cs -= ncs;
        cph ^= 1u;
      }
      if ((s += 2) >= nas) {
        s -= nas;
        sph ^= 1u;
      }
    };
    if constexpr (WT == kINT4 && ATM) {
      // ---------------- INT4, A in tensor memory ----------------
      // One weight row per thread (row r = 32 (w % 4) + t, the lanes warp w
      // may reach), one 128-k group per stage; group g takes stages g, g + 2.
      // In the packed block of row tile T, rows r0 and r0 + 8 (r0 = r % 8)
      // share 64 contiguous bytes per half-group, 16 words: word 4t + j holds
      // four k of both rows, k = 64 h + 32 (j >> 1) + 8 t + 4 (j & 1) + 0..3,
      // row r0 in nibbles 0, 4, 2, 6 (k + 0, + 1, + 2, + 3) and row r0 + 8 in
      // nibbles 1, 5, 3, 7. Shifting the word right by 4 for the upper row
      // puts (k, k + 1) in nibbles 0 and 4 and (k + 2, k + 3) in nibbles 2
      // and 6: two bf16x2 of 128 + q each with the 0x4300 magic, then the
      // exact subtraction of 128 + z and one rounded multiply by the scale.
      // The code slot holds tile tl's half h with its 16-byte chunk t of row
      // pair r0 at tl * 1024 + h * 512 + t * 128 + r0 * 16 (the TMA box
      // reorders rows and chunks), so the eight rows of a quarter-warp read
      // eight consecutive chunks: no bank conflicts.
      const int quarter = warp & 3;
      const int tl = quarter * 2 + (lane >> 4);  // row tile within the CTA
      const int r0 = lane & 7;
      const uint32_t shift = (lane & 8) ? 4u : 0u;
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16) + a_tcol;
      const int G = (int)(a.k / 128);
      const bool live = tile0 + tl < ntiles;
      const uint8_t* zp = a.wz + (tile0 + tl) * G * 8 + r0;  // zero byte of group gr at zp[8 gr]
      int gr = (jb >> 1) + grp;
      uint32_t znext = (live && gr < G) ? ldg_u8(zp + 8 * gr) : 0u;
      for (int u = grp; u < nu; u += 2) {
        const uint32_t zz = int4_zero_pair(znext >> shift);
        znext = (live && gr + 2 < G) ? ldg_u8(zp + 8 * (gr + 2)) : 0u;
        gr += 2;
        if (!__all_sync(0xffffffffu, mbar_wait(cfull + 8 * cs, cph))) {
          ok = false;
          break;
        }
        if (u >= nas && !__all_sync(0xffffffffu, mbar_wait(aempty + 8 * s, sph ^ 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read this stage's previous contents are complete
        const uint32_t slot = cring + cs * CSLOT;
        const uint32_t sw = lds32(slot + 2 * kI4Codes + tl * 32 + r0 * 4);
        const uint32_t ss = shift ? prmt(sw, 0u, 0x3232u) : prmt(sw, 0u, 0x1010u);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint4 w4 = lds128(slot + tl * 1024 + h * 512 + t * 128 + r0 * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t wv = word(w4, j) >> shift;
              const int c0 = 16 * (j >> 1) + 4 * t + 2 * (j & 1);
              v[c0] = bf16x2_mul(bf16x2_sub(and_or(wv, 0x000F000Fu, 0x43004300u), zz), ss);
              v[c0 + 1] = bf16x2_mul(bf16x2_sub(and_or(wv >> 8, 0x000F000Fu, 0x43004300u), zz), ss);
            }
          }
          tmem_st32(trow + (uint32_t)(s * 64 + h * 32), v);
        }
        tmem_wait_st();
        tc_fence_before();  // the stores are ordered before the arrival below
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(afull + 8 * s);
          mbar_arrive(cempty + 8 * cs);  // after the loaded codes and scales were used
        }
        advance();
      }
    } else if constexpr (WT == kINT4) {
      // ---------------- INT4: warp gw of a group owns 16-row tiles 2 gw, 2 gw + 1 ----------------
      // Group 0 dequantises the first 64-k half of every 128-k group, group 1
      // the second, so each iteration starts a new group: zero points are
      // fetched one iteration ahead.
      const int g = lane >> 2, t = lane & 3;
      const int G = (int)(a.k / 128);
      const uint8_t* zp[2];
      bool live[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int64_t tile = tile0 + 2 * gw + q;
        live[q] = tile < ntiles;
        zp[q] = a.wz + tile * G * 8 + g;  // zero byte of group gr at zp[q][8 gr]
      }
      int gr = (jb + grp) >> 1;
      uint32_t znext[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) znext[q] = (live[q] && gr < G) ? ldg_u8(zp[q] + 8 * gr) : 0u;
      // Lanes of odd g store their two 32-k halves in the opposite order, so
      // that each quarter-warp's 16-byte stores cover all 32 banks once.
      const uint32_t godd = g & 1;
      for (int i = grp; i < nl; i += 2) {
        uint32_t zcur[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          zcur[q] = znext[q];
          znext[q] = (live[q] && gr + 1 < G) ? ldg_u8(zp[q] + 8 * (gr + 1)) : 0u;
        }
        ++gr;
        if (!__all_sync(0xffffffffu, mbar_wait(cfull + 8 * cs, cph))) {  // warp-uniform: one arrival per warp
          ok = false;
          break;
        }
        uint4 u[2];
        uint32_t sc[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tt = 2 * gw + q;
          u[q] = lds128(cring + cs * CSLOT + tt * 512 + lane * 16);
          sc[q] = lds32(cring + cs * CSLOT + kI4Codes + tt * 32 + g * 4);
        }
        if (i >= nas && !__all_sync(0xffffffffu, mbar_wait(aempty + 8 * s, sph ^ 1u))) {
          ok = false;
          break;
        }
        const uint32_t base = aring + s * kABytes;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tt = 2 * gw + q;
          uint4 w = u[q];
          if (godd) {
            const uint32_t x0 = w.x, x1 = w.y;
            w.x = w.z;
            w.y = w.w;
            w.z = x0;
            w.w = x1;
          }
          const uint32_t slo = prmt(sc[q], 0u, 0x1010u), shi = prmt(sc[q], 0u, 0x3232u);
          const uint32_t zlo = int4_zero_pair(zcur[q]), zhi = int4_zero_pair(zcur[q] >> 4);
          const uint32_t row_lo = 2 * tt * 1024 + g * 128;  // row 16 tt + g; row + 8 is 1024 bytes on
          // words 2c, 2c+1 (after the swap) hold k = 32c' + 8t .. +7 of rows g
          // and g + 8, with c' = c ^ godd
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const Int4Frag f0 = int4_unpack(word(w, 2 * c), zlo, zhi);
            const Int4Frag f1 = int4_unpack(word(w, 2 * c + 1), zlo, zhi);
            const uint32_t a_lo = base + row_lo + (((4 * ((uint32_t)c ^ godd) + t) ^ g) << 4);
            sts128(a_lo, bf16x2_mul(f0.a0, slo), bf16x2_mul(f0.a2, slo), bf16x2_mul(f1.a0, slo),
                   bf16x2_mul(f1.a2, slo));
            sts128(a_lo + 1024, bf16x2_mul(f0.a1, shi), bf16x2_mul(f0.a3, shi), bf16x2_mul(f1.a1, shi),
                   bf16x2_mul(f1.a3, shi));
          }
        }
        // Every lane makes its generic-proxy stores visible to the tensor core;
        // after the warp has converged, lane 0 arrives for the warp (one
        // arrival per warp: per-lane arrivals on one barrier word serialise).
        // The code slot is released only now: an arrive does not wait for
        // shared loads still in flight, so it must follow the use of their
        // values, which every lane has made before the __syncwarp.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(afull + 8 * s);
          mbar_arrive(cempty + 8 * cs);
        }
        advance();
      }
    } else if constexpr (WT == kFP8 && ATM) {
      // ---------------- FP8, A in tensor memory ----------------
      // One weight row per thread: warp w may only reach tensor-memory lanes
      // 32 (w % 4) .. + 31, so thread t of warp w converts row 32 (w % 4) + t.
      // Group g takes stages g, g + 2, ...: each is one code slot, whose row
      // of 128 codes (eight 16-byte chunks, swizzled by row & 7, so that each
      // quarter-warp's loads of eight consecutive rows cover all 32 banks)
      // becomes the stage's 64 tensor-memory columns, with two tcgen05.st.
      // The code and A cursors (cs, s) start at the group's first stage and
      // advance by two stages: both rings hold an even number of them.
      const int quarter = warp & 3;
      const int r = quarter * 32 + lane;
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16) + a_tcol;
      for (int u = grp; u < nu; u += 2) {
        if (!__all_sync(0xffffffffu, mbar_wait(cfull + 8 * cs, cph))) {
          ok = false;
          break;
        }
        if (u >= nas && !__all_sync(0xffffffffu, mbar_wait(aempty + 8 * s, sph ^ 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read this stage's previous contents are complete
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint4 cw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            cw[j] = lds128(cring + cs * CSLOT + r * 128 + (((4 * h + j) ^ (r & 7)) << 4));
          uint32_t v[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[8 * j + 0] = fp8_lo_to_bf16x2(cw[j].x);
            v[8 * j + 1] = fp8_hi_to_bf16x2(cw[j].x);
            v[8 * j + 2] = fp8_lo_to_bf16x2(cw[j].y);
            v[8 * j + 3] = fp8_hi_to_bf16x2(cw[j].y);
            v[8 * j + 4] = fp8_lo_to_bf16x2(cw[j].z);
            v[8 * j + 5] = fp8_hi_to_bf16x2(cw[j].z);
            v[8 * j + 6] = fp8_lo_to_bf16x2(cw[j].w);
            v[8 * j + 7] = fp8_hi_to_bf16x2(cw[j].w);
          }
          tmem_st32(trow + (uint32_t)(s * 64 + h * 32), v);
        }
        tmem_wait_st();
        tc_fence_before();  // the stores are ordered before the arrival below
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(afull + 8 * s);
          mbar_arrive(cempty + 8 * cs);  // after the loaded codes were used
        }
        advance();
      }
    } else if constexpr (WT == kFP8) {
      // ---------------- FP8 ----------------
      // A code slot holds rows of 128 codes (slabs 2c, 2c + 1, 128-byte
      // swizzled); group h converts the h-th 64-code half of each row. Pass p:
      // thread d takes row 32 p + 8 (d >> 5) + 4 ((d >> 2) & 1) + ((d >> 3) & 3),
      // 16-code chunk d & 3: a quarter-warp reads rows r and r + 4, whose
      // swizzled chunks are disjoint, and the lanes of row r + 4 store their
      // odd 8-code chunk first, so loads and stores are free of conflicts.
      const int d = gw * 32 + lane, c4 = d & 3, rsel = (d >> 2) & 1;
      const int rbase = 8 * (d >> 5) + 4 * rsel + ((d >> 3) & 3);
      int ks = 0;
      uint32_t kph = 0;  // code slot cursor: one slot per slab pair
      for (int i = grp; i < nl; i += 2) {
        if (!__all_sync(0xffffffffu, mbar_wait(cfull + 8 * ks, kph))) {
          ok = false;
          break;
        }
        uint4 cw[4];
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
          const int r = 32 * pass + rbase;
          cw[pass] = lds128(cring + ks * CSLOT + r * 128 + (((4 * grp + c4) ^ (r & 7)) << 4));
        }
        if (i >= nas && !__all_sync(0xffffffffu, mbar_wait(aempty + 8 * s, sph ^ 1u))) {
          ok = false;
          break;
        }
        const uint32_t base = aring + s * kABytes;
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
          const int r = 32 * pass + rbase;
          const uint32_t rowb = base + (r >> 3) * 1024 + (r & 7) * 128;
          const uint32_t e0 = rowb + (((2 * c4) ^ (r & 7)) << 4), e1 = rowb + (((2 * c4 + 1) ^ (r & 7)) << 4);
          const uint32_t lo0 = fp8_lo_to_bf16x2(cw[pass].x), lo1 = fp8_hi_to_bf16x2(cw[pass].x);
          const uint32_t lo2 = fp8_lo_to_bf16x2(cw[pass].y), lo3 = fp8_hi_to_bf16x2(cw[pass].y);
          const uint32_t hi0 = fp8_lo_to_bf16x2(cw[pass].z), hi1 = fp8_hi_to_bf16x2(cw[pass].z);
          const uint32_t hi2 = fp8_lo_to_bf16x2(cw[pass].w), hi3 = fp8_hi_to_bf16x2(cw[pass].w);
          if (rsel) {
            sts128(e1, hi0, hi1, hi2, hi3);
            sts128(e0, lo0, lo1, lo2, lo3);
          } else {
            sts128(e0, lo0, lo1, lo2, lo3);
            sts128(e1, hi0, hi1, hi2, hi3);
          }
        }
        fence_proxy_async_smem();  // as for INT4: per-lane fence, one arrival per warp
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(afull + 8 * s);
          mbar_arrive(cempty + 8 * ks);  // after the loaded codes were used
        }
        if (++ks == ncs) {
          ks = 0;
          kph ^= 1u;
        }
        if ((s += 2) >= nas) {
          s -= nas;
          sph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) atomicOr(&g_tc_error, kErrWaitTimeout);
  } else {
    // ---------------- MMA issuers ----------------
    // One thread of each issuing warp: warp kMmaWarp takes the even slabs into
    // the accumulator at column 0, the next warp the odd slabs into the one at
    // column kAccCols; the epilogue adds the two. A single issuer spends some
    // 800-950 cycles per slab on its barrier checks, MMA issues and commits
    // (measured with per-slab clock stamps, with both operands long in place),
    // which caps a slab below the time HBM needs for its dequantised weights;
    // two issuers overlap those latencies.
    const int e = warp - kMmaWarp;
    if (lane == 0 && e < min(nu, kMmaWarps)) {
      const uint32_t idesc = idesc_bf16(kRows, a.ntok);
      const uint32_t acc = tmem + (uint32_t)e * acc_off;
      int sa = e, sb = e;  // slab i's slots i % nas, i % nbs and their parities, kept
      uint32_t pa = 0, pb = 0;  // incrementally (every ring holds an even number >= 2)
      for (int i = e; i < nu; i += kMmaWarps) {
        if (!mbar_wait(afull + 8 * sa, pa) || !mbar_wait(bfull + 8 * sb, pb)) {
          atomicOr(&g_tc_error, kErrWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t bbase = bring + sb * bstage;
        if constexpr (ATM) {
          // eight 16-k steps over the stage's two slabs: A 8 columns per step,
          // B 32 bytes per step within each slab's swizzled rows
          const uint32_t at = tmem + a_tcol + (uint32_t)(sa * 64);
#pragma unroll
          for (int kk = 0; kk < SK * kSlabK / 16; ++kk)
            umma_bf16_ta(acc, at + kk * 8, sw128_desc(bbase + (kk >> 2) * bslot_bytes + (kk & 3) * 32), idesc,
                         (i > e || kk > 0) ? 1u : 0u);
        } else {
          const uint32_t abase = aring + sa * kABytes;
#pragma unroll
          for (int kk = 0; kk < kSlabK / 16; ++kk)
            umma_bf16(acc, sw128_desc(abase + kk * 32), sw128_desc(bbase + kk * 32), idesc,
                      (i > e || kk > 0) ? 1u : 0u);
        }
        // both slots are free once these MMAs have read them
        umma_commit(aempty + 8 * sa);
        umma_commit(bempty + 8 * sb);
        if ((sa += kMmaWarps) >= nas) {
          sa -= nas;
          pa ^= 1u;
        }
        if ((sb += kMmaWarps) >= nbs) {
          sb -= nbs;
          pb ^= 1u;
        }
      }
      umma_commit(done);
    }
  }

  // ---------------- epilogue: warps w and w + 4 share lane quarter w % 4 ----------------
  if (warp >= kDeq0 && warp < kMmaWarp) {
    const int quarter = warp & 3;
    const int half = (warp - kDeq0) >> 2;
    const bool good = ok && mbar_wait(done, 0);
    if (!good && lane == 0) atomicOr(&g_tc_error, kErrWaitTimeout);
    __syncwarp();  // tcgen05.ld is warp-collective
    tc_fence_after();
    const int64_t row = row0 + quarter * 32 + lane;  // weight row = output column
    const int nchunks = (a.ntok + 31) / 32;
    float* part = a.splits > 1 ? a.part + (int64_t)blockIdx.z * a.m * a.n : nullptr;
    const float rscale = (WT == kFP8 && row < a.n) ? a.wscale[row] : 1.f;
    const bool two = nu >= 2;  // the second issuer's accumulator holds a sum
#pragma unroll 1
    for (int cc = half; cc < nchunks; cc += 2) {
      uint32_t r[32];
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + cc * 32;
      tmem_ld32(taddr, r);
      if (two) {
        uint32_t r2[32];
        tmem_ld32(taddr + acc_off, r2);
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
      }
      if (ROPE && !part) {
        // stage the projection's bf16 outputs, [token][128 rows of one head],
        // in the ring memory (free once `done` has fired); every warp of the
        // CTA then rotates and places them, four pairs per thread, after the
        // barrier below
#pragma unroll
        for (int j = 0; j < 32; ++j)
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(aring + (cc * 32 + j) * 256 + (quarter * 32 + lane) * 2),
                       "h"(f32_to_bf16(__uint_as_float(r[j]) * rscale))
                       : "memory");
      } else if (good && row < a.n) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int64_t mm = m0 + cc * 32 + j;
          if (cc * 32 + j < a.ntok && mm < a.m) {
            if (part)
              part[mm * a.n + row] = __uint_as_float(r[j]);
            else
              a.y[mm * a.n + row] = f32_to_bf16(__uint_as_float(r[j]) * rscale);
          }
        }
      }
    }
    if (a.splits > 1) {
      // publish the partials; the last CTA of this output tile reduces
      __threadfence();
      deq_barrier();
      unsigned* cnt = a.counters + (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
      if (warp == kDeq0 && lane == 0) last_sh = atomicAdd(cnt, 1u) == (unsigned)(a.splits - 1);
      deq_barrier();
      if (last_sh) {
        __threadfence();
        const int rows = (int)min((int64_t)kRows, a.n - row0);
        const int toks = (int)min((int64_t)a.ntok, a.m - m0);
        if (reduce_splits<ROPE>(a, row0, rows, m0, toks, threadIdx.x - kDeq0 * 32, kDeqWarps * 32, epi))
          atomicOr(&g_tc_error, kErrBadInput);
        if (warp == kDeq0 && lane == 0) *cnt = 0u;  // leave the ticket at zero for the next call
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (ROPE) {
    if (a.splits == 1) {
      // the CTA's 128 rows are one head (n is a multiple of 128); unit u is
      // eight dims of one token
      const int toks = (int)min((int64_t)a.ntok, a.m - m0);
      const int head = (int)(row0 >> 7);
      bool bad = false;
      for (int u = threadIdx.x; u < toks * 16; u += kThreads) {
        const int tl = u >> 4, ch = u & 15;
        const int64_t mm = m0 + tl;
        const uint4 x = lds128(aring + tl * 256 + ch * 16);
        bad |= rope_store8(epi, mm, (int)(mm / epi.w), (int)(mm % epi.w), head, ch * 8, x);
      }
      if (bad) atomicOr(&g_tc_error, kErrBadInput);
    }
  }
}

template <int WT, bool ROPE, bool ATM>
void* tc_kernel() {
  return reinterpret_cast<void*>(dq_gemm_tc_kernel<WT, ROPE, ATM>);
}

template <int WT, bool ATM, class E>
cudaError_t launch_tc(dim3 grid, size_t smem, cudaStream_t s, const CUtensorMap& tmx, const CUtensorMap& tmw,
                      const CUtensorMap& tms, const TcArgs& a, const E& epi) {
  constexpr bool ROPE = !std::is_same<E, NoEpi>::value;
  return launch_pdl(dq_gemm_tc_kernel<WT, ROPE, ATM>, grid, dim3(kThreads), smem, s, tmx, tmw, tms, a, epi);
}

}  // namespace

bool tc_supported(int wtype, int64_t m, int64_t n, int64_t k) {
  if (m > (int64_t)INT32_MAX || n <= 0 || (n + 127) / 128 > 65535 || k <= 0) return false;
  switch (wtype) {
    // INT4 and FP8 from m = 17, where the warp-MMA kernels need a third
    // m-tile and the tcgen05 kernel (A in tensor memory up to N = 64) runs at
    // a nearly flat cost. Measured against the warp-MMA kernels at m = 20..32:
    // FP8 faster on every 8B and 70B projection (70B gate+up 87.6 vs 139.4 us
    // at m = 20); INT4 faster on the 70B layer as a whole (m = 24: qkv + o +
    // gate+up + down 214 vs 242 us), within 10% behind on the 8B gate+up
    // (28672 x 4096: 40.4 vs 36.6 us). At m = 12..16 FP8 wins on the 70B
    // projections but loses on the 8B gate+up (38.9 vs 34.6 us), INT4 loses.
    case kINT4: return m >= 17 && k % 128 == 0 && k / 128 <= 65535;
    case kFP8: return m >= 17 && k % 16 == 0;
    // BF16 from m = 17, measured on the 8B and 70B projections against the
    // warp-MMA kernel with four m-tiles (m = 17..32): at m = 17, 70B
    // gate+up / down / qkv / o 144 / 79 / 39 / 27 us against 157 / 95 / 44 / 32.
    // Below that the warp-MMA kernels win or tie on nearly every shape (m = 16:
    // 4096 x 14336 down 22.6 vs 24.7 us); the 8B gate+up (28672 x 4096, 224
    // CTAs: a second wave half full) stays faster on them throughout (m = 32:
    // 46 vs 53 us).
    case kBF16: return m >= 17 && k % 8 == 0;
    default: return false;
  }
}

GemmPlan plan_dq_gemm_tc(int wtype, int64_t m, int64_t n, int64_t k, int num_sms) {
  GemmPlan p{};
  p.tc = 1;
  p.mt = 8;
  p.kc = kSlabK;
  p.slot_bytes = kABytes;
  p.smem_bytes = kSmem;
  p.grid_x = (int)((((n + 15) / 16) + 7) / 8);
  // Choose tokens per CTA (N, a multiple of 16 in [16, 256] covering m in
  // equal chunks) and the k split from a cost model: CTAs run in waves of one
  // per SM; a 64-wide slab costs its shared-memory traffic (weights in,
  // dequantised tile out and back to the tensor core, activations in and
  // back: about base + 2 N cycles; measured never below about 700 cycles, what
  // the two MMA issuers' barrier checks, MMA issues and commits take per slab
  // between them) or, with every SM
  // streaming, its share of HBM (weight bytes at about 21 bytes per SM
  // cycle), whichever is larger;
  // plus a fixed 6 slabs of fill, drain and epilogue; a split adds its fp32
  // partial traffic at about 6 TB/s.
  const int64_t nslabs = (k + kSlabK - 1) / kSlabK, sms = std::max(num_sms, 1);
  const int unit = wtype == kBF16 ? 1 : 2;  // INT4 splits on groups, FP8 on code slots (slab pairs)
  const int64_t units = (nslabs + unit - 1) / unit;
  const double base = wtype == kINT4 ? 330.0 : (wtype == kFP8 ? 380.0 : 260.0);
  const double wslab = wtype == kINT4 ? 4352.0 : (wtype == kFP8 ? 8192.0 : 16384.0);
  const char* env = std::getenv("DQD_GEMM_SPLITS");
  const long forced = env ? std::strtol(env, nullptr, 10) : 0;
  // Test hook: DQD_GEMM_TC_N caps the tokens per CTA (a multiple of 16), which
  // fixes N and with it the ring layout.
  const char* n_env = std::getenv("DQD_GEMM_TC_N");
  const long forced_n = n_env ? std::strtol(n_env, nullptr, 10) : 0;
  double best = -1.0;
  int64_t best_n = kMaxN, best_sp = 1;
  for (int64_t cap = kMaxN; cap >= 16; cap -= 16) {
    if (forced_n >= 16 && forced_n <= kMaxN && forced_n % 16 == 0 && cap != forced_n) continue;
    const int64_t chunks = (m + cap - 1) / cap;
    const int64_t ntok = ((m + chunks - 1) / chunks + 15) / 16 * 16;  // <= cap
    const int64_t ctas = chunks * p.grid_x;
    for (int64_t sp = 1; sp <= std::min<int64_t>(units, 32); ++sp) {
      if (sp > 1 && (ctas * sp > (int64_t)(kCounterBytes / 4) || units / sp < 2)) break;
      if (forced >= 1 && sp != std::min<int64_t>(forced, units)) continue;
      const int64_t per = (units + sp - 1) / sp * unit;  // slabs per split
      const double waves = (double)((ctas * sp + sms - 1) / sms);
      // with A in tensor memory (FP8, INT4 at N <= 64) a slab measured about
      // 480 (FP8) and 560 (INT4) cycles whatever N
      const bool atm_n = wtype != kBF16 && ntok <= 64;
      const double own = atm_n ? (wtype == kINT4 ? 560.0 : 480.0) : std::max(base + 2.0 * ntok, 700.0);
      const double slab = std::max(own, ctas * sp >= sms ? wslab / 21.0 : 0.0);
      double cycles = waves * (per + 6.0) * slab;
      if (sp > 1) cycles += 8.0 * sp * m * n / 6e12 * 1.9e9;
      if (best < 0 || cycles < best * 0.97) {
        best = cycles;
        best_n = ntok;
        best_sp = sp;
      }
    }
  }
  p.ra = (int)best_n;
  p.m_chunks = (int)((m + best_n - 1) / best_n);
  // FP8 with N <= 64 keeps A in tensor memory, in 128-k stages: the shared
  // memory then carries codes and activations only, and each MMA issuer
  // checks two barriers and commits twice per eight MMAs. (70B gate+up at
  // m = 32: 87.5 against 128.5 us; at N = 96..128 the MMAs bound both forms
  // equally.) Test hook: DQD_GEMM_TC_ATM=0 keeps A in shared memory, =1 uses
  // tensor memory up to N = 128.
  {
    const char* atm_env = std::getenv("DQD_GEMM_TC_ATM");
    const int cap = atm_env ? (atm_env[0] == '0' ? 0 : 128) : 64;
    p.tc_atm = (wtype != kBF16 && best_n <= cap) ? 1 : 0;
  }
  const int64_t per_units = (units + best_sp - 1) / best_sp;
  p.splits = (int)((units + per_units - 1) / per_units);
  p.k_per_split = per_units * unit * kSlabK;
  p.ws_bytes = p.splits > 1 ? kCounterBytes + sizeof(float) * (size_t)p.splits * m * n : 0;
  return p;
}

cudaError_t launch_dq_gemm_tc(const GemmLaunch& l, const GemmPlan& p, cudaStream_t s) {
  const int64_t ntiles = (l.n + 15) / 16;
  CUtensorMap tmx, tmw, tms;
  std::memset(&tms, 0, sizeof tms);
  {
    const uint64_t dims[2] = {(uint64_t)l.k, (uint64_t)l.m};
    const uint64_t strides[1] = {(uint64_t)l.k * 2};
    const uint32_t box[2] = {kSlabK, (uint32_t)p.ra};
    cudaError_t e =
        tensor_map(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, l.x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaSuccess;
  if (l.wtype == kBF16) {  // W [n][k] bf16, 128 x 64 tiles, swizzled as the tensor core reads them
    const uint64_t dims[2] = {(uint64_t)l.k, (uint64_t)l.n};
    const uint64_t strides[1] = {(uint64_t)l.k * 2};
    const uint32_t box[2] = {kSlabK, kRows};
    e = tensor_map(&tmw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, l.data, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else if (l.wtype == kFP8) {  // W [n][k] E4M3 codes, 128 x 128 tiles (full 128-byte rows), swizzled
    const uint64_t dims[2] = {(uint64_t)l.k, (uint64_t)l.n};
    const uint64_t strides[1] = {(uint64_t)l.k};
    const uint32_t box[2] = {2 * kSlabK, kRows};
    e = tensor_map(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, l.data, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const int64_t G = l.k / 128;
    if (p.tc_atm && p.ra <= 128) {
      // packed codes as 32-bit words, five dimensions: 4 words of a 16-byte
      // chunk, row pair r0 (8, 64 bytes apart), chunk t (4, 16 bytes apart),
      // half-group (2 G, 512 bytes apart), tile (ntiles, G KB apart); the box
      // {4, 8, 4, 2, 8} lands as [tile][half][t][r0][16 bytes]
      const uint64_t dims[5] = {4, 8, 4, (uint64_t)G * 2, (uint64_t)ntiles};
      const uint64_t strides[4] = {64, 16, 512, (uint64_t)G * 1024};
      const uint32_t box[5] = {4, 8, 4, 2, 8};
      e = tensor_map(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 5, l.data, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {  // packed codes as 32-bit words: [tile][G * 256]
      const uint64_t dims[2] = {(uint64_t)G * 256, (uint64_t)ntiles};
      const uint64_t strides[1] = {(uint64_t)G * 1024};
      const uint32_t box[2] = {128, 8};
      e = tensor_map(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, l.data, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (e == cudaSuccess) {  // packed scales as 32-bit words: [tile][G * 8]
      const uint64_t dims[2] = {(uint64_t)G * 8, (uint64_t)ntiles};
      const uint64_t strides[1] = {(uint64_t)G * 32};
      const uint32_t box[2] = {8, 8};
      e = tensor_map(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, l.scales, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
    }
  }
  if (e != cudaSuccess) return e;
  const bool atm = p.tc_atm != 0 && l.wtype != kBF16 && p.ra <= 128;
  {  // the two MMA issuers need even rings (see Rings)
    const Rings R = rings(l.wtype, (int)p.ra, atm);
    if (((R.nas | R.nbs) & 1) || R.nas < 2 || R.nbs < 2 || (l.wtype != kBF16 && R.ncs < 2))
      return cudaErrorInvalidValue;
  }
  static std::atomic<int> configured[64][12];
  int dev = 0;
  cudaGetDevice(&dev);
  const int wi = l.wtype == kBF16 ? 0 : (l.wtype == kFP8 ? 1 : 2);
  const bool rope = l.rope != nullptr;
  const int fi = wi + (rope ? 3 : 0) + (atm ? 6 : 0);
  if (dev < 0 || dev >= 64 || !configured[dev][fi].load(std::memory_order_relaxed)) {
    void* fn = nullptr;
    if (atm)
      fn = wi == 1 ? (rope ? tc_kernel<kFP8, true, true>() : tc_kernel<kFP8, false, true>())
                   : (rope ? tc_kernel<kINT4, true, true>() : tc_kernel<kINT4, false, true>());
    else if (rope)
      fn = wi == 0 ? tc_kernel<kBF16, true, false>()
                   : (wi == 1 ? tc_kernel<kFP8, true, false>() : tc_kernel<kINT4, true, false>());
    else
      fn = wi == 0 ? tc_kernel<kBF16, false, false>()
                   : (wi == 1 ? tc_kernel<kFP8, false, false>() : tc_kernel<kINT4, false, false>());
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev][fi].store(1, std::memory_order_relaxed);
  }
  TcArgs a;
  a.wz = static_cast<const uint8_t*>(l.zeros);
  a.wscale = l.wtype == kFP8 ? static_cast<const float*>(l.scales) : nullptr;
  a.y = l.y;
  a.counters = static_cast<unsigned*>(l.workspace);
  a.part = l.workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(l.workspace) + kCounterBytes) : nullptr;
  a.m = l.m;
  a.n = l.n;
  a.k = l.k;
  a.ntok = p.ra;
  a.splits = p.splits;
  a.slabs_per_split = (int)(p.k_per_split / kSlabK);
  const dim3 grid(p.m_chunks, p.grid_x, p.splits);
  const size_t smem = (size_t)p.smem_bytes;
  if (rope) {
    const RopeEpi& r = *l.rope;
    if (atm) return wi == 1 ? launch_tc<kFP8, true>(grid, smem, s, tmx, tmw, tms, a, r)
                            : launch_tc<kINT4, true>(grid, smem, s, tmx, tmw, tms, a, r);
    switch (wi) {
      case 0: return launch_tc<kBF16, false>(grid, smem, s, tmx, tmw, tms, a, r);
      case 1: return launch_tc<kFP8, false>(grid, smem, s, tmx, tmw, tms, a, r);
      default: return launch_tc<kINT4, false>(grid, smem, s, tmx, tmw, tms, a, r);
    }
  }
  const NoEpi none{};
  if (atm) return wi == 1 ? launch_tc<kFP8, true>(grid, smem, s, tmx, tmw, tms, a, none)
                          : launch_tc<kINT4, true>(grid, smem, s, tmx, tmw, tms, a, none);
  switch (wi) {
    case 0: return launch_tc<kBF16, false>(grid, smem, s, tmx, tmw, tms, a, none);
    case 1: return launch_tc<kFP8, false>(grid, smem, s, tmx, tmw, tms, a, none);
    default: return launch_tc<kINT4, false>(grid, smem, s, tmx, tmw, tms, a, none);
  }
}

cudaError_t tc_take_device_error(uint32_t* flags) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_tc_error, &zero, sizeof zero);
  *flags |= v;
  return e;
}

}  // namespace dqd
