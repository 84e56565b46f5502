// dq_gemm: y[m][n] = sum_k x[m][k] * deq(W)[n][k] for small and mid m.
//
// Source: "降低每個 Token 的生成成本" (Making each token cheaper), section
// "量化省下什麼" (What quantisation saves): the decode kernel multiplies a
// quantised matrix by a full-precision vector and dequantises the weights on
// the fly; "LLM 推理是怎么变快的" §4.1: weight-only formats dequantise back to
// 16-bit, and decode time is weight bytes over bandwidth.
//
// Design (HBM-bound at decode m):
//  * Each warp owns one 16-row tile of W: the weights are the A operand of
//    mma.m16n8k16 ("swap-AB"), the m tokens its 8-column side. A CTA has 8
//    warps for m <= 16 (4 for wider m) that share the activation stage.
//  * W and x stream through a 3-stage cp.async ring in shared memory (one
//    barrier per stage), so the bytes in flight per SM are set by the ring,
//    not by registers. Rows past n, tokens past m and k past the end are
//    zero-filled by the copies themselves.
//  * Inside each 32-k (BF16/INT4) or 64-k (FP8) chunk, lane t owns a run of
//    8 (16) consecutive k for rows g and g+8, so one 16-byte shared load
//    feeds 2 (4) MMAs. The reduction index is thereby permuted inside the
//    chunk; x is read with the same permutation, so the sum is unchanged.
//    The 16-byte units of odd rows are XOR-swizzled so both operands' loads
//    are free of bank conflicts without padding.
//  * INT4: OR-ing a code into the mantissa of bf16 128.0 gives 128 + q
//    exactly and subtracting 128 + z in bf16 leaves q - z exactly, so the
//    group's fp32 MMA sum is sum x (q - z); the group scale multiplies it.
//    (A second MMA carrying the zero point would save three ALU operations
//    per eight weights, but mma.sync throughput on this part is the tighter
//    limit.) FP8: the E4M3 value is
//    built exactly in bf16; the row scale multiplies the fp32 total.
//  * Split-K when the n tiles alone cannot fill the GPU: each split writes
//    fp32 partials; the last CTA to arrive (atomic ticket, no waiting) sums
//    them in split order, so the result does not depend on arrival order.
#include "dqd_device.cuh"
#include "dqd_internal.h"
#include "rope_device.cuh"

#include <algorithm>
#include <atomic>
#include <cstdlib>

namespace dqd {
namespace {

constexpr int kStages = 3;

// Per-module device error word (kErrWaitTimeout when a bounded wait gave up).
__device__ unsigned int g_gemm_error;

__host__ __device__ constexpr int kc_base(int wt) { return wt == kBF16 ? 128 : (wt == kFP8 ? 256 : 512); }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int WT, int MT>
struct Cfg {
  static constexpr int WARPS = MT <= 2 ? 8 : 4;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int ROWS = 8 * MT;                        // activation rows per CTA pass
  static constexpr int KC = cmin(kc_base(WT), 8192 / ROWS);  // k per pipeline stage
  static constexpr int NG = KC / 128;                        // INT4 groups per stage
  static constexpr int ESZ = WT == kBF16 ? 2 : 1;            // bytes per BF16/FP8 weight
  static constexpr int WROWB = KC * ESZ;                     // bytes of one W row per stage
  static constexpr int WSTAGE = WT == kINT4 ? WARPS * NG * 1024 : WARPS * 16 * WROWB;
  static constexpr int MSTAGE = WT == kINT4 ? WARPS * NG * 48 : 0;  // INT4 scales + zeros
  static constexpr int XROWB = KC * 2;                       // bytes of one x row per stage
};

// XOR on the 16-byte unit index of row r (see the header comment).
template <int WT>
__device__ __forceinline__ int xswz(int r) { return WT == kFP8 ? (r & 1) : ((r & 1) << 2); }
__device__ __forceinline__ int wswz(int r) { return (r & 1) << 2; }

struct Args {
  const uint8_t* w;        // BF16 rows / FP8 rows / packed INT4 codes
  const uint8_t* ws;       // FP8 scales (f32) / packed INT4 scales
  const uint8_t* wz;       // packed INT4 zeros
  const uint16_t* x;
  uint16_t* y;
  float* part;             // [splits][m][n] fp32 (splits > 1)
  unsigned* counters;      // [m_chunks][grid_x]
  int64_t m, n, k;
  int64_t k_per_split;
  int splits;
  int cluster;             // splits reduce through distributed shared memory
  int ra;                  // activation rows held per stage (<= ROWS)
  int slot;                // bytes per ring slot
  int ns;                  // INT4: ring slots (2 or 3)
};

__device__ __forceinline__ void cp_async8(uint32_t saddr, const void* gptr, bool pred) {
  int n = pred ? 8 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(saddr), "l"(gptr), "r"(n) : "memory");
}

// Issue the weight copies of one k stage into one ring slot (no commit).
template <int WT, int MT>
__device__ __forceinline__ void issue_w(uint32_t slot, const Args& a, int64_t tile0, int64_t kst,
                                        int64_t kend) {
  using C = Cfg<WT, MT>;
  const int tid = threadIdx.x;
  if constexpr (WT != kINT4) {
    constexpr int UPR = C::WROWB / 16;
    constexpr int UNITS = C::WARPS * 16 * UPR;
    constexpr int EPU = 16 / C::ESZ;  // weights per 16-byte unit
#pragma unroll
    for (int i = 0; i < (UNITS + C::THREADS - 1) / C::THREADS; ++i) {
      const int u = tid + i * C::THREADS;
      if (UNITS % C::THREADS == 0 || u < UNITS) {
        const int r = u / UPR, cu = u % UPR;
        const int64_t row = tile0 * 16 + r, kk = kst + (int64_t)cu * EPU;
        const bool ok = row < a.n && kk < kend;
        const uint8_t* src = ok ? a.w + (row * a.k + kk) * C::ESZ : a.w;
        cp_async16(slot + r * C::WROWB + ((cu ^ wswz(r)) << 4), src, ok);
      }
    }
  } else {
    const int64_t G = a.k / 128, g0 = kst / 128, gend = kend / 128, NT = (a.n + 15) / 16;
    constexpr int UNITS = C::WARPS * C::NG * 64;
#pragma unroll
    for (int i = 0; i < UNITS / C::THREADS; ++i) {
      const int u = tid + i * C::THREADS;
      const int wi = u / (C::NG * 64), rem = u % (C::NG * 64), j = rem / 64, cu = rem % 64;
      const int64_t tile = tile0 + wi;
      const bool ok = tile < NT && g0 + j < gend;
      const uint8_t* src = ok ? a.w + (tile * G + g0 + j) * 1024 + cu * 16 : a.w;
      cp_async16(slot + (wi * C::NG + j) * 1024 + cu * 16, src, ok);
    }
    const uint32_t meta = slot + C::WSTAGE;
    for (int u = tid; u < C::WARPS * C::NG * 3; u += C::THREADS) {
      const int wi = u / (C::NG * 3), rem = u % (C::NG * 3), j = rem / 3, part = rem % 3;
      const int64_t tile = tile0 + wi;
      const bool ok = tile < NT && g0 + j < gend;
      const int64_t blk = tile * G + g0 + j;
      const uint32_t dst = meta + (wi * C::NG + j) * 48;
      if (part < 2)
        cp_async16(dst + part * 16, ok ? a.ws + blk * 32 + part * 16 : a.ws, ok);
      else
        cp_async8(dst + 32, ok ? a.wz + blk * 8 : a.wz, ok);
    }
  }
}

// Issue the activation copies of one k stage into one ring slot (no commit).
template <int WT, int MT>
__device__ __forceinline__ void issue_x(uint32_t slot, const Args& a, int64_t m0, int64_t kst, int64_t kend) {
  using C = Cfg<WT, MT>;
  const int tid = threadIdx.x;
  const uint32_t xbase = slot + C::WSTAGE + C::MSTAGE;
  constexpr int XUPR = C::XROWB / 16;
  for (int u = tid; u < a.ra * XUPR; u += C::THREADS) {
    const int r = u / XUPR, cu = u % XUPR;
    const int64_t mm = m0 + r, kk = kst + (int64_t)cu * 8;
    const bool ok = mm < a.m && kk < kend;
    cp_async16(xbase + r * C::XROWB + ((cu ^ xswz<WT>(r)) << 4), ok ? a.x + mm * a.k + kk : a.x, ok);
  }
}

__device__ __forceinline__ uint32_t lds8(uint32_t saddr) {
  uint16_t r;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(r) : "r"(saddr));
  return r;
}

// Activation row a lane reads for token column r of its MMA tiles: columns
// past the staged rows read row 0 instead of branching around the load (an
// MMA column depends only on its own B column, and those outputs are never
// stored), so no quarter-warp diverges at m < 8.
__device__ __forceinline__ int xrow(int r, int rows) { return r < rows ? r : 0; }

// One warp's MMAs for one stage. acc[j][*]: rows (g, g+8) x token columns
// (8j + 2t, 8j + 2t + 1). ngroups bounds the INT4 groups inside [kbeg, kend).
template <int WT, int MT>
__device__ __forceinline__ void compute_stage(float (&acc)[MT][4], uint32_t slot, int warp, int lane,
                                              int ra, int ngroups) {
  using C = Cfg<WT, MT>;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t xbase = slot + C::WSTAGE + C::MSTAGE;
  if constexpr (WT == kBF16) {
    const uint32_t wb = slot + warp * 16 * C::WROWB;
#pragma unroll
    for (int c = 0; c < C::KC / 32; ++c) {
      const int unit = 4 * c + t;
      const uint4 wa = lds128(wb + g * C::WROWB + ((unit ^ wswz(g)) << 4));
      const uint4 wc = lds128(wb + (g + 8) * C::WROWB + ((unit ^ wswz(g)) << 4));
      uint4 xv[MT];
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const int r = xrow(8 * j + g, ra);
        xv[j] = lds128(xbase + r * C::XROWB + ((unit ^ xswz<WT>(r)) << 4));
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
#pragma unroll
        for (int j = 0; j < MT; ++j)
          mma_bf16(acc[j], word(wa, 2 * e), word(wc, 2 * e), word(wa, 2 * e + 1), word(wc, 2 * e + 1),
                   word(xv[j], 2 * e), word(xv[j], 2 * e + 1));
      }
    }
  } else if constexpr (WT == kFP8) {
    const uint32_t wb = slot + warp * 16 * C::WROWB;
#pragma unroll
    for (int d = 0; d < C::KC / 64; ++d) {
      const int unit = 4 * d + t;
      const uint4 wa = lds128(wb + g * C::WROWB + ((unit ^ wswz(g)) << 4));
      const uint4 wc = lds128(wb + (g + 8) * C::WROWB + ((unit ^ wswz(g)) << 4));
      uint4 xa[MT], xb[MT];
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const int r = xrow(8 * j + g, ra);
        const int u0 = 8 * d + 2 * t;
        xa[j] = lds128(xbase + r * C::XROWB + ((u0 ^ xswz<WT>(r)) << 4));
        xb[j] = lds128(xbase + r * C::XROWB + (((u0 + 1) ^ xswz<WT>(r)) << 4));
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t ug = word(wa, e), uh = word(wc, e);
        const uint32_t a0 = fp8_lo_to_bf16x2(ug), a1 = fp8_lo_to_bf16x2(uh);
        const uint32_t a2 = fp8_hi_to_bf16x2(ug), a3 = fp8_hi_to_bf16x2(uh);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
          const uint4& xv = e < 2 ? xa[j] : xb[j];
          mma_bf16(acc[j], a0, a1, a2, a3, word(xv, 2 * (e & 1)), word(xv, 2 * (e & 1) + 1));
        }
      }
    }
  } else {
    const uint32_t wb = slot + warp * C::NG * 1024;
    const uint32_t meta = slot + C::WSTAGE + warp * C::NG * 48;
#pragma unroll
    for (int jg = 0; jg < C::NG; ++jg) {
      if (jg >= ngroups) break;  // past the end of k (warp-uniform)
      const uint32_t sc = lds32(meta + jg * 48 + g * 4);
      const uint32_t zr = lds8(meta + jg * 48 + 32 + g);
      const uint32_t zlo = int4_zero_pair(zr), zhi = int4_zero_pair(zr >> 4);
      const uint4 q0 = lds128(wb + jg * 1024 + lane * 16);
      const uint4 q1 = lds128(wb + jg * 1024 + 512 + lane * 16);
      float ga[MT][4];
#pragma unroll
      for (int j = 0; j < MT; ++j) ga[j][0] = ga[j][1] = ga[j][2] = ga[j][3] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 xv[MT];
#pragma unroll
        for (int j = 0; j < MT; ++j) {
          const int r = xrow(8 * j + g, ra);
          const int unit = 16 * jg + 4 * c + t;
          xv[j] = lds128(xbase + r * C::XROWB + ((unit ^ xswz<WT>(r)) << 4));
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = 2 * c + e;
          const Int4Frag f = int4_unpack(word(i < 4 ? q0 : q1, i & 3), zlo, zhi);
#pragma unroll
          for (int j = 0; j < MT; ++j)
            mma_bf16(ga[j], f.a0, f.a1, f.a2, f.a3, word(xv[j], 2 * e), word(xv[j], 2 * e + 1));
        }
      }
      const float slo = __uint_as_float(sc << 16), shi = __uint_as_float(sc & 0xFFFF0000u);
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        acc[j][0] = fmaf(slo, ga[j][0], acc[j][0]);
        acc[j][1] = fmaf(slo, ga[j][1], acc[j][1]);
        acc[j][2] = fmaf(shi, ga[j][2], acc[j][2]);
        acc[j][3] = fmaf(shi, ga[j][3], acc[j][3]);
      }
    }
  }
}

// Epilogue shared by the dq_gemm kernels (every thread of the CTA calls it):
// bf16 output, or fp32 split-K partials reduced by the last-arriving CTA.
// ROPE: the output is a QKV projection row per token (head dim 128, n a
// multiple of 16); instead of y, each bf16 output goes through rope_store
// with its rotation partner (column nn ^ 1, same token), which every path
// below has at hand: a lane 4 apart in the MMA fragment, or the pair a thread
// reduces itself.
template <int WT, int MT, int WARPS, int THREADS, bool ROPE>
__device__ __forceinline__ void finish(const Args& a, float (&acc)[MT][4], int64_t tile0, int64_t m0,
                                       bool tile_ok, const typename EpiOf<ROPE>::type& epi) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t tile = tile0 + warp;
  const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
  if (a.splits == 1) {
    if (!tile_ok) return;
    float s0 = 1.f, s1 = 1.f;
    if constexpr (WT == kFP8) {
      const float* sc = reinterpret_cast<const float*>(a.ws);
      s0 = r0 < a.n ? sc[r0] : 0.f;
      s1 = r1 < a.n ? sc[r1] : 0.f;
    }
    if constexpr (ROPE) {
      bool bad = false;
#pragma unroll
      for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t mm = m0 + 8 * j + 2 * t + (q & 1);
          const int64_t nn = (q & 2) ? r1 : r0;
          float v = acc[j][q];
          if constexpr (WT == kFP8) v *= (q & 2) ? s1 : s0;
          const float vb = bf16_round(v);
          const float partner = __shfl_xor_sync(0xffffffffu, vb, 4);  // row g ^ 1, same token
          if (mm < a.m && nn < a.n) bad |= rope_store(epi, mm, nn, vb, partner);
        }
      if (bad) atomicOr(&g_gemm_error, kErrBadInput);
    } else {
#pragma unroll
      for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t mm = m0 + 8 * j + 2 * t + (q & 1);
          const int64_t nn = (q & 2) ? r1 : r0;
          if (mm < a.m && nn < a.n) {
            float v = acc[j][q];
            if constexpr (WT == kFP8) v *= (q & 2) ? s1 : s0;
            a.y[mm * a.n + nn] = f32_to_bf16(v);
          }
        }
    }
    return;
  }
  if (a.cluster) {
    // split-K inside a thread-block cluster (the splits of this tile set, in
    // cluster rank order along y): every CTA stages its fp32 partial in its
    // own shared memory, column-major [token][tile row]; after a cluster
    // barrier, CTA r sums the r-th share of the valid outputs over the
    // cluster's CTAs in rank (= split) order, reading them through
    // distributed shared memory, and writes y. A second barrier keeps every
    // CTA alive until its partial has been read.
    constexpr int RT = WARPS * 16;          // tile rows of the CTA
    extern __shared__ __align__(128) uint8_t fin_smem[];
    float* stage = reinterpret_cast<float*>(fin_smem);
    __syncthreads();  // the ring is no longer read
    if (warp < WARPS) {
#pragma unroll
      for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          stage[(8 * j + 2 * t + (q & 1)) * RT + warp * 16 + g + 8 * (q >> 1)] = tile_ok ? acc[j][q] : 0.f;
    }
    cluster_sync_all();
    const int S = a.splits, rank = (int)blockIdx.y;
    const int cols = (int)min((int64_t)(8 * MT), a.m - m0);
    const uint32_t sbase = smem_addr(stage);
    if constexpr (ROPE) {
      // shares of whole (even row, odd row) pairs: a thread reduces both
      const int pv = cols * RT / 2, p0 = (int)((int64_t)rank * pv / S), p1 = (int)((int64_t)(rank + 1) * pv / S);
      bool bad = false;
      for (int pe = p0 + threadIdx.x; pe < p1; pe += THREADS) {
        const int e = 2 * pe, col = e / RT, rid = e % RT;
        const int64_t nn = tile0 * 16 + rid, mm = m0 + col;
        float v0 = 0.f, v1 = 0.f;
        for (int p = 0; p < S; ++p) {
          v0 += ld_dsmem_f32(sbase + 4u * (uint32_t)e, (uint32_t)p);
          v1 += ld_dsmem_f32(sbase + 4u * (uint32_t)(e + 1), (uint32_t)p);
        }
        if (nn < a.n) {
          if constexpr (WT == kFP8) {
            v0 *= reinterpret_cast<const float*>(a.ws)[nn];
            v1 *= reinterpret_cast<const float*>(a.ws)[nn + 1];
          }
          const float b0 = bf16_round(v0), b1 = bf16_round(v1);
          bad |= rope_store(epi, mm, nn, b0, b1);
          bad |= rope_store(epi, mm, nn + 1, b1, b0);
        }
      }
      if (bad) atomicOr(&g_gemm_error, kErrBadInput);
    } else {
      const int ev = cols * RT, e0 = (int)((int64_t)rank * ev / S), e1 = (int)((int64_t)(rank + 1) * ev / S);
      for (int e = e0 + threadIdx.x; e < e1; e += THREADS) {
        const int col = e / RT, rid = e % RT;
        const int64_t nn = tile0 * 16 + rid, mm = m0 + col;
        float v = 0.f;
        for (int p = 0; p < S; ++p) v += ld_dsmem_f32(sbase + 4u * (uint32_t)e, (uint32_t)p);
        if (nn < a.n) {
          if constexpr (WT == kFP8) v *= reinterpret_cast<const float*>(a.ws)[nn];
          a.y[mm * a.n + nn] = f32_to_bf16(v);
        }
      }
    }
    cluster_sync_all();
    return;
  }
  // split-K: publish fp32 partials, then the last-arriving CTA reduces.
  if (tile_ok) {
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t mm = m0 + 8 * j + 2 * t + (q & 1);
        const int64_t nn = (q & 2) ? r1 : r0;
        if (mm < a.m && nn < a.n) a.part[((int64_t)blockIdx.y * a.m + mm) * a.n + nn] = acc[j][q];
      }
  }
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  unsigned* cnt = a.counters + (int64_t)blockIdx.z * gridDim.x + blockIdx.x;
  if (threadIdx.x == 0) s_last = (atomicAdd(cnt, 1u) == (unsigned)(a.splits - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Cooperative reduction of the CTA's outputs: each thread owns whole outputs
  // and sums their split partials in split order (loads issued ahead of adds).
  const int64_t n0 = tile0 * 16;
  const int64_t S = a.splits, plane = a.m * a.n;
  if constexpr (ROPE) {
    // a thread owns the (even row, odd row) pair of one token
    bool bad = false;
    for (int e = threadIdx.x; e < WARPS * 8 * (8 * MT); e += THREADS) {
      const int64_t nn = n0 + 2 * (e / (8 * MT)), mm = m0 + e % (8 * MT);
      if (nn >= a.n || mm >= a.m) continue;
      const float* p = a.part + mm * a.n + nn;
      float v0 = 0.f, v1 = 0.f;
      for (int64_t sp = 0; sp < S; ++sp) {
        v0 += __ldcg(p + sp * plane);
        v1 += __ldcg(p + sp * plane + 1);
      }
      if constexpr (WT == kFP8) {
        v0 *= reinterpret_cast<const float*>(a.ws)[nn];
        v1 *= reinterpret_cast<const float*>(a.ws)[nn + 1];
      }
      const float b0 = bf16_round(v0), b1 = bf16_round(v1);
      bad |= rope_store(epi, mm, nn, b0, b1);
      bad |= rope_store(epi, mm, nn + 1, b1, b0);
    }
    if (bad) atomicOr(&g_gemm_error, kErrBadInput);
  } else {
    for (int e = threadIdx.x; e < WARPS * 16 * (8 * MT); e += THREADS) {
      const int64_t nn = n0 + e / (8 * MT), mm = m0 + e % (8 * MT);
      if (nn >= a.n || mm >= a.m) continue;
      const float* p = a.part + mm * a.n + nn;
      float sacc = 0.f;
      int64_t sp = 0;
      for (; sp + 4 <= S; sp += 4) {
        const float v0 = __ldcg(p + sp * plane), v1 = __ldcg(p + (sp + 1) * plane);
        const float v2 = __ldcg(p + (sp + 2) * plane), v3 = __ldcg(p + (sp + 3) * plane);
        sacc += v0;
        sacc += v1;
        sacc += v2;
        sacc += v3;
      }
      for (; sp < S; ++sp) sacc += __ldcg(p + sp * plane);
      if constexpr (WT == kFP8) sacc *= reinterpret_cast<const float*>(a.ws)[nn];
      a.y[mm * a.n + nn] = f32_to_bf16(sacc);
    }
  }
  if (threadIdx.x == 0) *cnt = 0u;  // leave the counter at zero for the next call
}

template <int WT, int MT, bool ROPE>
__global__ void __launch_bounds__(Cfg<WT, MT>::THREADS)
    dq_gemm_kernel(const Args a, const __grid_constant__ typename EpiOf<ROPE>::type epi) {
  using C = Cfg<WT, MT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tile0 = (int64_t)blockIdx.x * C::WARPS;
  const int64_t tile = tile0 + warp;
  const int64_t ntiles = (a.n + 15) / 16;
  const bool tile_ok = tile < ntiles;
  const int64_t m0 = (int64_t)blockIdx.z * C::ROWS;
  const int64_t kbeg = (int64_t)blockIdx.y * a.k_per_split;
  const int64_t kend = min(a.k, kbeg + a.k_per_split);
  const int nst = kend > kbeg ? (int)((kend - kbeg + C::KC - 1) / C::KC) : 0;
  const uint32_t ring = smem_addr(smem);

  float acc[MT][4];
#pragma unroll
  for (int j = 0; j < MT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  // Weights are constant: their first stages are fetched before waiting for
  // the preceding kernel; activations (and every write) come after the wait.
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s)
    if (s < nst) issue_w<WT, MT>(ring + s * a.slot, a, tile0, kbeg + (int64_t)s * C::KC, kend);
  grid_dependency_wait();
  allow_dependent_launch();
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nst) issue_x<WT, MT>(ring + s * a.slot, a, m0, kbeg + (int64_t)s * C::KC, kend);
    cp_async_commit();
  }
  for (int s = 0; s < nst; ++s) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    const int sn = s + kStages - 1;
    if (sn < nst) {
      const uint32_t slot = ring + (sn % kStages) * a.slot;
      issue_w<WT, MT>(slot, a, tile0, kbeg + (int64_t)sn * C::KC, kend);
      issue_x<WT, MT>(slot, a, m0, kbeg + (int64_t)sn * C::KC, kend);
    }
    cp_async_commit();
    if (tile_ok) {
      const int64_t kst = kbeg + (int64_t)s * C::KC;
      compute_stage<WT, MT>(acc, ring + (s % kStages) * a.slot, warp, lane, a.ra,
                            (int)((kend - kst + 127) / 128));
    }
  }
  cp_async_wait<0>();

  finish<WT, MT, C::WARPS, C::THREADS, ROPE>(a, acc, tile0, m0, tile_ok, epi);
}

// ------------------------------------------------------------------------
// INT4 g128, warp-specialised: WARPS consumer warps (one 16-row tile each)
// and one producer warp that moves each k stage with bulk asynchronous copies
// (the packed codes and scales of a tile are contiguous per stage, and so is
// each activation row), completing on a per-slot mbarrier. Consumers release
// a slot through a second mbarrier; nobody touches copy addressing except the
// producer. Zero points travel with the stage when their 8-byte blocks form
// 16-byte-aligned runs (an even number of groups in k and per stage);
// otherwise they are read with ordinary loads one stage ahead.
template <int MT, int W>
struct Int4Cfg {
  static constexpr int WARPS = W;  // consumer warps: 8 or 4 for m <= 16, 4 beyond
  static constexpr int THREADS = (WARPS + 1) * 32;
  static constexpr int ROWS = 8 * MT;
  static constexpr int KC = cmin(512, 8192 / ROWS);
  static constexpr int NG = KC / 128;
  static constexpr int NS_MAX = 3;                           // ring slots: 2 or 3, set per call
  static constexpr int CODES = WARPS * NG * 1024;
  static constexpr int SCALES = WARPS * NG * 32;
  static constexpr int ZEROS = WARPS * NG * 8;               // staged when their copies align
  static constexpr int META = SCALES + ZEROS;
  static constexpr int XSTR = KC * 2 + 64;                    // padded activation row
};

template <int MT, int W, bool ROPE>
__global__ void __launch_bounds__(Int4Cfg<MT, W>::THREADS)
    dq_gemm_int4_kernel(const Args a, const __grid_constant__ typename EpiOf<ROPE>::type epi) {
  using C = Int4Cfg<MT, W>;
  const int NS = a.ns;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2 * C::NS_MAX];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t tile0 = (int64_t)blockIdx.x * C::WARPS;
  const int64_t ntiles = (a.n + 15) / 16;
  const bool consumer = warp < C::WARPS;
  const int64_t tile = tile0 + warp;
  const bool tile_ok = consumer && tile < ntiles;
  const int64_t m0 = (int64_t)blockIdx.z * C::ROWS;
  const int64_t kbeg = (int64_t)blockIdx.y * a.k_per_split;
  const int64_t kend = min(a.k, kbeg + a.k_per_split);
  const int nst = kend > kbeg ? (int)((kend - kbeg + C::KC - 1) / C::KC) : 0;
  const int rows_valid = (int)min((int64_t)a.ra, a.m - m0);
  const int64_t G = a.k / 128;
  // Zero-point blocks of a tile's stage groups form a 16-byte-aligned run
  // when G and the groups per stage are even (stages start at even groups).
  const bool zbulk = (G % 2 == 0) && (C::NG % 2 == 0);
  const uint32_t ring = smem_addr(smem);
  const uint32_t full0 = smem_addr(&bars[0]), empty0 = smem_addr(&bars[C::NS_MAX]);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, C::WARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();

  float acc[MT][4];
#pragma unroll
  for (int j = 0; j < MT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  bool ok = true;

  if (!consumer) {
    // ---------------- producer warp ----------------
    auto stage_groups = [&](int s) { return (int)min((int64_t)C::NG, (kend - kbeg) / 128 - (int64_t)s * C::NG); };
    auto stage_bytes = [&](int s) {
      const int ng = stage_groups(s);
      int nt = (int)min((int64_t)C::WARPS, ntiles - tile0);
      return (uint32_t)(nt * ng * (1024 + 32 + (zbulk ? 8 : 0)) + rows_valid * ng * 256);
    };
    // lane w < WARPS copies tile w's codes and scales; lanes >= 16 copy activation rows
    auto issue_w = [&](int s) {
      const uint32_t slot = ring + (s % NS) * a.slot, fb = full0 + 8 * (s % NS);
      const int ng = stage_groups(s);
      if (lane == 0) mbar_arrive_expect_tx(fb, stage_bytes(s));
      __syncwarp();
      const int64_t g0 = (kbeg + (int64_t)s * C::KC) / 128;
      if (lane < C::WARPS && tile0 + lane < ntiles) {
        const int64_t blk = (tile0 + lane) * G + g0;
        bulk_load(slot + lane * C::NG * 1024, a.w + blk * 1024, ng * 1024, fb);
        bulk_load(slot + C::CODES + lane * C::NG * 32, a.ws + blk * 32, ng * 32, fb);
        if (zbulk) bulk_load(slot + C::CODES + C::SCALES + lane * C::NG * 8, a.wz + blk * 8, ng * 8, fb);
      }
    };
    auto issue_x = [&](int s) {
      const uint32_t slot = ring + (s % NS) * a.slot, fb = full0 + 8 * (s % NS);
      const int ng = stage_groups(s);
      const int64_t kst = kbeg + (int64_t)s * C::KC;
      for (int r = lane; r < rows_valid; r += 32)
        bulk_load(slot + C::CODES + C::META + r * C::XSTR, a.x + (m0 + r) * a.k + kst, ng * 256, fb);
    };
    const int pre = min(NS, nst);
    for (int s = 0; s < pre; ++s) issue_w(s);  // weights are constant: fetch ahead
    grid_dependency_wait();
    allow_dependent_launch();
    for (int s = 0; s < pre; ++s) issue_x(s);
    for (int s = NS; s < nst; ++s) {
      if (!mbar_wait(empty0 + 8 * (s % NS), ((s / NS) - 1) & 1)) {
        if (lane == 0) atomicOr(&g_gemm_error, kErrWaitTimeout);
        ok = false;
        break;
      }
      issue_w(s);
      issue_x(s);
    }
  } else {
    // ---------------- consumer warps ----------------
    grid_dependency_wait();
    allow_dependent_launch();
    uint32_t znext[C::NG];
    auto load_zeros = [&](int s, uint32_t (&z)[C::NG]) {
      const int64_t g0 = (kbeg + (int64_t)s * C::KC) / 128, gend = kend / 128;
#pragma unroll
      for (int j = 0; j < C::NG; ++j)
        z[j] = (tile_ok && g0 + j < gend) ? ldg_u8(a.wz + (tile * G + g0 + j) * 8 + g) : 0u;
    };
    if (nst > 0 && !zbulk) load_zeros(0, znext);
    for (int s = 0; s < nst; ++s) {
      const int slot_i = s % NS;
      if (!mbar_wait(full0 + 8 * slot_i, (s / NS) & 1)) {
        if (lane == 0) atomicOr(&g_gemm_error, kErrWaitTimeout);
        ok = false;
        break;
      }
      uint32_t zcur[C::NG];
#pragma unroll
      for (int j = 0; j < C::NG; ++j) zcur[j] = znext[j];
      if (s + 1 < nst && !zbulk) load_zeros(s + 1, znext);
      const uint32_t slot = ring + slot_i * a.slot;
      const uint32_t wb = slot + warp * C::NG * 1024;
      const uint32_t sb = slot + C::CODES + warp * C::NG * 32;
      const uint32_t xb = slot + C::CODES + C::META;
      const uint32_t zb = slot + C::CODES + C::SCALES + warp * C::NG * 8;
      const int64_t kst = kbeg + (int64_t)s * C::KC;
      const int ngroups = (int)((kend - kst) / 128);
      if (tile_ok) {
#pragma unroll
        for (int jg = 0; jg < C::NG; ++jg) {
          if (jg >= ngroups) break;
          const uint32_t sc = lds32(sb + jg * 32 + g * 4);
          const uint32_t zz = zbulk ? lds8(zb + jg * 8 + g) : zcur[jg];
          const uint32_t zlo = int4_zero_pair(zz), zhi = int4_zero_pair(zz >> 4);
          const uint4 q0 = lds128(wb + jg * 1024 + lane * 16);
          const uint4 q1 = lds128(wb + jg * 1024 + 512 + lane * 16);
          float ga[MT][4];
#pragma unroll
          for (int j = 0; j < MT; ++j) ga[j][0] = ga[j][1] = ga[j][2] = ga[j][3] = 0.f;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 xv[MT];
#pragma unroll
            for (int j = 0; j < MT; ++j) {
              const int r = xrow(8 * j + g, rows_valid);
              xv[j] = lds128(xb + r * C::XSTR + (jg * 128 + 32 * c + 8 * t) * 2);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int i = 2 * c + e;
              const Int4Frag f = int4_unpack(word(i < 4 ? q0 : q1, i & 3), zlo, zhi);
#pragma unroll
              for (int j = 0; j < MT; ++j)
                mma_bf16(ga[j], f.a0, f.a1, f.a2, f.a3, word(xv[j], 2 * e), word(xv[j], 2 * e + 1));
            }
          }
          const float slo = __uint_as_float(sc << 16), shi = __uint_as_float(sc & 0xFFFF0000u);
#pragma unroll
          for (int j = 0; j < MT; ++j) {
            acc[j][0] = fmaf(slo, ga[j][0], acc[j][0]);
            acc[j][1] = fmaf(slo, ga[j][1], acc[j][1]);
            acc[j][2] = fmaf(shi, ga[j][2], acc[j][2]);
            acc[j][3] = fmaf(shi, ga[j][3], acc[j][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot_i);
    }
  }
  if (!ok) {
    // Let the copies already in flight land (bounded) before the CTA moves on.
    for (int i = 0; i < min(NS, nst); ++i) (void)mbar_wait(full0 + 8 * i, 0);
  }
  finish<kINT4, MT, C::WARPS, C::THREADS, ROPE>(a, acc, tile0, m0, tile_ok, epi);
}

struct KernelInfo {
  int warps, kc, wstage, mstage, xrowb, rows, stages;
};

template <int WT, int MT, int W = (MT <= 2 ? 8 : 4)>
KernelInfo info_t() {
  if constexpr (WT == kINT4) {
    using C = Int4Cfg<MT, W>;
    return {C::WARPS, C::KC, C::CODES, C::META, C::XSTR, C::ROWS, C::NS_MAX};
  } else {
    using C = Cfg<WT, MT>;
    return {C::WARPS, C::KC, C::WSTAGE, C::MSTAGE, C::XROWB, C::ROWS, kStages};
  }
}

// warps: INT4 consumer warps per CTA (8 or 4 for mt <= 2); ignored otherwise.
KernelInfo info_of(int wt, int mt, int warps) {
#define DQD_INFO(W)                          \
  switch (mt) {                              \
    case 1: return info_t<W, 1>();           \
    case 2: return info_t<W, 2>();           \
    case 4: return info_t<W, 4>();           \
    default: return info_t<W, 8>();          \
  }
  if (wt == kBF16) { DQD_INFO(kBF16) }
  if (wt == kFP8) { DQD_INFO(kFP8) }
  if (mt == 1 && warps == 4) return info_t<kINT4, 1, 4>();
  if (mt == 2 && warps == 4) return info_t<kINT4, 2, 4>();
  DQD_INFO(kINT4)
#undef DQD_INFO
}

template <int WT, int MT, int W, bool ROPE>
cudaError_t launch_t(const GemmLaunch& l, const GemmPlan& p, cudaStream_t s) {
  using C = Cfg<WT, MT>;
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || configured[dev].load(std::memory_order_relaxed) < p.smem_bytes) {
    cudaError_t e = WT == kINT4 ? cudaFuncSetAttribute(dq_gemm_int4_kernel<MT, W, ROPE>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes)
                                : cudaFuncSetAttribute(dq_gemm_kernel<WT, MT, ROPE>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(p.smem_bytes, std::memory_order_relaxed);
  }
  Args a;
  a.w = static_cast<const uint8_t*>(l.data);
  a.ws = static_cast<const uint8_t*>(l.scales);
  a.wz = static_cast<const uint8_t*>(l.zeros);
  a.x = l.x;
  a.y = l.y;
  a.counters = static_cast<unsigned*>(l.workspace);
  a.part = l.workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(l.workspace) + kCounterBytes)
                       : nullptr;
  a.m = l.m;
  a.n = l.n;
  a.k = l.k;
  a.k_per_split = p.k_per_split;
  a.splits = p.splits;
  a.ra = p.ra;
  a.slot = p.slot_bytes;
  a.cluster = p.cluster;
  a.ns = p.int4_slots;
  typename EpiOf<ROPE>::type epi{};
  if constexpr (ROPE) epi = *l.rope;
  dim3 grid(p.grid_x, p.splits, p.m_chunks);
  if constexpr (WT == kINT4) {
    if (p.cluster)
      return launch_pdl_cluster(dq_gemm_int4_kernel<MT, W, ROPE>, grid, dim3(Int4Cfg<MT, W>::THREADS), p.smem_bytes,
                                s, (unsigned)p.splits, a, epi);
    return launch_pdl(dq_gemm_int4_kernel<MT, W, ROPE>, grid, dim3(Int4Cfg<MT, W>::THREADS), p.smem_bytes, s, a,
                      epi);
  } else {
    if (p.cluster)
      return launch_pdl_cluster(dq_gemm_kernel<WT, MT, ROPE>, grid, dim3(C::THREADS), p.smem_bytes, s,
                                (unsigned)p.splits, a, epi);
    return launch_pdl(dq_gemm_kernel<WT, MT, ROPE>, grid, dim3(C::THREADS), p.smem_bytes, s, a, epi);
  }
}

template <int WT, bool ROPE>
cudaError_t launch_wt(const GemmLaunch& l, const GemmPlan& p, cudaStream_t s) {
  if constexpr (WT == kINT4) {
    if (p.mt == 1 && p.warps == 4) return launch_t<WT, 1, 4, ROPE>(l, p, s);
    if (p.mt == 2 && p.warps == 4) return launch_t<WT, 2, 4, ROPE>(l, p, s);
  }
  switch (p.mt) {
    case 1: return launch_t<WT, 1, 8, ROPE>(l, p, s);
    case 2: return launch_t<WT, 2, 8, ROPE>(l, p, s);
    case 4: return launch_t<WT, 4, 4, ROPE>(l, p, s);
    default: return launch_t<WT, 8, 4, ROPE>(l, p, s);
  }
}

}  // namespace

namespace {

GemmPlan plan_warp_mma(int wtype, int64_t m, int64_t n, int64_t k, int num_sms, int warps, int int4_slots) {
  GemmPlan p{};
  p.mt = m <= 8 ? 1 : (m <= 16 ? 2 : (m <= 32 ? 4 : 8));
  const KernelInfo ki = info_of(wtype, p.mt, warps);
  p.warps = ki.warps;
  const int64_t rows = ki.rows;
  p.m_chunks = (int)((m + rows - 1) / rows);
  const int64_t ntiles = (n + 15) / 16;
  p.grid_x = (int)((ntiles + ki.warps - 1) / ki.warps);
  p.kc = ki.kc;
  p.ra = (int)std::min<int64_t>(rows, m);
  p.slot_bytes = (ki.wstage + ki.mstage + p.ra * ki.xrowb + 127) / 128 * 128;
  p.int4_slots = wtype == kINT4 ? std::max(2, std::min(ki.stages, int4_slots)) : 0;
  p.smem_bytes = (wtype == kINT4 ? p.int4_slots : ki.stages) * p.slot_bytes;
  const int64_t stages = std::max<int64_t>(1, (k + p.kc - 1) / p.kc);
  const int64_t base = (int64_t)p.grid_x * p.m_chunks;
  const int cps = std::max(1, std::min((227 * 1024 - 1024) / std::max(p.smem_bytes, 1), 16 / ki.warps));
  const int64_t slots = (int64_t)std::max(num_sms, 1) * cps;
  // Split k: when 2..8 splits keep the whole grid within 85% of one wave,
  // take as many as fit (they reduce inside a thread-block cluster, cheaply;
  // measured: a 6144 x 4096 BF16 GEMV takes 10.7 us with 5 such splits, 14.4
  // us with 6 global ones). Otherwise split only as far as needed to fill the
  // GPU, preferring the smallest split whose CTA count wastes little of the
  // last wave.
  const double wbytes = wtype == kBF16 ? 2.0 * n * k : (wtype == kFP8 ? 1.0 * n * k : 0.52 * n * k);
  const char* cl_env = std::getenv("DQD_GEMM_CLUSTER");
  const bool cluster_ok = !(cl_env && cl_env[0] == '0');
  const int64_t fit = std::min<int64_t>(8, (int64_t)(0.85 * (double)slots) / std::max<int64_t>(base, 1));
  int64_t splits = 1;
  if (cluster_ok && fit >= 2 && stages >= 2) {
    splits = fit;
  } else if (2 * base >= slots) {
    // The grid alone covers half the CTA slots: streaming is HBM-bound, and
    // splitting only adds waves and a global fixup (measured: a 28672 x 4096
    // BF16 GEMV takes 38.8 us unsplit, 44.3 us with 4 splits over 3 waves).
    splits = 1;
  } else if (base < 2 * slots) {
    double best = 0.0;
    for (int64_t sp = 1; sp <= std::min<int64_t>(stages, 64); ++sp) {
      if (sp > 1 && 8.0 * sp * m * n > 0.25 * wbytes) break;
      const int64_t ctas = base * sp;
      const double waves = (double)((ctas + slots - 1) / slots);
      const double eff = (double)ctas / (waves * slots);
      if (eff > best + 0.05) {
        best = eff;
        splits = sp;
      }
      if (eff >= 0.9) break;
    }
  }
  // counters must fit their reserved region
  if ((size_t)base * 4 > kCounterBytes) splits = 1;
  // Test hook: DQD_GEMM_SPLITS forces the k split (results must not depend on it
  // beyond rounding).
  if (const char* env = std::getenv("DQD_GEMM_SPLITS")) {
    const long v = std::strtol(env, nullptr, 10);
    if (v >= 1 && (size_t)base * 4 <= kCounterBytes) splits = v;
  }
  splits = std::min(splits, stages);
  const int64_t per = (stages + splits - 1) / splits;
  splits = (stages + per - 1) / per;
  p.splits = (int)splits;
  p.k_per_split = per * p.kc;
  // Up to 8 splits (the portable cluster size) reduce inside a cluster
  // through distributed shared memory when the whole grid fits in 85% of one
  // wave; measured, clusters lose on multi-wave or nearly full grids, where
  // co-scheduling whole clusters leaves slots idle. Otherwise the splits go
  // through global partials. Test hook: DQD_GEMM_CLUSTER=0 / 1 forces the
  // global / cluster path (1 still needs 2..8 splits).
  p.cluster = p.splits > 1 && p.splits <= 8 && (double)base * p.splits <= 0.85 * (double)slots;
  if (cl_env && cl_env[0] == '0') p.cluster = 0;
  if (cl_env && cl_env[0] == '1') p.cluster = p.splits > 1 && p.splits <= 8;
  p.ws_bytes = p.splits > 1 && !p.cluster ? kCounterBytes + sizeof(float) * (size_t)p.splits * m * n : 0;
  return p;
}

// Time model for choosing the INT4 CTA width: CTAs are dealt to SMs evenly,
// and an SM's time is its consumer warps' k stages, one tile per warp.
double warp_mma_cost(const GemmPlan& p, int num_sms) {
  const int64_t ctas = (int64_t)p.grid_x * p.splits * p.m_chunks;
  const int64_t per_sm = (ctas + num_sms - 1) / std::max(num_sms, 1);
  return (double)per_sm * p.warps * (double)((p.k_per_split + p.kc - 1) / p.kc);
}

}  // namespace

GemmPlan plan_dq_gemm(int wtype, int64_t m, int64_t n, int64_t k, int num_sms) {
  // Test hooks: DQD_GEMM_TC=0 keeps wide-m shapes on the warp-MMA kernels;
  // DQD_GEMM_TC=1 takes any m to the tcgen05 kernel where the shape allows it.
  const char* tc_env = std::getenv("DQD_GEMM_TC");
  const bool tc_on = tc_env && tc_env[0] == '1' ? tc_supported(wtype, std::max<int64_t>(m, 1024), n, k)
                                                 : tc_supported(wtype, m, n, k);
  if (tc_on && !(tc_env && tc_env[0] == '0')) return plan_dq_gemm_tc(wtype, m, n, k, num_sms);
  // INT4 ring depth: 2 slots from m = 5, 3 below. Measured on the 8B and 70B
  // projections: 2 slots free shared memory for one more CTA per SM once the
  // activation rows make slots large (m = 8: 70B gate+up 73.9 -> 61.3 us, 8B
  // gate+up 22.4 -> 19.3 us; m = 16: 70B qkv 29.1 -> 22.4 us), and are mixed
  // at m <= 4. Test hook: DQD_GEMM_INT4_NS=2 / 3 forces it.
  int ns = m >= 5 ? 2 : 3;
  if (const char* env = std::getenv("DQD_GEMM_INT4_NS")) ns = env[0] == '2' ? 2 : 3;
  GemmPlan p = plan_warp_mma(wtype, m, n, k, num_sms, 8, ns);
  if (wtype == kINT4 && m <= 16) {
    // INT4 at m <= 16: 8 or 4 consumer warps per CTA, whichever spreads the
    // 16-row tiles more evenly over the SMs (fewer warps on ties). Test hook:
    // DQD_GEMM_WARPS=4 / 8 forces the width.
    const GemmPlan p4 = plan_warp_mma(wtype, m, n, k, num_sms, 4, ns);
    const char* w_env = std::getenv("DQD_GEMM_WARPS");
    if (w_env && w_env[0] == '4') return p4;
    if (!(w_env && w_env[0] == '8') && warp_mma_cost(p4, num_sms) <= warp_mma_cost(p, num_sms)) return p4;
  }
  return p;
}

cudaError_t gemm_take_device_error(uint32_t* flags) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof zero);
  *flags |= v;
  if (e != cudaSuccess) return e;
  return tc_take_device_error(flags);
}

cudaError_t launch_dq_gemm(const GemmLaunch& l, const GemmPlan& p, cudaStream_t s) {
  if (p.tc) return launch_dq_gemm_tc(l, p, s);
  if (l.rope) {
    switch (l.wtype) {
      case kBF16: return launch_wt<kBF16, true>(l, p, s);
      case kFP8: return launch_wt<kFP8, true>(l, p, s);
      default: return launch_wt<kINT4, true>(l, p, s);
    }
  }
  switch (l.wtype) {
    case kBF16: return launch_wt<kBF16, false>(l, p, s);
    case kFP8: return launch_wt<kFP8, false>(l, p, s);
    default: return launch_wt<kINT4, false>(l, p, s);
  }
}

}  // namespace dqd
