// dq_gemm: y[m][n] = sum_k x[m][k] * deq(W)[n][k] for small and mid m.
//
// Source: "降低每個 Token 的生成成本" (Making each token cheaper), section
// "量化省下什麼" (What quantisation saves): the decode kernel multiplies a
// quantised matrix by a full-precision vector and dequantises the weights on
// the fly; "LLM 推理是怎么变快的" §4.1: weight-only formats dequantise back to
// 16-bit, and decode time is weight bytes over bandwidth.
//
// Design (HBM-bound at decode m):
//  * A CTA is 4 warps; each warp owns one 16-row tile of W (the A operand of
//    mma.m16n8k16, "swap-AB": weights fill the 16-row side, the m tokens the
//    8-column side) and walks a k range. W is streamed straight from HBM into
//    registers with 128-bit loads, double-buffered one pipeline stage ahead.
//  * Inside each 32-k (BF16/INT4) or 64-k (FP8) chunk, lane t owns a run of
//    8 (16) consecutive k for rows g and g+8, so one 16-byte load feeds 2 (4)
//    MMAs. The reduction index k is thereby permuted within the chunk; the
//    activations are read with the same permutation, so the sum is unchanged.
//  * x for the CTA's k stage sits in shared memory (cp.async, two stages),
//    shared by the 4 warps; row strides are padded so the B-fragment loads
//    are free of bank conflicts.
//  * INT4: per 128-group, (q - z) is formed exactly in bf16 and the group's
//    fp32 MMA sum is multiplied by the group scale. FP8: the E4M3 value is
//    built exactly in bf16 and the per-row scale multiplies the fp32 total.
//  * Split-K when the n tiles alone cannot fill the GPU: each split writes
//    fp32 partials; the last CTA to arrive (atomic ticket, no waiting) sums
//    them in split order, so the result does not depend on arrival order.
#include "dqd_device.cuh"
#include "dqd_internal.h"

#include <algorithm>
#include <cstdlib>

namespace dqd {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSmTarget = 3;

__host__ __device__ constexpr int kc_base(int wt) { return wt == kBF16 ? 128 : (wt == kFP8 ? 256 : 512); }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int WT, int MT>
struct Cfg {
  static constexpr int ROWS = 8 * MT;                        // activation rows per CTA pass
  static constexpr int KC = cmin(kc_base(WT), 8192 / ROWS);  // k per pipeline stage
  static constexpr int NLD = WT == kBF16 ? KC / 16 : (WT == kFP8 ? KC / 32 : KC / 64);  // 16B loads/lane/stage
  static constexpr int PADB = WT == kFP8 ? 16 : 64;          // bank-conflict-free B loads
  static constexpr int SROW = KC * 2 + PADB;                 // bytes per x row in smem
  static constexpr int STAGE = ROWS * SROW;
  static constexpr int SMEM = 2 * STAGE;
  static constexpr int NGRP = KC / 128;                      // INT4 groups per stage
};

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
};

template <int WT, int MT>
__device__ __forceinline__ void stage_x(uint32_t sbase, const Args& a, int64_t m0, int64_t kst,
                                        int64_t kend) {
  using C = Cfg<WT, MT>;
  constexpr int UPR = C::KC / 8;  // 16-byte units per row
#pragma unroll
  for (int i = 0; i < (C::ROWS * UPR + kThreads - 1) / kThreads; ++i) {
    int u = threadIdx.x + i * kThreads;
    if (u < C::ROWS * UPR) {
      int r = u / UPR, cu = u % UPR;
      int64_t mm = m0 + r, kk = kst + (int64_t)cu * 8;
      bool ok = mm < a.m && kk < kend;
      const uint16_t* src = ok ? a.x + mm * a.k + kk : a.x;
      cp_async16(sbase + r * C::SROW + cu * 16, src, ok);
    }
  }
  cp_async_commit();
}

template <int WT, int MT>
struct Warp {
  using C = Cfg<WT, MT>;
  uint4 w[C::NLD];
  uint32_t sc[C::NGRP > 0 ? C::NGRP : 1];
  uint32_t zr[C::NGRP > 0 ? C::NGRP : 1];

  __device__ __forceinline__ void load(const Args& a, int64_t tile, int lane, int64_t kst,
                                       int64_t kend, bool tile_ok) {
    const int g = lane >> 2, t = lane & 3;
    const uint4 z = make_uint4(0, 0, 0, 0);
    if constexpr (WT == kBF16) {
      const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
      const bool ok0 = tile_ok && r0 < a.n, ok1 = tile_ok && r1 < a.n;
#pragma unroll
      for (int c = 0; c < C::KC / 32; ++c) {
        int64_t kk = kst + 32 * c + 8 * t;
        bool kok = kk < kend;
        w[2 * c] = (ok0 && kok) ? ldg_stream(a.w + (r0 * a.k + kk) * 2) : z;
        w[2 * c + 1] = (ok1 && kok) ? ldg_stream(a.w + (r1 * a.k + kk) * 2) : z;
      }
    } else if constexpr (WT == kFP8) {
      const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
      const bool ok0 = tile_ok && r0 < a.n, ok1 = tile_ok && r1 < a.n;
#pragma unroll
      for (int d = 0; d < C::KC / 64; ++d) {
        int64_t kk = kst + 64 * d + 16 * t;
        bool kok = kk < kend;
        w[2 * d] = (ok0 && kok) ? ldg_stream(a.w + r0 * a.k + kk) : z;
        w[2 * d + 1] = (ok1 && kok) ? ldg_stream(a.w + r1 * a.k + kk) : z;
      }
    } else {
      const int64_t G = a.k / 128, g0 = kst / 128, gend = kend / 128;
#pragma unroll
      for (int j = 0; j < C::NGRP; ++j) {
        bool ok = tile_ok && g0 + j < gend;
        int64_t blk = tile * G + g0 + j;
        w[2 * j] = ok ? ldg_stream(a.w + blk * 1024 + lane * 16) : z;
        w[2 * j + 1] = ok ? ldg_stream(a.w + blk * 1024 + 512 + lane * 16) : z;
        sc[j] = ok ? ldg_u32(a.ws + blk * 32 + g * 4) : 0u;
        zr[j] = ok ? ldg_u8(a.wz + blk * 8 + g) : 0u;
      }
    }
  }

  // acc[j][*]: rows (g, g+8) x token columns (8j + 2t, 8j + 2t + 1).
  // ngroups: INT4 groups of this stage inside [kbeg, kend) (BF16/FP8 ignore it:
  // their loads past kend are zero-filled on both operands).
  __device__ __forceinline__ void compute(float (&acc)[MT][4], uint32_t sx, int lane,
                                          int ngroups) const {
    const int g = lane >> 2, t = lane & 3;
    if constexpr (WT == kBF16) {
#pragma unroll
      for (int c = 0; c < C::KC / 32; ++c) {
        uint4 xv[MT];
#pragma unroll
        for (int j = 0; j < MT; ++j) xv[j] = lds128(sx + (8 * j + g) * C::SROW + (32 * c + 8 * t) * 2);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t a0 = word(w[2 * c], 2 * e), a1 = word(w[2 * c + 1], 2 * e);
          uint32_t a2 = word(w[2 * c], 2 * e + 1), a3 = word(w[2 * c + 1], 2 * e + 1);
#pragma unroll
          for (int j = 0; j < MT; ++j)
            mma_bf16(acc[j], a0, a1, a2, a3, word(xv[j], 2 * e), word(xv[j], 2 * e + 1));
        }
      }
    } else if constexpr (WT == kFP8) {
#pragma unroll
      for (int d = 0; d < C::KC / 64; ++d) {
        uint4 xa[MT], xb[MT];
#pragma unroll
        for (int j = 0; j < MT; ++j) {
          uint32_t p = sx + (8 * j + g) * C::SROW + (64 * d + 16 * t) * 2;
          xa[j] = lds128(p);
          xb[j] = lds128(p + 16);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t ug = word(w[2 * d], e), uh = word(w[2 * d + 1], e);
          uint32_t a0 = fp8_lo_to_bf16x2(ug), a1 = fp8_lo_to_bf16x2(uh);
          uint32_t a2 = fp8_hi_to_bf16x2(ug), a3 = fp8_hi_to_bf16x2(uh);
#pragma unroll
          for (int j = 0; j < MT; ++j) {
            const uint4& xv = e < 2 ? xa[j] : xb[j];
            mma_bf16(acc[j], a0, a1, a2, a3, word(xv, 2 * (e & 1)), word(xv, 2 * (e & 1) + 1));
          }
        }
      }
    } else {
#pragma unroll
      for (int jg = 0; jg < C::NGRP; ++jg) {
        if (jg >= ngroups) break;  // past the end of k (warp-uniform)
        const uint32_t zlo = int4_zero_pair(zr[jg]), zhi = int4_zero_pair(zr[jg] >> 4);
        float ga[MT][4];
#pragma unroll
        for (int j = 0; j < MT; ++j) ga[j][0] = ga[j][1] = ga[j][2] = ga[j][3] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 xv[MT];
#pragma unroll
          for (int j = 0; j < MT; ++j)
            xv[j] = lds128(sx + (8 * j + g) * C::SROW + (128 * jg + 32 * c + 8 * t) * 2);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = 2 * c + e;
            Int4Frag f = int4_unpack(word(w[2 * jg + (i >> 2)], i & 3), zlo, zhi);
#pragma unroll
            for (int j = 0; j < MT; ++j)
              mma_bf16(ga[j], f.a0, f.a1, f.a2, f.a3, word(xv[j], 2 * e), word(xv[j], 2 * e + 1));
          }
        }
        const float slo = __uint_as_float(sc[jg] << 16), shi = __uint_as_float(sc[jg] & 0xFFFF0000u);
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
};

template <int WT, int MT>
__global__ void __launch_bounds__(kThreads) dq_gemm_kernel(const Args a) {
  using C = Cfg<WT, MT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t tile = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t ntiles = (a.n + 15) / 16;
  const bool tile_ok = tile < ntiles;
  const int64_t m0 = (int64_t)blockIdx.z * C::ROWS;
  const int64_t kbeg = (int64_t)blockIdx.y * a.k_per_split;
  const int64_t kend = min(a.k, kbeg + a.k_per_split);
  const int nst = (int)((kend - kbeg + C::KC - 1) / C::KC);
  const uint32_t sbuf0 = smem_addr(smem), sbuf1 = sbuf0 + C::STAGE;

  float acc[MT][4];
#pragma unroll
  for (int j = 0; j < MT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  Warp<WT, MT> wa, wb;
  if (nst > 0) {
    stage_x<WT, MT>(sbuf0, a, m0, kbeg, kend);
    wa.load(a, tile, lane, kbeg, kend, tile_ok);
  }
  for (int s = 0; s < nst; s += 2) {
    const int64_t k1 = kbeg + (int64_t)(s + 1) * C::KC;
    if (s + 1 < nst) {
      stage_x<WT, MT>(sbuf1, a, m0, k1, kend);
      wb.load(a, tile, lane, k1, kend, tile_ok);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (tile_ok) wa.compute(acc, sbuf0, lane, (int)((kend - (kbeg + (int64_t)s * C::KC) + 127) / 128));
    __syncthreads();
    if (s + 1 >= nst) break;
    const int64_t k2 = k1 + C::KC;
    if (s + 2 < nst) {
      stage_x<WT, MT>(sbuf0, a, m0, k2, kend);
      wa.load(a, tile, lane, k2, kend, tile_ok);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (tile_ok) wb.compute(acc, sbuf1, lane, (int)((kend - k1 + 127) / 128));
    __syncthreads();
  }

  // ---- epilogue ----
  const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
  auto scale_row = [&](int64_t r) -> float {
    if constexpr (WT == kFP8) return (tile_ok && r < a.n) ? reinterpret_cast<const float*>(a.ws)[r] : 0.f;
    return 1.f;
  };
  auto store = [&](float (&v)[MT][4]) {
    if (!tile_ok) return;
    const float s0 = scale_row(r0), s1 = scale_row(r1);
#pragma unroll
    for (int j = 0; j < MT; ++j) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t mm = m0 + 8 * j + 2 * t + (q & 1);
        const int64_t nn = (q & 2) ? r1 : r0;
        if (mm < a.m && nn < a.n) {
          float val = v[j][q];
          if constexpr (WT == kFP8) val *= (q & 2) ? s1 : s0;
          a.y[mm * a.n + nn] = f32_to_bf16(val);
        }
      }
    }
  };

  if (a.splits == 1) {
    store(acc);
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
  // Cooperative reduction of the CTA's 64 x ROWS outputs: each thread owns
  // whole outputs and sums their split partials in split order (loads issued
  // ahead of the adds, so they overlap).
  const int64_t n0 = (int64_t)blockIdx.x * kWarps * 16;
  const int64_t S = a.splits, plane = a.m * a.n;
  for (int e = threadIdx.x; e < kWarps * 16 * C::ROWS; e += kThreads) {
    const int64_t nn = n0 + e / C::ROWS, mm = m0 + e % C::ROWS;
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
  if (threadIdx.x == 0) *cnt = 0u;  // leave the counter at zero for the next call
}

template <int WT, int MT>
cudaError_t launch_t(const GemmLaunch& l, const GemmPlan& p, cudaStream_t s) {
  using C = Cfg<WT, MT>;
  static_assert(C::SMEM <= 48 * 1024, "x stages must fit the default shared-memory window");
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
  dim3 grid(p.grid_x, p.splits, p.m_chunks);
  dq_gemm_kernel<WT, MT><<<grid, kThreads, C::SMEM, s>>>(a);
  return cudaGetLastError();
}

template <int WT>
cudaError_t launch_wt(const GemmLaunch& l, const GemmPlan& p, cudaStream_t s) {
  switch (p.mt) {
    case 1: return launch_t<WT, 1>(l, p, s);
    case 2: return launch_t<WT, 2>(l, p, s);
    case 4: return launch_t<WT, 4>(l, p, s);
    default: return launch_t<WT, 8>(l, p, s);
  }
}

template <int WT>
int kc_of(int mt) {
  switch (mt) {
    case 1: return Cfg<WT, 1>::KC;
    case 2: return Cfg<WT, 2>::KC;
    case 4: return Cfg<WT, 4>::KC;
    default: return Cfg<WT, 8>::KC;
  }
}
template <int WT>
int smem_of(int mt) {
  switch (mt) {
    case 1: return Cfg<WT, 1>::SMEM;
    case 2: return Cfg<WT, 2>::SMEM;
    case 4: return Cfg<WT, 4>::SMEM;
    default: return Cfg<WT, 8>::SMEM;
  }
}

}  // namespace

GemmPlan plan_dq_gemm(int wtype, int64_t m, int64_t n, int64_t k, int num_sms) {
  GemmPlan p{};
  p.mt = m <= 8 ? 1 : (m <= 16 ? 2 : (m <= 32 ? 4 : 8));
  const int64_t rows = 8 * p.mt;
  p.m_chunks = (int)((m + rows - 1) / rows);
  const int64_t ntiles = (n + 15) / 16;
  p.grid_x = (int)((ntiles + kWarps - 1) / kWarps);
  switch (wtype) {
    case kBF16: p.kc = kc_of<kBF16>(p.mt); p.smem_bytes = smem_of<kBF16>(p.mt); break;
    case kFP8: p.kc = kc_of<kFP8>(p.mt); p.smem_bytes = smem_of<kFP8>(p.mt); break;
    default: p.kc = kc_of<kINT4>(p.mt); p.smem_bytes = smem_of<kINT4>(p.mt); break;
  }
  const int64_t stages = std::max<int64_t>(1, (k + p.kc - 1) / p.kc);
  const int64_t base = (int64_t)p.grid_x * p.m_chunks;
  const int64_t slots = (int64_t)std::max(num_sms, 1) * kCtasPerSmTarget;
  int64_t splits = 1;
  if (base < slots) splits = (slots + base - 1) / base;
  // fp32 partial traffic stays a small fraction of the weight stream
  const double wbytes = wtype == kBF16 ? 2.0 * n * k : (wtype == kFP8 ? 1.0 * n * k : 0.53 * n * k);
  while (splits > 1 && 8.0 * splits * m * n > 0.25 * wbytes) --splits;
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
  p.ws_bytes = p.splits > 1 ? kCounterBytes + sizeof(float) * (size_t)p.splits * m * n : 0;
  return p;
}

cudaError_t launch_dq_gemm(const GemmLaunch& l, const GemmPlan& p, cudaStream_t s) {
  switch (l.wtype) {
    case kBF16: return launch_wt<kBF16>(l, p, s);
    case kFP8: return launch_wt<kFP8>(l, p, s);
    default: return launch_wt<kINT4>(l, p, s);
  }
}

}  // namespace dqd
