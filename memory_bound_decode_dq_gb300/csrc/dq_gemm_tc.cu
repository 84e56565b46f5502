// dq_gemm for wide m (verify batches): INT4 g128 on the 5th-generation tensor
// cores (tcgen05), where the tile is a dense contraction.
//
// Source: "降低每個 Token 的生成成本" (Making each token cheaper), section
// "推測式解碼" (speculative decoding): verifying gamma + 1 positions per
// sequence multiplies the rows of the weight-only GEMM, and with INT4 weights
// the verify step turns compute-bound; sections "格式" (Formats) and "量化省下
// 什麼": weight-only INT4 dequantises to 16-bit before the matrix arithmetic.
//
// One CTA computes D[128 weight rows][N tokens] (N <= 256, a multiple of 16)
// over its k range (all of k, or one split of it), in 64-wide k slabs:
//  * warp 0 streams the packed INT4 codes of the CTA's eight 16-row tiles
//    (half of each 1 KB group block) and their group scales with TMA into a
//    six-deep ring; these are constants, requested before the wait on the
//    preceding kernel;
//  * warp 1 streams the activation slab x[N tokens][64 k] with TMA as one
//    128-byte-swizzled box (rows past the ends arrive as zeros) into a
//    128 KB ring (4 to 16 slabs deep, by N), so that activation reads run
//    well ahead of the MMAs;
//  * warps 2-9 (one 16-row tile each) dequantise each slab's codes to bf16
//    deq = RN((q - z) * s) (the exact bf16 subtraction, then one rounded bf16
//    multiply; zero points prefetched a group ahead into registers) into a
//    four-deep ring of K-major 128-byte-swizzled A tiles;
//  * one thread of warp 10 issues tcgen05.mma (M 128, N, K 16, bf16 in, fp32
//    accumulate in tensor memory) once both operands of a slab are in place,
//    and commits the slab's MMAs to the "empty" mbarriers of both slots;
//  * warps 2-9 read the accumulator back with tcgen05.ld (two warps per
//    32-lane quarter, splitting its columns) and write bf16 y, or with k
//    split, fp32 partials that the last-arriving CTA of the tile sums in
//    split order (deterministic).
// Every wait is bounded; tensor memory is released on every path.
#include "dqd_device.cuh"
#include "dqd_internal.h"

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

namespace dqd {
namespace {

__device__ unsigned int g_tc_error;

constexpr int kRows = 128;    // weight rows per CTA (MMA M)
constexpr int kMaxN = 256;    // tokens per CTA at most (MMA N)
constexpr int kSlabK = 64;    // k per slab: one 128-byte swizzle row of bf16
constexpr int kASlots = 4;    // dequantised weight tiles (A)
constexpr int kBRing = 128 * 1024;            // activation slabs (B): N x 128 bytes each
constexpr int kMaxBSlots = 16;
constexpr int kCSlots = 6;    // code slots
constexpr int kABytes = kRows * kSlabK * 2;   // 16 KB
constexpr int kCodeBytes = 8 * 512;           // 8 tiles x half a group block
constexpr int kScaleBytes = 8 * 32;           // group scales of the 8 tiles
constexpr int kCSlot = kCodeBytes + kScaleBytes;
constexpr int kDeqWarps = 8;
constexpr int kDeq0 = 2;                      // first dequantising warp
constexpr int kMmaWarp = kDeq0 + kDeqWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kSmem = kASlots * kABytes + kBRing + kCSlots * kCSlot + 1024;  // + alignment slack
static_assert(kABytes % 1024 == 0 && kCSlot % 128 == 0, "slot alignment");
static_assert(kBRing >= 4 * kMaxN * kSlabK * 2, "at least four activation slabs");
static_assert(kSmem + 1024 <= 227 * 1024, "shared memory");

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);        // start address
  d |= (uint64_t)1 << 16;                          // leading offset (unused by swizzled K-major)
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;   // stride offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 lanes x 32 columns of 32-bit accumulator per warp.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1)
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
  const uint8_t* wz;  // packed zeros
  uint16_t* y;
  unsigned* counters; // split-K tickets (splits > 1)
  float* part;        // split-K fp32 partials [split][m][n]
  int64_t m, n, k;
  int ntok;           // N: tokens per CTA
  int splits;
  int slabs_per_split;  // even: splits fall on group boundaries
};

__device__ __forceinline__ float4 ldcg4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

// Last-arriving CTA of a split-K tile: y = bf16(sum of the split partials in
// split order) over the tile's rows [r0, r0 + rows) and tokens [m0, m0 + toks).
// Each thread keeps four outputs' partial loads of up to four splits in flight.
__device__ __forceinline__ void reduce_splits(const TcArgs& a, int64_t r0, int rows, int64_t m0, int toks, int tid,
                                              int nthreads) {
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
        if (live[q]) {
          uint2 o;
          o.x = pack_bf16x2(acc[q].x, acc[q].y);
          o.y = pack_bf16x2(acc[q].z, acc[q].w);
          *reinterpret_cast<uint2*>(a.y + off[q]) = o;
        }
    }
  } else {
    const int units = rows * toks;
    for (int u = tid; u < units; u += nthreads) {
      const int64_t off = (m0 + u / rows) * a.n + r0 + u % rows;
      float acc = 0.f;
      for (int sp = 0; sp < a.splits; ++sp) acc += __ldcg(part + sp * plane + off);
      a.y[off] = f32_to_bf16(acc);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    dq_gemm_int4_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                           const __grid_constant__ CUtensorMap tms, const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kCSlots + 2 * kASlots + 2 * kMaxBSlots + 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int last_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t aring = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t bring = aring + kASlots * kABytes;
  const uint32_t cring = bring + kBRing;
  const uint32_t cfull = smem_addr(&bars[0]), cempty = cfull + 8 * kCSlots;
  const uint32_t afull = cempty + 8 * kCSlots, aempty = afull + 8 * kASlots;
  const uint32_t bfull = aempty + 8 * kASlots, bempty = bfull + 8 * kMaxBSlots;
  const uint32_t done = bempty + 8 * kMaxBSlots;
  const uint32_t bslot_bytes = (uint32_t)a.ntok * kSlabK * 2;
  const int nbs = min(kMaxBSlots, (int)(kBRing / bslot_bytes));  // activation slots
  // blockIdx.x walks the token chunks fastest, so the CTAs that dequantise
  // the same weight tile run together and share it through L2.
  const int64_t tile0 = (int64_t)blockIdx.y * 8;  // first 16-row tile
  const int64_t ntiles = (a.n + 15) / 16;
  const int64_t m0 = (int64_t)blockIdx.x * a.ntok;
  const int G = (int)(a.k / 128);
  const int jb = (int)blockIdx.z * a.slabs_per_split;
  const int nl = min(2 * G - jb, a.slabs_per_split);  // slabs of this CTA (even, >= 2)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kCSlots; ++i) {
      mbar_init(cfull + 8 * i, 1);
      mbar_init(cempty + 8 * i, kDeqWarps * 32);
    }
    for (int i = 0; i < kASlots; ++i) {
      mbar_init(afull + 8 * i, kDeqWarps * 32);
      mbar_init(aempty + 8 * i, 1);
    }
    for (int i = 0; i < kMaxBSlots; ++i) {
      mbar_init(bfull + 8 * i, 1);
      mbar_init(bempty + 8 * i, 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(&tmem_base_sh), kMaxN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  bool ok = true;

  // Slot cursors: slot index and the parity of its current use; a slot's
  // "empty" barrier is waited on with the opposite parity (its previous use).
  if (warp == 0) {
    // ---------------- codes + scales (constants) ----------------
    if (lane == 0) {
      allow_dependent_launch();
      int cs = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nl; ++i) {
        const int j = jb + i;
        if (i >= kCSlots && !mbar_wait(cempty + 8 * cs, ph ^ 1u)) {
          atomicOr(&g_tc_error, kErrWaitTimeout);
          break;
        }
        const uint32_t dst = cring + cs * kCSlot, fb = cfull + 8 * cs;
        mbar_arrive_expect_tx(fb, kCSlot);
        tma_load_2d(dst, &tmw, fb, j * 128, (int)tile0);
        tma_load_2d(dst + kCodeBytes, &tms, fb, (j >> 1) * 8, (int)tile0);
        if (++cs == kCSlots) {
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
      for (int i = 0; i < nl; ++i) {
        if (i >= nbs && !mbar_wait(bempty + 8 * s, ph ^ 1u)) {
          atomicOr(&g_tc_error, kErrWaitTimeout);
          break;
        }
        mbar_arrive_expect_tx(bfull + 8 * s, bslot_bytes);
        tma_load_2d(bring + s * bslot_bytes, &tmx, bfull + 8 * s, (jb + i) * kSlabK, (int)m0);
        if (++s == nbs) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp < kMmaWarp) {
    // ---------------- dequantisers: warp w owns 16-row tile w - 2 ----------------
    const int tt = warp - kDeq0, g = lane >> 2, t = lane & 3;
    grid_dependency_wait();
    allow_dependent_launch();
    const int64_t tile = tile0 + tt;
    const uint8_t* zp = a.wz + tile * G * 8 + g;  // zero byte of group gr at zp[8 gr]
    const bool live = tile < ntiles;
    int gr = jb >> 1;
    uint32_t znext = live ? ldg_u8(zp + 8 * gr) : 0u;
    // Lanes of odd g store their two 32-k halves in the opposite order, so
    // that each quarter-warp's 16-byte stores cover all 32 banks once.
    const uint32_t godd = g & 1;
    const uint32_t row_lo = 2 * tt * 1024 + g * 128;  // row 16 tt + g; row + 8 is 1024 bytes on
    const uint32_t o0 = row_lo + (((4 * godd + t) ^ g) << 4);
    const uint32_t o1 = row_lo + (((4 * (godd ^ 1u) + t) ^ g) << 4);
    const uint32_t csrc0 = cring + tt * 512 + lane * 16, ssrc0 = cring + kCodeBytes + tt * 32 + g * 4;
    int cs = 0, s = 0;
    uint32_t cph = 0, sph = 0;
    uint32_t zlo = 0, zhi = 0;
    for (int i = 0; i < nl; ++i) {
      if ((i & 1) == 0) {  // a new group: take its zero points, prefetch the next group's
        zlo = int4_zero_pair(znext);
        zhi = int4_zero_pair(znext >> 4);
        ++gr;
        znext = (live && gr < G) ? ldg_u8(zp + 8 * gr) : 0u;
      }
      if (!mbar_wait(cfull + 8 * cs, cph)) {
        ok = false;
        break;
      }
      uint4 u = lds128(csrc0 + cs * kCSlot);
      const uint32_t sc = lds32(ssrc0 + cs * kCSlot);
      if (i >= kASlots && !mbar_wait(aempty + 8 * s, sph ^ 1u)) {
        ok = false;
        break;
      }
      if (godd) {
        const uint32_t x0 = u.x, x1 = u.y;
        u.x = u.z;
        u.y = u.w;
        u.z = x0;
        u.w = x1;
      }
      const uint32_t slo = prmt(sc, 0u, 0x1010u), shi = prmt(sc, 0u, 0x3232u);
      const uint32_t base = aring + s * kABytes;
      // words 2c, 2c+1 (after the swap) hold k = 32c' + 8t .. +7 of rows g
      // and g + 8, with c' = c ^ godd
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const Int4Frag f0 = int4_unpack(word(u, 2 * c), zlo, zhi);
        const Int4Frag f1 = int4_unpack(word(u, 2 * c + 1), zlo, zhi);
        const uint32_t a_lo = base + (c == 0 ? o0 : o1);
        sts128(a_lo, bf16x2_mul(f0.a0, slo), bf16x2_mul(f0.a2, slo), bf16x2_mul(f1.a0, slo),
               bf16x2_mul(f1.a2, slo));
        sts128(a_lo + 1024, bf16x2_mul(f0.a1, shi), bf16x2_mul(f0.a3, shi), bf16x2_mul(f1.a1, shi),
               bf16x2_mul(f1.a3, shi));
      }
      fence_proxy_async_smem();  // make the generic-proxy stores visible to the tensor core
      mbar_arrive(afull + 8 * s);
      // Release the code slot only now: an arrive does not wait for shared
      // loads still in flight, so it must follow the use of their values.
      mbar_arrive(cempty + 8 * cs);
      if (++cs == kCSlots) {
        cs = 0;
        cph ^= 1u;
      }
      if (++s == kASlots) {
        s = 0;
        sph ^= 1u;
      }
    }
    if (!ok && lane == 0) atomicOr(&g_tc_error, kErrWaitTimeout);
  } else {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kRows, a.ntok);
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      for (int i = 0; i < nl; ++i) {
        if (!mbar_wait(afull + 8 * sa, pa) || !mbar_wait(bfull + 8 * sb, pb)) {
          atomicOr(&g_tc_error, kErrWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t abase = aring + sa * kABytes, bbase = bring + sb * bslot_bytes;
#pragma unroll
        for (int kk = 0; kk < kSlabK / 16; ++kk)
          umma_bf16(tmem, sw128_desc(abase + kk * 32), sw128_desc(bbase + kk * 32), idesc,
                    (i > 0 || kk > 0) ? 1u : 0u);
        // both slots are free once these MMAs have read them
        umma_commit(aempty + 8 * sa);
        umma_commit(bempty + 8 * sb);
        if (++sa == kASlots) {
          sa = 0;
          pa ^= 1u;
        }
        if (++sb == nbs) {
          sb = 0;
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
    const int64_t row = tile0 * 16 + quarter * 32 + lane;  // weight row = output column
    const int nchunks = (a.ntok + 31) / 32;
    float* part = a.splits > 1 ? a.part + (int64_t)blockIdx.z * a.m * a.n : nullptr;
#pragma unroll 1
    for (int cc = half; cc < nchunks; cc += 2) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + cc * 32, r);
      if (good && row < a.n) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int64_t mm = m0 + cc * 32 + j;
          if (cc * 32 + j < a.ntok && mm < a.m) {
            if (part)
              part[mm * a.n + row] = __uint_as_float(r[j]);
            else
              a.y[mm * a.n + row] = f32_to_bf16(__uint_as_float(r[j]));
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
        const int64_t r0 = tile0 * 16;
        const int rows = (int)min((int64_t)kRows, a.n - r0);
        const int toks = (int)min((int64_t)a.ntok, a.m - m0);
        reduce_splits(a, r0, rows, m0, toks, threadIdx.x - kDeq0 * 32, kDeqWarps * 32);
        if (warp == kDeq0 && lane == 0) *cnt = 0u;  // leave the ticket at zero for the next call
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kMaxN);
  }
}

}  // namespace

bool tc_supported(int wtype, int64_t m, int64_t n, int64_t k) {
  return wtype == kINT4 && m >= 128 && m <= (int64_t)INT32_MAX && k % 128 == 0 && k > 0 &&
         k / 128 <= 65535 && n > 0 && (n + 127) / 128 <= 65535;
}

GemmPlan plan_dq_gemm_tc(int64_t m, int64_t n, int64_t k, int num_sms) {
  GemmPlan p{};
  p.tc = 1;
  p.mt = 8;
  p.kc = kSlabK;
  p.slot_bytes = kABytes;
  p.smem_bytes = kSmem;
  p.grid_x = (int)((((n + 15) / 16) + 7) / 8);
  // Choose tokens per CTA (N, a multiple of 16 in [64, 256] covering m in
  // equal chunks) and the k split from a cost model: CTAs run in waves of one
  // per SM; a 64-wide slab costs the larger of its MMAs (2 N cycles at the
  // dense bf16 rate) and the dequantisation (about 330 cycles of issue for
  // 128 x 64 weights), plus a fixed 6 slabs of fill, drain and epilogue; a
  // split adds its fp32 partial traffic at about 6 TB/s.
  const int64_t G = k / 128, sms = std::max(num_sms, 1);
  const char* env = std::getenv("DQD_GEMM_SPLITS");
  const long forced = env ? std::strtol(env, nullptr, 10) : 0;
  double best = -1.0;
  int64_t best_n = kMaxN, best_sp = 1;
  for (int64_t cap = kMaxN; cap >= 64; cap -= 16) {
    const int64_t chunks = (m + cap - 1) / cap;
    const int64_t ntok = ((m + chunks - 1) / chunks + 15) / 16 * 16;  // <= cap
    const int64_t base = chunks * p.grid_x;
    const double slab = std::max(2.0 * ntok, 330.0) + 20.0;
    for (int64_t sp = 1; sp <= std::min<int64_t>(G, 32); ++sp) {
      if (sp > 1 && (base * sp > (int64_t)(kCounterBytes / 4) || G / sp < 2)) break;
      if (forced >= 1 && sp != std::min<int64_t>(forced, G)) continue;
      const int64_t gps = (G + sp - 1) / sp;
      const double waves = (double)((base * sp + sms - 1) / sms);
      double cycles = waves * (2.0 * gps + 6.0) * slab;
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
  const int64_t gps = (G + best_sp - 1) / best_sp;
  p.splits = (int)((G + gps - 1) / gps);
  p.k_per_split = gps * 128;
  p.ws_bytes = p.splits > 1 ? kCounterBytes + sizeof(float) * (size_t)p.splits * m * n : 0;
  return p;
}

cudaError_t launch_dq_gemm_tc(const GemmLaunch& l, const GemmPlan& p, cudaStream_t s) {
  const int64_t ntiles = (l.n + 15) / 16, G = l.k / 128;
  CUtensorMap tmx, tmw, tms;
  {
    const uint64_t dims[2] = {(uint64_t)l.k, (uint64_t)l.m};
    const uint64_t strides[1] = {(uint64_t)l.k * 2};
    const uint32_t box[2] = {kSlabK, (uint32_t)p.ra};
    cudaError_t e =
        tensor_map(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, l.x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  {  // packed codes as 32-bit words: [tile][G * 256]
    const uint64_t dims[2] = {(uint64_t)G * 256, (uint64_t)ntiles};
    const uint64_t strides[1] = {(uint64_t)G * 1024};
    const uint32_t box[2] = {128, 8};
    cudaError_t e =
        tensor_map(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, l.data, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  {  // packed scales as 32-bit words: [tile][G * 8]
    const uint64_t dims[2] = {(uint64_t)G * 8, (uint64_t)ntiles};
    const uint64_t strides[1] = {(uint64_t)G * 32};
    const uint32_t box[2] = {8, 8};
    cudaError_t e = tensor_map(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, l.scales, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(dq_gemm_int4_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(1, std::memory_order_relaxed);
  }
  TcArgs a;
  a.wz = static_cast<const uint8_t*>(l.zeros);
  a.y = l.y;
  a.counters = static_cast<unsigned*>(l.workspace);
  a.part = l.workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(l.workspace) + kCounterBytes) : nullptr;
  a.m = l.m;
  a.n = l.n;
  a.k = l.k;
  a.ntok = p.ra;
  a.splits = p.splits;
  a.slabs_per_split = (int)(p.k_per_split / kSlabK);
  return launch_pdl(dq_gemm_int4_tc_kernel, dim3(p.m_chunks, p.grid_x, p.splits), dim3(kThreads), (size_t)kSmem,
                    s, tmx, tmw, tms, a);
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
