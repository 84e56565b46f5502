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
// over the whole k range, in 64-wide k slabs through a ring of shared-memory
// slots:
//  * warp 0 (producer) moves each slab with TMA: the packed INT4 codes of the
//    CTA's eight 16-row tiles (half of each 1 KB group block), their group
//    scales, and the activation slab x[N tokens][64 k] as one 128-byte-
//    swizzled box (rows past the ends arrive as zeros). Weights for the first
//    slots are requested before the wait on the preceding kernel;
//  * warps 1-8 (one 16-row tile each) stage the CTA's zero points in shared
//    memory once, then dequantise each slab's codes to bf16
//    deq = RN((q - z) * s) (the exact bf16 subtraction, then one rounded bf16
//    multiply) into the K-major 128-byte-swizzled layout the tensor core reads;
//  * one thread of warp 9 issues tcgen05.mma (M 128, N, K 16, bf16 in, fp32
//    accumulate in tensor memory) and commits each slab's MMAs to the slot's
//    "empty" mbarrier, which returns the slot to the producer;
//  * warps 1-8 read the accumulator back with tcgen05.ld (warps w and w+4
//    share a 32-lane quarter and split its columns) and write bf16 y.
// Every wait is bounded; tensor memory is released on every path.
#include "dqd_device.cuh"
#include "dqd_internal.h"

#include <atomic>
#include <cstring>

namespace dqd {
namespace {

__device__ unsigned int g_tc_error;

constexpr int kRows = 128;    // weight rows per CTA (MMA M)
constexpr int kMaxN = 256;    // tokens per CTA at most (MMA N)
constexpr int kSlabK = 64;    // k per slab: one 128-byte swizzle row of bf16
constexpr int kSlots = 3;
constexpr int kABytes = kRows * kSlabK * 2;   // 16 KB
constexpr int kBBytes = kMaxN * kSlabK * 2;   // 32 KB
constexpr int kCodeBytes = 8 * 512;           // 8 tiles x half a group block
constexpr int kScaleBytes = 8 * 32;           // group scales of the 8 tiles
constexpr int kSlot = 54 * 1024;              // A | B | codes | scales, padded to 1 KB
constexpr int kMaxZeroBytes = 16 * 1024;      // 8 tiles x G groups x 8 bytes (k <= 32768)
constexpr int kDeqWarps = 8;
constexpr int kThreads = (kDeqWarps + 2) * 32;
constexpr int kMmaWarp = kDeqWarps + 1;
constexpr int kSmem = kSlots * kSlot + kMaxZeroBytes + 1024;  // + alignment slack
static_assert(kABytes + kBBytes + kCodeBytes + kScaleBytes <= kSlot, "slot layout");
static_assert(kSlot % 1024 == 0, "slots keep 1024-byte alignment");
static_assert(kSmem <= 227 * 1024, "shared memory");

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
__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t saddr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(saddr) : "memory");
  return v;
}
__device__ __forceinline__ void sts64(uint32_t saddr, uint2 v) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(saddr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ uint2 ldg64(const void* p) {
  uint2 r;
  asm("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
// Named barrier over the dequantising warps only.
__device__ __forceinline__ void deq_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDeqWarps * 32) : "memory");
}

struct TcArgs {
  const uint8_t* wz;  // packed zeros
  uint16_t* y;
  int64_t m, n, k;
  int ntok;           // N: tokens per CTA
};

__global__ void __launch_bounds__(kThreads, 1)
    dq_gemm_int4_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                           const __grid_constant__ CUtensorMap tms, const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[3 * kSlots + 1];
  __shared__ uint32_t tmem_base_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t zsm = ring + kSlots * kSlot;
  const uint32_t full_raw = smem_addr(&bars[0]), full_a = smem_addr(&bars[kSlots]),
                 empty = smem_addr(&bars[2 * kSlots]), done = smem_addr(&bars[3 * kSlots]);
  // blockIdx.x walks the token chunks fastest, so the CTAs that dequantise
  // the same weight tile run together and share it through L2.
  const int64_t tile0 = (int64_t)blockIdx.y * 8;  // first 16-row tile
  const int64_t ntiles = (a.n + 15) / 16;
  const int64_t m0 = (int64_t)blockIdx.x * a.ntok;
  const int G = (int)(a.k / 128);
  const int nslabs = 2 * G;
  const uint32_t tx_bytes = kCodeBytes + kScaleBytes + (uint32_t)a.ntok * kSlabK * 2;
  auto slot = [&](int s) { return ring + s * kSlot; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(full_raw + 8 * i, 1);
      mbar_init(full_a + 8 * i, kDeqWarps * 32);
      mbar_init(empty + 8 * i, 1);
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

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      // Weights are constants: the first slots' codes and scales are requested
      // before waiting for the preceding kernel; activations after it.
      const int pre = min(kSlots, nslabs);
      for (int j = 0; j < pre; ++j) {
        const uint32_t base = slot(j), fb = full_raw + 8 * j;
        mbar_arrive_expect_tx(fb, tx_bytes);
        tma_load_2d(base + kABytes + kBBytes, &tmw, fb, j * 128, (int)tile0);
        tma_load_2d(base + kABytes + kBBytes + kCodeBytes, &tms, fb, (j / 2) * 8, (int)tile0);
      }
      grid_dependency_wait();
      allow_dependent_launch();
      for (int j = 0; j < pre; ++j) tma_load_2d(slot(j) + kABytes, &tmx, full_raw + 8 * j, j * kSlabK, (int)m0);
      for (int j = pre; j < nslabs; ++j) {
        const int s = j % kSlots;
        if (!mbar_wait(empty + 8 * s, ((j / kSlots) - 1) & 1)) {
          atomicOr(&g_tc_error, kErrWaitTimeout);
          break;
        }
        const uint32_t base = slot(s), fb = full_raw + 8 * s;
        mbar_arrive_expect_tx(fb, tx_bytes);
        tma_load_2d(base + kABytes + kBBytes, &tmw, fb, j * 128, (int)tile0);
        tma_load_2d(base + kABytes + kBBytes + kCodeBytes, &tms, fb, (j / 2) * 8, (int)tile0);
        tma_load_2d(base + kABytes, &tmx, fb, j * kSlabK, (int)m0);
      }
    }
  } else if (warp <= kDeqWarps) {
    // ---------------- dequantisers: warp w owns 16-row tile w - 1 ----------------
    const int tt = warp - 1, g = lane >> 2, t = lane & 3;
    const int dt = threadIdx.x - 32;
    // zero points of the CTA's tiles for every group: 8 bytes per (tile, group)
    for (int i = dt; i < 8 * G; i += kDeqWarps * 32) {
      const int64_t tile = tile0 + i / G;
      const uint2 z = tile < ntiles ? ldg64(a.wz + (tile0 * G + i) * 8) : make_uint2(0, 0);
      sts64(zsm + i * 8, z);
    }
    deq_barrier();
    grid_dependency_wait();
    allow_dependent_launch();
    const uint32_t row_lo = 2 * tt * 1024 + g * 128;  // row 16 tt + g; row + 8 is 1024 bytes on
    for (int j = 0; j < nslabs; ++j) {
      const int s = j % kSlots;
      if (!mbar_wait(full_raw + 8 * s, (j / kSlots) & 1)) {
        if (lane == 0) atomicOr(&g_tc_error, kErrWaitTimeout);
        ok = false;
        break;
      }
      const uint32_t base = slot(s);
      const uint4 u = lds128(base + kABytes + kBBytes + tt * 512 + lane * 16);
      const uint32_t sc = lds32(base + kABytes + kBBytes + kCodeBytes + tt * 32 + g * 4);
      const uint32_t zb = lds8(zsm + (tt * G + (j >> 1)) * 8 + g);
      const uint32_t slo = (sc & 0xFFFFu) * 0x00010001u, shi = (sc >> 16) * 0x00010001u;
      const uint32_t zlo = int4_zero_pair(zb), zhi = int4_zero_pair(zb >> 4);
      // words 2c, 2c+1 of this lane hold k = 32c + 8t .. +7 of rows g and g+8
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const Int4Frag f0 = int4_unpack(word(u, 2 * c), zlo, zhi);
        const Int4Frag f1 = int4_unpack(word(u, 2 * c + 1), zlo, zhi);
        const uint32_t a_lo = base + row_lo + (((4 * c + t) ^ g) << 4);
        sts128(a_lo, bf16x2_mul(f0.a0, slo), bf16x2_mul(f0.a2, slo), bf16x2_mul(f1.a0, slo),
               bf16x2_mul(f1.a2, slo));
        sts128(a_lo + 1024, bf16x2_mul(f0.a1, shi), bf16x2_mul(f0.a3, shi), bf16x2_mul(f1.a1, shi),
               bf16x2_mul(f1.a3, shi));
      }
      fence_proxy_async_smem();  // make the generic-proxy stores visible to the tensor core
      mbar_arrive(full_a + 8 * s);
    }
  } else {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kRows, a.ntok);
      for (int j = 0; j < nslabs; ++j) {
        const int s = j % kSlots;
        if (!mbar_wait(full_a + 8 * s, (j / kSlots) & 1)) {
          atomicOr(&g_tc_error, kErrWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t abase = slot(s), bbase = abase + kABytes;
#pragma unroll
        for (int kk = 0; kk < kSlabK / 16; ++kk)
          umma_bf16(tmem, sw128_desc(abase + kk * 32), sw128_desc(bbase + kk * 32), idesc,
                    (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(empty + 8 * s);  // the slot is free once these MMAs have read it
      }
      umma_commit(done);
    }
  }

  // ---------------- epilogue: warps w and w + 4 share lane quarter w % 4 ----------------
  if (warp >= 1 && warp <= kDeqWarps) {
    const int quarter = warp & 3;
    const int half = (warp - 1) >> 2;
    const bool good = ok && mbar_wait(done, 0);
    if (!good && lane == 0) atomicOr(&g_tc_error, kErrWaitTimeout);
    tc_fence_after();
    const int64_t row = tile0 * 16 + quarter * 32 + lane;  // weight row = output column
    const int nchunks = (a.ntok + 31) / 32;
#pragma unroll 1
    for (int cc = half; cc < nchunks; cc += 2) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + cc * 32, r);
      if (good && row < a.n) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int64_t mm = m0 + cc * 32 + j;
          if (cc * 32 + j < a.ntok && mm < a.m) a.y[mm * a.n + row] = f32_to_bf16(__uint_as_float(r[j]));
        }
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
  return wtype == kINT4 && m >= 128 && m <= (int64_t)INT32_MAX && k % 128 == 0 && k > 0 && k <= 32768 &&
         n > 0 && (n + 127) / 128 <= 65535;
}

GemmPlan plan_dq_gemm_tc(int64_t m, int64_t n, int64_t k) {
  GemmPlan p{};
  p.tc = 1;
  // Fewest token chunks of at most 256, then the smallest multiple of 16 that
  // covers m in that many chunks.
  const int64_t chunks = (m + kMaxN - 1) / kMaxN;
  const int64_t per = (m + chunks - 1) / chunks;
  p.ra = (int)((per + 15) / 16 * 16);
  p.m_chunks = (int)((m + p.ra - 1) / p.ra);
  p.grid_x = (int)((((n + 15) / 16) + 7) / 8);
  p.mt = 8;
  p.splits = 1;
  p.k_per_split = k;
  p.kc = kSlabK;
  p.slot_bytes = kSlot;
  p.smem_bytes = kSmem;
  p.ws_bytes = 0;
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
  a.m = l.m;
  a.n = l.n;
  a.k = l.k;
  a.ntok = p.ra;
  return launch_pdl(dq_gemm_int4_tc_kernel, dim3(p.m_chunks, p.grid_x), dim3(kThreads), (size_t)kSmem, s, tmx, tmw,
                    tms, a);
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
