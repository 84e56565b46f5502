// Device helpers shared by the dqd kernels (sm_103a): streaming loads,
// cp.async staging, warp-level bf16 MMA and the in-register INT4/FP8 -> bf16
// unpacking. Inline PTX only; no library code.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; no driver symbols are linked)

#include <cstdint>

namespace dqd {

// ---------------------------------------------------------------- loads ----

// 16-byte read-only load of data that is used once (weights): bypass L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
  uint32_t r;
  asm("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_u8(const void* p) {
  uint16_t r;
  asm("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(saddr));
  return r;
}

__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(saddr));
  return r;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async of 16 bytes global -> shared; zero-fills when !pred (no bytes read).
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* gptr, bool pred) {
  int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(gptr), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ------------------------------------------------------------------ MMA ----

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col), warp-wide.
// Fragment ownership (lane = 4*g + t): a0 = A[g][2t..2t+1], a1 = A[g+8][2t..],
// a2 = A[g][2t+8..], a3 = A[g+8][2t+8..]; b0 = B[2t..2t+1][g],
// b1 = B[2t+8..][g]; d0,d1 = D[g][2t..2t+1], d2,d3 = D[g+8][2t..2t+1].
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------- bit utilities ----

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// bf16x2 -> f16x2: exact for magnitudes in [2^-14, 65504]; smaller ones
// round to the f16 subnormal grid (absolute error <= 2^-25).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  // cvt packs its first source into the upper half.
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
  uint16_t d;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(d) : "f"(v));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------ INT4 unpacking ----
//
// One 32-bit word of the packed INT4 layout holds the eight codes of one
// m16n8k16 A fragment: nibble v belongs to register v%4, half v/4. OR-ing a
// code into the mantissa of bf16 128.0 (0x4300) gives the exact bf16 value
// 128 + q; subtracting 128 + z (exact) leaves q - z in [-15, 15], exact.
struct Int4Frag {
  uint32_t a0, a1, a2, a3;
};

__device__ __forceinline__ Int4Frag int4_unpack(uint32_t u, uint32_t zlo, uint32_t zhi) {
  const uint32_t M = 0x000F000Fu, MAGIC = 0x43004300u;
  Int4Frag f;
  f.a0 = bf16x2_sub(and_or(u, M, MAGIC), zlo);
  f.a1 = bf16x2_sub(and_or(u >> 4, M, MAGIC), zhi);
  f.a2 = bf16x2_sub(and_or(u >> 8, M, MAGIC), zlo);
  f.a3 = bf16x2_sub(and_or(u >> 12, M, MAGIC), zhi);
  return f;
}

// bf16x2 holding 128 + z in both halves.
__device__ __forceinline__ uint32_t int4_zero_pair(uint32_t z) {
  return (0x4300u | (z & 15u)) * 0x00010001u;
}

// ------------------------------------------------------- FP8 unpacking ----
//
// E4M3 s.eeee.mmm -> bf16 bit pattern s.0000eeee.mmm0000 (exponent field
// e, mantissa m<<4), whose value is the E4M3 value times 2^-120 for every
// code, subnormals included; one exact bf16 multiply by 2^120 restores it.
// prmt's sign-replicating selectors (bit 3 set) fill the high byte of each
// 16-bit lane with the code's sign, so a shift by 4 and one mask place sign,
// exponent and mantissa.
__device__ __forceinline__ uint32_t fp8_pair_to_bf16x2(uint32_t u, uint32_t sel) {
  uint32_t h = prmt(u, 0u, sel);
  uint32_t p = (h << 4) & 0x87F087F0u;
  return bf16x2_mul(p, 0x7B807B80u);  // 2^120 in both halves
}
// Codes in bytes 0,1 of u -> (lo, hi) of a bf16x2; bytes 2,3 likewise.
__device__ __forceinline__ uint32_t fp8_lo_to_bf16x2(uint32_t u) {
  return fp8_pair_to_bf16x2(u, 0x9180u);
}
__device__ __forceinline__ uint32_t fp8_hi_to_bf16x2(uint32_t u) {
  return fp8_pair_to_bf16x2(u, 0xB3A2u);
}

// ------------------------------------------------- thread-block clusters ----

// Cluster-wide barrier over every thread of every CTA of the cluster, with
// release/acquire ordering of shared-memory writes.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Loads from the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t saddr, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t saddr, uint32_t rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// ------------------------------------------- programmatic dependent launch ----
// Kernels are launched so that the next kernel on the stream may start while
// this one drains. Every kernel waits (griddepcontrol.wait, a hardware wait
// for the preceding grid to complete and flush) before it reads anything a
// preceding kernel may have written or writes anything it may read; only
// constant operands (weights) are prefetched before that point.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------ mbarrier + TMA ----

// Upper bound on polls of one mbarrier phase before a wait gives up. Each
// poll suspends for up to ~1 us in hardware, so this is seconds: far beyond
// any legitimate wait, short enough that a broken pipeline ends by itself.
constexpr uint32_t kSpinLimit = 1u << 22;

// Bit set in a module's device error word when a bounded wait gives up.
constexpr uint32_t kErrWaitTimeout = 1u;
// Bit set when a kernel met an input outside its documented range and clamped
// it so that every access stays in bounds (a block-table entry outside
// [0, num_blocks), a context shorter than the verify width or longer than the
// caller's max_context); the output of that call is then not meaningful.
constexpr uint32_t kErrBadInput = 2u;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of the given parity to complete; false after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 4-D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

}  // namespace dqd
