// rope_kv_append: rotary embedding of the new tokens' q and k, and the
// append of their k and v to the paged KV cache (bf16 or FP8-E4M3).
//
// Source: "第 10 讲：推理" §2.2-2.3 (KV cache): for every new token compute q,
// k, v; rotate q and k at the token's global position (start .. end-1, not
// from 0); write k and v into the cache at those positions; then attend.
// Rotary form: dims (2i, 2i+1) of a head turn by pos * base^(-2i/d).
//
// Grid: (new token, group of 256 (head, pair) units). Token (b, i) sits at
// position pos = context_lens[b] - w + i, so the cache already counts the new
// tokens, as the attention expects. Each thread owns VEC consecutive pairs
// (2p, 2p+1) of one head of the token's qkv row and rotates them with
// rope_rotate (rope_device.cuh: the angle reduced exactly in turns, sin and
// cos and the rotation in binary32). q heads go to q_out (bf16, the
// attention's layout), k heads into the K pool, v heads are copied into the V
// pool, at slot pos % 16 of physical block block_table[b][pos / 16]. For an
// FP8 pool the value is divided by the pool's scale (IEEE binary32) and
// rounded to E4M3 with saturation, like quant_fp8_rowwise.
#include "dqd_device.cuh"
#include "dqd_internal.h"
#include "rope_device.cuh"

#include <cmath>

namespace dqd {
namespace {

constexpr int kRopeThreads = 256;

// Device error word of this module (kErrBadInput when a block-table entry was
// clamped into the pool).
__device__ unsigned int g_rope_error;

constexpr int kMaxHalfD = kRopeMaxHalfD;

struct RopeFreqs {
  uint64_t turns[kMaxHalfD];  // base^(-2p/d) / 2pi as a fraction of 2^64, p < d/2
};

// Rotates dims (2p, 2p+1) held as one bf16 pair in x, at position pos.
__device__ __forceinline__ void rope_pair(uint32_t x, int64_t pos, uint64_t turns, float& x0, float& x1) {
  rope_rotate(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u), pos, turns, x0, x1);
}

// VEC consecutive pairs per thread (4 with 16-byte accesses when d % 8 == 0, else 1).
template <bool F8, int VEC>
__global__ void __launch_bounds__(kRopeThreads)
rope_kv_append_kernel(const uint16_t* __restrict__ qkv, int w, int hq, int hkv, int d,
                      const __grid_constant__ RopeFreqs freqs, const int32_t* __restrict__ table, int max_blocks,
                      const int32_t* __restrict__ ctx, int64_t num_blocks, void* __restrict__ k_pool,
                      void* __restrict__ v_pool, float k_scale, float v_scale, uint16_t* __restrict__ q_out) {
  grid_dependency_wait();  // qkv comes from the projection kernel
  allow_dependent_launch();
  const int64_t row = blockIdx.x;
  const int half = d / 2;
  const int u = (blockIdx.y * kRopeThreads + threadIdx.x) * VEC;  // first pair of this thread
  if (u >= (hq + 2 * hkv) * half) return;
  const int head = u / half, p = u % half;  // VEC divides half: the pairs share a head
  const int b = (int)(row / w), i = (int)(row % w);
  const int64_t pos = (int64_t)ctx[b] - w + i;
  const uint32_t* src = reinterpret_cast<const uint32_t*>(qkv + row * (int64_t)(hq + 2 * hkv) * d) + u;
  uint32_t x[VEC];
  if constexpr (VEC == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
  } else {
    x[0] = src[0];
  }
  const bool rotate = head < hq + hkv;
  uint32_t y[VEC];           // bf16 pairs out
  float f[VEC][2];           // binary32 values (FP8 pools)
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    if (rotate) {
      rope_pair(x[j], pos, freqs.turns[p + j], f[j][0], f[j][1]);
      y[j] = pack_bf16x2(f[j][0], f[j][1]);
    } else {
      f[j][0] = __uint_as_float(x[j] << 16);
      f[j][1] = __uint_as_float(x[j] & 0xFFFF0000u);
      y[j] = x[j];  // v: the bits as they came
    }
  }
  uint32_t* dst;
  if (head < hq) {
    dst = reinterpret_cast<uint32_t*>(q_out + (row * hq + head) * (int64_t)d) + p;
  } else {
    if (pos < 0 || pos / 16 >= max_blocks) return;  // nowhere to append
    const int32_t entry = table[(int64_t)b * max_blocks + pos / 16];
    const int32_t phys = entry < 0 ? 0 : (entry >= num_blocks ? (int32_t)(num_blocks - 1) : entry);
    if (phys != entry) atomicOr(&g_rope_error, kErrBadInput);
    const int g = rotate ? head - hq : head - hq - hkv;
    const int64_t elem = (((int64_t)phys * hkv + g) * 16 + pos % 16) * d + 2 * p;
    void* pool = rotate ? k_pool : v_pool;
    if constexpr (F8) {
      const float sc = rotate ? k_scale : v_scale;
      uint16_t c[VEC];
#pragma unroll
      for (int j = 0; j < VEC; ++j) c[j] = e4m3x2_rn_satfinite(__fdiv_rn(f[j][0], sc), __fdiv_rn(f[j][1], sc));
      uint8_t* o = static_cast<uint8_t*>(pool) + elem;
      if constexpr (VEC == 4) {
        *reinterpret_cast<uint2*>(o) = make_uint2(c[0] | ((uint32_t)c[1] << 16), c[2] | ((uint32_t)c[3] << 16));
      } else {
        *reinterpret_cast<uint16_t*>(o) = c[0];
      }
      return;
    }
    dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(pool) + elem);
  }
  if constexpr (VEC == 4) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(y[0], y[1], y[2], y[3]);
  } else {
    dst[0] = y[0];
  }
}

}  // namespace

void rope_turns(double base, int d, int n, uint64_t* turns) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int p = 0; p < n; ++p) {
    const double t = std::pow(base, -2.0 * p / d) / two_pi;  // < 1/6: fits the fraction
    turns[p] = (uint64_t)std::ldexp(t, 64);
  }
}

cudaError_t rope_take_device_error(uint32_t* flags) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_rope_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_rope_error, &zero, sizeof zero);
  *flags |= v;
  return e;
}

cudaError_t launch_rope_kv_append(const uint16_t* qkv, int b, int w, int hq, int hkv, int d, double rope_base,
                                  const int32_t* table, int max_blocks, const int32_t* ctx, int64_t num_blocks,
                                  void* k_pool, void* v_pool, bool kv_fp8, float k_scale, float v_scale,
                                  uint16_t* q_out, cudaStream_t s) {
  RopeFreqs f{};
  rope_turns(rope_base, d, d / 2 < kMaxHalfD ? d / 2 : kMaxHalfD, f.turns);
  const int units = (hq + 2 * hkv) * (d / 2);
  const bool vec = d % 8 == 0;  // 4 pairs per thread, 16-byte rows and stores
  const int per_thread = vec ? 4 : 1;
  const dim3 grid((unsigned)((int64_t)b * w),
                  (unsigned)((units / per_thread + kRopeThreads - 1) / kRopeThreads));
#define DQD_ROPE_LAUNCH(F8, VEC)                                                                              \
  return launch_pdl(rope_kv_append_kernel<F8, VEC>, grid, dim3(kRopeThreads), 0, s, qkv, w, hq, hkv, d, f, table, \
                    max_blocks, ctx, num_blocks, k_pool, v_pool, k_scale, v_scale, q_out)
  if (kv_fp8) {
    if (vec) DQD_ROPE_LAUNCH(true, 4);
    DQD_ROPE_LAUNCH(true, 1);
  }
  if (vec) DQD_ROPE_LAUNCH(false, 4);
  DQD_ROPE_LAUNCH(false, 1);
#undef DQD_ROPE_LAUNCH
}

}  // namespace dqd
