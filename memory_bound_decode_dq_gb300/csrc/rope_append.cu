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
// tokens, as the attention expects. Each thread owns one unit: dims 2p, 2p+1
// of one head of the token's qkv row. The angle pos * theta_p is reduced
// exactly, in turns: the host computes theta_p / 2pi (theta_p = base^(-2p/d))
// once per call as a 64-bit fixed-point fraction F_p, and pos * F_p mod 2^64
// (an integer multiply) is the angle's fraction of a turn to 2^-45 turns for
// positions up to 2^20 (a binary32 angle would be off by 1e-2 rad there, and
// fp64 arithmetic is scarce on this part); its top 32 bits, centred on
// [-1/2, 1/2) turns, feed sincospi in binary32, and the rotation is binary32. q heads go to q_out (bf16, the attention's layout), k heads
// into the K pool, v heads are copied into the V pool, at slot pos % 16 of
// physical block block_table[b][pos / 16]. For an FP8 pool the value is
// divided by the pool's scale (IEEE binary32) and rounded to E4M3 with
// saturation, like quant_fp8_rowwise.
#include "dqd_device.cuh"
#include "dqd_internal.h"

#include <cmath>

namespace dqd {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kMaxHalfD = 256;

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t pair;
  // cvt packs its first source into the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi), "f"(lo));
  return pair;
}

struct RopeFreqs {
  uint64_t turns[kMaxHalfD];  // base^(-2p/d) / 2pi as a fraction of 2^64, p < d/2
};

// Rotates dims (2p, 2p+1) held as one bf16 pair in x, at position pos.
__device__ __forceinline__ void rope_pair(uint32_t x, int64_t pos, uint64_t turns, float& x0, float& x1) {
  x0 = __uint_as_float(x << 16);
  x1 = __uint_as_float(x & 0xFFFF0000u);
  const uint64_t frac = (uint64_t)pos * turns;  // mod 2^64: the angle in turns
  float t = (float)(uint32_t)(frac >> 32) * 0x1p-32f;
  t -= rintf(t);  // [-1/2, 1/2] turns
  float sv, cv;
  sincospif(2.f * t, &sv, &cv);
  const float y0 = x0 * cv - x1 * sv, y1 = x0 * sv + x1 * cv;
  x0 = y0;
  x1 = y1;
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
    int32_t phys = table[(int64_t)b * max_blocks + pos / 16];
    phys = phys < 0 ? 0 : (phys >= num_blocks ? (int32_t)(num_blocks - 1) : phys);
    const int g = rotate ? head - hq : head - hq - hkv;
    const int64_t elem = (((int64_t)phys * hkv + g) * 16 + pos % 16) * d + 2 * p;
    void* pool = rotate ? k_pool : v_pool;
    if constexpr (F8) {
      const float sc = rotate ? k_scale : v_scale;
      uint16_t c[VEC];
#pragma unroll
      for (int j = 0; j < VEC; ++j) c[j] = e4m3x2(__fdiv_rn(f[j][0], sc), __fdiv_rn(f[j][1], sc));
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

cudaError_t launch_rope_kv_append(const uint16_t* qkv, int b, int w, int hq, int hkv, int d, double rope_base,
                                  const int32_t* table, int max_blocks, const int32_t* ctx, int64_t num_blocks,
                                  void* k_pool, void* v_pool, bool kv_fp8, float k_scale, float v_scale,
                                  uint16_t* q_out, cudaStream_t s) {
  RopeFreqs f{};
  const double two_pi = 6.283185307179586476925286766559;
  for (int p = 0; p < d / 2 && p < kMaxHalfD; ++p) {
    const double turns = std::pow(rope_base, -2.0 * p / d) / two_pi;  // < 1/6: fits the fraction
    f.turns[p] = (uint64_t)std::ldexp(turns, 64);
  }
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
