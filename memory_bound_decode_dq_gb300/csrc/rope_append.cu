// rope_kv_append: rotary embedding of the new tokens' q and k, and the
// append of their k and v to the paged KV cache (bf16 or FP8-E4M3).
//
// Source: "第 10 讲：推理" §2.2-2.3 (KV cache): for every new token compute q,
// k, v; rotate q and k at the token's global position (start .. end-1, not
// from 0); write k and v into the cache at those positions; then attend.
// Rotary form: dims (2i, 2i+1) of a head turn by pos * base^(-2i/d).
//
// One CTA per new token (sequence b, verify position i; position
// pos = context_lens[b] - w + i, so the cache already counts the new tokens,
// as the attention expects). Threads 0 .. d/2-1 first build the token's
// cos/sin table: the angle pos * theta_i and its reduction to [-pi, pi] in
// double (pos reaches 2^17 and more, where a binary32 angle would be off by
// 1e-2), then sin and cos in binary32. Every thread then rotates (head, pair)
// units of the token's qkv row in binary32: q heads to q_out (bf16, the
// attention's layout), k heads into the K pool, v heads copied into the V
// pool, at slot pos % 16 of physical block block_table[b][pos / 16]. For an
// FP8 pool the value is divided by the pool's scale (IEEE binary32) and
// rounded to E4M3 with saturation, like quant_fp8_rowwise.
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

template <bool F8>
__global__ void __launch_bounds__(kRopeThreads)
rope_kv_append_kernel(const uint16_t* __restrict__ qkv, int w, int hq, int hkv, int d, double log2_base,
                      const int32_t* __restrict__ table, int max_blocks, const int32_t* __restrict__ ctx,
                      int64_t num_blocks, void* __restrict__ k_pool, void* __restrict__ v_pool, float k_scale,
                      float v_scale, uint16_t* __restrict__ q_out) {
  grid_dependency_wait();  // qkv comes from the projection kernel
  allow_dependent_launch();
  __shared__ float s_cos[kMaxHalfD], s_sin[kMaxHalfD];
  const int64_t row = blockIdx.x;
  const int b = (int)(row / w), i = (int)(row % w);
  const int64_t pos = (int64_t)ctx[b] - w + i;
  const int half = d / 2;
  if (threadIdx.x < half) {
    const double theta = exp2(-2.0 * (double)threadIdx.x / (double)d * log2_base);
    const double a = (double)pos * theta;
    const double two_pi = 6.283185307179586476925286766559;
    const double r = a - two_pi * rint(a / two_pi);  // in [-pi, pi]
    float sv, cv;
    sincosf((float)r, &sv, &cv);
    s_cos[threadIdx.x] = cv;
    s_sin[threadIdx.x] = sv;
  }
  __syncthreads();
  // where this token's k and v go (none for a position outside the table)
  int64_t kv_row = -1;
  if (pos >= 0 && pos / 16 < max_blocks) {
    int32_t phys = table[(int64_t)b * max_blocks + pos / 16];
    phys = phys < 0 ? 0 : (phys >= num_blocks ? (int32_t)(num_blocks - 1) : phys);
    kv_row = (int64_t)phys * hkv * 16 + pos % 16;  // + head * 16
  }
  const uint32_t* src = reinterpret_cast<const uint32_t*>(qkv + row * (int64_t)(hq + 2 * hkv) * d);
  const int units = (hq + 2 * hkv) * half;
  for (int u = threadIdx.x; u < units; u += kRopeThreads) {
    const int head = u / half, p = u % half;
    const uint32_t x = src[u];  // dims 2p, 2p+1 of head `head`
    float x0 = __uint_as_float(x << 16), x1 = __uint_as_float(x & 0xFFFF0000u);
    if (head < hq + hkv) {  // q and k rotate
      const float c = s_cos[p], s = s_sin[p];
      const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
      x0 = y0;
      x1 = y1;
    }
    if (head < hq) {
      reinterpret_cast<uint32_t*>(q_out + (row * hq + head) * (int64_t)d)[p] = pack_bf16x2(x0, x1);
      continue;
    }
    if (kv_row < 0) continue;
    const bool is_k = head < hq + hkv;
    const int g = is_k ? head - hq : head - hq - hkv;
    const int64_t elem = ((kv_row + (int64_t)g * 16) * d) + 2 * p;
    void* pool = is_k ? k_pool : v_pool;
    if constexpr (F8) {
      const float sc = is_k ? k_scale : v_scale;
      reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(pool) + elem)[0] =
          e4m3x2(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
    } else {
      reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(pool) + elem)[0] =
          is_k ? pack_bf16x2(x0, x1) : x;  // v: the bits as they came
    }
  }
}

}  // namespace

cudaError_t launch_rope_kv_append(const uint16_t* qkv, int b, int w, int hq, int hkv, int d, double rope_base,
                                  const int32_t* table, int max_blocks, const int32_t* ctx, int64_t num_blocks,
                                  void* k_pool, void* v_pool, bool kv_fp8, float k_scale, float v_scale,
                                  uint16_t* q_out, cudaStream_t s) {
  const dim3 grid((unsigned)((int64_t)b * w));
  const double l2b = std::log2(rope_base);
  if (kv_fp8)
    return launch_pdl(rope_kv_append_kernel<true>, grid, dim3(kRopeThreads), 0, s, qkv, w, hq, hkv, d, l2b, table,
                      max_blocks, ctx, num_blocks, k_pool, v_pool, k_scale, v_scale, q_out);
  return launch_pdl(rope_kv_append_kernel<false>, grid, dim3(kRopeThreads), 0, s, qkv, w, hq, hkv, d, l2b, table,
                    max_blocks, ctx, num_blocks, k_pool, v_pool, k_scale, v_scale, q_out);
}

}  // namespace dqd
