// Rotary embedding of one (2i, 2i+1) pair and the store of one element of a
// QKV projection row into q_out or the paged KV cache. Shared by
// rope_kv_append (a kernel of its own) and the QKV dq_gemm epilogue that
// fuses it, so the two compute the same bits.
//
// Source: "第 10 讲：推理" (CS336 lecture 10 notes) §2.2-2.3: each new token's
// q and k are rotated at the token's global position and its k and v are
// written into the cache at that position before attending. Rotary form (the
// pages fix none; reading: the pairwise form): dims (2i, 2i+1) of a head turn
// by pos * base^(-2i/d).
#pragma once

#include "dqd_device.cuh"
#include "dqd_internal.h"

#include <cstdint>

namespace dqd {

constexpr int kRopeMaxHalfD = 256;

// The angle pos * theta_i is reduced exactly, in turns: theta_i / 2pi is held
// as a 64-bit fixed-point fraction F_i (computed once per call on the host),
// and pos * F_i mod 2^64 (an integer multiply) is the angle's fraction of a
// turn, good to 2^-45 turns for positions up to 2^20 (a binary32 angle would
// be off by 1e-2 rad there). Its top 32 bits, centred on [-1/2, 1/2] turns,
// feed sincospi in binary32. The rotation uses unfused binary32 products and
// sums, so every caller rounds alike.
__device__ __forceinline__ void rope_rotate(float x0, float x1, int64_t pos, uint64_t turns, float& y0,
                                            float& y1) {
  const uint64_t frac = (uint64_t)pos * turns;  // mod 2^64: the angle in turns
  float t = (float)(uint32_t)(frac >> 32) * 0x1p-32f;
  t -= rintf(t);  // [-1/2, 1/2] turns
  float sv, cv;
  sincospif(2.f * t, &sv, &cv);
  y0 = __fadd_rn(__fmul_rn(x0, cv), -__fmul_rn(x1, sv));
  y1 = __fadd_rn(__fmul_rn(x0, sv), __fmul_rn(x1, cv));
}

// E4M3 codes of (lo, hi): round to nearest even, saturating at +-448.
__device__ __forceinline__ uint16_t e4m3x2_rn_satfinite(float lo, float hi) {
  uint16_t pair;
  // cvt packs its first source into the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi), "f"(lo));
  return pair;
}

// Empty stand-in for the epilogue parameter of the plain dq_gemm kernels.
struct NoEpi {};

template <bool ROPE>
struct EpiOf {
  using type = NoEpi;
};
template <>
struct EpiOf<true> {
  using type = RopeEpi;
};

// Stores element (token mm = b * w + i, column nn) of a QKV projection whose
// row holds the heads q_0.., k_0.., v_0.. (head dim 128). v is this element's
// value as the projection rounds it (bf16, widened back to binary32); partner
// is the same for column nn ^ 1 of the same token. q and k columns are
// rotated as a pair at position ctx[b] - w + i: q goes to q_out, k and v to
// row pos % 16 of block table[b][pos / 16] (nothing when the position is
// below 0 or past the table). Returns true when a table entry outside
// [0, num_blocks) was clamped into range.
__device__ __forceinline__ bool rope_store_bi(const RopeEpi& r, int64_t mm, int b, int i, int64_t nn, float v,
                                              float partner) {
  const int head = (int)(nn >> 7), dim = (int)(nn & 127);
  const bool odd = dim & 1;
  const int64_t pos = (int64_t)r.ctx[b] - r.w + i;
  const bool rotated = head < r.hq + r.hkv;
  float val = v;
  if (rotated) {
    float y0, y1;
    rope_rotate(odd ? partner : v, odd ? v : partner, pos, r.turns[dim >> 1], y0, y1);
    val = odd ? y1 : y0;
  }
  if (head < r.hq) {
    r.q_out[(mm * r.hq + head) * 128 + dim] = f32_to_bf16(val);
    return false;
  }
  if (pos < 0 || pos / 16 >= r.max_blocks) return false;  // nowhere to append
  const int32_t entry = r.table[(int64_t)b * r.max_blocks + pos / 16];
  const int32_t phys = entry < 0 ? 0 : (entry >= r.num_blocks ? (int32_t)(r.num_blocks - 1) : entry);
  const int g = rotated ? head - r.hq : head - r.hq - r.hkv;
  const int64_t elem = (((int64_t)phys * r.hkv + g) * 16 + pos % 16) * 128 + dim;
  if (r.kv_fp8) {
    const float sc = rotated ? r.k_scale : r.v_scale;
    static_cast<uint8_t*>(rotated ? r.k_pool : r.v_pool)[elem] =
        (uint8_t)(e4m3x2_rn_satfinite(__fdiv_rn(val, sc), 0.f) & 0xFFu);
  } else {
    static_cast<uint16_t*>(rotated ? r.k_pool : r.v_pool)[elem] = f32_to_bf16(val);
  }
  return phys != entry;
}

// Eight consecutive dims [dim0, dim0 + 8) of head `head` for token mm = b * w
// + i, as four bf16 pairs in x: the same arithmetic and placement as
// rope_store_bi on each element, with 16-byte stores (8-byte for E4M3 codes).
__device__ __forceinline__ bool rope_store8(const RopeEpi& r, int64_t mm, int b, int i, int head, int dim0,
                                            uint4 x) {
  const int64_t pos = (int64_t)r.ctx[b] - r.w + i;
  const bool rotated = head < r.hq + r.hkv;
  uint32_t y[4];
  float f[4][2];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t xj = word(x, j);
    const float x0 = __uint_as_float(xj << 16), x1 = __uint_as_float(xj & 0xFFFF0000u);
    if (rotated) {
      rope_rotate(x0, x1, pos, r.turns[(dim0 >> 1) + j], f[j][0], f[j][1]);
      y[j] = pack_bf16x2(f[j][0], f[j][1]);
    } else {
      f[j][0] = x0;
      f[j][1] = x1;
      y[j] = xj;  // v: the bits as they came
    }
  }
  if (head < r.hq) {
    *reinterpret_cast<uint4*>(r.q_out + (mm * r.hq + head) * 128 + dim0) = make_uint4(y[0], y[1], y[2], y[3]);
    return false;
  }
  if (pos < 0 || pos / 16 >= r.max_blocks) return false;  // nowhere to append
  const int32_t entry = r.table[(int64_t)b * r.max_blocks + pos / 16];
  const int32_t phys = entry < 0 ? 0 : (entry >= r.num_blocks ? (int32_t)(r.num_blocks - 1) : entry);
  const int g = rotated ? head - r.hq : head - r.hq - r.hkv;
  const int64_t elem = (((int64_t)phys * r.hkv + g) * 16 + pos % 16) * 128 + dim0;
  if (r.kv_fp8) {
    const float sc = rotated ? r.k_scale : r.v_scale;
    uint16_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = e4m3x2_rn_satfinite(__fdiv_rn(f[j][0], sc), __fdiv_rn(f[j][1], sc));
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(rotated ? r.k_pool : r.v_pool) + elem) =
        make_uint2(c[0] | ((uint32_t)c[1] << 16), c[2] | ((uint32_t)c[3] << 16));
  } else {
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(rotated ? r.k_pool : r.v_pool) + elem) =
        make_uint4(y[0], y[1], y[2], y[3]);
  }
  return phys != entry;
}

// As rope_store_bi, with the token's sequence and position in it derived
// from mm.
__device__ __forceinline__ bool rope_store(const RopeEpi& r, int64_t mm, int64_t nn, float v, float partner) {
  return rope_store_bi(r, mm, (int)(mm / r.w), (int)(mm % r.w), nn, v, partner);
}

// The projection's bf16 rounding of an fp32 output, widened back to binary32.
__device__ __forceinline__ float bf16_round(float v) { return __uint_as_float((uint32_t)f32_to_bf16(v) << 16); }

}  // namespace dqd
