// Offline weight preparation: pack_int4_g128, quant_fp8_rowwise and
// quant_int4_g128.
//
// Source: "降低每個 Token 的生成成本" (Making each token cheaper), section "格式"
// (Formats): weight-only INT4 keeps 4-bit integers with one scale per group
// of 128; E4M3 has 4 exponent and 3 mantissa bits with largest normal 448,
// and values are multiplied by a scale before the cast.
#include "dqd_device.cuh"
#include "dqd_internal.h"

#include <algorithm>

namespace dqd {
namespace {

// One thread per 32-bit word of the packed code stream. Word w of block
// (T, g): h = w/128, l = (w/4)%32, j = w%4; i = 4h+j, c = i/2, e = i%2,
// r0 = l/4, t = l%4; nibble v <- code[16T + r0 + 8(v&1)][128g + 32c + 8t + 4e
// + 2((v>>1)&1) + (v>>2)], rows past n -> 0.
__global__ void pack_int4_codes_kernel(const uint8_t* __restrict__ codes, int64_t n, int64_t k,
                                       uint32_t* __restrict__ packed, int64_t words) {
  const int64_t G = k / 128;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < words;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t blk = idx / 256;
    const int w = (int)(idx % 256);
    const int64_t T = blk / G, grp = blk % G;
    const int h = w / 128, l = (w / 4) % 32, j = w % 4;
    const int i = 4 * h + j, c = i / 2, e = i % 2, r0 = l / 4, t = l % 4;
    const int64_t col0 = 128 * grp + 32 * c + 8 * t + 4 * e;
    uint32_t word = 0;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int64_t row = 16 * T + r0 + 8 * (v & 1);
      const int64_t col = col0 + 2 * ((v >> 1) & 1) + (v >> 2);
      const uint32_t q = row < n ? (codes[row * k + col] & 15u) : 0u;
      word |= q << (4 * v);
    }
    packed[idx] = word;
  }
}

// One thread per (block, r0): scale word and zero byte of rows 16T+r0, +8.
__global__ void pack_int4_meta_kernel(const uint16_t* __restrict__ scales,
                                      const uint8_t* __restrict__ zeros, int64_t n, int64_t k,
                                      uint32_t* __restrict__ pscales, uint8_t* __restrict__ pzeros,
                                      int64_t entries) {
  const int64_t G = k / 128;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < entries;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t blk = idx / 8;
    const int r0 = (int)(idx % 8);
    const int64_t T = blk / G, grp = blk % G;
    const int64_t lo = 16 * T + r0, hi = lo + 8;
    const uint32_t slo = lo < n ? scales[lo * G + grp] : 0u;
    const uint32_t shi = hi < n ? scales[hi * G + grp] : 0u;
    const uint32_t zlo = lo < n ? (zeros[lo * G + grp] & 15u) : 0u;
    const uint32_t zhi = hi < n ? (zeros[hi * G + grp] & 15u) : 0u;
    pscales[idx] = slo | (shi << 16);
    pzeros[idx] = (uint8_t)(zlo | (zhi << 4));
  }
}

// One CTA per row: row max of |w| (exact), scale = max / 448 (IEEE fp32
// division), code = E4M3 RNE-satfinite of w / scale (IEEE fp32 division).
constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads)
quant_fp8_kernel(const uint16_t* __restrict__ w, int64_t n, int64_t k, uint8_t* __restrict__ codes,
                 float* __restrict__ scales) {
  const int64_t row = blockIdx.x;
  const uint16_t* wr = w + row * k;
  float amax = 0.f;
  for (int64_t j = threadIdx.x * 8; j < k; j += kQuantThreads * 8) {
    if (j + 8 <= k) {
      const uint4 v = *reinterpret_cast<const uint4*>(wr + j);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(u[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(u[i] & 0xFFFF0000u)));
      }
    } else {
      for (int64_t jj = j; jj < k; ++jj) amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)wr[jj] << 16)));
    }
  }
  __shared__ float red[kQuantThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < kQuantThreads / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float rmax = red[0];
  const float scale = rmax > 0.f ? __fdiv_rn(rmax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) scales[row] = scale;
  uint8_t* cr = codes + row * k;
  for (int64_t j = threadIdx.x * 2; j < k; j += kQuantThreads * 2) {
    const float v0 = __fdiv_rn(__uint_as_float((uint32_t)wr[j] << 16), scale);
    const float v1 = __fdiv_rn(__uint_as_float((uint32_t)wr[j + 1] << 16), scale);
    uint16_t pair;
    // cvt packs its first source into the upper byte.
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(v1), "f"(v0));
    *reinterpret_cast<uint16_t*>(cr + j) = pair;
  }
}

}  // namespace

cudaError_t launch_pack_int4(const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                             int64_t n, int64_t k, void* packed, void* pscales, void* pzeros,
                             cudaStream_t s) {
  const int64_t blocks = ((n + 15) / 16) * (k / 128);
  const int64_t words = blocks * 256, entries = blocks * 8;
  const int threads = 256;
  const int64_t g1 = std::min<int64_t>((words + threads - 1) / threads, 1 << 20);
  pack_int4_codes_kernel<<<(unsigned)g1, threads, 0, s>>>(codes, n, k, static_cast<uint32_t*>(packed),
                                                          words);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t g2 = std::min<int64_t>((entries + threads - 1) / threads, 1 << 20);
  pack_int4_meta_kernel<<<(unsigned)g2, threads, 0, s>>>(scales, zeros, n, k,
                                                         static_cast<uint32_t*>(pscales),
                                                         static_cast<uint8_t*>(pzeros), entries);
  return cudaGetLastError();
}

cudaError_t launch_quant_fp8(const uint16_t* w, int64_t n, int64_t k, uint8_t* codes, float* scales,
                             cudaStream_t s) {
  quant_fp8_kernel<<<(unsigned)n, kQuantThreads, 0, s>>>(w, n, k, codes, scales);
  return cudaGetLastError();
}

namespace {

// INT4 asymmetric min/max quantiser: one warp per (row, 128-group), 8 groups
// per CTA. Lane l holds weights 4l .. 4l+3 of the group. Every step that
// decides an integer is IEEE binary32 with round-to-nearest-even, so codes,
// scales and zeros are reproducible bit for bit.
constexpr int kInt4QuantWarps = 8;

__global__ void __launch_bounds__(kInt4QuantWarps * 32)
quant_int4_kernel(const uint16_t* __restrict__ w, int64_t n, int64_t k, uint8_t* __restrict__ codes,
                  uint16_t* __restrict__ scales, uint8_t* __restrict__ zeros) {
  const int lane = threadIdx.x & 31;
  const int64_t G = k / 128;
  const int64_t unit = (int64_t)blockIdx.x * kInt4QuantWarps + (threadIdx.x >> 5);
  if (unit >= n * G) return;
  const int64_t row = unit / G, g = unit % G;
  const int64_t off = row * k + g * 128 + 4 * lane;
  const uint2 raw = *reinterpret_cast<const uint2*>(w + off);
  const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  // the range always holds 0, so 0 stays exactly on the grid
  float lo = 0.f, hi = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo = fminf(lo, v[i]);
    hi = fmaxf(hi, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const float d = hi - lo;
  uint16_t sb = 0x3F80u;  // a group of zeros takes scale 1
  if (d > 0.f) {
    sb = f32_to_bf16(__fdiv_rn(d, 15.0f));
    if ((sb & 0x7FFFu) == 0) sb = 0x0001u;  // keep the scale positive
  }
  const float sf = __uint_as_float((uint32_t)sb << 16);
  const float zf = fminf(fmaxf(rintf(__fdiv_rn(-lo, sf)), 0.f), 15.f);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float q = fminf(fmaxf(rintf(__fdiv_rn(v[i], sf)) + zf, 0.f), 15.f);
    packed |= (uint32_t)q << (8 * i);
  }
  *reinterpret_cast<uint32_t*>(codes + off) = packed;
  if (lane == 0) {
    scales[row * G + g] = sb;
    zeros[row * G + g] = (uint8_t)zf;
  }
}

}  // namespace

cudaError_t launch_quant_int4(const uint16_t* w, int64_t n, int64_t k, uint8_t* codes, uint16_t* scales,
                              uint8_t* zeros, cudaStream_t s) {
  const int64_t units = n * (k / 128);
  if (units == 0) return cudaSuccess;
  const int64_t blocks = (units + kInt4QuantWarps - 1) / kInt4QuantWarps;
  quant_int4_kernel<<<(unsigned)blocks, kInt4QuantWarps * 32, 0, s>>>(w, n, k, codes, scales, zeros);
  return cudaGetLastError();
}

}  // namespace dqd
