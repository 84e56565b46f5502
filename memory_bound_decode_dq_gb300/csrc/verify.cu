// Speculative verify: the step right after the target's verify forward.
//
// Sources: "AcceptedTokens 阅读笔记", Algorithm 1 (greedy verify and state
// rollback): compare each draft with the target's greedy prediction from the
// first position, stop at the first mismatch, emit the matched prefix plus
// the target's own token, invalidate the rejected tail of the KV cache;
// "第 10 讲：推理" §6 (speculative sampling): accept draft x with probability
// min(1, q(x)/p(x)); on the first rejection draw from norm(max(q - p, 0));
// when every draft is accepted draw one more token from the target.
//
// Greedy: spec_argmax_kernel (a cluster of S CTAs per verify position, each
// streaming a contiguous share of the vocabulary with 16-byte loads; the
// shares' (value, index) pairs meet in rank 0 through distributed shared
// memory; ties go to the smallest token id) writes the target's predictions
// t_i; S grows when there are few positions, so that small batches still
// spread over the SMs; spec_accept_kernel (one thread per request,
// launched as a programmatic dependent) counts the leading matches a. The
// round's output is t_0 .. t_a: accepted drafts equal the predictions they
// were compared with.
//
// Sampling: spec_sample_kernel, one CTA per request. Thread 0 walks the
// drafts (the test u * p(x) < q(x) in binary32); the CTA then draws the one
// sampled token by inverse CDF over the vocabulary, with fp64 partial sums
// per thread, a block-wide scan, and a sequential walk inside the thread
// whose range holds the crossing.
#include "dqd_device.cuh"
#include "dqd_internal.h"

#include <cmath>

namespace dqd {
namespace {

constexpr int kArgmaxThreads = 512;
constexpr int kSampleThreads = 512;

// (value, index) with the larger value, the smaller index on ties.
__device__ __forceinline__ void arg_better(float& v, int& i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Eight logits (16 bytes) starting at token id `base`: the running (value,
// index) moves only when the chunk's maximum is strictly larger, so chunks
// visited in increasing id order keep the first maximum; three packed maxima
// and one compare per chunk, the scan for the index only on a new maximum.
__device__ __forceinline__ void arg_chunk(float& bv, int& bi, const uint4& x, int base) {
  const uint32_t m = bf16x2_max(bf16x2_max(x.x, x.y), bf16x2_max(x.z, x.w));
  const float mx = fmaxf(bf16_lo(m), bf16_hi(m));
  if (mx > bv) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    int e = 0;
#pragma unroll
    for (int j = 7; j >= 0; --j)  // the first element equal to the maximum
      if ((j & 1 ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1])) == mx) e = j;
    bv = mx;
    bi = base + e;
  }
}

__global__ void __launch_bounds__(kArgmaxThreads)
spec_argmax_kernel(const uint16_t* __restrict__ logits, int64_t vocab, int32_t* __restrict__ out) {
  grid_dependency_wait();  // the logits come from the previous kernel
  allow_dependent_launch();
  const int64_t row = blockIdx.y;
  const int S = gridDim.x, rank = blockIdx.x;  // the CTAs of one row form a cluster along x
  const uint16_t* lr = logits + row * vocab;
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  if ((vocab & 7) == 0) {
    // 16-byte loads, four in flight per thread, over this CTA's share
    const uint4* v4 = reinterpret_cast<const uint4*>(lr);
    const int64_t units = vocab / 8;
    const int64_t per = (units + S - 1) / S;
    const int64_t n4 = min(units, (rank + 1) * per);
    int64_t u = rank * per + threadIdx.x;
    for (; u + 3 * kArgmaxThreads < n4; u += 4 * kArgmaxThreads) {
      uint4 x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j] = ldg_stream(v4 + u + j * kArgmaxThreads);
#pragma unroll
      for (int j = 0; j < 4; ++j) arg_chunk(bv, bi, x[j], (int)(8 * (u + j * kArgmaxThreads)));
    }
    for (; u < n4; u += kArgmaxThreads) arg_chunk(bv, bi, ldg_stream(v4 + u), (int)(8 * u));
  } else {
    const int64_t per = (vocab + S - 1) / S;
    const int64_t end = min(vocab, (rank + 1) * per);
    for (int64_t j = rank * per + threadIdx.x; j < end; j += kArgmaxThreads)
      arg_better(bv, bi, __uint_as_float((uint32_t)lr[j] << 16), (int)j);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    arg_better(bv, bi, ov, oi);
  }
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ int si[kArgmaxThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kArgmaxThreads / 32 ? sv[lane] : -INFINITY;
    bi = lane < kArgmaxThreads / 32 ? si[lane] : 0x7FFFFFFF;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      arg_better(bv, bi, ov, oi);
    }
    if (lane == 0) {
      sv[0] = bv;
      si[0] = bi;
    }
  }
  if (S > 1) {
    // rank 0 takes the best of the cluster's shares, in rank order
    cluster_sync_all();
    if (rank == 0 && threadIdx.x == 0) {
      const uint32_t av = smem_addr(&sv[0]), ai = smem_addr(&si[0]);
      for (int r = 1; r < S; ++r)
        arg_better(bv, bi, ld_dsmem_f32(av, (uint32_t)r), (int)ld_dsmem_u32(ai, (uint32_t)r));
    }
    cluster_sync_all();  // peers stay alive until their shares have been read
  }
  // a row of -inf only: the first token
  if (rank == 0 && threadIdx.x == 0) out[row] = bi == 0x7FFFFFFF ? 0 : bi;
}

__global__ void spec_accept_kernel(const int32_t* __restrict__ draft, int32_t* __restrict__ out,
                                   int32_t* __restrict__ count, int32_t* __restrict__ ctx, int b, int w) {
  grid_dependency_wait();  // the predictions come from spec_argmax_kernel
  allow_dependent_launch();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= b) return;
  int a = 0;
  while (a < w - 1 && draft[(int64_t)r * (w - 1) + a] == out[(int64_t)r * w + a]) ++a;
  count[r] = a + 1;
  if (ctx) ctx[r] -= (w - 1) - a;
}

// Residual mass of token y: max(q - p, 0) in binary32, or q itself.
__device__ __forceinline__ float residual(const float* q, const float* p, int64_t y) {
  return p ? fmaxf(q[y] - p[y], 0.f) : q[y];
}

// Inverse CDF over one vocabulary row, by the whole CTA: the smallest y with
// sum_{z<=y} r(z) > u * sum_z r(z), sums in fp64. Thread t owns a contiguous
// range of the vocabulary; a scan of the thread sums gives every range its
// bounds [lo, hi), built so that hi of one thread is bitwise lo of the next,
// hence exactly one thread holds the threshold and walks its range. Returns
// -1 when the total is not positive.
__device__ int64_t inverse_cdf(const float* q, const float* p, int64_t vocab, double u, double* sred,
                               long long* spick) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kSampleThreads / 32;
  const int64_t chunk = (vocab + kSampleThreads - 1) / kSampleThreads;
  const int64_t y0 = min(vocab, tid * chunk), y1 = min(vocab, y0 + chunk);
  double part = 0.0;
  for (int64_t y = y0; y < y1; ++y) part += (double)residual(q, p, y);
  double incl = part;  // inclusive scan inside the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  double excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.0;
  if (lane == 31) sred[warp] = incl;
  if (tid == 0) *spick = -1;
  __syncthreads();
  if (warp == 0) {
    double wv = lane < NW ? sred[lane] : 0.0;  // inclusive scan of the warp totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double v = __shfl_up_sync(0xffffffffu, wv, o);
      if (lane >= o) wv += v;
    }
    if (lane < NW) sred[NW + lane] = wv;
  }
  __syncthreads();
  const double total = sred[2 * NW - 1];
  const double wo = warp > 0 ? sred[NW + warp - 1] : 0.0;
  const double lo = wo + excl;
  const double hi = lane == 31 ? sred[NW + warp] : wo + incl;
  if (total > 0.0) {
    const double thr = u * total;
    if (lo <= thr && thr < hi) {
      double acc = lo;
      int64_t pick = -1, last = -1;
      for (int64_t y = y0; y < y1; ++y) {
        const float r = residual(q, p, y);
        if (r > 0.f) last = y;
        acc += (double)r;
        if (acc > thr) {
          pick = y;
          break;
        }
      }
      *spick = pick >= 0 ? pick : last;  // last: the walk's rounding stayed below thr
    }
  }
  __syncthreads();
  const long long pick = *spick;
  __syncthreads();
  return total > 0.0 ? (int64_t)pick : -1;
}

__global__ void __launch_bounds__(kSampleThreads)
spec_sample_kernel(const float* __restrict__ p, const float* __restrict__ q, const int32_t* __restrict__ draft,
                   const float* __restrict__ u_accept, const float* __restrict__ u_sample, int K, int64_t vocab,
                   int32_t* __restrict__ out, int32_t* __restrict__ count, int32_t* __restrict__ ctx) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int64_t b = blockIdx.x;
  __shared__ int s_j;
  __shared__ double sred[2 * (kSampleThreads / 32)];
  __shared__ long long spick;
  if (threadIdx.x == 0) {
    int j = 0;
    while (j < K) {
      const int32_t x = draft[b * K + j];
      if (x < 0 || x >= vocab) break;
      const float px = p[(b * K + j) * vocab + x], qx = q[(b * (K + 1) + j) * vocab + x];
      if (!(u_accept[b * K + j] * px < qx)) break;
      out[b * (K + 1) + j] = x;
      ++j;
    }
    s_j = j;
  }
  __syncthreads();
  const int j = s_j;
  const float* qrow = q + (b * (K + 1) + j) * vocab;
  const float* prow = j < K ? p + (b * K + j) * vocab : nullptr;
  const double u = (double)u_sample[b];
  int64_t y = inverse_cdf(qrow, prow, vocab, u, sred, &spick);
  if (y < 0 && prow) y = inverse_cdf(qrow, nullptr, vocab, u, sred, &spick);  // residual lost to rounding
  if (threadIdx.x == 0) {
    out[b * (K + 1) + j] = (int32_t)(y < 0 ? 0 : y);
    count[b] = j + 1;
    if (ctx) ctx[b] -= K - j;
  }
}

}  // namespace

static int verify_argmax_split(int64_t rows, int64_t vocab, int num_sms) {
  // up to 8 CTAs per row while the rows alone fill fewer than 2 CTAs per SM,
  // each keeping at least 4096 logits
  int S = 1;
  while (S < 8 && rows * S < 2 * (int64_t)num_sms && vocab / (2 * S) >= 4096) S *= 2;
  return S;
}

cudaError_t launch_spec_verify_greedy(const uint16_t* logits, int b, int w, int64_t vocab, const int32_t* draft,
                                      int32_t* out, int32_t* count, int32_t* ctx, int num_sms, cudaStream_t s) {
  const int64_t rows = (int64_t)b * w;
  const int S = verify_argmax_split(rows, vocab, num_sms);
  cudaError_t e = S > 1 ? launch_pdl_cluster_x(spec_argmax_kernel, dim3((unsigned)S, (unsigned)rows),
                                                dim3(kArgmaxThreads), 0, s, (unsigned)S, logits, vocab, out)
                        : launch_pdl(spec_argmax_kernel, dim3(1, (unsigned)rows), dim3(kArgmaxThreads), 0, s,
                                     logits, vocab, out);
  if (e != cudaSuccess) return e;
  return launch_pdl(spec_accept_kernel, dim3((unsigned)((b + 127) / 128)), dim3(128), 0, s, draft, out, count, ctx,
                    b, w);
}

cudaError_t launch_spec_verify_sample(const float* p, const float* q, const int32_t* draft, const float* u_accept,
                                      const float* u_sample, int b, int k, int64_t vocab, int32_t* out,
                                      int32_t* count, int32_t* ctx, cudaStream_t s) {
  return launch_pdl(spec_sample_kernel, dim3((unsigned)b), dim3(kSampleThreads), 0, s, p, q, draft, u_accept,
                    u_sample, k, vocab, out, count, ctx);
}

}  // namespace dqd
