// gqa_decode_attn: paged GQA decode / speculative-verify attention.
//
// Sources: "第 10 讲：推理" (CS336 lecture 10 notes) §2.2 — append the new
// tokens' K,V, then each new query attends to all cached K,V; "LLM 推理是怎么
// 变快的" §2.1 softmax(q K^T / sqrt(d)) V, §2.3 GQA (query heads share KV heads),
// §3.1 PagedAttention (16-token blocks + block table), §6.1 online softmax is
// exact; "降低每個 Token 的生成成本" (Making each token cheaper), section
// "注意力 Kernel": Flash-Decoding splits K/V into chunks processed in parallel
// and combines them; "AcceptedTokens 阅读笔记", Algorithm 1: the verify
// positions go through one causal forward.
//
// Work item = (sequence b, kv head g, chunk of the context, group of up to
// four 16-row query tiles). The query rows of one kv head are the G = Hq/Hkv
// heads at each of the W verify positions (row r -> position r / G, head
// g*G + r % G). A CTA has 4 warps: warp = (query tile, key slot); the KS = 4/QT
// key slots split each pipeline stage's blocks between them.
//
//  * K/V blocks (4 KB each per kv head in bf16, 2 KB in FP8) are gathered
//    through the block table by TMA into a shared-memory ring per key slot,
//    128-byte swizzled (16-byte unit u of a 128-byte row r sits at u ^ (r & 7)).
//  * S = Q K^T and O += P V run on mma.m16n8k16 (bf16 in, fp32 accumulate).
//    The head dimension is permuted the same way for Q and K (lane t owns 16
//    consecutive d per 64 in bf16, per 32 in FP8). For PV the B operand needs
//    V[key 2t][d], V[key 2t+1][d] in one register: the lane loads consecutive
//    d of four keys and pairs them with prmt.
//  * FP8-E4M3 cache ("LLM 推理是怎么变快的" §4.2 C, KV cache quantisation):
//    codes are widened to bf16 exactly in registers (every E4M3 value is a
//    bf16 value); k_scale folds into the logit scale and v_scale into the
//    output, so the MMAs see the codes' values unscaled.
//  * Online softmax in the log2 domain (ex2), masked keys -> -inf by select:
//    key j is visible to row r iff j <= ctx - W + r / G. V rows past the
//    context are zeroed before the MMA so stale pool contents cannot leak.
//  * Warps sharing a query tile merge through shared memory; the CTA then
//    either writes the normalised bf16 output (one chunk) or an fp32 partial
//    (o, m, l) that attn_merge_kernel combines per output row.
#include "dqd_device.cuh"
#include "dqd_internal.h"
#include "tcgen05.cuh"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>

namespace dqd {
namespace {

constexpr int kD = 128;
constexpr int kBlk = 16;
constexpr int kThreads = 128;
constexpr int kBlockBytes = kBlk * kD * 2;  // one block, one kv head, K or V
constexpr float kNegInf = -INFINITY;

struct Args {
  const uint16_t* q;
  const int32_t* table;
  const int32_t* ctx;
  uint16_t* out;
  float* part_o;   // [rows][nchunks][128]
  float* part_ml;  // [rows][nchunks][2]
  int64_t num_blocks;
  int max_blocks, max_context, B, W, Hq, Hkv, G, QR;
  int chunk_blocks, nchunks, qgroups;
  float scale_log2;  // softmax scale (times k_scale for FP8) times log2(e)
  float v_scale;     // 1 for bf16
  // tensor-core form, balanced tail: the last tail_items work items (sequence,
  // kv head) are split into tail_pieces pieces of whole tiles, whose partials
  // (tail_o [tail row][piece][128], tail_ml [tail row][piece][2]) the tail
  // merge combines; the other items run whole
  int tail_items, tail_pieces;
  float* tail_o;
  float* tail_ml;
  uint8_t* tail_seq;  // [kLptMaxB] the longest-first order, written by CTA 0 for the tail merge
  // persistent tensor-core form: the work queue's ticket and finished-CTA
  // count (the workspace's counter region; zero on entry and on exit)
  unsigned* ctr;
  int lpt;  // tensor-core forms: 1 = longest-first order of the sequences (B <= kLptMaxB)
};

// Per-module device error word (kErrWaitTimeout when a bounded wait gave up,
// kErrBadInput when an input was clamped into range).
__device__ unsigned int g_attn_error;

// The context of sequence b, clamped to what the block table and the split
// plan (sized from the caller's max_context) can cover.
__device__ __forceinline__ int seq_ctx(const Args& a, int b) {
  const int c = a.ctx[b];
  return max(0, min(c, min(a.max_context, a.max_blocks * kBlk)));
}

template <int QT, bool F8>
struct Cfg {
  static constexpr int KS = 4 / QT;  // key-slot groups per CTA
  // ring slots per group: bf16 96/64/48 KB in all, FP8 64/64/48 KB
  static constexpr int NS = F8 ? (QT == 1 ? 4 : (QT == 2 ? 8 : 12)) : (QT == 1 ? 3 : (QT == 2 ? 4 : 6));
  // bf16: K (2 x 2 KB) + V (2 x 2 KB); FP8: K (2 KB) + V (2 KB)
  static constexpr int SLOT = F8 ? kBlockBytes : 2 * kBlockBytes;
  static constexpr int RING = KS * NS * SLOT;
  static constexpr int MERGE = 4 * 16 * (kD + 2) * 4;     // (o, m, l) per warp-row
  static constexpr int BODY = RING > MERGE ? RING : MERGE;
  static constexpr int BARS = 2 * KS * NS * 8;            // full + empty mbarriers
  static constexpr int BYTES = 1024 + BODY + BARS;        // + alignment slack
};

// bf16: K and V of one (block, kv head) arrive as four 2 KB TMA boxes of 16
// rows x 64 head dims, 128-byte swizzled: 16-byte unit u of row r sits at unit
// u ^ (r & 7) of that row. Offsets inside a slot: K d<64, K d>=64, V d<64, V d>=64.
// FP8: two 2 KB boxes of 16 rows x 128 codes, same swizzle: K, then V.
__device__ __forceinline__ uint32_t kv_unit(uint32_t half_base, int row, int unit) {
  return half_base + row * 128 + ((unit ^ (row & 7)) << 4);
}

// Four E4M3 codes (bytes 0..3 of u) -> two f16x2 (codes 0,1 and 2,3), exact:
// every E4M3 value is an f16 value.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t u, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(u));
}

template <int QT, bool F8>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(const __grid_constant__ CUtensorMap tmk,
                                                              const __grid_constant__ CUtensorMap tmv,
                                                              const Args a) {
  using C = Cfg<QT, F8>;
  constexpr int KS = C::KS, NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;
  const int chunk = blockIdx.x, g = blockIdx.y;
  const int b = blockIdx.z / a.qgroups, qg = blockIdx.z % a.qgroups;
  grid_dependency_wait();  // q, the tables and the cache may come from the previous kernel
  allow_dependent_launch();
  const int ctx = seq_ctx(a, b);
  if (chunk == 0 && g == 0 && qg == 0 && threadIdx.x == 0) {
    // one CTA per sequence reports a context outside [w, max_context]
    const int raw = a.ctx[b];
    if (raw < a.W || raw != ctx) atomicOr(&g_attn_error, kErrBadInput);
  }
  const int nblk_seq = (ctx + kBlk - 1) / kBlk;
  const int blk0 = chunk * a.chunk_blocks;
  if (blk0 >= nblk_seq) {  // whole CTA: nothing of this sequence here
    if (a.nchunks == 1 && nblk_seq == 0) {
      // empty context: the rows see no key and are written as zeros
      for (int i = threadIdx.x; i < QT * 16 * kD / 2; i += kThreads) {
        const int r = (qg * QT) * 16 + i / (kD / 2);
        if (r < a.QR) {
          const int64_t orow = ((int64_t)b * a.W + r / a.G) * a.Hq + g * a.G + r % a.G;
          reinterpret_cast<uint32_t*>(a.out + orow * kD)[i % (kD / 2)] = 0u;
        }
      }
    }
    return;
  }
  const int blk_end = min(blk0 + a.chunk_blocks, nblk_seq);
  const int qt = warp % QT, grp = warp / QT;
  const bool leader = qt == 0;
  const int row_base = (qg * QT + qt) * 16;  // first query row of this warp's tile

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t bars = ring + C::BODY;
  auto full_bar = [&](int s) { return bars + (grp * NS + s) * 8; };
  auto empty_bar = [&](int s) { return bars + (KS * NS + grp * NS + s) * 8; };
  auto slot_addr = [&](int s) { return ring + (grp * NS + s) * C::SLOT; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < KS * NS; ++i) {
      mbar_init(bars + i * 8, 1);
      mbar_init(bars + (KS * NS + i) * 8, QT);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // This group's blocks: blk0 + grp + KS * i for i in [0, nb).
  const int span = blk_end - blk0;
  const int nb = span > grp ? (span - grp + KS - 1) / KS : 0;
  const int64_t tab_row = (int64_t)b * a.max_blocks;

  // Leader warp: lane l caches the physical id of group block tab_base + l.
  int tab_base = -1;
  int32_t tab = 0;
  auto phys_of = [&](int i) -> int {
    if (tab_base < 0 || i - tab_base >= 32) {
      tab_base = i;
      const int blk = blk0 + grp + KS * (i + lane);
      const int32_t v = (i + lane < nb) ? a.table[tab_row + blk] : 0;
      tab = v < 0 ? 0 : (v >= a.num_blocks ? (int32_t)(a.num_blocks - 1) : v);
      if (tab != v) atomicOr(&g_attn_error, kErrBadInput);  // clamped: reads stay inside the pool
    }
    return __shfl_sync(0xffffffffu, tab, i - tab_base);
  };
  auto issue = [&](int i) {  // the whole leader warp calls; lane 0 issues
    const int phys = phys_of(i);
    if (lane == 0) {
      const int s = i % NS;
      const uint32_t dst = slot_addr(s), fb = full_bar(s);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(fb, C::SLOT);
      if constexpr (F8) {
        tma_load_4d(dst, &tmk, fb, 0, 0, g, phys);
        tma_load_4d(dst + 2048, &tmv, fb, 0, 0, g, phys);
      } else {
        tma_load_4d(dst, &tmk, fb, 0, 0, g, phys);
        tma_load_4d(dst + 2048, &tmk, fb, 64, 0, g, phys);
        tma_load_4d(dst + 4096, &tmv, fb, 0, 0, g, phys);
        tma_load_4d(dst + 6144, &tmv, fb, 64, 0, g, phys);
      }
    }
  };
  if (leader)
    for (int i = 0; i < min(NS, nb); ++i) issue(i);

  // Q fragments for this warp's 16 query rows. The head dimension is permuted:
  // in pass dh (0, 1) lane t owns 16 consecutive d starting at 64dh + 16t
  // (bf16: 16-byte units 2t, 2t+1 of the 64-wide half dh) or 32t + 16dh (FP8:
  // unit 2t + dh of the 128-code row); MMA i of the pass reads 4i .. 4i+3 of
  // them. K is read the same way.
  uint32_t qf[2][4][4];
  int pos_lo, pos_hi;  // last visible key index of rows gq and gq+8 (-1: none)
  {
    const int rl = row_base + gq, rh = rl + 8;
    const bool okl = rl < a.QR, okh = rh < a.QR;
    const int64_t ql = okl ? (((int64_t)b * a.W + rl / a.G) * a.Hq + g * a.G + rl % a.G) * kD : 0;
    const int64_t qh = okh ? (((int64_t)b * a.W + rh / a.G) * a.Hq + g * a.G + rh % a.G) * kD : 0;
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int dh = 0; dh < 2; ++dh)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int d = (F8 ? 32 * t + 16 * dh : 64 * dh + 16 * t) + 8 * u;
        uint4 vl = okl ? *reinterpret_cast<const uint4*>(a.q + ql + d) : z;
        uint4 vh = okh ? *reinterpret_cast<const uint4*>(a.q + qh + d) : z;
        if constexpr (F8) {  // the FP8 path multiplies in f16
          vl = make_uint4(bf16x2_to_f16x2(vl.x), bf16x2_to_f16x2(vl.y), bf16x2_to_f16x2(vl.z), bf16x2_to_f16x2(vl.w));
          vh = make_uint4(bf16x2_to_f16x2(vh.x), bf16x2_to_f16x2(vh.y), bf16x2_to_f16x2(vh.z), bf16x2_to_f16x2(vh.w));
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = 2 * u + e;
          qf[dh][i][0] = word(vl, 2 * e);
          qf[dh][i][1] = word(vh, 2 * e);
          qf[dh][i][2] = word(vl, 2 * e + 1);
          qf[dh][i][3] = word(vh, 2 * e + 1);
        }
      }
    pos_lo = okl ? ctx - a.W + rl / a.G : -1;
    pos_hi = okh ? ctx - a.W + rh / a.G : -1;
  }

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = kNegInf, m_hi = kNegInf, l_lo = 0.f, l_hi = 0.f;
  bool ok = true;

  for (int i = 0; i < nb; ++i) {
    const int s = i % NS;
    if (!mbar_wait(full_bar(s), (i / NS) & 1)) {
      if (lane == 0) atomicOr(&g_attn_error, kErrWaitTimeout);
      ok = false;
      break;
    }
    const uint32_t kb = slot_addr(s), vb = kb + (F8 ? 2048 : 4096);
    const int key0 = (blk0 + grp + KS * i) * kBlk;
    const int ntok = min(kBlk, ctx - key0);

    // ---- S = Q K^T for 16 keys: two n8 halves, two accumulators each ----
    float sc[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      const int r = 8 * h + gq;
#pragma unroll
      for (int dh = 0; dh < 2; ++dh) {
        float(&acc)[4] = dh ? sb : sa;
        if constexpr (F8) {
          // lanes t = 0..3 of rows gq, gq+1 hit units 2t+dh and (2t+dh)^1:
          // eight distinct 16-byte bank groups per quarter warp
          const uint4 c = lds128(kv_unit(kb, r, 2 * t + dh));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t b0, b1;
            e4m3x4_to_f16x2(word(c, i), b0, b1);
            mma_f16(acc, qf[dh][i][0], qf[dh][i][1], qf[dh][i][2], qf[dh][i][3], b0, b1);
          }
        } else {
          const uint4 k0 = lds128(kv_unit(kb + 2048 * dh, r, 2 * t));
          const uint4 k1 = lds128(kv_unit(kb + 2048 * dh, r, 2 * t + 1));
          mma_bf16(acc, qf[dh][0][0], qf[dh][0][1], qf[dh][0][2], qf[dh][0][3], k0.x, k0.y);
          mma_bf16(acc, qf[dh][1][0], qf[dh][1][1], qf[dh][1][2], qf[dh][1][3], k0.z, k0.w);
          mma_bf16(acc, qf[dh][2][0], qf[dh][2][1], qf[dh][2][2], qf[dh][2][3], k1.x, k1.y);
          mma_bf16(acc, qf[dh][3][0], qf[dh][3][1], qf[dh][3][2], qf[dh][3][3], k1.z, k1.w);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) sc[h][q] = sa[q] + sb[q];
    }
    // ---- mask, scale, online softmax ----
    float mx_lo = kNegInf, mx_hi = kNegInf;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int key = key0 + 8 * h + 2 * t + (q & 1);
        const int pos = (q & 2) ? pos_hi : pos_lo;
        const float v = key <= pos ? sc[h][q] * a.scale_log2 : kNegInf;
        sc[h][q] = v;
        if (q & 2) mx_hi = fmaxf(mx_hi, v); else mx_lo = fmaxf(mx_lo, v);
      }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
    }
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float base_lo = mn_lo == kNegInf ? 0.f : mn_lo;
    const float base_hi = mn_hi == kNegInf ? 0.f : mn_hi;
    const float al_lo = ex2(m_lo - base_lo), al_hi = ex2(m_hi - base_hi);  // exp2(-inf) = 0
    m_lo = mn_lo;
    m_hi = mn_hi;
    float p[2][4];
    float rs_lo = 0.f, rs_hi = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      p[h][0] = ex2(sc[h][0] - base_lo);
      p[h][1] = ex2(sc[h][1] - base_lo);
      p[h][2] = ex2(sc[h][2] - base_hi);
      p[h][3] = ex2(sc[h][3] - base_hi);
      rs_lo += p[h][0] + p[h][1];
      rs_hi += p[h][2] + p[h][3];
    }
    l_lo = l_lo * al_lo + rs_lo;
    l_hi = l_hi * al_hi + rs_hi;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= al_lo;
      o[j][1] *= al_lo;
      o[j][2] *= al_hi;
      o[j][3] *= al_hi;
    }
    uint32_t pa0, pa1, pa2, pa3;
    if constexpr (F8) {
      pa0 = pack_f16x2(p[0][0], p[0][1]);
      pa1 = pack_f16x2(p[0][2], p[0][3]);
      pa2 = pack_f16x2(p[1][0], p[1][1]);
      pa3 = pack_f16x2(p[1][2], p[1][3]);
    } else {
      pa0 = pack_bf16x2(p[0][0], p[0][1]);
      pa1 = pack_bf16x2(p[0][2], p[0][3]);
      pa2 = pack_bf16x2(p[1][0], p[1][1]);
      pa3 = pack_bf16x2(p[1][2], p[1][3]);
    }

    // ---- O += P V ----
    const int k0 = 2 * t, k1 = 2 * t + 1, k2 = 2 * t + 8, k3 = 2 * t + 9;
    if constexpr (F8) {
      // n8 tile jt, column s <-> d = 16s + jt: the lane loads unit gq (d =
      // 16gq .. +15) of its four keys and pairs code jt of key 2t with code jt
      // of key 2t+1 (and 2t+8 with 2t+9) while widening them.
      uint4 va = lds128(kv_unit(vb, k0, gq));
      uint4 vv = lds128(kv_unit(vb, k1, gq));
      uint4 vc = lds128(kv_unit(vb, k2, gq));
      uint4 vd = lds128(kv_unit(vb, k3, gq));
      if (ntok < kBlk) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        if (k0 >= ntok) va = z;
        if (k1 >= ntok) vv = z;
        if (k2 >= ntok) vc = z;
        if (k3 >= ntok) vd = z;
      }
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        // interleave codes 4w.. of keys 2t and 2t+1 (and 2t+8, 2t+9):
        // [a0 b0 a1 b1] and [a2 b2 a3 b3], then widen pairs to f16x2
        uint32_t x[4], y[4];
        e4m3x4_to_f16x2(prmt(word(va, w), word(vv, w), 0x5140u), x[0], x[1]);
        e4m3x4_to_f16x2(prmt(word(va, w), word(vv, w), 0x7362u), x[2], x[3]);
        e4m3x4_to_f16x2(prmt(word(vc, w), word(vd, w), 0x5140u), y[0], y[1]);
        e4m3x4_to_f16x2(prmt(word(vc, w), word(vd, w), 0x7362u), y[2], y[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_f16(o[4 * w + j], pa0, pa1, pa2, pa3, x[j], y[j]);
      }
    } else {
    // n8 tile (h, jj), column s <-> d = 64h + 8s + jj
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t hb = vb + 2048 * h;
      uint4 va = lds128(kv_unit(hb, k0, gq));
      uint4 vv = lds128(kv_unit(hb, k1, gq));
      uint4 vc = lds128(kv_unit(hb, k2, gq));
      uint4 vd = lds128(kv_unit(hb, k3, gq));
      if (ntok < kBlk) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        if (k0 >= ntok) va = z;
        if (k1 >= ntok) vv = z;
        if (k2 >= ntok) vc = z;
        if (k3 >= ntok) vd = z;
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const uint32_t sel = (jj & 1) ? 0x7632u : 0x5410u;
        const uint32_t b0 = prmt(word(va, jj >> 1), word(vv, jj >> 1), sel);
        const uint32_t b1 = prmt(word(vc, jj >> 1), word(vd, jj >> 1), sel);
        mma_bf16(o[8 * h + jj], pa0, pa1, pa2, pa3, b0, b1);
      }
    }
    }

    // ---- release the slot and refill it ----
    __syncwarp();
    if constexpr (QT > 1) {
      if (lane == 0) mbar_arrive(empty_bar(s));
    }
    if (leader && i + NS < nb) {
      if constexpr (QT > 1) {
        if (!mbar_wait(empty_bar(s), (i / NS) & 1)) {
          if (lane == 0) atomicOr(&g_attn_error, kErrWaitTimeout);
          ok = false;
          break;
        }
      }
      issue(i + NS);
    }
  }
  if (!ok) {
    // Drain the copies this group may still have in flight (bounded) before
    // the shared memory is reused or released.
    if (leader)
      for (int i = 0; i < min(NS, nb); ++i) (void)mbar_wait(full_bar(i), 0);
  }

  // ---- merge the KS warps of each query tile through shared memory ----
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  __syncthreads();  // every warp is done with the ring
  float* mo = reinterpret_cast<float*>(smem_raw + (ring - raw));  // [warp][16 rows][130]
  {
    float* wbase = mo + warp * 16 * (kD + 2);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      // columns 2t, 2t+1 of tile j
      const int d0 = F8 ? 32 * t + j : 64 * (j >> 3) + 16 * t + (j & 7);
      const int d1 = d0 + (F8 ? 16 : 8);
      wbase[gq * (kD + 2) + d0] = o[j][0];
      wbase[gq * (kD + 2) + d1] = o[j][1];
      wbase[(gq + 8) * (kD + 2) + d0] = o[j][2];
      wbase[(gq + 8) * (kD + 2) + d1] = o[j][3];
    }
    if (t == 0) {
      wbase[gq * (kD + 2) + kD] = m_lo;
      wbase[gq * (kD + 2) + kD + 1] = l_lo;
      wbase[(gq + 8) * (kD + 2) + kD] = m_hi;
      wbase[(gq + 8) * (kD + 2) + kD + 1] = l_hi;
    }
  }
  __syncthreads();
  // thread -> (query tile, row, 128/ (kThreads/(QT*16)) columns)
  constexpr int TPR = kThreads / (QT * 16);  // threads per row
  constexpr int CPT = kD / TPR;              // columns per thread
  const int row_id = threadIdx.x / TPR;      // 0 .. QT*16-1
  const int col0 = (threadIdx.x % TPR) * CPT;
  const int mqt = row_id / 16, mrow = row_id % 16;
  const int r = (qg * QT + mqt) * 16 + mrow;
  if (r >= a.QR) return;
  float mstar = kNegInf;
#pragma unroll
  for (int j = 0; j < KS; ++j) {
    const float* wb = mo + (j * QT + mqt) * 16 * (kD + 2) + mrow * (kD + 2);
    mstar = fmaxf(mstar, wb[kD]);
  }
  const float mbase = mstar == kNegInf ? 0.f : mstar;
  float wgt[KS];
  float L = 0.f;
#pragma unroll
  for (int j = 0; j < KS; ++j) {
    const float* wb = mo + (j * QT + mqt) * 16 * (kD + 2) + mrow * (kD + 2);
    wgt[j] = ex2(wb[kD] - mbase);
    L += wgt[j] * wb[kD + 1];
  }
  const int64_t orow = ((int64_t)b * a.W + r / a.G) * a.Hq + g * a.G + r % a.G;
  if (a.nchunks == 1) {
    const float inv = (L > 0.f ? 1.f / L : 0.f) * a.v_scale;
    for (int c = 0; c < CPT; c += 2) {
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        const float* wb = mo + (j * QT + mqt) * 16 * (kD + 2) + mrow * (kD + 2);
        v0 += wgt[j] * wb[col0 + c];
        v1 += wgt[j] * wb[col0 + c + 1];
      }
      *reinterpret_cast<uint32_t*>(a.out + orow * kD + col0 + c) = pack_bf16x2(v0 * inv, v1 * inv);
    }
  } else {
    float* po = a.part_o + (orow * a.nchunks + chunk) * kD;
    for (int c = 0; c < CPT; ++c) {
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        const float* wb = mo + (j * QT + mqt) * 16 * (kD + 2) + mrow * (kD + 2);
        v += wgt[j] * wb[col0 + c];
      }
      po[col0 + c] = v * a.v_scale;
    }
    if (threadIdx.x % TPR == 0) {
      a.part_ml[(orow * a.nchunks + chunk) * 2] = mstar;
      a.part_ml[(orow * a.nchunks + chunk) * 2 + 1] = L;
    }
  }
}

// One warp per output row: combine the chunk partials of that row. Lane c
// reads (m, l) of chunk c (32 chunks per pass); the o partials are then summed
// in chunk order with their loads issued ahead of the adds.
__global__ void __launch_bounds__(128) attn_merge_kernel(const Args a) {
  grid_dependency_wait();  // the partials come from the split kernel
  allow_dependent_launch();
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)a.B * a.W * a.Hq;
  if (row >= rows) return;
  const int b = (int)(row / ((int64_t)a.W * a.Hq));
  const int ctx = seq_ctx(a, b);
  const int nblk = (ctx + kBlk - 1) / kBlk;
  const int nch = min(a.nchunks, (nblk + a.chunk_blocks - 1) / a.chunk_blocks);
  const float* ml = a.part_ml + row * a.nchunks * 2;
  const float* po = a.part_o + row * a.nchunks * kD + lane * 4;
  float mstar = kNegInf;
  for (int c = lane; c < nch; c += 32) mstar = fmaxf(mstar, ml[2 * c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
  const float mbase = mstar == kNegInf ? 0.f : mstar;
  float lpart = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int c = c0 + lane;
    float wl = 0.f;
    if (c < nch) {
      wl = ex2(ml[2 * c] - mbase);
      lpart += wl * ml[2 * c + 1];
    }
    const int cnt = min(32, nch - c0);
    int j = 0;
    for (; j + 4 <= cnt; j += 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcg(reinterpret_cast<const float4*>(po + (int64_t)(c0 + j + u) * kD));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float w = __shfl_sync(0xffffffffu, wl, j + u);
        acc.x += w * v[u].x;
        acc.y += w * v[u].y;
        acc.z += w * v[u].z;
        acc.w += w * v[u].w;
      }
    }
    for (; j < cnt; ++j) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(po + (int64_t)(c0 + j) * kD));
      const float w = __shfl_sync(0xffffffffu, wl, j);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, off);
  const float inv = lpart > 0.f ? 1.f / lpart : 0.f;
  uint2 o;
  o.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  o.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(a.out + row * kD + lane * 4) = o;
}

// The merge for many chunks per row (8 or more): one CTA per output row, its
// four warps taking every fourth chunk with eight partial loads in flight per
// lane, then warp 0 adds the four warps' sums in warp order (the result does
// not depend on timing). A warp per row, as above, is bound by the latency of
// its chunk loads at small batch, where few rows have to fill the GPU.
__global__ void __launch_bounds__(128) attn_merge_wide_kernel(const Args a) {
  grid_dependency_wait();  // the partials come from the split kernel
  allow_dependent_launch();
  __shared__ float4 s_acc[4][32];
  __shared__ float s_l[4];
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = (int)(row / ((int64_t)a.W * a.Hq));
  const int ctx = seq_ctx(a, b);
  const int nblk = (ctx + kBlk - 1) / kBlk;
  const int nch = min(a.nchunks, (nblk + a.chunk_blocks - 1) / a.chunk_blocks);
  const float* ml = a.part_ml + row * a.nchunks * 2;
  const float* po = a.part_o + row * a.nchunks * kD + lane * 4;
  float mstar = kNegInf;
  for (int c = lane; c < nch; c += 32) mstar = fmaxf(mstar, ml[2 * c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
  const float mbase = mstar == kNegInf ? 0.f : mstar;
  float lpart = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = warp; c0 < nch; c0 += 32) {  // chunks c0 + 4 u, u < 8
    const int cj = c0 + 4 * lane;
    float wl = 0.f;
    if (lane < 8 && cj < nch) {
      wl = ex2(ml[2 * cj] - mbase);
      lpart += wl * ml[2 * cj + 1];
    }
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = c0 + 4 * u;
      v[u] = c < nch ? __ldcg(reinterpret_cast<const float4*>(po + (int64_t)c * kD)) : zero;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float w = __shfl_sync(0xffffffffu, wl, u);
      acc.x += w * v[u].x;
      acc.y += w * v[u].y;
      acc.z += w * v[u].z;
      acc.w += w * v[u].w;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, off);
  s_acc[warp][lane] = acc;
  if (lane == 0) s_l[warp] = lpart;
  __syncthreads();
  if (warp != 0) return;
  float4 t = s_acc[0][lane];
#pragma unroll
  for (int w = 1; w < 4; ++w) {
    const float4 u = s_acc[w][lane];
    t.x += u.x;
    t.y += u.y;
    t.z += u.z;
    t.w += u.w;
  }
  const float l = ((s_l[0] + s_l[1]) + s_l[2]) + s_l[3];
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint2 o;
  o.x = pack_bf16x2(t.x * inv, t.y * inv);
  o.y = pack_bf16x2(t.z * inv, t.w * inv);
  *reinterpret_cast<uint2*>(a.out + row * kD + lane * 4) = o;
}

// ---------------------------------------------------------------------------
// Tensor-core (tcgen05) form for wide query tiles: 17..128 query rows per kv
// head (verify widths), bf16 cache. One CTA per (sequence, kv head, chunk);
// the context chunk is walked in tiles of 128 tokens (eight 16-token blocks):
//  * warp 0: gathers each tile's K and V blocks through the block table by
//    TMA into one of three stages: K and V as two 64-dim halves of 128 token
//    rows each (16 KB per half, 128-byte swizzled, block i at rows
//    16 i .. 16 i + 15);
//  * warp 1, lane 0: S = Q K^T (M 128 query rows, N 128 tokens, K 128 dims;
//    Q K-major, K K-major) into the S buffer of the tile's parity in tensor
//    memory, then O += P V for the previous tile (M 128, N 128 dims, K 128
//    tokens; P read from tensor memory, where it overwrote that tile's S; V
//    MN-major: token rows with the dims contiguous, as the cache stores them)
//    into the O accumulator of that parity;
//  * warps 2-9: two softmax groups of four warps, for the even and the odd
//    tiles, each with its own S buffer, O accumulator and running (m, l); one
//    query row per thread (the tensor-memory lane the warp may reach): the
//    online softmax in the log2 domain on its S row (masked keys -> -inf by
//    select: past the context, past the causal limit of the row's verify
//    position, or in an absent block), O rescaled in tensor memory when the
//    row's reference maximum moves, P written as bf16 for the next MMA; V rows
//    past the context are zeroed first so stale pool contents cannot leak.
//    At the end the even group combines the two (m, l, O), as the merge of two
//    chunks would.
// The result is the normalised bf16 output (one chunk) or the same fp32
// partial (o, m, l) as the mma.sync form, merged by the same kernels.
namespace tca {
constexpr int kTileBlk = 8;                 // 16-token blocks per tile
constexpr int kTileTok = kTileBlk * kBlk;   // 128
constexpr int kHalf = 128 * 128;            // one 64-dim half: 128 rows x 128 B
constexpr int kQ = 0;                       // Q: two halves
constexpr int kStage0 = 2 * kHalf;          // stages: K halves then V halves
constexpr int kStageBytes = 4 * kHalf;
constexpr int kStages = 3;
constexpr int kBody = kStage0 + kStages * kStageBytes;  // 224 KB
constexpr int kSmem = kBody;  // the dynamic region starts 1024-byte aligned (checked at run time)
constexpr int kThreads = 320;
constexpr int kSoft0 = 2;                   // first softmax warp
// tensor-memory columns: S (then P) and O for the even and the odd tiles
__host__ __device__ constexpr uint32_t s_col(int parity) { return parity ? 128u : 0u; }
__host__ __device__ constexpr uint32_t o_col(int parity) { return parity ? 384u : 256u; }
}  // namespace tca

// o0 w0 + o1 w1 for the two softmax groups' accumulators, each product and
// the sum rounded on its own (no fused multiply-add), so that the result does
// not depend on which accumulator holds the even and which the odd tiles; an
// accumulator whose row saw no key (has = false) adds 0.
__device__ __forceinline__ float combine2(float o0, float w0, bool has0, float o1, float w1, bool has1) {
  return __fadd_rn(has0 ? __fmul_rn(o0, w0) : 0.f, has1 ? __fmul_rn(o1, w1) : 0.f);
}

// Work units of the tensor-core forms, in a longest-first order of the
// sequences when there are at most kLptMaxB of them and the order matters (the
// persistent form, whose CTAs take units in order; a balanced tail, whose
// pieces split the last items): the units of the longest contexts go first
// and the tail splits the shortest ones, so that no long unit starts last (a
// CTA that did would finish long after the others). Every kernel that maps
// units or tail rows to (sequence, kv head) then takes the same order, so the
// two forms split the same items. Ties go by index: the order is
// deterministic. Otherwise units follow the sequence index.
constexpr int kLptMaxB = 256;

// seq[p] = the sequence at position p of that order, for every p < B <=
// kLptMaxB. Every thread of the CTA takes part (the caller synchronises
// before reading): each lane loads its share of the context lengths once, and
// warp w ranks sequences w, w + warps, ... by a count over all of them. Not
// inlined: it runs once per CTA, and inlined its registers added spills to
// the tensor-core kernels' tile loops.
__device__ __noinline__ void lpt_order(const Args& a, uint8_t* seq) {
  constexpr int K = kLptMaxB / 32;
  if (!a.lpt) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int c[K];
#pragma unroll
  for (int k = 0; k < K; ++k) c[k] = lane + 32 * k < a.B ? seq_ctx(a, lane + 32 * k) : -1;
  for (int b = warp; b < a.B; b += nwarps) {
    int cb = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {  // warp-uniform: b is the same in every lane
      const int v = __shfl_sync(0xffffffffu, c[k], b & 31);
      if ((b >> 5) == k) cb = v;
    }
    int n = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = lane + 32 * k;
      n += (i < a.B && (c[k] > cb || (c[k] == cb && i < b))) ? 1 : 0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
    if (lane == 0) seq[n] = (uint8_t)b;
  }
}

struct TcUnit {
  int item;  // position of the (sequence, kv head) item in the order
  int b, g, chunk, piece, ctx, blk0, blk_end, ntiles;
};

// The item of unit u of the tensor-core forms: item u / nchunks (chunk u mod
// nchunks) or, with a balanced tail, the whole items first and then the
// pieces of the last tail_items items. Item i is kv head i mod Hkv of the
// sequence at position i / Hkv of the order.
__device__ __forceinline__ int tc_unit_item(const Args& a, int u) {
  if (a.tail_pieces > 0) {
    const int nwhole = a.B * a.Hkv - a.tail_items;
    return u < nwhole ? u : nwhole + (u - nwhole) / a.tail_pieces;
  }
  return u / a.nchunks;
}

// The sequence at position pos of the order: seq from lpt_order, or pos
// itself (seq null).
__device__ __forceinline__ int tc_seq_at(const uint8_t* seq, int pos) { return seq ? (int)seq[pos] : pos; }

// Unit u, whose item belongs to sequence b (tc_seq_at of the item's position).
__device__ __forceinline__ TcUnit tc_unit(const Args& a, int u, int b) {
  TcUnit t;
  t.piece = -1;
  t.chunk = 0;
  t.item = tc_unit_item(a, u);
  if (a.tail_pieces > 0) {
    const int nwhole = a.B * a.Hkv - a.tail_items;
    t.piece = u < nwhole ? -1 : (u - nwhole) % a.tail_pieces;
  } else {
    t.chunk = u % a.nchunks;
  }
  t.b = b;
  t.g = t.item % a.Hkv;
  t.ctx = seq_ctx(a, t.b);
  const int nblk_seq = (t.ctx + kBlk - 1) / kBlk;
  t.blk0 = t.chunk * a.chunk_blocks;
  t.blk_end = min(t.blk0 + a.chunk_blocks, nblk_seq);
  if (t.piece >= 0) {  // piece k of p: tiles [k T / p, (k + 1) T / p) of the item's T tiles
    const int T = (nblk_seq + tca::kTileBlk - 1) / tca::kTileBlk;
    t.blk0 = (t.piece * T / a.tail_pieces) * tca::kTileBlk;
    t.blk_end = min(((t.piece + 1) * T / a.tail_pieces) * tca::kTileBlk, nblk_seq);
  }
  t.ntiles = t.blk0 < t.blk_end ? (t.blk_end - t.blk0 + tca::kTileBlk - 1) / tca::kTileBlk : 0;
  return t;
}

// One 128-token tile of the online softmax for one query row (a thread) of
// the tensor-core forms, in the log2 domain: sv holds the row's raw q.k
// products (scaled in place), columns 0 .. vl are visible (the others become
// -inf by select), c is the softmax scale times log2(e). The row's reference
// maximum m moves only when the tile's maximum exceeds it by more than 8, so
// P stays below 2^8 and O is rescaled on few tiles. Updates (m, l), writes P
// as bf16 pairs over the first 64 columns of the S row at tS and returns
// alpha, the factor that the row's O must take. (Keeping the raw products and
// taking c s - m in one fused multiply-add saves two instructions an element
// but needs more registers; the spills made the attention 20% slower.)
__device__ __forceinline__ float tc_softmax_tile(float (&sv)[tca::kTileTok], int vl, float c, float& m, float& l,
                                                 uint32_t tS) {
  constexpr int T = tca::kTileTok;
  float mx[8];  // eight independent partial maxima (short dependency chains)
#pragma unroll
  for (int q = 0; q < 8; ++q) mx[q] = kNegInf;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    sv[t] = t <= vl ? sv[t] * c : kNegInf;
    mx[t & 7] = fmaxf(mx[t & 7], sv[t]);
  }
  const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
  const float mn = (mt > m + 8.f || m == kNegInf) ? fmaxf(m, mt) : m;
  const float mb = mn == kNegInf ? 0.f : mn;  // a row with no visible key so far keeps p = 0
  const float alpha = mn == m ? 1.f : ex2(m - mb);  // m = -inf: 0
  float pa[8];  // eight partial sums
#pragma unroll
  for (int q = 0; q < 8; ++q) pa[q] = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // P over its S, one 64-token half at a time
    uint32_t pw[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const float p0 = ex2(sv[64 * h + 2 * q] - mb), p1 = ex2(sv[64 * h + 2 * q + 1] - mb);
      pa[q & 7] += p0 + p1;
      pw[q] = pack_bf16x2(p0, p1);
    }
    tmem_st32(tS + 32 * h, pw);
  }
  const float ps = ((pa[0] + pa[1]) + (pa[2] + pa[3])) + ((pa[4] + pa[5]) + (pa[6] + pa[7]));
  l = l * alpha + ps;
  m = mn;
  return alpha;
}

__device__ __forceinline__ void sts128z(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
}
__device__ __forceinline__ void softmax_barrier() {  // the eight softmax warps
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// Ten warps: three share some SM sub-partitions, whose 16K registers then
// allow about 168 per thread.
__global__ void __launch_bounds__(tca::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const Args a) {
  using namespace tca;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // kv_full[kStages], kv_empty[kStages], s_full[2], p_full[2], pv_done[2]
  __shared__ __align__(8) uint64_t bars[2 * kStages + 6];
  __shared__ uint32_t tmem_base_sh;
  __shared__ float xm[2][128];  // the odd group's final (m, l) per row
  __shared__ uint8_t lpt_seq[kLptMaxB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();  // q, the tables and the cache may come from the previous kernel
  allow_dependent_launch();
  if (smem_addr(smem_raw) & 1023u) {  // the layout needs a 1024-byte aligned region
    if (threadIdx.x == 0) atomicOr(&g_attn_error, kErrBadInput);
    return;
  }
  // Work unit: a chunk of one (sequence position, kv head) on a 3-D grid, or,
  // with a balanced tail, a 1-D list: the whole items first, then the pieces
  // of the last tail_items items (piece >= 0), in the longest-first order of
  // the persistent form (so that both forms split the same items)
  int chunk = blockIdx.x, g = blockIdx.y, b = blockIdx.z, piece = -1, item = 0;
  if (a.tail_pieces > 0) {
    const int nwhole = a.B * a.Hkv - a.tail_items;
    const int u = blockIdx.x;
    item = u < nwhole ? u : nwhole + (u - nwhole) / a.tail_pieces;
    piece = u < nwhole ? -1 : (u - nwhole) % a.tail_pieces;
    chunk = 0;
    b = item / a.Hkv;
    g = item % a.Hkv;
    if (a.lpt) {  // uniform across the grid
      lpt_order(a, lpt_seq);
      __syncthreads();
      b = lpt_seq[b];
      if (blockIdx.x == 0)  // for the tail merge
        for (int p = threadIdx.x; p < a.B; p += blockDim.x) a.tail_seq[p] = lpt_seq[p];
    }
  }
  const int ctx = seq_ctx(a, b);
  if (chunk == 0 && g == 0 && piece <= 0 && threadIdx.x == 0) {
    const int raw = a.ctx[b];
    if (raw < a.W || raw != ctx) atomicOr(&g_attn_error, kErrBadInput);
  }
  const int nblk_seq = (ctx + kBlk - 1) / kBlk;
  int blk0 = chunk * a.chunk_blocks, blk_end = min(blk0 + a.chunk_blocks, nblk_seq);
  if (piece >= 0) {  // piece k of p: tiles [k T / p, (k + 1) T / p) of the item's T tiles
    const int T = (nblk_seq + kTileBlk - 1) / kTileBlk;
    blk0 = (piece * T / a.tail_pieces) * kTileBlk;
    blk_end = min(((piece + 1) * T / a.tail_pieces) * kTileBlk, nblk_seq);
  }
  const int tail_row0 = (item - (a.B * a.Hkv - a.tail_items)) * a.QR;  // pieces: first tail row of the item
  if (blk0 >= blk_end) {  // whole CTA: nothing of this sequence here
    if (piece >= 0) {  // an empty piece: (m, l, o) = (-inf, 0, 0)
      for (int i = threadIdx.x; i < a.QR * kD; i += tca::kThreads) {
        const int64_t pr = (int64_t)(tail_row0 + i / kD) * a.tail_pieces + piece;
        a.tail_o[pr * kD + i % kD] = 0.f;
        if (i % kD == 0) {
          a.tail_ml[pr * 2] = kNegInf;
          a.tail_ml[pr * 2 + 1] = 0.f;
        }
      }
    } else if (a.nchunks == 1 && nblk_seq == 0) {
      for (int i = threadIdx.x; i < a.QR * kD / 2; i += tca::kThreads) {
        const int r = i / (kD / 2);
        const int64_t orow = ((int64_t)b * a.W + r / a.G) * a.Hq + g * a.G + r % a.G;
        reinterpret_cast<uint32_t*>(a.out + orow * kD)[i % (kD / 2)] = 0u;
      }
    }
    return;
  }
  const int ntiles = (blk_end - blk0 + kTileBlk - 1) / kTileBlk;
  const uint32_t base = smem_addr(smem_raw);
  const uint32_t kv_full = smem_addr(&bars[0]), kv_empty = kv_full + 8 * kStages, s_full = kv_full + 16 * kStages,
                 p_full = s_full + 16, pv_done = s_full + 32;
  auto stage = [&](int st) { return base + kStage0 + st * kStageBytes; };
  bool ok = true;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(kv_full + 8 * i, 1);
      mbar_init(kv_empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(p_full + 8 * i, 4);  // the four warps of a softmax group
      mbar_init(pv_done + 8 * i, 1);
    }
    fence_mbar_init();
  }
  // Q: the QR rows of this kv head (row r: position r / G, head g G + r % G),
  // zero rows up to 128, K-major and 128-byte swizzled in two 64-dim halves;
  // thread (r, hh) of the softmax warps copies half hh of row r.
  if (warp >= kSoft0) {
    const int tq = threadIdx.x - kSoft0 * 32;
    const int r = tq & 127, hh = tq >> 7;
    const bool live = r < a.QR;
    const uint4* src = live ? reinterpret_cast<const uint4*>(
                                  a.q + (((int64_t)b * a.W + r / a.G) * a.Hq + g * a.G + r % a.G) * kD) + 8 * hh
                            : nullptr;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t dst = base + kQ + hh * kHalf + r * 128 + ((((uint32_t)c) ^ (uint32_t)(r & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(smem_addr(&tmem_base_sh), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  int issued = 0;  // tiles whose copies the gather warp issued
  if (warp == 0) {
    // ---------------- K/V gather ----------------
    // Lane i (< 8) issues the four copies of the tile's block i, so that a
    // tile's 32 copies go out eight at a time; lane l reads the block-table
    // entry of block 32 q + l of the chunk for groups of four tiles.
    const int64_t tab_row = (int64_t)b * a.max_blocks;
    const int nblk = blk_end - blk0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmk) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmv) : "memory");
    int tab = 0;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int st = j % kStages;
      if (j >= kStages && !__all_sync(0xffffffffu, mbar_wait(kv_empty + 8 * st, ((j - kStages) / kStages) & 1))) {
        ok = false;
        break;
      }
      if ((j & 3) == 0) {  // the table entries of tiles j .. j + 3
        const int bi = j * kTileBlk + lane;
        const int32_t v = bi < nblk ? a.table[tab_row + blk0 + bi] : 0;
        tab = v < 0 ? 0 : (v >= a.num_blocks ? (int)(a.num_blocks - 1) : v);
        if (tab != v) atomicOr(&g_attn_error, kErrBadInput);  // clamped: reads stay inside the pool
      }
      const int nb = min(kTileBlk, nblk - j * kTileBlk);
      const uint32_t fb = kv_full + 8 * st, dst = stage(st);
      if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)nb * 4u * 2048u);
      __syncwarp();
      const int phys = __shfl_sync(0xffffffffu, tab, (j & 3) * kTileBlk + (lane & 7));
      if (lane < nb) {
        const uint32_t d = dst + lane * 2048;
        tma_load_4d(d, &tmk, fb, 0, 0, g, phys);
        tma_load_4d(d + kHalf, &tmk, fb, 64, 0, g, phys);
        tma_load_4d(d + 2 * kHalf, &tmv, fb, 0, 0, g, phys);
        tma_load_4d(d + 3 * kHalf, &tmv, fb, 64, 0, g, phys);
      }
      issued = j + 1;
    }
    if (!ok && lane == 0) atomicOr(&g_attn_error, kErrWaitTimeout);
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    // The tensor pipe runs one thread's MMAs in order: S of tile j + 2
    // overwrites the buffer that P of tile j occupied only after P V of tile j
    // has read it.
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, kTileTok), id_pv = idesc_bf16_bmn(128, kD);
      auto issue_pv = [&](int j) {  // O[j & 1] += P V of tile j
        const int pg = j & 1;
        if (!mbar_wait(p_full + 8 * pg, (j >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t v0 = stage(j % kStages) + 2 * kHalf;
#pragma unroll
        for (int kk = 0; kk < kTileTok / 16; ++kk)  // 16 tokens = 8 columns of P
          umma_bf16_ta(tmem + o_col(pg), tmem + s_col(pg) + kk * 8, sw128_desc_mn(v0 + kk * 2048, kHalf, 1024), id_pv,
                       (j >= 2 || kk > 0) ? 1u : 0u);
        umma_commit(kv_empty + 8 * (j % kStages));  // the stage is free once these MMAs have read V
        umma_commit(pv_done + 8 * pg);
        return true;
      };
      for (int j = 0; j < ntiles && ok; ++j) {
        const int ks = j % kStages, sg = j & 1;
        if (!mbar_wait(kv_full + 8 * ks, (j / kStages) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k0 = stage(ks);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          umma_bf16(tmem + s_col(sg), sw128_desc(base + kQ + (kk >> 2) * kHalf + (kk & 3) * 32),
                    sw128_desc(k0 + (kk >> 2) * kHalf + (kk & 3) * 32), id_s, kk > 0 ? 1u : 0u);
        umma_commit(s_full + 8 * sg);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok && !issue_pv(ntiles - 1)) ok = false;
      if (!ok) atomicOr(&g_attn_error, kErrWaitTimeout);
    }
  } else {
    // ---------------- softmax: group grp takes tiles grp, grp + 2, ... ----------------
    const int grp = (warp - kSoft0) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row = tensor-memory lane
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = trow + s_col(grp), tO = trow + o_col(grp);
    const bool live = r < a.QR;
    // key j is visible to row r iff j < ctx and j <= ctx - W + r / G
    const int lim = live ? min(ctx - 1, ctx - a.W + r / a.G) : -1;
    float m = kNegInf, l = 0.f;
    int last = -1;  // this group's last tile
    for (int j = grp; j < ntiles; j += 2) {
      const int tok0 = (blk0 + j * kTileBlk) * kBlk;  // first token of the tile
      const int tok_end = min(blk_end * kBlk, ctx);   // tokens past this are absent or past the context
      if (!__all_sync(0xffffffffu, mbar_wait(s_full + 8 * grp, (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[kTileTok];
      {
        uint32_t u0[32], u1[32], u2[32], u3[32];  // four loads in flight, one wait
        tmem_ld32_nowait(tS, u0);
        tmem_ld32_nowait(tS + 32, u1);
        tmem_ld32_nowait(tS + 64, u2);
        tmem_ld32_nowait(tS + 96, u3);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          sv[t] = __uint_as_float(u0[t]);
          sv[32 + t] = __uint_as_float(u1[t]);
          sv[64 + t] = __uint_as_float(u2[t]);
          sv[96 + t] = __uint_as_float(u3[t]);
        }
      }
      const int vl = min(lim, tok_end - 1) - tok0;  // columns 0 .. vl are visible to this row
      const float alpha = tc_softmax_tile(sv, vl, a.scale_log2, m, l, tS);
      // V rows past the context (or of absent blocks) are zeroed before the
      // MMA reads them: 0 * NaN would otherwise leak stale pool contents
      if (tok0 + kTileTok > tok_end) {
        if (!__all_sync(0xffffffffu, mbar_wait(kv_full + 8 * (j % kStages), (j / kStages) & 1))) {
          ok = false;
          break;
        }
        const int t = r;  // this thread's token row of the tile
        if (tok0 + t >= tok_end) {
          const uint32_t v0 = stage(j % kStages) + 2 * kHalf + t * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            sts128z(v0 + c * 16);
            sts128z(v0 + kHalf + c * 16);
          }
        }
      }
      if (j >= 2) {
        // O holds this group's earlier tiles once the previous P V is
        // complete; it is rescaled only when some row of the warp moved its
        // reference maximum
        if (!__all_sync(0xffffffffu, mbar_wait(pv_done + 8 * grp, ((j - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t u[32];
            tmem_ld32(tO + c * 32, u);
#pragma unroll
            for (int t = 0; t < 32; ++t) u[t] = __float_as_uint(__uint_as_float(u[t]) * alpha);
            tmem_st32(tO + c * 32, u);
          }
        }
      }
      tmem_wait_st();  // P (and a rescaled O) in place
      fence_proxy_async_smem();  // zeroed V rows, if any
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + 8 * grp);
      last = j;
    }
    // ---------------- epilogue ----------------
    // each group waits for its last P V, the odd group hands over its (m, l),
    // and the even group combines both O accumulators row by row
    bool good = ok && (last < 0 || __all_sync(0xffffffffu, mbar_wait(pv_done + 8 * grp, (last >> 1) & 1)));
    if (!good && lane == 0) atomicOr(&g_attn_error, kErrWaitTimeout);
    if (grp == 1) {
      xm[0][r] = last < 0 ? kNegInf : m;
      xm[1][r] = last < 0 ? 0.f : l;
    }
    tc_fence_before();
    softmax_barrier();
    tc_fence_after();
    if (grp == 0) {
      const float m1 = xm[0][r], l1 = xm[1][r];
      const float ms = fmaxf(m, m1);
      const float mbs = ms == kNegInf ? 0.f : ms;
      const float w0 = ex2(m - mbs), w1 = ex2(m1 - mbs);  // -inf: 0
      const bool use1 = __any_sync(0xffffffffu, m1 != kNegInf);  // the odd accumulator holds data
      const float lt = __fadd_rn(__fmul_rn(l, w0), __fmul_rn(l1, w1));
      const int64_t orow = live ? ((int64_t)b * a.W + r / a.G) * a.Hq + g * a.G + r % a.G : 0;
      const float inv = (lt > 0.f ? 1.f / lt : 0.f) * a.v_scale;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32], u1[32];
        tmem_ld32(trow + o_col(0) + c * 32, u);  // warp-collective: every lane takes part
        if (use1) {
          tmem_ld32(trow + o_col(1) + c * 32, u1);
#pragma unroll
          for (int t = 0; t < 32; ++t)
            u[t] = __float_as_uint(
                combine2(__uint_as_float(u[t]), w0, m != kNegInf, __uint_as_float(u1[t]), w1, m1 != kNegInf));
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t)
            u[t] = __float_as_uint(combine2(__uint_as_float(u[t]), w0, m != kNegInf, 0.f, 0.f, false));
        }
        if (good && live) {
          if (piece >= 0) {
            float4* po = reinterpret_cast<float4*>(
                a.tail_o + ((int64_t)(tail_row0 + r) * a.tail_pieces + piece) * kD + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              po[q] = make_float4(__uint_as_float(u[4 * q]) * a.v_scale, __uint_as_float(u[4 * q + 1]) * a.v_scale,
                                  __uint_as_float(u[4 * q + 2]) * a.v_scale, __uint_as_float(u[4 * q + 3]) * a.v_scale);
          } else if (a.nchunks == 1) {
            uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kD + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * q]) * inv, __uint_as_float(u[8 * q + 1]) * inv),
                                  pack_bf16x2(__uint_as_float(u[8 * q + 2]) * inv, __uint_as_float(u[8 * q + 3]) * inv),
                                  pack_bf16x2(__uint_as_float(u[8 * q + 4]) * inv, __uint_as_float(u[8 * q + 5]) * inv),
                                  pack_bf16x2(__uint_as_float(u[8 * q + 6]) * inv, __uint_as_float(u[8 * q + 7]) * inv));
          } else {
            float4* po = reinterpret_cast<float4*>(a.part_o + (orow * a.nchunks + chunk) * kD + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              po[q] = make_float4(__uint_as_float(u[4 * q]) * a.v_scale, __uint_as_float(u[4 * q + 1]) * a.v_scale,
                                  __uint_as_float(u[4 * q + 2]) * a.v_scale, __uint_as_float(u[4 * q + 3]) * a.v_scale);
          }
        }
      }
      if (good && live && piece >= 0) {
        const int64_t pr = (int64_t)(tail_row0 + r) * a.tail_pieces + piece;
        a.tail_ml[pr * 2] = ms;
        a.tail_ml[pr * 2 + 1] = lt;
      } else if (good && live && a.nchunks > 1) {
        a.part_ml[(orow * a.nchunks + chunk) * 2] = ms;
        a.part_ml[(orow * a.nchunks + chunk) * 2 + 1] = lt;
      }
    }
  }
  if (threadIdx.x == 0) {
    // every issued copy has landed before the CTA exits (immediate unless a
    // wait gave up): the last tile issued into each stage, bounded
    for (int st = 0; st < kStages; ++st) {
      const int jl = issued - 1 - (((issued - 1 - st) % kStages + kStages) % kStages);
      if (jl >= 0) (void)mbar_wait(kv_full + 8 * st, (jl / kStages) & 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Persistent tensor-core form: the work units and the per-tile arithmetic of
// attn_tc_kernel, with one CTA per SM taking units from a queue (an atomic
// ticket in the workspace's counter region; the last CTA to find the queue
// empty resets it), so that the tiles of successive units flow through one
// pipeline instead of each CTA paying its own start-up and drain:
//  * warp 0 takes the next unit once it has issued the copies of the current
//    one (units in the longest-first order of their sequences), hands it and
//    its sequence to the other roles through a two-slot queue in shared
//    memory, loads its Q by TMA (into a second Q slot when the unit has at
//    most 64 query rows, so that it lands while the current Q is in use) and
//    gathers its K tiles; warp 10 gathers the V tiles of the same units;
//  * tiles are numbered across units: tile J uses K and V slot J mod 3, the S
//    buffer and softmax group of J's parity, whatever unit it belongs to;
//  * warp 1 issues S of a unit's first tile before P V of the previous unit's
//    last tile, and the first P V of a unit (which starts an O accumulator
//    afresh) only after the even group has read both accumulators of the
//    previous unit;
//  * the odd group hands its (m, l) to the even group through shared memory
//    (a full/empty barrier pair) and goes on to the next unit.
namespace tcp {
// With at most 64 query rows, Q slot 1 starts 64 rows (8 KB) into each of
// slot 0's halves: the rows past 64 that an M = 128 MMA reads from either slot
// are rows of the other slot or of K slot 0, and belong to masked query rows.
constexpr int kQSlot = 64 * 128;
// K and V have rings of their own (three 32 KB slots each: two 64-dim halves
// of 128 token rows), so that a K slot is free again once S has read it and
// only V waits for P V.
constexpr int kSlotBytes = 2 * tca::kHalf;
constexpr int kK0 = 2 * tca::kHalf;               // after Q
constexpr int kV0 = kK0 + tca::kStages * kSlotBytes;
static_assert(kV0 + tca::kStages * kSlotBytes == tca::kSmem, "the K and V rings fill the stages' space");
constexpr int kThreads = 352;  // gather K (warp 0), MMA (1), softmax (2-9), gather V (10)
constexpr int kVWarp = 10;
}  // namespace tcp

// Eleven warps: three share each of three SM sub-partitions, whose 16K
// registers then allow at most 168 per thread.
__global__ void __maxnreg__(168)
    attn_tcp_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ CUtensorMap tmq, const Args a) {
  using namespace tca;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // k_full[3], k_empty[3], v_full[3], v_empty[3], s_full[2], p_full[2],
  // pv_done[2], q_full[2], q_free[2], u_full[2], u_empty[2], o_free, xm_full,
  // xm_empty, fin
  __shared__ __align__(8) uint64_t bars[4 * kStages + 18];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int2 unit_sh[2];   // (unit, its sequence) handed from the queue to the other roles
  __shared__ float xm[2][128];  // the odd group's (m, l) per row for the unit being combined
  __shared__ uint8_t lpt_seq[kLptMaxB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();  // q, the tables, the cache and the queue's counters come from earlier kernels
  allow_dependent_launch();
  if (smem_addr(smem_raw) & 1023u) {  // the layout needs a 1024-byte aligned region
    if (threadIdx.x == 0) atomicOr(&g_attn_error, kErrBadInput);
    return;
  }
  const int items = a.B * a.Hkv;
  const int units = a.tail_pieces > 0 ? items - a.tail_items + a.tail_items * a.tail_pieces : items * a.nchunks;
  const int nq = a.QR <= 64 ? 2 : 1;  // Q slots
  const uint32_t base = smem_addr(smem_raw);
  const uint32_t k_full = smem_addr(&bars[0]), k_empty = k_full + 8 * kStages, v_full = k_full + 16 * kStages,
                 v_empty = k_full + 24 * kStages, s_full = k_full + 32 * kStages, p_full = s_full + 16,
                 pv_done = s_full + 32, q_full = s_full + 48, q_free = s_full + 64, u_full = s_full + 80,
                 u_empty = s_full + 96, o_free = s_full + 112, xm_full = s_full + 120, xm_empty = s_full + 128,
                 fin = s_full + 136;
  auto kslot = [&](int st) { return base + tcp::kK0 + st * tcp::kSlotBytes; };
  auto vslot = [&](int st) { return base + tcp::kV0 + st * tcp::kSlotBytes; };
  bool ok = true;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(k_full + 8 * i, 1);
      mbar_init(k_empty + 8 * i, 1);
      mbar_init(v_full + 8 * i, 1);
      mbar_init(v_empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(p_full + 8 * i, 4);  // the four warps of a softmax group
      mbar_init(pv_done + 8 * i, 1);
      mbar_init(q_full + 8 * i, 1);
      mbar_init(q_free + 8 * i, 1);
      mbar_init(u_full + 8 * i, 1);
      mbar_init(u_empty + 8 * i, 10);  // the MMA thread, the eight softmax warps and the V gather warp
    }
    mbar_init(o_free, 4);  // the even group's warps
    mbar_init(xm_full, 4);  // the odd group's warps
    mbar_init(xm_empty, 4);
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  lpt_order(a, lpt_seq);
  const uint8_t* useq = a.lpt ? lpt_seq : nullptr;
  if (warp == 1) tmem_alloc(smem_addr(&tmem_base_sh), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (blockIdx.x == 0 && a.lpt && a.tail_pieces > 0)  // for the tail merge
    for (int p = threadIdx.x; p < a.B; p += blockDim.x) a.tail_seq[p] = lpt_seq[p];

  if (warp == 0) {
    // ---------------- queue, Q and K gather ----------------
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmk) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmq) : "memory");
    int J = 0;   // tiles whose copies were issued
    int qi = 0;  // Q loads issued (one per unit with tiles)
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait(u_empty + 8 * slot, ((k >> 1) - 1) & 1))) {
        ok = false;
        break;
      }
      int u = 0;
      if (lane == 0) u = (int)atomicAdd(a.ctr, 1u);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u >= units) u = -1;
      const int ub = u < 0 ? 0 : tc_seq_at(useq, tc_unit_item(a, u) / a.Hkv);
      if (lane == 0) {
        unit_sh[slot] = make_int2(u, ub);
        mbar_arrive(u_full + 8 * slot);
      }
      if (u < 0) break;
      const TcUnit t = tc_unit(a, u, ub);
      if (lane == 0 && t.chunk == 0 && t.g == 0 && t.piece <= 0) {
        const int raw = a.ctx[t.b];
        if (raw < a.W || raw != t.ctx) atomicOr(&g_attn_error, kErrBadInput);
      }
      if (t.ntiles == 0) continue;
      // Q of the unit: the QR rows of its kv head (row r: position r / G,
      // head g G + r % G), two 64-dim halves, once the slot's previous unit has
      // issued its last S
      const int qs = qi % nq;
      if (qi >= nq && !__all_sync(0xffffffffu, mbar_wait(q_free + 8 * qs, ((qi / nq) - 1) & 1))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const uint32_t qb = q_full + 8 * qs, dst = base + kQ + qs * tcp::kQSlot;
        mbar_arrive_expect_tx(qb, (uint32_t)a.QR * 256u);
        tma_load_4d(dst, &tmq, qb, 0, t.g * a.G, 0, t.b);
        tma_load_4d(dst + kHalf, &tmq, qb, 64, t.g * a.G, 0, t.b);
      }
      ++qi;
      const int64_t tab_row = (int64_t)t.b * a.max_blocks;
      const int nblk = t.blk_end - t.blk0;
      int tab = 0;
      for (int j = 0; j < t.ntiles; ++j) {
        const int st = J % kStages;
        if (J >= kStages && !__all_sync(0xffffffffu, mbar_wait(k_empty + 8 * st, ((J - kStages) / kStages) & 1))) {
          ok = false;
          break;
        }
        if ((j & 3) == 0) {  // the table entries of tiles j .. j + 3
          const int bi = j * kTileBlk + lane;
          const int32_t v = bi < nblk ? a.table[tab_row + t.blk0 + bi] : 0;
          tab = v < 0 ? 0 : (v >= a.num_blocks ? (int)(a.num_blocks - 1) : v);
          if (tab != v) atomicOr(&g_attn_error, kErrBadInput);  // clamped: reads stay inside the pool
        }
        const int nb = min(kTileBlk, nblk - j * kTileBlk);
        const uint32_t fb = k_full + 8 * st;
        if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)nb * 2u * 2048u);
        __syncwarp();
        const int phys = __shfl_sync(0xffffffffu, tab, (j & 3) * kTileBlk + (lane & 7));
        if (lane < nb) {  // block i of the tile: K rows 16 i .. 16 i + 15 of both halves
          const uint32_t d = kslot(st) + lane * 2048;
          tma_load_4d(d, &tmk, fb, 0, 0, t.g, phys);
          tma_load_4d(d + kHalf, &tmk, fb, 64, 0, t.g, phys);
        }
        ++J;
      }
    }
    if (lane == 0) {
      if (!ok) atomicOr(&g_attn_error, kErrWaitTimeout);
      // Every CTA counts itself out once; the last one leaves both counters
      // at zero for the next call (every other CTA has taken its last ticket).
      __threadfence();
      if (atomicAdd(a.ctr + 1, 1u) == gridDim.x - 1) {
        atomicExch(a.ctr, 0u);
        atomicExch(a.ctr + 1, 0u);
      }
      // every issued copy has landed before the CTA exits (immediate unless a
      // wait gave up): the last K tile issued into each slot, the last Q load
      // into each Q slot, bounded
      for (int st = 0; st < kStages; ++st) {
        const int jl = J - 1 - (((J - 1 - st) % kStages + kStages) % kStages);
        if (jl >= 0) (void)mbar_wait(k_full + 8 * st, (jl / kStages) & 1);
      }
      for (int s = 0; s < nq; ++s) {
        const int il = qi - 1 - (((qi - 1 - s) % nq + nq) % nq);
        if (il >= 0) (void)mbar_wait(q_full + 8 * s, (il / nq) & 1);
      }
    }
  } else if (warp == tcp::kVWarp) {
    // ---------------- V gather: the units from the queue, in order ----------------
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmv) : "memory");
    int J = 0;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(u_full + 8 * slot, (k >> 1) & 1))) {
        ok = false;
        break;
      }
      const int2 uv = unit_sh[slot];
      const int u = uv.x;
      __syncwarp();
      if (lane == 0) mbar_arrive(u_empty + 8 * slot);
      if (u < 0) break;
      const TcUnit t = tc_unit(a, u, uv.y);
      const int64_t tab_row = (int64_t)t.b * a.max_blocks;
      const int nblk = t.blk_end - t.blk0;
      int tab = 0;
      for (int j = 0; j < t.ntiles; ++j) {
        const int st = J % kStages;
        if (J >= kStages && !__all_sync(0xffffffffu, mbar_wait(v_empty + 8 * st, ((J - kStages) / kStages) & 1))) {
          ok = false;
          break;
        }
        if ((j & 3) == 0) {  // clamped as the K gather clamps them (which reports it)
          const int bi = j * kTileBlk + lane;
          const int32_t v = bi < nblk ? a.table[tab_row + t.blk0 + bi] : 0;
          tab = v < 0 ? 0 : (v >= a.num_blocks ? (int)(a.num_blocks - 1) : v);
        }
        const int nb = min(kTileBlk, nblk - j * kTileBlk);
        const uint32_t fb = v_full + 8 * st;
        if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)nb * 2u * 2048u);
        __syncwarp();
        const int phys = __shfl_sync(0xffffffffu, tab, (j & 3) * kTileBlk + (lane & 7));
        if (lane < nb) {
          const uint32_t d = vslot(st) + lane * 2048;
          tma_load_4d(d, &tmv, fb, 0, 0, t.g, phys);
          tma_load_4d(d + kHalf, &tmv, fb, 64, 0, t.g, phys);
        }
        ++J;
      }
    }
    if (lane == 0) {
      if (!ok) atomicOr(&g_attn_error, kErrWaitTimeout);
      for (int st = 0; st < kStages; ++st) {  // the last V tile issued into each slot has landed, bounded
        const int jl = J - 1 - (((J - 1 - st) % kStages + kStages) % kStages);
        if (jl >= 0) (void)mbar_wait(v_full + 8 * st, (jl / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue ----------------
    // The tensor pipe runs one thread's MMAs in order: S of tile J + 2
    // overwrites the buffer that P of tile J occupied only after P V of tile J
    // has read it, and a Q slot is reloaded only after the commit that follows
    // its unit's last S.
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, kTileTok), id_pv = idesc_bf16_bmn(128, kD);
      int ofn = 0;  // o_free phases waited
      // O[J & 1] += P V of tile J; acc = 0 starts the accumulator afresh (the
      // group's first tile of a unit); wait_o: the even group must first have
      // read both accumulators of the previous unit
      auto issue_pv = [&](int Jp, bool acc, bool wait_o) {
        const int pg = Jp & 1;
        if (wait_o) {
          if (!mbar_wait(o_free, ofn & 1)) return false;
          ++ofn;
        }
        if (!mbar_wait(p_full + 8 * pg, (Jp >> 1) & 1)) return false;
        if (!mbar_wait(v_full + 8 * (Jp % kStages), (Jp / kStages) & 1)) return false;
        tc_fence_after();
        const uint32_t v0 = vslot(Jp % kStages);
#pragma unroll
        for (int kk = 0; kk < kTileTok / 16; ++kk)  // 16 tokens = 8 columns of P
          umma_bf16_ta(tmem + o_col(pg), tmem + s_col(pg) + kk * 8, sw128_desc_mn(v0 + kk * 2048, kHalf, 1024), id_pv,
                       (acc || kk > 0) ? 1u : 0u);
        umma_commit(v_empty + 8 * (Jp % kStages));  // the V slot is free once these MMAs have read it
        umma_commit(pv_done + 8 * pg);
        return true;
      };
      int J = 0, qi = 0;
      int pend = -1;                       // the tile whose P V is still to issue
      bool pend_acc = false, pend_wait = false;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!mbar_wait(u_full + 8 * slot, (k >> 1) & 1)) {
          ok = false;
          break;
        }
        const int2 uv = unit_sh[slot];
        const int u = uv.x;
        mbar_arrive(u_empty + 8 * slot);
        if (u < 0) break;
        const TcUnit t = tc_unit(a, u, uv.y);
        if (t.ntiles == 0) {
          // The last P V of the previous unit waits for no S here: issued now.
          // (Held back, it would wait for the next unit with tiles, which the
          // queue may publish only once the softmax warps, who need this P V
          // to finish their epilogue, have taken this empty unit.)
          if (pend >= 0 && !issue_pv(pend, pend_acc, pend_wait)) {
            ok = false;
            break;
          }
          pend = -1;
          continue;
        }
        const int qs = qi % nq;
        if (!mbar_wait(q_full + 8 * qs, (qi / nq) & 1)) {
          ok = false;
          break;
        }
        const uint32_t qa = base + kQ + qs * tcp::kQSlot;
        for (int j = 0; j < t.ntiles; ++j, ++J) {
          const int ks = J % kStages, sg = J & 1;
          if (!mbar_wait(k_full + 8 * ks, (J / kStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k0 = kslot(ks);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            umma_bf16(tmem + s_col(sg), sw128_desc(qa + (kk >> 2) * kHalf + (kk & 3) * 32),
                      sw128_desc(k0 + (kk >> 2) * kHalf + (kk & 3) * 32), id_s, kk > 0 ? 1u : 0u);
          umma_commit(k_empty + 8 * ks);  // the K slot is free once S has read it
          umma_commit(s_full + 8 * sg);
          if (j == t.ntiles - 1) umma_commit(q_free + 8 * qs);
          if (pend >= 0 && !issue_pv(pend, pend_acc, pend_wait)) {
            ok = false;
            break;
          }
          pend = J;
          pend_acc = j >= 2;
          pend_wait = j == 0 && qi > 0;
        }
        ++qi;
      }
      if (ok && pend >= 0 && !issue_pv(pend, pend_acc, pend_wait)) ok = false;
      if (!ok) atomicOr(&g_attn_error, kErrWaitTimeout);
      umma_commit(fin);  // completes once every MMA issued above has
      (void)mbar_wait(fin, 0);
    }
  } else {
    // ---------------- softmax: group grp takes the tiles J of parity grp ----------------
    const int grp = (warp - kSoft0) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row = tensor-memory lane
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = trow + s_col(grp), tO = trow + o_col(grp);
    const bool live = r < a.QR;
    int J = 0, qi = 0;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(u_full + 8 * slot, (k >> 1) & 1))) {
        ok = false;
        break;
      }
      const int2 uv = unit_sh[slot];
      const int u = uv.x;
      __syncwarp();
      if (lane == 0) mbar_arrive(u_empty + 8 * slot);
      if (u < 0) break;
      const TcUnit t = tc_unit(a, u, uv.y);
      const int tail_row0 = (t.item - (a.B * a.Hkv - a.tail_items)) * a.QR;  // pieces: first tail row of the item
      if (t.ntiles == 0) {  // nothing of the sequence in this unit
        if (grp == 0 && t.piece >= 0) {  // an empty piece: (m, l, o) = (-inf, 0, 0)
          for (int i = r; i < a.QR * kD; i += 128) {
            const int64_t pr = (int64_t)(tail_row0 + i / kD) * a.tail_pieces + t.piece;
            a.tail_o[pr * kD + i % kD] = 0.f;
            if (i % kD == 0) {
              a.tail_ml[pr * 2] = kNegInf;
              a.tail_ml[pr * 2 + 1] = 0.f;
            }
          }
        } else if (grp == 0 && a.nchunks == 1) {  // an empty sequence: zero rows
          for (int i = r; i < a.QR * kD / 2; i += 128) {
            const int rr = i / (kD / 2);
            const int64_t orow = ((int64_t)t.b * a.W + rr / a.G) * a.Hq + t.g * a.G + rr % a.G;
            reinterpret_cast<uint32_t*>(a.out + orow * kD)[i % (kD / 2)] = 0u;
          }
        }
        continue;
      }
      const int J0 = J;
      J += t.ntiles;
      // key j is visible to row r iff j < ctx and j <= ctx - W + r / G
      const int lim = live ? min(t.ctx - 1, t.ctx - a.W + r / a.G) : -1;
      const int tok_end = min(t.blk_end * kBlk, t.ctx);  // tokens past this are absent or past the context
      float m = kNegInf, l = 0.f;
      int last = -1;  // this group's last tile of the unit
      for (int Jt = J0 + ((J0 ^ grp) & 1); Jt < J; Jt += 2) {
        const int tok0 = (t.blk0 + (Jt - J0) * kTileBlk) * kBlk;  // first token of the tile
        if (!__all_sync(0xffffffffu, mbar_wait(s_full + 8 * grp, (Jt >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[kTileTok];
        {
          uint32_t u0[32], u1[32], u2[32], u3[32];  // four loads in flight, one wait
          tmem_ld32_nowait(tS, u0);
          tmem_ld32_nowait(tS + 32, u1);
          tmem_ld32_nowait(tS + 64, u2);
          tmem_ld32_nowait(tS + 96, u3);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = __uint_as_float(u0[c]);
            sv[32 + c] = __uint_as_float(u1[c]);
            sv[64 + c] = __uint_as_float(u2[c]);
            sv[96 + c] = __uint_as_float(u3[c]);
          }
        }
        const int vl = min(lim, tok_end - 1) - tok0;  // columns 0 .. vl are visible to this row
        const float alpha = tc_softmax_tile(sv, vl, a.scale_log2, m, l, tS);
        // V rows past the context (or of absent blocks) are zeroed before the
        // MMA reads them: 0 * NaN would otherwise leak stale pool contents
        if (tok0 + kTileTok > tok_end) {
          if (!__all_sync(0xffffffffu, mbar_wait(v_full + 8 * (Jt % kStages), (Jt / kStages) & 1))) {
            ok = false;
            break;
          }
          if (tok0 + r >= tok_end) {  // this thread's token row of the tile
            const uint32_t v0 = vslot(Jt % kStages) + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              sts128z(v0 + c * 16);
              sts128z(v0 + kHalf + c * 16);
            }
          }
        }
        if (last >= 0) {
          // O holds this group's earlier tiles of the unit once their P V is
          // complete; it is rescaled only when some row of the warp moved its
          // reference maximum
          if (!__all_sync(0xffffffffu, mbar_wait(pv_done + 8 * grp, (last >> 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
#pragma unroll
              for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
              tmem_st32(tO + c * 32, o);
            }
          }
        }
        tmem_wait_st();            // P (and a rescaled O) in place
        fence_proxy_async_smem();  // zeroed V rows, if any
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + 8 * grp);
        last = Jt;
      }
      if (!ok) break;
      // ---------------- the unit's epilogue ----------------
      // each group waits for its last P V; the odd group hands over its (m, l)
      // and goes on; the even group combines both O accumulators row by row,
      // then frees them for the next unit's first P V
      if (last >= 0 && !__all_sync(0xffffffffu, mbar_wait(pv_done + 8 * grp, (last >> 1) & 1))) {
        ok = false;
        break;
      }
      if (grp == 1) {
        if (qi >= 1 && !__all_sync(0xffffffffu, mbar_wait(xm_empty, (qi - 1) & 1))) {
          ok = false;
          break;
        }
        xm[0][r] = last < 0 ? kNegInf : m;
        xm[1][r] = last < 0 ? 0.f : l;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(xm_full);
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(xm_full, qi & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float m1 = xm[0][r], l1 = xm[1][r];
        __syncwarp();
        if (lane == 0) mbar_arrive(xm_empty);
        const float m0 = last < 0 ? kNegInf : m, l0 = last < 0 ? 0.f : l;
        const float ms = fmaxf(m0, m1);
        const float mbs = ms == kNegInf ? 0.f : ms;
        const float w0 = m0 != kNegInf ? ex2(m0 - mbs) : 0.f, w1 = m1 != kNegInf ? ex2(m1 - mbs) : 0.f;
        // an accumulator with no tile of this unit holds the previous unit's
        // values: it is neither read (warp-uniform) nor added (per row)
        const bool use0 = __any_sync(0xffffffffu, m0 != kNegInf), use1 = __any_sync(0xffffffffu, m1 != kNegInf);
        const float lt = __fadd_rn(__fmul_rn(l0, w0), __fmul_rn(l1, w1));
        const int64_t orow = live ? ((int64_t)t.b * a.W + r / a.G) * a.Hq + t.g * a.G + r % a.G : 0;
        const float inv = (lt > 0.f ? 1.f / lt : 0.f) * a.v_scale;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o0[32], o1[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) o0[q] = o1[q] = 0u;
          // warp-collective (every lane takes part); both loads in flight, one wait
          if (use0) tmem_ld32_nowait(trow + o_col(0) + c * 32, o0);
          if (use1) tmem_ld32_nowait(trow + o_col(1) + c * 32, o1);
          tmem_wait_ld();
          float v[32];
#pragma unroll
          for (int q = 0; q < 32; ++q)
            v[q] = combine2(__uint_as_float(o0[q]), w0, m0 != kNegInf, __uint_as_float(o1[q]), w1, m1 != kNegInf);
          if (live) {
            if (t.piece >= 0) {
              float4* po = reinterpret_cast<float4*>(
                  a.tail_o + ((int64_t)(tail_row0 + r) * a.tail_pieces + t.piece) * kD + c * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                po[q] = make_float4(v[4 * q] * a.v_scale, v[4 * q + 1] * a.v_scale, v[4 * q + 2] * a.v_scale,
                                    v[4 * q + 3] * a.v_scale);
            } else if (a.nchunks == 1) {
              uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kD + c * 32);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(pack_bf16x2(v[8 * q] * inv, v[8 * q + 1] * inv),
                                    pack_bf16x2(v[8 * q + 2] * inv, v[8 * q + 3] * inv),
                                    pack_bf16x2(v[8 * q + 4] * inv, v[8 * q + 5] * inv),
                                    pack_bf16x2(v[8 * q + 6] * inv, v[8 * q + 7] * inv));
            } else {
              float4* po = reinterpret_cast<float4*>(a.part_o + (orow * a.nchunks + t.chunk) * kD + c * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                po[q] = make_float4(v[4 * q] * a.v_scale, v[4 * q + 1] * a.v_scale, v[4 * q + 2] * a.v_scale,
                                    v[4 * q + 3] * a.v_scale);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);  // both accumulators read
        if (live && t.piece >= 0) {
          const int64_t pr = (int64_t)(tail_row0 + r) * a.tail_pieces + t.piece;
          a.tail_ml[pr * 2] = ms;
          a.tail_ml[pr * 2 + 1] = lt;
        } else if (live && a.nchunks > 1) {
          a.part_ml[(orow * a.nchunks + t.chunk) * 2] = ms;
          a.part_ml[(orow * a.nchunks + t.chunk) * 2 + 1] = lt;
        }
      }
      ++qi;
    }
    if (!ok && lane == 0) atomicOr(&g_attn_error, kErrWaitTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The balanced tail's merge: one warp per query row of a split item combines
// its pieces' (o, m, l) in piece order.
__global__ void __launch_bounds__(128) attn_tail_merge_kernel(const Args a) {
  grid_dependency_wait();  // the partials and the order come from the tensor-core kernel
  allow_dependent_launch();
  const int t = (int)blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= a.tail_items * a.QR) return;
  const int item = a.B * a.Hkv - a.tail_items + t / a.QR, r = t % a.QR;
  const int pos = item / a.Hkv, g = item % a.Hkv;
  const int b = a.lpt ? (int)a.tail_seq[pos] : pos;  // the tail items are the last ones of its order
  if (b >= a.B) {  // the order was not written (the tensor-core kernel bailed out): flag, write nothing
    if (lane == 0) atomicOr(&g_attn_error, kErrBadInput);
    return;
  }
  const int P = a.tail_pieces;
  const float* ml = a.tail_ml + (int64_t)t * P * 2;
  float mstar = kNegInf;
  for (int k = 0; k < P; ++k) mstar = fmaxf(mstar, __ldcg(ml + 2 * k));
  const float mbase = mstar == kNegInf ? 0.f : mstar;
  float l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < P; ++k) {
    const float w = ex2(__ldcg(ml + 2 * k) - mbase);
    l += w * __ldcg(ml + 2 * k + 1);
    const float4 v = __ldcg(reinterpret_cast<const float4*>(a.tail_o + ((int64_t)t * P + k) * kD) + lane);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int64_t orow = ((int64_t)b * a.W + r / a.G) * a.Hq + g * a.G + r % a.G;
  uint2 o;
  o.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  o.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(a.out + orow * kD + lane * 4) = o;
}

// A 4-D tensor map over a KV pool [num_blocks][hkv][16][128] whose box is 16
// tokens of one (block, kv head), 128 bytes wide (64 bf16 head dims or 128
// FP8 codes), 128-byte swizzled.
cudaError_t kv_tensor_map(const void* pool, bool f8, int hkv, int64_t num_blocks, CUtensorMap* out) {
  const uint64_t es = f8 ? 1 : 2;
  const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)kBlk, (uint64_t)hkv, (uint64_t)num_blocks};
  const uint64_t strides[3] = {(uint64_t)kD * es, (uint64_t)kBlk * kD * es, (uint64_t)hkv * kBlk * kD * es};
  const uint32_t box[4] = {f8 ? 128u : 64u, (uint32_t)kBlk, 1, 1};
  return tensor_map(out, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pool, dims,
                    strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Queries [b][w][hq][128] bf16 as a 4-D map (dims, heads, positions,
// sequences) whose box is one kv head's G heads at all W positions, one 64-dim
// half: it lands as the W x G query rows of that head, 128 bytes each,
// 128-byte swizzled.
cudaError_t q_tensor_map(const uint16_t* q, int b, int w, int hq, int hkv, CUtensorMap* out) {
  const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)hq, (uint64_t)w, (uint64_t)b};
  const uint64_t strides[3] = {(uint64_t)kD * 2, (uint64_t)hq * kD * 2, (uint64_t)w * hq * kD * 2};
  const uint32_t box[4] = {64u, (uint32_t)(hq / hkv), (uint32_t)w, 1};
  return tensor_map(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int QT, bool F8>
cudaError_t launch_split(const Args& a, const AttnPlan& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                         cudaStream_t s) {
  using C = Cfg<QT, F8>;
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(attn_split_kernel<QT, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(1, std::memory_order_relaxed);
  }
  dim3 grid(p.nchunks, a.Hkv, a.B * p.qgroups);
  return launch_pdl(attn_split_kernel<QT, F8>, grid, dim3(kThreads), C::BYTES, s, tmk, tmv, a);
}

template <int QT, bool F8>
constexpr int ctas_per_sm() {
  // shared memory (227 KB per SM usable) and registers (~165 per thread -> 3 CTAs)
  return std::min(227 * 1024 / Cfg<QT, F8>::BYTES, 3);
}

template <bool F8>
int ctas_per_sm_of(int qt) {
  return qt == 1 ? ctas_per_sm<1, F8>() : (qt == 2 ? ctas_per_sm<2, F8>() : ctas_per_sm<4, F8>());
}

template <bool F8>
int smem_of(int qt) {
  return qt == 1 ? Cfg<1, F8>::BYTES : (qt == 2 ? Cfg<2, F8>::BYTES : Cfg<4, F8>::BYTES);
}

// Fixed scratch for gqa_decode_attn_static_ws, for callers that cannot
// allocate device memory. Every GPU that loads this module holds it until the
// process exits. It is zero at load; the attention path never uses its
// counter region and writes every split-KV partial before reading it.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) uint8_t g_attn_static_scratch[kStaticScratchBytes];

}  // namespace

size_t attn_static_scratch_bytes() { return kStaticScratchBytes; }

// Device address of the static scratch in the current CUDA context. In host
// code the array's name is only a host-side stand-in, so the address is
// looked up with cudaGetSymbolAddress (the first lookup in a context may load
// this module there, which reserves the array) and cached under the context's
// id, which the driver never reuses within a process: after a device reset
// the new context looks the address up again instead of reusing a stale one.
namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

bool current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t attn_static_scratch(void** ptr) {
  static std::mutex mu;
  static unsigned long long ids[64];
  static void* addrs[64];
  static int used = 0, next = 0;
  unsigned long long id = 0;
  bool have_id = current_ctx_id(&id);
  if (have_id) {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
      if (ids[i] == id) {
        *ptr = addrs[i];
        return cudaSuccess;
      }
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
  if (e != cudaSuccess) return e;
  if (!have_id) have_id = current_ctx_id(&id);  // the lookup made the context current
  if (have_id) {
    std::lock_guard<std::mutex> lk(mu);
    ids[next] = id;
    addrs[next] = p;
    next = (next + 1) % 64;
    used = used < 64 ? used + 1 : 64;
  }
  *ptr = p;
  return cudaSuccess;
}

AttnPlan plan_attn(int b, int w, int hq, int hkv, int max_context, int num_sms, bool kv_fp8) {
  AttnPlan p{};
  const int G = hq / hkv;
  const int qr = G * w;
  const int tiles = (qr + 15) / 16;
  p.qt = tiles <= 1 ? 1 : (tiles <= 2 ? 2 : 4);
  p.qgroups = (tiles + p.qt - 1) / p.qt;
  const int ks = 4 / p.qt;
  const int maxblk = std::max(1, (max_context + kBlk - 1) / kBlk);
  const int64_t items = (int64_t)b * hkv * p.qgroups;
  const int cps = kv_fp8 ? ctas_per_sm_of<true>(p.qt) : ctas_per_sm_of<false>(p.qt);
  const int64_t slots = (int64_t)std::max(num_sms, 1) * cps;
  // About four waves of CTAs so that waves balance; each key-slot group gets
  // at least four blocks, and a chunk's partial (o, m, l) per query row stays
  // small next to the chunk's K/V bytes (cb >= 1.3 * rows), unless that would
  // leave SMs idle: a small problem (few sequences and heads) is latency
  // bound, so its chunks shrink until the CTAs fill one wave.
  const int64_t per_item = std::max<int64_t>(1, (slots + items - 1) / items);
  const int cb_wave = std::max<int>(ks, (int)((maxblk + per_item - 1) / per_item));
  const int cb_min = std::max(4 * ks, std::min((13 * qr + 9) / 10, cb_wave));
  int64_t nch = std::max<int64_t>(1, (4 * slots + items - 1) / items);
  int cb = std::max<int>((int)((maxblk + nch - 1) / nch), cb_min);
  // An FP8 block holds half the bytes of a bf16 block: twice the blocks keep
  // a chunk's bytes, and the per-CTA start-up cost they amortise, the same.
  if (kv_fp8) cb *= 2;
  // Fewer chunks when the sequences and heads already fill the GPU: time
  // ~ waves x blocks per chunk, with a quarter more for the merge pass that a
  // split needs. Taken only when it beats the plan above by 13% (measured on
  // the bf16 cache: 32 x 2048 tokens 55.0 -> 46.1 us, 64 x 2048 92.9 -> 82.0
  // us, 16 x 4096 53.8 -> 48.6 us; long contexts keep their plan).
  {
    auto rounded = [&](int64_t c) { return (std::min<int64_t>(c, maxblk) + ks - 1) / ks * ks; };
    auto cost = [&](int64_t n) {
      const int64_t c = rounded((maxblk + n - 1) / n);
      const int64_t n_eff = (maxblk + c - 1) / c;
      const int64_t waves = (items * n_eff + slots - 1) / slots;
      return (double)(waves * c) * (n_eff > 1 ? 1.25 : 1.0);
    };
    const int64_t cur = (maxblk + rounded(cb) - 1) / rounded(cb);
    const double cur_cost = cost(cur);
    int64_t best = cur;
    double best_cost = cur_cost;
    for (int64_t n = 1; n < cur; ++n) {
      const double c = cost(n);
      if (c < best_cost) {
        best_cost = c;
        best = n;
      }
    }
    if (best < cur && best_cost < 0.87 * cur_cost) cb = (int)rounded((maxblk + best - 1) / best);
    // Small problems (fewer items than SMs, at most about 2 MB of bf16 KV per
    // SM): one wave of CTAs, with the chunk count that minimises the blocks
    // the busiest SM streams (fewer chunks on ties). Measured at batch 1-4,
    // each wave of CTAs on an SM costs about as much as 30 more blocks
    // (start-up, first loads, the chunk's partial), so several waves of short
    // chunks lose to one wave of long ones: batch 1 x 32768 tokens 37.3 ->
    // about 27 us, batch 4 x 8192 34.5 -> about 28 us. Test hook:
    // DQD_ATTN_PLAN=0 keeps the plan above; =1 takes this one whenever there
    // are fewer items than SMs.
    const char* plan_env = std::getenv("DQD_ATTN_PLAN");
    const bool small = items < num_sms && (items * maxblk <= (int64_t)256 * std::max(num_sms, 1) ||
                                           (plan_env && plan_env[0] == '1'));
    if (small && !(plan_env && plan_env[0] == '0')) {
      const int64_t n_max = std::max<int64_t>(1, (int64_t)std::max(num_sms, 1) * cps / items);
      int64_t best_load = -1;
      for (int64_t n = 1; n <= std::min<int64_t>(n_max, maxblk); ++n) {
        const int64_t c = std::max<int64_t>(rounded((maxblk + n - 1) / n), cb_min);
        const int64_t n_eff = (maxblk + c - 1) / c;
        const int64_t load = (items * n_eff + num_sms - 1) / std::max(num_sms, 1) * c;
        if (best_load < 0 || load < best_load) {
          best_load = load;
          cb = (int)c;
        }
      }
    }
  }
  // Test hook: DQD_ATTN_CHUNK_BLOCKS forces the split-KV chunk size.
  if (const char* env = std::getenv("DQD_ATTN_CHUNK_BLOCKS")) {
    const long v = std::strtol(env, nullptr, 10);
    if (v >= 1) cb = (int)v;
  }
  cb = std::min(cb, maxblk);
  cb = (cb + ks - 1) / ks * ks;
  p.chunk_blocks = cb;
  p.nchunks = (maxblk + cb - 1) / cb;
  p.smem_bytes = kv_fp8 ? smem_of<true>(p.qt) : smem_of<false>(p.qt);
  p.kv_fp8 = kv_fp8 ? 1 : 0;
  // Wide query tiles over a bf16 cache (17..128 rows per kv head: verify
  // widths) take the tensor-core form: one CTA per SM, chunks of whole
  // 128-token tiles; the chunk count minimises waves x (chunk + a fixed cost
  // per CTA), with a quarter of a chunk more when the partials need merging.
  // The fixed cost (Q load, the first tile's copy latency, epilogue) is about
  // 96 blocks' worth: measured at batch 64, width 16, 144 blocks per
  // sequence, one chunk 140 us, two 173 us, three 207 us. Test hook:
  // DQD_ATTN_TC=0 keeps the mma.sync form.
  {
    const char* tc_env = std::getenv("DQD_ATTN_TC");
    p.tc = (!kv_fp8 && qr > 16 && qr <= 128 && !(tc_env && tc_env[0] == '0')) ? 1 : 0;
  }
  if (p.tc) {
    const int64_t titems = (int64_t)b * hkv, tslots = std::max(num_sms, 1);
    auto round8 = [](int64_t c) { return (c + 7) / 8 * 8; };
    double best = -1.0;
    int64_t best_c = round8(maxblk);
    for (int64_t n = 1; n <= std::min<int64_t>(64, (maxblk + 7) / 8); ++n) {
      const int64_t c = round8((maxblk + n - 1) / n);
      const int64_t n_eff = (maxblk + c - 1) / c;
      const int64_t waves = (titems * n_eff + tslots - 1) / tslots;
      const double cost = (double)waves * (double)(c + 96) + (n_eff > 1 ? 0.25 * (double)c : 0.0);
      if (best < 0 || cost < best) {
        best = cost;
        best_c = c;
      }
    }
    int64_t c = best_c;
    if (const char* env = std::getenv("DQD_ATTN_CHUNK_BLOCKS")) {
      const long v = std::strtol(env, nullptr, 10);
      if (v >= 1) c = v;
    }
    c = std::min<int64_t>(c, maxblk);
    p.chunk_blocks = (int)c;
    p.nchunks = (int)((maxblk + c - 1) / c);
    p.qt = 4;
    p.qgroups = 1;
    p.smem_bytes = tca::kSmem;
    // Balanced tail: with one chunk per item and more items than SMs, the
    // last partial wave's R items are split into floor(SMs / R) pieces each,
    // so that they finish together instead of leaving most SMs idle (batch
    // 64, width 16: 512 items, 3.37 waves). Test hook: DQD_ATTN_TAIL=0 keeps
    // whole items.
    const char* tail_env = std::getenv("DQD_ATTN_TAIL");
    const int64_t R = titems % tslots;
    int64_t pieces = R > 0 ? std::min<int64_t>(8, tslots / R) : 0;
    if (const char* env = std::getenv("DQD_ATTN_TAIL_PIECES")) {  // test hook: pieces per tail item
      const long v = std::strtol(env, nullptr, 10);
      if (v >= 2 && v <= 64 && R > 0) pieces = v;
    }
    if (p.nchunks == 1 && titems > tslots && pieces >= 2 && !std::getenv("DQD_ATTN_CHUNK_BLOCKS") &&
        !(tail_env && tail_env[0] == '0')) {
      p.tail_items = (int)R;
      p.tail_pieces = (int)pieces;
    }
    // Persistent form when there are more units than SMs: one CTA per SM
    // takes the units from a queue in the workspace's counter region (with
    // fewer units it only adds the queue's cost: batch 1, width 16, 8192
    // tokens 17.6 -> 19.0 us). Test hook: DQD_ATTN_PERSIST=0 keeps one CTA per
    // unit, =1 takes the persistent form whatever the unit count.
    const char* persist_env = std::getenv("DQD_ATTN_PERSIST");
    const int64_t units = p.tail_pieces > 0 ? titems - p.tail_items + (int64_t)p.tail_items * p.tail_pieces
                                            : titems * p.nchunks;
    const bool force = persist_env && persist_env[0] == '1', off = persist_env && persist_env[0] == '0';
    if (!off && (force || units > tslots)) p.persist = (int)std::min<int64_t>(units, tslots);
  }
  const size_t rows = (size_t)b * w * hq;
  p.ws_bytes = p.nchunks > 1 ? kCounterBytes + rows * p.nchunks * (kD + 2) * sizeof(float) : 0;
  if (p.tail_pieces > 0)  // partials, then the longest-first order of the sequences
    p.ws_bytes = kCounterBytes + (size_t)p.tail_items * qr * p.tail_pieces * (kD + 2) * sizeof(float) + kLptMaxB;
  if (p.persist > 0) p.ws_bytes = std::max(p.ws_bytes, kCounterBytes);
  return p;
}

cudaError_t attn_take_device_error(uint32_t* flags) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_attn_error, &zero, sizeof zero);
  *flags |= v;
  return e;
}

cudaError_t launch_attn(const AttnLaunch& l, const AttnPlan& p, cudaStream_t s) {
  Args a;
  a.q = l.q;
  a.table = l.block_table;
  a.ctx = l.context_lens;
  a.out = l.out;
  const size_t rows = (size_t)l.b * l.w * l.hq;
  if (p.nchunks > 1) {
    a.part_o = reinterpret_cast<float*>(static_cast<uint8_t*>(l.workspace) + kCounterBytes);
    a.part_ml = a.part_o + rows * p.nchunks * kD;
  } else {
    a.part_o = nullptr;
    a.part_ml = nullptr;
  }
  a.tail_items = p.tail_items;
  a.tail_pieces = p.tail_pieces;
  a.ctr = p.persist > 0 ? static_cast<unsigned*>(l.workspace) : nullptr;
  {  // test hook: DQD_ATTN_ORDER=0 keeps the sequences in index order
    const char* env = std::getenv("DQD_ATTN_ORDER");
    a.lpt = p.tc && l.b <= kLptMaxB && !(env && env[0] == '0') ? 1 : 0;
  }
  a.tail_o = nullptr;
  a.tail_ml = nullptr;
  a.tail_seq = nullptr;
  if (p.tail_pieces > 0) {
    const size_t trows = (size_t)p.tail_items * (l.hq / l.hkv) * l.w;
    a.tail_o = reinterpret_cast<float*>(static_cast<uint8_t*>(l.workspace) + kCounterBytes);
    a.tail_ml = a.tail_o + trows * p.tail_pieces * kD;
    a.tail_seq = reinterpret_cast<uint8_t*>(a.tail_ml + trows * p.tail_pieces * 2);
  }
  a.num_blocks = l.num_blocks;
  a.max_blocks = l.max_blocks;
  a.max_context = l.max_context;
  a.B = l.b;
  a.W = l.w;
  a.Hq = l.hq;
  a.Hkv = l.hkv;
  a.G = l.hq / l.hkv;
  a.QR = a.G * l.w;
  a.chunk_blocks = p.chunk_blocks;
  a.nchunks = p.nchunks;
  a.qgroups = p.qgroups;
  const bool f8 = p.kv_fp8 != 0;
  a.scale_log2 = f8 ? l.softmax_scale * l.k_scale * 1.4426950408889634f : l.softmax_scale * 1.4426950408889634f;
  a.v_scale = f8 ? l.v_scale : 1.f;
  CUtensorMap tmk, tmv;
  cudaError_t e = kv_tensor_map(l.k_pool, f8, l.hkv, l.num_blocks, &tmk);
  if (e == cudaSuccess) e = kv_tensor_map(l.v_pool, f8, l.hkv, l.num_blocks, &tmv);
  if (e != cudaSuccess) return e;
  if (p.tc && p.persist > 0) {
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(attn_tcp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tca::kSmem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) configured[dev].store(1, std::memory_order_relaxed);
    }
    CUtensorMap tmq;
    e = q_tensor_map(l.q, l.b, l.w, l.hq, l.hkv, &tmq);
    if (e != cudaSuccess) return e;
    e = launch_pdl(attn_tcp_kernel, dim3((unsigned)p.persist), dim3(tcp::kThreads), (size_t)tca::kSmem, s, tmk, tmv,
                   tmq, a);
    if (e == cudaSuccess && p.tail_pieces > 0) {
      const unsigned trows = (unsigned)(p.tail_items * a.QR);
      return launch_pdl(attn_tail_merge_kernel, dim3((trows + 3) / 4), dim3(128), 0, s, a);
    }
  } else if (p.tc) {
    static std::atomic<int> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tca::kSmem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) configured[dev].store(1, std::memory_order_relaxed);
    }
    const dim3 grid = p.tail_pieces > 0
                          ? dim3((unsigned)(a.B * a.Hkv - p.tail_items + p.tail_items * p.tail_pieces))
                          : dim3(p.nchunks, a.Hkv, a.B);
    e = launch_pdl(attn_tc_kernel, grid, dim3(tca::kThreads), (size_t)tca::kSmem, s, tmk, tmv, a);
    if (e == cudaSuccess && p.tail_pieces > 0) {
      const unsigned trows = (unsigned)(p.tail_items * a.QR);
      return launch_pdl(attn_tail_merge_kernel, dim3((trows + 3) / 4), dim3(128), 0, s, a);
    }
  } else if (f8) {
    switch (p.qt) {
      case 1: e = launch_split<1, true>(a, p, tmk, tmv, s); break;
      case 2: e = launch_split<2, true>(a, p, tmk, tmv, s); break;
      default: e = launch_split<4, true>(a, p, tmk, tmv, s); break;
    }
  } else {
    switch (p.qt) {
      case 1: e = launch_split<1, false>(a, p, tmk, tmv, s); break;
      case 2: e = launch_split<2, false>(a, p, tmk, tmv, s); break;
      default: e = launch_split<4, false>(a, p, tmk, tmv, s); break;
    }
  }
  if (e != cudaSuccess || p.nchunks == 1) return e;
  if (p.nchunks >= 8) return launch_pdl(attn_merge_wide_kernel, dim3((unsigned)rows), dim3(128), 0, s, a);
  const int64_t blocks = ((int64_t)rows + 3) / 4;
  return launch_pdl(attn_merge_kernel, dim3((unsigned)blocks), dim3(128), 0, s, a);
}

}  // namespace dqd
