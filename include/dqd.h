/*
 * dqd — memory-bound LLM decode kernels for GB300 (sm_103a), C ABI.
 *
 * Two operations make up the hot path of one decode (or speculative-verify)
 * step, and offline operations prepare weights for it:
 *
 *   dq_gemm          y = x * deq(W)^T, a weight-only quantised skinny GEMM.
 *   gqa_decode_attn  GQA attention of the new tokens' queries over a paged
 *                    BF16 KV cache, causal inside the verify block
 *                    (gqa_decode_attn_fp8kv: the same over an FP8-E4M3 cache).
 *   pack_int4_g128   re-lay INT4 g128 codes/scales/zeros for dq_gemm.
 *   quant_fp8_rowwise  BF16 W -> FP8 E4M3 codes + per-output-row fp32 scales.
 *   quant_int4_g128  BF16 W -> INT4 codes + per-group bf16 scales and zeros.
 *
 * the step between the QKV projection and the attention:
 *
 *   rope_kv_append   rotate the new tokens' q and k, append k and v to the cache,
 *
 * and the step after the verify forward:
 *
 *   spec_verify_greedy / spec_verify_sample  accept a speculative draft
 *                    block and invalidate the rejected KV tail.
 *
 * Sources (web pages):
 *   [MTC]  "降低每個 Token 的生成成本" (Making each token cheaper), optiverse-tech.com
 *   [LIF]  "LLM 推理是怎么变快的" (How LLM inference gets fast), random.sdx88.com
 *   [CS10] "第 10 讲：推理" (CS336 lecture 10 notes), semidirectx.com
 *   [ATC]  "AcceptedTokens 阅读笔记" (speculative-decoding energy notes), zhongzhuzhou.org
 *
 * Conventions for every call:
 *   - Buffers are owned by the caller. Pointers named in a signature are
 *     DEVICE pointers (unless documented otherwise) and must be 16-byte
 *     aligned. The library never allocates, frees or synchronises.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     A status is returned after all host-side checks and the launches;
 *     argument errors are detected on the host and returned before anything
 *     is enqueued. Device-side faults surface at the caller's next sync.
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Workspace: calls that need scratch take (workspace, ws_bytes); query the
 *     size with the *_workspace_bytes function for the same arguments on the
 *     same device. The first DQD_WS_COUNTER_BYTES bytes of a workspace hold
 *     arrival counters: they must be zero before the first call that uses
 *     the buffer, and every call leaves them zero again. Calls that share a
 *     workspace must not overlap on the GPU.
 *   - Thread safety: calls may be made from several host threads; the last
 *     error message is kept per host thread (dqd_last_error()).
 */
#ifndef DQD_H_
#define DQD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DQD_API __attribute__((visibility("default")))
#else
#define DQD_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* dqd_stream;

typedef enum {
  DQD_OK = 0,
  DQD_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or shape      */
  DQD_ERR_UNSUPPORTED = 2, /* shape or parameter outside what the kernels do  */
  DQD_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required      */
  DQD_ERR_CUDA = 4         /* a CUDA runtime call or a launch failed          */
} dqd_status;

typedef enum {
  DQD_W_BF16 = 0,      /* data: bf16 [n][k] row-major; scales, zeros: NULL   */
  DQD_W_FP8_E4M3 = 1,  /* data: E4M3 codes u8 [n][k]; scales: fp32 [n];
                          zeros: NULL                                        */
  DQD_W_INT4_G128 = 2  /* data/scales/zeros: the packed buffers written by
                          pack_int4_g128 (layout below)                      */
} dqd_wtype;

/* A weight matrix W [n out][k in]. */
typedef struct {
  int32_t type;        /* dqd_wtype */
  int64_t n, k;
  const void* data;
  const void* scales;
  const void* zeros;
} dqd_weight;

/* Bytes of arrival counters at the start of every workspace. */
#define DQD_WS_COUNTER_BYTES 65536

/* Human-readable name of a status; never NULL. */
DQD_API const char* dqd_status_string(dqd_status status);

/* Detail of the error of the last library call made on the calling host
 * thread (empty string if it succeeded). Valid until that thread's next call. */
DQD_API const char* dqd_last_error(void);

/* Library version, e.g. "dqd 0.1 sm_103a". */
DQD_API const char* dqd_version(void);

/* Errors that only the device can see are recorded in device error words:
 *  - bit 0 (DQD_DEVICE_ERR_WAIT_TIMEOUT): kernels never spin without bound;
 *    every wait on an asynchronous copy gives up after a fixed number of polls
 *    (seconds), records this flag and ends the kernel (its output is then
 *    meaningless);
 *  - bit 1 (DQD_DEVICE_ERR_BAD_INPUT): a kernel met an input outside its
 *    documented range and clamped it, so that every access stays in bounds: a
 *    block-table entry outside [0, num_blocks) (attention, RoPE + append), or
 *    a context_lens[b] below the verify width w or above max_context
 *    (attention). The output of that call is not meaningful.
 * This call synchronises with the current device, returns the OR of the flags
 * raised since the last call in *flags (0: none) and clears them. */
#define DQD_DEVICE_ERR_WAIT_TIMEOUT 1u
#define DQD_DEVICE_ERR_BAD_INPUT 2u
DQD_API dqd_status dqd_device_errors(uint32_t* flags);

/* Diagnostic for failure detection: launches one kernel that waits, with the
 * same bounded polling as every pipeline wait of the library but at most
 * `polls` polls (1 <= polls <= 2^22), on a barrier that nothing completes.
 * The wait gives up, sets DQD_DEVICE_ERR_WAIT_TIMEOUT (read and cleared by
 * dqd_device_errors) and the kernel returns; the context stays usable. */
DQD_API dqd_status dqd_selftest_wait_timeout(uint32_t polls, dqd_stream stream);

/* ------------------------------------------------------------------------
 * pack_int4_g128 — re-lay W4A16 INT4 g128 weights for dq_gemm.
 *
 * Source: [MTC, section "格式" (Formats)]: weight-only INT4 stores 4-bit
 * integers with one scale per group (group size 128) and dequantises to
 * 16-bit before the arithmetic; [CS10 §5.2] scale and zero point.
 * Reading: codes are unsigned 0..15, the zero point is a 4-bit value per
 * group, deq = bf16_RNE((q - z) * s).
 *
 * Inputs (device):
 *   codes        u8 [n][k], values 0..15 (only the low 4 bits are read)
 *   scales_bf16  bf16 [n][k/128]
 *   zeros        u8 [n][k/128], values 0..15 (low 4 bits read)
 * Outputs (device), sizes from pack_int4_g128_bytes:
 *   packed, packed_scales, packed_zeros
 * Requirements: n >= 1, k >= 128, k % 128 == 0, all pointers 16-byte aligned.
 *
 * Packed layout (frozen). NT = ceil(n/16) row tiles, G = k/128 groups,
 * block b = T*G + g for row tile T and group g.
 *   packed:        NT*G blocks of 1024 bytes = 256 little-endian uint32 words.
 *                  Word w = 128*h + 4*l + j (h in 0..1, l in 0..31, j in 0..3).
 *                  With i = 4h + j, c = i/2, e = i%2, r0 = l/4, t = l%4,
 *                  nibble v (bits 4v..4v+3) of word w is the code of
 *                    row    16*T + r0 + 8*(v & 1)
 *                    column 128*g + 32*c + 8*t + 4*e + 2*((v >> 1) & 1) + (v >> 2)
 *                  (This puts, for lane l of a warp, the A-operand fragment
 *                  of eight m16n8k16 MMAs in two 16-byte loads.)
 *   packed_scales: NT*G blocks of 8 uint32 words; word r0 holds the bf16
 *                  scale of row 16T+r0 in bits 0..15 and of row 16T+r0+8 in
 *                  bits 16..31.
 *   packed_zeros:  NT*G blocks of 8 bytes; byte r0 holds the zero point of
 *                  row 16T+r0 in bits 0..3 and of row 16T+r0+8 in bits 4..7.
 *   Rows at or beyond n (padding of the last tile) hold 0 everywhere.
 * Storage: 4 + 16/128 + 4/128 = 4.15625 bits per weight.
 * ---------------------------------------------------------------------- */

/* which: 0 = packed codes, 1 = packed scales, 2 = packed zeros.
 * Returns 0 for invalid arguments. Host-only arithmetic. */
DQD_API size_t pack_int4_g128_bytes(int64_t n, int64_t k, int which);

DQD_API dqd_status pack_int4_g128(const uint8_t* codes, const uint16_t* scales_bf16,
                          const uint8_t* zeros, int64_t n, int64_t k,
                          void* packed, void* packed_scales, void* packed_zeros,
                          dqd_stream stream);

/* ------------------------------------------------------------------------
 * quant_fp8_rowwise — BF16 W [n][k] -> FP8 E4M3 codes [n][k] + fp32 scales [n].
 *
 * Source: [MTC, section "格式" (Formats)]: E4M3 has 4 exponent bits, 3
 * mantissa bits and largest normal 448; values are multiplied by a scale
 * before the cast to fit that range. Reading: per output row n,
 *   scale[n] = fp32(max_k |W[n][k]|) / 448        (IEEE binary32 division)
 *   code[n][k] = e4m3_RNE_satfinite(fp32(W[n][k]) / scale[n])
 * and a row whose entries are all zero takes scale 1. W must be finite.
 * Requirements: n >= 1, k >= 1, k % 16 == 0, pointers 16-byte aligned.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status quant_fp8_rowwise(const uint16_t* w_bf16, int64_t n, int64_t k,
                             uint8_t* codes, float* scales, dqd_stream stream);

/* ------------------------------------------------------------------------
 * quant_int4_g128 — BF16 W [n][k] -> INT4 g128 codes, bf16 scales, zero points
 * (the logical inputs of pack_int4_g128), asymmetric min/max per group.
 *
 * Source: [CS10 §5.2] a scale and a zero point map values onto the integer
 * grid, x ~ (q - z) * s; the granularity demo there: an outlier widens its
 * own group's scale, finer groups are more accurate; [MTC, "格式"] INT4 with
 * one scale per group of 128. The notes' worked example is garbled; reading,
 * for row n and group j (weights W[n][128j .. 128j+127]):
 *   lo = min(0, min W), hi = max(0, max W)          (0 stays on the grid)
 *   s  = bf16_RNE(fp32(fp32(hi - lo) / 15)); all-zero group: s = 1; an s that
 *        rounds to 0 becomes the smallest positive bf16
 *   z  = clamp(rint(fp32(-lo / s)), 0, 15)
 *   q  = clamp(rint(fp32(W / s)) + z, 0, 15)       (rint: ties to even)
 * with IEEE binary32 division; dequantisation is (q - z) * s.
 *
 * w_bf16: [n][k] (device); codes: u8 [n][k], 0..15 (device);
 * scales_bf16: [n][k/128] (device); zeros: u8 [n][k/128] (device).
 * Requirements: n >= 1, k >= 128, k % 128 == 0, W finite, pointers 16-byte
 * aligned.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status quant_int4_g128(const uint16_t* w_bf16, int64_t n, int64_t k,
                           uint8_t* codes, uint16_t* scales_bf16, uint8_t* zeros,
                           dqd_stream stream);

/* ------------------------------------------------------------------------
 * dq_gemm — y[m][n] = sum_k x[m][k] * deq(W)[n][k], bf16 in/out, fp32 accumulate.
 *
 * Source: [MTC, section "量化省下什麼" (What quantisation saves)]: the decode
 * kernel multiplies a quantised matrix by a full-precision vector,
 * dequantising the weights on the fly without quantising the activations;
 * [LIF §4.1] weight-only quantisation dequantises back to 16-bit and wins at
 * small batch because decode is bandwidth-bound.
 * Per weight type:
 *   BF16: y = x W^T.
 *   FP8:  y[m][n] = scale[n] * sum_k x[m][k] * e4m3(code[n][k]); the E4M3
 *         value is exact in bf16 and the scale multiplies the fp32 sum.
 *   INT4: y = x deq^T with deq = (q - z) * s of each 128-group; (q - z) is
 *         formed exactly in bf16 and s multiplies each group's fp32 sum.
 * Rounding: fp32 accumulation (tensor-core MMA), one fp32 -> bf16 RNE at the
 * output. Summation order is fixed for a given (shape, device), so results
 * are reproducible run to run.
 *
 * x: bf16 [m][k] row-major (device); y: bf16 [m][n] row-major (device).
 * Requirements: 1 <= m <= 65536, n >= 1, k >= 0; k % 8 == 0 (BF16),
 * k % 16 == 0 (FP8), k % 128 == 0 (INT4); pointers 16-byte aligned.
 * m == 0 or n == 0 is a no-op; k == 0 writes zeros.
 * Workspace: may be NULL when dq_gemm_workspace_bytes reports 0.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status dq_gemm_workspace_bytes(const dqd_weight* w, int64_t m, size_t* bytes);

DQD_API dqd_status dq_gemm(const dqd_weight* w, const uint16_t* x_bf16, int64_t m,
                   uint16_t* y_bf16, void* workspace, size_t ws_bytes,
                   dqd_stream stream);

/* ------------------------------------------------------------------------
 * gqa_decode_attn — paged GQA decode / speculative-verify attention.
 *
 * Sources: [CS10 §2.2] the new tokens' K,V are appended to the cache, then
 * each new token's query attends to all cached K,V; [LIF §2.1]
 * softmax(q K^T / sqrt(d)) V; [LIF §2.3] Hq query heads share Hkv KV heads;
 * [LIF §3.1, CS10 §7.3] KV stored in 16-token blocks addressed through a
 * block table; [MTC, section "注意力 Kernel"] split K/V into chunks processed
 * in parallel, then combine (Flash-Decoding), exact online softmax
 * (FlashAttention); [ATC, Algorithm 1] verify positions form one causal
 * forward: later draft tokens cannot affect earlier ones.
 *
 * For sequence b, verify position i (0 <= i < w) and query head h:
 *   kv head  g   = h / (hq / hkv)
 *   position p   = context_lens[b] - w + i
 *   out[b][i][h] = sum_{j<=p} softmax_j(softmax_scale * q[b][i][h] . K_j) V_j
 * where K_j, V_j are row (j % 16) of physical block block_table[b][j / 16],
 * kv head g.
 *
 * q:            bf16 [b][w][hq][d]              (device)
 * k_pool,v_pool:bf16 [num_blocks][hkv][16][d]   (device)
 * block_table:  int32 [b][max_blocks_per_seq]   (device)
 * context_lens: int32 [b]                        (device); includes the w new
 *               tokens, so w <= context_lens[b] <= max_context is required
 * max_context:  host upper bound of context_lens (plans the split)
 * out:          bf16 [b][w][hq][d]              (device)
 * Requirements: d == 128, 1 <= w <= 16, hq % hkv == 0, 1 <= b,
 * max_context <= 16 * max_blocks_per_seq, num_blocks >= 1.
 * Inputs the host cannot check are clamped on the device, so that no memory
 * outside the pool is read, and reported through DQD_DEVICE_ERR_BAD_INPUT
 * (dqd_device_errors); the output of such a call is not meaningful:
 *  - a block-table entry outside [0, num_blocks) is clamped into range;
 *  - a context_lens[b] above max_context is taken as max_context;
 *  - a query row that sees no key (context_lens[b] < w) is written as zeros.
 * Workspace (size from gqa_decode_attn_workspace_bytes for the same b, w, hq,
 * hkv, d, max_context on the same device): the split-KV partials and, for
 * 17-128 query rows per kv head, the pieces of a balanced last wave, the
 * order of the sequences, and a work queue in the counter region when there
 * are more work units than SMs; so it can be needed with a single split.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status gqa_decode_attn_workspace_bytes(int32_t b, int32_t w, int32_t hq,
                                           int32_t hkv, int32_t d,
                                           int32_t max_context, size_t* bytes);

DQD_API dqd_status gqa_decode_attn(const uint16_t* q, const uint16_t* k_pool,
                           const uint16_t* v_pool, int64_t num_blocks,
                           const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t max_context,
                           int32_t b, int32_t w, int32_t hq, int32_t hkv, int32_t d,
                           float softmax_scale, uint16_t* out, void* workspace,
                           size_t ws_bytes, dqd_stream stream);

/* ------------------------------------------------------------------------
 * gqa_decode_attn_fp8kv — gqa_decode_attn over an FP8-E4M3 KV cache.
 *
 * Sources: [LIF §4.2 C, KV-cache quantisation] K/V cached as FP8 halve the
 * cache bytes and are close to lossless; [MTC, speculative-decoding
 * exercises] the step bound with an idealised 1-byte FP8 KV. The pages leave
 * the scale factors open; here each pool has one fp32 scale:
 *   K_j = e4m3(k_pool code) * k_scale,  V_j = e4m3(v_pool code) * v_scale
 * and the result is gqa_decode_attn's formula on those K_j, V_j.
 *
 * k_pool,v_pool: uint8 E4M3 codes [num_blocks][hkv][16][d]  (device); the
 *               NaN codes 0x7F and 0xFF must not occur (the kernel reads
 *               them as +-480)
 * k_scale, v_scale: finite host floats (0 allowed)
 * The products are taken in f16 (every E4M3 value is an f16 value): q is
 * converted to f16, so |q| <= 65504 is required (entries below 2^-14 keep an
 * absolute error <= 2^-25), and the softmax weights enter P V as f16.
 * Every other argument, the layouts, requirements and results are those of
 * gqa_decode_attn; the workspace size comes from
 * gqa_decode_attn_fp8kv_workspace_bytes.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status gqa_decode_attn_fp8kv_workspace_bytes(int32_t b, int32_t w, int32_t hq,
                                                 int32_t hkv, int32_t d,
                                                 int32_t max_context, size_t* bytes);

DQD_API dqd_status gqa_decode_attn_fp8kv(const uint16_t* q, const uint8_t* k_pool,
                                 const uint8_t* v_pool, int64_t num_blocks,
                                 const int32_t* block_table, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, int32_t max_context,
                                 int32_t b, int32_t w, int32_t hq, int32_t hkv, int32_t d,
                                 float softmax_scale, float k_scale, float v_scale,
                                 uint16_t* out, void* workspace, size_t ws_bytes,
                                 dqd_stream stream);

/* ------------------------------------------------------------------------
 * gqa_decode_attn_static_ws — gqa_decode_attn without a caller workspace.
 *
 * The pages have no counterpart to this entry point: it is an interface for
 * callers that cannot allocate device memory. Examples are a runtime that
 * forbids cudaMalloc once serving has started (an allocation can stall the
 * device or fail under memory pressure) and a plug-in running inside a host
 * process whose memory allocator it does not own. Such callers still own q,
 * the pools, the tables and out; only the split-KV scratch changes hands.
 *
 * Arguments, layouts and results are those of gqa_decode_attn. The scratch
 * is a fixed 32 MiB array inside the library (a static device variable). A
 * call that needs more than that (b * w * hq * chunks * 520 bytes, plus
 * 64 KiB) returns DQD_ERR_WORKSPACE with a message and launches nothing; use
 * gqa_decode_attn with a caller workspace instead.
 *
 * Set-up, once per device: the first call that needs scratch in a CUDA
 * context looks up the array's device address there (with that device
 * current) and caches it under the context's id. Because CUDA loads a
 * library's kernels on a device lazily, that first call (like the first
 * call of any entry point of the attention module) may load them, and
 * loading reserves the 32 MiB array and the kernel code on the device: an
 * allocation made by the driver, which can fail under memory pressure. Make
 * that first call at start-up, before serving and before any CUDA stream
 * capture; from then on the GPU holds the array until the process exits, and
 * later calls allocate nothing and call no allocating routine. After a device
 * reset the new context makes its own first call.
 *
 * All calls on a device share the one scratch array, which keeps whatever the
 * previous call left in it; each call writes the partial results it reads,
 * so nothing has to start at zero. Calls whose executions overlap on the GPU
 * (different streams, or different host threads) race on the scratch and
 * give wrong results: serialise them, e.g. on a single stream.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status gqa_decode_attn_static_ws(const uint16_t* q, const uint16_t* k_pool,
                                     const uint16_t* v_pool, int64_t num_blocks,
                                     const int32_t* block_table, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t max_context,
                                     int32_t b, int32_t w, int32_t hq, int32_t hkv, int32_t d,
                                     float softmax_scale, uint16_t* out, dqd_stream stream);

/* ------------------------------------------------------------------------
 * rope_kv_append — rotary embedding of the new tokens' q and k, and the
 * append of their k and v to the paged KV cache (the step between the QKV
 * projection and the attention).
 *
 * Source: [CS10 §2.2-2.3] for each new token compute q, k, v; rotate q and k
 * at the token's global position (not from 0); write k and v into the cache
 * at those positions; then attend. Rotary form (the pages do not fix one;
 * reading: the pairwise form): dims (2i, 2i+1) of every q and k head turn by
 * angle pos * base^(-2i/d):
 *   [x_2i', x_2i+1'] = [x_2i cos - x_2i+1 sin, x_2i sin + x_2i+1 cos].
 * (A checkpoint in the half-split form is brought to it by permuting the
 * rows of its q and k projections.)
 * Token (r, i), r < b, i < w, reads row r*w + i of qkv and sits at position
 * pos = context_lens[r] - w + i (the cache already counts the w new tokens,
 * as gqa_decode_attn expects). q_out[r][i][h] = rotated q head h (bf16 RNE of
 * the binary32 rotation); k head g (rotated) and v head g (unchanged) go to
 * row pos % 16 of kv head g of block block_table[r][pos / 16]. A position
 * below 0 or past the table appends nothing; table entries outside
 * [0, num_blocks) are clamped into range and reported through
 * DQD_DEVICE_ERR_BAD_INPUT (dqd_device_errors).
 * kv_fp8 = 0: bf16 pools (v is copied bit for bit). kv_fp8 = 1: E4M3 pools as
 * in gqa_decode_attn_fp8kv: code = e4m3_RNE_satfinite(binary32(x / scale)).
 * The angle pos * base^(-2i/d) is reduced exactly in turns: each frequency
 * over 2 pi is held as a 64-bit fixed-point fraction (computed in double on
 * the host), pos times it modulo 2^64 is the angle's fraction of a turn; sin
 * and cos of it, and the rotation, are taken in binary32.
 *
 * qkv: bf16 [b*w][(hq + 2*hkv) * d], heads ordered q_0.., k_0.., v_0..
 * (device); q_out: bf16 [b][w][hq][d] (device); pools: [num_blocks][hkv][16][d]
 * bf16 or u8 (device); block_table, context_lens as in gqa_decode_attn.
 * Requirements: b, w, hq, hkv >= 1; d even, 2 <= d <= 512; rope_base > 1;
 * qkv, q_out and pools 16-byte aligned; int32 arrays 4-byte aligned.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status rope_kv_append(const uint16_t* qkv, int32_t b, int32_t w, int32_t hq,
                          int32_t hkv, int32_t d, float rope_base,
                          const int32_t* block_table, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, int64_t num_blocks, void* k_pool,
                          void* v_pool, int32_t kv_fp8, float k_scale, float v_scale,
                          uint16_t* q_out, dqd_stream stream);

/* ------------------------------------------------------------------------
 * dq_gemm_qkv_rope_append — the QKV projection of the new tokens fused with
 * rope_kv_append: the step from a layer's input to the attention's q and
 * cache in one launch.
 *
 * Source: [CS10 §2.2-2.3] for each new token compute q, k, v (the QKV
 * projection), rotate q and k at the token's global position, write k and v
 * into the cache, then attend; [MTC, section "量化省下什麼"] the projection is
 * the dequantising GEMM (BF16, FP8-E4M3 or INT4 g128 weights).
 *
 * Result: exactly (bit for bit) what
 *   dq_gemm(w, x, b*wv, qkv)  followed by
 *   rope_kv_append(qkv, b, wv, hq, hkv, 128, rope_base, ...)
 * produce, without qkv: each bf16 output of the projection's epilogue is
 * rotated with its pair (columns 2i, 2i+1 of a q or k head) and stored into
 * q_out, the K pool or the V pool (positions, slots, FP8 encoding and the
 * handling of out-of-range table entries as in rope_kv_append).
 *
 * w:     the QKV weight [(hq + 2*hkv) * 128 out][k in], rows ordered
 *        q_0.., k_0.., v_0.. (any dqd_wtype, layout as in dq_gemm)
 * x_bf16:bf16 [b*wv][k] (device): row r*wv + i is token i of sequence r
 * d:     head dimension, must be 128
 * other arguments: as in rope_kv_append (w there is wv here)
 * workspace: as dq_gemm's for (w, m = b*wv): dq_gemm_workspace_bytes gives
 *        its size; counters left at zero, as dq_gemm leaves them.
 * Requirements: those of dq_gemm and rope_kv_append, d == 128,
 * b*wv <= 65536, x, q_out and the pools 16-byte aligned.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status dq_gemm_qkv_rope_append(const dqd_weight* w, const uint16_t* x_bf16, int32_t b,
                                   int32_t wv, int32_t hq, int32_t hkv, int32_t d,
                                   float rope_base, const int32_t* block_table,
                                   int32_t max_blocks_per_seq, const int32_t* context_lens,
                                   int64_t num_blocks, void* k_pool, void* v_pool,
                                   int32_t kv_fp8, float k_scale, float v_scale,
                                   uint16_t* q_out, void* workspace, size_t ws_bytes,
                                   dqd_stream stream);

/* ------------------------------------------------------------------------
 * spec_verify_greedy — greedy verify of a speculative draft block, with
 * KV-tail invalidation (the step right after the target's verify forward).
 *
 * Source: [ATC, Algorithm 1 "贪心验证及状态回退" (greedy verify and state
 * rollback)]: compare each draft with the target's greedy prediction from
 * the first position, stop at the first mismatch, keep the matched prefix,
 * add the target's token (the correction, or the extra token when every
 * draft matched), invalidate the KV behind the accepted boundary; the
 * correction token is the next round's input.
 * Per request r, with verify width w = k + 1 (position 0 is the round's input
 * token, positions 1..k the drafts d_1..d_k):
 *   t_i       = argmax_v logits[r][i][v]   (ties: the smallest token id)
 *   a         = number of leading i with d_{i+1} == t_i   (0 <= a <= k)
 *   out[r][i] = t_i for every i; the round emits out[r][0 .. a]
 *   count[r]  = a + 1
 *   context_lens[r] -= k - a     (when context_lens is not NULL: the w verify
 *                                 tokens sit at the end of the cache; the
 *                                 rejected drafts' KV becomes invalid)
 * A draft id outside [0, vocab) never matches.
 *
 * logits_bf16: [b][w][vocab] (device), not NaN; draft: int32 [b][w-1]
 * (device; may be NULL when w == 1); out_tokens: int32 [b][w] (device);
 * out_count: int32 [b] (device); context_lens: int32 [b] (device, in/out)
 * or NULL.
 * Requirements: b >= 1, 1 <= w <= 1024, 1 <= vocab < 2^31, logits 16-byte
 * aligned, int32 buffers 4-byte aligned.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status spec_verify_greedy(const uint16_t* logits_bf16, int32_t b, int32_t w,
                              int64_t vocab, const int32_t* draft, int32_t* out_tokens,
                              int32_t* out_count, int32_t* context_lens, dqd_stream stream);

/* ------------------------------------------------------------------------
 * spec_verify_sample — speculative sampling accept / resample.
 *
 * Source: [CS10 §6 "推测采样" (speculative sampling)]: draft token x is
 * accepted with probability min(1, q(x)/p(x)); at the first rejection one
 * token is drawn from norm(max(q - p, 0)) and the rest of the draft is
 * dropped; when all k drafts are accepted one more token is drawn from the
 * target's distribution at position k+1. The output is then distributed
 * exactly as the target's q.
 * The random numbers are inputs: draft i is accepted iff
 * u_accept[r][i] * p(x) < q(x) (binary32); the one drawn token is the smallest
 * y with sum_{z<=y} r(z) > u_sample[r] * sum_z r(z) (sums in double), with
 * r = max(q - p, 0) (binary32 difference) after a rejection and r = q for the
 * extra token; a residual that sums to 0 (through rounding only) falls back
 * to q. out_tokens[r][0 .. j-1] = accepted drafts, out_tokens[r][j] = drawn
 * token, count[r] = j + 1, context_lens[r] -= k - j.
 *
 * p_draft: f32 [b][k][vocab]; q_target: f32 [b][k+1][vocab]; draft: int32
 * [b][k]; u_accept: f32 [b][k] in [0, 1); u_sample: f32 [b] in [0, 1) (all
 * device). out_tokens: int32 [b][k+1]; out_count: int32 [b]; context_lens as
 * above. Requirements: b >= 1, 0 <= k <= 1023, 1 <= vocab < 2^31; p, q
 * non-negative and finite; 4-byte aligned pointers.
 * ---------------------------------------------------------------------- */
DQD_API dqd_status spec_verify_sample(const float* p_draft, const float* q_target,
                              const int32_t* draft, const float* u_accept,
                              const float* u_sample, int32_t b, int32_t k, int64_t vocab,
                              int32_t* out_tokens, int32_t* out_count,
                              int32_t* context_lens, dqd_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* DQD_H_ */
