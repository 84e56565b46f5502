// C-ABI layer of libdqd: argument checks, planning and launches. Every check
// that can be made on the host is made before anything is enqueued.
#include "../../include/dqd.h"
#include "dqd_internal.h"

#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <string>

static_assert(DQD_WS_COUNTER_BYTES == dqd::kCounterBytes, "counter region size mismatch");

namespace {

thread_local std::string g_last_error;

dqd_status fail(dqd_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

dqd_status ok() { return DQD_OK; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device, cached per device.
dqd_status sm_count(int* out) {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DQD_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64) {
    int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return DQD_OK;
    }
  }
  int c = 0;
  e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(DQD_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64) cache[dev].store(c, std::memory_order_relaxed);
  *out = c;
  return DQD_OK;
}

dqd_status check_launch(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(DQD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return DQD_OK;
}

dqd_status check_weight(const dqd_weight* w) {
  if (!w) return fail(DQD_ERR_INVALID_ARG, "weight descriptor is NULL");
  if (w->n < 0 || w->k < 0) return fail(DQD_ERR_INVALID_ARG, "negative weight shape");
  if (w->n > (int64_t)1 << 31 || w->k > (int64_t)1 << 31)
    return fail(DQD_ERR_UNSUPPORTED, "weight dimension above 2^31");
  switch (w->type) {
    case DQD_W_BF16:
      if (w->k % 8) return fail(DQD_ERR_INVALID_ARG, "BF16 weights need k %% 8 == 0 (k=%lld)", (long long)w->k);
      break;
    case DQD_W_FP8_E4M3:
      if (w->k % 16) return fail(DQD_ERR_INVALID_ARG, "FP8 weights need k %% 16 == 0 (k=%lld)", (long long)w->k);
      if (w->n > 0 && (!w->scales || !aligned16(w->scales)))
        return fail(DQD_ERR_INVALID_ARG, "FP8 weights need 16-byte aligned fp32 row scales");
      break;
    case DQD_W_INT4_G128:
      if (w->k % 128) return fail(DQD_ERR_INVALID_ARG, "INT4 g128 weights need k %% 128 == 0 (k=%lld)", (long long)w->k);
      if (w->n > 0 && w->k > 0 &&
          (!w->scales || !w->zeros || !aligned16(w->scales) || !aligned16(w->zeros)))
        return fail(DQD_ERR_INVALID_ARG, "INT4 weights need 16-byte aligned packed scales and zeros");
      break;
    default:
      return fail(DQD_ERR_INVALID_ARG, "unknown weight type %d", (int)w->type);
  }
  if (w->n > 0 && w->k > 0 && (!w->data || !aligned16(w->data)))
    return fail(DQD_ERR_INVALID_ARG, "weight data must be a 16-byte aligned device pointer");
  return DQD_OK;
}

}  // namespace

extern "C" {

const char* dqd_status_string(dqd_status s) {
  switch (s) {
    case DQD_OK: return "DQD_OK";
    case DQD_ERR_INVALID_ARG: return "DQD_ERR_INVALID_ARG";
    case DQD_ERR_UNSUPPORTED: return "DQD_ERR_UNSUPPORTED";
    case DQD_ERR_WORKSPACE: return "DQD_ERR_WORKSPACE";
    case DQD_ERR_CUDA: return "DQD_ERR_CUDA";
  }
  return "DQD_ERR_UNKNOWN";
}

const char* dqd_last_error(void) { return g_last_error.c_str(); }

const char* dqd_version(void) { return "dqd 0.1 sm_103a"; }

dqd_status dqd_device_errors(uint32_t* flags) {
  g_last_error.clear();
  if (!flags) return fail(DQD_ERR_INVALID_ARG, "flags is NULL");
  *flags = 0;
  cudaError_t e = dqd::attn_take_device_error(flags);
  if (e == cudaSuccess) e = dqd::gemm_take_device_error(flags);
  if (e == cudaSuccess) e = dqd::rope_take_device_error(flags);
  if (e == cudaSuccess) e = dqd::selftest_take_device_error(flags);
  if (e != cudaSuccess) return fail(DQD_ERR_CUDA, "reading the device error words: %s", cudaGetErrorString(e));
  return DQD_OK;
}

dqd_status dqd_selftest_wait_timeout(uint32_t polls, dqd_stream stream) {
  g_last_error.clear();
  if (polls < 1 || polls > (1u << 22)) return fail(DQD_ERR_INVALID_ARG, "polls must be in [1, 2^22]");
  return check_launch(dqd::launch_selftest_wait(polls, reinterpret_cast<cudaStream_t>(stream)),
                      "dqd_selftest_wait_timeout launch");
}

size_t pack_int4_g128_bytes(int64_t n, int64_t k, int which) {
  if (n < 1 || k < 128 || k % 128) return 0;
  const size_t blocks = (size_t)((n + 15) / 16) * (size_t)(k / 128);
  switch (which) {
    case 0: return blocks * 1024;
    case 1: return blocks * 32;
    case 2: return blocks * 8;
  }
  return 0;
}

dqd_status pack_int4_g128(const uint8_t* codes, const uint16_t* scales_bf16, const uint8_t* zeros,
                          int64_t n, int64_t k, void* packed, void* packed_scales,
                          void* packed_zeros, dqd_stream stream) {
  g_last_error.clear();
  if (n < 1 || k < 128 || k % 128)
    return fail(DQD_ERR_INVALID_ARG, "pack_int4_g128 needs n >= 1, k >= 128, k %% 128 == 0 (n=%lld k=%lld)",
                (long long)n, (long long)k);
  if (n > (int64_t)1 << 31 || k > (int64_t)1 << 31) return fail(DQD_ERR_UNSUPPORTED, "dimension above 2^31");
  const void* ptrs[] = {codes, scales_bf16, zeros, packed, packed_scales, packed_zeros};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(DQD_ERR_INVALID_ARG, "pack_int4_g128: NULL or misaligned pointer");
  return check_launch(dqd::launch_pack_int4(codes, scales_bf16, zeros, n, k, packed, packed_scales,
                                            packed_zeros, reinterpret_cast<cudaStream_t>(stream)),
                      "pack_int4_g128 launch");
}

dqd_status quant_fp8_rowwise(const uint16_t* w_bf16, int64_t n, int64_t k, uint8_t* codes,
                             float* scales, dqd_stream stream) {
  g_last_error.clear();
  if (n < 1 || k < 1 || k % 16)
    return fail(DQD_ERR_INVALID_ARG, "quant_fp8_rowwise needs n >= 1, k >= 1, k %% 16 == 0 (n=%lld k=%lld)",
                (long long)n, (long long)k);
  if (n > ((int64_t)1 << 31) - 1 || k > ((int64_t)1 << 31)) return fail(DQD_ERR_UNSUPPORTED, "dimension above 2^31");
  if (!w_bf16 || !codes || !scales || !aligned16(w_bf16) || !aligned16(codes) || !aligned16(scales))
    return fail(DQD_ERR_INVALID_ARG, "quant_fp8_rowwise: NULL or misaligned pointer");
  return check_launch(dqd::launch_quant_fp8(w_bf16, n, k, codes, scales,
                                            reinterpret_cast<cudaStream_t>(stream)),
                      "quant_fp8_rowwise launch");
}

dqd_status quant_int4_g128(const uint16_t* w_bf16, int64_t n, int64_t k, uint8_t* codes,
                           uint16_t* scales_bf16, uint8_t* zeros, dqd_stream stream) {
  g_last_error.clear();
  if (n < 1 || k < 128 || k % 128)
    return fail(DQD_ERR_INVALID_ARG, "quant_int4_g128 needs n >= 1, k >= 128, k %% 128 == 0 (n=%lld k=%lld)",
                (long long)n, (long long)k);
  if (n > ((int64_t)1 << 31) - 1 || k > ((int64_t)1 << 31) || n * (k / 128) > ((int64_t)1 << 36))
    return fail(DQD_ERR_UNSUPPORTED, "quant_int4_g128: dimension too large");
  if (!w_bf16 || !codes || !scales_bf16 || !zeros || !aligned16(w_bf16) || !aligned16(codes) ||
      !aligned16(scales_bf16) || !aligned16(zeros))
    return fail(DQD_ERR_INVALID_ARG, "quant_int4_g128: NULL or misaligned pointer");
  return check_launch(dqd::launch_quant_int4(w_bf16, n, k, codes, scales_bf16, zeros,
                                             reinterpret_cast<cudaStream_t>(stream)),
                      "quant_int4_g128 launch");
}

static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

dqd_status rope_kv_append(const uint16_t* qkv, int32_t b, int32_t w, int32_t hq, int32_t hkv, int32_t d,
                          float rope_base, const int32_t* block_table, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, int64_t num_blocks, void* k_pool, void* v_pool,
                          int32_t kv_fp8, float k_scale, float v_scale, uint16_t* q_out, dqd_stream stream) {
  g_last_error.clear();
  if (b < 1 || w < 1 || hq < 1 || hkv < 1 || d < 2 || d > 512 || d % 2 || num_blocks < 1 ||
      max_blocks_per_seq < 1)
    return fail(DQD_ERR_INVALID_ARG, "rope_kv_append needs b, w, hq, hkv >= 1, even d in [2, 512], "
                                     "num_blocks >= 1, max_blocks_per_seq >= 1");
  if ((int64_t)b * w > INT32_MAX || (int64_t)(hq + 2 * (int64_t)hkv) * (d / 2) > ((int64_t)1 << 24))
    return fail(DQD_ERR_UNSUPPORTED, "rope_kv_append: b * w or the head count too large");
  if (!(rope_base > 1.f) || rope_base == INFINITY) return fail(DQD_ERR_INVALID_ARG, "rope_base must be finite and > 1");
  if (kv_fp8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY))
    return fail(DQD_ERR_INVALID_ARG, "an FP8 cache needs finite positive k_scale and v_scale");
  const void* p16[] = {qkv, q_out, k_pool, v_pool};
  for (const void* p : p16)
    if (!p || !aligned16(p)) return fail(DQD_ERR_INVALID_ARG, "rope_kv_append: NULL or misaligned pointer");
  if (!block_table || !context_lens || !aligned4(block_table) || !aligned4(context_lens))
    return fail(DQD_ERR_INVALID_ARG, "rope_kv_append: NULL or misaligned table or context_lens");
  return check_launch(dqd::launch_rope_kv_append(qkv, b, w, hq, hkv, d, (double)rope_base, block_table,
                                                 max_blocks_per_seq, context_lens, num_blocks, k_pool, v_pool,
                                                 kv_fp8 != 0, k_scale, v_scale, q_out,
                                                 reinterpret_cast<cudaStream_t>(stream)),
                      "rope_kv_append launch");
}

dqd_status spec_verify_greedy(const uint16_t* logits_bf16, int32_t b, int32_t w, int64_t vocab,
                              const int32_t* draft, int32_t* out_tokens, int32_t* out_count,
                              int32_t* context_lens, dqd_stream stream) {
  g_last_error.clear();
  if (b < 1 || w < 1 || w > 1024 || vocab < 1 || vocab > INT32_MAX)
    return fail(DQD_ERR_INVALID_ARG, "spec_verify_greedy needs b >= 1, 1 <= w <= 1024, 1 <= vocab < 2^31");
  if ((int64_t)b * w > INT32_MAX) return fail(DQD_ERR_UNSUPPORTED, "spec_verify_greedy: b * w too large");
  if (!logits_bf16 || !aligned16(logits_bf16) || !out_tokens || !aligned4(out_tokens) || !out_count ||
      !aligned4(out_count) || (w > 1 && (!draft || !aligned4(draft))) || (context_lens && !aligned4(context_lens)))
    return fail(DQD_ERR_INVALID_ARG, "spec_verify_greedy: NULL or misaligned pointer");
  int sms = 0;
  dqd_status st = sm_count(&sms);
  if (st != DQD_OK) return st;
  return check_launch(dqd::launch_spec_verify_greedy(logits_bf16, b, w, vocab, draft, out_tokens, out_count,
                                                     context_lens, sms, reinterpret_cast<cudaStream_t>(stream)),
                      "spec_verify_greedy launch");
}

dqd_status spec_verify_sample(const float* p_draft, const float* q_target, const int32_t* draft,
                              const float* u_accept, const float* u_sample, int32_t b, int32_t k, int64_t vocab,
                              int32_t* out_tokens, int32_t* out_count, int32_t* context_lens,
                              dqd_stream stream) {
  g_last_error.clear();
  if (b < 1 || k < 0 || k > 1023 || vocab < 1 || vocab > INT32_MAX)
    return fail(DQD_ERR_INVALID_ARG, "spec_verify_sample needs b >= 1, 0 <= k <= 1023, 1 <= vocab < 2^31");
  const void* always[] = {q_target, u_sample, out_tokens, out_count};
  for (const void* p : always)
    if (!p || !aligned4(p)) return fail(DQD_ERR_INVALID_ARG, "spec_verify_sample: NULL or misaligned pointer");
  if (k > 0) {
    const void* drafts[] = {p_draft, draft, u_accept};
    for (const void* p : drafts)
      if (!p || !aligned4(p)) return fail(DQD_ERR_INVALID_ARG, "spec_verify_sample: NULL or misaligned pointer");
  }
  if (context_lens && !aligned4(context_lens))
    return fail(DQD_ERR_INVALID_ARG, "spec_verify_sample: misaligned context_lens");
  return check_launch(dqd::launch_spec_verify_sample(p_draft, q_target, draft, u_accept, u_sample, b, k, vocab,
                                                     out_tokens, out_count, context_lens,
                                                     reinterpret_cast<cudaStream_t>(stream)),
                      "spec_verify_sample launch");
}

dqd_status dq_gemm_workspace_bytes(const dqd_weight* w, int64_t m, size_t* bytes) {
  g_last_error.clear();
  if (!bytes) return fail(DQD_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = 0;
  dqd_status st = check_weight(w);
  if (st != DQD_OK) return st;
  if (m < 0 || m > 65536) return fail(DQD_ERR_UNSUPPORTED, "m must be in [0, 65536] (m=%lld)", (long long)m);
  if (m == 0 || w->n == 0) return DQD_OK;
  int sms = 0;
  if ((st = sm_count(&sms)) != DQD_OK) return st;
  *bytes = dqd::plan_dq_gemm(w->type, m, w->n, w->k, sms).ws_bytes;
  return DQD_OK;
}

dqd_status dq_gemm(const dqd_weight* w, const uint16_t* x_bf16, int64_t m, uint16_t* y_bf16,
                   void* workspace, size_t ws_bytes, dqd_stream stream) {
  g_last_error.clear();
  dqd_status st = check_weight(w);
  if (st != DQD_OK) return st;
  if (m < 0 || m > 65536) return fail(DQD_ERR_UNSUPPORTED, "m must be in [0, 65536] (m=%lld)", (long long)m);
  if (m == 0 || w->n == 0) return ok();
  if (!y_bf16 || !aligned16(y_bf16)) return fail(DQD_ERR_INVALID_ARG, "y must be a 16-byte aligned device pointer");
  if (w->k > 0 && (!x_bf16 || !aligned16(x_bf16)))
    return fail(DQD_ERR_INVALID_ARG, "x must be a 16-byte aligned device pointer");
  int sms = 0;
  if ((st = sm_count(&sms)) != DQD_OK) return st;
  const dqd::GemmPlan plan = dqd::plan_dq_gemm(w->type, m, w->n, w->k, sms);
  if (plan.ws_bytes > 0) {
    if (!workspace || !aligned16(workspace))
      return fail(DQD_ERR_WORKSPACE, "dq_gemm needs a 16-byte aligned workspace of %zu bytes", plan.ws_bytes);
    if (ws_bytes < plan.ws_bytes)
      return fail(DQD_ERR_WORKSPACE, "dq_gemm workspace too small: %zu < %zu bytes", ws_bytes, plan.ws_bytes);
  }
  dqd::GemmLaunch l;
  l.rope = nullptr;
  l.wtype = w->type;
  l.data = w->data;
  l.scales = w->scales;
  l.zeros = w->zeros;
  l.x = x_bf16 ? x_bf16 : y_bf16;  // k == 0: x is never read
  l.y = y_bf16;
  l.m = m;
  l.n = w->n;
  l.k = w->k;
  l.workspace = plan.ws_bytes > 0 ? workspace : nullptr;
  return check_launch(dqd::launch_dq_gemm(l, plan, reinterpret_cast<cudaStream_t>(stream)),
                      "dq_gemm launch");
}

dqd_status dq_gemm_qkv_rope_append(const dqd_weight* w, const uint16_t* x_bf16, int32_t b, int32_t wv,
                                   int32_t hq, int32_t hkv, int32_t d, float rope_base,
                                   const int32_t* block_table, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int64_t num_blocks, void* k_pool, void* v_pool,
                                   int32_t kv_fp8, float k_scale, float v_scale, uint16_t* q_out,
                                   void* workspace, size_t ws_bytes, dqd_stream stream) {
  g_last_error.clear();
  dqd_status st = check_weight(w);
  if (st != DQD_OK) return st;
  if (b < 1 || wv < 1 || hq < 1 || hkv < 1 || num_blocks < 1 || max_blocks_per_seq < 1)
    return fail(DQD_ERR_INVALID_ARG, "dq_gemm_qkv_rope_append needs b, w, hq, hkv, num_blocks, "
                                     "max_blocks_per_seq >= 1");
  if (d != 128) return fail(DQD_ERR_UNSUPPORTED, "dq_gemm_qkv_rope_append: head_dim must be 128 (d=%d)", d);
  const int64_t m = (int64_t)b * wv;
  if (m > 65536) return fail(DQD_ERR_UNSUPPORTED, "dq_gemm_qkv_rope_append: b * w must be <= 65536");
  if (w->n != ((int64_t)hq + 2 * (int64_t)hkv) * d)
    return fail(DQD_ERR_INVALID_ARG, "dq_gemm_qkv_rope_append: W has %lld rows, (hq + 2 hkv) * d = %lld",
                (long long)w->n, ((long long)hq + 2LL * hkv) * d);
  if (w->k < 1) return fail(DQD_ERR_INVALID_ARG, "dq_gemm_qkv_rope_append needs k >= 1");
  if (!(rope_base > 1.f) || rope_base == INFINITY) return fail(DQD_ERR_INVALID_ARG, "rope_base must be finite and > 1");
  if (kv_fp8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY))
    return fail(DQD_ERR_INVALID_ARG, "an FP8 cache needs finite positive k_scale and v_scale");
  const void* p16[] = {x_bf16, q_out, k_pool, v_pool};
  for (const void* p : p16)
    if (!p || !aligned16(p)) return fail(DQD_ERR_INVALID_ARG, "dq_gemm_qkv_rope_append: NULL or misaligned pointer");
  if (!block_table || !context_lens || !aligned4(block_table) || !aligned4(context_lens))
    return fail(DQD_ERR_INVALID_ARG, "dq_gemm_qkv_rope_append: NULL or misaligned table or context_lens");
  int sms = 0;
  if ((st = sm_count(&sms)) != DQD_OK) return st;
  const dqd::GemmPlan plan = dqd::plan_dq_gemm(w->type, m, w->n, w->k, sms);
  if (plan.ws_bytes > 0) {
    if (!workspace || !aligned16(workspace))
      return fail(DQD_ERR_WORKSPACE, "dq_gemm_qkv_rope_append needs a 16-byte aligned workspace of %zu bytes",
                  plan.ws_bytes);
    if (ws_bytes < plan.ws_bytes)
      return fail(DQD_ERR_WORKSPACE, "dq_gemm_qkv_rope_append workspace too small: %zu < %zu bytes", ws_bytes,
                  plan.ws_bytes);
  }
  dqd::RopeEpi r;
  dqd::rope_turns((double)rope_base, d, d / 2, r.turns);
  r.table = block_table;
  r.ctx = context_lens;
  r.k_pool = k_pool;
  r.v_pool = v_pool;
  r.q_out = q_out;
  r.num_blocks = num_blocks;
  r.max_blocks = max_blocks_per_seq;
  r.w = wv;
  r.hq = hq;
  r.hkv = hkv;
  r.kv_fp8 = kv_fp8 ? 1 : 0;
  r.k_scale = k_scale;
  r.v_scale = v_scale;
  dqd::GemmLaunch l;
  l.rope = &r;
  l.wtype = w->type;
  l.data = w->data;
  l.scales = w->scales;
  l.zeros = w->zeros;
  l.x = x_bf16;
  l.y = nullptr;  // never written: the epilogue stores into q_out and the pools
  l.m = m;
  l.n = w->n;
  l.k = w->k;
  l.workspace = plan.ws_bytes > 0 ? workspace : nullptr;
  return check_launch(dqd::launch_dq_gemm(l, plan, reinterpret_cast<cudaStream_t>(stream)),
                      "dq_gemm_qkv_rope_append launch");
}

static dqd_status check_attn_shape(int32_t b, int32_t w, int32_t hq, int32_t hkv, int32_t d,
                                   int32_t max_context) {
  if (b < 1 || w < 1 || hq < 1 || hkv < 1)
    return fail(DQD_ERR_INVALID_ARG, "gqa_decode_attn needs b, w, hq, hkv >= 1");
  if (d != 128) return fail(DQD_ERR_UNSUPPORTED, "head_dim must be 128 (d=%d)", d);
  if (w > 16) return fail(DQD_ERR_UNSUPPORTED, "verify width must be <= 16 (w=%d)", w);
  if (hq % hkv) return fail(DQD_ERR_INVALID_ARG, "hq %% hkv != 0 (hq=%d hkv=%d)", hq, hkv);
  if (max_context < 1) return fail(DQD_ERR_INVALID_ARG, "max_context must be >= 1");
  if ((int64_t)b * hkv > 65535 * 64) return fail(DQD_ERR_UNSUPPORTED, "b * hkv too large");
  return DQD_OK;
}

dqd_status gqa_decode_attn_workspace_bytes(int32_t b, int32_t w, int32_t hq, int32_t hkv,
                                           int32_t d, int32_t max_context, size_t* bytes) {
  g_last_error.clear();
  if (!bytes) return fail(DQD_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = 0;
  dqd_status st = check_attn_shape(b, w, hq, hkv, d, max_context);
  if (st != DQD_OK) return st;
  int sms = 0;
  if ((st = sm_count(&sms)) != DQD_OK) return st;
  *bytes = dqd::plan_attn(b, w, hq, hkv, max_context, sms, false).ws_bytes;
  return DQD_OK;
}

dqd_status gqa_decode_attn_fp8kv_workspace_bytes(int32_t b, int32_t w, int32_t hq, int32_t hkv,
                                                 int32_t d, int32_t max_context, size_t* bytes) {
  g_last_error.clear();
  if (!bytes) return fail(DQD_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = 0;
  dqd_status st = check_attn_shape(b, w, hq, hkv, d, max_context);
  if (st != DQD_OK) return st;
  int sms = 0;
  if ((st = sm_count(&sms)) != DQD_OK) return st;
  *bytes = dqd::plan_attn(b, w, hq, hkv, max_context, sms, true).ws_bytes;
  return DQD_OK;
}

}  // extern "C"

// Argument checks and the plan shared by the attention entry points; fills
// everything in *l but the workspace.
static dqd_status prepare_attn(const uint16_t* q, const void* k_pool, const void* v_pool,
                               int64_t num_blocks, const int32_t* block_table,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               int32_t max_context, int32_t b, int32_t w, int32_t hq, int32_t hkv,
                               int32_t d, float softmax_scale, bool kv_fp8, float k_scale,
                               float v_scale, uint16_t* out, dqd::AttnLaunch* l,
                               dqd::AttnPlan* plan) {
  dqd_status st = check_attn_shape(b, w, hq, hkv, d, max_context);
  if (st != DQD_OK) return st;
  if (num_blocks < 1) return fail(DQD_ERR_INVALID_ARG, "num_blocks must be >= 1");
  if (max_blocks_per_seq < 1 || (int64_t)max_context > 16 * (int64_t)max_blocks_per_seq)
    return fail(DQD_ERR_INVALID_ARG, "max_context (%d) exceeds 16 * max_blocks_per_seq (%d)", max_context,
                max_blocks_per_seq);
  const float scales[] = {softmax_scale, k_scale, v_scale};
  for (float v : scales)
    if (!(v == v) || v == INFINITY || v == -INFINITY)
      return fail(DQD_ERR_INVALID_ARG, "softmax_scale, k_scale and v_scale must be finite");
  const void* ptrs[] = {q, k_pool, v_pool, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(DQD_ERR_INVALID_ARG, "q, pools and out must be 16-byte aligned device pointers");
  if (!block_table || !context_lens || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(DQD_ERR_INVALID_ARG, "block_table and context_lens must be 4-byte aligned device pointers");
  int sms = 0;
  if ((st = sm_count(&sms)) != DQD_OK) return st;
  *plan = dqd::plan_attn(b, w, hq, hkv, max_context, sms, kv_fp8);
  if ((int64_t)b * plan->qgroups > 65535)
    return fail(DQD_ERR_UNSUPPORTED, "b * query groups exceeds the grid limit (b=%d)", b);
  l->q = q;
  l->k_pool = k_pool;
  l->v_pool = v_pool;
  l->num_blocks = num_blocks;
  l->block_table = block_table;
  l->max_blocks = max_blocks_per_seq;
  l->context_lens = context_lens;
  l->max_context = max_context;
  l->b = b;
  l->w = w;
  l->hq = hq;
  l->hkv = hkv;
  l->softmax_scale = softmax_scale;
  l->k_scale = k_scale;
  l->v_scale = v_scale;
  l->out = out;
  l->workspace = nullptr;
  return DQD_OK;
}

static dqd_status attn_with_workspace(const char* who, dqd::AttnLaunch& l, const dqd::AttnPlan& plan,
                                      void* workspace, size_t ws_bytes, dqd_stream stream) {
  if (plan.ws_bytes > 0) {
    if (!workspace || !aligned16(workspace))
      return fail(DQD_ERR_WORKSPACE, "%s needs a 16-byte aligned workspace of %zu bytes", who, plan.ws_bytes);
    if (ws_bytes < plan.ws_bytes)
      return fail(DQD_ERR_WORKSPACE, "%s workspace too small: %zu < %zu bytes", who, ws_bytes, plan.ws_bytes);
    l.workspace = workspace;
  }
  return check_launch(dqd::launch_attn(l, plan, reinterpret_cast<cudaStream_t>(stream)), who);
}

extern "C" {

dqd_status gqa_decode_attn(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                           int64_t num_blocks, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t max_context, int32_t b, int32_t w, int32_t hq, int32_t hkv,
                           int32_t d, float softmax_scale, uint16_t* out, void* workspace,
                           size_t ws_bytes, dqd_stream stream) {
  g_last_error.clear();
  dqd::AttnLaunch l;
  dqd::AttnPlan plan;
  dqd_status st = prepare_attn(q, k_pool, v_pool, num_blocks, block_table, max_blocks_per_seq, context_lens,
                               max_context, b, w, hq, hkv, d, softmax_scale, false, 1.f, 1.f, out, &l, &plan);
  if (st != DQD_OK) return st;
  return attn_with_workspace("gqa_decode_attn", l, plan, workspace, ws_bytes, stream);
}

dqd_status gqa_decode_attn_fp8kv(const uint16_t* q, const uint8_t* k_pool, const uint8_t* v_pool,
                                 int64_t num_blocks, const int32_t* block_table,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens,
                                 int32_t max_context, int32_t b, int32_t w, int32_t hq, int32_t hkv,
                                 int32_t d, float softmax_scale, float k_scale, float v_scale,
                                 uint16_t* out, void* workspace, size_t ws_bytes, dqd_stream stream) {
  g_last_error.clear();
  dqd::AttnLaunch l;
  dqd::AttnPlan plan;
  dqd_status st = prepare_attn(q, k_pool, v_pool, num_blocks, block_table, max_blocks_per_seq, context_lens,
                               max_context, b, w, hq, hkv, d, softmax_scale, true, k_scale, v_scale, out, &l,
                               &plan);
  if (st != DQD_OK) return st;
  return attn_with_workspace("gqa_decode_attn_fp8kv", l, plan, workspace, ws_bytes, stream);
}

dqd_status gqa_decode_attn_static_ws(const uint16_t* q, const uint16_t* k_pool,
                                     const uint16_t* v_pool, int64_t num_blocks,
                                     const int32_t* block_table, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t max_context, int32_t b,
                                     int32_t w, int32_t hq, int32_t hkv, int32_t d,
                                     float softmax_scale, uint16_t* out, dqd_stream stream) {
  g_last_error.clear();
  dqd::AttnLaunch l;
  dqd::AttnPlan plan;
  dqd_status st = prepare_attn(q, k_pool, v_pool, num_blocks, block_table, max_blocks_per_seq, context_lens,
                               max_context, b, w, hq, hkv, d, softmax_scale, false, 1.f, 1.f, out, &l, &plan);
  if (st != DQD_OK) return st;
  const size_t cap = dqd::attn_static_scratch_bytes();
  if (plan.ws_bytes > cap)
    return fail(DQD_ERR_WORKSPACE,
                "gqa_decode_attn_static_ws: this call needs %zu bytes of scratch but the library's "
                "static scratch holds %zu; use gqa_decode_attn with a caller workspace",
                plan.ws_bytes, cap);
  if (plan.ws_bytes > 0) {
    cudaError_t e = dqd::attn_static_scratch(&l.workspace);
    if (e != cudaSuccess)
      return fail(DQD_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
  }
  return check_launch(dqd::launch_attn(l, plan, reinterpret_cast<cudaStream_t>(stream)),
                      "gqa_decode_attn_static_ws launch");
}

}  // extern "C"
