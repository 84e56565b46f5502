// Internal interface between the C-ABI layer (dqd_api.cu) and the kernel
// launchers. Host-only declarations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

namespace dqd {

// Launch `kernel` on `stream` with programmatic stream serialisation, so that
// it may begin while the previous kernel on the stream finishes (the kernel
// itself waits for that kernel before touching dependent data).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// As launch_pdl, with CTAs grouped in thread-block clusters of cluster_y CTAs
// along y (grid.y must be a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               unsigned cluster_y, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = cluster_y;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// As launch_pdl, with CTAs grouped in thread-block clusters of cluster_x CTAs
// along x (grid.x must be a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster_x(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

enum WType { kBF16 = 0, kFP8 = 1, kINT4 = 2 };

// Tiled TMA tensor map over `base` (rank <= 5; dims innermost first; strides
// in bytes for dims 1..rank-1), zero fill out of bounds. Encoded maps are
// cached, keyed by every argument.
cudaError_t tensor_map(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle);

constexpr size_t kCounterBytes = 65536;  // = DQD_WS_COUNTER_BYTES

// ---------------------------------------------------------------- dq_gemm --

struct GemmPlan {
  int tc;            // 1: tensor-core (tcgen05) kernel for wide m
  int tc_atm;        // tcgen05: 1 = A (dequantised weights) in tensor memory
  int mt;            // m8 tiles per CTA pass (1, 2, 4, 8)
  int warps;         // warp-MMA kernels: compute warps per CTA (one 16-row tile each)
  int int4_slots;    // INT4 warp-MMA kernel: ring slots (2 or 3)
  int m_chunks;      // ceil(m / (8*mt))
  int grid_x;        // CTAs along n (one 16-row tile per warp)
  int splits;        // CTAs along k
  int cluster;       // 1: the splits of a tile form a thread-block cluster and reduce through DSMEM
  int64_t k_per_split;
  int kc;            // k per pipeline stage
  int ra;            // activation rows staged per CTA (<= 8 * mt)
  int slot_bytes;    // bytes per shared-memory ring slot
  int smem_bytes;    // dynamic shared memory per CTA
  size_t ws_bytes;   // workspace needed (0 if splits == 1)
};

GemmPlan plan_dq_gemm(int wtype, int64_t m, int64_t n, int64_t k, int num_sms);


// The destinations of the QKV projection fused with RoPE and the paged KV
// append (dq_gemm_qkv_rope_append): the rotation frequencies for head dim 128
// and what rope_kv_append takes. Passed by value as a kernel parameter.
struct RopeEpi {
  uint64_t turns[64];     // base^(-2i/128) / 2pi as fractions of 2^64, i < 64
  const int32_t* table;   // [b][max_blocks]
  const int32_t* ctx;     // [b]
  void* k_pool;           // [num_blocks][hkv][16][128] bf16 or E4M3 codes
  void* v_pool;
  uint16_t* q_out;        // [b][w][hq][128] bf16
  int64_t num_blocks;
  int max_blocks, w, hq, hkv;
  int kv_fp8;
  float k_scale, v_scale;
};

// Fixed-point rotation frequencies of RoPE: base^(-2i/d) / 2pi as a fraction
// of 2^64 for i < n (n <= d / 2), computed in double.
void rope_turns(double base, int d, int n, uint64_t* turns);

struct GemmLaunch {
  const RopeEpi* rope;  // non-null: the fused QKV + RoPE + append epilogue
  int wtype;
  const void* data;
  const void* scales;
  const void* zeros;
  const uint16_t* x;
  uint16_t* y;
  int64_t m, n, k;
  void* workspace;
};

cudaError_t launch_dq_gemm(const GemmLaunch& a, const GemmPlan& p, cudaStream_t s);

// tcgen05 path (dq_gemm_tc.cu): whether it takes this shape, its plan, its
// launch, and its device error word.
bool tc_supported(int wtype, int64_t m, int64_t n, int64_t k);
GemmPlan plan_dq_gemm_tc(int wtype, int64_t m, int64_t n, int64_t k, int num_sms);
cudaError_t launch_dq_gemm_tc(const GemmLaunch& a, const GemmPlan& p, cudaStream_t s);
cudaError_t tc_take_device_error(uint32_t* flags);

// OR the GEMM module's device error word into *flags and clear it.
cudaError_t gemm_take_device_error(uint32_t* flags);

// ------------------------------------------------------------ attention --

struct AttnPlan {
  int qt;            // 16-row query tiles per CTA (1, 2, 4)
  int qgroups;       // CTAs needed to cover all query rows of one kv head
  int chunk_blocks;  // 16-token blocks per split-KV chunk
  int nchunks;
  int smem_bytes;
  int kv_fp8;        // 1: FP8-E4M3 cache codes, 0: bf16 cache
  int tc;            // 1: tensor-core (tcgen05) form for wide query tiles
  int tail_items;    // tensor-core form: items of the last partial wave, split ...
  int tail_pieces;   // ... into this many pieces (0: none)
  int persist;       // tensor-core form: > 0 = persistent, with this many CTAs taking units from a queue
  size_t ws_bytes;   // 0 if nchunks == 1 and no tail
};

AttnPlan plan_attn(int b, int w, int hq, int hkv, int max_context, int num_sms, bool kv_fp8);

struct AttnLaunch {
  const uint16_t* q;
  const void* k_pool;  // bf16 or FP8-E4M3 codes, as the plan says
  const void* v_pool;
  int64_t num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* context_lens;
  int max_context;  // the caller's bound on context_lens (the plan covers it)
  int b, w, hq, hkv;
  float softmax_scale;
  float k_scale, v_scale;  // FP8 cache only
  uint16_t* out;
  void* workspace;
};

cudaError_t launch_attn(const AttnLaunch& a, const AttnPlan& p, cudaStream_t s);

// Library-owned attention scratch (a static __device__ array in attn.cu):
// its size, and its device address in the current CUDA context (looked up on
// the first call in each context, cached by context id).
size_t attn_static_scratch_bytes();
cudaError_t attn_static_scratch(void** ptr);

// ORs the attention module's device error word into *flags and clears it.
cudaError_t attn_take_device_error(uint32_t* flags);

// -------------------------------------------------------------- formats --

cudaError_t launch_pack_int4(const uint8_t* codes, const uint16_t* scales, const uint8_t* zeros,
                             int64_t n, int64_t k, void* packed, void* pscales, void* pzeros,
                             cudaStream_t s);

cudaError_t launch_quant_fp8(const uint16_t* w, int64_t n, int64_t k, uint8_t* codes,
                             float* scales, cudaStream_t s);

cudaError_t launch_quant_int4(const uint16_t* w, int64_t n, int64_t k, uint8_t* codes, uint16_t* scales,
                              uint8_t* zeros, cudaStream_t s);

// ------------------------------------------------------ RoPE and append --

// ORs the RoPE/append module's device error word into *flags and clears it.
cudaError_t rope_take_device_error(uint32_t* flags);

cudaError_t launch_rope_kv_append(const uint16_t* qkv, int b, int w, int hq, int hkv, int d, double rope_base,
                                  const int32_t* table, int max_blocks, const int32_t* ctx, int64_t num_blocks,
                                  void* k_pool, void* v_pool, bool kv_fp8, float k_scale, float v_scale,
                                  uint16_t* q_out, cudaStream_t s);

// --------------------------------------------------------------- verify --

cudaError_t launch_spec_verify_greedy(const uint16_t* logits, int b, int w, int64_t vocab, const int32_t* draft,
                                      int32_t* out, int32_t* count, int32_t* ctx, int num_sms, cudaStream_t s);

cudaError_t launch_spec_verify_sample(const float* p, const float* q, const int32_t* draft, const float* u_accept,
                                      const float* u_sample, int b, int k, int64_t vocab, int32_t* out,
                                      int32_t* count, int32_t* ctx, cudaStream_t s);

// ----------------------------------------------------------- diagnostics --

// One bounded wait (polls polls) on an mbarrier nothing completes; it gives
// up, sets the self-test error word and returns.
cudaError_t launch_selftest_wait(uint32_t polls, cudaStream_t s);
cudaError_t selftest_take_device_error(uint32_t* flags);

}  // namespace dqd
