// Host-side TMA tensor-map encoding shared by the kernels that use tensor
// copies. The driver's encoder is reached through the runtime's driver entry
// point, so the library does not link the driver API.
#include "dqd_internal.h"

#include <cstring>
#include <mutex>

namespace dqd {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

struct Key {
  const void* base;
  int dtype, rank, swizzle;
  uint64_t dims[5], strides[4];
  uint32_t box[5];
  bool operator==(const Key& o) const { return std::memcmp(this, &o, sizeof(Key)) == 0; }
};

}  // namespace

cudaError_t tensor_map(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle) {
  static std::mutex mu;
  static Key keys[32];
  static CUtensorMap maps[32];
  static int used = 0, next = 0;
  Key key;
  std::memset(&key, 0, sizeof key);
  key.base = base;
  key.dtype = (int)dtype;
  key.rank = rank;
  key.swizzle = (int)swizzle;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides_bytes[i];
  }
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
      if (keys[i] == key) {
        *out = maps[i];
        return cudaSuccess;
      }
  }
  EncodeTiledFn fn = encoder();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], el[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    el[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUtensorMap m;
  std::memset(&m, 0, sizeof m);
  const CUresult r = fn(&m, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, el,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lk(mu);
  keys[next] = key;
  maps[next] = m;
  next = (next + 1) % 32;
  used = used < 32 ? used + 1 : 32;
  *out = m;
  return cudaSuccess;
}

}  // namespace dqd
