// Host-side encoding of TMA tensor maps (bf16, 4-D, 128-byte swizzle) for the
// tcgen05 kernels. The driver entry point is looked up once per process
// through the runtime, so the library needs no link against the driver API.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace jt {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 4-D bf16 map, dims innermost first, 128-byte swizzle.
inline bool make_map(CUtensorMap* m, const void* base, const uint64_t (&dims)[4],
              const uint32_t (&box)[4]) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t gd[4], gs[3];
  cuuint32_t bx[4], es[4] = {1, 1, 1, 1};
  for (int i = 0; i < 4; ++i) { gd[i] = dims[i] ? dims[i] : 1; bx[i] = box[i]; }
  gs[0] = gd[0] * 2;
  gs[1] = gs[0] * gd[1];
  gs[2] = gs[1] * gd[2];
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gd, gs, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace jt
