// Host side of the TMA loads: cuTensorMapEncodeTiled reached through the
// runtime's driver entry point (no link against the driver library).
#pragma once

#include <cuda.h>   // CUtensorMap and its enums
#include <cuda_runtime.h>

namespace csa2 {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once; the initialisation of a function-local static is
// thread-safe, so concurrent first calls all see the finished lookup.
inline EncodeTiled encode_tiled() {
  static const EncodeTiled fn = []() -> EncodeTiled {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult res;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &res) == cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiled>(p);
    return nullptr;
  }();
  return fn;
}

}  // namespace csa2
