// tmap.cu -- the one place that builds TMA tensor maps (cuTensorMapEncodeTiled, reached through
// the runtime's driver entry-point query, so the library links no driver stub).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "internal.h"

namespace da {

static PFN_cuTensorMapEncodeTiled_v12000 encode_entry() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult res;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &res) == cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tmap_4d(CUtensorMap* m, CUtensorMapDataType type, const void* base,
                    const cuuint64_t (&dims)[4], const cuuint64_t (&byte_strides)[3],
                    const cuuint32_t (&box)[4], char* err, size_t err_len) {
  auto fn = encode_entry();
  if (!fn) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled entry point unavailable");
    return false;
  }
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, type, 4, const_cast<void*>(base), dims, byte_strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return false;
  }
  return true;
}

}  // namespace da
