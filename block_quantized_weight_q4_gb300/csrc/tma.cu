// tma.cu -- host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled, obtained from the
// driver through the runtime's entry-point query, so the library links no libcuda).
#include <mutex>

#include <cudaTypedefs.h>

#include "qmv_internal.h"

namespace qmv {

namespace {
std::once_flag g_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess) {
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
}
}  // namespace

cudaError_t encode_tmap_2d(CUtensorMap* map, int dtype, const void* base, uint64_t inner_elems, uint64_t outer,
                           uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle) {
  std::call_once(g_once, resolve);
  if (g_encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {inner_elems, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, static_cast<CUtensorMapDataType>(dtype), 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              static_cast<CUtensorMapSwizzle>(swizzle), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace qmv
