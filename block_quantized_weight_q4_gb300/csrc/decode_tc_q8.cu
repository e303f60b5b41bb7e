// decode_tc_q8.cu -- tensor-memory decode kernels for Q8_0 weights (float16 and float32 scales).
#include "decode_tc.cuh"

namespace qmv {
namespace dtc {

cudaError_t launch_q8(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch, bool xsplit, bool pdl,
                      const DeviceInfo& dev, const Workspace& ws, cudaStream_t stream) {
  return ms[0].scale_f16 ? launch_wtype<QMV_Q8_0, true>(ms, xs, ys, n, batch, xsplit, pdl, dev, ws, stream)
                         : launch_wtype<QMV_Q8_0, false>(ms, xs, ys, n, batch, xsplit, pdl, dev, ws, stream);
}

}  // namespace dtc
}  // namespace qmv
