// matvec_qx_q8.cu -- the activation-quantized product for Q8_0 weights (kernels in matvec_qx.cuh),
// and the entry that picks the weight type.
#include "matvec_qx.cuh"

namespace qmv {

cudaError_t launch_matvec_qx_q4(const MatrixRef& m, const int8_t* xq, const float* xd, int batch, float* y,
                                const DeviceInfo& dev, cudaStream_t stream);

cudaError_t launch_matvec_qx(const MatrixRef& m, const int8_t* xq, const float* xd, int batch, float* y,
                             const DeviceInfo& dev, cudaStream_t stream) {
  if (m.wtype == QMV_Q8_0) return qx::launch_wtype<QMV_Q8_0>(m, xq, xd, batch, y, dev, stream);
  return launch_matvec_qx_q4(m, xq, xd, batch, y, dev, stream);
}

}  // namespace qmv
