// matvec_qx_q4.cu -- the activation-quantized product for Q4_0 weights (kernels in matvec_qx.cuh).
#include "matvec_qx.cuh"

namespace qmv {

cudaError_t launch_matvec_qx_q4(const MatrixRef& m, const int8_t* xq, const float* xd, int batch, float* y,
                                const DeviceInfo& dev, cudaStream_t stream) {
  return qx::launch_wtype<QMV_Q4_0>(m, xq, xd, batch, y, dev, stream);
}

}  // namespace qmv
