// matvec_qx_fused_q4.cu -- the activation-quantized product with in-kernel activation
// quantization, Q4_0 weights (kernels in matvec_qx.cuh).
#include "matvec_qx.cuh"

namespace qmv {

cudaError_t launch_matvec_qx_fused_q4(const MatrixRef* ms, const void* const* xs, float* const* ys, int n,
                                      bool x_bf16, int batch, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  return x_bf16 ? qx::launch_fused_wtype<QMV_Q4_0, true>(ms, xs, ys, n, batch, pdl, dev, stream)
                : qx::launch_fused_wtype<QMV_Q4_0, false>(ms, xs, ys, n, batch, pdl, dev, stream);
}

}  // namespace qmv
