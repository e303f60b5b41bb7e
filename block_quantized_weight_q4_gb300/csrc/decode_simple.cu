// decode_simple.cu -- warp-per-row product for any shape (cols a multiple of 32).
//
// The general path, used where the fast kernel's alignment needs are not met (a row's run
// of scales not 16-byte aligned, i.e. cols not a multiple of 256).  Lane l of a warp takes
// blocks l, l+32, ... of the row; per block it forms sum_j level_j * x_j in float32, scales
// by d and adds into its accumulator; the warp then sums its lanes with shuffles.
// (Krafla ".mlb model format v1": "Q8_0", "Q4_0", and y[r] = sum_c W[r][c] x[c].)
#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {

template <bool XBF16>
__device__ __forceinline__ void load_x32(const void* x, int64_t off, float (&xv)[32]) {
  if (XBF16) {
    const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(x) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(p + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        xv[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
        xv[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + off);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = __ldg(p + i);
      xv[4 * i] = v.x;
      xv[4 * i + 1] = v.y;
      xv[4 * i + 2] = v.z;
      xv[4 * i + 3] = v.w;
    }
  }
}

template <int WT, bool F16, bool XBF16, int NB>
__global__ void __launch_bounds__(256) matvec_simple_kernel(const uint8_t* __restrict__ q,
                                                            const uint8_t* __restrict__ d,
                                                            const void* __restrict__ x, float* __restrict__ y,
                                                            int64_t rows, int64_t cols, int batch) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t nblk = cols / 32;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    for (int64_t k = lane; k < nblk; k += 32) {
      const int64_t sidx = r * nblk + k;
      const float dv = F16 ? f16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(d) + sidx))
                           : __ldg(reinterpret_cast<const float*>(d) + sidx);
      float lv[32];
      if (WT == QMV_Q4_0) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(q + r * (cols / 2) + 16 * k));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t byte = (w[j >> 2] >> (8 * (j & 3))) & 0xFF;
          lv[j] = (float)((int)(byte & 0xF) - 8);
          lv[j + 16] = (float)((int)(byte >> 4) - 8);
        }
      } else {
        const uint4* p = reinterpret_cast<const uint4*>(q + r * cols + 32 * k);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint4 v = __ldg(p + i);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 16; ++j) lv[16 * i + j] = (float)(int8_t)(w[j >> 2] >> (8 * (j & 3)));
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < batch) {
          float xv[32];
          load_x32<XBF16>(x, (int64_t)b * cols + 32 * k, xv);
          float s = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) s = fmaf(lv[j], xv[j], s);
          acc[b] = fmaf(dv, s, acc[b]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float v = acc[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && b < batch) y[(int64_t)b * rows + r] = v;
    }
  }
}

template <int WT, bool F16, bool XBF16>
static cudaError_t launch_nb(const MatrixRef& m, const void* x, float* y, int batch, int blocks,
                             cudaStream_t stream) {
  if (batch <= 1)
    matvec_simple_kernel<WT, F16, XBF16, 1><<<blocks, 256, 0, stream>>>(m.q, m.d, x, y, m.rows, m.cols, batch);
  else if (batch <= 2)
    matvec_simple_kernel<WT, F16, XBF16, 2><<<blocks, 256, 0, stream>>>(m.q, m.d, x, y, m.rows, m.cols, batch);
  else if (batch <= 4)
    matvec_simple_kernel<WT, F16, XBF16, 4><<<blocks, 256, 0, stream>>>(m.q, m.d, x, y, m.rows, m.cols, batch);
  else
    matvec_simple_kernel<WT, F16, XBF16, 8><<<blocks, 256, 0, stream>>>(m.q, m.d, x, y, m.rows, m.cols, batch);
  return cudaGetLastError();
}

cudaError_t launch_matvec_simple(const MatrixRef& m, const void* x, bool x_bf16, float* y, int batch,
                                 const DeviceInfo& dev, cudaStream_t stream) {
  int64_t blocks = (m.rows + 7) / 8;  // 8 warps per block, one row per warp
  const int64_t cap = (int64_t)dev.sm_count * 8;
  if (blocks > cap) blocks = cap;
  const int nb = (int)blocks;
  if (m.wtype == QMV_Q4_0) {
    if (m.scale_f16) return x_bf16 ? launch_nb<QMV_Q4_0, true, true>(m, x, y, batch, nb, stream)
                                   : launch_nb<QMV_Q4_0, true, false>(m, x, y, batch, nb, stream);
    return x_bf16 ? launch_nb<QMV_Q4_0, false, true>(m, x, y, batch, nb, stream)
                  : launch_nb<QMV_Q4_0, false, false>(m, x, y, batch, nb, stream);
  }
  if (m.scale_f16) return x_bf16 ? launch_nb<QMV_Q8_0, true, true>(m, x, y, batch, nb, stream)
                                 : launch_nb<QMV_Q8_0, true, false>(m, x, y, batch, nb, stream);
  return x_bf16 ? launch_nb<QMV_Q8_0, false, true>(m, x, y, batch, nb, stream)
                : launch_nb<QMV_Q8_0, false, false>(m, x, y, batch, nb, stream);
}

}  // namespace qmv
