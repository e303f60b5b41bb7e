// dequant.cu -- elementwise kernels: bit-exact dequantization and the Q8_0 -128 scan.
//
// Dequantization (Krafla ".mlb model format v1", sections "Q8_0" and "Q4_0"):
//   w = level * d, one float32 multiplication rounded to nearest even; f16 scales are
//   converted to float32 exactly first.  No flush of subnormals (built without fast math).
// Validation ("Validation done by the loader"): a Q8_0 byte equal to -128 is a format error.
#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {

// One thread writes 4 consecutive weights (16 bytes of output).  Weights 4i..4i+3 lie in
// one block (blocks are 32 consecutive weights of a row and tile the rows exactly):
//   Q8_0: their quants are the 4 bytes at 4i.
//   Q4_0: element e of block b sits in byte 16b + (e mod 16), low nibble for e < 16 and
//         high nibble otherwise, so the 4 quants are one aligned word.
template <int WT, bool F16>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ q,
                                                      const uint8_t* __restrict__ d,
                                                      float4* __restrict__ out, int64_t n_quads) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_quads; i += stride) {
    const int64_t e = i * 4;
    const int64_t blk = e >> 5;
    const int j = (int)(e & 31);
    const float dv = F16 ? f16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(d) + blk))
                         : __ldg(reinterpret_cast<const float*>(d) + blk);
    int lv[4];
    if (WT == QMV_Q8_0) {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(q + e));
#pragma unroll
      for (int k = 0; k < 4; ++k) lv[k] = (int)(int8_t)(w >> (8 * k));
    } else {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(q + blk * 16 + (j & 15)));
      const int shift = (j < 16) ? 0 : 4;
#pragma unroll
      for (int k = 0; k < 4; ++k) lv[k] = (int)((w >> (8 * k + shift)) & 0xF) - 8;
    }
    float4 o;
    o.x = __fmul_rn((float)lv[0], dv);
    o.y = __fmul_rn((float)lv[1], dv);
    o.z = __fmul_rn((float)lv[2], dv);
    o.w = __fmul_rn((float)lv[3], dv);
    out[i] = o;
  }
}

cudaError_t launch_dequant(const MatrixRef& m, float* out, cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t err = current_device_info(&dev);
  if (err != cudaSuccess) return err;
  const int64_t n_quads = m.rows * m.cols / 4;
  const int threads = 256;
  int64_t blocks = (n_quads + threads - 1) / threads;
  const int64_t cap = (int64_t)dev.sm_count * 16;
  if (blocks > cap) blocks = cap;
  float4* o = reinterpret_cast<float4*>(out);
  if (m.wtype == QMV_Q8_0) {
    if (m.scale_f16) dequant_kernel<QMV_Q8_0, true><<<(int)blocks, threads, 0, stream>>>(m.q, m.d, o, n_quads);
    else dequant_kernel<QMV_Q8_0, false><<<(int)blocks, threads, 0, stream>>>(m.q, m.d, o, n_quads);
  } else {
    if (m.scale_f16) dequant_kernel<QMV_Q4_0, true><<<(int)blocks, threads, 0, stream>>>(m.q, m.d, o, n_quads);
    else dequant_kernel<QMV_Q4_0, false><<<(int)blocks, threads, 0, stream>>>(m.q, m.d, o, n_quads);
  }
  return cudaGetLastError();
}

__global__ void validate_init_kernel(unsigned long long* first_bad) { *first_bad = ~0ull; }

// Smallest index of a 0x80 byte in q[0, n).  ~0 (that is, -1 as int64) when none.
__global__ void __launch_bounds__(256) validate_q8_kernel(const uint8_t* __restrict__ q, int64_t n,
                                                          unsigned long long* first_bad) {
  const int64_t n16 = n / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(q) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (((w[k] >> (8 * b)) & 0xFF) == 0x80) {
          atomicMin(first_bad, (unsigned long long)(i * 16 + 4 * k + b));
        }
      }
    }
  }
  // tail bytes (q size not a multiple of 16)
  const int64_t t = n16 * 16 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n && q[t] == 0x80) atomicMin(first_bad, (unsigned long long)t);
}

cudaError_t launch_validate(const MatrixRef& m, int64_t* first_bad, cudaStream_t stream) {
  unsigned long long* fb = reinterpret_cast<unsigned long long*>(first_bad);
  validate_init_kernel<<<1, 1, 0, stream>>>(fb);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || m.wtype != QMV_Q8_0) return err;
  DeviceInfo dev;
  err = current_device_info(&dev);
  if (err != cudaSuccess) return err;
  const int64_t n = m.rows * m.cols;
  const int threads = 256;
  int64_t blocks = (n / 16 + threads - 1) / threads;
  if (blocks < 1) blocks = 1;
  const int64_t cap = (int64_t)dev.sm_count * 16;
  if (blocks > cap) blocks = cap;
  validate_q8_kernel<<<(int)blocks, threads, 0, stream>>>(m.q, n, fb);
  return cudaGetLastError();
}

}  // namespace qmv
