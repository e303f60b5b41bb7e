// quantize.cu -- the writer rules on the device: float32 rows x cols into the two-array
// layout (Krafla ".mlb model format v1", "Quantization rule" and "Body").
//
//   Q8_0 (per block of 32): amax = max |x|.  amax < 1e-30: d = 0 and every quant 0.
//     f32 scale: d = amax / 127, q = trunc(x * (127 / amax) + copysign(0.5, x)).
//     f16 scale: d = the f16 nearest amax / 127 (ties to even; a d beyond the f16 range is
//     refused), q = trunc(x * (1 / d) + copysign(0.5, x)) with the f16 d (d rounding to
//     f16 zero gives the zero block).  q clamped to +-127.
//   Q4_0, the "round" rule: d = (element of largest magnitude, the first of equals) / -8,
//     first rounded to f16 (to nearest) with f16 scales (refused beyond the f16 range);
//     nibble = min(15, trunc(x * (1 / d) + 8.5)), kept at or above 0; 1 / d taken as 0
//     for d = 0.  Element j's nibble is the low half of byte j, element j + 16's the high.
// Every product, quotient and sum is one IEEE float32 operation rounded to nearest even
// (written with the _rn intrinsics, so nothing is contracted), so the bytes equal the
// writer rules' bytes.  Inputs are meant to be finite; what a NaN or infinity produces is
// not specified.
#include <mutex>

#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {

namespace {

// Kernel code of the Q4_0 best-fit rule (its output is a Q4_0 matrix).
constexpr int kQ4Fit = kQuantQ4Fit;

// The Q4_0 best-fit rule for one block: the largest-magnitude element m (first of equals) is
// mapped to each candidate level L = -(60 + 2k) / 10, k = 0..12 (-6 .. -8.4); levels
// l_j = clamp(rint(x_j / s), -8, 7) with s = m / L; d = sum(x^3 l) / sum(x^2 l^2); the candidate
// with the smallest sum(x^2 (x - d l)^2) wins (the first on ties).  A block below 1e-6 is
// fitted at unit scale and d scaled back; the zero block is d = 0, level 0.  Every operation
// is one float32 operation rounded to nearest (ties to even for rint), in element order.
template <bool F16>
__device__ __forceinline__ void quantize_block_fit(const float (&xin)[32], long long blk, uint8_t* __restrict__ q,
                                                   uint8_t* __restrict__ d, unsigned long long* first_bad) {
  float x[32];
  float m = xin[0], a = fabsf(xin[0]);
#pragma unroll
  for (int j = 1; j < 32; ++j)
    if (fabsf(xin[j]) > a) {
      a = fabsf(xin[j]);
      m = xin[j];
    }
  uint32_t best_w[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};  // level 0 everywhere
  float best_d = 0.f;
  if (a != 0.f) {
    const bool small = a < 1e-6f;
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = small ? __fdiv_rn(xin[j], a) : xin[j];
    if (small) m = __fdiv_rn(m, a);
    float best_err = 0.f;
#pragma unroll 1
    for (int k = 0; k <= 12; ++k) {
      const float L = __fdiv_rn((float)(-(60 + 2 * k)), 10.0f);
      const float s = __fdiv_rn(m, L);
      float lv[32];
      float num = 0.f, den = 0.f;
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float r = rintf(__fdiv_rn(x[j], s));
        r = fminf(fmaxf(r, -8.0f), 7.0f);
        lv[j] = r;
        const float t = __fmul_rn(x[j], x[j]);
        num = __fadd_rn(num, __fmul_rn(__fmul_rn(t, x[j]), r));
        den = __fadd_rn(den, __fmul_rn(__fmul_rn(t, r), r));
        const uint32_t nib = (uint32_t)((int)r + 8);
        if (j < 16) {
          w[j >> 2] |= nib << (8 * (j & 3));
        } else {
          w[(j - 16) >> 2] |= nib << (8 * ((j - 16) & 3) + 4);
        }
      }
      const float dk = den == 0.f ? 0.f : __fdiv_rn(num, den);
      float err = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float e = __fsub_rn(x[j], __fmul_rn(dk, lv[j]));
        err = __fadd_rn(err, __fmul_rn(__fmul_rn(x[j], x[j]), __fmul_rn(e, e)));
      }
      if (k == 0 || err < best_err) {
        best_err = err;
        best_d = dk;
#pragma unroll
        for (int i = 0; i < 4; ++i) best_w[i] = w[i];
      }
    }
    if (small) best_d = __fmul_rn(best_d, a);
  }
  uint32_t dbits;
  bool bad = false;
  if (F16) {
    const unsigned short h = __half_as_ushort(__float2half_rn(best_d));
    if ((h & 0x7fffu) >= 0x7c00u) {
      bad = true;  // refused: written as d = 0, every nibble 8
      dbits = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) best_w[i] = 0x88888888u;
    } else {
      dbits = h;
    }
  } else {
    dbits = __float_as_uint(best_d);
  }
  *reinterpret_cast<uint4*>(q + blk * 16) = make_uint4(best_w[0], best_w[1], best_w[2], best_w[3]);
  if (F16) {
    reinterpret_cast<uint16_t*>(d)[blk] = (uint16_t)dbits;
  } else {
    reinterpret_cast<uint32_t*>(d)[blk] = dbits;
  }
  if (bad) atomicMin(first_bad, (unsigned long long)blk);
}

// The rules for one block, held whole by one lane (x[e] = element e).
template <int WT, bool F16>
__device__ __forceinline__ void quantize_block(const float (&x)[32], long long blk, uint8_t* __restrict__ q,
                                               uint8_t* __restrict__ d, unsigned long long* first_bad) {
  uint32_t dbits = 0;
  bool bad = false;
  if (WT == QMV_Q8_0) {
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float a = fabsf(x[e]);
      if (a > amax) amax = a;
    }
    float inv = 0.f;  // 0: the zero block
    if (!(amax < 1e-30f)) {
      if (F16) {
        const unsigned short h = __half_as_ushort(__float2half_rn(__fdiv_rn(amax, 127.0f)));
        if ((h & 0x7fffu) >= 0x7c00u) {
          bad = true;  // refused: written as the zero block
        } else {
          const float dv = __half2float(__ushort_as_half(h));
          if (dv != 0.f) {
            inv = __fdiv_rn(1.0f, dv);
            dbits = h;
          }
        }
      } else {
        inv = __fdiv_rn(127.0f, amax);
        dbits = __float_as_uint(__fdiv_rn(amax, 127.0f));
      }
    }
    uint32_t w[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      uint32_t packed = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // inv = 0 (the zero block) gives trunc(+-0.5) = 0 with no branch; the conversion
        // truncates, and clamping its integer equals clamping the truncated float
        const float xe = x[4 * g + k];
        int v = (int)__fadd_rn(__fmul_rn(xe, inv), copysignf(0.5f, xe));
        v = v > 127 ? 127 : (v < -127 ? -127 : v);
        packed |= (uint32_t)(v & 0xFF) << (8 * k);
      }
      w[g] = packed;
    }
    uint4* dst = reinterpret_cast<uint4*>(q + blk * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
    // element of largest magnitude, the first of equals (strict > in element order)
    float best = fabsf(x[0]), bval = x[0];
#pragma unroll
    for (int e = 1; e < 32; ++e)
      if (fabsf(x[e]) > best) {
        best = fabsf(x[e]);
        bval = x[e];
      }
    float dv = __fdiv_rn(bval, -8.0f);
    if (F16) {
      const unsigned short h = __half_as_ushort(__float2half_rn(dv));
      if ((h & 0x7fffu) >= 0x7c00u) {
        bad = true;  // refused: written as d = 0, every nibble 8
        dv = 0.f;
      } else {
        dv = __half2float(__ushort_as_half(h));
        dbits = h;
      }
    } else {
      dbits = __float_as_uint(dv);
    }
    const float id = (dv != 0.f) ? __fdiv_rn(1.0f, dv) : 0.f;
    uint32_t nib[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int n = (int)__fadd_rn(__fmul_rn(x[e], id), 8.5f);  // the conversion truncates
      nib[e] = (uint32_t)(n > 15 ? 15 : (n < 0 ? 0 : n));
    }
    // byte j = nibble of element j | nibble of element j + 16 << 4
    uint32_t w[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t packed = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) packed |= (nib[4 * g + k] | (nib[4 * g + k + 16] << 4)) << (8 * k);
      w[g] = packed;
    }
    *reinterpret_cast<uint4*>(q + blk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (F16) {
    reinterpret_cast<uint16_t*>(d)[blk] = (uint16_t)dbits;
  } else {
    reinterpret_cast<uint32_t*>(d)[blk] = dbits;
  }
  if (bad) atomicMin(first_bad, (unsigned long long)blk);
}

// A warp takes a chunk of 32 consecutive blocks (4 KB of float32) at a time, lane i the
// chunk's block i.  The chunk comes into shared memory by cp.async, coalesced (the warp's
// 16-byte copies cover 512 contiguous bytes each); block i lands in a slot of 36 floats, so
// that the lanes' 16-byte reads of their own blocks hit distinct banks in every phase.  Each
// warp keeps its own ring of kQStages chunks: kQStages - 1 are in flight while it works on
// one, and cp.async.wait_group (a hardware wait) orders them; nothing spins.
constexpr int kQWarps = 8;
constexpr int kQStages = 2;
constexpr int kQSlot = 36;
constexpr int kQStageFloats = 32 * kQSlot;
constexpr int kQSmem = kQWarps * kQStages * kQStageFloats * 4;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int WT, bool F16>
__global__ void __launch_bounds__(kQWarps * 32) quantize_kernel(const float* __restrict__ src,
                                                                uint8_t* __restrict__ q, uint8_t* __restrict__ d,
                                                                long long nblk, unsigned long long* first_bad) {
  extern __shared__ __align__(16) float qsm[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const uint32_t ring = smem_u32(qsm) + (uint32_t)(wid * kQStages * kQStageFloats * 4);
  const long long chunks = (nblk + 31) / 32;
  const long long W = (long long)gridDim.x * kQWarps;
  const long long gw = (long long)blockIdx.x * kQWarps + wid;

  // copy chunk c (if there is one) into stage st; one commit group either way
  auto issue = [&](long long c, int st) {
    if (c < chunks) {
      const long long b0 = c * 32;
      const long long left = nblk - b0;
      const int nb = left < 32 ? (int)left : 32;
      const float* g = src + b0 * 32;
      const uint32_t base = ring + (uint32_t)(st * kQStageFloats * 4);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int j = 32 * t + lane;  // 16-byte piece j of the chunk: block j / 8, quarter j % 8
        if (j < nb * 8) cp_async16(base + (uint32_t)(((j >> 3) * kQSlot + 4 * (j & 7)) * 4), g + 4 * j);
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int st = 0; st < kQStages - 1; ++st) issue(gw + st * W, st);
  long long k = 0;
  for (long long c = gw; c < chunks; c += W, ++k) {
    // the stage refilled here was read in the previous pass, which every lane has left
    issue(c + (kQStages - 1) * W, (int)((k + kQStages - 1) % kQStages));
    cp_async_wait<kQStages - 1>();  // this lane's copies of chunk c have landed
    __syncwarp();                   // ... and every other lane's are visible
    const uint32_t slot = ring + (uint32_t)(((int)(k % kQStages) * kQStageFloats + lane * kQSlot) * 4);
    float x[32];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      float f[4];
      lds_f32x4(slot + 16 * v, f);
      x[4 * v] = f[0];
      x[4 * v + 1] = f[1];
      x[4 * v + 2] = f[2];
      x[4 * v + 3] = f[3];
    }
    const long long blk = c * 32 + lane;
    if (blk < nblk) {
      if constexpr (WT == kQ4Fit) {
        quantize_block_fit<F16>(x, blk, q, d, first_bad);
      } else {
        quantize_block<WT, F16>(x, blk, q, d, first_bad);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
}

// Grid: every CTA resident at once (the occupancy of this instance times the SMs), and no
// more warps than chunks.
template <int WT, bool F16>
cudaError_t launch_typed(const float* src, uint8_t* q, uint8_t* d, long long nblk, unsigned long long* fb,
                         const DeviceInfo& dev, cudaStream_t stream) {
  auto kern = quantize_kernel<WT, F16>;
  static std::mutex mu;
  static int ctas_per_sm[64] = {};  // 0 = not yet known
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidValue;
  if ((size_t)kQSmem > dev.smem_optin) return cudaErrorInvalidConfiguration;
  int per_sm;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (ctas_per_sm[dev.device] == 0) {
      cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
      if (err != cudaSuccess) return err;
      int k = 0;
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, kern, kQWarps * 32, kQSmem);
      if (err != cudaSuccess) return err;
      ctas_per_sm[dev.device] = k > 0 ? k : 1;
    }
    per_sm = ctas_per_sm[dev.device];
  }
  const long long chunks = (nblk + 31) / 32;
  long long grid = (chunks + kQWarps - 1) / kQWarps;
  const long long cap = (long long)dev.sm_count * per_sm;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kQWarps * 32, kQSmem, stream>>>(src, q, d, nblk, fb);
  return cudaGetLastError();
}

// The runtime's activation quantizer: the Q8_0 rule with an f32 scale on blocks of 32
// activations (float32, or bfloat16 widened exactly), four lanes to a block (lane 4g + p holds
// values 8p .. 8p + 7 of the warp's block g).  The block's amax comes from two xor shuffles (the
// maximum does not depend on the order; NaN is skipped); lane pair (4g, 4g + 1) takes the rule's
// two divisions, and every value's quant is the rule's float32 steps.  Activations are a few KB
// to a few MB, so this is launch-latency bound: four lanes shorten each thread's chain to 8
// values (one thread per block took about 0.6 us more).
// The x arrays of a group are blockIdx.y; the kernel lets the next launch start at once (its
// dependents wait for it to finish), and with a programmatic launch of this kernel x is read
// only after the preceding kernel has finished.
template <bool BF16>
__global__ void __launch_bounds__(128) quantize_x_group_kernel(const __grid_constant__ QxImages a) {
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  const int i = blockIdx.y;
  const long long t = (long long)blockIdx.x * 128 + threadIdx.x;
  const long long blk = t >> 2;
  const int part = (int)(t & 3);
  const bool live = blk < a.nblk[i];  // every lane takes part in the shuffles
  float v[8];
  if (!live) {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.f;
  } else if (BF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x[i]) + blk * 32 + 8 * part));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.x[i]) + blk * 32 + 8 * part);
    const float4 f0 = __ldg(p), f1 = __ldg(p + 1);
    v[0] = f0.x, v[1] = f0.y, v[2] = f0.z, v[3] = f0.w, v[4] = f1.x, v[5] = f1.y, v[6] = f1.z, v[7] = f1.w;
  }
  float amax = 0.f;  // fmaxf skips a NaN operand, so amax never is NaN
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // lane 4g divides for d = amax / 127, lane 4g + 1 for 127 / amax; the zero block (amax below
  // 1e-30) has d = 0 and its inverse taken as 0
  const int lane = threadIdx.x & 31;
  const float quot = amax < 1e-30f ? 0.f : ((lane & 1) ? __fdiv_rn(127.0f, amax) : __fdiv_rn(amax, 127.0f));
  const float d = __shfl_sync(0xffffffffu, quot, lane & ~3);
  const float inv = __shfl_sync(0xffffffffu, quot, (lane & ~3) + 1);
  uint32_t w[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint32_t packed = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // inv = 0 gives trunc(+-0.5) = 0; the conversion truncates
      const float xe = v[4 * g + k];
      int q = (int)__fadd_rn(__fmul_rn(xe, inv), copysignf(0.5f, xe));
      q = q > 127 ? 127 : (q < -127 ? -127 : q);
      packed |= (uint32_t)(q & 0xFF) << (8 * k);
    }
    w[g] = packed;
  }
  if (live) {
    *reinterpret_cast<uint2*>(a.q[i] + blk * 32 + 8 * part) = make_uint2(w[0], w[1]);
    if (part == 0) a.d[i][blk] = d;
  }
}

}  // namespace

cudaError_t launch_quantize_x_group(bool x_bf16, const QxImages& a, int n, bool pdl, cudaStream_t stream) {
  if (n < 1 || n > QxImages::kMax) return cudaErrorInvalidValue;
  long long most = 0;
  for (int i = 0; i < n; ++i) most = a.nblk[i] > most ? a.nblk[i] : most;
  if (most == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((4 * most + 127) / 128), (unsigned)n);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return x_bf16 ? cudaLaunchKernelEx(&cfg, quantize_x_group_kernel<true>, a)
                : cudaLaunchKernelEx(&cfg, quantize_x_group_kernel<false>, a);
}

cudaError_t launch_quantize_x(bool x_bf16, int64_t batch, int64_t cols, const void* x, uint8_t* xq, int64_t d_off,
                              int64_t q_bytes, cudaStream_t stream) {
  if (d_off > q_bytes) {
    const cudaError_t err = cudaMemsetAsync(xq + q_bytes, 0, (size_t)(d_off - q_bytes), stream);
    if (err != cudaSuccess) return err;
  }
  QxImages a{};
  a.x[0] = x;
  a.q[0] = xq;
  a.d[0] = reinterpret_cast<float*>(xq + d_off);
  a.nblk[0] = batch * (cols / 32);
  return launch_quantize_x_group(x_bf16, a, 1, false, stream);
}

cudaError_t launch_quantize(int wtype, bool scale_f16, int64_t rows, int64_t cols, const float* src, uint8_t* W,
                            int64_t d_off, int64_t q_bytes, int64_t* first_bad, const DeviceInfo& dev,
                            cudaStream_t stream) {
  const long long nblk = rows * (cols / 32);
  cudaError_t err = cudaMemsetAsync(first_bad, 0xFF, sizeof(int64_t), stream);  // -1: none refused
  if (err != cudaSuccess) return err;
  if (d_off > q_bytes) {
    err = cudaMemsetAsync(W + q_bytes, 0, (size_t)(d_off - q_bytes), stream);  // the padding between the arrays
    if (err != cudaSuccess) return err;
  }
  unsigned long long* fb = reinterpret_cast<unsigned long long*>(first_bad);
  uint8_t* d = W + d_off;
  if (wtype == QMV_Q8_0) {
    return scale_f16 ? launch_typed<QMV_Q8_0, true>(src, W, d, nblk, fb, dev, stream)
                     : launch_typed<QMV_Q8_0, false>(src, W, d, nblk, fb, dev, stream);
  }
  if (wtype == kQ4Fit) {
    return scale_f16 ? launch_typed<kQ4Fit, true>(src, W, d, nblk, fb, dev, stream)
                     : launch_typed<kQ4Fit, false>(src, W, d, nblk, fb, dev, stream);
  }
  return scale_f16 ? launch_typed<QMV_Q4_0, true>(src, W, d, nblk, fb, dev, stream)
                   : launch_typed<QMV_Q4_0, false>(src, W, d, nblk, fb, dev, stream);
}

}  // namespace qmv
