// gguf.cu -- tensors given in GGUF interleaved blocks (minfer "02 - GGUF load" page, §2.3-2.4:
// a Q4_0 block is an f16 d then 16 bytes of nibbles, 18 bytes; a Q8_0 block d then 32 int8
// quants, 34 bytes; a row is cols/32 consecutive blocks, rows follow without padding) into the
// two-array layout the product kernels stream (Krafla ".mlb model format v1", "Body": the q
// array, zeros to a multiple of 64 bytes, then the d array, here f16).  The bytes are moved,
// never decoded: record i's quants become q block i, its d the i-th scale.
//
// A warp takes chunks of 32 records (576 or 1088 bytes, a multiple of 16): it loads a chunk
// with 16-byte loads (each load instruction 512 contiguous bytes) into its own shared buffer,
// then lane i writes record i: its quants as 16-byte stores (a warp store instruction covers
// 512 or 1024 contiguous bytes of q) and its d as one f16 (64 contiguous bytes per warp).
// The last, partial chunk is read in 2-byte pieces, so that no load passes the tensor's end.
#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {

namespace {

constexpr int kGWarps = 8;

template <int WT>
struct Rec {
  static constexpr int QB = WT == QMV_Q8_0 ? 32 : 16;  // quant bytes of a block
  static constexpr int BS = 2 + QB;                      // GGUF record bytes
  static constexpr int CHUNK = 32 * BS;                  // bytes of 32 records
  static constexpr int NP = CHUNK / 16;                  // 16-byte pieces of a chunk: 36 or 68
  static constexpr int PPL = (NP + 31) / 32;             // pieces per lane
};

// Lane `lane` writes record `rec` from the chunk in shared memory (record lane at lane * BS).
template <int WT>
__device__ __forceinline__ void emit(const uint8_t* buf, int lane, long long rec, uint8_t* __restrict__ q,
                                     uint16_t* __restrict__ d) {
  using R = Rec<WT>;
  const uint16_t* r16 = reinterpret_cast<const uint16_t*>(buf + lane * R::BS);  // BS is even
  d[rec] = r16[0];
  uint32_t w[R::QB / 4];
#pragma unroll
  for (int i = 0; i < R::QB / 4; ++i) w[i] = (uint32_t)r16[1 + 2 * i] | ((uint32_t)r16[2 + 2 * i] << 16);
  uint4* dst = reinterpret_cast<uint4*>(q + rec * R::QB);
#pragma unroll
  for (int i = 0; i < R::QB / 16; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

template <int WT>
__global__ void __launch_bounds__(kGWarps * 32) gguf_to_mlb_kernel(const uint8_t* __restrict__ src,
                                                                   uint8_t* __restrict__ q, uint16_t* __restrict__ d,
                                                                   long long nrec) {
  using R = Rec<WT>;
  __shared__ __align__(16) uint8_t sbuf[kGWarps][R::CHUNK];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  uint8_t* buf = sbuf[wid];
  const long long full = nrec / 32;
  const long long W = (long long)gridDim.x * kGWarps;
  const long long gw = (long long)blockIdx.x * kGWarps + wid;
  for (long long c = gw; c < full; c += W) {
    const uint4* p = reinterpret_cast<const uint4*>(src + c * R::CHUNK);
    uint4 v[R::PPL];
#pragma unroll
    for (int t = 0; t < R::PPL; ++t) {
      const int j = 32 * t + lane;
      if (j < R::NP) v[t] = __ldcs(p + j);
    }
#pragma unroll
    for (int t = 0; t < R::PPL; ++t) {
      const int j = 32 * t + lane;
      if (j < R::NP) reinterpret_cast<uint4*>(buf)[j] = v[t];
    }
    __syncwarp();
    emit<WT>(buf, lane, c * 32 + lane, q, d);
    __syncwarp();
  }
  // the partial chunk, by the warp whose turn it would be
  const long long rem = nrec - full * 32;
  if (rem > 0 && gw == full % W) {
    const uint16_t* p16 = reinterpret_cast<const uint16_t*>(src + full * R::CHUNK);
    const int n16 = (int)(rem * R::BS / 2);
    for (int j = lane; j < n16; j += 32) reinterpret_cast<uint16_t*>(buf)[j] = p16[j];
    __syncwarp();
    if (lane < rem) emit<WT>(buf, lane, full * 32 + lane, q, d);
  }
}

}  // namespace

cudaError_t launch_gguf_to_mlb(int wtype, int64_t rows, int64_t cols, const void* src, uint8_t* W, int64_t d_off,
                               int64_t q_bytes, const DeviceInfo& dev, cudaStream_t stream) {
  const long long nrec = rows * (cols / 32);
  if (d_off > q_bytes) {
    const cudaError_t err = cudaMemsetAsync(W + q_bytes, 0, (size_t)(d_off - q_bytes), stream);
    if (err != cudaSuccess) return err;
  }
  const long long chunks = (nrec + 31) / 32;
  long long grid = (chunks + kGWarps - 1) / kGWarps;
  const long long cap = (long long)dev.sm_count * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const uint8_t* s = static_cast<const uint8_t*>(src);
  uint16_t* d = reinterpret_cast<uint16_t*>(W + d_off);
  if (wtype == QMV_Q8_0) {
    gguf_to_mlb_kernel<QMV_Q8_0><<<(unsigned)grid, kGWarps * 32, 0, stream>>>(s, W, d, nrec);
  } else {
    gguf_to_mlb_kernel<QMV_Q4_0><<<(unsigned)grid, kGWarps * 32, 0, stream>>>(s, W, d, nrec);
  }
  return cudaGetLastError();
}

}  // namespace qmv
