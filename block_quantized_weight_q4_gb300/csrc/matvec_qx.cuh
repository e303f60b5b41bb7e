// matvec_qx.cuh -- the activation-quantized product: weights as stored (Q8_0 or Q4_0, f32 or
// f16 scales) against activations already quantized to Q8_0 blocks with f32 scales (the
// runtime's activation quantizer, Krafla ".mlb model format v1", "Quantization rule"; the
// minfer "02 - GGUF load" page on products taken in quantized space).
//
//   y[v][r] = sum over blocks b of (d_w[r][b] * d_x[v][b]) * isum,
//   isum    = sum_j level_w[r][32b + j] * q_x[v][32b + j]   (an exact integer, |isum| < 2^20)
//
// isum is formed with dp4a (four int8 products and their sum per instruction, exact).  Q4_0
// nibbles n enter as they are (0..15) and the level offset is taken out afterwards:
// sum_j (n_j - 8) q_j = sum_j n_j q_j - 8 sum_j q_j, the activation block's sum coming from
// one more dp4a per word against 0x01010101.  Each block then adds (d_w * d_x) * isum to an
// f32 accumulator (isum converts to f32 exactly), and the 32 lanes' sums meet by shuffles.
//
// Work split: a warp takes R consecutive rows and one of KS column slices; slice s holds the
// 32-block chunks s, s + KS, s + 2 KS, ... of those rows, and lane l block l of each chunk, so
// that each weight load instruction of the warp covers 512 (Q4_0) or 1024 (Q8_0) contiguous
// bytes of one row, and one activation block, loaded once per lane, serves R rows.  A CTA's 8
// warps are 8 / KS row groups times KS slices: the slices of a row group read neighbouring
// pieces of the same rows at the same time, and their sums meet in shared memory, added in
// slice order (results do not depend on timing).  The next chunk's weights are loaded before
// the current ones are used.  Vectors: up to NV per launch (1, 2, 4 or 8; a batch that is not
// a power of two repeats its last vector's loads and does not store them).
#pragma once

#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace qx {

constexpr int kWarps = 8;  // warps per CTA

template <int WT>
struct Words {
  static constexpr int N = WT == QMV_Q8_0 ? 8 : 4;  // 32-bit words of one block's quants
};

template <bool F16>
__device__ __forceinline__ float load_scale(const uint8_t* __restrict__ d, long long idx) {
  if (F16) return __half2float(__ushort_as_half(__ldcs(reinterpret_cast<const unsigned short*>(d) + idx)));
  return __ldcs(reinterpret_cast<const float*>(d) + idx);
}

template <int WT, bool F16, int R>
struct WeightTile {
  uint32_t w[R][Words<WT>::N];
  float dw[R];

  __device__ __forceinline__ void load(const uint8_t* __restrict__ q, const uint8_t* __restrict__ d,
                                       const long long (&row)[R], long long nb, long long b) {
    constexpr int NW = Words<WT>::N;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint4* p = reinterpret_cast<const uint4*>(q + (row[r] * nb + b) * (NW * 4));
#pragma unroll
      for (int i = 0; i < NW / 4; ++i) {
        const uint4 u = __ldcs(p + i);
        w[r][4 * i] = u.x;
        w[r][4 * i + 1] = u.y;
        w[r][4 * i + 2] = u.z;
        w[r][4 * i + 3] = u.w;
      }
      dw[r] = load_scale<F16>(d, row[r] * nb + b);
    }
  }
};

// Passes of one vector: three CTAs per SM (24 warps, more loads in flight; the tile fits 80
// registers); larger passes two.
template <int R, int NV>
struct MinCtas {
  static constexpr int value = NV == 1 ? 3 : 2;
};

template <int WT, bool F16, int R, int NV>
__global__ void __launch_bounds__(kWarps * 32, MinCtas<R, NV>::value)
    matvec_qx_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ d, const int8_t* __restrict__ xq,
                     const float* __restrict__ xd, long long rows, long long nb, int nv, int ks,
                     float* __restrict__ y) {
  __shared__ float red[kWarps][NV][R];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int slice = warp % ks;
  const long long r0 = ((long long)blockIdx.x * (kWarps / ks) + warp / ks) * R;
  const bool live = r0 < rows;  // warp-uniform; every warp reaches the barrier below
  long long row[R];
#pragma unroll
  for (int r = 0; r < R; ++r) row[r] = r0 + r < rows ? r0 + r : rows - 1;  // loads stay in the matrix

  float acc[NV][R];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[v][r] = 0.f;

  WeightTile<WT, F16, R> cur, nxt;
  const long long step = 32LL * ks;
  const long long b0 = live ? 32LL * slice + lane : nb;
  if (b0 < nb) cur.load(q, d, row, nb, b0);
  for (long long b = b0; b < nb; b += step) {
    if (b + step < nb) nxt.load(q, d, row, nb, b + step);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const long long vv = v < nv ? v : nv - 1;
      const int4* xp = reinterpret_cast<const int4*>(xq + (vv * nb + b) * 32);
      const int4 xa = __ldg(xp), xb = __ldg(xp + 1);
      const int xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      const float dx = __ldg(xd + vv * nb + b);
      int sx = 0;  // sum of the block's activation quants (Q4_0's level offset)
      if (WT == QMV_Q4_0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) sx = __dp4a(xw[i], 0x01010101, sx);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        int dot = 0;
        if (WT == QMV_Q8_0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) dot = __dp4a((int)cur.w[r][i], xw[i], dot);
        } else {
          // word i: low nibbles are elements 4i..4i+3 (activation word i), high nibbles the
          // elements 16 later (activation word i + 4)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dot = __dp4a((int)(cur.w[r][i] & 0x0F0F0F0Fu), xw[i], dot);
            dot = __dp4a((int)((cur.w[r][i] >> 4) & 0x0F0F0F0Fu), xw[i + 4], dot);
          }
          dot -= 8 * sx;
        }
        acc[v][r] = __fmaf_rn(__fmul_rn(cur.dw[r], dx), (float)dot, acc[v][r]);
      }
    }
    cur = nxt;
  }

#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[v][r] += __shfl_xor_sync(0xffffffffu, acc[v][r], o);
  if (ks == 1) {
    if (lane == 0 && live) {
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (v < nv && r0 + r < rows) y[(long long)v * rows + r0 + r] = acc[v][r];
    }
    return;
  }
  if (lane == 0) {
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int r = 0; r < R; ++r) red[warp][v][r] = acc[v][r];
  }
  __syncthreads();
  // lane (v, r) of the row group's first warp adds the slices in order
  if (slice == 0 && live && lane < NV * R) {
    const int v = lane / R, r = lane % R;
    float sum = red[warp][v][r];
    for (int s2 = 1; s2 < ks; ++s2) sum += red[warp + s2][v][r];
    if (v < nv && r0 + r < rows) y[(long long)v * rows + r0 + r] = sum;
  }
}

// Warps a launch wants: one wave at two 8-warp CTAs per SM.
inline long long warps_wanted(int sm_count) { return (long long)sm_count * 2 * kWarps; }

// Column slices per row group: the fewest (1, 2, 4 or 8, each with at least one 32-block
// chunk of the row) that give the launch the warps it wants; max_slices: the most allowed.
inline int slices_for(long long row_groups, long long nb, int sm_count, bool max_slices = false) {
  int ks = 1;
  while (ks < kWarps && (max_slices || row_groups * ks < warps_wanted(sm_count)) && 32LL * 2 * ks <= nb) ks *= 2;
  return ks;
}

template <int WT, bool F16, int R, int NV>
cudaError_t launch_rnv(const MatrixRef& m, const int8_t* xq, const float* xd, int nv, float* y,
                       const DeviceInfo& dev, cudaStream_t stream) {
  const long long nb = m.cols / 32;
  const long long groups = (m.rows + R - 1) / R;
  const int ks = slices_for(groups, nb, dev.sm_count);
  const long long per_cta = kWarps / ks;
  const long long grid = (groups + per_cta - 1) / per_cta;
  matvec_qx_kernel<WT, F16, R, NV><<<(unsigned)grid, kWarps * 32, 0, stream>>>(m.q, m.d, xq, xd, m.rows, nb, nv,
                                                                                 ks, y);
  return cudaGetLastError();
}

// Four rows per warp only for passes of one or two vectors (more accumulators do not fit
// the registers of two CTAs per SM).
template <int WT, bool F16, int R>
cudaError_t launch_r(const MatrixRef& m, const int8_t* xq, const float* xd, int nv, float* y,
                     const DeviceInfo& dev, cudaStream_t stream) {
  if (nv == 1) return launch_rnv<WT, F16, R, 1>(m, xq, xd, nv, y, dev, stream);
  if constexpr (R == 4) {
    return launch_rnv<WT, F16, R, 2>(m, xq, xd, nv, y, dev, stream);
  } else {
    if (nv == 2) return launch_rnv<WT, F16, R, 2>(m, xq, xd, nv, y, dev, stream);
    if (nv <= 4) return launch_rnv<WT, F16, R, 4>(m, xq, xd, nv, y, dev, stream);
    return launch_rnv<WT, F16, R, 8>(m, xq, xd, nv, y, dev, stream);
  }
}

// One weight type: passes of up to 8 vectors.
template <int WT>
cudaError_t launch_wtype(const MatrixRef& m, const int8_t* xq, const float* xd, int batch, float* y,
                         const DeviceInfo& dev, cudaStream_t stream) {
  // rows per warp: Q4_0 four (two for passes of more than two vectors), Q8_0 two; fewer where
  // the row groups, each split into as many column slices as the row allows, would not give
  // the launch the warps it wants
  constexpr int R4 = WT == QMV_Q4_0 ? 4 : 2;
  const long long nb = m.cols / 32;
  const int ks_max = slices_for(1, nb, dev.sm_count, true);
  int R = R4;
  while (R > 1 && (m.rows + R - 1) / R * ks_max < warps_wanted(dev.sm_count)) R /= 2;
  for (int v0 = 0; v0 < batch; v0 += 8) {
    const int nv = batch - v0 < 8 ? batch - v0 : 8;
    const int8_t* xqp = xq + (long long)v0 * m.cols;
    const float* xdp = xd + (long long)v0 * nb;
    float* yp = y + (long long)v0 * m.rows;
    const int Rp = R == 4 && nv > 2 ? 2 : R;
    cudaError_t err;
    if (m.scale_f16) {
      err = Rp == 4  ? launch_r<WT, true, R4>(m, xqp, xdp, nv, yp, dev, stream)
            : Rp == 2 ? launch_r<WT, true, 2>(m, xqp, xdp, nv, yp, dev, stream)
                     : launch_r<WT, true, 1>(m, xqp, xdp, nv, yp, dev, stream);
    } else {
      err = Rp == 4  ? launch_r<WT, false, R4>(m, xqp, xdp, nv, yp, dev, stream)
            : Rp == 2 ? launch_r<WT, false, 2>(m, xqp, xdp, nv, yp, dev, stream)
                     : launch_r<WT, false, 1>(m, xqp, xdp, nv, yp, dev, stream);
    }
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace qx
}  // namespace qmv
