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

#include <mutex>

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

// ------------------------------------------------------------------------ fused activations
// The same product for several problems in one launch, each with its float activations (bf16
// or f32) quantized inside the kernel with the runtime's rule (the bytes qmv_quantize_x
// writes) into shared memory, from where the loop above reads them.  CTAs are
// persistent (one wave, by occupancy) and walk items of kWarps / ks row groups, problem after
// problem; a CTA quantizes a problem's activations when it first meets them (problems that
// share one x pointer share one quantization), so the quantizer's work is spread over all the
// rows a CTA takes.  Shared layout per vector: quants of block b in two 16-byte planes
// (elements 0..15 at lo[b], 16..31 at hi[b], so that the lanes' 16-byte reads of consecutive
// blocks are contiguous), then the scales.  With programmatic overlap the first weight tile is
// requested before the activations are read.
constexpr int kMaxFused = 8;

struct FusedProblem {
  const uint8_t* q;
  const uint8_t* d;
  long long rows;
  long long nb;    // blocks per row (cols / 32)
  const void* x;   // nv vectors of cols activations, row-major
  float* y;        // nv x rows
  int item0;       // first item of this problem
};

struct FusedParams {
  FusedProblem pr[kMaxFused];
  int nprob;
  int nitems;
  int nv;
  int ks;
  long long snb;   // blocks per vector in shared memory (the largest nb of the group)
};

// Eight activations (float32, or bfloat16 widened exactly) from element `first` of x.
template <bool BF16>
__device__ __forceinline__ void load_act8(const void* __restrict__ x, long long first, float (&v)[8]) {
  if (BF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + first));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + first);
    const float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
  }
}

template <int WT, bool F16, int R, int NV, bool BF16X>
__global__ void __launch_bounds__(kWarps * 32, MinCtas<R, NV>::value)
    matvec_qx_fused_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(16) uint8_t qsm[];
  __shared__ float red[kWarps][NV][R];
  const long long snb = p.snb;
  const int nv = p.nv, ks = p.ks;
  uint8_t* qlo = qsm;                               // [nv][snb][16]
  uint8_t* qhi = qsm + (size_t)nv * snb * 16;       // [nv][snb][16]
  float* xds = reinterpret_cast<float*>(qsm + (size_t)nv * snb * 32);  // [nv][snb]
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int slice = warp % ks;
  const void* quantized = nullptr;  // activations now in shared memory
  bool first = true;
  int pi = 0;

  for (int item = (int)blockIdx.x; item < p.nitems; item += (int)gridDim.x) {
    while (pi + 1 < p.nprob && item >= p.pr[pi + 1].item0) ++pi;
    const FusedProblem& P = p.pr[pi];
    const long long rows = P.rows, nb = P.nb;
    const long long r0 = ((long long)(item - P.item0) * (kWarps / ks) + warp / ks) * R;
    const bool live = r0 < rows;  // warp-uniform; every warp reaches the barriers below
    long long row[R];
#pragma unroll
    for (int r = 0; r < R; ++r) row[r] = r0 + r < rows ? r0 + r : rows - 1;

    WeightTile<WT, F16, R> cur, nxt;
    const long long step = 32LL * ks;
    const long long b0 = live ? 32LL * slice + lane : nb;
    if (b0 < nb) cur.load(P.q, P.d, row, nb, b0);  // weights: independent of the preceding kernel
    if (first) griddep_wait();  // the activations may be the preceding kernel's output
    if (P.x != quantized) {
      // the runtime's rule with each block spread over four consecutive lanes,
      // eight values each (few registers next to the prefetched tile): the block's amax by two
      // shuffles, then every lane the same scale and its eight quants
      __syncthreads();  // the previous activations are no longer read
      const long long nq = 4LL * nv * nb;
      for (long long t0 = 0; t0 < nq; t0 += kWarps * 32) {
        const long long t = t0 + threadIdx.x;
        const bool act = t < nq;  // the loop runs warp-uniformly for the shuffles
        const long long blk = act ? t >> 2 : 0;
        const int part = (int)(t & 3);
        const long long v = blk / nb, b = blk - v * nb;
        float vals[8];
        if (act) {
          load_act8<BF16X>(P.x, (v * nb + b) * 32 + 8 * part, vals);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) vals[e] = 0.f;
        }
        float amax = 0.f;  // fmaxf skips a NaN operand
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(vals[e]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        float inv = 0.f, dv = 0.f;  // the zero block
        if (!(amax < 1e-30f)) {
          inv = __fdiv_rn(127.0f, amax);
          dv = __fdiv_rn(amax, 127.0f);
        }
        uint32_t w[2];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t packed = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float xe = vals[4 * g + k];
            int qv = (int)__fadd_rn(__fmul_rn(xe, inv), copysignf(0.5f, xe));
            qv = qv > 127 ? 127 : (qv < -127 ? -127 : qv);
            packed |= (uint32_t)(qv & 0xFF) << (8 * k);
          }
          w[g] = packed;
        }
        if (act) {
          uint8_t* plane = part < 2 ? qlo : qhi;
          *reinterpret_cast<uint2*>(plane + (v * snb + b) * 16 + 8 * (part & 1)) = make_uint2(w[0], w[1]);
          if (part == 0) xds[v * snb + b] = dv;
        }
      }
      __syncthreads();
      quantized = P.x;
    }
    if (first && threadIdx.x == 0) griddep_launch_dependents();
    first = false;

    float acc[NV][R];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[v][r] = 0.f;
    for (long long b = b0; b < nb; b += step) {
      if (b + step < nb) nxt.load(P.q, P.d, row, nb, b + step);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const long long vv = v < nv ? v : nv - 1;
        const int4 xa = *reinterpret_cast<const int4*>(qlo + (vv * snb + b) * 16);
        const int4 xb = *reinterpret_cast<const int4*>(qhi + (vv * snb + b) * 16);
        const int xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const float dx = xds[vv * snb + b];
        int sx = 0;
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
            if (v < nv && r0 + r < rows) P.y[(long long)v * rows + r0 + r] = acc[v][r];
      }
      continue;
    }
    if (lane == 0) {
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) red[warp][v][r] = acc[v][r];
    }
    __syncthreads();
    if (slice == 0 && live && lane < NV * R) {
      const int v = lane / R, r = lane % R;
      float sum = red[warp][v][r];
      for (int s2 = 1; s2 < ks; ++s2) sum += red[warp + s2][v][r];
      if (v < nv && r0 + r < rows) P.y[(long long)v * rows + r0 + r] = sum;
    }
    __syncthreads();  // red is read before the next item writes it
  }
  if (first) {
    // a CTA with no item still lets the dependent launch proceed
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();
  }
}

// Shared memory of the fused kernel for nv vectors of snb blocks.
inline size_t fused_smem(int nv, long long snb) { return (size_t)nv * (size_t)snb * 36; }

template <int WT, bool F16, int R, int NV, bool BF16X>
cudaError_t launch_fused_rnv(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int nv,
                             bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  auto kern = matvec_qx_fused_kernel<WT, F16, R, NV, BF16X>;
  FusedParams p{};
  long long total_groups = 0, min_nb = 1LL << 40, snb = 0;
  for (int i = 0; i < n; ++i) {
    total_groups += (ms[i].rows + R - 1) / R;
    const long long nb = ms[i].cols / 32;
    if (nb < min_nb) min_nb = nb;
    if (nb > snb) snb = nb;
  }
  const int ks = slices_for(total_groups, min_nb, dev.sm_count);
  const long long per_item = kWarps / ks;
  long long items = 0;
  for (int i = 0; i < n; ++i) {
    p.pr[i].q = ms[i].q;
    p.pr[i].d = ms[i].d;
    p.pr[i].rows = ms[i].rows;
    p.pr[i].nb = ms[i].cols / 32;
    p.pr[i].x = xs[i];
    p.pr[i].y = ys[i];
    p.pr[i].item0 = (int)items;
    items += ((ms[i].rows + R - 1) / R + per_item - 1) / per_item;
  }
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.nprob = n;
  p.nitems = (int)items;
  p.nv = nv;
  p.ks = ks;
  p.snb = snb;
  const size_t smem = fused_smem(nv, snb);
  if (smem > dev.smem_optin) return cudaErrorInvalidValue;
  // per device: the shared-memory attribute (raised as larger groups come) and the resident
  // CTAs per SM at each size met
  static std::mutex mu;
  static size_t set_to[64] = {};
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (set_to[dev.device] < smem) {
      const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      set_to[dev.device] = smem;
    }
    const cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, smem);
    if (err != cudaSuccess) return err;
  }
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const long long cap = (long long)per_sm * dev.sm_count;
  const long long grid = items < cap ? (items > 0 ? items : 1) : cap;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int WT, bool F16, int R, bool BF16X>
cudaError_t launch_fused_r(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int nv, bool pdl,
                           const DeviceInfo& dev, cudaStream_t stream) {
  if (nv == 1) return launch_fused_rnv<WT, F16, R, 1, BF16X>(ms, xs, ys, n, nv, pdl, dev, stream);
  if constexpr (R == 4) {
    return launch_fused_rnv<WT, F16, R, 2, BF16X>(ms, xs, ys, n, nv, pdl, dev, stream);
  } else {
    if (nv == 2) return launch_fused_rnv<WT, F16, R, 2, BF16X>(ms, xs, ys, n, nv, pdl, dev, stream);
    if (nv <= 4) return launch_fused_rnv<WT, F16, R, 4, BF16X>(ms, xs, ys, n, nv, pdl, dev, stream);
    return launch_fused_rnv<WT, F16, R, 8, BF16X>(ms, xs, ys, n, nv, pdl, dev, stream);
  }
}

// A group of problems of one weight type, passes of up to 8 vectors; rows per warp as for the
// plain launch, from the group's total rows.
template <int WT, bool BF16X>
cudaError_t launch_fused_wtype(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch,
                               bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  constexpr int R4 = WT == QMV_Q4_0 ? 4 : 2;
  long long rows = 0, min_nb = 1LL << 40;
  for (int i = 0; i < n; ++i) {
    rows += ms[i].rows;
    if (ms[i].cols / 32 < min_nb) min_nb = ms[i].cols / 32;
  }
  const int ks_max = slices_for(1, min_nb, dev.sm_count, true);
  int R = R4;
  while (R > 1 && (rows + R - 1) / R * ks_max < warps_wanted(dev.sm_count)) R /= 2;
  const size_t xsz = BF16X ? 2 : 4;
  for (int v0 = 0; v0 < batch; v0 += 8) {
    const int nv = batch - v0 < 8 ? batch - v0 : 8;
    const void* xp[kMaxFused];
    float* yp[kMaxFused];
    for (int i = 0; i < n; ++i) {
      xp[i] = static_cast<const uint8_t*>(xs[i]) + (size_t)v0 * (size_t)ms[i].cols * xsz;
      yp[i] = ys[i] + (size_t)v0 * (size_t)ms[i].rows;
    }
    const int Rp = R == 4 && nv > 2 ? 2 : R;
    const bool f16 = ms[0].scale_f16 != 0;
    cudaError_t err;
    if (f16) {
      err = Rp == 4  ? launch_fused_r<WT, true, R4, BF16X>(ms, xp, yp, n, nv, pdl, dev, stream)
            : Rp == 2 ? launch_fused_r<WT, true, 2, BF16X>(ms, xp, yp, n, nv, pdl, dev, stream)
                     : launch_fused_r<WT, true, 1, BF16X>(ms, xp, yp, n, nv, pdl, dev, stream);
    } else {
      err = Rp == 4  ? launch_fused_r<WT, false, R4, BF16X>(ms, xp, yp, n, nv, pdl, dev, stream)
            : Rp == 2 ? launch_fused_r<WT, false, 2, BF16X>(ms, xp, yp, n, nv, pdl, dev, stream)
                     : launch_fused_r<WT, false, 1, BF16X>(ms, xp, yp, n, nv, pdl, dev, stream);
    }
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace qx
}  // namespace qmv
