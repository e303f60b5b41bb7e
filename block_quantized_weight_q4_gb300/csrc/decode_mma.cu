// decode_mma.cu -- the decode product (batch 1..8 per pass) for cols % 256 == 0.
//
// What is computed (Krafla ".mlb model format v1", "Q8_0", "Q4_0", "Body"):
//   y[n][r] = sum_k d[r][k] * sum_{j<32} level[r][32k+j] * x[n][32k+j]
// with level = nibble - 8 (Q4_0) or the int8 quant (Q8_0), d the block's scale.
//
// How (one warp = one tile of 16 rows x a slice of the columns):
//   * Weight stream.  Each warp owns a ring of S shared-memory stages.  A stage holds 16
//     rows x 256 weights of q plus their 8 scales per row; the 32 lanes each issue one
//     cp.async.bulk per stage (lanes 0-15 the q runs of rows 0-15, lanes 16-31 their scale
//     runs), completing on the stage's mbarrier.  S-1 stages are always in flight.
//   * Unpack.  ldmatrix hands thread (g = lane/4, t = lane%4) the 4 quant bytes 4t..4t+3 of
//     a block for row g and for row g+8.  They become exact bfloat16 levels in registers
//     (Q4_0: 0x4300|nibble = 128+n, minus 136; Q8_0: via the float32 2^23 trick).
//   * Block dot.  Per block, two m16n8k16 bf16 MMAs (elements 0-15 and 16-31 of the block)
//     into a zeroed f32 fragment give sum_j level*x for 16 rows x 8 activation vectors.
//     Inside an MMA the k order is permuted (slot 2t <-> element 4t, 2t+1 <-> 4t+2,
//     2t+8 <-> 4t+1, 2t+9 <-> 4t+3); the B fragment (x) uses the same permutation.
//   * Scale and accumulate.  acc += d[row][block] * fragment, in float32 FFMA.
//   * Split-K.  The warps of a CTA that share a tile add their partial sums through shared
//     memory in a fixed order; one warp writes y.
// f32 activations are split x = hi + lo (two bfloat16s, hi = RN(x)) and take two MMAs,
// which keeps 16 significant bits of x.
#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {

namespace {

constexpr int kWarps = 4;     // warps per CTA
constexpr int kTK = 256;      // weights per stage and row
constexpr int kBlocksPerStage = kTK / 32;

template <int WT, bool F16>
struct Cfg {
  static constexpr int QROW = (WT == QMV_Q4_0) ? kTK / 2 : kTK;  // q bytes per row per stage
  static constexpr int QPITCH = QROW + 16;                       // padded: conflict-free ldmatrix
  static constexpr int DROW = kBlocksPerStage * (F16 ? 2 : 4);   // scale bytes per row per stage
  static constexpr int STAGE_BYTES = 16 * QPITCH + 16 * DROW;
  static constexpr int S = (WT == QMV_Q4_0) ? 6 : 4;             // ring depth
  static constexpr int WARP_BYTES = S * STAGE_BYTES;
  static constexpr int RED_BYTES = kWarps * 16 * 8 * 4;
  static constexpr int SMEM_BYTES = kWarps * WARP_BYTES + RED_BYTES + kWarps * S * 8;
};

struct Params {
  const uint8_t* q;
  const uint8_t* d;
  const void* x;
  float* y;
  int64_t rows;
  int64_t cols;
  int batch;    // 1..8
  int64_t ntiles;
  int ks;       // k-slices per tile (1, 2, 4)
  int* status;  // per-device status word
};

// B fragments (x) for one 16-element half of block kb, batch vector n = g, permuted to
// match the A fragment's k order.
template <bool XBF16>
__device__ __forceinline__ void load_b(const Params& p, int g, int t, int64_t kb, int half, uint32_t (&bh)[2],
                                       uint32_t (&bl)[2]) {
  bh[0] = bh[1] = bl[0] = bl[1] = 0u;
  if (g >= p.batch) return;
  const int64_t off = (int64_t)g * p.cols + kb * 32 + half * 16 + 4 * t;
  if (XBF16) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.x) + off));
    bh[0] = prmt(v.x, v.y, 0x5410);  // (e0, e2)
    bh[1] = prmt(v.x, v.y, 0x7632);  // (e1, e3)
  } else {
    const float4 v = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.x) + off));
    bh[0] = pack_bf16x2(v.x, v.z);
    bh[1] = pack_bf16x2(v.y, v.w);
    bl[0] = pack_bf16x2(v.x - __uint_as_float(bh[0] << 16), v.z - __uint_as_float(bh[0] & 0xFFFF0000u));
    bl[1] = pack_bf16x2(v.y - __uint_as_float(bh[1] << 16), v.w - __uint_as_float(bh[1] & 0xFFFF0000u));
  }
}

template <int WT, bool F16, bool XBF16>
__global__ void __launch_bounds__(kWarps * 32) matvec_mma_kernel(const Params p) {
  using C = Cfg<WT, F16>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;

  uint8_t* ring = smem + warp * C::WARP_BYTES;
  float* red = reinterpret_cast<float*>(smem + kWarps * C::WARP_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * C::WARP_BYTES + C::RED_BYTES) + warp * C::S;

  const int tiles_per_cta = kWarps / p.ks;
  const int tile_local = warp / p.ks;
  const int kslice = warp % p.ks;
  const int64_t tile = (int64_t)blockIdx.x * tiles_per_cta + tile_local;
  const bool active = tile < p.ntiles;
  const int64_t row0 = tile * 16;

  const int64_t nchunks = p.cols / kTK;
  const int64_t c_begin = kslice * nchunks / p.ks;
  const int64_t c_end = (kslice + 1) * nchunks / p.ks;
  const int niter = active ? (int)(c_end - c_begin) : 0;

  const int64_t nblk = p.cols / 32;
  const int64_t qrow_bytes = (WT == QMV_Q4_0) ? p.cols / 2 : p.cols;
  const int nvalid = active ? (p.rows - row0 < 16 ? (int)(p.rows - row0) : 16) : 0;
  const uint32_t stage_tx = (uint32_t)nvalid * (C::QROW + C::DROW);

  if (lane == 0) {
    for (int s = 0; s < C::S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t pol = l2_policy_evict_first();
  const int my_row = lane & 15;
  const bool my_valid = my_row < nvalid;

  // issue chunk (c_begin + i) into stage i % S
  auto issue = [&](int i) {
    const int s = i % C::S;
    uint8_t* st = ring + s * C::STAGE_BYTES;
    const int64_t c = c_begin + i;
    if (lane == 0) mbar_arrive_expect_tx(&bars[s], stage_tx);
    __syncwarp();
    fence_proxy_async_smem();
    if (my_valid) {
      const int64_t r = row0 + my_row;
      if (lane < 16) {
        bulk_copy_g2s(st + my_row * C::QPITCH, p.q + r * qrow_bytes + c * C::QROW, C::QROW, &bars[s], pol);
      } else {
        bulk_copy_g2s(st + 16 * C::QPITCH + my_row * C::DROW,
                      p.d + (r * nblk + c * kBlocksPerStage) * (F16 ? 2 : 4), C::DROW, &bars[s], pol);
      }
    }
  };

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int pre = niter < C::S - 1 ? niter : C::S - 1;
  for (int i = 0; i < pre; ++i) issue(i);

  // ldmatrix row address for this lane: matrix m = lane/8 covers rows (m&1)*8 .. +7
  const int lm = lane >> 3;
  const int lrow = (lane & 7) + ((lm & 1) << 3);
  const int lsub = lm >> 1;  // which 16-byte chunk of the pair

  bool failed = false;
  for (int it = 0; it < niter; ++it) {
    if (it + C::S - 1 < niter) issue(it + C::S - 1);
    const int s = it % C::S;
    if (!mbar_wait_bounded(&bars[s], (uint32_t)(it / C::S) & 1u)) {
      record_status(p.status, QMV_E_TIMEOUT);
      // drain this warp's other copies in flight (bounded), then stop
      const int issued = (it + C::S - 1 < niter) ? it + C::S : niter;
      for (int j = it + 1; j < issued; ++j) mbar_wait_bounded(&bars[j % C::S], (uint32_t)(j / C::S) & 1u);
      failed = true;
      break;
    }
    const uint8_t* st = ring + s * C::STAGE_BYTES;
    const uint32_t qbase = smem_u32(st) + lrow * C::QPITCH + lsub * 16;
    const uint8_t* dst = st + 16 * C::QPITCH;

    // scales of rows g and g+8 for the 8 blocks of this stage, as float32
    float dg[kBlocksPerStage], dh[kBlocksPerStage];
    if (F16) {
      const uint4 a = *reinterpret_cast<const uint4*>(dst + g * C::DROW);
      const uint4 b = *reinterpret_cast<const uint4*>(dst + (g + 8) * C::DROW);
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
      const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        dg[2 * k] = f16_bits_to_f32((uint16_t)(wa[k] & 0xFFFF));
        dg[2 * k + 1] = f16_bits_to_f32((uint16_t)(wa[k] >> 16));
        dh[2 * k] = f16_bits_to_f32((uint16_t)(wb[k] & 0xFFFF));
        dh[2 * k + 1] = f16_bits_to_f32((uint16_t)(wb[k] >> 16));
      }
    } else {
      const float4* a = reinterpret_cast<const float4*>(dst + g * C::DROW);
      const float4* b = reinterpret_cast<const float4*>(dst + (g + 8) * C::DROW);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float4 u = a[k], v = b[k];
        dg[4 * k] = u.x; dg[4 * k + 1] = u.y; dg[4 * k + 2] = u.z; dg[4 * k + 3] = u.w;
        dh[4 * k] = v.x; dh[4 * k + 1] = v.y; dh[4 * k + 2] = v.z; dh[4 * k + 3] = v.w;
      }
    }

    const int64_t kb0 = (c_begin + it) * kBlocksPerStage;
    if (WT == QMV_Q4_0) {
#pragma unroll
      for (int bp = 0; bp < kBlocksPerStage / 2; ++bp) {
        uint32_t w[4];  // row g blk 2bp, row g+8 blk 2bp, row g blk 2bp+1, row g+8 blk 2bp+1
        ldmatrix_x4(w[0], w[1], w[2], w[3], qbase + bp * 32);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kbl = 2 * bp + h;
          uint32_t ag[4], ah[4];
          q4_word_to_bf16_levels(w[2 * h], ag[0], ag[1], ag[2], ag[3]);
          q4_word_to_bf16_levels(w[2 * h + 1], ah[0], ah[1], ah[2], ah[3]);
          uint32_t bh0[2], bl0[2], bh1[2], bl1[2];
          load_b<XBF16>(p, g, t, kb0 + kbl, 0, bh0, bl0);
          load_b<XBF16>(p, g, t, kb0 + kbl, 1, bh1, bl1);
          float c[4] = {0.f, 0.f, 0.f, 0.f};
          // elements 0..15 (low nibbles): A = (lo0,lo2),(lo1,lo3) of rows g / g+8
          mma_bf16_16816(c, ag[0], ah[0], ag[2], ah[2], bh0[0], bh0[1], c);
          // elements 16..31 (high nibbles)
          mma_bf16_16816(c, ag[1], ah[1], ag[3], ah[3], bh1[0], bh1[1], c);
          if (!XBF16) {
            mma_bf16_16816(c, ag[0], ah[0], ag[2], ah[2], bl0[0], bl0[1], c);
            mma_bf16_16816(c, ag[1], ah[1], ag[3], ah[3], bl1[0], bl1[1], c);
          }
          acc[0] = fmaf(dg[kbl], c[0], acc[0]);
          acc[1] = fmaf(dg[kbl], c[1], acc[1]);
          acc[2] = fmaf(dh[kbl], c[2], acc[2]);
          acc[3] = fmaf(dh[kbl], c[3], acc[3]);
        }
      }
    } else {
#pragma unroll
      for (int kbl = 0; kbl < kBlocksPerStage; ++kbl) {
        uint32_t w[4];  // row g half 0, row g+8 half 0, row g half 1, row g+8 half 1
        ldmatrix_x4(w[0], w[1], w[2], w[3], qbase + kbl * 32);
        uint32_t ag0[2], ah0[2], ag1[2], ah1[2];
        q8_word_to_bf16_levels(w[0], ag0[0], ag0[1]);
        q8_word_to_bf16_levels(w[1], ah0[0], ah0[1]);
        q8_word_to_bf16_levels(w[2], ag1[0], ag1[1]);
        q8_word_to_bf16_levels(w[3], ah1[0], ah1[1]);
        uint32_t bh0[2], bl0[2], bh1[2], bl1[2];
        load_b<XBF16>(p, g, t, kb0 + kbl, 0, bh0, bl0);
        load_b<XBF16>(p, g, t, kb0 + kbl, 1, bh1, bl1);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16_16816(c, ag0[0], ah0[0], ag0[1], ah0[1], bh0[0], bh0[1], c);
        mma_bf16_16816(c, ag1[0], ah1[0], ag1[1], ah1[1], bh1[0], bh1[1], c);
        if (!XBF16) {
          mma_bf16_16816(c, ag0[0], ah0[0], ag0[1], ah0[1], bl0[0], bl0[1], c);
          mma_bf16_16816(c, ag1[0], ah1[0], ag1[1], ah1[1], bl1[0], bl1[1], c);
        }
        acc[0] = fmaf(dg[kbl], c[0], acc[0]);
        acc[1] = fmaf(dg[kbl], c[1], acc[1]);
        acc[2] = fmaf(dh[kbl], c[2], acc[2]);
        acc[3] = fmaf(dh[kbl], c[3], acc[3]);
      }
    }
    __syncwarp();
  }

  // split-K: partials to shared memory, fixed-order sum, coalesced store of y
  float* my = red + warp * 128;  // [16 rows][8 vectors]
  my[g * 8 + 2 * t] = acc[0];
  my[g * 8 + 2 * t + 1] = acc[1];
  my[(g + 8) * 8 + 2 * t] = acc[2];
  my[(g + 8) * 8 + 2 * t + 1] = acc[3];
  __syncthreads();
  if (active && kslice == 0 && !failed) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = i * 32 + lane;
      const int n = v >> 4;
      const int r = v & 15;
      if (n < p.batch && r < nvalid) {
        float s = 0.f;
        for (int k = 0; k < p.ks; ++k) s += red[(warp + k) * 128 + r * 8 + n];
        p.y[(int64_t)n * p.rows + row0 + r] = s;
      }
    }
  }
}

template <int WT, bool F16, bool XBF16>
cudaError_t launch_typed(const Params& p, int grid, int dev, cudaStream_t stream) {
  using C = Cfg<WT, F16>;
  auto kern = matvec_mma_kernel<WT, F16, XBF16>;
  static bool attr_set[64] = {};  // per device: raise the dynamic shared memory limit once
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  kern<<<grid, kWarps * 32, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool matvec_mma_supported(const MatrixRef& m) { return m.cols % kTK == 0; }

cudaError_t launch_matvec_mma(const MatrixRef& m, const void* x, bool x_bf16, float* y, int batch,
                              const DeviceInfo& dev, cudaStream_t stream) {
  Params p;
  p.q = m.q;
  p.d = m.d;
  p.x = x;
  p.y = y;
  p.rows = m.rows;
  p.cols = m.cols;
  p.batch = batch;
  p.status = dev.status;
  p.ntiles = (m.rows + 15) / 16;
  const int64_t nchunks = m.cols / kTK;
  // enough warps in flight to cover HBM latency: split the columns while tiles are few
  const int64_t target = (int64_t)dev.sm_count * 8;
  int ks = 1;
  while (ks < kWarps && p.ntiles * ks < target && nchunks >= 2 * ks) ks *= 2;
  p.ks = ks;
  const int64_t tiles_per_cta = kWarps / ks;
  const int grid = (int)((p.ntiles + tiles_per_cta - 1) / tiles_per_cta);
  if (m.wtype == QMV_Q4_0) {
    if (m.scale_f16) return x_bf16 ? launch_typed<QMV_Q4_0, true, true>(p, grid, dev.device, stream)
                                   : launch_typed<QMV_Q4_0, true, false>(p, grid, dev.device, stream);
    return x_bf16 ? launch_typed<QMV_Q4_0, false, true>(p, grid, dev.device, stream)
                  : launch_typed<QMV_Q4_0, false, false>(p, grid, dev.device, stream);
  }
  if (m.scale_f16) return x_bf16 ? launch_typed<QMV_Q8_0, true, true>(p, grid, dev.device, stream)
                                 : launch_typed<QMV_Q8_0, true, false>(p, grid, dev.device, stream);
  return x_bf16 ? launch_typed<QMV_Q8_0, false, true>(p, grid, dev.device, stream)
                : launch_typed<QMV_Q8_0, false, false>(p, grid, dev.device, stream);
}

}  // namespace qmv
