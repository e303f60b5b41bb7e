// decode_tc.cuh -- the decode product (1..16 bfloat16 activation vectors per pass) on the
// 5th-generation tensor core, with the quantized weights unpacked into tensor memory.
//
// What is computed (Krafla ".mlb model format v1", "Q8_0", "Q4_0", "Body"):
//   y[n][r] = sum_k d[r][k] * sum_{j<32} level[r][32k+j] * x[n][32k+j]
// level = nibble - 8 (Q4_0) or the int8 quant (Q8_0), exact in bfloat16.  The tensor core
// forms each block's dot product in float32; the rows' threads scale it (float32 FFMA) and
// add the blocks in column order.
//
// Work.  Units of 128 rows x 256 columns (a tile and a chunk), ordered problem, tile, chunk.
// The persistent CTAs (two per SM) take equal contiguous shares of the units (stream-K), so a
// tile may be split between consecutive CTAs.  A CTA that holds a whole tile stores y; the
// parts of a split tile are written to a workspace, and the CTA that finishes its part last
// (an arrival counter per split tile) adds the parts in CTA order and stores y, so the result
// does not depend on timing; it also sets the counter back to zero for the next launch.
//
// Roles (224 threads; two CTAs per SM):
//   warp 0     TMA producer: per unit, the q box(es) (128 rows x 128 bytes, 128-byte
//              swizzle), the d box (128 rows x 8 scales) and the activation box (16 vectors
//              x 256 bf16 in four 64-wide boxes, 128-byte swizzle; vectors past the batch
//              are zero-filled) into a ring slot.  The activation box is the MMA's B operand.
//   warps 1-2  MMA issuers (warp 1 also allocates the 256 tensor-memory columns): warp 1+h
//              issues, per unit, the 8 tcgen05.mma (M 128, N 16, K 16, A from tensor memory,
//              B from shared memory) of half h (blocks 4h .. 4h+3), block k accumulating into
//              columns 128+16k .. 128+16k+15.  One thread issues about one MMA per 90 cycles,
//              so the SM's four issuing warps (two CTAs) keep four streams of MMAs going.
//   warps 3-6  128 rows, thread = row.  Per unit and half (blocks 0-3, 4-7): load the row's
//              quant bytes of that half from the ring slot, read the previous unit's block
//              sums of that half from tensor memory and add d * sum into the row's
//              accumulators, unpack the quants to bf16 levels and store them to tensor memory
//              (tcgen05.st) as the next MMA's A operand.  A half's MMAs run while the rows
//              work on the other half.
// Tensor memory: A in columns 0..127 (row r in lane r, two K elements per column), block sums
// in columns 128..255.
// Every wait is bounded; a wait that runs out records QMV_E_TIMEOUT and the roles unwind.
#pragma once

#include <cstring>

#include "qmv_common.cuh"
#include "qmv_internal.h"
#include "tcgen05.cuh"

namespace qmv {
namespace dtc {

constexpr int kM = 128;                 // rows per CTA tile = MMA M = tensor-memory lanes
constexpr int kTileRows = kM;           // rows per unit
constexpr int kKS = 256;                // columns per unit
constexpr int kBlk = kKS / 32;          // blocks per unit
constexpr int kN = 16;                  // MMA N: activation vectors, zero-padded
constexpr int kMaxVec = kN;             // vectors per pass (bf16 activations)
constexpr int kMaxBatch = 8;            // vectors per pass given as hi + lo pairs (16 MMA columns)
constexpr int kMaxProblems = 8;
constexpr int kIssuers = 2;             // MMA-issuing warps, one per half unit
constexpr int kRowWarps = 4;
constexpr int kFirstRowWarp = 1 + kIssuers;  // after the producer and the MMA issuers
constexpr int kThreads = 32 * (kFirstRowWarp + kRowWarps);
constexpr int kHalfBlk = kBlk / 2;      // blocks per half unit
constexpr int kTmemCols = 256;          // A, then block sums
constexpr int kSumCol = 128;            // first block-sum column
constexpr int kXBox = 64;               // activation box width (one 128-byte swizzle span of bf16)
constexpr int kXBoxBytes = kN * 128;

template <int WT, bool F16>
struct Cfg {
  static constexpr int QROW = WT == QMV_Q4_0 ? 128 : 256;  // q bytes per row per unit
  static constexpr int NQBOX = QROW / 128;
  static constexpr int QWORDS = QROW / 4;
  static constexpr int QHALF = QWORDS / 2;                   // quant words per row per half
  static constexpr int Q_BOX = kTileRows * 128;
  static constexpr int Q_STAGE = NQBOX * Q_BOX;
  static constexpr int DROW = kBlk * (F16 ? 2 : 4);         // scale bytes per row per unit
  static constexpr int DWORDS = DROW / 4;
  static constexpr int D_STAGE = kTileRows * DROW;
  static constexpr int X_STAGE = (kKS / kXBox) * kXBoxBytes;
  static constexpr int OFF_D = Q_STAGE;                      // within a slot
  static constexpr int OFF_X = Q_STAGE + D_STAGE;            // 1024-aligned
  static constexpr int STAGE = Q_STAGE + D_STAGE + X_STAGE;  // multiple of 1024
  // ring depth: two CTAs per SM within 228 KB of shared memory (and 120 registers per
  // thread, so that two CTAs fit the register file)
  static constexpr int S = WT == QMV_Q4_0 ? (F16 ? 4 : 3) : 2;
  static constexpr int OFF_BAR = S * STAGE;
  // full[S], empty[S], afull[2], dfull[2], flush_bar, flush_done, mma_idle[kIssuers]
  static constexpr int NBARS = 2 * S + 4 + 2 + kIssuers;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;       // tensor-memory base, failed, last
  static constexpr int SMEM = 1024 + OFF_MISC + 16;
};

struct Problem {
  float* y;
  int rows;
  int nchunks;     // cols / 256
  int ntiles;      // ceil(rows / 128)
  long long unit0; // first unit of this problem
};

struct Params {
  int nprob;
  int batch;
  int xsplit;  // 1: x[i] is 16 rows of bfloat16, hi parts of the vectors in rows 0..7, lo in 8..15
  int grid;
  long long units;
  int early;  // the weights may be read before the preceding kernel has finished
  int* status;
  float* partials;              // [2 * grid][NV][kTileRows] parts of split tiles (NV: the kernel's)
  unsigned* counters;           // [grid] arrivals, zero between launches
  Problem pr[kMaxProblems];
};

struct Maps {
  CUtensorMap q[kMaxProblems];
  CUtensorMap d[kMaxProblems];
  CUtensorMap x[kMaxProblems];
};

struct Unit {
  int prob, tile, chunk;
};

__device__ __forceinline__ void unit_at(const Params& p, long long u, Unit& w) {
  int pr = 0;
  while (pr + 1 < p.nprob && u >= p.pr[pr + 1].unit0) ++pr;
  const long long local = u - p.pr[pr].unit0;
  w.prob = pr;
  w.tile = (int)(local / p.pr[pr].nchunks);
  w.chunk = (int)(local - (long long)w.tile * p.pr[pr].nchunks);
}

__device__ __forceinline__ void unit_next(const Params& p, Unit& w) {
  if (++w.chunk == p.pr[w.prob].nchunks) {
    w.chunk = 0;
    if (++w.tile == p.pr[w.prob].ntiles) {
      w.tile = 0;
      ++w.prob;
    }
  }
}

// first unit of CTA c, and the CTA whose share holds unit u
__device__ __forceinline__ long long cta_first_unit(const Params& p, long long c) { return c * p.units / p.grid; }
__device__ __forceinline__ int cta_of_unit(const Params& p, long long u) {
  return (int)(((u + 1) * p.grid + p.units - 1) / p.units - 1);
}

__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned* addr, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

// Bounded wait that gives up at once when another role has already failed.
__device__ __forceinline__ bool twait(uint64_t* bar, uint32_t parity, volatile int* failed, int* status) {
  if (*failed) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  record_status(status, QMV_E_TIMEOUT);
  *failed = 1;
  return false;
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

// One Q4_0 block (16 quant bytes in w[0..3]) to 32 exact bf16 levels in K order, two per
// 32-bit column: out[j] = (e[2j], e[2j+1]); elements 0..15 are the low nibbles of bytes
// 0..15, elements 16..31 the high nibbles.  0x4300 | n is the bfloat16 of 128 + n.
__device__ __forceinline__ void q4_block_levels(const uint32_t* w, uint32_t (&out)[16]) {
  constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u, kOffset = 0x43084308u;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t b01 = prmt(w[m], 0u, 0x4140);  // bytes 4m, 4m+1 in the low bytes of the two halves
    const uint32_t b23 = prmt(w[m], 0u, 0x4342);
    out[2 * m] = bf16x2_sub(lop_and_or(b01, kMask, kMagic), kOffset);
    out[2 * m + 1] = bf16x2_sub(lop_and_or(b23, kMask, kMagic), kOffset);
    out[8 + 2 * m] = bf16x2_sub(lop_and_or(b01 >> 4, kMask, kMagic), kOffset);
    out[9 + 2 * m] = bf16x2_sub(lop_and_or(b23 >> 4, kMask, kMagic), kOffset);
  }
}

// One Q8_0 block (32 int8 quants in w[0..7]) to 32 exact bf16 levels in K order.  In a
// 16-bit lane holding quant byte b (m = b & 0x7F, s its sign bit, q = m - 128 s):
// 0x4300 | m is the bfloat16 of 128 + m, 0x4300 | (b & 0x80) that of 128 or 256.
__device__ __forceinline__ void q8_block_levels(const uint32_t* w, uint32_t (&out)[16]) {
  constexpr uint32_t kLow7 = 0x007F007Fu, kSign = 0x00800080u, kMagic = 0x43004300u;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const uint32_t b01 = prmt(w[m], 0u, 0x4140);
    const uint32_t b23 = prmt(w[m], 0u, 0x4342);
    out[2 * m] = bf16x2_sub(lop_and_or(b01, kLow7, kMagic), lop_and_or(b01, kSign, kMagic));
    out[2 * m + 1] = bf16x2_sub(lop_and_or(b23, kLow7, kMagic), lop_and_or(b23, kSign, kMagic));
  }
}

// acc[n] += d[k] * S[k][n] over blocks k = k0 .. k0+3 in order, S read from the block-sum
// columns (block k at column 16k).
template <int NV>
__device__ __forceinline__ void add_block_sums(uint32_t tsum, int k0, const float (&dk)[kBlk], float (&acc)[NV]) {
  constexpr int G = NV <= 4 ? kHalfBlk : NV <= 8 ? 2 : 1;  // blocks per tensor-memory read batch
#pragma unroll
  for (int kb = 0; kb < kHalfBlk; kb += G) {
    uint32_t v[G][NV];
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const uint32_t a = tsum + (uint32_t)(16 * (k0 + kb + k));
      if constexpr (NV == 1) tmem_ld1(a, v[k]);
      else if constexpr (NV == 2) tmem_ld2(a, v[k]);
      else if constexpr (NV == 4) tmem_ld4(a, v[k]);
      else if constexpr (NV == 8) tmem_ld8(a, v[k]);
      else tmem_ld16(a, v[k]);
    }
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < G; ++k)
#pragma unroll
      for (int n = 0; n < NV; ++n) acc[n] = fmaf(dk[k0 + kb + k], __uint_as_float(v[k][n]), acc[n]);
  }
}

// The same with float32 activations given as bfloat16 pairs x = hi + lo: the MMA's B rows
// 0..7 hold the vectors' hi parts and rows 8..15 their lo parts, so vector n's block sum is
// S[k][n] + S[k][8 + n].
template <int NV>
__device__ __forceinline__ void add_block_sums_split(uint32_t tsum, int k0, const float (&dk)[kBlk],
                                                     float (&acc)[NV]) {
  constexpr int G = NV <= 4 ? kHalfBlk : 1;  // blocks per tensor-memory read batch
#pragma unroll
  for (int kb = 0; kb < kHalfBlk; kb += G) {
    uint32_t hi[G][NV], lo[G][NV];
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const uint32_t a = tsum + (uint32_t)(16 * (k0 + kb + k));
      if constexpr (NV == 1) {
        tmem_ld1(a, hi[k]);
        tmem_ld1(a + 8, lo[k]);
      } else if constexpr (NV == 2) {
        tmem_ld2(a, hi[k]);
        tmem_ld2(a + 8, lo[k]);
      } else if constexpr (NV == 4) {
        tmem_ld4(a, hi[k]);
        tmem_ld4(a + 8, lo[k]);
      } else {
        tmem_ld8(a, hi[k]);
        tmem_ld8(a + 8, lo[k]);
      }
    }
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < G; ++k)
#pragma unroll
      for (int n = 0; n < NV; ++n)
        acc[n] = fmaf(dk[k0 + kb + k], __uint_as_float(hi[k][n]) + __uint_as_float(lo[k][n]), acc[n]);
  }
}

template <int WT, bool F16, int NV>
__global__ void __maxnreg__(NV > 8 ? 128 : 120) decode_tc_kernel(const __grid_constant__ Maps maps,
                                                                const __grid_constant__ Params p) {
  using C = Cfg<WT, F16>;
  constexpr int S = C::S;
  constexpr int kPart = NV * kTileRows;  // floats of one part of a split tile
  // launched early without leave to read the weights meanwhile: nothing global before the wait
  if (!p.early) griddep_wait();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);  // 1024-aligned: swizzle atoms
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* afull = bars + 2 * S;  // [half]
  uint64_t* dfull = afull + 2;     // [half]
  uint64_t* flush_bar = dfull + 2;
  uint64_t* flush_done = flush_bar + 1;
  uint64_t* mma_idle = flush_done + 1;  // [issuer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const long long u0 = cta_first_unit(p, blockIdx.x);
  const long long u1 = cta_first_unit(p, (long long)blockIdx.x + 1);
  const int nunits = (int)(u1 - u0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kRowWarps + kIssuers);  // every row warp has read the slot; its MMAs are done
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&afull[h], kRowWarps);
      mbar_init(&dfull[h], 1);  // the issuer of that half
    }
    mbar_init(flush_bar, kRowWarps);
    mbar_init(flush_done, 1);
    for (int j = 0; j < kIssuers; ++j) mbar_init(&mma_idle[j], 1);
    *failed = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      Unit w;
      unit_at(p, u0, w);
      Unit deferred[S];
      int issued = 0;
      bool waited = false;
      auto load_x = [&](int s, const Unit& wx) {
        uint8_t* xs = smem + s * C::STAGE + C::OFF_X;
#pragma unroll
        for (int j = 0; j < kKS / kXBox; ++j)
          tma_load_2d_keep(xs + j * kXBoxBytes, &maps.x[wx.prob], wx.chunk * kKS + j * kXBox, 0, &full[s]);
      };
      for (int i = 0; i < nunits; ++i) {
        const int s = i % S;
        if (i >= S && !twait(&empty[s], (uint32_t)((i / S - 1) & 1), failed, p.status)) break;
        mbar_arrive_expect_tx(&full[s], (uint32_t)C::STAGE);
        uint8_t* slot = smem + s * C::STAGE;
#pragma unroll
        for (int b = 0; b < C::NQBOX; ++b)
          tma_load_2d(slot + b * C::Q_BOX, &maps.q[w.prob], w.chunk * C::QROW + b * 128, w.tile * kTileRows,
                      &full[s], pol);
        tma_load_2d(slot + C::OFF_D, &maps.d[w.prob], w.chunk * C::DROW, w.tile * kTileRows, &full[s], pol);
        if (waited) {
          load_x(s, w);
        } else {
          deferred[i] = w;
        }
        issued = i + 1;
        if (!waited && (i == S - 1 || i == nunits - 1)) {
          // weights of the first stages are in flight; activations only once the preceding
          // kernel has finished
          griddep_wait();
          griddep_launch_dependents();
          waited = true;
          for (int j = 0; j <= i; ++j) load_x(j, deferred[j]);
        }
        unit_next(p, w);
      }
      if (!waited) {
        griddep_wait();
        griddep_launch_dependents();
      }
      if (*failed) {
        // let the copies still in flight land before the shared memory is released
        for (int s = 0; s < S && s < issued; ++s) {
          const int last = issued - 1 - ((issued - 1 - s) % S);  // last stage issued into slot s
          mbar_wait_bounded(&full[last % S], (uint32_t)((last / S) & 1), 400000000LL);
        }
      }
    }
  } else if (warp < kFirstRowWarp) {
    // ------------------------------------------------------------------ MMA issuers
    const int j = warp - 1;  // issuer j: half h = j of every unit
    const int h = j;
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kM, kN);
      bool any = false;
      for (int i = 0; i < nunits; ++i) {
        const int s = i % S;
        if (!twait(&full[s], (uint32_t)((i / S) & 1), failed, p.status)) break;
        if (!twait(&afull[h], (uint32_t)(i & 1), failed, p.status)) break;
        tc_fence_after();
        const uint32_t xb = sbase + s * C::STAGE + C::OFF_X;
#pragma unroll
        for (int k = h * kHalfBlk; k < (h + 1) * kHalfBlk; ++k) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kk = 32 * k + 16 * e;  // first K element of this MMA
            const uint32_t b = xb + (uint32_t)((kk / kXBox) * kXBoxBytes + (kk % kXBox) * 2);
            tc_mma_f16_ts(tmem + kSumCol + 16 * k, tmem + 16 * k + 8 * e, smem_desc_sw128(b), idesc, e != 0);
          }
        }
        tc_commit(smem_u32(&dfull[h]));
        tc_commit(smem_u32(&empty[s]));
        any = true;
      }
      if (any) {
        // every MMA issued above has completed before the tensor memory is released
        tc_commit(smem_u32(&mma_idle[j]));
        mbar_wait_bounded(&mma_idle[j], 0u, 400000000LL);
      }
    }
  } else {
    // ------------------------------------------------------------------ rows
    const int quarter = warp & 3;  // the tensor-memory lane quarter this warp may access
    const int rt = quarter * 32 + lane;  // row within the unit
    const int sw = rt & 7;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t ta = tl;             // A columns
    const uint32_t tsum = tl + kSumCol;  // block-sum columns

    float acc[NV];
#pragma unroll
    for (int n = 0; n < NV; ++n) acc[n] = 0.f;
    uint32_t dprev[C::DWORDS];
    Unit cur, prev;
    unit_at(p, u0, cur);
    prev = cur;
    long long seg0 = u0;  // first unit of the open segment
    int flushes = 0;

    // the open segment [seg0, ue] of tile (pw.prob, pw.tile) is complete in acc: store it
    auto flush = [&](const Unit& pw, long long ue) {
      griddep_wait();  // y and the workspace are written only after the preceding kernel
      const Problem& P = p.pr[pw.prob];
      const long long t0 = P.unit0 + (long long)pw.tile * P.nchunks;  // the tile's first unit
      const int grow = pw.tile * kTileRows + rt;
      if (seg0 == t0 && ue == t0 + P.nchunks - 1) {
        if (grow < P.rows) {
#pragma unroll
          for (int n = 0; n < NV; ++n)
            if (n < p.batch) P.y[(size_t)n * P.rows + grow] = acc[n];
        }
        return;
      }
      const int me = (int)blockIdx.x;
      const int cfirst = cta_of_unit(p, t0);
      const int clast = cta_of_unit(p, t0 + P.nchunks - 1);
      // the tile is this CTA's first segment when it starts at or before the first unit
      const int myslot = 2 * me + (t0 <= u0 ? 0 : 1);
      float* mine = p.partials + (size_t)myslot * kPart;
#pragma unroll
      for (int n = 0; n < NV; ++n) mine[n * kTileRows + rt] = acc[n];
      __syncwarp();
      if (lane == 0) mbar_arrive(flush_bar);
      if (threadIdx.x == 32 * kFirstRowWarp) {
        // the CTA's parts are all written (the barrier orders them before this thread's
        // release): count this CTA's arrival at the tile
        bool last = false;
        if (twait(flush_bar, (uint32_t)(flushes & 1), failed, p.status)) {
          const unsigned before = atomic_add_acq_rel(p.counters + cfirst, 1u);
          last = (int)before + 1 == clast - cfirst + 1;
          if (last) p.counters[cfirst] = 0u;  // every part has arrived: ready for the next launch
        }
        *last_flag = last ? 1 : 0;
        mbar_arrive(flush_done);
      }
      const bool ok = twait(flush_done, (uint32_t)(flushes & 1), failed, p.status);
      ++flushes;
      if (!ok || !*last_flag) return;
      // the last part of the tile: add all parts in CTA order, QF in flight at a time
      float sum[NV];
#pragma unroll
      for (int n = 0; n < NV; ++n) sum[n] = 0.f;
      constexpr int QF = NV <= 8 ? 4 : WT == QMV_Q4_0 ? 2 : 1;  // parts in flight (registers: QF x NV)
      for (int c = cfirst; c <= clast; c += QF) {
        float v[QF][NV];
#pragma unroll
        for (int q = 0; q < QF; ++q) {
          const int cc = c + q;
          const int slot = 2 * cc + (t0 * p.grid <= (long long)cc * p.units ? 0 : 1);
          const float* part = p.partials + (size_t)slot * kPart;
#pragma unroll
          for (int n = 0; n < NV; ++n) v[q][n] = cc <= clast ? __ldcg(part + n * kTileRows + rt) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < QF; ++q)
#pragma unroll
          for (int n = 0; n < NV; ++n) sum[n] += v[q][n];
      }
      if (grow < P.rows) {
#pragma unroll
        for (int n = 0; n < NV; ++n)
          if (n < p.batch) P.y[(size_t)n * P.rows + grow] = sum[n];
      }
    };
    auto scales = [&](const uint32_t (&dw)[C::DWORDS], float (&dk)[kBlk]) {
#pragma unroll
      for (int k = 0; k < kBlk; ++k) {
        if (F16) {
          const uint32_t v = dw[k >> 1];
          dk[k] = f16_bits_to_f32((uint16_t)((k & 1) ? (v >> 16) : (v & 0xFFFFu)));
        } else {
          dk[k] = __uint_as_float(dw[k]);
        }
      }
    };
    // this row's quant words of half h of the unit in slot s
    auto load_half = [&](int s, int h, uint32_t (&w)[C::QHALF]) {
      const uint32_t qrow = sbase + s * C::STAGE + rt * 128;
      constexpr int CH = C::QHALF / 4;  // 16-byte chunks per half
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int chunk = h * CH + c;            // chunk of the row's unit bytes
        const int box = chunk / 8, cb = chunk % 8;  // 128-byte box and chunk within it
        lds128(qrow + box * C::Q_BOX + ((cb ^ sw) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      }
    };
    // the levels of half h into tensor memory: the next A operand of that half
    auto unpack_half = [&](const uint32_t (&w)[C::QHALF], int h) {
#pragma unroll
      for (int k = 0; k < kHalfBlk; ++k) {
        uint32_t lv[16];
        if (WT == QMV_Q4_0) {
          q4_block_levels(&w[4 * k], lv);
        } else {
          q8_block_levels(&w[8 * k], lv);
        }
        tmem_st16(ta + (uint32_t)(16 * (h * kHalfBlk + k)), lv);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[h]);
    };
    // block sums of half h of unit j into acc
    auto take_half = [&](int j, int h, const float (&dk)[kBlk]) -> bool {
      if (!twait(&dfull[h], (uint32_t)(j & 1), failed, p.status)) return false;
      tc_fence_after();
      if constexpr (NV <= kMaxBatch) {
        if (p.xsplit) {
          add_block_sums_split<NV>(tsum, h * kHalfBlk, dk, acc);
          return true;
        }
      }
      add_block_sums<NV>(tsum, h * kHalfBlk, dk, acc);
      return true;
    };

    int done = 0;  // units whose A has been handed to the MMA
    for (int i = 0; i < nunits; ++i) {
      const int s = i % S;
      if (!twait(&full[s], (uint32_t)((i / S) & 1), failed, p.status)) break;
      uint32_t w[C::QHALF];
      uint32_t dcur[C::DWORDS];
      load_half(s, 0, w);
      const uint32_t drow = sbase + s * C::STAGE + C::OFF_D + rt * C::DROW;
#pragma unroll
      for (int k = 0; k < C::DWORDS; k += 4) lds128(drow + 4 * k, dcur[k], dcur[k + 1], dcur[k + 2], dcur[k + 3]);
      float dk[kBlk];
      if (i > 0) scales(dprev, dk);
      // half 0: the previous unit's first-half sums free A and sums of half 0
      if (i > 0 && !take_half(i - 1, 0, dk)) break;
      unpack_half(w, 0);
      load_half(s, 1, w);
      if (i > 0) {
        if (!take_half(i - 1, 1, dk)) break;
        const long long ue = u0 + i - 1;
        if (prev.chunk == p.pr[prev.prob].nchunks - 1) {  // unit i-1 ends its tile
          flush(prev, ue);
          if (*failed) break;
#pragma unroll
          for (int n = 0; n < NV; ++n) acc[n] = 0.f;
          seg0 = ue + 1;
        }
      }
      unpack_half(w, 1);
      if (lane == 0) mbar_arrive(&empty[s]);  // every lane's loads of the slot are consumed
      ++done;
#pragma unroll
      for (int k = 0; k < C::DWORDS; ++k) dprev[k] = dcur[k];
      prev = cur;
      unit_next(p, cur);
    }
    if (done == nunits && nunits > 0 && !*failed) {
      float dk[kBlk];
      scales(dprev, dk);
      if (take_half(nunits - 1, 0, dk) && take_half(nunits - 1, 1, dk)) flush(prev, u1 - 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int WT, bool F16, int NV>
cudaError_t launch_typed(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch, bool xsplit,
                         bool pdl,
                         const DeviceInfo& dev, const Workspace& ws, cudaStream_t stream) {
  using C = Cfg<WT, F16>;
  auto kern = decode_tc_kernel<WT, F16, NV>;
  static bool ready[64] = {};
  if (dev.device < 0 || dev.device >= 64 || n < 1 || n > kMaxProblems || batch < 1 || batch > NV ||
      (xsplit && batch > kMaxBatch))
    return cudaErrorInvalidValue;
  constexpr int kPart = NV * kTileRows;
  if (!ready[dev.device]) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    // the whole carve-out for shared memory, so that two CTAs fit on an SM
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    ready[dev.device] = true;
  }
  Params p{};
  p.nprob = n;
  p.batch = batch;
  p.xsplit = xsplit ? 1 : 0;
  p.early = pdl ? 1 : 0;
  p.status = dev.status;
  p.partials = ws.partials;
  p.counters = ws.counters;
  long long units = 0;
  for (int i = 0; i < n; ++i) {
    p.pr[i].y = ys[i];
    p.pr[i].rows = (int)ms[i].rows;
    p.pr[i].nchunks = (int)(ms[i].cols / kKS);
    p.pr[i].ntiles = (int)((ms[i].rows + kTileRows - 1) / kTileRows);
    p.pr[i].unit0 = units;
    units += (long long)p.pr[i].ntiles * p.pr[i].nchunks;
  }
  // two CTAs per SM: shared memory (<= 113 KB each), registers (at most 128 a thread: the 14
  // warps put four on some sub-partition, whose 16K registers then hold 4 x 32 x 128) and tensor
  // memory (256 columns each) hold two.  (The occupancy query reports one CTA per SM for any
  // kernel that allocates tensor memory, so it is not used here.)  Within the workspace's
  // counters and parts, and no more CTAs than units.
  static_assert(2 * (C::SMEM + 1024) <= 233472, "two CTAs per SM by shared memory");
  static_assert(2 * kTmemCols <= 512, "two CTAs per SM by tensor memory");
  long long cap = 2LL * dev.sm_count;
  if (cap > ws.max_counters) cap = ws.max_counters;
  const long long by_parts = (long long)(ws.max_partial_floats / ((size_t)2 * kPart));
  if (cap > by_parts) cap = by_parts;
  if (cap > units) cap = units;
  const int grid = (int)cap;
  p.units = units;
  p.grid = grid;

  Maps maps;
  memset(&maps, 0, sizeof(maps));
  for (int i = 0; i < n; ++i) {
    const MatrixRef& m = ms[i];
    const uint64_t qrow = (WT == QMV_Q4_0) ? (uint64_t)m.cols / 2 : (uint64_t)m.cols;
    const uint64_t drow = (uint64_t)(m.cols / 32) * (F16 ? 2 : 4);
    cudaError_t err = encode_tmap_2d(&maps.q[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, m.q, qrow, (uint64_t)m.rows, qrow,
                                     128, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    err = encode_tmap_2d(&maps.d[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, m.d, drow, (uint64_t)m.rows, drow, C::DROW,
                         kTileRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
    err = encode_tmap_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xs[i], (uint64_t)m.cols,
                         (uint64_t)(xsplit ? kN : batch),
                         (uint64_t)m.cols * 2, kXBox, kN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
  }

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  // always a programmatic dependent: the CTAs start during the preceding kernel's tail; without
  // pdl they wait for it before their first global access (p.early = 0)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

template <int WT, bool F16>
cudaError_t launch_wtype(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch, bool xsplit,
                         bool pdl, const DeviceInfo& dev, const Workspace& ws, cudaStream_t stream) {
  if (batch <= 1) return launch_typed<WT, F16, 1>(ms, xs, ys, n, batch, xsplit, pdl, dev, ws, stream);
  if (batch <= 2) return launch_typed<WT, F16, 2>(ms, xs, ys, n, batch, xsplit, pdl, dev, ws, stream);
  if (batch <= 4) return launch_typed<WT, F16, 4>(ms, xs, ys, n, batch, xsplit, pdl, dev, ws, stream);
  if (batch <= 8) return launch_typed<WT, F16, 8>(ms, xs, ys, n, batch, xsplit, pdl, dev, ws, stream);
  return launch_typed<WT, F16, 16>(ms, xs, ys, n, batch, xsplit, pdl, dev, ws, stream);
}

cudaError_t launch_q4(const MatrixRef*, const void* const*, float* const*, int, int, bool, bool, const DeviceInfo&,
                      const Workspace&, cudaStream_t);
cudaError_t launch_q8(const MatrixRef*, const void* const*, float* const*, int, int, bool, bool, const DeviceInfo&,
                      const Workspace&, cudaStream_t);

}  // namespace dtc
}  // namespace qmv
