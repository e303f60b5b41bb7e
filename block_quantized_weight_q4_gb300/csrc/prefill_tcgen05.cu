// prefill_tcgen05.cu -- the batched product Y = X W^T for 16..128 activation vectors per pass
// on the 5th-generation tensor core.
//
// What is computed (Krafla ".mlb model format v1", "Q8_0", "Q4_0", "Body"): for each row r
// and vector n, y[n][r] = sum_c w[r][c] * x[n][c], where each weight w = fl32(level * d) is
// the exact dequantized value (as qmv_dequant forms it).  The tensor core takes bfloat16
// operands, so each weight enters it as two bfloat16 parts: hi = RN_bf16(w) and
// lo = RN_bf16(w - hi), and every 16-column step issues two MMAs into the same float32
// accumulator, one with hi and one with lo.  For Q4_0 with f16 scales hi + lo equals w
// exactly (w has at most 15 significant bits, hi takes 8 and w - hi fits in the other 7); in
// the other formats the part lost is below 2^-17 |w|.  A single bfloat16 rounding of w (the
// "bf16 weights" variant, one MMA per step) loses up to 2^-9 |w| per term, which is more than
// a 1e-3 * sum |w x| tolerance allows when one term dominates an output; that variant is kept
// for callers that ask for it.
//
// One CTA owns 128 rows (the MMA's M) over all columns, or, when the matrix has fewer
// 128-row tiles than the GPU has SMs, over one of ksplit ranges of its columns (split-K: the
// ksplit CTAs of a tile each write their 128 x N partial product to the stream's prefill
// workspace and count their arrival on the tile's counter; the last to arrive adds the parts
// in split order, stores y and resets the counter, so the result does not depend on timing).
// The activation vectors are the MMA's N (their count rounded up to 16).  Roles:
//   warp 0     TMA producer of the raw stages (128 rows x 256 weights of q, 128 x 8 scales).
//   warp 18    TMA producer of the X stages (N x 64 bf16, 128-byte swizzle); a stage's slot is
//              free once the MMAs that read it complete, and the weight loads must not wait
//              for that, hence a producer of their own.
//   warp 1     allocates tensor memory (128 lanes x 512 columns: two f32 accumulators of 128
//              columns, then a ring of bf16-weight stages: 4 stages of 64 columns, hi then lo
//              parts, or 8 stages of 32 columns with bf16 weights).
//   warps 1, 19  lane 0 issues, per 64-column stage (warp 1 the even ones into accumulator 0,
//              warp 19 the odd ones into accumulator 1), four tcgen05.mma (M 128, N, K 16,
//              bf16 in, f32 accumulate) with the hi parts and four with the lo parts (or four
//              with bf16 weights), A from the weight stage in tensor memory and B from the X
//              stage in shared memory, then commits to the stage's "empty" barriers; after its
//              last stage, to "accumulator full".  One issuing thread could not keep up: each
//              instruction costs it tens of cycles while the tensor core finishes a stage in
//              fewer.
//   warps 2-17 dequantize, in two groups of eight (warps 2-9 and 10-17) that take turns
//              with the pairs of 64-column stages: thread (row, half) of a group turns one
//              32-weight block of its row per stage into 32 bf16 weights (or their hi and lo
//              parts) and stores them (tcgen05.st) to its row's tensor-memory lane, where the
//              MMA reads them, so the weights cross shared memory only in their quantized
//              form.  One pass of waits per pair of stages (per-stage synchronisation, not the
//              arithmetic, set the pace when every stage had its own); two groups keep four
//              warps per scheduler busy.  Then they read the accumulators from tensor memory
//              (each warp its 32-lane quarter and a quarter of the columns) and store y, or,
//              for a split tile, the CTA's part (vector-major) for the last CTA to add.
// Every wait is bounded; a wait that runs out records QMV_E_TIMEOUT and the roles unwind.
#include "qmv_common.cuh"
#include "qmv_internal.h"
#include "tcgen05.cuh"

namespace qmv {

namespace {

constexpr int kPM = 128;      // rows of W per CTA tile = MMA M = tensor-memory lanes
constexpr int kKB = 64;       // columns per MMA stage: one 128-byte swizzle span of bf16
constexpr int kRawK = 256;    // columns per raw (quantized) stage
constexpr int kMaxXS = 16;    // deepest X ring (its depth is set per launch by the batch)
constexpr int kRS = 4;        // ring depth of the raw stages
constexpr int kDeqWarps = 16;  // dequantize (two groups of 8); the first group drains the accumulators
constexpr int kXWarp = 2 + kDeqWarps;  // the X-stage producer
constexpr int kMmaWarp2 = 3 + kDeqWarps;  // the second MMA issuer (odd stages)
constexpr int kThreads = 32 * (4 + kDeqWarps);
constexpr int kMaxN = 128;    // activation vectors per pass
constexpr int kMaxKS = 8;     // deepest ring of weight stages in tensor memory
constexpr int kAccCol = 0;    // accumulators: columns 0..127 (even stages), 128..255 (odd stages)
constexpr int kACol = 256;    // weight ring from column 256 (128 lanes x 64 bf16 per part of a stage)
constexpr int kTmemCols = 512;
// ring of weight stages in tensor memory: HILO (hi and lo parts, 64 columns per stage) 4
// stages, bf16 weights (32 columns per stage) 8; a multiple of 4, since the two dequantize
// groups take turns with pairs of stages
template <bool HILO>
struct Ring {
  static constexpr int kStageCols = HILO ? 64 : 32;
  static constexpr int kKS = HILO ? 4 : 8;
  static_assert(kACol + kStageCols * kKS <= kTmemCols && kKS <= kMaxKS && kKS % 4 == 0, "tensor memory");
};

template <int WT, bool F16>
struct PCfg {
  static constexpr int QRAW_ROW = (WT == QMV_Q4_0) ? kRawK / 2 : kRawK;  // q bytes per row per raw stage
  static constexpr int NQBOX = QRAW_ROW / 128;                           // 128-byte q boxes per raw stage
  static constexpr int Q_RAW = kPM * QRAW_ROW;
  static constexpr int ESZ = F16 ? 2 : 4;
  static constexpr int DROW = (kRawK / 32) * ESZ;                        // scale bytes per row per raw stage
  static constexpr int D_RAW = kPM * DROW;
  static constexpr int OFF_Q = 0;  // raw ring, then scales, barriers, flags, then the X ring
  static constexpr int OFF_D = OFF_Q + kRS * Q_RAW;
  static constexpr int OFF_BAR = OFF_D + kRS * D_RAW;
  // barriers: raw_full[kRS], raw_empty[kRS], a_full[kMaxKS], empty[kMaxKS], x_full[kMaxXS],
  // x_empty[kMaxXS], acc_full
  static constexpr int NBARS = 2 * kRS + 2 * kMaxKS + 2 * kMaxXS + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;  // tensor-memory base, failure and last flags
  static constexpr int OFF_X = (OFF_MISC + 16 + 1023) / 1024 * 1024;  // X ring (1024-aligned stages)
  // shared memory of a launch with xs X stages of npad vectors
  static constexpr int smem_bytes(int xs, int npad) { return 1024 + OFF_X + xs * npad * 128; }
  static_assert(smem_bytes(4, kMaxN) <= 227 * 1024, "shared memory of one CTA");
};

struct PParams {
  float* y;
  int rows;
  int cols;
  int batch;  // vectors in this pass (1..128)
  int npad;   // batch rounded up to 16
  int* status;
  int xs;              // X ring depth (2..kMaxXS, even)
  int ksplit;          // column ranges per tile (1: no workspace used)
  unsigned* counters;  // per tile arrival counters, zero between launches
  float* parts;        // per (tile, split): npad x 128 partial sums, vector-major
  int early;           // the weights may be read before the preceding kernel has finished
};

__device__ __forceinline__ unsigned atomic_add_acq_rel_u32(unsigned* addr, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void epilogue_barrier() {  // the dequantize warps
  asm volatile("bar.sync 1, %0;" ::"r"(32 * kDeqWarps) : "memory");
}

// fl32(a * d) and fl32(b * d) (one packed float32 multiply) rounded to a bfloat16 pair,
// a in the low half.
__device__ __forceinline__ uint32_t scale2_bf16(float a, float b, float d) {
  float ra, rb;
  asm("{\n\t.reg .b64 va, vd, vr;\n\t"
      "mov.b64 va, {%2, %3};\n\t"
      "mov.b64 vd, {%4, %4};\n\t"
      "mul.rn.f32x2 vr, va, vd;\n\t"
      "mov.b64 {%0, %1}, vr;\n\t}"
      : "=f"(ra), "=f"(rb)
      : "f"(a), "f"(b), "f"(d));
  return pack_bf16x2(ra, rb);
}

// An IEEE-half level pair (exact small integers) times d, as bfloat16: RN(fl32(level * d)).
__device__ __forceinline__ uint32_t scale_half_levels(uint32_t h2, float d) {
  return scale2_bf16(__half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16))), d);
}

// One Q4_0 block (quant bytes in w[0..3], byte j = word j/4 bits 8(j%4)) to 32 bf16 weights
// RN(fl32(level * d)) in element order: out[0..7] elements 0..15 (low nibbles of bytes
// 0..15), out[8..15] elements 16..31 (high nibbles).  The levels are formed as exact halves
// (q4_word_to_f16_levels) and widened to float32 exactly.
__device__ __forceinline__ void q4_block_to_bf16(const uint32_t (&w)[4], float d, uint32_t (&out)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo01, lo23, hi01, hi23;
    q4_word_to_f16_levels(w[i], lo01, lo23, hi01, hi23);
    out[2 * i] = scale_half_levels(lo01, d);          // elements 4i, 4i+1
    out[2 * i + 1] = scale_half_levels(lo23, d);      // 4i+2, 4i+3
    out[8 + 2 * i] = scale_half_levels(hi01, d);      // 16+4i, 16+4i+1
    out[8 + 2 * i + 1] = scale_half_levels(hi23, d);  // 16+4i+2, 16+4i+3
  }
}

// An IEEE-half scale d (as float32) as two bfloat16 parts, each in both halves of a word:
// hi = RN_bf16(d) and lo = d - hi.  d has at most 11 significant bits, so lo has at most 3
// and is itself a bfloat16 (exact).  A scale that is not finite keeps lo = 0.
__device__ __forceinline__ void split_half_scale(float d, uint32_t& hi2, uint32_t& lo2) {
  hi2 = pack_bf16x2(d, d);
  const float lo = isfinite(d) ? d - __uint_as_float(hi2 << 16) : 0.0f;
  lo2 = pack_bf16x2(lo, lo);
}

__device__ __forceinline__ uint32_t bf16x2_mul_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_fma_rn(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// A bfloat16 level pair (exact integers, |level| <= 8) times the split scale: level * lo has
// at most 3 + 3 significant bits, so it is exact in bfloat16, and the fused multiply-add
// rounds level * hi + level * lo = level * d once: RN_bf16(level * d), which equals
// RN_bf16(fl32(level * d)) since level * d (at most 4 + 11 bits) is exact in float32.
__device__ __forceinline__ uint32_t scale_bf16_levels(uint32_t l2, uint32_t hi2, uint32_t lo2) {
  return bf16x2_fma_rn(l2, hi2, bf16x2_mul_rn(l2, lo2));
}

// One Q4_0 block with an IEEE-half scale (split by split_half_scale) to the same 32 bfloat16
// weights as q4_block_to_bf16, from exact bfloat16 levels (q4_word_to_bf16_levels) in two
// packed bfloat16 operations per pair instead of two widenings, a multiply and a narrowing.
__device__ __forceinline__ void q4_block_to_bf16_split(const uint32_t (&w)[4], uint32_t hi2, uint32_t lo2,
                                                       uint32_t (&out)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo01, lo23, hi01, hi23;
    q4_word_to_bf16_levels(w[i], lo01, lo23, hi01, hi23);
    out[2 * i] = scale_bf16_levels(lo01, hi2, lo2);
    out[2 * i + 1] = scale_bf16_levels(lo23, hi2, lo2);
    out[8 + 2 * i] = scale_bf16_levels(hi01, hi2, lo2);
    out[8 + 2 * i + 1] = scale_bf16_levels(hi23, hi2, lo2);
  }
}

// One Q8_0 block (32 int8 quants in w[0..7]) to 32 bf16 weights RN(fl32(q * d)), in order:
// 0x4B000000 | (q + 128) is 2^23 + q + 128, minus 2^23 + 128 gives q exactly (packed pairs).
__device__ __forceinline__ void q8_block_to_bf16(const uint32_t (&w)[8], float d, uint32_t (&out)[16]) {
  const float bias = 8388736.0f;  // 2^23 + 128
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t u = w[i] ^ 0x80808080u;  // q + 128 per byte
    const float f0 = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7440)), bias);
    const float f1 = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7441)), bias);
    const float f2 = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7442)), bias);
    const float f3 = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7443)), bias);
    out[2 * i] = scale2_bf16(f0, f1, d);
    out[2 * i + 1] = scale2_bf16(f2, f3, d);
  }
}

// ---------------------------------------------------------------- hi and lo parts
// hi = RN_bf16(v) with finite values beyond the bfloat16 range (and infinities) saturated to
// the largest finite bfloat16, so that v - hi stays meaningful; lo = RN_bf16(v - hi).  v - hi is
// exact in float32 (hi is v rounded to fewer bits, within a factor of two of v).  An infinite v
// gives hi = +-max and lo = +-inf, a NaN gives NaN in both, so hi x + lo x follows v x.
__device__ __forceinline__ void split2_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.satfinite.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(b), "f"(a));
  float ra, rb;
  asm("{\n\t.reg .b64 va, vh, vr;\n\t"
      "mov.b64 va, {%2, %3};\n\t"
      "mov.b64 vh, {%4, %5};\n\t"
      "sub.rn.f32x2 vr, va, vh;\n\t"
      "mov.b64 {%0, %1}, vr;\n\t}"
      : "=f"(ra), "=f"(rb)
      : "f"(a), "f"(b), "f"(__uint_as_float(hi << 16)), "f"(__uint_as_float(hi & 0xFFFF0000u)));
  lo = pack_bf16x2(ra, rb);
}

// fl32(a * d), fl32(b * d) (one packed float32 multiply) as hi and lo bfloat16 pairs.
__device__ __forceinline__ void scale2_hilo(float a, float b, float d, uint32_t& hi, uint32_t& lo) {
  float ra, rb;
  asm("{\n\t.reg .b64 va, vd, vr;\n\t"
      "mov.b64 va, {%2, %3};\n\t"
      "mov.b64 vd, {%4, %4};\n\t"
      "mul.rn.f32x2 vr, va, vd;\n\t"
      "mov.b64 {%0, %1}, vr;\n\t}"
      : "=f"(ra), "=f"(rb)
      : "f"(a), "f"(b), "f"(d));
  split2_bf16(ra, rb, hi, lo);
}

__device__ __forceinline__ uint32_t bf16x2_add_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// A bfloat16 level pair l (exact integers, |l| <= 8) times an IEEE-half scale d split as
// d = dh + dl (dh = RN_bf16(d), dl exact with at most 3 significant bits; split_half_scale):
//   m  = l * dl                (at most 7 bits: exact)
//   hi = RN_bf16(l * dh + m)   = RN_bf16(l * d)
//   t  = l * dh - hi           (exact: a multiple of ulp(dh) of magnitude below 16 ulp(dh))
//   lo = t + m                 = l * d - hi (exact: w = l * d has at most 15 significant bits,
//                               hi the leading 8, so w - hi fits in bfloat16's 8)
// so hi + lo = l * d exactly.  Four packed bfloat16 operations per pair.
__device__ __forceinline__ void scale_bf16_levels_hilo(uint32_t l2, uint32_t hi2, uint32_t lo2, uint32_t& h,
                                                       uint32_t& l) {
  const uint32_t m = bf16x2_mul_rn(l2, lo2);
  h = bf16x2_fma_rn(l2, hi2, m);
  const uint32_t t = bf16x2_fma_rn(l2, hi2, h ^ 0x80008000u);  // fma with -hi (sign bits flipped)
  l = bf16x2_add_rn(t, m);
}

// One Q4_0 block with an IEEE-half scale (split by split_half_scale) to the hi and lo parts
// of its 32 weights (hi + lo = level * d exactly; pairs in the order of q4_block_to_bf16).
// A scale that is not finite gives lo = 0 (hi then carries the infinity or NaN).
__device__ __forceinline__ void q4_block_to_hilo_split(const uint32_t (&w)[4], uint32_t hi2, uint32_t lo2,
                                                       bool finite, uint32_t (&hi)[16], uint32_t (&lo)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo01, lo23, hi01, hi23;
    q4_word_to_bf16_levels(w[i], lo01, lo23, hi01, hi23);
    scale_bf16_levels_hilo(lo01, hi2, lo2, hi[2 * i], lo[2 * i]);
    scale_bf16_levels_hilo(lo23, hi2, lo2, hi[2 * i + 1], lo[2 * i + 1]);
    scale_bf16_levels_hilo(hi01, hi2, lo2, hi[8 + 2 * i], lo[8 + 2 * i]);
    scale_bf16_levels_hilo(hi23, hi2, lo2, hi[8 + 2 * i + 1], lo[8 + 2 * i + 1]);
  }
  if (!finite) {
#pragma unroll
    for (int i = 0; i < 16; ++i) lo[i] = 0u;
  }
}

// One Q4_0 block with a float32 scale to the hi and lo parts of fl32(level * d).
__device__ __forceinline__ void q4_block_to_hilo(const uint32_t (&w)[4], float d, uint32_t (&hi)[16],
                                                 uint32_t (&lo)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo01, lo23, hi01, hi23;
    q4_word_to_f16_levels(w[i], lo01, lo23, hi01, hi23);
#define QMV_HALF_PAIR(h2, k)                                                                                 \
  scale2_hilo(__half2float(__ushort_as_half(static_cast<unsigned short>((h2) & 0xFFFFu))),                  \
              __half2float(__ushort_as_half(static_cast<unsigned short>((h2) >> 16))), d, hi[k], lo[k])
    QMV_HALF_PAIR(lo01, 2 * i);
    QMV_HALF_PAIR(lo23, 2 * i + 1);
    QMV_HALF_PAIR(hi01, 8 + 2 * i);
    QMV_HALF_PAIR(hi23, 8 + 2 * i + 1);
#undef QMV_HALF_PAIR
  }
}

// One Q8_0 block (32 int8 quants in w[0..7]) to the hi and lo parts of fl32(q * d).
__device__ __forceinline__ void q8_block_to_hilo(const uint32_t (&w)[8], float d, uint32_t (&hi)[16],
                                                 uint32_t (&lo)[16]) {
  const float bias = 8388736.0f;  // 2^23 + 128
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t u = w[i] ^ 0x80808080u;  // q + 128 per byte
    const float f0 = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7440)), bias);
    const float f1 = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7441)), bias);
    const float f2 = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7442)), bias);
    const float f3 = __fsub_rn(__uint_as_float(prmt(u, 0x4B000000u, 0x7443)), bias);
    scale2_hilo(f0, f1, d, hi[2 * i], lo[2 * i]);
    scale2_hilo(f2, f3, d, hi[2 * i + 1], lo[2 * i + 1]);
  }
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

// 16 columns of accumulator 0 plus the same columns of accumulator 1 (128 columns on).
__device__ __forceinline__ void acc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  uint32_t u[16];
  tmem_ld16(taddr, v);
  tmem_ld16(taddr + 128u, u);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(u[i]));
}

// Bounded wait that gives up at once when another role has already failed (a phase that has
// already completed returns without reading the failure flag).
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, volatile int* failed, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*failed) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  record_status(status, QMV_E_TIMEOUT);
  *failed = 1;
  return false;
}

template <int WT, bool F16, bool HILO>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tq,
                                                              const __grid_constant__ CUtensorMap td,
                                                              const __grid_constant__ CUtensorMap tx,
                                                              const PParams p) {
  using C = PCfg<WT, F16>;
  constexpr int kKS = Ring<HILO>::kKS;
  constexpr int kSC = Ring<HILO>::kStageCols;
  // launched early without leave to read the weights meanwhile: nothing global (and no tensor
  // memory) before the wait
  if (!p.early) griddep_wait();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);  // 1024-aligned: swizzle atoms
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = bars + kRS;
  uint64_t* a_full = bars + 2 * kRS;
  uint64_t* empty = a_full + kMaxKS;
  uint64_t* x_full = empty + kMaxKS;
  uint64_t* x_empty = x_full + kMaxXS;
  uint64_t* acc_full = x_empty + kMaxXS;
  const uint32_t xstage = (uint32_t)p.npad * 128;  // bytes of one X stage
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  // this CTA's tile and column range: raw stages [q0, q1) = 64-column stages kb0 + [0, nkb)
  const int tile = (int)blockIdx.x / p.ksplit;
  const int split = (int)blockIdx.x - tile * p.ksplit;
  const int row0 = tile * kPM;
  const int nq = p.cols / kRawK;
  const int q0 = split * nq / p.ksplit;
  const int q1 = (split + 1) * nq / p.ksplit;
  const int kb0 = 4 * q0;
  const int nkb = 4 * (q1 - q0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRS; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kDeqWarps);  // both groups read every raw stage
    }
    for (int i = 0; i < kMaxXS; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);
    }
    for (int i = 0; i < kKS; ++i) {
      mbar_init(&a_full[i], 8);
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 2);
    *failed = 0;
    fence_mbar_init();
    griddep_launch_dependents();  // the next kernel may be scheduled (it waits for this one before its activations)
    prefetch_tmap(&tq);
    prefetch_tmap(&td);
    prefetch_tmap(&tx);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- raw-stage producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int nqs = q1 - q0;
      int raw_issued = 0;
      for (int q = 0; q < nqs && !*failed; ++q) {
        const int r = q % kRS;
        if (q >= kRS && !pwait(&raw_empty[r], (uint32_t)((q / kRS - 1) & 1), failed, p.status)) break;
        mbar_arrive_expect_tx(&raw_full[r], C::Q_RAW + C::D_RAW);
#pragma unroll
        for (int b = 0; b < C::NQBOX; ++b)
          tma_load_2d(smem + C::OFF_Q + r * C::Q_RAW + b * (kPM * 128), &tq, (q0 + q) * C::QRAW_ROW + b * 128, row0,
                      &raw_full[r], pol);
        tma_load_2d(smem + C::OFF_D + r * C::D_RAW, &td, (q0 + q) * C::DROW, row0, &raw_full[r], pol);
        raw_issued = q + 1;
      }
      if (*failed) {
        // let the copies still in flight land before the shared memory is released
        for (int r = 0; r < kRS && r < raw_issued; ++r) {
          const int last = raw_issued - 1 - ((raw_issued - 1 - r) % kRS);  // last raw stage in slot r
          mbar_wait_bounded(&raw_full[last % kRS], (uint32_t)((last / kRS) & 1), 400000000LL);
        }
      }
    }
  } else if (warp == kXWarp) {
    // ---------------------------------------------------------------- X-stage producer
    if (lane == 0) {
      // the activations (and, after them, the y and workspace writes) wait for the preceding
      // kernel to complete when this launch overlaps it; the weights do not
      griddep_wait();
      int x_issued = 0;
      int xs = 0;         // slot of stage kb in the X ring (kb % p.xs)
      uint32_t xph = 0;   // its phase ((kb / p.xs) & 1)
      for (int kb = 0; kb < nkb && !*failed; ++kb) {
        if (kb >= p.xs && !pwait(&x_empty[xs], xph ^ 1u, failed, p.status)) break;
        mbar_arrive_expect_tx(&x_full[xs], xstage);
        tma_load_2d_keep(smem + C::OFF_X + xs * xstage, &tx, (kb0 + kb) * kKB, 0, &x_full[xs]);
        x_issued = kb + 1;
        if (++xs == p.xs) {
          xs = 0;
          xph ^= 1u;
        }
      }
      if (*failed) {
        for (int s = 0; s < p.xs && s < x_issued; ++s) {
          const int last = x_issued - 1 - ((x_issued - 1 - s) % p.xs);
          mbar_wait_bounded(&x_full[last % p.xs], (uint32_t)((last / p.xs) & 1), 400000000LL);
        }
      }
    }
  } else if (warp == 1 || warp == kMmaWarp2) {
    // ---------------------------------------------------------------- MMA issuers
    // Warp 1 issues the even stages into accumulator 0 (columns 0..127), the other warp the
    // odd ones into accumulator 1 (columns 128..255): a single issuing thread, not the
    // tensor core, set the pace with one.
    if (lane == 0) {
      const int m = warp == 1 ? 0 : 1;
      const uint32_t acc = tmem + (uint32_t)(kAccCol + m * 128);
      const uint32_t idesc = idesc_bf16_f32(kPM, p.npad);
      int xs = m;        // slot of stage kb in the X ring (kb % p.xs; p.xs even)
      uint32_t xph = 0;  // its phase
      int s = m;         // slot of stage kb in the weight ring (kb % kKS)
      uint32_t aph = 0;  // its phase
      for (int kb = m; kb < nkb; kb += 2) {
        if (!pwait(&x_full[xs], xph, failed, p.status) || !pwait(&a_full[s], aph, failed, p.status)) break;
        tc_fence_after();
        // A: 128 lanes x 32 columns (two bf16 each) of hi parts (or bf16 weights), then as many
        // of lo parts
        const uint32_t a0 = tmem + (uint32_t)(kACol + kSC * s);
        const uint32_t b0 = sbase + C::OFF_X + xs * xstage;
#pragma unroll
        for (int k = 0; k < kKB / 16; ++k) {
          const uint64_t bdesc = smem_desc_sw128(b0 + 32 * k);
          tc_mma_f16_ts(acc, a0 + 8 * k, bdesc, idesc, ((kb - m) | k) != 0);
          if (HILO) tc_mma_f16_ts(acc, a0 + 32 + 8 * k, bdesc, idesc, true);
        }
        tc_commit(smem_u32(&empty[s]));     // the weight stage is free once these MMAs complete
        tc_commit(smem_u32(&x_empty[xs]));  // and so is the X stage
        xs += 2;
        if (xs >= p.xs) {
          xs -= p.xs;
          xph ^= 1u;
        }
        s += 2;
        if (s >= kKS) {
          s -= kKS;
          aph ^= 1u;
        }
      }
      tc_commit(smem_u32(acc_full));  // arrives once every MMA this thread issued has completed
    }
  } else {
    // ---------------------------------------------------------------- dequantize, then drain
    // thread (row, h): a warp may write only its own 32-lane quarter of tensor memory, so
    // the row is 32 (warp % 4) + lane; the group's first four warps take block 0 of each
    // stage, the others block 1
    const int grp = (warp - 2) >> 3;
    const int dt = threadIdx.x - 64 - 256 * grp;
    const int row = 32 * (warp & 3) + lane;
    const int h = (dt >> 7) & 1;  // which block of each 64-column stage
    const int sw = row & 7;
    const uint32_t a_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(kACol + 16 * h);  // hi part
    // stages kb and kb + 1 (slots s and s + 1 of the weight ring, blocks blk and blk + 2 of
    // the raw stage)
    int s = 2 * grp;   // slot of stage kb in the weight ring (kb % kKS; stage kb + 1 takes s + 1)
    uint32_t ph = 0;   // its phase
    for (int kb = 2 * grp; kb < nkb; kb += 4) {
      const int q = kb / 4, r = q % kRS;
      const bool ok = pwait(&raw_full[r], (uint32_t)((q / kRS) & 1), failed, p.status) &&
                      (kb < kKS || (pwait(&empty[s], ph ^ 1u, failed, p.status) &&
                                    pwait(&empty[s + 1], ph ^ 1u, failed, p.status)));
      // the tensor-memory stores below are warp-wide: the warp leaves together
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();  // the MMAs that read these stages' tensor memory are complete
      const int blk = 2 * (kb & 3) + h;
      float d0, d1;
      if (F16) {
        const uint16_t* ds = reinterpret_cast<const uint16_t*>(smem + C::OFF_D + r * C::D_RAW + row * C::DROW);
        d0 = f16_bits_to_f32(ds[blk]);
        d1 = f16_bits_to_f32(ds[blk + 2]);
      } else {
        const float* ds = reinterpret_cast<const float*>(smem + C::OFF_D + r * C::D_RAW + row * C::DROW);
        d0 = ds[blk];
        d1 = ds[blk + 2];
      }
      uint32_t out0[16], out1[16];  // hi parts (or bf16 weights) of blocks blk and blk + 2
      uint32_t lo0[16], lo1[16];    // lo parts (HILO)
      const uint32_t qrow = sbase + C::OFF_Q + r * C::Q_RAW + row * 128;
      if (WT == QMV_Q4_0) {
        uint32_t w0[4], w1[4];
        lds128(qrow + ((blk ^ sw) << 4), w0[0], w0[1], w0[2], w0[3]);
        lds128(qrow + (((blk + 2) ^ sw) << 4), w1[0], w1[1], w1[2], w1[3]);
        if (F16) {
          uint32_t h0, l0, h1, l1;
          split_half_scale(d0, h0, l0);
          split_half_scale(d1, h1, l1);
          if (HILO) {
            q4_block_to_hilo_split(w0, h0, l0, isfinite(d0), out0, lo0);
            q4_block_to_hilo_split(w1, h1, l1, isfinite(d1), out1, lo1);
          } else {
            q4_block_to_bf16_split(w0, h0, l0, out0);
            q4_block_to_bf16_split(w1, h1, l1, out1);
          }
        } else if (HILO) {
          q4_block_to_hilo(w0, d0, out0, lo0);
          q4_block_to_hilo(w1, d1, out1, lo1);
        } else {
          q4_block_to_bf16(w0, d0, out0);
          q4_block_to_bf16(w1, d1, out1);
        }
      } else {
        uint32_t w0[8], w1[8];
        const uint32_t box = qrow + (blk >> 2) * (kPM * 128);
        const int c0 = 2 * (blk & 3);  // blk + 2 lies in the same 128-byte box (blk & 3 < 2)
        lds128(box + ((c0 ^ sw) << 4), w0[0], w0[1], w0[2], w0[3]);
        lds128(box + (((c0 + 1) ^ sw) << 4), w0[4], w0[5], w0[6], w0[7]);
        lds128(box + (((c0 + 4) ^ sw) << 4), w1[0], w1[1], w1[2], w1[3]);
        lds128(box + (((c0 + 5) ^ sw) << 4), w1[4], w1[5], w1[6], w1[7]);
        if (HILO) {
          q8_block_to_hilo(w0, d0, out0, lo0);
          q8_block_to_hilo(w1, d1, out1, lo1);
        } else {
          q8_block_to_bf16(w0, d0, out0);
          q8_block_to_bf16(w1, d1, out1);
        }
      }
      // the block's 32 bf16 weights (pairs in element order) into 16 columns of this row's lane;
      // the lo parts 32 columns further on
      tmem_st16(a_lane + (uint32_t)(kSC * s), out0);
      tmem_st16(a_lane + (uint32_t)(kSC * (s + 1)), out1);
      if (HILO) {
        tmem_st16(a_lane + (uint32_t)(kSC * s + 32), lo0);
        tmem_st16(a_lane + (uint32_t)(kSC * (s + 1) + 32), lo1);
      }
      tmem_st_wait();
      tc_fence_before();  // the stores are complete before the arrivals below
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&a_full[s]);
        mbar_arrive(&a_full[s + 1]);
        mbar_arrive(&raw_empty[r]);
      }
      s += 4;
      if (s >= kKS) {
        s -= kKS;
        ph ^= 1u;
      }
    }
    // drain the accumulators and store y (all dequantize warps): warp w reads tensor-memory
    // lanes 32*(w%4) .. +31 (its rows) and the 16-column chunks (w-2)/4 + 4k of both
    // accumulators, and adds them (even stages + odd stages)
    const bool ok = mbar_wait_bounded(acc_full, 0u);
    if (!ok) {
      record_status(p.status, QMV_E_TIMEOUT);
      *failed = 1;
    }
    tc_fence_after();
    const int quarter = warp & 3;
    const int cg = (warp - 2) >> 2;  // which 16-column chunks: cg, cg + 4, ...
    const int trow = quarter * 32 + lane;  // row within the tile
    const int grow = row0 + trow;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    if (p.ksplit == 1) {
      if (ok && !*failed) {
        for (int c = cg * 16; c < p.npad; c += 64) {
          uint32_t v[16];
          acc_ld16(tl + (uint32_t)c, v);
          if (grow < p.rows) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c + i < p.batch) p.y[(size_t)(c + i) * p.rows + grow] = __uint_as_float(v[i]);
          }
        }
      }
    } else {
      // this split's part, vector-major (the 128 sums of vector n contiguous) so that its
      // stores here and the loads of the last CTA below are coalesced; then the last CTA of
      // the tile to arrive adds the parts in split order
      float* part = p.parts + (size_t)blockIdx.x * kPM * p.npad;
      if (ok && !*failed) {
        for (int c = cg * 16; c < p.npad; c += 64) {
          uint32_t v[16];
          acc_ld16(tl + (uint32_t)c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) part[(size_t)(c + i) * kPM + trow] = __uint_as_float(v[i]);
        }
      }
      epilogue_barrier();  // every part of this CTA is written before the release below
      if (threadIdx.x == 64) {
        const unsigned before = atomic_add_acq_rel_u32(p.counters + tile, 1u);
        const bool last = before + 1 == (unsigned)p.ksplit;
        if (last) p.counters[tile] = 0u;  // every part has arrived: ready for the next launch
        *last_flag = last ? 1 : 0;
      }
      epilogue_barrier();  // the acquire above is ordered before the loads below
      if (*last_flag && !*failed) {
        // units of 4 consecutive rows of one vector; each thread takes kUnits of them at a
        // time and loads every split's values (4 splits at a time) before adding them in order
        constexpr int kUnits = 2;
        constexpr int kEpi = 32 * kDeqWarps;  // threads
        const float* tpart = p.parts + (size_t)tile * p.ksplit * kPM * p.npad;
        const size_t sstride = (size_t)kPM * p.npad;  // floats between the splits of the tile
        const int units = p.npad * (kPM / 4);
        const int et = threadIdx.x - 64;
        for (int u0 = et; u0 < units; u0 += kUnits * kEpi) {
          float4 acc[kUnits];
          for (int sp0 = 0; sp0 < p.ksplit; sp0 += 4) {
            float4 q[kUnits][4];
#pragma unroll
            for (int j = 0; j < kUnits; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (u0 + j * kEpi < units && sp0 + e < p.ksplit)
                  q[j][e] = __ldcg(reinterpret_cast<const float4*>(tpart + (sp0 + e) * sstride) + u0 + j * kEpi);
#pragma unroll
            for (int j = 0; j < kUnits; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (u0 + j * kEpi < units && sp0 + e < p.ksplit) {
                  if (sp0 + e == 0) {
                    acc[j] = q[j][e];
                  } else {
                    acc[j].x += q[j][e].x;
                    acc[j].y += q[j][e].y;
                    acc[j].z += q[j][e].z;
                    acc[j].w += q[j][e].w;
                  }
                }
          }
#pragma unroll
          for (int j = 0; j < kUnits; ++j) {
            const int u = u0 + j * kEpi;
            const int n = u / (kPM / 4);
            const int r = row0 + (u % (kPM / 4)) * 4;
            if (u < units && n < p.batch) {
              float* dst = p.y + (size_t)n * p.rows + r;
              if (r + 3 < p.rows && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {  // y is 4-byte aligned
                *reinterpret_cast<float4*>(dst) = acc[j];
              } else {
                if (r < p.rows) dst[0] = acc[j].x;
                if (r + 1 < p.rows) dst[1] = acc[j].y;
                if (r + 2 < p.rows) dst[2] = acc[j].z;
                if (r + 3 < p.rows) dst[3] = acc[j].w;
              }
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool prefill_supported(const MatrixRef& m, bool x_bf16) {
  return x_bf16 && m.cols % kRawK == 0 && m.rows < (1LL << 31) - kPM && m.cols < (1LL << 30);
}

int prefill_max_batch() { return kMaxN; }

// Column ranges per tile: enough to give every SM a CTA when the matrix has fewer tiles than
// SMs (at least two raw stages per range), within the workspace; 1 without one.
static int prefill_ksplit(const MatrixRef& m, int npad, const DeviceInfo& dev, const Workspace* ws) {
  const long long tiles = (m.rows + kPM - 1) / kPM;
  const long long nq = m.cols / kRawK;
  if (ws == nullptr || tiles >= dev.sm_count || tiles > ws->max_counters) return 1;
  long long k = dev.sm_count / tiles;
  if (k > nq / 2) k = nq / 2;
  if (k > 16) k = 16;
  while (k > 1 && (size_t)(tiles * k * npad * kPM) > ws->max_partial_floats) --k;
  return k < 1 ? 1 : (int)k;
}

template <int WT, bool F16, bool HILO>
static cudaError_t launch_prefill_typed(const MatrixRef& m, const void* x, float* y, int batch, const DeviceInfo& dev,
                                        const Workspace* ws, bool pdl, cudaStream_t stream) {
  using C = PCfg<WT, F16>;
  auto kern = prefill_kernel<WT, F16, HILO>;
  static bool ready[64] = {};
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev.device]) {
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev.smem_optin);
    if (err != cudaSuccess) return err;
    ready[dev.device] = true;
  }
  PParams p;
  p.y = y;
  p.rows = (int)m.rows;
  p.cols = (int)m.cols;
  p.batch = batch;
  p.npad = (batch + 15) / 16 * 16;
  p.status = dev.status;
  p.early = pdl ? 1 : 0;
  // X ring: as many stages as the shared memory left by the raw ring holds, in an even
  // number (the two MMA warps take alternate stages, so with an even depth each slot always
  // serves the same warp and no warp can wait for a phase two ahead of the slot's barrier,
  // which a parity wait would take as done)
  p.xs = ((int)dev.smem_optin - C::smem_bytes(0, p.npad)) / (p.npad * 128);
  if (p.xs > kMaxXS) p.xs = kMaxXS;
  p.xs &= ~1;
  if (p.xs < 2) return cudaErrorInvalidConfiguration;
  p.ksplit = prefill_ksplit(m, p.npad, dev, ws);
  p.counters = p.ksplit > 1 ? ws->counters : nullptr;
  p.parts = p.ksplit > 1 ? ws->partials : nullptr;
  CUtensorMap tq, td, tx;
  const uint64_t qrow = (WT == QMV_Q4_0) ? (uint64_t)m.cols / 2 : (uint64_t)m.cols;
  const uint64_t drow = (uint64_t)(m.cols / 32) * C::ESZ;
  cudaError_t err = encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, m.q, qrow, (uint64_t)m.rows, qrow, 128, kPM,
                                   CU_TENSOR_MAP_SWIZZLE_128B);
  if (err != cudaSuccess) return err;
  err = encode_tmap_2d(&td, CU_TENSOR_MAP_DATA_TYPE_UINT8, m.d, drow, (uint64_t)m.rows, drow, C::DROW, kPM,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
  if (err != cudaSuccess) return err;
  err = encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)m.cols, (uint64_t)batch,
                       (uint64_t)m.cols * 2, kKB, p.npad, CU_TENSOR_MAP_SWIZZLE_128B);
  if (err != cudaSuccess) return err;
  const int grid = (int)((m.rows + kPM - 1) / kPM) * p.ksplit;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::smem_bytes(p.xs, p.npad);
  cfg.stream = stream;
  // always a programmatic dependent (without pdl the kernel waits before its first global access)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, td, tx, p);
}

template <bool HILO>
static cudaError_t launch_prefill_ring(const MatrixRef& m, const void* x, float* y, int batch, const DeviceInfo& dev,
                                       const Workspace* ws, bool pdl, cudaStream_t stream) {
  if (m.wtype == QMV_Q4_0) {
    return m.scale_f16 ? launch_prefill_typed<QMV_Q4_0, true, HILO>(m, x, y, batch, dev, ws, pdl, stream)
                       : launch_prefill_typed<QMV_Q4_0, false, HILO>(m, x, y, batch, dev, ws, pdl, stream);
  }
  return m.scale_f16 ? launch_prefill_typed<QMV_Q8_0, true, HILO>(m, x, y, batch, dev, ws, pdl, stream)
                     : launch_prefill_typed<QMV_Q8_0, false, HILO>(m, x, y, batch, dev, ws, pdl, stream);
}

cudaError_t launch_prefill(const MatrixRef& m, const void* x, float* y, int batch, bool bf16_weights,
                           const DeviceInfo& dev, const Workspace* ws, bool pdl, cudaStream_t stream) {
  if (batch < 1 || batch > kMaxN) return cudaErrorInvalidValue;
  return bf16_weights ? launch_prefill_ring<false>(m, x, y, batch, dev, ws, pdl, stream)
                      : launch_prefill_ring<true>(m, x, y, batch, dev, ws, pdl, stream);
}

}  // namespace qmv
