// qmv_common.cuh -- device helpers shared by the libqmv kernels (sm_103a).
//
// Format facts used throughout (Krafla ".mlb model format v1", "Body", "Q8_0", "Q4_0"):
//   q array first, d array at round_up(q bytes, 64); one scale per 32 consecutive
//   weights of a row; Q4_0 block = 16 bytes, byte j = element j (low nibble) and
//   element j+16 (high nibble), weight (nibble - 8) * d; Q8_0 weight = int8 * d.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qmv.h"

namespace qmv {

// A kernel whose bounded wait runs out records QMV_E_TIMEOUT in the per-device status word
// (passed to it as a pointer) and returns; qmv_check_device() reads and clears it.
__device__ __forceinline__ void record_status(int* status, int code) { atomicCAS(status, 0, code); }

// ---------------------------------------------------------------------------- numbers
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// ---------------------------------------------------------------------------- smem / PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after about `limit_cycles` SM cycles.
// Returns false on time-out (the caller records QMV_E_TIMEOUT and unwinds).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_cycles = 4000000000LL) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit_cycles) return false;
  }
}

// Programmatic dependent launch: wait until the preceding kernel in the stream has finished
// and its writes are visible (a no-op when the launch did not allow overlap), and let the
// next kernel be scheduled early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 policy for data read exactly once (the weight stream): evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk (non-tensor) asynchronous copy global -> shared, completion counted in bytes on an
// mbarrier.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                             uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 2-D tiled TMA load of one box into shared memory (coordinates: x innermost, in elements).
__device__ __forceinline__ void tma_load_2d(void* dst_smem, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// The same without a cache hint (data that many CTAs re-read, such as the activations).
__device__ __forceinline__ void tma_load_2d_keep(void* dst_smem, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory loads by 32-bit shared address (ordered after the barrier waits).
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t a;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a) : "r"(addr) : "memory");
  return a;
}

__device__ __forceinline__ void lds_u32x2(uint32_t addr, uint32_t& a, uint32_t& b) {
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr) : "memory");
}

__device__ __forceinline__ void lds_f32x4(uint32_t addr, float (&v)[4]) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ldmatrix: four 8x8 matrices of 16-bit elements; lane l supplies the address of row
// (l % 8) of matrix (l / 8); thread (g = lane/4, t = lane%4) receives, for each matrix,
// the 32-bit word t of row g.
__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, f32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(orv));  // (a & b) | c
  return r;
}

// bf16x2 a - b (exact here: both operands are small integers).
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Four Q4_0 quant bytes (bytes i = 0..3 of one 32-bit word; byte i holds element i in its
// low nibble lo_i and element i+16 in its high nibble hi_i) to exact bfloat16 levels
// (nibble - 8), in natural pairs (low half first):
//   lo01 = (lo0, lo1)  lo23 = (lo2, lo3)  hi01 = (hi0, hi1)  hi23 = (hi2, hi3)
// prmt spreads bytes 0,1 (2,3) into the two 16-bit halves; 0x4300 | n is the bfloat16 of
// 128 + n (n < 16 sits in the mantissa), and (128 + n) - 136 = n - 8 is exact.
__device__ __forceinline__ void q4_word_to_bf16_levels(uint32_t w, uint32_t& lo01, uint32_t& lo23, uint32_t& hi01,
                                                       uint32_t& hi23) {
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kMagic = 0x43004300u;   // bf16 128.0 in both halves
  constexpr uint32_t kOffset = 0x43084308u;  // bf16 136.0 in both halves
  const uint32_t b01 = prmt(w, 0u, 0x4140);  // bytes: w.b0, 0, w.b1, 0
  const uint32_t b23 = prmt(w, 0u, 0x4342);  // bytes: w.b2, 0, w.b3, 0
  lo01 = bf16x2_sub(lop_and_or(b01, kMask, kMagic), kOffset);
  hi01 = bf16x2_sub(lop_and_or(b01 >> 4, kMask, kMagic), kOffset);
  lo23 = bf16x2_sub(lop_and_or(b23, kMask, kMagic), kOffset);
  hi23 = bf16x2_sub(lop_and_or(b23 >> 4, kMask, kMagic), kOffset);
}

// Four Q8_0 quant bytes q0..q3 (one word) to exact bfloat16 levels in natural pairs
//   q01 = (q0, q1)  q23 = (q2, q3)
// via float32: 0x4B000000 | u is 2^23 + u; with u = q + 128 the float32 subtraction of
// 2^23 + 128 gives q exactly, and an integer of magnitude <= 128 is exact in bfloat16,
// so its bfloat16 code is the upper half of its float32 code.
__device__ __forceinline__ void q8_word_to_bf16_levels(uint32_t w, uint32_t& q01, uint32_t& q23) {
  const uint32_t u = w ^ 0x80808080u;  // q + 128 in each byte
  const float bias = 8388736.0f;       // 2^23 + 128
  const float f0 = __uint_as_float(prmt(u, 0x4B000000u, 0x7440)) - bias;
  const float f1 = __uint_as_float(prmt(u, 0x4B000000u, 0x7441)) - bias;
  const float f2 = __uint_as_float(prmt(u, 0x4B000000u, 0x7442)) - bias;
  const float f3 = __uint_as_float(prmt(u, 0x4B000000u, 0x7443)) - bias;
  q01 = prmt(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
  q23 = prmt(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
}

// Round-to-nearest-even bfloat16 pair from two floats: low half from lo, high half from hi.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------- half precision
// IEEE half pair arithmetic on packed registers (all uses below are exact).
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t f16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// A bfloat16 pair (low half first) as an IEEE half pair; `exact` is cleared unless both
// values convert exactly (checked by converting back: zero, and bfloat16 values with
// 2^-17 <= |x| <= 65280, pass; larger and tinier values and NaN do not).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t p, bool& exact) {
  const float lo = __uint_as_float(p << 16);
  const float hi = __uint_as_float(p & 0xFFFF0000u);
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  const float blo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
  const float bhi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
  exact = exact & (blo == lo) & (bhi == hi);
  return h;
}

// The power of two xs = 2^s that brings a stage's largest magnitude amax into [2^14, 2^15)
// (s = 141 - the biased exponent of amax), and xinv = 2^-s, both exact; amax == 0 gives
// xs = xinv = 1.  False (xs = xinv = 1) when no such power is a normal float32: amax below
// 2^-112, infinite or NaN.
__device__ __forceinline__ bool half_stage_scale(float amax, float& xs, float& xinv) {
  const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  const bool ok = amax == 0.f || (eb >= 15 && eb <= 254);
  const int se = (amax == 0.f || !ok) ? 127 : 268 - eb;  // biased exponent of 2^s
  xs = __uint_as_float((uint32_t)se << 23);
  xinv = __uint_as_float((uint32_t)(254 - se) << 23);
  return ok;
}

// Two float32 values times a power of two `scale` rounded to an IEEE half pair (to nearest
// even); `fits` is cleared unless each value is zero or its result is a normal half (magnitude
// 2^-14 .. 65504), where the rounding's relative error is at most 2^-11.  A product that left
// the float32 normal range (so was not exact) gives a subnormal or zero half and clears `fits`.
__device__ __forceinline__ uint32_t f32x2_to_f16x2_normal(float lo, float hi, float scale, bool& fits) {
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi * scale), "f"(lo * scale));
  const float blo = fabsf(__half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu))));
  const float bhi = fabsf(__half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16))));
  const bool okl = (blo >= 0x1p-14f && blo <= 65504.0f) || lo == 0.0f;
  const bool okh = (bhi >= 0x1p-14f && bhi <= 65504.0f) || hi == 0.0f;
  fits = fits & okl & okh;
  return h;
}

// The same for a bfloat16 pair times a power of two `scale` (exact in float32).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t p, float scale, bool& exact) {
  const float lo = __uint_as_float(p << 16) * scale;
  const float hi = __uint_as_float(p & 0xFFFF0000u) * scale;
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  const float blo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
  const float bhi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
  exact = exact & (blo == lo) & (bhi == hi);
  return h;
}

// Four Q4_0 quant bytes (as for q4_word_to_bf16_levels) to exact IEEE half levels in natural
// pairs.  prmt puts byte b under the half exponent of 1024 (0x6400 | b is 1024 + b: the
// 10-bit mantissa takes the whole byte); H = 1024 + 16 hi + 8 (the low nibble replaced by 8);
// then (1024 + b) - H = lo - 8 and H / 16 - 72.5 = hi - 8, both exact.
__device__ __forceinline__ void q4_word_to_f16_levels(uint32_t w, uint32_t& lo01, uint32_t& lo23, uint32_t& hi01,
                                                      uint32_t& hi23) {
  constexpr uint32_t kExp = 0x64646464u;       // 0x64: the high byte of half 1024
  constexpr uint32_t kSixteenth = 0x2C002C00u;  // half 1/16
  constexpr uint32_t kOff = 0xD488D488u;        // half -72.5
  const uint32_t p01 = prmt(w, kExp, 0x4140);   // 1024 + b0, 1024 + b1
  const uint32_t p23 = prmt(w, kExp, 0x4342);   // 1024 + b2, 1024 + b3
  const uint32_t h01 = lop_and_or(p01, 0xFFF0FFF0u, 0x00080008u);
  const uint32_t h23 = lop_and_or(p23, 0xFFF0FFF0u, 0x00080008u);
  lo01 = f16x2_sub(p01, h01);
  lo23 = f16x2_sub(p23, h23);
  hi01 = f16x2_fma(h01, kSixteenth, kOff);
  hi23 = f16x2_fma(h23, kSixteenth, kOff);
}

// Four Q8_0 quant bytes q0..q3 to exact IEEE half levels q01 = (q0, q1), q23 = (q2, q3):
// with u = q + 128, 0x6400 | u is 1024 + u, and (1024 + u) - 1152 = q.
__device__ __forceinline__ void q8_word_to_f16_levels(uint32_t w, uint32_t& q01, uint32_t& q23) {
  constexpr uint32_t kExp = 0x64646464u;
  constexpr uint32_t kBias = 0x64806480u;  // half 1152
  const uint32_t u = w ^ 0x80808080u;
  q01 = f16x2_sub(prmt(u, kExp, 0x4140), kBias);
  q23 = f16x2_sub(prmt(u, kExp, 0x4342), kBias);
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + C, f32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ void lds_u32x4(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void sts_u32x4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}


// ---------------------------------------------------------------------------- gated activation
// The FFN's gated activation (Krafla page, "Body": w1 gate, w3 up, header field act):
// SiLU(g) = g / (1 + e^-g) (act 0), GELU_tanh(g) = g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))
// (act 1), times up; float32 operations with CUDA's expf and tanhf.
__device__ __forceinline__ float glu(int act, float g, float u) {
  float h;
  if (act == 0) {
    h = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  } else {
    const float k = 0.7978845608028654f;  // sqrt(2 / pi)
    const float inner = __fmul_rn(k, __fadd_rn(g, __fmul_rn(0.044715f, __fmul_rn(g, __fmul_rn(g, g)))));
    h = __fmul_rn(__fmul_rn(0.5f, g), __fadd_rn(1.0f, tanhf(inner)));
  }
  return __fmul_rn(h, u);
}

// bfloat16 bits of v rounded to nearest (ties to even); finite v beyond the bfloat16 range
// (which would round to infinity) are truncated instead, so that hi + lo stays finite.
__device__ __forceinline__ uint16_t bf16_bits_rn_finite(float v) {
  const uint32_t r = pack_bf16x2(v, v) & 0xFFFFu;
  const float back = __uint_as_float(r << 16);
  if (isfinite(v) && !isfinite(back)) return static_cast<uint16_t>(__float_as_uint(v) >> 16);
  return static_cast<uint16_t>(r);
}

// A float32 activation as a bfloat16 pair: hi = RN_bf16(v), lo = RN_bf16(v - hi) (v - hi is
// exact in float32; lo = 0 for v that is not finite): 16 significant bits of v kept.
__device__ __forceinline__ void split_bf16_pair(float v, uint16_t& hi, uint16_t& lo) {
  hi = bf16_bits_rn_finite(v);
  const float h = __uint_as_float((uint32_t)hi << 16);
  lo = isfinite(v) ? bf16_bits_rn_finite(v - h) : 0;
}


// ---------------------------------------------------------------------------- activation rule
// The runtime's activation quantizer (Krafla page, "Quantization rule", Q8_0 with a float32
// scale) on a block of 32 values: amax = max |x|; amax < 1e-30 gives the zero block (d = 0, every
// quant 0); else d = amax / 127 and q = trunc(x * (127 / amax) + copysign(0.5, x)), clamped to
// +-127; each step one float32 operation rounded to nearest.  The kernels that apply it hold a
// block in four lanes, eight values each.
//
// The rule on NCH blocks at once, each held by four lanes (lanes 4g .. 4g+3 of the warp hold
// block g of chunk h, 8 values each, v[h]): each block's amax by two xor shuffles (the maximum
// does not depend on the order; NaN is skipped); the divisions 127 / amax and amax / 127 of all
// NCH blocks in one pass over the four lanes (lane 4g + 2h + r divides for chunk h, r = 0: d, r = 1: 1 / d), then
// each value's quant by the same float32 steps, returned as IEEE half pairs (exact: |q| <= 127),
// hq[h][i] = (q(v[h][2i]) low, q(v[h][2i+1]) high), and d[h] the block's scale.
template <int NCH>
__device__ __forceinline__ void act_q8_lane_quarters(const float (&v)[NCH][8], uint32_t (&hq)[NCH][4],
                                                     float (&d)[NCH]) {
  static_assert(NCH == 1 || NCH == 2, "one or two chunks");
  const int lane = threadIdx.x & 31;
  float amax[NCH];
#pragma unroll
  for (int h = 0; h < NCH; ++h) {
    float m = 0.f;
    // fmaxf returns the operand that is not NaN, so a NaN value is skipped, and m never is NaN
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[h][e]));
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    amax[h] = m;
  }
  const int r = lane & 1;
  const float am = (NCH == 2 && (lane & 2)) ? amax[NCH - 1] : amax[0];
  // the zero block (amax below 1e-30) has d = 0 and 1 / d taken as 0
  const float num = r ? 127.0f : am, den = r ? am : 127.0f;
  const float quot = am < 1e-30f ? 0.f : __fdiv_rn(num, den);
  const int base = lane & ~3;
#pragma unroll
  for (int h = 0; h < NCH; ++h) {
    d[h] = __shfl_sync(0xffffffffu, quot, base + 2 * h);
    const float inv = __shfl_sync(0xffffffffu, quot, base + 2 * h + 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float q[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        // the rule's clamp to +-127 never acts here: |x| <= amax gives |x * inv| <= 127 (1 + 2^-23)
        // and a sum below 128 before the truncation; a value that is not finite gives NaN, whose
        // conversion is 0 with or without the clamp
        const float xe = v[h][2 * i + j];
        q[j] = (float)(int)__fadd_rn(__fmul_rn(xe, inv), copysignf(0.5f, xe));
      }
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hq[h][i]) : "f"(q[1]), "f"(q[0]));
    }
  }
}

}  // namespace qmv
