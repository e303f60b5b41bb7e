// decode_bdiag.cu -- the decode product for one bfloat16 activation vector, cols % 256 == 0.
//
// What is computed (Krafla ".mlb model format v1", "Q8_0", "Q4_0", "Body"):
//   y[r] = sum_k d[r][k] * sum_{j<32} level[r][32k+j] * x[32k+j]
// with level = nibble - 8 (Q4_0) or the int8 quant (Q8_0), d the block's scale.
//
// The stream of stages, the work split (warp tiles of 16*MT rows, items of NW/ks tiles x ks
// column slices walked persistently), the per-warp TMA rings and the overlap with the
// preceding kernel are those of the general decode kernel (decode_mma.cu), with three
// changes: a stage is two 256-column chunks (one TMA issue of each kind, one wait and one
// activation check per 512 columns: the per-stage bookkeeping and the many 16-byte rows of
// the scale box measured as costly as a third of the stage's work); the ks warps of a tile
// take interleaved stages (warp k: stages k, k + ks, ...), so that they read neighbouring
// pieces of the same rows at a time (DRAM pages are reused: one warp walking a row alone
// measured 20% slower); and ks is chosen by an estimate that counts waves of items (see
// plan_typed).  What changes with a single vector:
//   * Block-diagonal activations.  The 8 columns of an m16n8k16 MMA are spent on the 8
//     weight blocks of a chunk instead of on 8 vectors: the MMA of block j multiplies 16
//     rows' levels of block j by an activation fragment whose column j holds x of block j
//     and whose other columns are zero.  After the chunk's 16 MMAs (8 blocks x 2 halves)
//     column j of the accumulator is each row's block-j dot product, and the thread holding
//     it (g, t with j = 2t or 2t+1) applies that row's block-j scale: 4 FFMA per 16 rows and
//     chunk instead of 32.  Lanes g = j hold x of block j in the fragment of block j; each
//     lane writes its 16 activation bytes to a slot of its own and reads, for block j, that
//     slot (j = g) or a shared zero line (j != g).  At the end of an item the four lanes t
//     that share rows g, g+8 add their blocks' sums (two xor shuffles).
//   * Half-precision operands.  When every activation of the stage converts exactly to IEEE
//     half (zero, and bfloat16 values with 2^-17 <= |x| <= 65280; tested by converting back),
//     levels and activations enter the MMA as f16, whose 10-bit mantissa holds a whole quant
//     byte (0x6400 | b is 1024 + b): Q4_0 levels then cost 2 integer and 2 half operations
//     per byte pair instead of 4 and 2 (see q4_word_to_f16_levels).  The products are the
//     same exact products as with bfloat16 operands.  A stage whose activations are not all
//     exact halves (larger, tinier, NaN) uses bfloat16 operands, as the general kernel does.
//   * Gated pair (Q4_0).  For the FFN's w1 (gate) and w3 (up) projections of one x (Krafla
//     page, "Body"), a warp tile's two 16-row MMA tiles are rows 16t..16t+15 of w1 and the
//     same rows of w3 (two 16-row TMA boxes into the same 32-row swizzled stage), so that at
//     the end of its item the warp holds gate and up of the same rows and writes
//     h = act(gate) * up directly as the bfloat16 pair hi = RN_bf16(h), lo = RN_bf16(h - hi)
//     that the down projection's float32 route takes (the same bits the split kernel writes
//     from float32 gate and up).
#include <cstring>
#include <mutex>

#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {

namespace {

constexpr int kTK = 256;             // weights per chunk and row
constexpr int kBlocksPerStage = kTK / 32;  // blocks per chunk (the MMA's 8 columns)
constexpr int kRows = 16;            // rows per MMA tile
constexpr int kBox = 128;            // q box inner extent in bytes (the 128-byte swizzle span)
constexpr int kMaxProblems = 8;      // problems per grouped launch

// XS: float32 activations given as two bfloat16 vectors hi + lo (x = hi + lo); each stage
// then carries both.  A warp first forms x = hi + lo of its stage, scales it by the power of
// two 2^s that brings the stage's largest magnitude into [2^14, 2^15) and rounds it once to
// IEEE half: when every value is zero or a normal half after that (the stage's nonzero
// magnitudes lie within 2^28 of one another and are finite), each block runs one MMA as for a
// bfloat16 vector and its sums are multiplied by 2^-s (exact) before the scale; the rounding
// errs by at most 2^-11 of each term.  Otherwise every block's MMAs run once with hi and once
// with lo, into the same sums (16 significant bits of x).
// RD: ring depth (stages per warp in shared memory).  2: the next stage is requested before the
// current one is used; 1: only for launches where every warp has a single stage (half the
// shared memory, so twice the CTAs per SM), whose one stage is requested before the
// dependency wait.
// XH: the activations were rounded to half ahead of the product (per 256-column chunk, as above),
// with the bfloat16 pair kept in device memory for the chunks that do not round: the stage holds
// the half values (as a bfloat16 vector's), the slots room for both parts.
// X4: the stage's activation box holds four bytes a value (float32 activations).
template <int WT, bool F16, int NW, int CH, bool XS = false, int RD = 2, bool XH = false, bool X4 = false>
struct Cfg {
  static constexpr int kCH = CH;                                   // chunks per stage
  static constexpr int XPARTS = XS ? 2 : 1;                        // activation vectors per stage
  static constexpr int X_PART = CH * kTK * 2;                      // bfloat16 activations of one vector
  static constexpr int X_STAGE = (XS || X4 ? 2 : 1) * X_PART;       // activations of one stage
  static constexpr int MT = (WT == QMV_Q4_0) ? 2 : 1;           // 16-row MMA tiles per warp tile
  static constexpr int WROWS = MT * kRows;                        // rows per warp tile
  static constexpr int CBOX = (WT == QMV_Q4_0) ? 1 : 2;         // q boxes per chunk
  static constexpr int NQBOX = CBOX * CH;                        // q boxes per stage
  static constexpr int Q_BOX_BYTES = WROWS * kBox;
  static constexpr int Q_CHUNK = CBOX * Q_BOX_BYTES;              // 4096 bytes, multiple of 1024
  static constexpr int Q_STAGE = CH * Q_CHUNK;
  static constexpr int QROW = CBOX * kBox;                         // q bytes per row per chunk
  static constexpr int DCHUNK = kBlocksPerStage * (F16 ? 2 : 4);  // scale bytes per row per chunk
  static constexpr int DROW = CH * DCHUNK;                        // scale bytes per row per stage
  static constexpr int D_STAGE = WROWS * DROW;                     // multiple of 512
  static constexpr int S = RD;  // ring depth
  static constexpr int Q_WARP = S * Q_STAGE;
  static constexpr int D_WARP = S * D_STAGE;
  static constexpr int X_WARP = S * X_STAGE;
  // q rings, d rings, activation rings, activation slots (per chunk and vector: 32 lanes x
  // 16 bytes), zero area (a zero line as long as a warp's slots), reduction buffer (split-K),
  // barriers
  static constexpr int OFF_D = NW * Q_WARP;
  static constexpr int OFF_X = OFF_D + NW * D_WARP;
  static constexpr int OFF_SLOT = OFF_X + NW * X_WARP;
  static constexpr int SLOT_WARP = (XS || XH ? 2 : 1) * CH * 512;  // a warp's slots: [vector][chunk][lane]
  static constexpr int OFF_ZERO = OFF_SLOT + NW * SLOT_WARP;
  static constexpr int OFF_RED = OFF_ZERO + SLOT_WARP;
  static constexpr int OFF_BAR = OFF_RED + ((NW * WROWS * 4 + 127) / 128) * 128;
  static constexpr int SMEM = 1024 + OFF_BAR + ((NW * S * 8 + 127) / 128) * 128;
};

struct Problem {
  float* y;
  int rows;
  int ntiles;   // warp tiles (16*MT rows)
  int nst;      // stages per tile row: ceil(cols / 256 / CH) (chunks past the end read zeros)
  int item0;    // first item of this problem in the group's item list
  int nchunks;  // cols / 256
  const uint16_t* xg;  // XH: the bfloat16 hi parts (cols), then the lo parts (cols)
  const float* xinv;   // XH: per chunk 2^-s of its half values, 0 for a chunk that keeps hi + lo
};

struct Params {
  int nprob;
  int ks;       // column slices per tile (1, 2, 4, 8); at most every problem's nst
  int lgks;     // log2(ks)
  int nitems;
  int* status;
  // gated pair: problem 0 is the w1 / w3 pair (rows = w1's rows, 16 of each per warp tile)
  int early;      // the weights may be read before the preceding kernel has finished
  int act;        // 0 SiLU, 1 GELU-tanh
  uint16_t* h;    // the down projection's activations: hi parts at h[r], lo parts at h[rows + r]
  Problem pr[kMaxProblems];
};

struct Maps {  // per problem: q (128-byte swizzle), d, and activation (viewed as [cols/256][256]) tensor maps
  CUtensorMap q[kMaxProblems];
  CUtensorMap d[kMaxProblems];
  CUtensorMap x[kMaxProblems];
  CUtensorMap xl[kMaxProblems];  // the lo vectors (XS)
};

// Position of a warp in its stream of stages: item (global index), its problem and warp
// tile, this warp's first stage and stage count in the item (stage c0 + j * ks is the j-th;
// stage c covers chunks CH c .. CH c + CH - 1).
struct Cursor {
  int item, prob, tile, c0, n, j;
};

__device__ __forceinline__ void cursor_load(Cursor& c, const Params& p, int tiles_per_item, int tile_local,
                                            int kslice) {
  if (c.item >= p.nitems) return;
  int pr = 0;
  while (pr + 1 < p.nprob && c.item >= p.pr[pr + 1].item0) ++pr;
  c.prob = pr;
  c.tile = (c.item - p.pr[pr].item0) * tiles_per_item + tile_local;
  // stages kslice, kslice + ks, ... (ks <= nst: at least one)
  c.c0 = kslice;
  c.n = (p.pr[pr].nst - kslice + p.ks - 1) >> p.lgks;
  c.j = 0;
}

// One chunk of a stage of one warp: the 16*MT x 256 weights at qs (q, swizzled) and ds
// (the chunk's first scale in each DROW-byte row), x block j read at bsrc[j] + boff; adds each
// row's scaled block sums of blocks 2t, 2t+1 to acc.
// SC: the activations were scaled by a power of two for the MMAs; xinv (its inverse) takes
// each block sum back before the block's scale is applied (exact).
// QX: the activations are Q8_0 quants with a scale per block; dx0, dx1 are those of blocks 2t
// and 2t+1, and each block's sum is scaled by the product d_w * d_x.
template <int WT, bool F16, int NW, int CH, bool HALF, bool XS = false, bool SC = false, bool QX = false>
__device__ __forceinline__ void chunk_math(float (&acc)[Cfg<WT, F16, NW, CH>::MT][2], uint32_t qs, const uint8_t* ds,
                                           const uint32_t (&bsrc)[kBlocksPerStage], uint32_t boff, int lrow,
                                           int lsub, int sw, int g, int t, float xinv = 1.0f, float dx0 = 1.0f,
                                           float dx1 = 1.0f) {
  using C = Cfg<WT, F16, NW, CH>;
  constexpr int MT = C::MT;
  float da[MT][4];  // block sums (both halves of a block), column j = block j
  float dl[MT][4];  // XS: the same for the lo vector (scaled by 2^9 in HALF stages)
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) da[mt][i] = dl[mt][i] = 0.f;
#pragma unroll
  for (int bp = 0; bp < kBlocksPerStage / 2; ++bp) {
    uint32_t w[MT][4];  // Q4_0: [tile][row g blk 2bp, row g+8 blk 2bp, row g blk 2bp+1, row g+8 blk 2bp+1]
    if (WT == QMV_Q4_0) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        ldmatrix_x4(w[mt][0], w[mt][1], w[mt][2], w[mt][3],
                    qs + (16 * mt + lrow) * kBox + (((2 * bp + lsub) ^ sw) << 4));
    }
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int k = 2 * bp + hb;
      uint32_t b[4];  // elements (4t, 4t+1), (4t+2, 4t+3), (16+4t, ..), (18+4t, ..) of block k, or zeros
      lds_u32x4(bsrc[k] + boff, b);
      uint32_t bl[4];  // the same of the lo vector (XS: its slots follow the hi ones)
      if (XS) lds_u32x4(bsrc[k] + boff + (uint32_t)(CH * 512), bl);
      if (WT == QMV_Q4_0) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t g01, g23, gh01, gh23, h01, h23, hh01, hh23;
          if (HALF) {
            q4_word_to_f16_levels(w[mt][2 * hb], g01, g23, gh01, gh23);      // row g
            q4_word_to_f16_levels(w[mt][2 * hb + 1], h01, h23, hh01, hh23);  // row g + 8
            mma_f16_16816(da[mt], g01, h01, g23, h23, b[0], b[1], da[mt]);
            mma_f16_16816(da[mt], gh01, hh01, gh23, hh23, b[2], b[3], da[mt]);
            if (XS) {
              mma_f16_16816(dl[mt], g01, h01, g23, h23, bl[0], bl[1], dl[mt]);
              mma_f16_16816(dl[mt], gh01, hh01, gh23, hh23, bl[2], bl[3], dl[mt]);
            }
          } else {
            q4_word_to_bf16_levels(w[mt][2 * hb], g01, g23, gh01, gh23);
            q4_word_to_bf16_levels(w[mt][2 * hb + 1], h01, h23, hh01, hh23);
            mma_bf16_16816(da[mt], g01, h01, g23, h23, b[0], b[1], da[mt]);
            mma_bf16_16816(da[mt], gh01, hh01, gh23, hh23, b[2], b[3], da[mt]);
            if (XS) {
              mma_bf16_16816(dl[mt], g01, h01, g23, h23, bl[0], bl[1], dl[mt]);
              mma_bf16_16816(dl[mt], gh01, hh01, gh23, hh23, bl[2], bl[3], dl[mt]);
            }
          }
        }
      } else {
        // Q8_0: block k = chunks 2k, 2k+1 of the stage (box k / 4)
        uint32_t q[4];  // row g half 0, row g+8 half 0, row g half 1, row g+8 half 1
        const int chunk = 2 * (k & 3) + lsub;
        ldmatrix_x4(q[0], q[1], q[2], q[3], qs + (k >> 2) * C::Q_BOX_BYTES + lrow * kBox + ((chunk ^ sw) << 4));
        uint32_t g0a, g0b, h0a, h0b, g1a, g1b, h1a, h1b;
        if (HALF) {
          q8_word_to_f16_levels(q[0], g0a, g0b);
          q8_word_to_f16_levels(q[1], h0a, h0b);
          q8_word_to_f16_levels(q[2], g1a, g1b);
          q8_word_to_f16_levels(q[3], h1a, h1b);
          mma_f16_16816(da[0], g0a, h0a, g0b, h0b, b[0], b[1], da[0]);
          mma_f16_16816(da[0], g1a, h1a, g1b, h1b, b[2], b[3], da[0]);
          if (XS) {
            mma_f16_16816(dl[0], g0a, h0a, g0b, h0b, bl[0], bl[1], dl[0]);
            mma_f16_16816(dl[0], g1a, h1a, g1b, h1b, bl[2], bl[3], dl[0]);
          }
        } else {
          q8_word_to_bf16_levels(q[0], g0a, g0b);
          q8_word_to_bf16_levels(q[1], h0a, h0b);
          q8_word_to_bf16_levels(q[2], g1a, g1b);
          q8_word_to_bf16_levels(q[3], h1a, h1b);
          mma_bf16_16816(da[0], g0a, h0a, g0b, h0b, b[0], b[1], da[0]);
          mma_bf16_16816(da[0], g1a, h1a, g1b, h1b, b[2], b[3], da[0]);
          if (XS) {
            mma_bf16_16816(dl[0], g0a, h0a, g0b, h0b, bl[0], bl[1], dl[0]);
            mma_bf16_16816(dl[0], g1a, h1a, g1b, h1b, bl[2], bl[3], dl[0]);
          }
        }
      }
    }
  }
  // columns 2t, 2t+1 = blocks 2t, 2t+1; fragment entries [2h], [2h+1] are row g + 8h
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint8_t* dr = ds + (16 * mt + 8 * h + g) * C::DROW;
      float d0, d1;
      if (F16) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(dr + 4 * t);
        d0 = f16_bits_to_f32((uint16_t)(v & 0xFFFF));
        d1 = f16_bits_to_f32((uint16_t)(v >> 16));
      } else {
        const float2 v = *reinterpret_cast<const float2*>(dr + 8 * t);
        d0 = v.x;
        d1 = v.y;
      }
      // XS: the lo vector's sums, scaled back (2^-9 is exact) in HALF stages
      constexpr float kLoBack = HALF ? 0x1p-9f : 1.0f;
      float s0 = XS ? da[mt][2 * h] + dl[mt][2 * h] * kLoBack : da[mt][2 * h];
      float s1 = XS ? da[mt][2 * h + 1] + dl[mt][2 * h + 1] * kLoBack : da[mt][2 * h + 1];
      if (SC) {
        s0 *= xinv;
        s1 *= xinv;
      }
      if (QX) {
        d0 *= dx0;
        d1 *= dx1;
      }
      acc[mt][h] = fmaf(d1, s1, fmaf(d0, s0, acc[mt][h]));
    }
  }
}

// XF (with XS): the activations arrive as float32 (one box of CH x 256 values per stage, the
// bytes of the hi and lo boxes); a stage that rounds to half as above takes them directly, the
// others are split by each lane into hi = RN_bf16(x) and lo = RN_bf16(x - hi) in registers
// (split_bf16_pair, the split kernel's rule), so float32 activations take one launch.
// XQ: the runtime's activation-quantized product: each stage's activations (bfloat16, or float32
// with XF) are quantized by the Q8_0 activation rule in the stage (lanes 4g..4g+3 share block g of
// a chunk: its largest magnitude by two shuffles), the quants enter the MMA as exact halves, so
// each block's dot product is the exact integer sum, scaled by d_w * d_x.
template <int WT, bool F16, int NW, int CH, bool XS, bool GLU = false, bool XF = false, int RD = 2, bool XH = false,
          bool XQ = false>
__global__ void __launch_bounds__(NW * 32) matvec_bdiag_kernel(const __grid_constant__ Maps maps,
                                                               const __grid_constant__ Params p) {
  using C = Cfg<WT, F16, NW, CH, XS, RD, XH, XQ && XF>;
  constexpr int MT = C::MT;
  static_assert(!GLU || (MT == 2 && !XS), "the gated pair takes two 16-row MMA tiles per warp tile");
  static_assert(!XF || XS || XQ, "float32 activations are split into the hi and lo parts, or quantized");
  static_assert(!XQ || (!XS && !XH && !GLU), "the activation-quantized product is a route of its own");
  static_assert(!XH || (!XS && !XF && !GLU), "pre-rounded half activations are a route of their own");
  constexpr bool XP = XS || XH;  // activations with hi and lo parts
  constexpr int TROWS = GLU ? kRows : C::WROWS;  // rows of each matrix per warp tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);  // 1024-aligned: swizzle atoms

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;

  uint8_t* qring = smem + warp * C::Q_WARP;
  uint8_t* dring = smem + C::OFF_D + warp * C::D_WARP;
  uint8_t* xring = smem + C::OFF_X + warp * C::X_WARP;
  const uint32_t slot = smem_u32(smem + C::OFF_SLOT + warp * C::SLOT_WARP + lane * 16);
  const uint32_t zline = smem_u32(smem + C::OFF_ZERO);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + warp * C::S;

  const int tiles_per_item = NW / p.ks;
  const int tile_local = warp / p.ks;
  const int kslice = warp % p.ks;
  constexpr uint32_t stage_tx = (uint32_t)(C::Q_STAGE + C::D_STAGE + C::X_STAGE);

  for (int i = threadIdx.x; i < C::SLOT_WARP / 4; i += NW * 32) reinterpret_cast<uint32_t*>(smem + C::OFF_ZERO)[i] = 0u;
  if (lane == 0) {
    for (int s = 0; s < C::S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();  // zero line and barriers visible
  const uint64_t pol_stream = l2_policy_evict_first();

  // producer cursor: runs S-1 stages ahead of the consumer cursor
  Cursor pc;
  pc.item = (int)blockIdx.x;
  cursor_load(pc, p, tiles_per_item, tile_local, kslice);
  int ps = 0;
  int issued = 0;
  // fill ring slot ps from the producer cursor; with_x = false defers the activation box
  auto issue = [&](bool with_x) {
    if (lane == 0) {
      const Problem& P = p.pr[pc.prob];
      if (pc.tile < P.ntiles) {
        const int c = pc.c0 + (pc.j << p.lgks);  // stage: chunks CH c ..
        mbar_arrive_expect_tx(&bars[ps], stage_tx);
        fence_proxy_async_smem();
        if (GLU) {
          // rows 16t.. of w1 into the stage's first 16 rows, the same rows of w3 into the next 16
#pragma unroll
          for (int b = 0; b < C::NQBOX; ++b)
#pragma unroll
            for (int m = 0; m < 2; ++m)
              tma_load_2d(qring + ps * C::Q_STAGE + b * C::Q_BOX_BYTES + m * kRows * kBox, &maps.q[m],
                          c * (C::kCH * C::QROW) + b * kBox, pc.tile * TROWS, &bars[ps], pol_stream);
#pragma unroll
          for (int m = 0; m < 2; ++m)
            tma_load_2d(dring + ps * C::D_STAGE + m * kRows * C::DROW, &maps.d[m], c * C::DROW, pc.tile * TROWS,
                        &bars[ps], pol_stream);
        } else {
#pragma unroll
          for (int b = 0; b < C::NQBOX; ++b)
            tma_load_2d(qring + ps * C::Q_STAGE + b * C::Q_BOX_BYTES, &maps.q[pc.prob],
                        c * (C::kCH * C::QROW) + b * kBox, pc.tile * C::WROWS, &bars[ps], pol_stream);
          tma_load_2d(dring + ps * C::D_STAGE, &maps.d[pc.prob], c * C::DROW, pc.tile * C::WROWS, &bars[ps],
                      pol_stream);
        }
        if (with_x) {
          tma_load_2d_keep(xring + ps * C::X_STAGE, &maps.x[pc.prob], 0, c * C::kCH, &bars[ps]);
          if (XS && !XF)
            tma_load_2d_keep(xring + ps * C::X_STAGE + C::X_PART, &maps.xl[pc.prob], 0, c * C::kCH, &bars[ps]);
        }
      } else {
        mbar_arrive(&bars[ps]);  // a tile past the end of its problem: complete the phase, no data
      }
    }
  };
  auto advance = [&](Cursor& c) {
    if (++c.j == c.n) {
      c.item += (int)gridDim.x;
      cursor_load(c, p, tiles_per_item, tile_local, kslice);
    }
  };

  // prologue: weight boxes of the first S-1 stages (of the one stage with a ring of one) may be
  // requested before the preceding kernel has finished; activations only after
  // griddepcontrol.wait
  constexpr int kPre = C::S > 1 ? C::S - 1 : 1;
  int pre_c[C::S], pre_prob[C::S];
  bool pre_valid[C::S];
  int pre = 0;
  // launched early without leave to read the weights meanwhile: nothing global before the wait
  if (!p.early) griddep_wait();
  while (pre < kPre && pc.item < p.nitems) {
    pre_c[pre] = pc.c0 + (pc.j << p.lgks);
    pre_prob[pre] = pc.prob;
    pre_valid[pre] = pc.tile < p.pr[pc.prob].ntiles;
    issue(false);
    ps = (ps + 1 == C::S) ? 0 : ps + 1;
    advance(pc);
    ++pre;
  }
  issued = pre;
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (lane == 0) {
    for (int i = 0; i < pre; ++i)
      if (pre_valid[i]) {
        tma_load_2d_keep(xring + i * C::X_STAGE, &maps.x[pre_prob[i]], 0, pre_c[i] * C::kCH, &bars[i]);
        if (XS && !XF)
          tma_load_2d_keep(xring + i * C::X_STAGE + C::X_PART, &maps.xl[pre_prob[i]], 0, pre_c[i] * C::kCH, &bars[i]);
      }
  }

  // ldmatrix: lane supplies row (lane & 7) + 8 * (matrix & 1), 16-byte chunk (matrix >> 1)
  const int lm = lane >> 3;
  const int lrow = (lane & 7) + ((lm & 1) << 3);
  const int lsub = lm >> 1;
  const int sw = lrow & 7;  // 128-byte swizzle: physical chunk = logical chunk ^ (row & 7)
  // activation fragment source of block j: this lane's slot for j = g, else the zero line
  uint32_t bsrc[kBlocksPerStage];
#pragma unroll
  for (int j = 0; j < kBlocksPerStage; ++j) bsrc[j] = (j == g) ? slot : zline;

  float acc[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = 0.f;
  bool failed = false;
  int cs = 0;          // consumer ring slot
  uint32_t phase = 0;  // its parity
  int consumed = 0;
  Cursor cc;
  cc.item = (int)blockIdx.x;
  cursor_load(cc, p, tiles_per_item, tile_local, kslice);
  while (cc.item < p.nitems) {
    const Problem& P = p.pr[cc.prob];
    const bool valid = cc.tile < P.ntiles;
    if (!failed) {
      if (C::S > 1 && pc.item < p.nitems) {
        issue(true);
        ps = (ps + 1 == C::S) ? 0 : ps + 1;
        advance(pc);
        ++issued;
      }
      if (!mbar_wait_bounded(&bars[cs], phase)) {
        record_status(p.status, QMV_E_TIMEOUT);
        failed = true;
      } else {
        ++consumed;
        if (valid) {
          const uint32_t qs = smem_u32(qring + cs * C::Q_STAGE);
          const uint8_t* ds = dring + cs * C::D_STAGE;
          bool rounded = false;
          if constexpr (XS) {
            // activations given as hi + lo (or float32): scaled by a power of two 2^s (from the
            // stage's largest magnitude, so that it lies in [2^14, 2^15)) and rounded once to
            // IEEE half (11 significant bits: at most 2^-11 relative error per term, under half
            // the product's tolerance), one MMA per block as for bfloat16 activations, the block
            // sums taken back by 2^-s; where some value of the stage would round to a subnormal
            // half (a range over 2^28 within the stage) or is not finite, the exact two-part path
            float v[C::kCH][8];
            float amax = 0.f;
#pragma unroll
            for (int h = 0; h < C::kCH; ++h) {
              if (XF) {
                const uint8_t* xf = xring + cs * C::X_STAGE + h * (kTK * 4) + g * 128 + t * 16;
                const float4 fa = *reinterpret_cast<const float4*>(xf);
                const float4 fb = *reinterpret_cast<const float4*>(xf + 64);
                v[h][0] = fa.x, v[h][1] = fa.y, v[h][2] = fa.z, v[h][3] = fa.w;
                v[h][4] = fb.x, v[h][5] = fb.y, v[h][6] = fb.z, v[h][7] = fb.w;
              } else {
                const uint8_t* xh = xring + cs * C::X_STAGE + h * (kTK * 2) + g * 64 + t * 8;
                const uint8_t* xl = xh + C::kCH * (kTK * 2);
                const uint2 ha = *reinterpret_cast<const uint2*>(xh), hb = *reinterpret_cast<const uint2*>(xh + 32);
                const uint2 la = *reinterpret_cast<const uint2*>(xl), lb = *reinterpret_cast<const uint2*>(xl + 32);
                const uint32_t hw[4] = {ha.x, ha.y, hb.x, hb.y}, lw[4] = {la.x, la.y, lb.x, lb.y};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  // exact for a split x (lo under half an ulp of hi); one float32 rounding otherwise
                  v[h][2 * i] = __uint_as_float(hw[i] << 16) + __uint_as_float(lw[i] << 16);
                  v[h][2 * i + 1] = __uint_as_float(hw[i] & 0xFFFF0000u) + __uint_as_float(lw[i] & 0xFFFF0000u);
                }
              }
#pragma unroll
              for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[h][k]));  // a NaN is not taken
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            float xs, xinv;
            bool fits = half_stage_scale(amax, xs, xinv);
            uint32_t rx[C::kCH][4];
#pragma unroll
            for (int h = 0; h < C::kCH; ++h)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                rx[h][i] = f32x2_to_f16x2_normal(v[h][2 * i], v[h][2 * i + 1], xs, fits);
            if (__all_sync(0xffffffffu, fits)) {
              rounded = true;
#pragma unroll
              for (int h = 0; h < C::kCH; ++h) sts_u32x4(slot + h * 512, rx[h][0], rx[h][1], rx[h][2], rx[h][3]);
#pragma unroll
              for (int h = 0; h < C::kCH; ++h)
                chunk_math<WT, F16, NW, CH, true, false, true>(acc, qs + h * C::Q_CHUNK, ds + h * C::DCHUNK, bsrc,
                                                               h * 512u, lrow, lsub, sw, g, t, xinv);
            }
          }
          if constexpr (XQ) {
            // this lane's 8 values of block g of each chunk (elements 4t..4t+3, 16+4t..16+4t+3),
            // quantized with the block's scale; the quants as half pairs in the slot's order
            uint32_t hq[C::kCH][4];
            float dxb[C::kCH];  // the scale of block g of chunk h
            float v[C::kCH][8];
#pragma unroll
            for (int h = 0; h < C::kCH; ++h) {
              if (XF) {
                const uint8_t* xf = xring + cs * C::X_STAGE + h * (kTK * 4) + g * 128 + t * 16;
                const float4 fa = *reinterpret_cast<const float4*>(xf);
                const float4 fb = *reinterpret_cast<const float4*>(xf + 64);
                v[h][0] = fa.x, v[h][1] = fa.y, v[h][2] = fa.z, v[h][3] = fa.w;
                v[h][4] = fb.x, v[h][5] = fb.y, v[h][6] = fb.z, v[h][7] = fb.w;
              } else {
                const uint8_t* xl = xring + cs * C::X_STAGE + h * (kTK * 2) + g * 64 + t * 8;
                const uint2 a = *reinterpret_cast<const uint2*>(xl);
                const uint2 b = *reinterpret_cast<const uint2*>(xl + 32);
                const uint32_t w[4] = {a.x, a.y, b.x, b.y};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  v[h][2 * i] = __uint_as_float(w[i] << 16);
                  v[h][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                }
              }
            }
            act_q8_lane_quarters<C::kCH>(v, hq, dxb);
#pragma unroll
            for (int h = 0; h < C::kCH; ++h) sts_u32x4(slot + h * 512, hq[h][0], hq[h][1], hq[h][2], hq[h][3]);
#pragma unroll
            for (int h = 0; h < C::kCH; ++h) {
              // the scales of blocks 2t and 2t+1 (computed by lanes 8t.. and 8t+4..)
              const float dx0 = __shfl_sync(0xffffffffu, dxb[h], 8 * t);
              const float dx1 = __shfl_sync(0xffffffffu, dxb[h], 8 * t + 4);
              chunk_math<WT, F16, NW, CH, true, false, false, true>(acc, qs + h * C::Q_CHUNK, ds + h * C::DCHUNK,
                                                                    bsrc, h * 512u, lrow, lsub, sw, g, t, 1.0f, dx0,
                                                                    dx1);
            }
            rounded = true;
          }
          const int stage = cc.c0 + (cc.j << p.lgks);  // chunks CH stage ..
          if constexpr (XH) {
            // half values rounded ahead: the stage's chunks all rounded (chunk scales from device
            // memory, the same for every lane), one MMA per block, sums taken back by 2^-s
            float xinv[C::kCH];
            bool all = true;
#pragma unroll
            for (int h = 0; h < C::kCH; ++h) {
              const int ch = stage * C::kCH + h;
              xinv[h] = ch < P.nchunks ? __ldg(P.xinv + ch) : 1.0f;  // chunks past the end: zeros
              all = all && xinv[h] != 0.f;
            }
            if (all) {
              rounded = true;
#pragma unroll
              for (int h = 0; h < C::kCH; ++h) {
                const uint8_t* xl = xring + cs * C::X_STAGE + h * (kTK * 2) + g * 64 + t * 8;
                const uint2 a = *reinterpret_cast<const uint2*>(xl);
                const uint2 b = *reinterpret_cast<const uint2*>(xl + 32);
                sts_u32x4(slot + h * 512, a.x, a.y, b.x, b.y);
              }
#pragma unroll
              for (int h = 0; h < C::kCH; ++h)
                chunk_math<WT, F16, NW, CH, true, false, true>(acc, qs + h * C::Q_CHUNK, ds + h * C::DCHUNK, bsrc,
                                                               h * 512u, lrow, lsub, sw, g, t, xinv[h]);
            }
          }
          // this lane's activations of each chunk h: block g, elements 4t..4t+3 and
          // 16+4t..16+4t+3; its slot for chunk h is 512 bytes after the one for chunk h-1
          // (XS, XH: the same of the lo vector, whose slots follow the hi ones: chunk h at CH + h)
          constexpr int NX = (XP ? 2 : 1) * C::kCH;
          uint2 xa[NX], xb[NX];
          uint32_t hx[NX][4];
          bool exact = true;
          if (!XQ && !rounded) {
          if (XF) {
            // float32 activations: elements 4t..4t+3 and 16+4t..16+4t+3 of block g of each chunk,
            // split into the bf16 hi (chunk h) and lo (chunk CH + h) parts
#pragma unroll
            for (int h = 0; h < C::kCH; ++h) {
              const uint8_t* xf = xring + cs * C::X_STAGE + h * (kTK * 4) + g * 128 + t * 16;
              const float4 fa = *reinterpret_cast<const float4*>(xf);
              const float4 fb = *reinterpret_cast<const float4*>(xf + 64);
              const float v[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
              uint16_t hi[8], lo[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) split_bf16_pair(v[k], hi[k], lo[k]);
              xa[h] = make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
              xb[h] = make_uint2(hi[4] | ((uint32_t)hi[5] << 16), hi[6] | ((uint32_t)hi[7] << 16));
              xa[C::kCH + h] = make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
              xb[C::kCH + h] = make_uint2(lo[4] | ((uint32_t)lo[5] << 16), lo[6] | ((uint32_t)lo[7] << 16));
            }
          }
#pragma unroll
          for (int e = 0; e < NX; ++e) {
            if (XH) {
              // the pair from device memory (hi row, then lo row), zeros past the end
              const int ch = stage * C::kCH + (e % C::kCH);
              xa[e] = xb[e] = make_uint2(0u, 0u);
              if (ch < P.nchunks) {
                const uint16_t* src = P.xg + (e >= C::kCH ? (size_t)P.nchunks * kTK : 0) + (size_t)ch * kTK +
                                      g * 32 + t * 4;
                xa[e] = __ldg(reinterpret_cast<const uint2*>(src));
                xb[e] = __ldg(reinterpret_cast<const uint2*>(src + 16));
              }
            } else if (!XF) {
              const uint8_t* xl = xring + cs * C::X_STAGE + e * (kTK * 2) + g * 64 + t * 8;
              xa[e] = *reinterpret_cast<const uint2*>(xl);
              xb[e] = *reinterpret_cast<const uint2*>(xl + 32);
            }
            // XS, XH: the lo vector (about 2^-9 of hi) scaled by 2^9, exactly, so that its values
            // lie where IEEE half holds them exactly as often as hi's do
            const float sc = (XP && e >= C::kCH) ? 512.0f : 1.0f;
            hx[e][0] = bf16x2_to_f16x2_scaled(xa[e].x, sc, exact);
            hx[e][1] = bf16x2_to_f16x2_scaled(xa[e].y, sc, exact);
            hx[e][2] = bf16x2_to_f16x2_scaled(xb[e].x, sc, exact);
            hx[e][3] = bf16x2_to_f16x2_scaled(xb[e].y, sc, exact);
          }
          if (__all_sync(0xffffffffu, exact)) {
#pragma unroll
            for (int e = 0; e < NX; ++e) sts_u32x4(slot + e * 512, hx[e][0], hx[e][1], hx[e][2], hx[e][3]);
#pragma unroll
            for (int h = 0; h < C::kCH; ++h)
              chunk_math<WT, F16, NW, CH, true, XP>(acc, qs + h * C::Q_CHUNK, ds + h * C::DCHUNK, bsrc, h * 512u,
                                                    lrow, lsub, sw, g, t);
          } else {
#pragma unroll
            for (int e = 0; e < NX; ++e) sts_u32x4(slot + e * 512, xa[e].x, xa[e].y, xb[e].x, xb[e].y);
#pragma unroll
            for (int h = 0; h < C::kCH; ++h)
              chunk_math<WT, F16, NW, CH, false, XP>(acc, qs + h * C::Q_CHUNK, ds + h * C::DCHUNK, bsrc, h * 512u,
                                                     lrow, lsub, sw, g, t);
          }
          }  // !rounded
        }
      }
      __syncwarp();
      // a ring of one: the slot is free only now (every lane has read it)
      if (C::S == 1 && !failed && pc.item < p.nitems) {
        issue(true);
        advance(pc);
        ++issued;
      }
    }

    if (cc.j == cc.n - 1) {  // end of an item: add the lanes' blocks and the column slices, store y
      const int row0 = cc.tile * TROWS;
      // row sums over the four lanes t that share rows g, g + 8 (the same value in all four)
      float v[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float s = acc[mt][h];
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          s += __shfl_xor_sync(0xffffffffu, s, 2);
          v[mt][h] = s;
        }
      // lane t keeps row g + 8 (t & 1) of MMA tile t >> 1 (t < 2 * MT)
      float mine = (t & 1) ? v[0][1] : v[0][0];
      if (MT == 2 && t >= 2) mine = (t & 1) ? v[MT - 1][1] : v[MT - 1][0];
      const int r = 16 * (t >> 1) + 8 * (t & 1) + g;
      const bool holder = t < 2 * MT;
      if (GLU) {
        // gate of row row0 + i in lane i of the tile's first warp, up in lane 16 + i (rows 16..31
        // of the warp tile are w3's); h = act(gate) * up as the bf16 pair
        float sum = 0.f;
        if (p.ks == 1) {
          sum = __shfl_sync(0xffffffffu, mine, ((lane & 15) << 2 & 28) | ((lane >> 4) << 1) | ((lane >> 3) & 1));
        } else {
          if (holder) red[warp * C::WROWS + r] = mine;
          __syncthreads();
          if (kslice == 0)
            for (int k = 0; k < p.ks; ++k) sum += red[(warp + k) * C::WROWS + lane];
        }
        const float up = __shfl_down_sync(0xffffffffu, sum, 16);
        if (kslice == 0 && valid && !failed && lane < kRows && row0 + lane < P.rows) {
          uint16_t hi, lo;
          split_bf16_pair(glu(p.act, sum, up), hi, lo);
          p.h[row0 + lane] = hi;
          p.h[P.rows + row0 + lane] = lo;
        }
        if (p.ks != 1) __syncthreads();
      } else if (p.ks == 1) {
        if (valid && !failed && holder && row0 + r < P.rows) P.y[row0 + r] = mine;
      } else {
        if (holder) red[warp * C::WROWS + r] = mine;
        __syncthreads();
        if (kslice == 0 && valid && !failed && lane < C::WROWS && row0 + lane < P.rows) {
          float sum = 0.f;
          for (int k = 0; k < p.ks; ++k) sum += red[(warp + k) * C::WROWS + lane];
          P.y[row0 + lane] = sum;
        }
        __syncthreads();
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = 0.f;
    }
    cs = (cs + 1 == C::S) ? 0 : cs + 1;
    if (cs == 0) phase ^= 1u;
    advance(cc);
  }
  if (failed) {
    // let this warp's copies still in flight land before the CTA's shared memory is released
    for (int j = consumed; j < issued; ++j)
      mbar_wait_bounded(&bars[j % C::S], (uint32_t)(j / C::S) & 1u, 400000000LL);
  }
}

// One warps-per-CTA choice's plan for a launch: the column split ks with the smallest
// estimate of the launch's duration, in 1/40 stage.  A launch with more items than resident
// CTAs runs in waves of `grid` items (the last one partly filled), each as long as one item:
// ceil(nst / ks) stages plus, for ks > 1, a CTA-wide reduction (about a quarter stage);
// with ks = 1 a warp walks a row alone, which measured about 10% slower per stage.
struct Plan {
  int ks = 1, nitems = 0, grid = 0, smem = 0;
  long long cost = -1;
  long long longest = 0;  // stages of the longest warp's item
  long long waves = 0;
};

template <int WT, bool F16, int NW, int CH, bool XS, bool GLU = false, bool XF = false, int RD = 2, bool XH = false,
          bool XQ = false>
cudaError_t plan_typed(const MatrixRef* ms, int n, const DeviceInfo& dev, Plan* out) {
  using C = Cfg<WT, F16, NW, CH, XS, RD, XH, XQ && XF>;
  auto kern = matvec_bdiag_kernel<WT, F16, NW, CH, XS, GLU, XF, RD, XH, XQ>;
  // per device: the shared-memory attribute set and the occupancy known (0 = does not fit)
  static std::mutex mu;
  static bool ready[64] = {};
  static int ctas_per_sm[64] = {};
  if (dev.device < 0 || dev.device >= 64 || n < 1 || n > kMaxProblems) return cudaErrorInvalidValue;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev.device]) {
      int k = 0;
      if ((size_t)C::SMEM <= dev.smem_optin) {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (err != cudaSuccess) return err;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, kern, NW * 32, C::SMEM);
        if (err != cudaSuccess) return err;
      }
      ctas_per_sm[dev.device] = k;
      ready[dev.device] = true;
    }
  }
  *out = Plan{};
  if (ctas_per_sm[dev.device] == 0) return cudaSuccess;  // does not fit: cost stays -1
  const long long slots = (long long)ctas_per_sm[dev.device] * dev.sm_count;
  long long min_stages = 1LL << 30;
  for (int i = 0; i < n; ++i) {
    const long long nst = (ms[i].cols / kTK + C::kCH - 1) / C::kCH;
    if (nst < min_stages) min_stages = nst;
  }
  Plan best;
  for (int ks = 1; ks <= NW && ks <= min_stages; ks *= 2) {
    const int tpi = NW / ks;
    long long items = 0, longest = 0;
    for (int i = 0; i < n; ++i) {
      items += ((ms[i].rows + C::WROWS - 1) / C::WROWS + tpi - 1) / tpi;
      const long long st = ((ms[i].cols / kTK + C::kCH - 1) / C::kCH + ks - 1) / ks;
      if (st > longest) longest = st;
    }
    const long long grid = items < slots ? items : slots;
    const long long waves = (items + grid - 1) / grid;
    const long long cost = waves * (longest * (ks == 1 ? 44 : 40) + (ks > 1 ? 10 : 0));
    if (best.cost < 0 || cost < best.cost || (cost == best.cost && grid < best.grid)) {
      best.cost = cost;
      best.ks = ks;
      best.nitems = (int)items;
      best.grid = (int)grid;
      best.longest = longest;
      best.waves = waves;
    }
  }
  best.smem = C::SMEM;
  *out = best;
  return cudaSuccess;
}

// GLU: ms = {w1, w3} (same shape), one x (xs[0]); the pair is one problem whose warp tiles are
// 16 rows of each; act and h as in Params.
// XH: xs[i] is the problem's area of the half route's buffer: the bfloat16 hi row and lo row
// (cols each), the half row, then the chunks' inverse scales (cols / 256 floats).
template <int WT, bool F16, int NW, int CH, bool XS, bool GLU = false, bool XF = false, int RD = 2, bool XH = false,
          bool XQ = false>
cudaError_t launch_typed(const Plan& plan, const MatrixRef* ms, const void* const* xs, float* const* ys, int n,
                         bool pdl, const DeviceInfo& dev, cudaStream_t stream, int act = -1, uint16_t* h = nullptr) {
  using C = Cfg<WT, F16, NW, CH, XS, RD, XH, XQ && XF>;
  constexpr int TROWS = GLU ? kRows : C::WROWS;  // rows of each matrix per warp tile
  if (GLU && (n != 2 || ms[0].rows != ms[1].rows || ms[0].cols != ms[1].cols || h == nullptr))
    return cudaErrorInvalidValue;
  Params p{};
  p.nprob = GLU ? 1 : n;
  p.status = dev.status;
  p.ks = plan.ks;
  p.lgks = 31 - __builtin_clz((unsigned)plan.ks);
  p.act = act;
  p.early = pdl ? 1 : 0;
  p.h = h;
  const int tpi = NW / plan.ks;
  int items = 0;
  for (int i = 0; i < p.nprob; ++i) {
    p.pr[i].y = GLU ? nullptr : ys[i];
    p.pr[i].rows = (int)ms[i].rows;
    p.pr[i].ntiles = (int)((ms[i].rows + TROWS - 1) / TROWS);
    p.pr[i].nst = (int)((ms[i].cols / kTK + C::kCH - 1) / C::kCH);
    p.pr[i].item0 = items;
    p.pr[i].nchunks = (int)(ms[i].cols / kTK);
    if (XH) {
      p.pr[i].xg = static_cast<const uint16_t*>(xs[i]);
      p.pr[i].xinv = reinterpret_cast<const float*>(static_cast<const uint16_t*>(xs[i]) + 3 * ms[i].cols);
    }
    items += (p.pr[i].ntiles + tpi - 1) / tpi;
  }
  if (items != plan.nitems) return cudaErrorInvalidValue;
  p.nitems = items;

  Maps maps;
  memset(&maps, 0, sizeof(maps));
  for (int i = 0; i < n; ++i) {
    const MatrixRef& m = ms[i];
    const uint64_t qrow = (WT == QMV_Q4_0) ? (uint64_t)m.cols / 2 : (uint64_t)m.cols;
    const uint64_t drow = (uint64_t)(m.cols / 32) * (F16 ? 2 : 4);
    cudaError_t err = encode_tmap_2d(&maps.q[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, m.q, qrow, (uint64_t)m.rows, qrow,
                                     kBox, TROWS, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    err = encode_tmap_2d(&maps.d[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, m.d, drow, (uint64_t)m.rows, drow, C::DROW,
                         TROWS, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
    if (GLU && i == 1) continue;  // one x for the pair
    if (XF) {  // float32 activations, split in the kernel
      err = encode_tmap_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xs[i], kTK, (uint64_t)(m.cols / kTK), kTK * 4,
                           kTK, C::kCH, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (err != cudaSuccess) return err;
      continue;
    }
    // (XH: the half row; two-byte elements as a bfloat16 vector's)
    const void* xb = XH ? static_cast<const void*>(static_cast<const uint16_t*>(xs[i]) + 2 * m.cols) : xs[i];
    err = encode_tmap_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xb, kTK, (uint64_t)(m.cols / kTK), kTK * 2,
                         kTK, C::kCH, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
    if (XS) {  // the lo vector follows the hi one
      const void* lo = static_cast<const uint8_t*>(xs[i]) + (size_t)m.cols * 2;
      err = encode_tmap_2d(&maps.xl[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lo, kTK, (uint64_t)(m.cols / kTK), kTK * 2,
                           kTK, C::kCH, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (err != cudaSuccess) return err;
    }
  }

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  // always a programmatic dependent: the CTAs start and set up during the preceding kernel's
  // tail; without pdl they wait for it before their first global access (p.early = 0)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, matvec_bdiag_kernel<WT, F16, NW, CH, XS, GLU, XF, RD, XH, XQ>, maps, p);
}

// Q4_0 launches of at least this many weight bytes take one-chunk stages.
constexpr long long kOneChunkBytes = 32LL << 20;

// Stages of two chunks in 4-warp CTAs; when that leaves SMs without a CTA (a launch with few
// tiles), 8-warp CTAs instead if their estimate is smaller.  One-chunk stages fit more warps per
// SM (five 4-warp CTAs instead of two): measured faster on large Q4_0 launches, slower on
// launches of a few tens of MB (the Llama-7B layer's, the 4096 x 4096 product) and on Q8_0.
// GLU: ms = {w1, w3}, planned as one matrix of twice the rows (the same warp tiles: 16 rows of
// each per tile); act and h as in launch_typed.
template <int WT, bool F16, bool XS, bool GLU = false, bool XF = false, bool XH = false, bool XQ = false>
cudaError_t launch_best(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                        const DeviceInfo& dev, cudaStream_t stream, int act = -1, uint16_t* h = nullptr) {
  MatrixRef pair[1];
  const MatrixRef* pm = ms;
  int pn = n;
  if (GLU) {
    pair[0] = ms[0];
    pair[0].rows = 2 * ms[0].rows;
    pm = pair;
    pn = 1;
  }
  Plan p4, p8;
  cudaError_t err;
  if (WT == QMV_Q4_0 && !XS) {
    long long bytes = 0;
    for (int i = 0; i < pn; ++i) bytes += pm[i].rows * pm[i].cols / 2;
    if (bytes >= kOneChunkBytes) {
      Plan p1;
      err = plan_typed<WT, F16, 4, 1, XS, GLU, XF, 2, XH, XQ>(pm, pn, dev, &p1);
      if (err != cudaSuccess) return err;
      if (p1.cost >= 0 && p1.grid > dev.sm_count)
        return launch_typed<WT, F16, 4, 1, XS, GLU, XF, 2, XH, XQ>(p1, ms, xs, ys, n, pdl, dev, stream, act, h);
    }
  }
  err = plan_typed<WT, F16, 4, 2, XS, GLU, XF, 2, XH, XQ>(pm, pn, dev, &p4);
  if (err != cudaSuccess) return err;
  if constexpr (!XS && !GLU) {
    if (p4.cost >= 0 && p4.longest > 1) {
      // 8-warp CTAs with a ring of one: every warp one stage, in one wave, where 4-warp CTAs
      // give each warp two or more stages one after the other
      Plan p1;
      err = plan_typed<WT, F16, 8, 2, XS, GLU, XF, 1, XH, XQ>(pm, pn, dev, &p1);
      if (err != cudaSuccess) return err;
      if (p1.cost >= 0 && p1.longest == 1 && p1.waves == 1 && p1.grid > dev.sm_count)
        return launch_typed<WT, F16, 8, 2, XS, GLU, XF, 1, XH, XQ>(p1, ms, xs, ys, n, pdl, dev, stream, act, h);
    }
  }
  if (p4.cost >= 0 && p4.grid > dev.sm_count)
    return launch_typed<WT, F16, 4, 2, XS, GLU, XF, 2, XH, XQ>(p4, ms, xs, ys, n, pdl, dev, stream, act, h);
  err = plan_typed<WT, F16, 8, 2, XS, GLU, XF, 2, XH, XQ>(pm, pn, dev, &p8);
  if (err != cudaSuccess) return err;
  if (p8.cost >= 0 && (p4.cost < 0 || p8.cost < p4.cost))
    return launch_typed<WT, F16, 8, 2, XS, GLU, XF, 2, XH, XQ>(p8, ms, xs, ys, n, pdl, dev, stream, act, h);
  if (p4.cost < 0) return cudaErrorInvalidConfiguration;
  return launch_typed<WT, F16, 4, 2, XS, GLU, XF, 2, XH, XQ>(p4, ms, xs, ys, n, pdl, dev, stream, act, h);
}

template <bool XS, bool XF = false, bool XH = false, bool XQ = false>
cudaError_t launch_any(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                       const DeviceInfo& dev, cudaStream_t stream) {
  const MatrixRef& m = ms[0];
  if (m.wtype == QMV_Q4_0)
    return m.scale_f16 ? launch_best<QMV_Q4_0, true, XS, false, XF, XH, XQ>(ms, xs, ys, n, pdl, dev, stream)
                       : launch_best<QMV_Q4_0, false, XS, false, XF, XH, XQ>(ms, xs, ys, n, pdl, dev, stream);
  return m.scale_f16 ? launch_best<QMV_Q8_0, true, XS, false, XF, XH, XQ>(ms, xs, ys, n, pdl, dev, stream)
                     : launch_best<QMV_Q8_0, false, XS, false, XF, XH, XQ>(ms, xs, ys, n, pdl, dev, stream);
}

}  // namespace

cudaError_t launch_matvec_bdiag(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                const DeviceInfo& dev, cudaStream_t stream) {
  return launch_any<false>(ms, xs, ys, n, pdl, dev, stream);
}

cudaError_t launch_matvec_bdiag_split(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                      const DeviceInfo& dev, cudaStream_t stream) {
  return launch_any<true>(ms, xs, ys, n, pdl, dev, stream);
}

cudaError_t launch_matvec_bdiag_half(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                     const DeviceInfo& dev, cudaStream_t stream) {
  return launch_any<false, false, true>(ms, xs, ys, n, pdl, dev, stream);
}

cudaError_t launch_matvec_bdiag_qx(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool x_bf16,
                                   bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  return x_bf16 ? launch_any<false, false, false, true>(ms, xs, ys, n, pdl, dev, stream)
                : launch_any<false, true, false, true>(ms, xs, ys, n, pdl, dev, stream);
}

cudaError_t launch_matvec_bdiag_f32in(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                      const DeviceInfo& dev, cudaStream_t stream) {
  return launch_any<true, true>(ms, xs, ys, n, pdl, dev, stream);
}

bool matvec_bdiag_glu_supported(const MatrixRef& w1, const MatrixRef& w3) {
  return w1.wtype == QMV_Q4_0 && w3.wtype == QMV_Q4_0 && w1.scale_f16 == w3.scale_f16 && w1.rows == w3.rows &&
         w1.cols == w3.cols && w1.cols % kTK == 0 && w1.rows < (1LL << 30);
}

cudaError_t launch_matvec_bdiag_glu(const MatrixRef& w1, const MatrixRef& w3, const void* x, int act, uint16_t* h,
                                    bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  if (!matvec_bdiag_glu_supported(w1, w3) || (act != 0 && act != 1)) return cudaErrorInvalidValue;
  const MatrixRef ms[2] = {w1, w3};
  const void* xs[2] = {x, x};
  float* ys[2] = {nullptr, nullptr};
  return w1.scale_f16 ? launch_best<QMV_Q4_0, true, false, true>(ms, xs, ys, 2, pdl, dev, stream, act, h)
                      : launch_best<QMV_Q4_0, false, false, true>(ms, xs, ys, 2, pdl, dev, stream, act, h);
}

}  // namespace qmv
