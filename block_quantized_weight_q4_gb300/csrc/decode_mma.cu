// decode_mma.cu -- the decode product (batch 1..8 per pass) for cols % 256 == 0.
//
// What is computed (Krafla ".mlb model format v1", "Q8_0", "Q4_0", "Body"):
//   y[n][r] = sum_k d[r][k] * sum_{j<32} level[r][32k+j] * x[n][32k+j]
// with level = nibble - 8 (Q4_0) or the int8 quant (Q8_0), d the block's scale.
//
// How:
//   * Work.  A warp owns tiles of 16*MT rows (MT = 2 for Q4_0, 1 for Q8_0: one or two 16-row
//     MMA tiles sharing the activation fragments); the columns are cut into chunks of 256
//     weights (8 blocks).  A CTA of NW warps (4, or 8 or 16 for launches with few tiles) takes items
//     of (NW/ks) tiles x ks column slices and walks its items persistently (item =
//     blockIdx.x, + gridDim.x, ...); each warp sees one continuous stream of stages across
//     its items.
//   * Streams.  Each warp has its own ring of S shared-memory stages.  Lane 0 fills a stage
//     with 2-D TMA loads: the (16*MT)-row x 128-byte q box (128-byte swizzle; two boxes for
//     Q8_0), the (16*MT)-row x 8-scale d box, and the batch x 256 activation box.  Rows past
//     the end of the matrix read as zeros and are never stored.
//   * Unpack.  ldmatrix (addresses swizzled like the TMA box) hands thread (g = lane/4,
//     t = lane%4) the 4 quant bytes 4t..4t+3 of a block for rows g and g+8.  They become
//     exact bfloat16 levels in registers (Q4_0: 0x4300|nibble = 128+n, minus 136; Q8_0:
//     through the float32 2^23 trick), paired as elements (4t, 4t+1) and (4t+2, 4t+3).
//   * Block dot.  Per block, two m16n8k16 bf16 MMAs (elements 0-15 and 16-31 of the block)
//     into a zeroed f32 fragment give sum_j level*x for 16 rows x 8 activation vectors.
//     Inside an MMA, k slots (2t, 2t+1, 2t+8, 2t+9) hold elements (4t .. 4t+3) of the half
//     block, for A and B alike, so thread t's B fragment is the 8 contiguous bytes
//     x[n][4t .. 4t+3] of vector n = g: one shared-memory load.  Lanes whose g is past the
//     batch read a zero area instead.
//   * Scale and accumulate.  acc += d[row][block] * fragment, float32 FFMA.
//   * Split-K.  Warps of one item that share a tile add their partial sums through shared
//     memory in a fixed order (a reduction area, or, in the variant without one, the q slot
//     each warp has just consumed); one warp writes y.
//   * Groups.  One launch may carry up to 8 problems of the same types and batch (for
//     example the projections of a layer that read the same input); items of all problems
//     form one list that the persistent CTAs walk.
//   * Launched as a programmatic dependent of the preceding kernel: the CTAs start and set up
//     during its tail.  With the overlap flag the weight boxes of the first stages are also
//     requested before griddepcontrol.wait (the weights must then not be written by the
//     preceding kernel); without it nothing global is touched before the wait.  The
//     activations are read and y is written only after it.
// f32 activations are split x = hi + lo (two bfloat16s, hi = RN(x)) and take two MMAs each,
// which keeps 16 significant bits of x.
// XQ: the runtime's activation-quantized product on an activation image of Q8_0 quants with a
// float32 scale per block (qmv_quantize_x's bytes): the stage's activation boxes are the quants
// (batch x 256 bytes) and the scales (batch x 8 floats); quants and levels enter the MMA as
// exact IEEE halves (m16n8k16 f16), so each block's dot product is the exact integer sum, and
// acc += (d_w * d_x) * sum, the float32 steps of the dp4a product.
#include <cstring>
#include <mutex>

#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {

namespace {

constexpr int kTK = 256;             // weights per stage and row
constexpr int kBlocksPerStage = kTK / 32;
constexpr int kRows = 16;            // rows per MMA tile
constexpr int kBox = 128;            // q box inner extent in bytes (the 128-byte swizzle span)
constexpr int kMaxBatch = 8;         // activation vectors per pass (the MMA's N)
constexpr int kMaxProblems = 8;      // problems per grouped launch

template <int WT, bool F16, bool XBF16, int NW, bool XQ = false, bool RS = false>
struct Cfg {
  static constexpr int kWarps = NW;
  static constexpr int MT = (WT == QMV_Q4_0) ? 2 : 1;           // 16-row MMA tiles per warp tile
  static constexpr int WROWS = MT * kRows;                        // rows per warp tile
  static constexpr int NQBOX = (WT == QMV_Q4_0) ? 1 : 2;        // q boxes per stage
  static constexpr int Q_BOX_BYTES = WROWS * kBox;
  static constexpr int Q_STAGE = NQBOX * Q_BOX_BYTES;             // bytes, multiple of 1024
  static constexpr int QROW = NQBOX * kBox;                        // q bytes per row per stage
  static constexpr int DROW = kBlocksPerStage * (F16 ? 2 : 4);    // scale bytes per row per stage
  static constexpr int D_STAGE = WROWS * DROW;                     // multiple of 128
  static constexpr int XROW = XQ ? kTK : kTK * (XBF16 ? 2 : 4);    // activation bytes per vector per stage
  static constexpr int XDROW = XQ ? kBlocksPerStage * 4 : 0;       // XQ: activation scale bytes per vector
  // ring depth: 2 (3 measured slower: it halves the CTAs per SM that shared memory allows, e.g.
  // 14336 x 4096 Q4_0 at 8 vectors 14.0 against 10.0 us)
  static constexpr int S = 2;
  static constexpr int Q_WARP = S * Q_STAGE;
  static constexpr int D_WARP = S * D_STAGE;
  static constexpr int ZERO_BYTES = 128;
  // fixed part: q rings, d rings, zero area, reduction area (WROWS x 8 floats per warp, where
  // a split tile's column slices meet), barriers; the activation rings (S x batch x XROW per
  // warp) follow.  RS: no reduction area -- the slices meet in the q slot each warp has just
  // consumed, whose index each warp leaves after the barriers.  That saves 4 KB per CTA and is
  // taken where it lets an SM hold one CTA more and the launch fills them (65536 x 4096 Q4_0 at
  // 8 quantized vectors, three to four CTAs per SM: 42.5 against 45.6 us, at 4 bf16 vectors
  // 36.9 against 39.5 us); in launches whose occupancy it does not raise it measured 2-4% slower
  static constexpr int OFF_D = kWarps * Q_WARP;
  static constexpr int OFF_ZERO = OFF_D + kWarps * D_WARP;
  static constexpr int OFF_RED = OFF_ZERO + ZERO_BYTES;
  static constexpr int RED_FLOATS = RS ? 0 : kWarps * WROWS * 8;
  static constexpr int OFF_BAR = OFF_RED + RED_FLOATS * 4;
  static constexpr int OFF_SLOT = OFF_BAR + kWarps * S * 8;
  static constexpr int OFF_X = RS ? (OFF_SLOT + kWarps * 4 + 127) / 128 * 128
                                  : OFF_BAR + ((kWarps * S * 8 + 127) / 128) * 128;
  static_assert(WROWS * 8 * 4 <= Q_STAGE, "a q slot holds a warp's partial sums");
  // activation bytes of one stage (quants then scales with XQ), a multiple of 128 (TMA destinations)
  static __host__ __device__ int x_stage(int batch) { return (batch * (XROW + XDROW) + 127) / 128 * 128; }
  static int smem_bytes(int batch) { return 1024 + OFF_X + kWarps * S * x_stage(batch); }
};

struct Problem {
  float* y;
  int rows;
  int cols;
  int ntiles;   // warp tiles (16*MT rows)
  int nchunks;  // cols / 256
  int item0;    // first item of this problem in the group's item list
};

struct Params {
  int nprob;
  int batch;    // 1..8
  int ks;       // column slices per tile (1, 2, 4, 8, 16); at most every problem's nchunks
  int nitems;
  int early;    // the weights may be read before the preceding kernel has finished
  int* status;
  Problem pr[kMaxProblems];
};

struct Maps {  // per problem: q (128-byte swizzle), d, and activation tensor maps
  CUtensorMap q[kMaxProblems];
  CUtensorMap d[kMaxProblems];
  CUtensorMap x[kMaxProblems];
  CUtensorMap xd[kMaxProblems];  // XQ: the activation scales
};

// Position of a warp in its stream of stages: item (global index), its problem and warp
// tile, this warp's first chunk and chunk count in the item, and the position within.
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
  const int nch = p.pr[pr].nchunks;
  const int lg = 31 - __clz(p.ks);  // ks is a power of two
  c.c0 = (kslice * nch) >> lg;
  c.n = (((kslice + 1) * nch) >> lg) - c.c0;
  c.j = 0;
}

template <int WT, bool F16, bool XBF16, int NW, bool XQ = false, bool RS = false>
__global__ void __launch_bounds__(NW * 32) matvec_mma_kernel(const __grid_constant__ Maps maps,
                                                             const __grid_constant__ Params p) {
  using C = Cfg<WT, F16, XBF16, NW, XQ, RS>;
  constexpr int kWarps = NW;
  constexpr int MT = C::MT;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);  // 1024-aligned: swizzle atoms

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;

  const int x_stage = C::x_stage(p.batch);
  uint8_t* qring = smem + warp * C::Q_WARP;
  uint8_t* dring = smem + C::OFF_D + warp * C::D_WARP;
  uint8_t* xring = smem + C::OFF_X + warp * C::S * x_stage;
  uint8_t* zero = smem + C::OFF_ZERO;
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  int* red_slot = reinterpret_cast<int*>(smem + C::OFF_SLOT);  // RS: per warp, the q slot holding its partial sums
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + warp * C::S;

  const int tiles_per_item = kWarps / p.ks;
  const int tile_local = warp / p.ks;
  const int kslice = warp % p.ks;
  // bytes the copies of one stage deliver (the activation area may be padded beyond them)
  const uint32_t stage_tx = (uint32_t)(C::Q_STAGE + C::D_STAGE + p.batch * (C::XROW + C::XDROW));

  if (threadIdx.x < C::ZERO_BYTES / 4) reinterpret_cast<uint32_t*>(zero)[threadIdx.x] = 0u;
  if (lane == 0) {
    for (int s = 0; s < C::S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();  // zero area and barriers visible
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
        const int c = pc.c0 + pc.j;
        mbar_arrive_expect_tx(&bars[ps], stage_tx);
        fence_proxy_async_smem();
#pragma unroll
        for (int b = 0; b < C::NQBOX; ++b)
          tma_load_2d(qring + ps * C::Q_STAGE + b * C::Q_BOX_BYTES, &maps.q[pc.prob], c * C::QROW + b * kBox,
                      pc.tile * C::WROWS, &bars[ps], pol_stream);
        tma_load_2d(dring + ps * C::D_STAGE, &maps.d[pc.prob], c * C::DROW, pc.tile * C::WROWS, &bars[ps],
                    pol_stream);
        if (with_x) {
          tma_load_2d_keep(xring + ps * x_stage, &maps.x[pc.prob], c * kTK, 0, &bars[ps]);
          if (XQ)
            tma_load_2d_keep(xring + ps * x_stage + p.batch * C::XROW, &maps.xd[pc.prob], c * kBlocksPerStage, 0,
                             &bars[ps]);
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

  // prologue: weight boxes of the first S-1 stages may be requested before the preceding
  // kernel has finished; activations only after griddepcontrol.wait
  int pre_c[C::S], pre_prob[C::S];
  bool pre_valid[C::S];
  int pre = 0;
  // launched early without leave to read the weights meanwhile: nothing global before the wait
  if (!p.early) griddep_wait();
  while (pre < C::S - 1 && pc.item < p.nitems) {
    pre_c[pre] = pc.c0 + pc.j;
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
        tma_load_2d_keep(xring + i * x_stage, &maps.x[pre_prob[i]], pre_c[i] * kTK, 0, &bars[i]);
        if (XQ)
          tma_load_2d_keep(xring + i * x_stage + p.batch * C::XROW, &maps.xd[pre_prob[i]], pre_c[i] * kBlocksPerStage,
                           0, &bars[i]);
      }
  }

  // ldmatrix: lane supplies row (lane & 7) + 8 * (matrix & 1), 16-byte chunk (matrix >> 1)
  const int lm = lane >> 3;
  const int lrow = (lane & 7) + ((lm & 1) << 3);
  const int lsub = lm >> 1;
  const int sw = lrow & 7;  // 128-byte swizzle: physical chunk = logical chunk ^ (row & 7)
  // B fragment source of this lane: vector g of the stage's activation box, or the zero area
  constexpr int XESZ = XQ ? 1 : XBF16 ? 2 : 4;
  const bool xlive = g < p.batch;
  const uint32_t xblk = xlive ? 32 * XESZ : 0;   // byte step per block
  const uint32_t xhalf = xlive ? 16 * XESZ : 0;  // byte step to elements 16..31
  const uint32_t xlane = (xlive ? (uint32_t)(g * C::XROW) : 0u) + 4 * XESZ * t;

  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
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
      if (pc.item < p.nitems) {
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
        const uint32_t xs = (xlive ? smem_u32(xring + cs * x_stage) : smem_u32(zero)) + xlane;
#pragma unroll
        for (int bp = 0; bp < kBlocksPerStage / 2; ++bp) {
          uint32_t w[MT][4];  // Q4_0: [tile][row g blk 2bp, row g+8 blk 2bp, row g blk 2bp+1, row g+8 blk 2bp+1]
          if (WT == QMV_Q4_0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
              ldmatrix_x4(w[mt][0], w[mt][1], w[mt][2], w[mt][3],
                          qs + (16 * mt + lrow) * kBox + (((2 * bp + lsub) ^ sw) << 4));
          }
          // scales of blocks 2bp, 2bp+1 for rows g + 16 mt (h = 0) and g + 8 + 16 mt (h = 1)
          float dsc[MT][2][2];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint8_t* dr = ds + (16 * mt + 8 * h + g) * C::DROW;
              if (F16) {
                const uint32_t v = *reinterpret_cast<const uint32_t*>(dr + 4 * bp);
                dsc[mt][h][0] = f16_bits_to_f32((uint16_t)(v & 0xFFFF));
                dsc[mt][h][1] = f16_bits_to_f32((uint16_t)(v >> 16));
              } else {
                const float2 v = *reinterpret_cast<const float2*>(dr + 8 * bp);
                dsc[mt][h][0] = v.x;
                dsc[mt][h][1] = v.y;
              }
            }
          }
          // XQ: the activation scales of blocks 2bp, 2bp+1 for vectors 2t, 2t+1 (the fragment's
          // columns of this thread; 0 past the batch)
          float dxb[2][2];
          if (XQ) {
            const float* xdq = reinterpret_cast<const float*>(xring + cs * x_stage + p.batch * C::XROW);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int n = 2 * t + j;
                dxb[hb][j] = n < p.batch ? xdq[n * kBlocksPerStage + 2 * bp + hb] : 0.f;
              }
          }
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const int k = 2 * bp + hb;
            // B fragments: [half][pair]; hi/lo split for f32 activations
            uint32_t xh[2][2], xl[2][2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t a = xs + k * xblk + h * xhalf;
              if (XQ) {
                q8_word_to_f16_levels(lds_u32(a), xh[h][0], xh[h][1]);  // quants as exact halves
              } else if (XBF16) {
                lds_u32x2(a, xh[h][0], xh[h][1]);
              } else {
                float v[4];
                lds_f32x4(a, v);
                xh[h][0] = pack_bf16x2(v[0], v[1]);
                xh[h][1] = pack_bf16x2(v[2], v[3]);
                xl[h][0] = pack_bf16x2(v[0] - __uint_as_float(xh[h][0] << 16),
                                       v[1] - __uint_as_float(xh[h][0] & 0xFFFF0000u));
                xl[h][1] = pack_bf16x2(v[2] - __uint_as_float(xh[h][1] << 16),
                                       v[3] - __uint_as_float(xh[h][1] & 0xFFFF0000u));
              }
            }
            if (WT == QMV_Q4_0) {
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                uint32_t g01, g23, gh01, gh23, h01, h23, hh01, hh23;
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                if (XQ) {
                  q4_word_to_f16_levels(w[mt][2 * hb], g01, g23, gh01, gh23);      // row g
                  q4_word_to_f16_levels(w[mt][2 * hb + 1], h01, h23, hh01, hh23);  // row g + 8
                  mma_f16_16816(c, g01, h01, g23, h23, xh[0][0], xh[0][1], c);      // elements 0..15
                  mma_f16_16816(c, gh01, hh01, gh23, hh23, xh[1][0], xh[1][1], c);  // elements 16..31
                } else {
                  q4_word_to_bf16_levels(w[mt][2 * hb], g01, g23, gh01, gh23);      // row g
                  q4_word_to_bf16_levels(w[mt][2 * hb + 1], h01, h23, hh01, hh23);  // row g + 8
                  mma_bf16_16816(c, g01, h01, g23, h23, xh[0][0], xh[0][1], c);      // elements 0..15
                  mma_bf16_16816(c, gh01, hh01, gh23, hh23, xh[1][0], xh[1][1], c);  // elements 16..31
                  if (!XBF16) {
                    mma_bf16_16816(c, g01, h01, g23, h23, xl[0][0], xl[0][1], c);
                    mma_bf16_16816(c, gh01, hh01, gh23, hh23, xl[1][0], xl[1][1], c);
                  }
                }
                if (XQ) {
                  acc[mt][0] = fmaf(dsc[mt][0][hb] * dxb[hb][0], c[0], acc[mt][0]);
                  acc[mt][1] = fmaf(dsc[mt][0][hb] * dxb[hb][1], c[1], acc[mt][1]);
                  acc[mt][2] = fmaf(dsc[mt][1][hb] * dxb[hb][0], c[2], acc[mt][2]);
                  acc[mt][3] = fmaf(dsc[mt][1][hb] * dxb[hb][1], c[3], acc[mt][3]);
                } else {
                  acc[mt][0] = fmaf(dsc[mt][0][hb], c[0], acc[mt][0]);
                  acc[mt][1] = fmaf(dsc[mt][0][hb], c[1], acc[mt][1]);
                  acc[mt][2] = fmaf(dsc[mt][1][hb], c[2], acc[mt][2]);
                  acc[mt][3] = fmaf(dsc[mt][1][hb], c[3], acc[mt][3]);
                }
              }
            } else {
              // Q8_0: block k = chunks 2k, 2k+1 of the stage (box k / 4)
              uint32_t q[4];  // row g half 0, row g+8 half 0, row g half 1, row g+8 half 1
              const int chunk = 2 * (k & 3) + lsub;
              ldmatrix_x4(q[0], q[1], q[2], q[3], qs + (k >> 2) * C::Q_BOX_BYTES + lrow * kBox + ((chunk ^ sw) << 4));
              uint32_t g0a, g0b, h0a, h0b, g1a, g1b, h1a, h1b;
              float c[4] = {0.f, 0.f, 0.f, 0.f};
              if (XQ) {
                q8_word_to_f16_levels(q[0], g0a, g0b);
                q8_word_to_f16_levels(q[1], h0a, h0b);
                q8_word_to_f16_levels(q[2], g1a, g1b);
                q8_word_to_f16_levels(q[3], h1a, h1b);
                mma_f16_16816(c, g0a, h0a, g0b, h0b, xh[0][0], xh[0][1], c);
                mma_f16_16816(c, g1a, h1a, g1b, h1b, xh[1][0], xh[1][1], c);
                acc[0][0] = fmaf(dsc[0][0][hb] * dxb[hb][0], c[0], acc[0][0]);
                acc[0][1] = fmaf(dsc[0][0][hb] * dxb[hb][1], c[1], acc[0][1]);
                acc[0][2] = fmaf(dsc[0][1][hb] * dxb[hb][0], c[2], acc[0][2]);
                acc[0][3] = fmaf(dsc[0][1][hb] * dxb[hb][1], c[3], acc[0][3]);
              } else {
                q8_word_to_bf16_levels(q[0], g0a, g0b);
                q8_word_to_bf16_levels(q[1], h0a, h0b);
                q8_word_to_bf16_levels(q[2], g1a, g1b);
                q8_word_to_bf16_levels(q[3], h1a, h1b);
                mma_bf16_16816(c, g0a, h0a, g0b, h0b, xh[0][0], xh[0][1], c);
                mma_bf16_16816(c, g1a, h1a, g1b, h1b, xh[1][0], xh[1][1], c);
                if (!XBF16) {
                  mma_bf16_16816(c, g0a, h0a, g0b, h0b, xl[0][0], xl[0][1], c);
                  mma_bf16_16816(c, g1a, h1a, g1b, h1b, xl[1][0], xl[1][1], c);
                }
                acc[0][0] = fmaf(dsc[0][0][hb], c[0], acc[0][0]);
                acc[0][1] = fmaf(dsc[0][0][hb], c[1], acc[0][1]);
                acc[0][2] = fmaf(dsc[0][1][hb], c[2], acc[0][2]);
                acc[0][3] = fmaf(dsc[0][1][hb], c[3], acc[0][3]);
              }
            }
          }
        }
        }
      }
      __syncwarp();
    }

    if (cc.j == cc.n - 1) {  // end of an item: add the column slices, store y
      const int row0 = cc.tile * C::WROWS;
      if (p.ks == 1) {
        if (valid && !failed) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int r0 = row0 + 16 * mt + g, r1 = r0 + 8;
            const int n0 = 2 * t, n1 = 2 * t + 1;
            if (n0 < p.batch && r0 < P.rows) P.y[(size_t)n0 * P.rows + r0] = acc[mt][0];
            if (n1 < p.batch && r0 < P.rows) P.y[(size_t)n1 * P.rows + r0] = acc[mt][1];
            if (n0 < p.batch && r1 < P.rows) P.y[(size_t)n0 * P.rows + r1] = acc[mt][2];
            if (n1 < p.batch && r1 < P.rows) P.y[(size_t)n1 * P.rows + r1] = acc[mt][3];
          }
        }
      } else {
        // RS: slot cs was consumed above (all lanes, __syncwarp) and is filled again only after
        // the second __syncthreads below (the next issue(), whose proxy fence orders these
        // accesses before its copies)
        float* my = RS ? reinterpret_cast<float*>(qring + cs * C::Q_STAGE) : red + warp * (C::WROWS * 8);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          my[(16 * mt + g) * 8 + 2 * t] = acc[mt][0];
          my[(16 * mt + g) * 8 + 2 * t + 1] = acc[mt][1];
          my[(16 * mt + g + 8) * 8 + 2 * t] = acc[mt][2];
          my[(16 * mt + g + 8) * 8 + 2 * t + 1] = acc[mt][3];
        }
        if (RS && lane == 0) red_slot[warp] = cs;
        __syncthreads();
        if (kslice == 0 && valid && !failed) {
#pragma unroll
          for (int i = 0; i < C::WROWS * 8 / 32; ++i) {
            const int v = i * 32 + lane;
            const int n = v / C::WROWS;
            const int r = v % C::WROWS;
            if (n < p.batch && row0 + r < P.rows) {
              float sum = 0.f;
              for (int k = 0; k < p.ks; ++k) {
                const float* part =
                    RS ? reinterpret_cast<const float*>(smem + (warp + k) * C::Q_WARP + red_slot[warp + k] * C::Q_STAGE)
                       : red + (warp + k) * (C::WROWS * 8);
                sum += part[r * 8 + n];
              }
              P.y[(size_t)n * P.rows + row0 + r] = sum;
            }
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
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

// One warps-per-CTA choice's plan for a launch: column split, item count, grid, and the
// estimated stages on the critical path (the stages of an even share of all items plus one
// item's stages for the tail, plus half a stage per item for the CTA-wide reduction that a
// split needs).
struct Plan {
  int ks = 1, nitems = 0, grid = 0, smem = 0;
  int per_sm = 0;  // CTAs an SM can hold
  bool rs = false;  // the kernel without the reduction area (Cfg::RS)
  long cost = -1;
};

// The kernel's dynamic shared-memory limit raised to at least `smem` on this device (one
// record per kernel and device, shared by the planner and the launcher).
template <int WT, bool F16, bool XBF16, int NW, bool XQ, bool RS>
cudaError_t raise_smem_limit(int device, int smem) {
  static std::mutex mu;
  static int attr_smem[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (smem <= attr_smem[device]) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(matvec_mma_kernel<WT, F16, XBF16, NW, XQ, RS>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err == cudaSuccess) attr_smem[device] = smem;
  return err;
}

template <int WT, bool F16, bool XBF16, int NW, bool XQ = false>
cudaError_t plan_typed(const MatrixRef* ms, int n, int batch, const DeviceInfo& dev, Plan* out) {
  using C = Cfg<WT, F16, XBF16, NW, XQ, false>;
  int smem_rs = 0;  // the RS variant's shared memory (four warps per CTA only)
  if constexpr (NW == 4) smem_rs = Cfg<WT, F16, XBF16, NW, XQ, true>::smem_bytes(batch);
  // per device and batch: occupancy known, with the reduction area [0] and without [1] (four
  // warps per CTA only); 0 = does not fit
  static std::mutex mu;
  static bool ready[64][kMaxBatch + 1] = {};
  static int ctas_per_sm[64][kMaxBatch + 1][2] = {};
  if (dev.device < 0 || dev.device >= 64 || batch < 1 || batch > kMaxBatch || n < 1 || n > kMaxProblems)
    return cudaErrorInvalidValue;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev.device][batch]) {
      int k = 0;
      if ((size_t)C::smem_bytes(batch) <= dev.smem_optin) {
        cudaError_t err = raise_smem_limit<WT, F16, XBF16, NW, XQ, false>(dev.device, C::smem_bytes(batch));
        if (err != cudaSuccess) return err;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, matvec_mma_kernel<WT, F16, XBF16, NW, XQ, false>,
                                                            NW * 32, C::smem_bytes(batch));
        if (err != cudaSuccess) return err;
      }
      ctas_per_sm[dev.device][batch][0] = k;
      k = 0;
      if constexpr (NW == 4) {
        if ((size_t)smem_rs <= dev.smem_optin) {
          cudaError_t err = raise_smem_limit<WT, F16, XBF16, NW, XQ, true>(dev.device, smem_rs);
          if (err != cudaSuccess) return err;
          err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, matvec_mma_kernel<WT, F16, XBF16, NW, XQ, true>,
                                                              NW * 32, smem_rs);
          if (err != cudaSuccess) return err;
        }
      }
      ctas_per_sm[dev.device][batch][1] = k;
      ready[dev.device][batch] = true;
    }
  }
  *out = Plan{};
  const int occ = ctas_per_sm[dev.device][batch][0];
  const int occ_slot = ctas_per_sm[dev.device][batch][1];
  if (occ == 0) return cudaSuccess;  // does not fit: cost stays -1
  const long slots = (long)occ * dev.sm_count;
  long min_chunks = 1L << 30;
  for (int i = 0; i < n; ++i)
    if (ms[i].cols / kTK < min_chunks) min_chunks = ms[i].cols / kTK;
  Plan best;
  for (int ks = 1; ks <= NW && ks <= min_chunks; ks *= 2) {
    const int tpi = NW / ks;
    long items = 0, units = 0, longest = 0;
    for (int i = 0; i < n; ++i) {
      const long it = ((ms[i].rows + C::WROWS - 1) / C::WROWS + tpi - 1) / tpi;
      const long st = (ms[i].cols / kTK + ks - 1) / ks;
      items += it;
      units += it * st;
      if (st > longest) longest = st;
    }
    const long grid = items < slots ? items : slots;
    const long per_cta = (items + grid - 1) / grid;
    const long cost = 2 * ((units + grid - 1) / grid + longest) + (ks > 1 ? per_cta : 0);
    if (best.cost < 0 || cost < best.cost) {
      best.cost = cost;
      best.ks = ks;
      best.nitems = (int)items;
      best.grid = (int)grid;
    }
  }
  best.smem = C::smem_bytes(batch);
  best.per_sm = occ;
  // without the reduction area an SM may hold more CTAs: taken when the items fill them
  if (occ_slot > occ && best.nitems >= (long)occ_slot * dev.sm_count) {
    best.rs = true;
    best.smem = smem_rs;
    best.per_sm = occ_slot;
    best.grid = occ_slot * dev.sm_count;
  }
  *out = best;
  return cudaSuccess;
}

// XQ: xs[i] is the problem's activation quants (batch x cols bytes), xds[i] their scales
// (batch x cols / 32 floats).
template <int WT, bool F16, bool XBF16, int NW, bool XQ = false, bool RS = false>
cudaError_t launch_typed(const Plan& plan, const MatrixRef* ms, const void* const* xs, float* const* ys, int n,
                         int batch, bool pdl, const DeviceInfo& dev, cudaStream_t stream,
                         const float* const* xds = nullptr) {
  using C = Cfg<WT, F16, XBF16, NW, XQ, RS>;
  if (plan.rs != RS || plan.smem < C::smem_bytes(batch)) return cudaErrorInvalidValue;
  Params p{};
  p.nprob = n;
  p.batch = batch;
  p.status = dev.status;
  p.ks = plan.ks;
  p.early = pdl ? 1 : 0;
  const int tpi = NW / plan.ks;
  int items = 0;
  for (int i = 0; i < n; ++i) {
    p.pr[i].y = ys[i];
    p.pr[i].rows = (int)ms[i].rows;
    p.pr[i].cols = (int)ms[i].cols;
    p.pr[i].ntiles = (int)((ms[i].rows + C::WROWS - 1) / C::WROWS);
    p.pr[i].nchunks = (int)(ms[i].cols / kTK);
    p.pr[i].item0 = items;
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
                                     kBox, C::WROWS, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    err = encode_tmap_2d(&maps.d[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, m.d, drow, (uint64_t)m.rows, drow, C::DROW,
                         C::WROWS, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
    if (XQ) {
      err = encode_tmap_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, xs[i], (uint64_t)m.cols, (uint64_t)batch,
                           (uint64_t)m.cols, kTK, batch, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (err != cudaSuccess) return err;
      err = encode_tmap_2d(&maps.xd[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xds[i], (uint64_t)(m.cols / 32),
                           (uint64_t)batch, (uint64_t)(m.cols / 32) * 4, kBlocksPerStage, batch,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
      if (err != cudaSuccess) return err;
      continue;
    }
    err = encode_tmap_2d(&maps.x[i], XBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xs[i],
                         (uint64_t)m.cols, (uint64_t)batch, (uint64_t)m.cols * (XBF16 ? 2 : 4), kTK, batch,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
  }

  // A grid smaller than the SMs can hold: each CTA asks for enough shared memory that an SM
  // holds no more CTAs than the grid needs per SM, so the hardware spreads the CTAs over all
  // SMs instead of filling some (14336 x 4096 Q4_0 at 4 bf16 vectors, 344 CTAs, four per SM
  // allowed: 11.0 against 9.2 us with at most three)
  int smem = plan.smem;
  const int need = (plan.grid + dev.sm_count - 1) / dev.sm_count;
  if (need < plan.per_sm && dev.smem_per_sm > 0) {
    const size_t spread = (dev.smem_per_sm / (size_t)(need + 1) + 128 - dev.smem_reserved + 127) / 128 * 128;
    if (spread > (size_t)smem && spread <= dev.smem_optin) smem = (int)spread;
  }
  if (smem > plan.smem) {
    const cudaError_t err = raise_smem_limit<WT, F16, XBF16, NW, XQ, RS>(dev.device, smem);
    if (err != cudaSuccess) return err;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // always a programmatic dependent: the CTAs start and set up during the preceding kernel's
  // tail; without pdl they wait for it before their first global access (p.early = 0)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, matvec_mma_kernel<WT, F16, XBF16, NW, XQ, RS>, maps, p);
}

// 4 warps per CTA; when that leaves SMs without a CTA (a launch with few tiles), 8 or 16
// warps per CTA instead if the plan estimates them shorter (ties to fewer warps).  With
// every SM busy, more warps per CTA measured slower (they share the SM's issue slots).
template <int WT, bool F16, bool XBF16, bool XQ = false>
cudaError_t launch_best(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch, bool pdl,
                        const DeviceInfo& dev, cudaStream_t stream, const float* const* xds = nullptr) {
  Plan p4, p8, p16;
  cudaError_t err = plan_typed<WT, F16, XBF16, 4, XQ>(ms, n, batch, dev, &p4);
  if (err != cudaSuccess) return err;
  auto launch4 = [&]() {
    return p4.rs ? launch_typed<WT, F16, XBF16, 4, XQ, true>(p4, ms, xs, ys, n, batch, pdl, dev, stream, xds)
                 : launch_typed<WT, F16, XBF16, 4, XQ>(p4, ms, xs, ys, n, batch, pdl, dev, stream, xds);
  };
  if (p4.cost >= 0 && p4.grid > dev.sm_count) return launch4();
  err = plan_typed<WT, F16, XBF16, 8, XQ>(ms, n, batch, dev, &p8);
  if (err != cudaSuccess) return err;
  err = plan_typed<WT, F16, XBF16, 16, XQ>(ms, n, batch, dev, &p16);
  if (err != cudaSuccess) return err;
  auto better = [](const Plan& a, const Plan& b) { return a.cost >= 0 && (b.cost < 0 || a.cost < b.cost); };
  if (better(p16, p8) && better(p16, p4))
    return launch_typed<WT, F16, XBF16, 16, XQ>(p16, ms, xs, ys, n, batch, pdl, dev, stream, xds);
  if (better(p8, p4)) return launch_typed<WT, F16, XBF16, 8, XQ>(p8, ms, xs, ys, n, batch, pdl, dev, stream, xds);
  if (p4.cost < 0) return cudaErrorInvalidConfiguration;
  return launch4();
}

}  // namespace

bool matvec_mma_supported(const MatrixRef& m) {
  return m.cols % kTK == 0 && m.rows < (1LL << 31) - 64 && m.cols < (1LL << 30);
}

int matvec_mma_max_problems() { return kMaxProblems; }

cudaError_t launch_matvec_qx_mma(const MatrixRef* ms, const int8_t* const* xq, const float* const* xd, int n,
                                 int batch, float* const* ys, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  if (batch < 1 || n < 1 || n > kMaxProblems) return cudaErrorInvalidValue;
  for (int i = 0; i < n; ++i)
    if (!matvec_mma_supported(ms[i]) || ms[i].wtype != ms[0].wtype || ms[i].scale_f16 != ms[0].scale_f16)
      return cudaErrorInvalidValue;
  const MatrixRef& m = ms[0];
  for (int b0 = 0; b0 < batch; b0 += kMaxBatch) {
    const int nb = (batch - b0) < kMaxBatch ? (batch - b0) : kMaxBatch;
    const void* xs[kMaxProblems];
    const float* xds[kMaxProblems];
    float* yp[kMaxProblems];
    for (int i = 0; i < n; ++i) {
      xs[i] = xq[i] + (size_t)b0 * (size_t)ms[i].cols;
      xds[i] = xd[i] + (size_t)b0 * (size_t)(ms[i].cols / 32);
      yp[i] = ys[i] + (size_t)b0 * (size_t)ms[i].rows;
    }
    cudaError_t err;
    if (m.wtype == QMV_Q4_0)
      err = m.scale_f16 ? launch_best<QMV_Q4_0, true, true, true>(ms, xs, yp, n, nb, pdl, dev, stream, xds)
                        : launch_best<QMV_Q4_0, false, true, true>(ms, xs, yp, n, nb, pdl, dev, stream, xds);
    else
      err = m.scale_f16 ? launch_best<QMV_Q8_0, true, true, true>(ms, xs, yp, n, nb, pdl, dev, stream, xds)
                        : launch_best<QMV_Q8_0, false, true, true>(ms, xs, yp, n, nb, pdl, dev, stream, xds);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_matvec_mma(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool x_bf16,
                              int batch, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  const MatrixRef& m = ms[0];
  if (m.wtype == QMV_Q4_0) {
    if (m.scale_f16) return x_bf16 ? launch_best<QMV_Q4_0, true, true>(ms, xs, ys, n, batch, pdl, dev, stream)
                                   : launch_best<QMV_Q4_0, true, false>(ms, xs, ys, n, batch, pdl, dev, stream);
    return x_bf16 ? launch_best<QMV_Q4_0, false, true>(ms, xs, ys, n, batch, pdl, dev, stream)
                  : launch_best<QMV_Q4_0, false, false>(ms, xs, ys, n, batch, pdl, dev, stream);
  }
  if (m.scale_f16) return x_bf16 ? launch_best<QMV_Q8_0, true, true>(ms, xs, ys, n, batch, pdl, dev, stream)
                                 : launch_best<QMV_Q8_0, true, false>(ms, xs, ys, n, batch, pdl, dev, stream);
  return x_bf16 ? launch_best<QMV_Q8_0, false, true>(ms, xs, ys, n, batch, pdl, dev, stream)
                : launch_best<QMV_Q8_0, false, false>(ms, xs, ys, n, batch, pdl, dev, stream);
}

}  // namespace qmv
