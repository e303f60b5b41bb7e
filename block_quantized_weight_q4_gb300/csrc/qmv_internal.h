// qmv_internal.h -- launchers shared between the libqmv translation units (host side).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qmv {

// Validated description of one matrix image (see include/qmv.h).
struct MatrixRef {
  int wtype;        // QMV_Q8_0 or QMV_Q4_0
  int scale_f16;    // 0: f32 scales, 1: f16 scales
  int64_t rows;
  int64_t cols;     // multiple of 32
  const uint8_t* q; // q array (device)
  const uint8_t* d; // d array (device) = q + round_up(q bytes, 64)
};

struct DeviceInfo {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  size_t smem_optin;
  size_t smem_per_sm;     // shared memory of one SM
  size_t smem_reserved;   // of it, what the system keeps per resident CTA
  int* status;  // device address of this device's status word
};

// Scratch of the tensor-memory decode kernel: arrival counters and the parts of tiles split
// between CTAs.  One per stream (calls on one stream never overlap).  The counters are zero
// between launches (the last arrival at a tile resets its counter).
struct Workspace {
  unsigned* counters;         // arrival counters
  int max_counters;
  float* partials;            // parts of split tiles
  size_t max_partial_floats;
};
// Bytes of the counter region for n counters (a multiple of 256); carve `bytes` at `base`
// into n counters followed by the parts.
size_t workspace_counter_bytes(int n);
void workspace_carve(void* base, size_t bytes, int n, Workspace* ws);
// The workspace of (current device, stream), allocated and zeroed on first use; returns
// cudaErrorNotReady when there is none yet and the stream is being captured.
cudaError_t stream_workspace(const DeviceInfo& dev, cudaStream_t stream, Workspace* ws);
// The same for the prefill kernel's split tiles (a separate, larger workspace per stream).
cudaError_t stream_prefill_workspace(const DeviceInfo& dev, cudaStream_t stream, Workspace* ws);
// Zero the counters of every workspace (decode and prefill) of the current device (after a kernel gave up on a
// bounded wait, a counter may have been left part-way); synchronous.
cudaError_t reset_workspaces();

// 2-D tiled tensor map over a row-major array: inner_elems elements of `dtype`
// (a CUtensorMapDataType) per row, `outer` rows, rows row_stride_bytes apart; box of
// box_inner x box_outer elements; swizzle is a CUtensorMapSwizzle; out-of-range reads
// are zero-filled.
cudaError_t encode_tmap_2d(CUtensorMap* map, int dtype, const void* base, uint64_t inner_elems, uint64_t outer,
                           uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle);

// Cached properties of the current device.
cudaError_t current_device_info(DeviceInfo* info);

cudaError_t launch_dequant(const MatrixRef& m, float* out, cudaStream_t stream);
// The writer rules into W (q at W, d at W + d_off; zeros between q_bytes and d_off).  wtype:
// QMV_Q8_0, QMV_Q4_0 (the round rule) or kQuantQ4Fit (the Q4_0 best-fit rule).
constexpr int kQuantQ4Fit = 3;
cudaError_t launch_quantize(int wtype, bool scale_f16, int64_t rows, int64_t cols, const float* src, uint8_t* W,
                            int64_t d_off, int64_t q_bytes, int64_t* first_bad, const DeviceInfo& dev,
                            cudaStream_t stream);
cudaError_t launch_validate(const MatrixRef& m, int64_t* first_bad, cudaStream_t stream);
// Create every per-stream workspace of `stream` now (not while it is captured), and free them.
cudaError_t prepare_stream_workspaces(const DeviceInfo& dev, cudaStream_t stream);
cudaError_t release_stream_workspaces(int device, cudaStream_t stream);
// GGUF interleaved records (18-byte Q4_0, 34-byte Q8_0) into the two-array layout with f16
// scales at W (q at W, d at W + d_off; zeros between q_bytes and d_off).
cudaError_t launch_gguf_to_mlb(int wtype, int64_t rows, int64_t cols, const void* src, uint8_t* W, int64_t d_off,
                               int64_t q_bytes, const DeviceInfo& dev, cudaStream_t stream);
// The activation quantizer (Q8_0 rule, f32 scale) into xq (q at xq, d at xq + d_off).
cudaError_t launch_quantize_x(bool x_bf16, int64_t batch, int64_t cols, const void* x, uint8_t* xq, int64_t d_off,
                              int64_t q_bytes, cudaStream_t stream);
// The same rule for up to 8 activation arrays in one launch (x[i]: nblk[i] blocks of 32, bf16 or
// f32; the quants to q[i], the scales to d[i]).  The kernel lets the next launch start at once
// (its dependents wait for it to finish); pdl: launch as a programmatic dependent (x is read
// only after the preceding kernel has finished).
struct QxImages {
  static constexpr int kMax = 8;
  const void* x[kMax];
  uint8_t* q[kMax];
  float* d[kMax];
  long long nblk[kMax];
};
cudaError_t launch_quantize_x_group(bool x_bf16, const QxImages& a, int n, bool pdl, cudaStream_t stream);
// The activation-quantized product y[v][r] = sum_b d_w d_x (integer dot of levels and quants);
// xq / xd: the quants and scales of the batch x cols Q8_0 / f32 activation image.
cudaError_t launch_matvec_qx(const MatrixRef& m, const int8_t* xq, const float* xd, int batch, float* y,
                             const DeviceInfo& dev, cudaStream_t stream);
// The same product on the tensor core (quants and levels as exact halves, mma.sync), cols % 256
// == 0, for 1..matvec_mma_max_problems() problems of one weight type and scale type (problem i:
// ms[i], its image xq[i] / xd[i], ys[i]), batch in passes of up to 8.  pdl: launch as a
// programmatic dependent.
cudaError_t launch_matvec_qx_mma(const MatrixRef* ms, const int8_t* const* xq, const float* const* xd, int n,
                                 int batch, float* const* ys, bool pdl, const DeviceInfo& dev, cudaStream_t stream);
// The stream's split buffer (split_buffer_bytes(), 256-byte aligned, allocated on first use and
// kept), which the float32 split routes and the grouped activation-quantized route write into.
size_t split_buffer_bytes();
cudaError_t stream_split_buffer(const DeviceInfo& dev, cudaStream_t stream, uint8_t** base);
// The same product for 1..8 problems of one weight type and scale type in one launch per pass
// of 8 vectors, each with its float activations (batch x cols, bf16 or f32), which the kernel
// quantizes itself (the bytes launch_quantize_x writes) into shared memory: needs
// min(batch, 8) * cols * 9 / 8 bytes of shared memory for the largest cols of the group.
cudaError_t launch_matvec_qx_fused(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool x_bf16,
                                   int batch, bool pdl, const DeviceInfo& dev, cudaStream_t stream);

// Any shape with cols % 32 == 0; batch 1..8 per call.
cudaError_t launch_matvec_simple(const MatrixRef& m, const void* x, bool x_bf16, float* y, int batch,
                                 const DeviceInfo& dev, cudaStream_t stream);

// cols % 256 == 0; 1..matvec_mma_max_problems() problems of the same wtype, scale type and
// x type per launch (ms[i], xs[i], ys[i]); batch 1..8.  pdl: launch as a programmatic
// dependent of the preceding kernel (weights are read before that kernel finishes).
bool matvec_mma_supported(const MatrixRef& m);
int matvec_mma_max_problems();
cudaError_t launch_matvec_mma(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool x_bf16,
                              int batch, bool pdl, const DeviceInfo& dev, cudaStream_t stream);

// The same problems with one bfloat16 activation vector (batch 1), block-diagonal
// activation fragments and half-precision operands where exact (decode_bdiag.cu); takes
// every problem matvec_mma_supported() accepts.
cudaError_t launch_matvec_bdiag(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                const DeviceInfo& dev, cudaStream_t stream);
// The same with each activation vector given as two bfloat16 vectors hi and lo (x = hi + lo,
// lo in the cols following hi): every block's MMAs run once with each into the same sums.
cudaError_t launch_matvec_bdiag_split(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                      const DeviceInfo& dev, cudaStream_t stream);
// The FFN's gated pair (Q4_0, one bfloat16 vector x): w1 x and w3 x in one launch, written as
// h = act(w1 x) * (w3 x) in the bfloat16 pair layout launch_matvec_bdiag_split reads (hi parts
// at h[r], lo parts at h[rows + r]); act 0 SiLU, 1 GELU-tanh.
bool matvec_bdiag_glu_supported(const MatrixRef& w1, const MatrixRef& w3);
cudaError_t launch_matvec_bdiag_glu(const MatrixRef& w1, const MatrixRef& w3, const void* x, int act, uint16_t* h,
                                    bool pdl, const DeviceInfo& dev, cudaStream_t stream);
// The runtime's activation-quantized product (the same quants, scales and float32 steps as
// launch_matvec_qx after launch_quantize_x) for one activation vector per problem (bfloat16, or
// float32 16-byte aligned), quantized in the kernel's activation stage; every problem
// matvec_mma_supported().
cudaError_t launch_matvec_bdiag_qx(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool x_bf16,
                                   bool pdl, const DeviceInfo& dev, cudaStream_t stream);
// The same problems with the activations rounded to half ahead of the product: xs[i] is the
// problem's area written by the half route's split (launch_matvec_bdiag_f32): the bfloat16 hi and
// lo rows, the half row and the chunks' inverse scales (0: that chunk takes hi and lo).
cudaError_t launch_matvec_bdiag_half(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                     const DeviceInfo& dev, cudaStream_t stream);
// One float32 activation vector per problem (16-byte aligned), split into bfloat16 hi + lo in
// the kernel's activation stage (one launch; the same parts and results as below).
cudaError_t launch_matvec_bdiag_f32in(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                      const DeviceInfo& dev, cudaStream_t stream);
// One float32 activation vector per problem: split in the stream's split buffer into the hi + lo
// bfloat16 rows and, per 256-column chunk, the values rounded to half after a power-of-two scale
// (about 6 bytes per column: up to about 340,000 columns over the problems), then the half route
// above.  Fails (nothing launched) when the buffer would not hold them, or cannot be created
// while the stream is being captured.
// act >= 0: xs are gates, the activations act(gate) * up with up at gate + up_batch * cols floats.
cudaError_t launch_matvec_bdiag_f32(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                    const DeviceInfo& dev, cudaStream_t stream, int act = -1, long long up_batch = 0);

// Batched product on the 5th-generation tensor core (weights dequantized in tensor memory as
// bf16 hi + lo parts, or rounded once to bf16 when bf16_weights; tcgen05 MMA, f32 accumulators
// in tensor memory): bf16 activations, cols % 256 == 0, 1..128 vectors per launch (meant for
// 16 and more).  ws: the stream's prefill workspace, or null (then no tile is split between
// CTAs).  pdl: launch as a programmatic dependent of the preceding kernel (weights are read
// before that kernel finishes).
bool prefill_supported(const MatrixRef& m, bool x_bf16);
int prefill_max_batch();
cudaError_t launch_prefill(const MatrixRef& m, const void* x, float* y, int batch, bool bf16_weights,
                           const DeviceInfo& dev, const Workspace* ws, bool pdl, cudaStream_t stream);

// Decode product on the 5th-generation tensor core with the weights unpacked into tensor
// memory: bf16 activations, cols % 256 == 0, 1..8 vectors, 1..decode_tc_max_problems()
// problems of the same wtype and scale type per launch.
bool decode_tc_supported(const MatrixRef& m);
int decode_tc_max_problems();
cudaError_t launch_decode_tc(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch, bool pdl,
                             const DeviceInfo& dev, const Workspace& ws, cudaStream_t stream);

// The same product for float32 activations: x is first split into bfloat16 pairs hi + lo
// (hi = RN_bf16(x), lo = RN_bf16(x - hi)) in a buffer of the stream, 16 rows per problem
// (hi of the vectors in rows 0..7, lo in 8..15), which the kernel takes as its 16 MMA
// columns and adds per vector.  Needs decode_tc_f32_fits (the buffer holds 65,536 columns
// over the problems) and a stream that is not being captured when it has no buffer yet.
bool decode_tc_f32_fits(const MatrixRef* ms, int n);
cudaError_t launch_decode_tc_f32(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch,
                                 bool pdl, const DeviceInfo& dev, const Workspace& ws, cudaStream_t stream,
                                 int act = -1, long long up_batch = 0);

}  // namespace qmv
