/*
 * qmv.h -- C ABI of libqmv: products against block-quantized (Q8_0 / Q4_0) weight
 * matrices on NVIDIA GB300 (sm_103a).
 *
 * Format (Krafla ".mlb model format v1" page, sections "Body", "Q8_0", "Q4_0"):
 *   A rows x cols matrix (cols a multiple of 32) is stored as its q array, then its d
 *   array, each array's length rounded up to a 64-byte boundary with zero bytes (the tail
 *   of the last array is never read here, so whether a file carries it does not matter):
 *     q : Q8_0: rows*cols int8 quants, row-major.
 *         Q4_0: rows*cols/2 bytes; block k of row r is the 16 bytes at r*cols/2 + 16k;
 *               the low four bits of byte j are the block's element j, the high four bits
 *               its element j+16; the weight is (nibble - 8) * d.
 *     d : rows*cols/32 scales: the scale of row r's k-th run of 32 weights at index
 *         r*cols/32 + k; float32, or IEEE binary16 when the file's scale_f16 flag is 1.
 *         Q8_0 weight = q * d.
 *   Row r of the matrix gives output r: y[r] = sum_c W[r][c] * x[c].
 *
 * Conventions for every entry point:
 *   - W points at the q array.  The d array starts at W + qmv_scale_offset(...), i.e.
 *     at q's size rounded up to 64 bytes, exactly as in the file.  W must be a device
 *     pointer aligned to 16 bytes (the file format gives 64).
 *   - x is batch x cols, row-major, float32 or bfloat16; y is batch x rows float32,
 *     row-major.  Device pointers, 16-byte aligned for x and out, 4 for y.  The y of the
 *     products (qmv_matvec, qmv_matvec_grouped, qmv_matvec_grouped_noalloc, qmv_matvec_qx,
 *     qmv_matvec_qx_grouped) may instead be pinned host memory that the device addresses
 *     directly (cudaHostAlloc or cudaHostRegister memory under unified addressing, the same
 *     address on both sides): the kernels only store to y, and their stores then cross to
 *     the host, which saves a copy after the launch.
 *   - All memory is owned by the caller; the library allocates no device memory per
 *     call.  Work is enqueued on `stream` (0 = the legacy default stream) of the calling
 *     thread's current device, and the call returns without waiting, except where noted.
 *   - Argument errors are found on the host, before anything is launched; nothing is
 *     written then.  A CUDA launch error returns QMV_E_CUDA.
 *   - Errors met inside a running kernel (a bounded wait that ran out) are recorded in
 *     a per-device status word that qmv_check_device() returns; the kernel then returns
 *     without finishing its output.
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* wtype: the .mlb header's wtype field (offset 44). */
#define QMV_Q8_0 1
#define QMV_Q4_0 2

/* scale_dtype: the header's scale_f16 field (offset 120). */
#define QMV_SCALE_F32 0
#define QMV_SCALE_F16 1

/* x_dtype: element type of the activations. */
#define QMV_X_F32 0
#define QMV_X_BF16 1
/* Gated activations, the FFN down projection's input (Krafla page, "Body": w1 gate, w3 up,
 * w2 down; header field act): x holds two batch x cols float32 arrays one after the other,
 * gate (w1 x) then up (w3 x), and the product's activations are act(gate) * up, formed in
 * float32 in the activation prep of the float32 routes (no launch of its own):
 *   QMV_X_SILU_GLU_F32: act(g) = g / (1 + e^-g)
 *   QMV_X_GELU_GLU_F32: act(g) = g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))
 * with CUDA's expf / tanhf.  They need cols % 256 == 0 (QMV_E_SHAPE otherwise), at most
 * 65,536 columns over a group's problems when batch >= 2, and the stream's split buffer (made
 * on the stream's first float32 or gated call outside stream capture, or by qmv_step_create);
 * QMV_E_ARG otherwise.  The tolerance of the product is taken against the exact
 * act(gate) * up. */
#define QMV_X_SILU_GLU_F32 2
#define QMV_X_GELU_GLU_F32 3
/* One activation vector given as a bfloat16 pair (batch must be 1): x holds cols bfloat16 hi
 * parts followed by cols bfloat16 lo parts, the activations being hi + lo (formed in float32);
 * the block-diagonal kernel takes them as it takes one float32 vector (each stage rounded once
 * to half after a power-of-two scale, or both parts where that would not hold every value as a
 * normal half).  This is the layout qmv_matvec_glu writes.  cols % 256 == 0 (QMV_E_SHAPE
 * otherwise), batch other than 0 or 1 gives QMV_E_ARG. */
#define QMV_X_BF16_PAIR 4

/* act of qmv_matvec_glu (the .mlb header's act field): */
#define QMV_ACT_SILU 0      /* SiLU(g) = g / (1 + e^-g) */
#define QMV_ACT_GELU_TANH 1 /* GELU(g) = g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) */

/* Status codes.  QMV_E_FORMAT and QMV_E_SHAPE mirror the loader's ML_E_FORMAT and
 * ML_E_SHAPE classes (Krafla page, "Validation done by the loader"): an unknown enum
 * value or an invalid quant is a format error; a zero dimension, cols not a multiple of
 * 32, or a size that overflows is a shape error. */
#define QMV_OK 0
#define QMV_E_FORMAT 2
#define QMV_E_SHAPE 3
#define QMV_E_ARG 4     /* null pointer, negative batch                             */
#define QMV_E_ALIGN 5   /* a pointer not aligned as stated above                    */
#define QMV_E_CUDA 6    /* a CUDA call failed (launch error, no device, no sm_103a) */
#define QMV_E_TIMEOUT 7 /* a kernel's bounded wait ran out (see qmv_check_device)   */

/* q8_mask class bits (Krafla page, header offset 72: the mask has a bit for each class of
 * matrix).  wq/wk also cover wg and lqkv; wv covers lz; wo covers lout. */
#define QMV_CLASS_TOK_EMB 1
#define QMV_CLASS_WCLS 2
#define QMV_CLASS_WQ_WK 4
#define QMV_CLASS_WV 8
#define QMV_CLASS_WO 16
#define QMV_CLASS_W1_W3 32
#define QMV_CLASS_W2 64

/* Bytes of a matrix image: q, its padding to 64, then d (no trailing pad).
 * Every size is computed with overflow checks, as the page requires.  Returns 0 for an
 * invalid wtype, scale_dtype or shape.  Host only. */
size_t qmv_weight_bytes(int wtype, int scale_dtype, int64_t rows, int64_t cols);

/* Offset of the d array from W (q's size rounded up to 64).  -1 if invalid.  Host only. */
int64_t qmv_scale_offset(int wtype, int scale_dtype, int64_t rows, int64_t cols);

/* Storage type of one matrix of a mixed model (Krafla page, header offset 72): a Q4_0
 * file stores the classes whose bit is set in q8_mask as Q8_0; with a shared classifier
 * (header offset 48 non-zero) tok_emb is Q8_0 when bit 1 or bit 2 is set.  A Q8_0 file
 * stores everything as Q8_0.  class_bit is one QMV_CLASS_* value.  Returns QMV_Q8_0 or
 * QMV_Q4_0, or -1 for an unknown file_wtype or class bit.  Host only. */
int qmv_matrix_wtype(int file_wtype, uint32_t q8_mask, int class_bit, int shared_classifier);

/* y = W x for a batch of activation vectors (Krafla page, "Body": row r of a matrix gives
 * output r, y[r] = sum_c W[r][c] x[c]).
 *   W     : device, the matrix image described above (q array first).
 *   x     : device, batch x cols, x_dtype (QMV_X_F32 or QMV_X_BF16), row-major.
 *   y     : device, batch x rows float32, row-major; fully overwritten.
 *   batch : number of activation vectors, >= 0; 0 launches nothing and returns QMV_OK.
 * Each block contributes d * sum_j level_j * x_j; sums are kept in float32.  Batches
 * below 16 (and 16 in groups of 8 MB of weights or more, and float32 activations) run
 * through the decode kernels (weights decoded to exact levels, one tensor-core dot product
 * per block, f32 scale and accumulate) in passes of up to 8 vectors, or of up to 16 for bf16
 * batches of 9..16 in groups of 8 MB of weights or more: those 16-vector passes and bf16
 * passes of 8 vectors over 128 MB of weights take the tensor-memory kernel (levels stored to
 * tensor memory, tcgen05 MMA); the other passes of 2..8 bf16 vectors the mma.sync kernel,
 * which measured faster there; a pass of one bf16 vector takes the block-diagonal kernel (one MMA
 * column per weight block; IEEE-half operands for the 256-column stages whose activations
 * are exact halves, bfloat16 otherwise).  float32 activations, 2..8 vectors, are split into
 * bfloat16 pairs hi + lo (hi = RN_bf16(x), lo = RN_bf16(x - hi): 16 bits of x kept): on
 * launches of 96 MB of weights or more (and for gated activations) in a 2 MiB buffer of the
 * calling stream (allocated on its first such call; without it, and while the stream is
 * captured before it exists, the mma.sync kernel takes them) for the tensor-memory kernel (hi
 * and lo as its 16 MMA columns), on smaller launches in the mma.sync kernel's own stages.  One float32 vector takes the
 * block-diagonal kernel (launches under 256K weights the mma.sync kernel, which splits x as
 * above in one launch): under 16 MB of weights it reads x as float32, larger launches after
 * the split into the buffer.  There each warp's stage of 256 or 512 columns is scaled by the
 * power of two that brings its largest magnitude into [2^14, 2^15) and rounded once to IEEE
 * half (at most 2^-11 relative error per term, one MMA per block, the sums scaled back
 * exactly); a stage holding a nonzero value that would round to a subnormal half (nonzero
 * magnitudes more than 2^28 apart) or a non-finite one runs each block's MMAs with hi and
 * with lo instead.  The same holds for QMV_X_BF16_PAIR and for gated activations at batch 1.
 * The rest take the mma.sync kernel.  The tensor-memory kernel splits tiles between CTAs;
 * their parts meet in a workspace of the calling stream (8 MiB of device memory, allocated
 * on the stream's first such call and kept; while a stream without one is being captured,
 * the call takes the mma.sync kernel instead).  Results do not depend on timing.
 * bfloat16 batches of 17 and more (and of 16 in groups under 8 MB of weights; cols % 256 ==
 * 0) run in passes of up to 128 through the prefill kernel: each weight w is dequantized as
 * qmv_dequant does and enters the tensor core
 * as two bfloat16 parts hi = RN_bf16(w) and lo = RN_bf16(w - hi) (for Q4_0 with f16 scales
 * hi + lo = w exactly; otherwise within 2^-17 |w|, and within 2^-134 absolute for the
 * weights below 2^-117 that only float32 scales under 2^-120 produce), stored to tensor
 * memory; two tcgen05 MMAs per 16 columns (hi, then lo) accumulate in f32 in tensor memory.  A matrix with fewer
 * 128-row tiles than the GPU has SMs has its columns split between CTAs, whose parts meet in
 * a second workspace of the calling stream (32 MiB, allocated like the first; without it the
 * call does not split).
 * Products agree with an
 * exact evaluation to within 1e-3 * sum_c |W[r][c] x[c]| per output (on the prefill route with
 * float32 scales, for weights of magnitude 2^-124 or more).  A Q8_0 byte of
 * -128 is not rejected here: it decodes as -128 * d (see qmv_validate).
 * Returns QMV_OK, or QMV_E_FORMAT / QMV_E_SHAPE / QMV_E_ARG / QMV_E_ALIGN before any
 * launch, or QMV_E_CUDA. */
int qmv_matvec(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void *W,
               const void *x, int x_dtype, float *y, int batch, cudaStream_t stream);

/* One problem of a grouped product: y = W x for this matrix with its own activations.
 * Layout and alignment of W, x and y as for qmv_matvec. */
typedef struct qmv_problem {
  int64_t rows;
  int64_t cols;
  const void *W;
  const void *x;
  float *y;
} qmv_problem;

#define QMV_MAX_GROUP 8

/* Flags of qmv_matvec_grouped.
 * QMV_FLAG_OVERLAP: this launch's first weight tiles are fetched while the kernel that
 *   precedes it on the stream finishes (a programmatic dependent launch).  Activations are
 *   read, and y written, only after the preceding kernel has completed; the WEIGHTS however
 *   may be read earlier, so they must not be written by the immediately preceding kernel
 *   (true for model weights after loading).  Without the flag the decode and prefill kernels
 *   still launch as programmatic dependents (their CTAs start and set up during the preceding
 *   kernel's tail) but touch no global memory, and allocate no tensor memory, before that
 *   kernel has completed.
 * QMV_FLAG_BF16_WEIGHTS: for the problems that take the prefill kernel (16 or more bf16
 *   vectors), round each dequantized weight once to bfloat16 instead of passing it as hi + lo
 *   parts: one MMA per 16 columns instead of two.  Each term then carries a relative error of
 *   up to 2^-9, so an output dominated by a few terms (short rows, concentrated activations)
 *   can miss the 1e-3 * sum |W x| tolerance stated for qmv_matvec; with many comparable terms
 *   the rounding errors largely cancel.  No effect on the other kernels, which use exact
 *   levels. */
#define QMV_FLAG_OVERLAP 1u
#define QMV_FLAG_BF16_WEIGHTS 2u

/* Several products in one launch (Krafla page, "Body": the projections of a layer, e.g.
 * wq, wk, wv reading the same normalized input, or w1 and w3).  All n problems share
 * wtype, scale_dtype, x_dtype and batch; each has its own rows, cols, W, x and y.  Same
 * results as n calls of qmv_matvec (without QMV_FLAG_BF16_WEIGHTS).  problems is a host array
 * of n entries, read during the call only; 1 <= n <= QMV_MAX_GROUP, else QMV_E_ARG; flags
 * other than the QMV_FLAG_* above give QMV_E_ARG.  Returns as qmv_matvec (the first failing
 * problem decides the code; nothing is launched then). */
int qmv_matvec_grouped(int wtype, int scale_dtype, int x_dtype, int batch, const qmv_problem *problems, int n,
                       unsigned flags, cudaStream_t stream);

/* Limits of qmv_matvec_grouped_noalloc. */
#define QMV_NOALLOC_MAX_BATCH 8   /* activation vectors per call */
#define QMV_NOALLOC_MAX_CTAS 320  /* CTAs its scratch array holds partial sums for */
#define QMV_NOALLOC_SCRATCH_BYTES 2622976 /* size of that array (2.5 MiB + 1536 bytes) */

/* Allocation-free variant of qmv_matvec_grouped (the Krafla page has no counterpart: this
 * is a property of this library's runtime, not of the format).  For callers that cannot
 * let a library allocate device memory after start-up: an inference server that hands all
 * free device memory to its own pool at start-up (a later cudaMalloc would fail, or eat
 * into that pool), or a latency-critical path that cannot take cudaMalloc's implicit
 * device synchronization.
 *
 * It runs the tensor-memory decode kernel (bf16 activations, weights unpacked into tensor
 * memory, tcgen05 MMA), whose tiles may be split between CTAs; the split tiles' partial
 * sums and arrival counters live in one fixed array inside the library
 * (QMV_NOALLOC_SCRATCH_BYTES of device memory per device) instead of the per-stream workspace
 * that qmv_matvec_grouped allocates on a stream's first such call.  Nothing is allocated,
 * freed or resized by this call.
 *
 * Set-up on first use.  CUDA loads the library's device code lazily: the array, and the
 * kernel it serves, come into existence on a device at the first call that needs them there,
 * and the first call on each device also looks up the array's address (cudaGetSymbolAddress,
 * with that device current) and sets the kernel's shared-memory limit.  That first call
 * therefore takes device memory (the array and the kernel's code); make one call per device
 * (any valid arguments) before handing the remaining device memory to a pool, and before
 * capturing a stream if the calls are to be captured.  Later calls take no memory.
 *
 * Same arguments and results as qmv_matvec_grouped, restricted to what that kernel takes.
 * The checks, all made before any launch, in this order:
 *   problems non-null and 1 <= n <= QMV_MAX_GROUP, else QMV_E_ARG;
 *   x_dtype must be QMV_X_BF16, else QMV_E_FORMAT;
 *   0 <= batch <= QMV_NOALLOC_MAX_BATCH, else QMV_E_ARG (larger batches: call once per
 *     group of at most 8 vectors);
 *   flags only QMV_FLAG_OVERLAP, else QMV_E_ARG;
 *   per problem as qmv_matvec_grouped, and cols % 256 == 0 and rows < 2^31 - 256, else
 *     QMV_E_SHAPE.
 * The kernel uses at most QMV_NOALLOC_MAX_CTAS CTAs (fewer on a device with fewer SMs).
 *
 * The arrival counters in the array must be zero when the kernel starts.  A call that
 * completes leaves them at zero; a kernel that gave up on a bounded wait (QMV_E_TIMEOUT from
 * qmv_check_device) may leave them part-way, and qmv_check_device() then clears them.  The
 * array is shared by all calls on a device, so calls that may overlap in time (on different
 * streams, or from different host threads without ordering) race on it and give wrong
 * results: order them on one stream. */
int qmv_matvec_grouped_noalloc(int wtype, int scale_dtype, int x_dtype, int batch, const qmv_problem *problems,
                               int n, unsigned flags, cudaStream_t stream);

/* The FFN's gate and up projections with the gated activation as their epilogue (Krafla page,
 * "Body": w1 gate, w3 up, both hidden_dim x dim; header field act): for one bfloat16 activation
 * vector x (device, cols bfloat16, 16-byte aligned),
 *   gate = W1 x,  up = W3 x  (each as qmv_matvec computes it, float32 sums),
 *   h[r] = act(gate[r]) * up[r]  (float32 operations, CUDA's expf / tanhf),
 * written to h (device, 2 * rows bfloat16, 16-byte aligned) as the pair hi[r] = RN_bf16(h[r]) at
 * h[r] and lo[r] = RN_bf16(h[r] - hi[r]) at h[rows + r] (a finite h beyond the bfloat16 range
 * keeps a truncated hi; lo = 0 for h that is not finite): the layout of QMV_X_BF16_PAIR, so the
 * down projection takes it directly (qmv_matvec_grouped with x_dtype QMV_X_BF16_PAIR, batch 1).
 * One launch: each warp tile holds 16 rows of W1 and the same 16 rows of W3, so gate and up
 * meet in registers and neither is written to memory.  The result has the bits that the
 * grouped product of {W1, W3} followed by the float32 gated route (QMV_X_SILU_GLU_F32 /
 * QMV_X_GELU_GLU_F32) forms from the same sums.
 *   wtype must be QMV_Q4_0 (QMV_E_FORMAT otherwise; other types: qmv_matvec_grouped on {W1, W3},
 *   then the gated float32 route); x_dtype must be QMV_X_BF16 (QMV_E_FORMAT); act QMV_ACT_SILU
 *   or QMV_ACT_GELU_TANH (QMV_E_FORMAT); cols % 256 == 0 (QMV_E_SHAPE); flags QMV_FLAG_OVERLAP
 *   or 0 (QMV_E_ARG).
 * W1 and W3 are matrix images as for qmv_matvec (same wtype, scale_dtype, rows and cols).
 * Allocates nothing.  Asynchronous.  Returns as qmv_matvec. */
int qmv_matvec_glu(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void *W1, const void *W3,
                   const void *x, int x_dtype, int act, void *h, unsigned flags, cudaStream_t stream);

/* out[r][c] = level * d as float32, with one float32 multiplication rounded to nearest
 * even (Krafla page, "Q8_0" and "Q4_0"; an f16 scale is first widened to float32, which is
 * exact, as the runtime does when it loads a file).  No flush of subnormals;
 * NaN and infinite scales propagate by IEEE rules.
 *   out : device, rows x cols float32, row-major, 16-byte aligned; fully overwritten.
 * Returns as qmv_matvec. */
int qmv_dequant(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void *W,
                float *out, cudaStream_t stream);

/* The loader's quant check (Krafla page, "Q8_0": a file whose Q8_0 quants contain the byte
 * -128 fails to load, with ML_E_FORMAT).  Scans the q array on the device and writes to
 * *first_bad (device, 8-byte aligned) the smallest byte index into q that holds -128,
 * or -1 when there is none.  Q4_0 has no invalid nibble (the page accepts every scale and
 * every nibble), so for Q4_0 it writes -1.  Asynchronous: the caller reads
 * *first_bad after the stream has reached this point.  Returns as qmv_matvec. */
int qmv_validate(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void *W,
                 int64_t *first_bad, cudaStream_t stream);

/* The writer rules on the device (Krafla page, "Quantization rule"): float32 rows x cols
 * (src, device, row-major, 16-byte aligned) into the two-array layout at W (device, 16-byte
 * aligned, qmv_weight_bytes() bytes; the padding between the arrays is written as zeros).
 *   Q8_0, per block of 32: amax = max |x|; amax < 1e-30 gives d = 0 and zero quants;
 *     f32 scale: d = amax / 127, q = trunc(x * (127 / amax) + copysign(0.5, x));
 *     f16 scale: d = the f16 nearest amax / 127, q = trunc(x * (1 / d) + copysign(0.5, x))
 *     (a d that rounds to f16 zero gives the zero block); q clamped to +-127.
 *   Q4_0 ("round" rule): d = (element of largest magnitude, the first of equals) / -8,
 *     first rounded to f16 (to nearest) with f16 scales; nibble = trunc(x * (1 / d) + 8.5)
 *     kept in 0..15, with 1 / d = 0 for d = 0.
 * Each operation is one float32 operation rounded to nearest even, so the bytes equal those
 * of the rules evaluated in that order.  src is meant to be finite (what a NaN or an
 * infinity gives is not specified).  A block whose f16 scale would lie beyond the f16 range
 * is refused: it is written as d = 0 (Q8_0: zero quants, Q4_0: nibbles 8), and *first_bad
 * (device, 8-byte aligned) receives the smallest such block index (row * cols / 32 +
 * column block), or -1 when there is none.  Asynchronous.  Returns as qmv_dequant, and
 * QMV_E_ARG for a null first_bad. */
int qmv_quantize(int wtype, int scale_dtype, int64_t rows, int64_t cols, const float *src, void *W,
                 int64_t *first_bad, cudaStream_t stream);

/* Size in bytes of a rows x cols tensor stored as GGUF interleaved blocks (minfer "02 - GGUF
 * load" page, §2.3-2.4): rows * cols/32 records of 18 bytes (Q4_0: f16 d, then 16 bytes of
 * nibbles) or 34 bytes (Q8_0: f16 d, then 32 int8 quants), a row being cols/32 consecutive
 * records.  0 for invalid arguments. */
size_t qmv_gguf_bytes(int wtype, int64_t rows, int64_t cols);

/* A tensor in GGUF interleaved blocks (src, device, 16-byte aligned, qmv_gguf_bytes() bytes)
 * into the two-array layout with f16 scales at W (device, 16-byte aligned,
 * qmv_weight_bytes(wtype, QMV_SCALE_F16, rows, cols) bytes; the padding between the arrays is
 * written as zeros), the layout every product entry point reads.  Bytes are moved, not decoded:
 * record k of row r gives q block r*cols/32 + k (its quants, unchanged; for Q4_0 the nibble
 * order is the Krafla page's: byte j holds element j low, element j + 16 high) and that
 * block's scale (its f16 code, unchanged).  src and W must not overlap.  Asynchronous.
 * Returns QMV_OK, QMV_E_FORMAT (wtype), QMV_E_SHAPE, QMV_E_ARG (null pointer), QMV_E_ALIGN, or
 * QMV_E_CUDA. */
int qmv_gguf_to_mlb(int wtype, int64_t rows, int64_t cols, const void *src, void *W, cudaStream_t stream);

/* The runtime's activation quantizer (Krafla page, "Quantization rule": the writer's Q8_0
 * operations, applied by the runtime to its activations; f32 scale): x (device, batch x cols,
 * x_dtype QMV_X_F32 or QMV_X_BF16, row-major, 16-byte aligned; bfloat16 is widened to float32
 * exactly) into xq (device, 16-byte aligned, qmv_weight_bytes(QMV_Q8_0, QMV_SCALE_F32, batch,
 * cols) bytes): the two-array Q8_0 / f32-scale image of the batch x cols matrix, the padding
 * between its arrays written as zeros.  For float32 x the bytes equal those of
 * qmv_quantize(QMV_Q8_0, QMV_SCALE_F32, batch, cols, x, ...).  batch 0 writes nothing.
 * Asynchronous.  Returns QMV_OK, QMV_E_FORMAT (x_dtype), QMV_E_SHAPE (cols not a positive
 * multiple of 32, or a size that overflows), QMV_E_ARG (batch < 0, null pointer),
 * QMV_E_ALIGN, or QMV_E_CUDA. */
int qmv_quantize_x(int x_dtype, int64_t batch, int64_t cols, const void *x, void *xq, cudaStream_t stream);

/* The activation-quantized product (the runtime's CPU path, which multiplies in quantized
 * space; minfer "02 - GGUF load" page): W as for qmv_matvec; xq the Q8_0 / f32-scale image of
 * batch x cols activations as qmv_quantize_x writes it (device, 16-byte aligned).  For each
 * vector v, row r and block b:
 *   isum = sum_j level_w[r][32b + j] * q_x[v][32b + j]   (exact integer),
 *   y[v][r] = sum_b (d_w[r][b] * d_x[v][b]) * isum        (float32 products and sums),
 * y device, batch x rows float32, row-major, 4-byte aligned, fully overwritten.  Results agree
 * with an exact evaluation to within 1e-3 * sum_b |d_w d_x| sum_j |level_w q_x| per output and
 * do not depend on timing.  Runs in passes of up to 8 vectors: with 2 or more vectors and cols a
 * multiple of 256 on the tensor core (mma.sync m16n8k16 with the quants and the levels as IEEE
 * halves, exact, so each block dot is the exact integer sum), else with dp4a integer dot
 * products (one warp per 1, 2 or 4 rows).  batch 0 launches nothing.  Asynchronous.  Returns as
 * qmv_matvec. */
int qmv_matvec_qx(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void *W, const void *xq,
                  float *y, int batch, cudaStream_t stream);

/* The activation-quantized product with the activation quantizer inside it, for several
 * products in one launch: for each problem, y = qmv_matvec_qx(W, qmv_quantize_x(x)) -- the same
 * activation quants and scales (the runtime's Q8_0 / f32-scale rule), the same integer block dots
 * and float32 steps -- without the separate quantizer launch or the intermediate image.  One
 * vector (batch 1) in groups under 96 MB of weights with every problem's cols a multiple of 256
 * runs the block-diagonal kernel: each warp quantizes the 256-column chunks it streams (four
 * lanes to a block of 32), and the quants and the levels enter the tensor core as IEEE halves,
 * whose block dot products are the exact integer sums.  Two or more vectors with every
 * problem's cols a multiple of 256 take two launches: a quantizer writes the image of each
 * distinct activation array (qmv_quantize_x's bytes) into the calling stream's split buffer
 * (2 MiB of device memory, allocated on the stream's first such call and kept), and the
 * tensor-core mode of qmv_matvec_qx, launched as its programmatic dependent (its weight loads
 * overlap the quantizer), reads them there.  Every other batch and group (one vector on
 * larger groups, where it measured faster; images beyond the buffer; a stream captured before
 * it has its buffer) runs the dp4a kernel, whose CTAs each quantize their problem's
 * activations into shared memory (a few KB per vector) and read them from there.  All n
 * problems share wtype, scale_dtype, x_dtype and batch; each has its own rows, cols, W, x and y
 * (problems of one layer that read the same activations: pass the same x).
 *   x_dtype : QMV_X_F32 or QMV_X_BF16 (QMV_E_FORMAT otherwise); x : device, batch x cols,
 *             row-major, 16-byte aligned.  y : device, batch x rows float32, 4-byte aligned.
 *   min(batch, 8) * (the largest cols of the group) <= QMV_QX_MAX_VEC_COLS, else QMV_E_SHAPE
 *   (the shared memory of one pass); 1 <= n <= QMV_MAX_GROUP, flags 0 or QMV_FLAG_OVERLAP,
 *   else QMV_E_ARG.
 * Results agree with those of qmv_quantize_x followed by qmv_matvec_qx within the tolerance stated
 * there (the column slices may be added in a different grouping) and do not depend on timing.
 * Allocates nothing but the split buffer.  Asynchronous.  Returns as qmv_matvec_grouped. */
#define QMV_QX_MAX_VEC_COLS 200704
int qmv_matvec_qx_grouped(int wtype, int scale_dtype, int x_dtype, int batch, const qmv_problem *problems, int n,
                          unsigned flags, cudaStream_t stream);

/* The Q4_0 best-fit writer (Krafla page, "Quantization rule": the search tools/mlb.py runs
 * per block), arguments, layout and refusal as qmv_quantize with wtype QMV_Q4_0.  Per block:
 * m = the element of largest magnitude (the first of equals); for the candidate levels
 * L = -(60 + 2k)/10, k = 0..12 (-6 .. -8.4): s = m / L, l_j = clamp(rint(x_j / s), -8, 7)
 * (ties to even), d = sum(x^3 l) / sum(x^2 l^2) (0 when the denominator is 0), and the
 * lowest sum(x^2 (x - d l)^2) picks the candidate (the first on ties); a block with
 * max |x| under 1e-6 is divided by that maximum before the fit and d multiplied by it after;
 * the zero block is d = 0 with every level 0; with f16 scales only the winning d goes to f16
 * (to nearest).
 * Every step is one float32 operation rounded to nearest, sums in element order.  About 13x
 * the round rule's arithmetic per block.  Returns as qmv_quantize. */
int qmv_quantize_q4_fit(int scale_dtype, int64_t rows, int64_t cols, const float *src, void *W,
                        int64_t *first_bad, cudaStream_t stream);

/* A compiled step: copies and grouped products recorded once as a CUDA graph and replayed by
 * one call (a decode step's host input, its products and its host output, launched together).
 *   qmv_copy  : bytes from src to dst, any mix of device and pinned host pointers (the
 *               direction follows from the addresses); pageable host memory is not allowed.
 *               A copy between device memory and pinned host memory mapped into the device's
 *               address space is recorded as a small copy kernel reading or writing the host
 *               memory directly (cheaper than a copy node for the few KB of a decode step);
 *               other copies as cudaMemcpyAsync.
 *   qmv_group : the arguments of one qmv_matvec_grouped call.
 * qmv_step_create runs the step once, eagerly, on a private stream (the `before` copies in
 * order, the groups in order, the `after` copies in order): that run sets up the kernels and
 * the private stream's workspaces and checks every argument; it then records the same
 * sequence as a graph.  The products take the kernels an eager call on that stream takes, so a
 * run's results are bit-identical to the eager calls'.  Pointers are fixed at creation: a run
 * reads and writes the same buffers (new inputs are new contents of the same buffers).
 * Returns the status of the first call that failed (as qmv_matvec_grouped, QMV_E_CUDA for a
 * copy), QMV_E_ARG for null arrays with a positive count or a null `step`; nothing is
 * recorded then and *step is NULL. */
typedef struct qmv_copy {
  void *dst;
  const void *src;
  size_t bytes;
} qmv_copy;

typedef struct qmv_group {
  int wtype;
  int scale_dtype;
  int x_dtype;
  int batch;
  const qmv_problem *problems;
  int n;
  unsigned flags;
} qmv_group;

typedef struct qmv_step qmv_step;

int qmv_step_create(const qmv_copy *before, int n_before, const qmv_group *groups, int n_groups,
                    const qmv_copy *after, int n_after, qmv_step **step);

/* Enqueues one run of the step on `stream` (the graph's launch; asynchronous).  Runs of one
 * step must not overlap each other (they share its workspaces): issue them on one stream, or
 * order them.  Returns QMV_OK, QMV_E_ARG (null step) or QMV_E_CUDA. */
int qmv_step_run(qmv_step *step, cudaStream_t stream);

/* One run of the step on `stream` followed by a wait for the stream (what a decode loop does
 * before it reads its host results): one call instead of qmv_step_run and a separate
 * synchronization.  Returns QMV_OK, QMV_E_ARG (null step) or QMV_E_CUDA (a failed launch, or an
 * error the stream reported). */
int qmv_step_run_wait(qmv_step *step, cudaStream_t stream);

/* A gated step: the same step (created, checked and recorded the same way), whose runs each
 * start with a gate kernel that waits on the device until the host opens the run, and end with
 * a kernel that reports the run done to the host through pinned host memory.  A decode loop
 * then enqueues the next run (qmv_step_run) while the current one computes, and after its
 * host-side work (the next token) only opens it: the graph's launch leaves the critical path,
 * and the first products load their first weights while the run waits for the host (they
 * launch as programmatic dependents of the gate).  Every `before` copy must go from pinned host
 * memory the device addresses directly to device memory (the gate kernel copies them once the
 * run is opened), at most 8, else QMV_E_ARG; the step's results can be stored straight into
 * such host memory by the products (see the conventions above) or copied by `after` copies.
 *   qmv_step_run  : enqueues a run; it holds its stream at the gate until opened.  A run that
 *                   is never opened proceeds after one second with stale inputs and records
 *                   QMV_E_TIMEOUT in the status word (qmv_check_device).
 *   qmv_step_open : opens the oldest enqueued run that is not yet open (host memory write,
 *                   release order after the caller's writes of the inputs); QMV_E_ARG for a
 *                   step that is not gated or has no enqueued run left to open.
 *   qmv_step_wait : waits on the host (spinning) until every opened run has finished, at most
 *                   timeout_us microseconds (10 s when <= 0): QMV_OK, QMV_E_TIMEOUT, or QMV_E_ARG
 *                   for a step that is not gated.  After QMV_OK the run's host results are
 *                   visible to the calling thread.
 *   qmv_step_run_wait on a gated step enqueues, opens and waits.
 * Runs of one gated step follow each other on one stream.  qmv_step_destroy opens the runs
 * still closed before it waits for the device.  The gate's counters are 64 bytes of pinned
 * host memory and 8 bytes of device memory, allocated at creation. */
int qmv_step_create_gated(const qmv_copy *before, int n_before, const qmv_group *groups, int n_groups,
                          const qmv_copy *after, int n_after, qmv_step **step);
int qmv_step_open(qmv_step *step);
int qmv_step_wait(qmv_step *step, long long timeout_us);
/* A decode loop's step in one call: qmv_step_open(step), then qmv_step_run(next, stream) when
 * next is not NULL (the following token's run, which waits at its gate), then
 * qmv_step_wait(step, timeout_us).  Both steps gated, else QMV_E_ARG; otherwise the first
 * failing call's status. */
int qmv_step_open_wait(qmv_step *step, qmv_step *next, cudaStream_t stream, long long timeout_us);

/* Waits for the device, then frees the step and its workspaces.  NULL is a no-op.  Returns
 * QMV_OK or QMV_E_CUDA. */
int qmv_step_destroy(qmv_step *step);

/* Synchronizes the current device, then returns and clears the status word that the
 * kernels set when a bounded wait runs out (QMV_E_TIMEOUT); QMV_OK when none was set,
 * QMV_E_CUDA when the device reports a CUDA error.  When the word was set it also zeroes the
 * split-tile arrival counters of every workspace on the device (the per-stream ones and the
 * array of qmv_matvec_grouped_noalloc), which a kernel that gave up may have left part-way.
 * This is the library's sticky device-error query: the errors a running kernel can meet are
 * recorded here rather than in a per-thread "last error". */
int qmv_check_device(void);

/* Short English text for a status code; never NULL. */
const char *qmv_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
