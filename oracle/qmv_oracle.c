/*
 * qmv_oracle.c -- plain CPU oracle for block-quantized (Q8_0 / Q4_0) weight matrices.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this file's library.  It shares no code, header,
 * table or constant with the CUDA library, and the CUDA library never calls it.
 *
 * Source of every definition below: the Krafla ".mlb model format v1" page, sections
 * "Body", "Q8_0", "Q4_0", "Quantization rule" and "Validation done by the loader".  Size arithmetic is also
 * checked against the worked byte counts of the minfer "02 - GGUF load" page, §2.3-2.4.
 *
 * Everything is written the slow, obvious way: one weight at a time, values taken
 * straight from their definitions, products in double precision.  Compile with
 * -O2 -ffp-contract=off -fno-fast-math so that every float operation is one IEEE
 * operation with round-to-nearest-even, as the pages require ("exact float32
 * operations").
 *
 * Parity status of each function (what pins it is in tests/test_oracle_pins.py):
 *   oracle_weight_bytes / oracle_scale_offset : pinned (worked byte counts, closed forms)
 *   oracle_f16_value / oracle_f16_bits_rne    : pinned (all 65536 codes; IEEE rounding cases)
 *   oracle_level / oracle_scale / oracle_dequant : pinned (hand-built blocks)
 *   oracle_matvec / oracle_matvec_rows        : pinned (brute force, one-hot, closed forms)
 *   oracle_validate                           : pinned (hand-built -128 byte)
 *   oracle_quant_q8_block                     : pinned (invariants of the rule)
 *   oracle_quant_q4_round_block               : pinned (invariants of the rule)
 *   oracle_quantize_x                         : pinned (exactly representable activations
 *                                               give back their integers and power-of-two scale)
 *   oracle_matvec_qx                          : pinned (equals the plain product on exactly
 *                                               representable activations; equals the product
 *                                               with the dequantized activations; a hand block)
 *   oracle_gguf_bytes                         : pinned (the minfer page's GGUF tensor sizes)
 *   oracle_gguf_to_mlb                        : pinned (hand blocks written as GGUF records)
 *   oracle_quant_q4_fit_block / _quantize_q4_fit : pinned by invariants only (exactly
 *                                               representable blocks come back exactly; the
 *                                               weighted error never exceeds the round rule's;
 *                                               scaling a block scales d); the float order is a
 *                                               reading: parity of the printed rule unpinned
 *   oracle_matvec_glu                         : pinned (act(g) - act(-g) = g turns a pair of
 *                                               gated products into the plain product; SiLU at
 *                                               ln 3 and GELU where its tanh is 1/2 give 3g/4)
 *   oracle_glu                                : pinned (the same identities value by value, and
 *                                               act(0) = 0, large |g|: act(g) -> max(g, 0))
 *   corner readings of the writers (f16 scale that rounds to 0, all-zero Q4 block,
 *   ties of the largest magnitude) : parity unpinned (writer-only, not on the product path)
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* Status values.  They mirror the loader's ML_E_* classes ("Validation done by the
 * loader"): a bad value in the data is a format error, a bad dimension a shape error. */
#define ORACLE_OK 0
#define ORACLE_E_FORMAT 2
#define ORACLE_E_SHAPE 3

/* wtype values of the .mlb header (offset 44): 1 = Q8_0, 2 = Q4_0. */
#define ORACLE_Q8_0 1
#define ORACLE_Q4_0 2

/* ---------------------------------------------------------------------------
 * Size arithmetic ("Body": a quantized matrix is its q array followed by its d array, each
 * array's length rounded up to a 64-byte boundary with zeros; a file may leave out the tail
 * of the last array, which is never read).
 * ------------------------------------------------------------------------- */

static int64_t round_up_64(int64_t n) { return ((n + 63) / 64) * 64; }

/* Checks the dimensions and fills the byte counts of the two arrays.  Returns a status.
 * q bytes: Q8_0 rows*cols, Q4_0 rows*cols/2.  d bytes: rows*cols/32 scales of 4 (f32)
 * or 2 (f16, scale_f16 = 1) bytes.  cols must be a multiple of 32 (one block is 32
 * consecutive weights of a row); zero dimensions are shape errors, as in the loader. */
static int layout(int wtype, int scale_f16, int64_t rows, int64_t cols,
                  int64_t *q_bytes, int64_t *d_off, int64_t *d_bytes)
{
    if (wtype != ORACLE_Q8_0 && wtype != ORACLE_Q4_0) return ORACLE_E_FORMAT;
    if (scale_f16 != 0 && scale_f16 != 1) return ORACLE_E_FORMAT;
    if (rows <= 0 || cols <= 0 || cols % 32 != 0) return ORACLE_E_SHAPE;
    /* overflow-checked: the product rows*cols must fit comfortably in 63 bits */
    if (rows > INT64_MAX / cols) return ORACLE_E_SHAPE;
    int64_t n = rows * cols;
    if (n > INT64_MAX / 4) return ORACLE_E_SHAPE;
    int64_t q = (wtype == ORACLE_Q8_0) ? n : n / 2;
    int64_t nscales = n / 32;
    int64_t dsz = nscales * (scale_f16 ? 2 : 4);
    int64_t off = round_up_64(q);
    if (off > INT64_MAX - dsz) return ORACLE_E_SHAPE;
    *q_bytes = q;
    *d_off = off;
    *d_bytes = dsz;
    return ORACLE_OK;
}

/* Smallest buffer that holds the matrix: q, its padding, then d (no trailing pad).
 * Returns -1 for invalid arguments. */
int64_t oracle_weight_bytes(int wtype, int scale_f16, int64_t rows, int64_t cols)
{
    int64_t q, off, dsz;
    if (layout(wtype, scale_f16, rows, cols, &q, &off, &dsz) != ORACLE_OK) return -1;
    return off + dsz;
}

/* Offset of the d array from the start of the matrix.  -1 for invalid arguments. */
int64_t oracle_scale_offset(int wtype, int scale_f16, int64_t rows, int64_t cols)
{
    int64_t q, off, dsz;
    if (layout(wtype, scale_f16, rows, cols, &q, &off, &dsz) != ORACLE_OK) return -1;
    return off;
}

/* ---------------------------------------------------------------------------
 * Number formats
 * ------------------------------------------------------------------------- */

/* Value of an IEEE 754 binary16 code, from the format's definition: sign bit,
 * 5-bit biased exponent (bias 15), 10-bit fraction; exponent 0 is subnormal
 * (fraction * 2^-24), exponent 31 is infinity or NaN.  Every binary16 value is a
 * float32 value, so the result is exact (the page has the runtime widen f16 scales to
 * f32, exactly, on loading). */
float oracle_f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double mag;
    if (e == 0) {
        mag = ldexp((double)m, -24);
    } else if (e == 31) {
        if (m != 0) return NAN;
        mag = INFINITY;
    } else {
        mag = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return (float)(sign ? -mag : mag);
}

/* binary16 code nearest to v, ties to even (IEEE default rounding).  Used by the
 * writer rules with f16 scales, which round d to f16 (to nearest). */
uint16_t oracle_f16_bits_rne(float v)
{
    if (isnan(v)) return 0x7e00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs((double)v);
    /* 65504 is the largest finite half; the midpoint to the next step (65536) is 65520,
     * and a tie there goes to the even neighbour, 65536, i.e. overflow. */
    if (a >= 65520.0) return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: multiples of 2^-24; 1024 * 2^-24 is the smallest normal,
         * whose code 0x0400 equals the integer 1024, so the encoding stays right. */
        double m = nearbyint(a * 16777216.0);
        return sign | (uint16_t)m;
    }
    int e2;
    frexp(a, &e2);          /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;         /* unbiased exponent */
    double quantum = ldexp(1.0, E - 10);
    double m = nearbyint(a / quantum); /* 1024 .. 2048, exact division */
    if (m == 2048.0) {
        m = 1024.0;
        E += 1;
    }
    if (E > 15) return sign | 0x7c00;
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(m - 1024.0));
}

/* Value of a bfloat16 code: the upper half of a float32. */
float oracle_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t load_le32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t bits_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* ---------------------------------------------------------------------------
 * Decoding one weight ("Q8_0", "Q4_0")
 * ------------------------------------------------------------------------- */

/* Integer level of weight (r, c).  Q8_0: the int8 byte (rows*cols bytes, row-major).
 * Q4_0: block k = c/32 of row r is 16 bytes at r*cols/2 + 16k; element j of the block is
 * the low four bits of byte j, element j+16 the high four bits; level = nibble - 8. */
int oracle_level(const uint8_t *W, int wtype, int64_t cols, int64_t r, int64_t c)
{
    if (wtype == ORACLE_Q8_0) {
        return (int)(int8_t)W[r * cols + c];
    }
    int64_t k = c / 32;
    int64_t j = c % 32;
    uint8_t byte = W[r * (cols / 2) + 16 * k + (j % 16)];
    int nibble = (j < 16) ? (byte & 0x0f) : (byte >> 4);
    return nibble - 8;
}

/* Scale d of block k of row r, as float32: stored f32, or f16 converted exactly. */
float oracle_scale(const uint8_t *W, int wtype, int scale_f16, int64_t rows, int64_t cols,
                   int64_t r, int64_t k)
{
    int64_t q, off, dsz;
    if (layout(wtype, scale_f16, rows, cols, &q, &off, &dsz) != ORACLE_OK) return NAN;
    int64_t idx = r * (cols / 32) + k;
    if (scale_f16) {
        const uint8_t *p = W + off + 2 * idx;
        return oracle_f16_value((uint16_t)(p[0] | (p[1] << 8)));
    }
    return f32_from_bits(load_le32(W + off + 4 * idx));
}

/* Dequantized matrix, float32, rows x cols row-major: w = level * d with one float32
 * multiplication (round to nearest even).  With f16 scales the product is exact. */
int oracle_dequant(int wtype, int scale_f16, int64_t rows, int64_t cols, const uint8_t *W,
                   float *out)
{
    int64_t q, off, dsz;
    int st = layout(wtype, scale_f16, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t c = 0; c < cols; c++) {
            float level = (float)oracle_level(W, wtype, cols, r, c);
            float d = oracle_scale(W, wtype, scale_f16, rows, cols, r, c / 32);
            out[r * cols + c] = level * d;
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * The product y[r] = sum_c W[r][c] * x[c]  ("Body": row r of a matrix gives output r), for
 * a batch of activation vectors.  x is batch x cols row-major, f32
 * or bf16 (x_bf16 = 1); y and absref are batch x n_rows row-major, double.
 * Each weight is level * d evaluated exactly in double (level has 8 bits, d 24), each
 * activation is converted exactly to double, and the sum runs in double in column order.
 * absref[b][i] = sum_c |w * x|, the scale of the tolerance.
 * ------------------------------------------------------------------------- */

static double x_value(const void *x, int x_bf16, int64_t cols, int64_t b, int64_t c)
{
    if (x_bf16) return (double)oracle_bf16_value(((const uint16_t *)x)[b * cols + c]);
    return (double)((const float *)x)[b * cols + c];
}

int oracle_matvec_rows(int wtype, int scale_f16, int64_t rows, int64_t cols, const uint8_t *W,
                       const void *x, int x_bf16, int batch, const int64_t *row_ids,
                       int64_t n_rows, double *y, double *absref)
{
    int64_t q, off, dsz;
    int st = layout(wtype, scale_f16, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    for (int b = 0; b < batch; b++) {
        for (int64_t i = 0; i < n_rows; i++) {
            int64_t r = row_ids[i];
            if (r < 0 || r >= rows) return ORACLE_E_SHAPE;
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t c = 0; c < cols; c++) {
                double w = (double)oracle_level(W, wtype, cols, r, c) *
                           (double)oracle_scale(W, wtype, scale_f16, rows, cols, r, c / 32);
                double t = w * x_value(x, x_bf16, cols, b, c);
                acc += t;
                acc_abs += fabs(t);
            }
            y[(int64_t)b * n_rows + i] = acc;
            absref[(int64_t)b * n_rows + i] = acc_abs;
        }
    }
    return ORACLE_OK;
}

int oracle_matvec(int wtype, int scale_f16, int64_t rows, int64_t cols, const uint8_t *W,
                  const void *x, int x_bf16, int batch, double *y, double *absref)
{
    int64_t q, off, dsz;
    int st = layout(wtype, scale_f16, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    for (int b = 0; b < batch; b++) {
        for (int64_t r = 0; r < rows; r++) {
            int st2 = oracle_matvec_rows(wtype, scale_f16, rows, cols, W,
                                         (const char *)x + (size_t)b * cols * (x_bf16 ? 2 : 4),
                                         x_bf16, 1, &r, 1, &y[(int64_t)b * rows + r],
                                         &absref[(int64_t)b * rows + r]);
            if (st2 != ORACLE_OK) return st2;
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Validation ("Validation done by the loader": a Q8_0 quant of -128 makes the file a format
 * error: the x86 kernels flip the sign of weights, and -128 has no int8 opposite).  Every
 * Q4_0 nibble and every scale is accepted.
 * ------------------------------------------------------------------------- */
int oracle_validate(int wtype, int scale_f16, int64_t rows, int64_t cols, const uint8_t *W)
{
    int64_t q, off, dsz;
    int st = layout(wtype, scale_f16, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    if (wtype == ORACLE_Q8_0) {
        for (int64_t i = 0; i < q; i++)
            if (W[i] == 0x80) return ORACLE_E_FORMAT;
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Writer rules ("Quantization rule"), used to make test matrices from float data
 * and for round-trip checks.  Not on the product path.
 * ------------------------------------------------------------------------- */

static float clamp127(float t)
{
    if (t > 127.0f) return 127.0f;
    if (t < -127.0f) return -127.0f;
    return t;
}

/* One Q8_0 block of 32 floats.  f32 scale: amax = max |x|; amax < 1e-30 gives d = 0,
 * q = 0; otherwise d = amax / 127 and q = trunc(x * (127 / amax) + copysign(0.5, x)),
 * clamped to +-127.  f16 scale: d = amax / 127 rounded to f16, to nearest (a d above
 * 65504 is refused), then q = trunc(x * (1 / d) + copysign(0.5, x)) with the f16 d.
 * Reading for a d that rounds to f16 zero (1 / d infinite): the block is stored as the
 * zero block (parity unpinned: writer-only corner).  d_bits receives the stored scale
 * bits (f32 bits, or the f16 code in the low half). */
int oracle_quant_q8_block(const float *x, int scale_f16, int8_t *q, uint32_t *d_bits)
{
    float amax = 0.0f;
    for (int j = 0; j < 32; j++) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    if (amax < 1e-30f) {
        for (int j = 0; j < 32; j++) q[j] = 0;
        *d_bits = 0;
        return ORACLE_OK;
    }
    if (!scale_f16) {
        float d = amax / 127.0f;
        float inv = 127.0f / amax;
        for (int j = 0; j < 32; j++) {
            float t = x[j] * inv;
            float u = t + copysignf(0.5f, x[j]);
            q[j] = (int8_t)clamp127(truncf(u));
        }
        *d_bits = bits_from_f32(d);
        return ORACLE_OK;
    }
    uint16_t h = oracle_f16_bits_rne(amax / 127.0f);
    if ((h & 0x7fff) >= 0x7c00) return ORACLE_E_FORMAT; /* above 65504: refused */
    float d = oracle_f16_value(h);
    if (d == 0.0f) {
        for (int j = 0; j < 32; j++) q[j] = 0;
        *d_bits = 0;
        return ORACLE_OK;
    }
    float inv = 1.0f / d;
    for (int j = 0; j < 32; j++) {
        float t = x[j] * inv;
        float u = t + copysignf(0.5f, x[j]);
        q[j] = (int8_t)clamp127(truncf(u));
    }
    *d_bits = h;
    return ORACLE_OK;
}

/* One Q4_0 block with the "--q4-rule round" rule: d = (element of largest magnitude) /
 * -8; level = min(15, trunc(x * (1 / d) + 8.5)) - 8.  Readings (parity unpinned,
 * writer-only): the first index wins a tie of magnitudes; an all-zero block (d = 0)
 * uses 1/d = 0, so every level is trunc(8.5) - 8 = 0; with f16 scales d is first rounded
 * to f16 (to nearest), as the Q8_0 f16 rule and the best-fit writer do, and the
 * nibble is also kept at or above 0 (the rounded d can push x/d a hair past -8).
 * qs receives the 16 packed bytes (element j low nibble, element j+16 high nibble). */
int oracle_quant_q4_round_block(const float *x, int scale_f16, uint8_t *qs, uint32_t *d_bits)
{
    int im = 0;
    float best = fabsf(x[0]);
    for (int j = 1; j < 32; j++) {
        if (fabsf(x[j]) > best) {
            best = fabsf(x[j]);
            im = j;
        }
    }
    float d = x[im] / -8.0f;
    uint32_t bits;
    if (scale_f16) {
        uint16_t h = oracle_f16_bits_rne(d);
        if ((h & 0x7fff) >= 0x7c00) return ORACLE_E_FORMAT;
        d = oracle_f16_value(h);
        bits = h;
    } else {
        bits = bits_from_f32(d);
    }
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    int nib[32];
    for (int j = 0; j < 32; j++) {
        float t = x[j] * id;
        float u = t + 8.5f;
        int n = (int)truncf(u);
        if (n > 15) n = 15;
        if (n < 0) n = 0;
        nib[j] = n;
    }
    for (int j = 0; j < 16; j++) qs[j] = (uint8_t)(nib[j] | (nib[j + 16] << 4));
    *d_bits = bits;
    return ORACLE_OK;
}

/* Whole matrix from float data into the two-array layout: Q8_0 blocks by the Q8_0
 * rule, Q4_0 blocks by the round rule.  W must hold oracle_weight_bytes() bytes; the
 * padding between the arrays is written as zeros. */
int oracle_quantize(int wtype, int scale_f16, int64_t rows, int64_t cols, const float *src,
                    uint8_t *W)
{
    int64_t q, off, dsz;
    int st = layout(wtype, scale_f16, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    memset(W, 0, (size_t)(off + dsz));
    int64_t nblk = cols / 32;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t k = 0; k < nblk; k++) {
            const float *xb = src + r * cols + 32 * k;
            uint32_t bits = 0;
            if (wtype == ORACLE_Q8_0) {
                st = oracle_quant_q8_block(xb, scale_f16, (int8_t *)(W + r * cols + 32 * k), &bits);
            } else {
                st = oracle_quant_q4_round_block(xb, scale_f16, W + r * (cols / 2) + 16 * k, &bits);
            }
            if (st != ORACLE_OK) return st;
            int64_t idx = r * nblk + k;
            if (scale_f16) {
                W[off + 2 * idx] = (uint8_t)(bits & 0xff);
                W[off + 2 * idx + 1] = (uint8_t)((bits >> 8) & 0xff);
            } else {
                for (int i = 0; i < 4; i++) W[off + 4 * idx + i] = (uint8_t)((bits >> (8 * i)) & 0xff);
            }
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * The runtime's activation-quantized product.  Krafla page, "Quantization rule": the
 * runtime's activation quantizer uses the same float32 operations as the Q8_0 writer
 * (f32 scale); the minfer "02 - GGUF load" page (why weights stay raw until run time):
 * activations are held in float32 and turned into Q8_0 blocks by the CPU at each product,
 * whose kernels then work on the two sets of integers.  Reading: the pages do not spell
 * out the float steps of that dot, so
 * it is taken as its definition, block by block: the integer dot product of the weight
 * levels and the activation quants (exact), times d_w * d_x, summed over the blocks.
 * ------------------------------------------------------------------------- */

/* Activations (batch x cols, float32 or bfloat16 codes with x_bf16 = 1; bfloat16 is
 * widened to float32 exactly) into xq, the Q8_0 / f32-scale two-array image of a
 * batch x cols matrix, block by block with the Q8_0 rule.  xq must hold
 * oracle_weight_bytes(Q8_0, 0, batch, cols) bytes; its padding is written as zeros. */
int oracle_quantize_x(int x_bf16, int64_t batch, int64_t cols, const void *x, uint8_t *xq)
{
    int64_t q, off, dsz;
    int st = layout(ORACLE_Q8_0, 0, batch, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    memset(xq, 0, (size_t)(off + dsz));
    int64_t nblk = cols / 32;
    for (int64_t b = 0; b < batch; b++) {
        for (int64_t k = 0; k < nblk; k++) {
            float xb[32];
            for (int j = 0; j < 32; j++) xb[j] = (float)x_value(x, x_bf16, cols, b, 32 * k + j);
            uint32_t bits = 0;
            st = oracle_quant_q8_block(xb, 0, (int8_t *)(xq + b * cols + 32 * k), &bits);
            if (st != ORACLE_OK) return st;
            int64_t idx = b * nblk + k;
            for (int i = 0; i < 4; i++) xq[off + 4 * idx + i] = (uint8_t)((bits >> (8 * i)) & 0xff);
        }
    }
    return ORACLE_OK;
}

/* y[b][r] = sum over blocks k of d_w(r, k) * d_x(b, k) * sum_j level_w(r, 32k + j) * q_x(b, 32k + j)
 * for W (wtype, scale_f16, rows x cols) and xq as oracle_quantize_x writes it (batch x
 * cols).  The inner sum is an exact integer; d_w * d_x is exact in double (24-bit
 * significands); the blocks are summed in double in column order.  absref[b][r] = sum over
 * blocks |d_w d_x| * sum_j |level_w q_x|, the scale of the tolerance. */
int oracle_matvec_qx(int wtype, int scale_f16, int64_t rows, int64_t cols, const uint8_t *W,
                     const uint8_t *xq, int batch, double *y, double *absref)
{
    int64_t q, off, dsz;
    int st = layout(wtype, scale_f16, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    if (batch < 1) return ORACLE_E_SHAPE;
    st = layout(ORACLE_Q8_0, 0, batch, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    int64_t nblk = cols / 32;
    for (int b = 0; b < batch; b++) {
        for (int64_t r = 0; r < rows; r++) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < nblk; k++) {
                int64_t isum = 0, iabs = 0;
                for (int j = 0; j < 32; j++) {
                    int64_t t = (int64_t)oracle_level(W, wtype, cols, r, 32 * k + j) *
                                (int64_t)oracle_level(xq, ORACLE_Q8_0, cols, b, 32 * k + j);
                    isum += t;
                    iabs += t < 0 ? -t : t;
                }
                double s = (double)oracle_scale(W, wtype, scale_f16, rows, cols, r, k) *
                           (double)oracle_scale(xq, ORACLE_Q8_0, 0, batch, cols, b, k);
                acc += s * (double)isum;
                acc_abs += fabs(s) * (double)iabs;
            }
            y[(int64_t)b * rows + r] = acc;
            absref[(int64_t)b * rows + r] = acc_abs;
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * GGUF interleaved blocks (minfer "02 - GGUF load" page, §2.3-2.4): a Q4_0 block is an f16
 * scale d followed by 16 bytes of nibbles (18 bytes), a Q8_0 block d followed by 32 int8
 * quants (34 bytes); a row of cols values is cols/32 consecutive blocks (row stride
 * (cols/32) * block bytes), rows follow one another with no padding.  Reading: the nibble
 * order inside qs is the Krafla page's Q4_0 order (byte j: element j low, element j + 16
 * high); the pages do not restate it for GGUF.
 * ------------------------------------------------------------------------- */

/* Bytes of a rows x cols tensor in GGUF blocks; -1 for invalid arguments. */
int64_t oracle_gguf_bytes(int wtype, int64_t rows, int64_t cols)
{
    int64_t q, off, dsz;
    if (layout(wtype, 1, rows, cols, &q, &off, &dsz) != ORACLE_OK) return -1;
    int64_t block_bytes = (wtype == ORACLE_Q8_0) ? 34 : 18;
    return rows * (cols / 32) * block_bytes;
}

/* The same matrix in the two-array layout with f16 scales (W must hold
 * oracle_weight_bytes(wtype, 1, rows, cols) bytes; its padding is written as zeros): block
 * k of row r is the GGUF record at (r * (cols/32) + k) * block bytes; its first two bytes
 * are d (little-endian f16 code), the rest its quants, copied unchanged. */
int oracle_gguf_to_mlb(int wtype, int64_t rows, int64_t cols, const uint8_t *gguf, uint8_t *W)
{
    int64_t q, off, dsz;
    int st = layout(wtype, 1, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    memset(W, 0, (size_t)(off + dsz));
    int64_t nblk = cols / 32;
    int64_t qb = (wtype == ORACLE_Q8_0) ? 32 : 16;
    int64_t block_bytes = 2 + qb;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t k = 0; k < nblk; k++) {
            const uint8_t *rec = gguf + (r * nblk + k) * block_bytes;
            int64_t idx = r * nblk + k;
            W[off + 2 * idx] = rec[0];
            W[off + 2 * idx + 1] = rec[1];
            for (int64_t j = 0; j < qb; j++) W[idx * qb + j] = rec[2 + j];
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * The FFN's gated activation feeding the down projection (Krafla page, "Body": w1 is the gate
 * and w3 the up projection, hidden_dim x dim, w2 the down projection, dim x hidden_dim; header
 * field act: 0 = SiLU, 1 = GELU in its tanh form).  Reading: the down projection's
 * input is h = act(w1 x) * (w3 x), element by element, and the product is y = w2 h.
 *   SiLU(g) = g / (1 + e^-g);   GELU_tanh(g) = g/2 * (1 + tanh(sqrt(2/pi) * (g + 0.044715 g^3))).
 * gate and up are batch x cols float32 (the products w1 x, w3 x); h is evaluated in double.
 * ------------------------------------------------------------------------- */

static double glu_act(int act, double g)
{
    if (act == 0) return g / (1.0 + exp(-g));
    const double k = sqrt(2.0 / acos(-1.0));
    return 0.5 * g * (1.0 + tanh(k * (g + 0.044715 * g * g * g)));
}

/* h[i] = act(gate[i]) * up[i] for n values given in double (the exact products w1 x and w3 x of
 * a layer, as the oracle's matvec returns them), evaluated in double. */
int oracle_glu(int act, int64_t n, const double *gate, const double *up, double *h)
{
    if (act != 0 && act != 1) return ORACLE_E_FORMAT;
    if (n < 0) return ORACLE_E_SHAPE;
    for (int64_t i = 0; i < n; i++) h[i] = glu_act(act, gate[i]) * up[i];
    return ORACLE_OK;
}

/* y[b][r] = sum_c W[r][c] * act(gate[b][c]) * up[b][c], absref = sum_c |W[r][c] * h[b][c]|. */
int oracle_matvec_glu(int wtype, int scale_f16, int64_t rows, int64_t cols, const uint8_t *W, int act,
                      const float *gate, const float *up, int batch, double *y, double *absref)
{
    int64_t q, off, dsz;
    int st = layout(wtype, scale_f16, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    if (act != 0 && act != 1) return ORACLE_E_FORMAT;
    for (int b = 0; b < batch; b++) {
        for (int64_t r = 0; r < rows; r++) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t c = 0; c < cols; c++) {
                double w = (double)oracle_level(W, wtype, cols, r, c) *
                           (double)oracle_scale(W, wtype, scale_f16, rows, cols, r, c / 32);
                double h = glu_act(act, (double)gate[(int64_t)b * cols + c]) * (double)up[(int64_t)b * cols + c];
                acc += w * h;
                acc_abs += fabs(w * h);
            }
            y[(int64_t)b * rows + r] = acc;
            absref[(int64_t)b * rows + r] = acc_abs;
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * The Q4_0 best-fit writer (Krafla page, "Quantization rule": the search tools/mlb.py runs
 * per block).  What the page fixes: 13 candidates send the element of largest magnitude
 * to the levels -6, -6.2, ..., -8.4 (all levels clamped to [-8, 7]); each candidate's d is
 * the x^2-weighted least-squares scale for its levels; the lowest weighted error picks the
 * candidate; blocks with max |x| under 1e-6 are brought to unit size for the fit and d is
 * scaled back; d can come out negative; f16 scales round the chosen d to f16 (to nearest).  Readings (parity pinned only by the invariants in the
 * tests, not by printed values): every step is one float32 operation rounded to nearest even,
 * in this order --
 *   m = the element of largest magnitude (the first of equals), a = |m|;
 *   a == 0: the zero block (d = 0, every level 0); a < 1e-6: x_j <- x_j / a, and d <- d * a
 *   at the end;
 *   candidate k = 0..12: L = (float)(-(60 + 2k)) / 10;  s = m / L;
 *     l_j = clamp(rint(x_j / s), -8, 7)  (ties to even, as numpy rounds);
 *     t_j = x_j * x_j;  num += (t_j * x_j) * l_j;  den += (t_j * l_j) * l_j  (j = 0..31 in order);
 *     d = den == 0 ? 0 : num / den;
 *     err += t_j * (e_j * e_j), e_j = x_j - d * l_j  (j in order);
 *   the first candidate with the smallest err wins (strict <); nibble = l + 8.
 * ------------------------------------------------------------------------- */

/* One block; d_bits receives the stored scale bits.  ORACLE_E_FORMAT for an f16 d beyond
 * 65504 (refused, as the other f16 rules). */
int oracle_quant_q4_fit_block(const float *xin, int scale_f16, uint8_t *qs, uint32_t *d_bits)
{
    float x[32];
    float m = xin[0], a = fabsf(xin[0]);
    for (int j = 1; j < 32; j++)
        if (fabsf(xin[j]) > a) {
            a = fabsf(xin[j]);
            m = xin[j];
        }
    int best_l[32];
    float best_d = 0.0f;
    if (a == 0.0f) {
        for (int j = 0; j < 32; j++) best_l[j] = 0;
    } else {
        const int small = a < 1e-6f;
        for (int j = 0; j < 32; j++) x[j] = small ? xin[j] / a : xin[j];
        if (small) m = m / a;
        float best_err = 0.0f;
        for (int k = 0; k <= 12; k++) {
            const float L = (float)(-(60 + 2 * k)) / 10.0f;
            const float s = m / L;
            int l[32];
            float num = 0.0f, den = 0.0f;
            for (int j = 0; j < 32; j++) {
                float r = rintf(x[j] / s);
                if (r < -8.0f) r = -8.0f;
                if (r > 7.0f) r = 7.0f;
                l[j] = (int)r;
                const float t = x[j] * x[j];
                num += (t * x[j]) * (float)l[j];
                den += (t * (float)l[j]) * (float)l[j];
            }
            const float d = den == 0.0f ? 0.0f : num / den;
            float err = 0.0f;
            for (int j = 0; j < 32; j++) {
                const float e = x[j] - d * (float)l[j];
                err += (x[j] * x[j]) * (e * e);
            }
            if (k == 0 || err < best_err) {
                best_err = err;
                best_d = d;
                for (int j = 0; j < 32; j++) best_l[j] = l[j];
            }
        }
        if (small) best_d = best_d * a;
    }
    for (int j = 0; j < 16; j++) qs[j] = (uint8_t)((best_l[j] + 8) | ((best_l[j + 16] + 8) << 4));
    if (scale_f16) {
        uint16_t h = oracle_f16_bits_rne(best_d);
        if ((h & 0x7fff) >= 0x7c00) return ORACLE_E_FORMAT;
        *d_bits = h;
    } else {
        *d_bits = bits_from_f32(best_d);
    }
    return ORACLE_OK;
}

/* A whole matrix by the best-fit rule into the two-array layout (as oracle_quantize). */
int oracle_quantize_q4_fit(int scale_f16, int64_t rows, int64_t cols, const float *src, uint8_t *W)
{
    int64_t q, off, dsz;
    int st = layout(ORACLE_Q4_0, scale_f16, rows, cols, &q, &off, &dsz);
    if (st != ORACLE_OK) return st;
    memset(W, 0, (size_t)(off + dsz));
    int64_t nblk = cols / 32;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t k = 0; k < nblk; k++) {
            uint32_t bits = 0;
            st = oracle_quant_q4_fit_block(src + r * cols + 32 * k, scale_f16, W + r * (cols / 2) + 16 * k, &bits);
            if (st != ORACLE_OK) return st;
            int64_t idx = r * nblk + k;
            if (scale_f16) {
                W[off + 2 * idx] = (uint8_t)(bits & 0xff);
                W[off + 2 * idx + 1] = (uint8_t)((bits >> 8) & 0xff);
            } else {
                for (int i = 0; i < 4; i++) W[off + 4 * idx + i] = (uint8_t)((bits >> (8 * i)) & 0xff);
            }
        }
    }
    return ORACLE_OK;
}
