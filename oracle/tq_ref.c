/*
 * tq_ref.c -- plain CPU oracle of the ternary pq2_0 x q8_K matrix product.
 *
 * TEST INFRASTRUCTURE (see tq_ref.h): callable only from the tests, the smoke
 * check and the benchmark's CPU-baseline leg. Every function is the plain
 * definition written out with loops, in the order the pages state it.
 */
#include "tq_ref.h"

#include <math.h>
#include <string.h>

typedef char ref_q8K_size_check[(sizeof(ref_block_q8K) == REF_Q8K_BYTES) ? 1 : -1];

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float ref_fp16_to_f32(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1F;
    const int m = h & 0x3FF;
    float v;
    if (e == 0) {
        v = ldexpf((float)m, -24);                 /* zero or subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexpf((float)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/*
 * q8_K quantization of activations (ciot README: 256 int8 values, a float
 * scale and 16 partial sums per block). Symmetric scale from the block's
 * largest magnitude over 127 ("Quantization and the CPU"); a block whose
 * absolute max is 127 quantizes with scale 1 (the ternary post, *stuff that
 * went wrong*). Rounding is to nearest, ties to even.
 */
void ref_quantize_q8K(const float *x, int64_t ntok, int64_t cols, ref_block_q8K *y)
{
    const int64_t nb = cols / REF_QK;
    for (int64_t t = 0; t < ntok; ++t) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + t * cols + b * REF_QK;
            ref_block_q8K *yb = y + t * nb + b;
            float amax = 0.0f;
            for (int k = 0; k < REF_QK; ++k) {
                const float a = fabsf(xb[k]);
                if (a > amax) amax = a;
            }
            if (amax == 0.0f) {
                yb->d = 0.0f;
                memset(yb->qs, 0, sizeof(yb->qs));
                memset(yb->bsums, 0, sizeof(yb->bsums));
                continue;
            }
            const float iscale = 127.0f / amax;
            yb->d = amax / 127.0f;
            for (int k = 0; k < REF_QK; ++k) {
                const float p = xb[k] * iscale;
                long q = lrintf(p);                 /* default mode: nearest, ties to even */
                if (q > 127) q = 127;
                if (q < -127) q = -127;
                yb->qs[k] = (int8_t)q;
            }
            for (int i = 0; i < REF_QK / 16; ++i) {
                int s = 0;
                for (int j = 0; j < 16; ++j) s += yb->qs[16 * i + j];
                yb->bsums[i] = (int16_t)s;
            }
        }
    }
}

/* Code u of weight k of a pq2_0 block: byte k >> 2, bits 2*(k & 3). */
static int pq2_code(const uint8_t *block, int k)
{
    return (block[2 + (k >> 2)] >> (2 * (k & 3))) & 3;
}

static uint16_t pq2_scale_bits(const uint8_t *block)
{
    return (uint16_t)(block[0] | (block[1] << 8));
}

void ref_decode_pq2_0(const uint8_t *wpq, int64_t rows, int64_t cols,
                      int8_t *w, uint16_t *scale_bits)
{
    const int64_t ng = cols / REF_GROUP;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < ng; ++g) {
            const uint8_t *blk = wpq + (r * ng + g) * REF_PQ2_BYTES;
            scale_bits[r * ng + g] = pq2_scale_bits(blk);
            for (int k = 0; k < REF_GROUP; ++k)
                w[r * cols + g * REF_GROUP + k] = (int8_t)(pq2_code(blk, k) - 1);
        }
    }
}

/*
 * ptq1_0 (declared with its readings in tq_ref.h). A code byte's trit n is
 * the page's formula as written: floor(3 * ((b * 3^n) mod 256) / 256).
 */
int ref_ptq1_trit(uint8_t b, int n)
{
    int p = 1;
    for (int i = 0; i < n; ++i) p *= 3;
    const int v = (b * p) % 256;
    return (3 * v) / 256;
}

uint8_t ref_ptq1_byte(const int *t)
{
    int q = 0;
    for (int n = 0; n < 5; ++n) q = 3 * q + t[n];   /* sum t_n 3^(4 - n) */
    return (uint8_t)((256 * q + 242) / 243);         /* ceil(256 q / 243) */
}

void ref_encode_ptq1_0(const int8_t *w, const uint16_t *scale_bits, int64_t rows,
                       int64_t cols, uint8_t *wpt)
{
    const int64_t ng = cols / REF_GROUP;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < ng; ++g) {
            uint8_t *blk = wpt + (r * ng + g) * REF_PTQ1_BYTES;
            const uint16_t sb = scale_bits[r * ng + g];
            blk[0] = (uint8_t)(sb & 0xFF);
            blk[1] = (uint8_t)(sb >> 8);
            for (int c = 0; c < REF_PTQ1_CODES; ++c) {
                int t[5];
                for (int n = 0; n < 5; ++n) {
                    const int k = 5 * c + n;
                    t[n] = k < REF_GROUP ? w[r * cols + g * REF_GROUP + k] + 1 : 0;
                }
                blk[2 + c] = ref_ptq1_byte(t);
            }
        }
    }
}

void ref_ptq1_0_to_pq2_0(const uint8_t *wpt, int64_t rows, int64_t cols, uint8_t *wpq)
{
    const int64_t ng = cols / REF_GROUP;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < ng; ++g) {
            const uint8_t *src = wpt + (r * ng + g) * REF_PTQ1_BYTES;
            uint8_t *dst = wpq + (r * ng + g) * REF_PQ2_BYTES;
            memset(dst, 0, REF_PQ2_BYTES);
            dst[0] = src[0];
            dst[1] = src[1];
            for (int k = 0; k < REF_GROUP; ++k) {
                const int u = ref_ptq1_trit(src[2 + k / 5], k % 5);
                dst[2 + (k >> 2)] |= (uint8_t)(u << (2 * (k & 3)));
            }
        }
    }
}

/*
 * The GPU weight layout ("tq"). Same bits as pq2_0, another order:
 *  - rows are taken in blocks of 32 (the last block padded); groups of 128
 *    weights along a row as in pq2_0;
 *  - tile (row block rb, group g) is 1088 bytes at offset (rb * G + g) * 1088,
 *    G = cols / 128: 1024 code bytes, then the 32 fp16 scales of the block's
 *    rows (row l at byte 1024 + 2 l, little-endian);
 *  - weight k of the group for row l: with h = k / 64, wd = (k % 64) / 16,
 *    s = (k % 16) / 4, j = k % 4, its code sits in byte h*512 + l*16 + wd*4 + j
 *    at bits 2s .. 2s+1.
 * So one 32-bit word holds 16 consecutive weights, and masking it with
 * 0x03030303 << 2s leaves 4 consecutive weights, times 4^s, one per byte.
 * Padding rows get code 1 (w = 0) and scale 0.
 */
#define TQ_ROWS_PER_BLOCK 32
#define TQ_TILE_BYTES 1088
#define TQ_CODE_BYTES 1024

int64_t ref_repacked_bytes(int64_t rows, int64_t cols)
{
    const int64_t rb = (rows + TQ_ROWS_PER_BLOCK - 1) / TQ_ROWS_PER_BLOCK;
    return rb * (cols / REF_GROUP) * TQ_TILE_BYTES;
}

static int64_t tq_code_byte(int l, int k)
{
    const int h = k / 64, wd = (k % 64) / 16, j = k % 4;
    return (int64_t)h * 512 + l * 16 + wd * 4 + j;
}

static int tq_code_shift(int k)
{
    return 2 * ((k % 16) / 4);
}

void ref_repack(const uint8_t *wpq, int64_t rows, int64_t cols, uint8_t *wtq)
{
    const int64_t ng = cols / REF_GROUP;
    const int64_t nrb = (rows + TQ_ROWS_PER_BLOCK - 1) / TQ_ROWS_PER_BLOCK;
    memset(wtq, 0, (size_t)ref_repacked_bytes(rows, cols));
    for (int64_t rb = 0; rb < nrb; ++rb) {
        for (int64_t g = 0; g < ng; ++g) {
            uint8_t *tile = wtq + (rb * ng + g) * TQ_TILE_BYTES;
            for (int l = 0; l < TQ_ROWS_PER_BLOCK; ++l) {
                const int64_t r = rb * TQ_ROWS_PER_BLOCK + l;
                uint16_t sb = 0;
                for (int k = 0; k < REF_GROUP; ++k) {
                    int u = 1;
                    if (r < rows) u = pq2_code(wpq + (r * ng + g) * REF_PQ2_BYTES, k);
                    tile[tq_code_byte(l, k)] |= (uint8_t)(u << tq_code_shift(k));
                }
                if (r < rows) sb = pq2_scale_bits(wpq + (r * ng + g) * REF_PQ2_BYTES);
                tile[TQ_CODE_BYTES + 2 * l] = (uint8_t)(sb & 0xFF);
                tile[TQ_CODE_BYTES + 2 * l + 1] = (uint8_t)(sb >> 8);
            }
        }
    }
}

void ref_unrepack(const uint8_t *wtq, int64_t rows, int64_t cols, uint8_t *wpq)
{
    const int64_t ng = cols / REF_GROUP;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t rb = r / TQ_ROWS_PER_BLOCK;
        const int l = (int)(r % TQ_ROWS_PER_BLOCK);
        for (int64_t g = 0; g < ng; ++g) {
            const uint8_t *tile = wtq + (rb * ng + g) * TQ_TILE_BYTES;
            uint8_t *blk = wpq + (r * ng + g) * REF_PQ2_BYTES;
            memset(blk, 0, REF_PQ2_BYTES);
            blk[0] = tile[TQ_CODE_BYTES + 2 * l];
            blk[1] = tile[TQ_CODE_BYTES + 2 * l + 1];
            for (int k = 0; k < REF_GROUP; ++k) {
                const int u = (tile[tq_code_byte(l, k)] >> tq_code_shift(k)) & 3;
                blk[2 + (k >> 2)] |= (uint8_t)(u << (2 * (k & 3)));
            }
        }
    }
}

/* Activation q of token t at column c. */
static int q8K_value(const ref_block_q8K *xq, int64_t nb, int64_t t, int64_t c)
{
    return xq[t * nb + c / REF_QK].qs[c % REF_QK];
}

/*
 * Exact group sum of (u - 1) * q over the 128 weights of group g, taken
 * directly from the definition (w = u - 1, the ternary post, *what's
 * running*), not through bsums, so that the bsums identity stays a check.
 */
static int32_t group_sum(const uint8_t *wpq, const ref_block_q8K *xq, int64_t ng,
                         int64_t nb, int64_t r, int64_t g, int64_t t)
{
    const uint8_t *blk = wpq + (r * ng + g) * REF_PQ2_BYTES;
    int32_t s = 0;
    for (int k = 0; k < REF_GROUP; ++k)
        s += (pq2_code(blk, k) - 1) * q8K_value(xq, nb, t, g * REF_GROUP + k);
    return s;
}

void ref_groupsums(const uint8_t *wpq, const ref_block_q8K *xq, int64_t rows,
                   int64_t cols, int64_t ntok, int32_t *S)
{
    const int64_t ng = cols / REF_GROUP, nb = cols / REF_QK;
    for (int64_t t = 0; t < ntok; ++t)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t g = 0; g < ng; ++g)
                S[(t * rows + r) * ng + g] = group_sum(wpq, xq, ng, nb, r, g, t);
}

/*
 * y[t][r] = sum_g fp16(d_w[r][g]) * d_x[t][g/2] * isum[t][r][g]. Each term is
 * exact in double (11 + 24 + 15 significant bits); the sum is taken in double
 * and rounded once to f32. abs_sum collects |term| for the tolerance
 * |y_gpu - y| <= 1e-5 * abs_sum.
 */
void ref_matmul(const uint8_t *wpq, const ref_block_q8K *xq, int64_t rows,
                int64_t cols, int64_t ntok, float *y, double *abs_sum)
{
    const int64_t ng = cols / REF_GROUP, nb = cols / REF_QK;
    for (int64_t t = 0; t < ntok; ++t) {
        for (int64_t r = 0; r < rows; ++r) {
            double acc = 0.0, mag = 0.0;
            for (int64_t g = 0; g < ng; ++g) {
                const uint8_t *blk = wpq + (r * ng + g) * REF_PQ2_BYTES;
                const double dw = (double)ref_fp16_to_f32(pq2_scale_bits(blk));
                const double dx = (double)xq[t * nb + g / 2].d;
                const double isum = (double)group_sum(wpq, xq, ng, nb, r, g, t);
                const double term = dw * dx * isum;
                acc += term;
                mag += fabs(term);
            }
            y[t * rows + r] = (float)acc;
            abs_sum[t * rows + r] = mag;
        }
    }
}
