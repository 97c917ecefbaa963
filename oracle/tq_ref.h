/*
 * tq_ref.h -- plain CPU oracle of the ternary pq2_0 x q8_K matrix product.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may call this code. It shares nothing with the CUDA path:
 * no headers, tables or helpers. Single-threaded C99, no SIMD, no fast-math,
 * no floating-point contraction.
 *
 * Sources (web pages on the method):
 *  - "how i made a 27b ternary model 3.8x faster on a laptop cpu by reordering
 *    its bits", sections *what's running* (pq2_0: u = w + 1 in 2 bits, one fp16
 *    scale per 128 weights), *the trick with 4 and 16* (dot(w,y) = dot(u,y) -
 *    sum(y); the int32 bound), *stuff that went wrong* (block absmax 127 gives
 *    scale 1) and *did i break the model?* (exact integer oracle).
 *  - the ciot README (q8_K: 256 int8 values, a float scale and 16 partial sums
 *    per block; pq2_0 is 2.125 bits per weight).
 *  - "Quantization and the CPU", section *Quantizing the weights and
 *    activations* (symmetric int8: largest magnitude divided by 127).
 *
 * Readings where the pages are silent:
 *  - pq2_0 block = { uint16 fp16 scale; uint8 codes[32] }, 34 bytes; weight k
 *    of the block in code byte k >> 2, bits 2*(k & 3).
 *  - q8_K block = { float d; int8 qs[256]; int16 bsums[16] }, 292 bytes.
 *  - q8_K scale: amax = max |x|; d = amax / 127; q = round-half-even(x * (127 /
 *    amax)) clamped to [-127, 127]; an all-zero block has d = 0 and q = 0.
 *  - bsums[i] = sum of qs[16 i .. 16 i + 15].
 *  - output y[t][r] = sum over groups g of d_w[r][g] * d_x[t][g/2] * isum, with
 *    isum = sum_{k in g} (u - 1) * q, accumulated here in double.
 *
 * Parity of the exact f32 output bits between this oracle and the GPU is
 * unpinned (the float sum order is free); only the tolerance is contractual.
 */
#ifndef TQ_REF_H
#define TQ_REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define REF_QK 256
#define REF_GROUP 128
#define REF_PQ2_BYTES 34
#define REF_Q8K_BYTES 292

typedef struct {
    float d;
    int8_t qs[REF_QK];
    int16_t bsums[REF_QK / 16];
} ref_block_q8K;

/* IEEE binary16 bit pattern -> binary32 value (exact). */
float ref_fp16_to_f32(uint16_t h);

/* x[ntok][cols] -> y[ntok][cols/256]; cols % 256 == 0. */
void ref_quantize_q8K(const float *x, int64_t ntok, int64_t cols, ref_block_q8K *y);

/* pq2_0 -> ternary w[rows][cols] (u - 1, with code 3 giving 2) and scale bits. */
void ref_decode_pq2_0(const uint8_t *wpq, int64_t rows, int64_t cols,
                      int8_t *w, uint16_t *scale_bits);

/* The GPU weight layout ("tq"), see ref_repack in tq_ref.c for its definition. */
int64_t ref_repacked_bytes(int64_t rows, int64_t cols);
void ref_repack(const uint8_t *wpq, int64_t rows, int64_t cols, uint8_t *wtq);
void ref_unrepack(const uint8_t *wtq, int64_t rows, int64_t cols, uint8_t *wpq);

/*
 * ptq1_0, the 1.75-bit file ("how i made a 27b ternary model ... faster",
 * section *the detour that lost*): five weights per byte in base 3, since
 * 3^5 = 243 fits in 256; weight n of byte b is floor(3 * (b * 3^n mod 256) /
 * 256), which the page notes equals (v >= 86) + (v >= 171) for
 * v = b * 3^n mod 256. Readings where the page is silent:
 *  - block = { uint16 fp16 scale; uint8 codes[26] }, 28 bytes per 128
 *    weights: 1.75 bits per weight, and 28 / 34 makes the file 18% smaller
 *    than pq2_0, as the page says;
 *  - weight k of the block is trit k % 5 of code byte k / 5; the last byte
 *    holds weights 125..127 as trits 0..2 and zero trits 3 and 4;
 *  - a trit is the code u = w + 1 in {0, 1, 2}, as in pq2_0;
 *  - a byte for trits t0..t4 is the smallest b whose trits decode to them:
 *    b = ceil(256 q / 243) with q = sum_n t_n 3^(4 - n).
 */
#define REF_PTQ1_BYTES 28
#define REF_PTQ1_CODES 26

/* Trit n (0..4) of a ptq1_0 code byte, from the page's formula. */
int ref_ptq1_trit(uint8_t b, int n);
/* The code byte of trits t[0..4], each in {0, 1, 2}. */
uint8_t ref_ptq1_byte(const int *t);
/* ternary w[rows][cols] (-1, 0, 1) and scale bits -> ptq1_0 blocks. */
void ref_encode_ptq1_0(const int8_t *w, const uint16_t *scale_bits, int64_t rows,
                       int64_t cols, uint8_t *wpt);
/* ptq1_0 -> pq2_0 blocks of the same weights and scales. */
void ref_ptq1_0_to_pq2_0(const uint8_t *wpt, int64_t rows, int64_t cols, uint8_t *wpq);

/* S[t][r][g] = sum_{k<128} (u[r][128g+k] - 1) * q[t][128g+k]. */
void ref_groupsums(const uint8_t *wpq, const ref_block_q8K *xq, int64_t rows,
                   int64_t cols, int64_t ntok, int32_t *S);

/* y[t][r] (f32) and abs_sum[t][r] = sum_g |term| of the f64 terms. */
void ref_matmul(const uint8_t *wpq, const ref_block_q8K *xq, int64_t rows,
                int64_t cols, int64_t ntok, float *y, double *abs_sum);

#ifdef __cplusplus
}
#endif
#endif
