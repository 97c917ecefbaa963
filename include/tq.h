/*
 * tq.h -- C ABI of the ternary-weight x int8-activation matrix product
 * (pq2_0 weights, q8_K activations) on NVIDIA GB300 (sm_103a).
 *
 * The method (web pages "how i made a 27b ternary model 3.8x faster on a
 * laptop cpu by reordering its bits" and the ciot README):
 *   - weights are ternary, w in {-1, 0, +1}, stored as u = w + 1 in 2 bits
 *     with one fp16 scale d_w per 128 weights of a row (format pq2_0,
 *     2.125 bits per weight);
 *   - activations are quantized on the fly to q8_K: blocks of 256 int8
 *     values q with one f32 scale d_x and 16 partial sums (bsums);
 *   - y[t][r] = sum over 128-weight groups g of
 *       d_w[r][g] * d_x[t][g/2] * isum[t][r][g],
 *     isum[t][r][g] = sum_{k in g} (u - 1) * q, an exact integer;
 *   - the weights are repacked once at load time into an order that makes
 *     unpacking cheap (post, section "the layout"; README "the repack runs
 *     once at model load").
 *
 * Conventions shared by every call:
 *   - all buffer pointers are DEVICE pointers (cudaMalloc, torch, or managed
 *     memory) of the current CUDA device, owned by the caller; the library
 *     allocates no memory and never synchronizes the device;
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream); work is enqueued on it and the call returns at once;
 *   - sizes are int64_t; a call with any size equal to 0 (no rows, no tokens)
 *     enqueues nothing and returns TQ_OK, except as stated below;
 *   - every call returns TQ_OK (0) or a negative TQ_ERR_* code; an error is
 *     returned before anything is enqueued, except TQ_ERR_CUDA, which reports
 *     a failed launch (tq_last_cuda_error() gives the cudaError_t);
 *   - buffers marked "16-byte aligned" must start on a 16-byte boundary
 *     (TQ_ERR_ALIGN otherwise); input and output buffers must not overlap.
 */
#ifndef TQ_H
#define TQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_OK            0
#define TQ_ERR_SHAPE    -1  /* cols % 256 != 0, or a negative size */
#define TQ_ERR_NULL     -2  /* a required pointer is NULL */
#define TQ_ERR_ALIGN    -3  /* a buffer breaks its alignment rule */
#define TQ_ERR_CUDA     -4  /* a CUDA launch or runtime call failed */
#define TQ_ERR_TIMEOUT  -5  /* a kernel gave up a bounded wait (tq_device_status) */
#define TQ_ERR_ALIAS    -6  /* an output buffer overlaps an input buffer */
#define TQ_ERR_WORKSPACE -7 /* workspace smaller than tq_matmul_workspace_bytes */

#define TQ_QK_K 256          /* activations per q8_K block */
#define TQ_GROUP 128         /* weights per pq2_0 scale */
#define TQ_PQ2_0_BYTES 34    /* bytes per pq2_0 block (fp16 scale + 32 code bytes) */
#define TQ_PTQ1_0_BYTES 28   /* bytes per ptq1_0 block (fp16 scale + 26 code bytes) */
#define TQ_Q8K_BYTES 292     /* bytes per q8_K block */
#define TQ_TILE_ROWS 32      /* rows per tile of the repacked layout */
#define TQ_TILE_BYTES 1088   /* bytes per tile: 32 rows x 128 weights */
#define TQ_STATIC_WS_BYTES (8 << 20)  /* fixed workspace of tq_matmul_static_ws: 8 MiB */

/*
 * q8_K block (ciot README: "256 int8 values, a float scale and 16 partial
 * sums per block"). Packed, 292 bytes, no padding; blocks of one token are
 * contiguous and tokens follow each other: block b of token t is element
 * t * (cols/256) + b of the array.
 */
typedef struct {
    float d;             /* scale: x ~= d * q */
    int8_t qs[256];      /* q in [-127, 127] */
    int16_t bsums[16];   /* bsums[i] = qs[16i] + ... + qs[16i+15] */
} tq_block_q8K;

/*
 * pq2_0 block (post, "what's running": 2 bits per weight as u = w + 1, one
 * fp16 scale per 128 weights; README: 2.125 bits per weight). The byte order
 * inside the block is this library's reading, the pages leave it open:
 * bytes 0..1 hold the fp16 scale (little-endian), bytes 2..33 the codes, and
 * weight k (0..127) of the block is in code byte k >> 2 at bits
 * 2*(k & 3) .. 2*(k & 3)+1. A weight matrix [rows][cols] is rows * cols/128
 * blocks, row-major: block (r, g) starts at byte (r * cols/128 + g) * 34.
 *
 * Repacked layout ("tq"), produced by tq_repack: the same bits in a GPU
 * order. Rows are taken in tiles of 32 (the last tile padded with code 1,
 * i.e. w = 0, and scale 0). Tile (row block rb, group g) is 1088 bytes at
 * offset (rb * cols/128 + g) * 1088: 1024 code bytes, then the 32 fp16
 * scales of its rows (row l at byte 1024 + 2l). The code of weight k of the
 * group, row l of the tile, is in byte h*512 + l*16 + wd*4 + j at bits 2s,
 * where h = k/64, wd = (k%64)/16, s = (k%16)/4, j = k%4. Hence:
 *   - each 32-bit word holds 16 consecutive weights of one row, and
 *     word & (0x03030303 << 2s) is 4 consecutive weights times 4^s, one per
 *     byte, lined up with 4 consecutive int8 activations (one AND per
 *     dp4a operand: the post's "trick with 4 and 16", on 32-bit lanes);
 *   - a warp reading 16 bytes per lane reads 512 contiguous bytes: 64
 *     weights of each of 32 rows.
 */

/*
 * tq_quantize_q8K -- quantize activations to q8_K (ciot README: activations
 * are quantized on the fly to q8_K). For each block of 256 values:
 * amax = max |x|; if amax == 0 the block is all zero (d = 0); otherwise
 * d = amax / 127 and q = round-to-nearest-even(x * (127 / amax)) clamped to
 * [-127, 127] (one IEEE division for 127/amax, one for d); bsums[i] is the
 * sum of qs[16i .. 16i+15]. Inputs must be finite, with every nonzero
 * block's amax at least 2^-126 (smaller values are out of contract).
 *   X   [ntok][cols] f32, row-major, 16-byte aligned.
 *   Xq  [ntok][cols/256] tq_block_q8K, 16-byte aligned, written.
 * Errors: TQ_ERR_SHAPE if cols % 256 != 0 or a size is negative.
 */
int tq_quantize_q8K(const float *X, void *Xq, int64_t ntok, int64_t cols, void *stream);

/* Bytes of the repacked weights: ceil(rows/32) * (cols/128) * 1088, which is
 * rows * cols/128 * 34 (the pq2_0 size) when rows % 32 == 0; -1 if
 * cols % 128 != 0 or a size is negative. */
int64_t tq_repacked_bytes(int64_t rows, int64_t cols);

/*
 * tq_repack -- load-time repack of pq2_0 weights into the tq layout (post,
 * "the layout": "it runs once when the model loads"). A pure permutation of
 * bits: every code, including the unused value 3, is moved as is.
 * Out-of-place (the pages repack in place; on the GPU the copy avoids
 * hazards between thread blocks).
 *   Wpq2 [rows][cols/128] pq2_0 blocks, 16-byte aligned.
 *   Wtq  tq_repacked_bytes(rows, cols) bytes, 16-byte aligned, written.
 * Errors: TQ_ERR_SHAPE if cols % 128 != 0; TQ_ERR_ALIAS if the buffers overlap.
 */
int tq_repack(const void *Wpq2, void *Wtq, int64_t rows, int64_t cols, void *stream);

/* tq_unrepack -- the exact inverse of tq_repack (padding rows are dropped). */
int tq_unrepack(const void *Wtq, void *Wpq2, int64_t rows, int64_t cols, void *stream);

/*
 * ptq1_0, the 1.75-bit file (post, "the detour that lost"): five ternary
 * weights per code byte in base 3 (3^5 = 243 fits in 256); trit n of byte b
 * is floor(3 * (b * 3^n mod 256) / 256) = (v >= 86) + (v >= 171) with
 * v = b * 3^n mod 256, and a trit is the code u = w + 1. Block (where the
 * post is silent, our reading): { uint16 fp16 scale; uint8 codes[26] } per
 * 128 weights of a row, 28 bytes, weight k in trit k % 5 of code byte k / 5;
 * blocks row-major like pq2_0.
 *
 * tq_ptq1_0_bytes -- rows * cols/128 * 28; -1 if cols % 128 != 0 or a size is
 * negative.
 *
 * tq_repack_ptq1_0 -- load-time decode of ptq1_0 weights into the tq layout:
 * writes exactly the bytes tq_repack writes for the pq2_0 file of the same
 * weights and scales, so every matmul entry point takes the result. The file
 * is 18% smaller; the weights stream at 2.125 bits per weight, because base-3
 * decoding costs several integer operations per weight where the tq layout
 * needs one AND per four (the post found the same trade on the CPU).
 *   Wpt [rows][cols/128] ptq1_0 blocks, 16-byte aligned.
 *   Wtq tq_repacked_bytes(rows, cols) bytes, 16-byte aligned, written.
 * Errors: as tq_repack.
 */
int64_t tq_ptq1_0_bytes(int64_t rows, int64_t cols);
int tq_repack_ptq1_0(const void *Wpt, void *Wtq, int64_t rows, int64_t cols, void *stream);

/*
 * The streamed 1.75-bit form (post, "the detour that lost": the file is 18%
 * smaller, and on a machine limited by memory that should win; on the CPU the
 * decode cost more than the bytes saved). Here the GEMV streams the ptq1_0
 * bytes themselves and decodes them in the kernel: each code byte goes
 * through a 256-entry shared-memory table (byte -> its five trits as 2-bit
 * codes), the five-weight chunks are laid end to end into the same 2-bit code
 * words the pq2_0 path uses, and the activations are staged in the matching
 * order, so the dot product is the same AND-per-slot dp4a. Measured on GB300
 * with one token on the 32768 x 8192 decode matrix it takes 30.6 us per
 * launch against 12.8 us for the 2-bit stream of the same weights: the
 * decode costs about 2.5 times the 2-bit unpack's instructions, more than the
 * 18% fewer bytes save. As on the CPU, the file is therefore decoded once at
 * load (tq_repack_ptq1_0) for the product path; this form is kept so that the
 * trade can be measured.
 *
 * tq_ptq1_0_stream_bytes -- ceil(rows/32) * (cols/128) * 896; -1 if
 * cols % 128 != 0 or a size is negative.
 *
 * tq_repack_ptq1_0_stream -- load-time re-tiling of a ptq1_0 file, no decode:
 * tile (row block rb, group g) is 896 bytes at (rb * cols/128 + g) * 896, the
 * 28-byte blocks of rows 32 rb .. 32 rb + 31 and group g, row l at byte 28 l
 * (rows past the matrix: scale 0 and code bytes 0x80, five trits of 1: w = 0).
 *   Wpt [rows][cols/128] ptq1_0 blocks, 16-byte aligned.
 *   Wt1 tq_ptq1_0_stream_bytes(rows, cols) bytes, 16-byte aligned, written.
 * Errors: as tq_repack_ptq1_0.
 *
 * tq_matmul_ptq1_0_stream / tq_matmul_ptq1_0_stream_groupsums -- tq_matmul and
 * tq_matmul_groupsums over the stream tiles: the same results (the same exact
 * group sums, the same tolerance on Y), in launches of up to 8 tokens, each
 * reading the weights once.
 *   Wt1 the stream tiles, 16-byte aligned; Xq, Y, S as tq_matmul(_groupsums).
 * Errors: as tq_matmul.
 */
int64_t tq_ptq1_0_stream_bytes(int64_t rows, int64_t cols);
int tq_repack_ptq1_0_stream(const void *Wpt, void *Wt1, int64_t rows, int64_t cols, void *stream);
int tq_matmul_ptq1_0_stream(const void *Wt1, const void *Xq, float *Y, int64_t rows, int64_t cols,
                            int64_t ntok, void *stream);
int tq_matmul_ptq1_0_stream_groupsums(const void *Wt1, const void *Xq, int32_t *S, int64_t rows,
                                      int64_t cols, int64_t ntok, void *stream);

/*
 * tq_matmul -- Y = the ternary x q8_K product (definition at the top).
 * Each group sum is exact in int32 (post, "the trick with 4 and 16": the
 * largest scaled intermediate is 520,192); the scale products and the sum
 * over groups are f32, accumulated in an order the library chooses, within
 * 1e-5 of sum_g |d_w d_x isum| of the exact value.
 * Routing by ntok (post, "the leftovers": never one weight pass per leftover
 * token): ntok <= 16 runs a bandwidth-bound GEMV that reads the weights once
 * for all tokens (dp4a for 1 to 3 tokens, warp-level f16 MMAs over 8-column
 * token blocks from 4; once per half of the tokens where the activations of
 * all do not fit in shared memory, as 8 tokens of 17408 columns or 16 of
 * 8192; the tensor-core path only where not even one token's do); larger
 * ntok runs a tcgen05 tensor-core kernel with the token dimension
 * zero-padded to its tile, storing only the real outputs.
 *   Wtq [tq layout] repacked weights, 16-byte aligned.
 *   Xq  [ntok][cols/256] q8_K blocks, 16-byte aligned.
 *   Y   [ntok][rows] f32, 4-byte aligned, overwritten (not accumulated).
 * With cols == 0 and rows, ntok > 0, Y is set to zero.
 * Overlap: the kernels are launched as programmatic dependents, so they may
 * start while the kernel enqueued before them on the stream is finishing; they
 * wait for it before reading Xq. When the previous call this library received
 * for the stream was tq_quantize_q8K, the GEMV also starts reading Wtq before
 * that wait, since the quantizer never writes weights; so do not write Wtq
 * with a kernel of your own between tq_quantize_q8K and tq_matmul on one
 * stream (copies and events are fine).
 * GEMV chains in a graph: a GEMV lets the next kernel start only after its
 * own wait. While a stream is being captured, a GEMV whose one dependency in
 * the capture is the previous call's GEMV node (nothing else was captured
 * between them), and none of whose inputs (Wtq, Xq, or X for
 * tq_quantize_matmul) overlaps that GEMV's outputs (Y or S, and Xq it
 * wrote), reads its inputs before waiting and waits only before its first
 * store: after its first ring stage where a 32-row tile column takes three
 * or more stages (more than 8192 columns at 1 to 3 tokens), else after its
 * first tile column where every CTA has two or more (the 32768 x 8192 decode
 * matrix), else at its start as usual; the group-sum form always waits
 * first. Back-to-back decode matmuls in a graph then overlap each other's
 * start and end. Outside a capture the library cannot see what else is on
 * the stream and always waits first.
 * Errors: TQ_ERR_SHAPE if cols % 256 != 0; TQ_ERR_ALIAS if Y overlaps an input.
 */
int tq_matmul(const void *Wtq, const void *Xq, float *Y, int64_t rows, int64_t cols,
              int64_t ntok, void *stream);

/*
 * tq_matmul_groupsums -- parity/debug form of tq_matmul: runs the same
 * kernels (chosen by ntok the same way) but stores the exact integer group
 * sums instead of Y.
 *   S [ntok][rows][cols/128] int32, 4-byte aligned: S[t][r][g] = isum[t][r][g].
 */
int tq_matmul_groupsums(const void *Wtq, const void *Xq, int32_t *S, int64_t rows,
                        int64_t cols, int64_t ntok, void *stream);

/*
 * tq_matmul_workspace_bytes -- scratch needed by tq_matmul_ws for this shape:
 * 0 when ntok <= 3 (the GEMV needs none). From 4 to 8 tokens the GEMV's
 * activations staged once, as f16 rows: with R = round16(ntok * (2*cols + 8)),
 * round16(R + ntok * (cols/128) * 4 + ntok * (cols/256) * 4) bytes (round16:
 * up to a multiple of 16); 0 below 3072 columns (staging does not pay there)
 * and where that GEMV would need more than the 227 KB of shared memory a
 * block may opt in to (cols > 9984 at 8 tokens, cols > 19968 at 4).
 * Otherwise, with the token tile T = 16 for
 * ntok <= 16, 32 for ntok <= 32, else 64,
 * ceil(ntok/T) * (cols/128) * 256*T + ceil(ntok/T) * (cols/256) * 12*T bytes.
 * -1 for a bad shape.
 */
int64_t tq_matmul_workspace_bytes(int64_t rows, int64_t cols, int64_t ntok);

/*
 * tq_matmul_ws -- tq_matmul with a caller-provided workspace, the faster form
 * for ntok >= 9 (measured on GB300 on a 17408 x 5120 matrix: 1.25-1.4x at 9
 * to 16 tokens, where tq_matmul runs the GEMV; 1.8-2.2x from 17 to 130
 * tokens): a pre-pass converts the q8_K activations once into the
 * tensor cores' operand layout in the workspace (each int8 split exactly
 * into two e4m3 parts, instead of every 128-row tile of the weights
 * converting them again), then the tensor-core kernel reads them with one
 * bulk copy per q8_K block. Same results
 * and tolerance as tq_matmul. For ntok <= 8 it runs tq_matmul's GEMV; from 4
 * tokens and 5120 columns (where the workspace size is not 0) a small kernel
 * first converts the activations once into the GEMV's f16 layout in the
 * workspace, which every CTA of the GEMV then loads with one bulk copy
 * instead of converting them itself (measured in graph chains: 1.0-1.15x
 * faster from 5120 columns, slower below, where each CTA converts before
 * waiting for the launch before it). From 9 tokens on it runs the tensor-core
 * kernel on token tiles of 16, 32 or 64 where tq_matmul would still run the
 * GEMV up to 16.
 *   workspace  device buffer of at least tq_matmul_workspace_bytes(rows, cols,
 *              ntok) bytes, 16-byte aligned, owned by the caller; its contents
 *              are overwritten and meaningless after the call; it must not
 *              overlap Wtq, Xq or Y. Calls that share a workspace must be
 *              ordered (the same stream, or synchronized streams).
 * Errors: as tq_matmul; TQ_ERR_NULL if the workspace is needed and NULL;
 * TQ_ERR_WORKSPACE if it is smaller than needed; TQ_ERR_ALIGN if it is
 * misaligned; TQ_ERR_ALIAS if it overlaps another buffer.
 */
int tq_matmul_ws(const void *Wtq, const void *Xq, float *Y, int64_t rows, int64_t cols,
                 int64_t ntok, void *workspace, int64_t workspace_bytes, void *stream);

/* tq_matmul_groupsums_ws -- tq_matmul_groupsums through the kernels of
 * tq_matmul_ws (parity/debug): S[t][r][g] = isum[t][r][g]. */
int tq_matmul_groupsums_ws(const void *Wtq, const void *Xq, int32_t *S, int64_t rows,
                           int64_t cols, int64_t ntok, void *workspace,
                           int64_t workspace_bytes, void *stream);

/*
 * tq_quantize_matmul -- tq_quantize_q8K then tq_matmul_ws in one call: Xq =
 * the q8_K blocks of X, Y = the product of Wtq and Xq. For ntok <= 3 (and up
 * to 8 where the workspace size is 0, as below 3072 columns) it is one
 * fused launch: every CTA of the GEMV quantizes X into its shared memory
 * itself (with the quantizer's arithmetic, so Xq and Y carry the bits of the
 * two separate calls), and writes Xq (CTA 0 at its start; in the graph chains
 * tq_matmul describes, every CTA a share after its wait). That removes a launch and the
 * quantizer's place on the critical path of each matmul. From 4 to 8 tokens
 * with a workspace, one small kernel quantizes X (the same arithmetic),
 * writes Xq and stages the GEMV's activations in the workspace, then the
 * GEMV runs (measured in graph chains: 1.02-1.7x faster than the fused launch
 * from 3072 columns; 11.4 against 12.6 us at 4 tokens on 17408 x 5120).
 * For ntok >= 9 one
 * kernel quantizes X (the same arithmetic), writes Xq and packs the
 * workspace, which the tensor-core kernel then reads: two launches instead
 * of three, the same bits.
 *   X  [ntok][cols] f32, 16-byte aligned (as tq_quantize_q8K).
 *   Xq [ntok][cols/256] q8_K, 16-byte aligned: written.
 *   Wtq, Y, workspace, workspace_bytes: as tq_matmul_ws (the workspace is
 *   used from 4 tokens on where its size is not 0).
 * Overlap: like tq_matmul after tq_quantize_q8K, the launch may start
 * reading Wtq before the kernel enqueued just before it ends when the
 * previous call this library received for the stream was the quantizer or a
 * matmul; so do not write Wtq with a kernel of your own between such a call
 * and this one on one stream. In a captured chain of GEMVs it may read X and
 * Wtq before the previous GEMV ends, under the conditions tq_matmul states.
 * Errors: those of tq_quantize_q8K and tq_matmul_ws, checked before anything
 * is enqueued.
 */
int tq_quantize_matmul(const void *Wtq, const float *X, void *Xq, float *Y, int64_t rows,
                       int64_t cols, int64_t ntok, void *workspace, int64_t workspace_bytes,
                       void *stream);

/*
 * tq_matmul_host -- one whole step from host memory to host memory, in one
 * call: copy X from the host, quantize and multiply (tq_quantize_matmul),
 * copy Y back to the host. Everything is enqueued on `stream`
 * with cudaMemcpyAsync and kernel launches; the call returns at once, so the
 * caller synchronizes the stream before reading Y_host.
 *   X_host [ntok][cols] f32 host memory, pinned (page-locked) for the copy
 *          to be asynchronous; it must stay unchanged until the copy is done.
 *   X      [ntok][cols] f32 device staging buffer, 16-byte aligned.
 *   Xq     [ntok][cols/256] q8_K device buffer, 16-byte aligned.
 *   Y      [ntok][rows] f32 device buffer, 4-byte aligned.
 *   Y_host [ntok][rows] f32 host memory, pinned; written when the stream
 *          reaches the copy.
 *   Wtq, workspace, workspace_bytes: as tq_matmul_ws.
 * Errors: those of tq_quantize_q8K and tq_matmul_ws, checked before anything
 * is enqueued; TQ_ERR_NULL for a NULL host or staging buffer; TQ_ERR_CUDA if
 * a copy or launch fails (work already enqueued stays enqueued).
 */
int tq_matmul_host(const void *Wtq, const float *X_host, float *X, void *Xq, float *Y,
                   float *Y_host, int64_t rows, int64_t cols, int64_t ntok, void *workspace,
                   int64_t workspace_bytes, void *stream);

/*
 * tq_matmul_static_ws -- tq_matmul_ws without a caller workspace: the
 * workspace is a fixed device array of TQ_STATIC_WS_BYTES inside this
 * library, so the call allocates nothing. The paper has no counterpart to
 * this entry point; it exists for callers that cannot allocate device memory
 * where they run the matmul (a plugin that only receives input and output
 * pointers from its host application, an engine that allows no allocation
 * after start-up because cudaMalloc can synchronize the device, code whose
 * caching allocator must not be bypassed).
 *   Same arguments, results and errors as tq_matmul_ws, minus the workspace.
 *   Limit: tq_matmul_workspace_bytes(rows, cols, ntok) <= TQ_STATIC_WS_BYTES,
 *   else TQ_ERR_WORKSPACE before anything runs (for example cols = 5120
 *   allows ntok <= 768; ntok <= 8 needs at most the GEMV's staged
 *   activations, under 227 KB, and has no limit).
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current), which may also load the
 *   library's code for the array onto that device; make that first call
 *   before any stream capture. TQ_ERR_CUDA if the look-up fails.
 *   Memory: the array occupies TQ_STATIC_WS_BYTES on every GPU where it has
 *   been loaded, until the process exits. The looked-up address is kept for
 *   the life of the process: do not use the library on a device after
 *   cudaDeviceReset (or any reset of its primary context) there, since the
 *   array then moves and the kept address is stale.
 *   Sharing: every call uses the same array, which keeps the last call's
 *   contents (nothing in it needs to start at zero: the pre-pass rewrites all
 *   of it that the matmul reads). Calls whose kernels overlap on the GPU
 *   (different streams, different host threads) race on it and give wrong
 *   results; order them on one stream or synchronize between them.
 */
int tq_matmul_static_ws(const void *Wtq, const void *Xq, float *Y, int64_t rows, int64_t cols,
                        int64_t ntok, void *stream);

/* Human-readable name of a TQ_* code. */
const char *tq_strerror(int code);

/* cudaError_t of the last TQ_ERR_CUDA returned on this host thread (0 if none). */
int tq_last_cuda_error(void);

/*
 * tq_device_status -- read and clear the device-side status word of the
 * current device. Kernels that wait on a barrier bound the wait; one that
 * gives up sets this word and returns early (its outputs are then
 * undefined). Returns TQ_OK, TQ_ERR_TIMEOUT, or TQ_ERR_CUDA. This call
 * synchronizes the device (it copies the word to the host).
 */
int tq_device_status(void);

/*
 * tq_probe_read_sum -- measurement aid: the memory-read ceiling the GEMV is
 * judged against (the post measures its DRAM read ceiling the same way, in
 * "the ceiling": a sum over a large buffer). Adds every 32-bit word of buf,
 * as unsigned integers modulo 2^32, to *out, reading buf once with 128-bit
 * streaming loads and nothing else; time it to get the read rate.
 *   buf    bytes of device memory, 16-byte aligned; bytes a multiple of 16.
 *   out    one uint32 in device memory, 4-byte aligned; added to (atomically).
 *   early  nonzero: the loads may start before the kernel enqueued just
 *          before on the stream finishes (the caller promises that kernel
 *          does not write buf); the store into out still waits for it.
 * Errors: TQ_ERR_SHAPE if bytes < 0 or bytes % 16 != 0; TQ_ERR_NULL;
 * TQ_ERR_ALIGN; TQ_ERR_ALIAS if out lies in buf.
 */
int tq_probe_read_sum(const void *buf, int64_t bytes, uint32_t *out, int early, void *stream);

/*
 * tq_debug_stall_next_launch -- test facility for the timeout path (the pages
 * have no counterpart). The next matmul kernel this library launches, from
 * any host thread and on any stream, runs with its first thread block (the
 * first pair of blocks for the tensor-core kernel, which runs on CTA pairs)
 * requesting none of its input copies, as if they never arrived: those
 * blocks' waits expire after wait_limit_ns (instead of the usual 2 s), they
 * set the device status word and return; the other blocks finish normally.
 * Its outputs are then undefined, and tq_device_status() reports
 * TQ_ERR_TIMEOUT (and clears the word). The block still waits for any copy
 * it did request before it exits, so no copy outlives it. Nothing faults and
 * nothing waits without bound. Kernels that take it: the GEMV (ntok <= 16, or <= 8
 * in the workspace forms) and
 * the tensor-core kernel of the workspace forms. wait_limit_ns = 0 cancels a
 * pending stall.
 * Errors: TQ_ERR_SHAPE if wait_limit_ns < 0.
 */
int tq_debug_stall_next_launch(int64_t wait_limit_ns);

/* Library version as "major.minor.patch". */
const char *tq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
