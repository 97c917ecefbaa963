// tq_repack.cu -- load-time permutation of pq2_0 weights into the tq layout,
// its inverse, and the load-time decode of the 1.75-bit ptq1_0 file into the
// same layout.
//
// The ternary post ("the layout") repacks once at model load so that
// unpacking costs one AND per vector; this is the GPU version of that step,
// with a GPU-chosen order (layout defined in include/tq.h).
//
// One warp per tile (32 rows x 128 weights); lane l handles row l. A 32-bit
// word of pq2_0 codes covers 16 consecutive weights: byte s holds weights
// 4s..4s+3 at bits 0, 2, 4, 6. The tq word of the same 16 weights holds in
// byte j the weights j, 4+j, 8+j, 12+j at bits 0, 2, 4, 6. Viewing the word as
// a 4x4 matrix of 2-bit fields (row = byte), one layout is the transpose of
// the other, done with two delta swaps (off-diagonal 2x2 blocks, then within
// each block). A transpose is its own inverse, so unrepack uses the same swap.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ uint32_t transpose_2bit_4x4(uint32_t x) {
  uint32_t t = (x ^ (x >> 12)) & 0x0000F0F0u;  // fields (s<2, j>=2) <-> (s+2, j-2)
  x ^= t ^ (t << 12);
  t = (x ^ (x >> 6)) & 0x00CC00CCu;            // fields (s even, j odd) <-> (s+1, j-1)
  x ^= t ^ (t << 6);
  return x;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
repack_kernel(const uint8_t* __restrict__ Wpq2, uint8_t* __restrict__ Wtq, int64_t rows,
              int64_t ngroups, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  const int64_t tile = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (tile >= ntiles) return;
  const int64_t rb = tile / ngroups, g = tile - rb * ngroups;
  const int64_t r = rb * kTileRows + lane;
  uint8_t* out = Wtq + tile * kTileBytes;

  uint32_t w[8];
  uint16_t scale = 0;
  if (r < rows) {
    // pq2_0 blocks are 34 bytes, so only 2-byte alignment is guaranteed.
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(Wpq2 + (r * ngroups + g) * kPq2Bytes);
    scale = blk[0];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = transpose_2bit_4x4((uint32_t)blk[1 + 2 * i] | ((uint32_t)blk[2 + 2 * i] << 16));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0x55555555u;  // padding rows: code 1, w = 0
  }
  // words 0..3 cover weights 0..63 (h = 0), words 4..7 weights 64..127 (h = 1)
  *reinterpret_cast<uint4*>(out + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(out + 512 + lane * 16) = make_uint4(w[4], w[5], w[6], w[7]);
  reinterpret_cast<uint16_t*>(out + kTileCodeBytes)[lane] = scale;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
unrepack_kernel(const uint8_t* __restrict__ Wtq, uint8_t* __restrict__ Wpq2, int64_t rows,
                int64_t ngroups, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  const int64_t tile = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (tile >= ntiles) return;
  const int64_t rb = tile / ngroups, g = tile - rb * ngroups;
  const int64_t r = rb * kTileRows + lane;
  if (r >= rows) return;
  const uint8_t* in = Wtq + tile * kTileBytes;
  const uint4 lo = *reinterpret_cast<const uint4*>(in + lane * 16);
  const uint4 hi = *reinterpret_cast<const uint4*>(in + 512 + lane * 16);
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint16_t* blk = reinterpret_cast<uint16_t*>(Wpq2 + (r * ngroups + g) * kPq2Bytes);
  blk[0] = reinterpret_cast<const uint16_t*>(in + kTileCodeBytes)[lane];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t p = transpose_2bit_4x4(w[i]);
    blk[1 + 2 * i] = (uint16_t)(p & 0xFFFFu);
    blk[2 + 2 * i] = (uint16_t)(p >> 16);
  }
}

// ptq1_0 (five weights per code byte in base 3; block = fp16 scale + 26 code
// bytes, 28 bytes per 128 weights; weight k is trit k % 5 of code byte k / 5)
// into the tq layout: lane l decodes row l of the tile. Trit n of byte b is
// floor(3 * (b * 3^n mod 256) / 256) (the ternary post, "the detour that
// lost"), the code u = w + 1, written where tq_repack puts weight k.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
repack_ptq1_kernel(const uint8_t* __restrict__ Wpt, uint8_t* __restrict__ Wtq, int64_t rows,
                   int64_t ngroups, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  const int64_t tile = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (tile >= ntiles) return;
  const int64_t rb = tile / ngroups, g = tile - rb * ngroups;
  const int64_t r = rb * kTileRows + lane;
  uint8_t* out = Wtq + tile * kTileBytes;

  uint32_t w[8];
  uint16_t scale = 0;
  if (r < rows) {
    // 28-byte blocks: 4-byte alignment. Byte 2 + c of the block is code byte c.
    const uint32_t* blk = reinterpret_cast<const uint32_t*>(Wpt + (r * ngroups + g) * kPtq1Bytes);
    uint32_t bw[kPtq1Bytes / 4];
#pragma unroll
    for (int i = 0; i < kPtq1Bytes / 4; ++i) bw[i] = blk[i];
    scale = (uint16_t)(bw[0] & 0xFFFFu);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0u;
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
      const int c = k / 5, n = k % 5;
      const uint32_t b = (bw[(2 + c) >> 2] >> (8 * ((2 + c) & 3))) & 0xFFu;
      const uint32_t u = ptq1_trit(b, n);
      // tq position of weight k: word (k / 64) * 4 + (k % 64) / 16, byte k % 4,
      // bits 2 * ((k % 16) / 4)
      w[(k >> 6) * 4 + ((k & 63) >> 4)] |= u << (8 * (k & 3) + 2 * ((k & 15) >> 2));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0x55555555u;  // padding rows: code 1, w = 0
  }
  *reinterpret_cast<uint4*>(out + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(out + 512 + lane * 16) = make_uint4(w[4], w[5], w[6], w[7]);
  reinterpret_cast<uint16_t*>(out + kTileCodeBytes)[lane] = scale;
}

// ptq1_0 stream layout: one warp per (32-row block, group) tile; lane l
// copies row l's 28-byte block (seven words) to byte 28 l of the tile. Rows
// past the matrix get scale 0 and code bytes 0x80 (five trits of 1: w = 0).
__global__ void __launch_bounds__(kWarpsPerCta * 32)
repack_ptq1_stream_kernel(const uint8_t* __restrict__ Wpt, uint8_t* __restrict__ Wt1, int64_t rows,
                          int64_t ngroups, int64_t ntiles) {
  const int lane = threadIdx.x & 31;
  const int64_t tile = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (tile >= ntiles) return;
  const int64_t rb = tile / ngroups, g = tile - rb * ngroups;
  const int64_t r = rb * kTileRows + lane;
  uint32_t* out = reinterpret_cast<uint32_t*>(Wt1 + tile * kTq1TileBytes + lane * kPtq1Bytes);
  if (r < rows) {
    const uint32_t* blk = reinterpret_cast<const uint32_t*>(Wpt + (r * ngroups + g) * kPtq1Bytes);
#pragma unroll
    for (int i = 0; i < kPtq1Bytes / 4; ++i) out[i] = blk[i];
  } else {
    out[0] = 0x80800000u;
#pragma unroll
    for (int i = 1; i < kPtq1Bytes / 4; ++i) out[i] = 0x80808080u;
  }
}

int64_t tile_count(int64_t rows, int64_t cols) {
  return (rows + kTileRows - 1) / kTileRows * (cols / kGroup);
}

}  // namespace

cudaError_t launch_repack(const uint8_t* Wpq2, uint8_t* Wtq, int64_t rows, int64_t cols,
                          cudaStream_t s) {
  const int64_t ntiles = tile_count(rows, cols);
  if (ntiles <= 0) return cudaSuccess;
  const int64_t grid = (ntiles + kWarpsPerCta - 1) / kWarpsPerCta;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  repack_kernel<<<(unsigned)grid, kWarpsPerCta * 32, 0, s>>>(Wpq2, Wtq, rows, cols / kGroup,
                                                             ntiles);
  return cudaGetLastError();
}

cudaError_t launch_repack_ptq1(const uint8_t* Wpt, uint8_t* Wtq, int64_t rows, int64_t cols,
                               cudaStream_t s) {
  const int64_t ntiles = tile_count(rows, cols);
  if (ntiles <= 0) return cudaSuccess;
  const int64_t grid = (ntiles + kWarpsPerCta - 1) / kWarpsPerCta;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  repack_ptq1_kernel<<<(unsigned)grid, kWarpsPerCta * 32, 0, s>>>(Wpt, Wtq, rows, cols / kGroup,
                                                                  ntiles);
  return cudaGetLastError();
}

cudaError_t launch_repack_ptq1_stream(const uint8_t* Wpt, uint8_t* Wt1, int64_t rows,
                                      int64_t cols, cudaStream_t s) {
  const int64_t ntiles = tile_count(rows, cols);
  if (ntiles <= 0) return cudaSuccess;
  const int64_t grid = (ntiles + kWarpsPerCta - 1) / kWarpsPerCta;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  repack_ptq1_stream_kernel<<<(unsigned)grid, kWarpsPerCta * 32, 0, s>>>(Wpt, Wt1, rows,
                                                                         cols / kGroup, ntiles);
  return cudaGetLastError();
}

cudaError_t launch_unrepack(const uint8_t* Wtq, uint8_t* Wpq2, int64_t rows, int64_t cols,
                            cudaStream_t s) {
  const int64_t ntiles = tile_count(rows, cols);
  if (ntiles <= 0) return cudaSuccess;
  const int64_t grid = (ntiles + kWarpsPerCta - 1) / kWarpsPerCta;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  unrepack_kernel<<<(unsigned)grid, kWarpsPerCta * 32, 0, s>>>(Wtq, Wpq2, rows, cols / kGroup,
                                                               ntiles);
  return cudaGetLastError();
}

}  // namespace tq
