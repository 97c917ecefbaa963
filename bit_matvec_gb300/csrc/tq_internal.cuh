// tq_internal.cuh -- shared internals of the CUDA path: layout constants,
// small PTX wrappers and the launchers each kernel file exports to the C ABI
// file. Nothing here is visible outside the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/tq.h"

namespace tq {

constexpr int kQK = TQ_QK_K;             // activations per q8_K block
constexpr int kGroup = TQ_GROUP;         // weights per scale
constexpr int kPq2Bytes = TQ_PQ2_0_BYTES;
constexpr int kQ8KBytes = TQ_Q8K_BYTES;
constexpr int kTileRows = TQ_TILE_ROWS;  // rows per tile of the tq layout
constexpr int kTileBytes = TQ_TILE_BYTES;
constexpr int kTileCodeBytes = 1024;     // code bytes per tile; fp16 scales follow
constexpr int kQ8KQsOffset = 4;          // byte offset of qs in a q8_K block
constexpr int kQ8KBsumsOffset = 260;     // byte offset of bsums in a q8_K block

// Status word values written by kernels on the device.
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 1;

// ---------------------------------------------------------------- loads

// 16-byte streaming load through the non-coherent path, not kept in L1:
// weights are read exactly once per launch.
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ldg_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Unsigned-by-signed 4-way byte dot product with accumulate:
// c + sum_i a.u8[i] * b.s8[i]. The unsigned left operand lets a masked
// weight byte reach 128 (code 2 at bits 6..7) without wrapping.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ---------------------------------------------------------------- launchers
// Each returns a cudaError_t from the launch (cudaSuccess if nothing ran).

cudaError_t launch_quantize_q8K(const float* X, uint8_t* Xq, int64_t nblocks, cudaStream_t s);
cudaError_t launch_repack(const uint8_t* Wpq2, uint8_t* Wtq, int64_t rows, int64_t cols,
                          cudaStream_t s);
cudaError_t launch_unrepack(const uint8_t* Wtq, uint8_t* Wpq2, int64_t rows, int64_t cols,
                            cudaStream_t s);

// GEMV for 1..8 tokens. Returns cudaErrorNotSupported (without launching)
// when the activations of all tokens do not fit in shared memory.
cudaError_t launch_gemv(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                        int64_t rows, int64_t cols, int ntok, cudaStream_t s);
int64_t gemv_smem_bytes(int64_t cols, int ntok);
int gemv_max_tokens();

// Tensor-core path for any ntok >= 1 (used for ntok > gemv_max_tokens()).
cudaError_t launch_gemm_tc(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                           int64_t rows, int64_t cols, int64_t ntok, int* dev_status,
                           cudaStream_t s);

// Opt a kernel in to `bytes` of dynamic shared memory on the current device
// (cached per device and kernel).
cudaError_t ensure_dynamic_smem(const void* kernel, int bytes);

}  // namespace tq
