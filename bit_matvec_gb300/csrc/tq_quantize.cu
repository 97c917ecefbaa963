// tq_quantize.cu -- f32 activations -> q8_K blocks on the GPU.
//
// q8_K (ciot README): 256 int8 values, one f32 scale and 16 partial sums per
// block. Scale: the block's largest magnitude over 127, symmetric ("Quantization
// and the CPU", section "Quantizing the weights and activations"); a block whose
// absolute max is 127 quantizes with scale 1 (ternary post, "stuff that went
// wrong"). Rounding to nearest, ties to even.
//
// One warp per block (q8K_warp in tq_internal.cuh): each lane holds 8
// consecutive values (two float4 loads), the absolute max is a warp max over
// the float bit patterns, and each partial sum of 16 values is the sum of two
// neighbouring lanes.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kWarpsPerCta = 8;

__global__ void __launch_bounds__(kWarpsPerCta * 32)
quantize_q8K_kernel(const float* __restrict__ X, uint8_t* __restrict__ Xq, int64_t nblocks) {
  // Launched as a programmatic dependent: start early, but touch no memory
  // before the previous kernel in the stream has finished; let the next kernel
  // start only after that wait, so that when it starts this kernel is the only
  // one before it that can still run (the matmuls rely on that to request
  // their weights early).
  pdl_wait_primary();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t blk = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (blk >= nblocks) return;  // whole warp leaves together

  const float4* src = reinterpret_cast<const float4*>(X + blk * kQK) + 2 * lane;
  uint32_t w0, w1;
  int s8;
  float d;
  q8K_warp(__ldg(src), __ldg(src + 1), w0, w1, s8, d);
  q8K_store(Xq + blk * kQ8KBytes, lane, w0, w1, s8, d);
}

}  // namespace

cudaError_t launch_quantize_q8K(const float* X, uint8_t* Xq, int64_t nblocks, cudaStream_t s) {
  if (nblocks <= 0) return cudaSuccess;
  const int64_t grid = (nblocks + kWarpsPerCta - 1) / kWarpsPerCta;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  return launch_pdl(quantize_q8K_kernel, dim3((unsigned)grid), dim3(kWarpsPerCta * 32), 0, s, X,
                    Xq, nblocks);
}

}  // namespace tq
