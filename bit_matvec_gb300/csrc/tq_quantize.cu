// tq_quantize.cu -- f32 activations -> q8_K blocks on the GPU.
//
// q8_K (ciot README): 256 int8 values, one f32 scale and 16 partial sums per
// block. Scale: the block's largest magnitude over 127, symmetric ("Quantization
// and the CPU", section "Quantizing the weights and activations"); a block whose
// absolute max is 127 quantizes with scale 1 (ternary post, "stuff that went
// wrong"). Rounding to nearest, ties to even.
//
// One warp per block: each lane holds 8 consecutive values (two float4 loads),
// the absolute max is a warp max over the float bit patterns (non-negative
// floats order like their bits), and each partial sum of 16 values is the sum
// of two neighbouring lanes.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ uint32_t pack4_s8(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xFF) | ((uint32_t)(b & 0xFF) << 8) | ((uint32_t)(c & 0xFF) << 16) |
         ((uint32_t)(d & 0xFF) << 24);
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
quantize_q8K_kernel(const float* __restrict__ X, uint8_t* __restrict__ Xq, int64_t nblocks) {
  // Launched as a programmatic dependent: start early, but touch no memory
  // before the previous kernel in the stream has finished.
  pdl_launch_dependents();
  pdl_wait_primary();
  const int lane = threadIdx.x & 31;
  const int64_t blk = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (blk >= nblocks) return;  // whole warp leaves together

  const float4* src = reinterpret_cast<const float4*>(X + blk * kQK) + 2 * lane;
  const float4 a = __ldg(src), b = __ldg(src + 1);
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};

  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));

  uint8_t* out = Xq + blk * kQ8KBytes;
  uint32_t* qs_out = reinterpret_cast<uint32_t*>(out + kQ8KQsOffset) + 2 * lane;
  int16_t* bsums_out = reinterpret_cast<int16_t*>(out + kQ8KBsumsOffset);

  if (amax == 0.0f) {  // uniform across the warp
    qs_out[0] = 0u;
    qs_out[1] = 0u;
    if ((lane & 1) == 0) bsums_out[lane >> 1] = 0;
    if (lane == 0) *reinterpret_cast<float*>(out) = 0.0f;
    return;
  }

  const float iscale = __fdiv_rn(127.0f, amax);
  int q[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int qi = __float2int_rn(__fmul_rn(v[i], iscale));
    qi = max(-127, min(127, qi));
    q[i] = qi;
    sum += qi;
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);

  qs_out[0] = pack4_s8(q[0], q[1], q[2], q[3]);
  qs_out[1] = pack4_s8(q[4], q[5], q[6], q[7]);
  if ((lane & 1) == 0) bsums_out[lane >> 1] = (int16_t)sum;
  if (lane == 0) *reinterpret_cast<float*>(out) = __fdiv_rn(amax, 127.0f);
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
