// tq_probe.cu -- the memory-read ceiling probe behind the GEMV's roofline.
//
// The ternary post measures its machine's DRAM read ceiling before judging
// its kernels against it ("the ceiling": a sum over a large buffer, one
// thread and then several). This is the GB300 counterpart: a plain streaming
// sum of a buffer's 32-bit words with 128-bit loads, eight loads in flight
// per thread, four CTAs of 256 threads per SM, and no other work; the rate it
// reaches on a buffer of the decode matrix's size is the most any kernel that
// only reads that many bytes can expect.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 4;
constexpr int kProbeInFlight = 8;

__device__ __forceinline__ uint32_t add4(uint4 v) { return v.x + v.y + v.z + v.w; }

__global__ void __launch_bounds__(kProbeThreads) read_sum_kernel(const uint4* __restrict__ p,
                                                                 int64_t n16, uint32_t* out,
                                                                 int early) {
  // Launched as a programmatic dependent: with `early` the loads start before
  // the previous kernel in the stream has finished (it must not write p).
  if (!early) pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (kProbeInFlight - 1) * stride < n16; i += kProbeInFlight * stride) {
    uint4 v[kProbeInFlight];
#pragma unroll
    for (int u = 0; u < kProbeInFlight; ++u) v[u] = ldg_stream_v4(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < kProbeInFlight; ++u) acc += add4(v[u]);
  }
  for (; i < n16; i += stride) acc += add4(ldg_stream_v4(p + i));
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (early) pdl_wait_primary();   // before the store: out may be the previous kernel's
  if ((threadIdx.x & 31) == 0) atomicAdd(out, acc);
}

}  // namespace

cudaError_t launch_read_sum(const void* buf, int64_t bytes, uint32_t* out, bool early,
                            cudaStream_t s) {
  DeviceLimits lim;
  cudaError_t e = device_limits(&lim);
  if (e != cudaSuccess) return e;
  return launch_pdl(read_sum_kernel, dim3(lim.sms * kProbeCtasPerSm), dim3(kProbeThreads), 0, s,
                    static_cast<const uint4*>(buf), bytes / 16, out, early ? 1 : 0);
}

}  // namespace tq
