// tq_static_ws.cu -- tq_matmul_static_ws: the workspace form of the matmul
// with its workspace in a fixed device array of this library instead of a
// buffer the caller allocates.
//
// Some callers cannot allocate device memory at the point where they run the
// matmul: a plugin handed only input and output pointers by a host
// application that owns all device memory, an engine that forbids allocation
// after start-up because cudaMalloc can synchronize the device and stall
// other work, or code under a caching allocator whose pool must not be
// bypassed. They can still get the faster workspace path through this entry.
//
// The array below is the workspace. Every call shares it and it keeps the
// last call's contents; nothing in it has to start at zero, because the
// activation pre-pass writes every byte the tensor-core kernel reads before
// that kernel reads it. Two calls whose kernels overlap on the GPU (other
// streams, other host threads) race on it; callers must order them.
#include <mutex>

#include "tq_internal.cuh"

namespace tq {
namespace {

// The device array. In host code this name is only a host-side stand-in for
// the symbol: its device address comes from cudaGetSymbolAddress, once per
// device, with that device current.
static __device__ __align__(256) uint8_t g_static_ws[TQ_STATIC_WS_BYTES];

constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxStaticDevices] = {};

// Device address of g_static_ws on the current device, looked up on the first
// call there (which may also load this file's module onto that device).
cudaError_t static_ws_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxStaticDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace tq

extern "C" int tq_matmul_static_ws(const void* Wtq, const void* Xq, float* Y, int64_t rows,
                                   int64_t cols, int64_t ntok, void* stream) {
  if (rows < 0 || cols < 0 || ntok < 0 || cols % TQ_QK_K != 0) return TQ_ERR_SHAPE;
  // Beyond these, the tensor-core path's workspace (at least 4 KB per 128
  // columns, and 16 KB per 64 tokens and 128 columns) exceeds the array;
  // rejecting them first also keeps the size product below from overflowing.
  constexpr int64_t kMaxFactor = TQ_STATIC_WS_BYTES / 4096;
  if (ntok > tq::ws_gemv_max_tokens() && cols > 0 &&
      (cols / TQ_GROUP > kMaxFactor || ntok / 64 > kMaxFactor))
    return TQ_ERR_WORKSPACE;
  const int64_t need = tq_matmul_workspace_bytes(rows, cols, ntok);
  if (need < 0) return TQ_ERR_SHAPE;
  if (need > TQ_STATIC_WS_BYTES) return TQ_ERR_WORKSPACE;
  void* ws = nullptr;
  const cudaError_t e = tq::static_ws_ptr(&ws);
  if (e != cudaSuccess) {
    tq::record_cuda_error(e);
    return TQ_ERR_CUDA;
  }
  return tq_matmul_ws(Wtq, Xq, Y, rows, cols, ntok, ws, TQ_STATIC_WS_BYTES, stream);
}
