// tq_api.cu -- the C ABI declared in include/tq.h: argument checks, routing by
// token count, error reporting. Kernels live in the other files of csrc/.
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <unordered_map>
#include <utility>

#include "tq_internal.cuh"

namespace tq {
namespace {

thread_local int g_last_cuda_error = 0;

// Device-side status word: kernels that bound a wait set it when they give up.
__device__ int g_device_status = kDevOk;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
std::map<std::pair<int, const void*>, int> g_smem_optin;

bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return na > 0 && nb > 0 && x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

// What this library last enqueued on each stream, and, inside a stream
// capture, that kernel's graph node. A kernel of this library may read its
// weights (or all its inputs) before waiting for the kernel before it only
// when the host can prove what that kernel is: inside a capture whose one
// dependency is the node this library recorded for its own last kernel on the
// stream (so nothing else was captured between the two), and whose outputs
// miss the new kernel's inputs. Outside a capture the library cannot see
// other work on the stream (a caller's kernel between two calls could write
// the weights), so its kernels always wait first there.
enum LastOp { kOpOther = 0, kOpQuantize = 1, kOpMatmul = 2, kOpGemv = 3 };
constexpr int kMaxOuts = 5;
struct StreamLast {
  int op = kOpOther;
  unsigned long long capture_id = 0;   // inside a capture: its id and the
  cudaGraphNode_t node = nullptr;      // kernel's node (else 0, null)
  const void* out[kMaxOuts] = {};
  int64_t out_bytes[kMaxOuts] = {};
};
std::mutex g_stream_mu;
std::unordered_map<cudaStream_t, StreamLast> g_last_op;

void note_op(cudaStream_t s, int op) {
  StreamLast l;
  l.op = op;
  std::lock_guard<std::mutex> lk(g_stream_mu);
  g_last_op[s] = l;
}

// The single node the next captured operation on s will depend on; false when
// s is not capturing or depends on several nodes (or none).
bool capture_tail(cudaStream_t s, unsigned long long* id, cudaGraphNode_t* node) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  const cudaGraphNode_t* deps = nullptr;
  const cudaGraphEdgeData* edges = nullptr;
  size_t n = 0;
  if (cudaStreamGetCaptureInfo(s, &st, id, nullptr, &deps, &edges, &n) != cudaSuccess) {
    (void)cudaGetLastError();   // a failed query is no error of the caller's
    return false;
  }
  if (st != cudaStreamCaptureStatusActive || n != 1 || !deps) return false;
  *node = deps[0];
  return true;
}

// Called right after this library launched a kernel of kind `op` on s, with
// the ranges that kernel (or a kernel before it that may still be running)
// writes.
void note_kernel(cudaStream_t s, int op, const void* out0, int64_t bytes0,
                 const void* out1 = nullptr, int64_t bytes1 = 0, const void* out2 = nullptr,
                 int64_t bytes2 = 0) {
  StreamLast l;
  l.op = op;
  if (!capture_tail(s, &l.capture_id, &l.node)) {
    l.capture_id = 0;
    l.node = nullptr;
  }
  l.out[0] = out0;
  l.out_bytes[0] = bytes0;
  l.out[1] = out1;
  l.out_bytes[1] = bytes1;
  l.out[2] = out2;
  l.out_bytes[2] = bytes2;
  std::lock_guard<std::mutex> lk(g_stream_mu);
  g_last_op[s] = l;
}

// Like note_kernel, for a kernel that lets its successor start at its own
// start: the kernel before it (record prev, when proven) may then still run
// beside that successor, so prev's outputs join this kernel's.
void note_early_trigger_kernel(cudaStream_t s, int op, const StreamLast& prev, bool proven,
                               const void* out0, int64_t bytes0, const void* out1 = nullptr,
                               int64_t bytes1 = 0) {
  StreamLast l;
  l.op = op;
  if (!proven || !capture_tail(s, &l.capture_id, &l.node)) {
    l.capture_id = 0;
    l.node = nullptr;
  }
  l.out[0] = out0;
  l.out_bytes[0] = bytes0;
  l.out[1] = out1;
  l.out_bytes[1] = bytes1;
  int k = 2;
  for (int i = 0; i < kMaxOuts && proven; ++i)
    if (prev.out_bytes[i] > 0) {
      if (k == kMaxOuts) {   // no room: the successor must not be trusted
        l.node = nullptr;
        break;
      }
      l.out[k] = prev.out[i];
      l.out_bytes[k++] = prev.out_bytes[i];
    }
  std::lock_guard<std::mutex> lk(g_stream_mu);
  g_last_op[s] = l;
}

bool misses_outputs(const StreamLast& l, const void* p, int64_t n) {
  for (int i = 0; i < kMaxOuts; ++i)
    if (overlap(p, n, l.out[i], l.out_bytes[i])) return false;
  return true;
}

// The kernel enqueued just before on s is, provably, this library's last
// kernel there (see StreamLast); its record is returned in *l.
bool proven_predecessor(cudaStream_t s, StreamLast* l) {
  {
    std::lock_guard<std::mutex> lk(g_stream_mu);
    auto it = g_last_op.find(s);
    if (it == g_last_op.end()) return false;
    *l = it->second;
  }
  if (l->op == kOpOther || !l->node) return false;
  unsigned long long id = 0;
  cudaGraphNode_t node = nullptr;
  return capture_tail(s, &id, &node) && id == l->capture_id && node == l->node;
}

// The GEMV about to be enqueued on s may request its weights W before
// waiting for the kernel before it: that kernel is this library's and writes
// no part of W, and every kernel of this library that is recorded here lets
// its successor start only after its own wait (or at its end), so no older
// kernel can still be running, or else (the GEMV's staging kernel) its
// record also holds the outputs of the one kernel before it that can.
bool early_weights_ok(cudaStream_t s, const void* W, int64_t w_bytes) {
  StreamLast l;
  return proven_predecessor(s, &l) && misses_outputs(l, W, w_bytes);
}

// The GEMV about to be enqueued on s may read all its inputs (the activations
// in0 and the weights in1) before waiting: the kernel before it is this
// library's GEMV, which lets its successor start only after its own wait (so
// nothing older can still run), and none of its outputs overlaps them.
bool gemv_inputs_final(cudaStream_t s, const void* in0, int64_t bytes0, const void* in1,
                       int64_t bytes1) {
  StreamLast l;
  return proven_predecessor(s, &l) && l.op == kOpGemv && misses_outputs(l, in0, bytes0) &&
         misses_outputs(l, in1, bytes1);
}

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return TQ_ERR_CUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

cudaError_t device_status_ptr(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

int64_t q8K_bytes(int64_t ntok, int64_t cols) { return ntok * (cols / kQK) * kQ8KBytes; }

// With a workspace, tokens beyond this many go to the tensor cores (a token
// tile of 16, 32 or 64); without one the GEMV takes up to gemv_max_tokens().
// From 4 tokens up to it (and from 3072 columns) the workspace holds the
// mma.sync GEMV's activations, staged once instead of in every CTA.
constexpr int kWsGemvMaxTok = 8;

int64_t workspace_bytes(int64_t rows, int64_t cols, int64_t ntok) {
  if (rows <= 0 || cols <= 0) return 0;
  if (ntok <= kWsGemvMaxTok) return gemv_stage_bytes(cols, (int)ntok);
  return tc_workspace_bytes(cols, ntok);
}

// The staging kernel about to be enqueued on s: *proven when the kernel
// before it is provably this library's (record *prev), and then the staging
// kernel lets the GEMV start at once; the result says whether it may also
// read its input in (bytes n) before waiting (that kernel is a GEMV, which
// lets its successor start only after its own wait, and writes none of it).
bool stage_input_final(cudaStream_t s, const void* in, int64_t n, StreamLast* prev,
                       bool* proven) {
  *proven = proven_predecessor(s, prev);
  return *proven && prev->op == kOpGemv && misses_outputs(*prev, in, n);
}

int matmul_impl(const void* Wtq, const void* Xq, float* Y, int32_t* S, int64_t rows,
                int64_t cols, int64_t ntok, void* ws, int64_t ws_bytes, bool use_ws,
                void* stream) {
  if (rows < 0 || cols < 0 || ntok < 0 || cols % kQK != 0) return TQ_ERR_SHAPE;
  if (rows == 0 || ntok == 0) return TQ_OK;
  void* out = Y ? (void*)Y : (void*)S;
  if (!out) return TQ_ERR_NULL;
  const int64_t out_bytes = Y ? ntok * rows * 4 : ntok * rows * (cols / kGroup) * 4;
  if (!aligned4(out)) return TQ_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cols == 0) {
    if (Y) {
      note_op(s, kOpOther);
      cudaError_t e = cudaMemsetAsync(Y, 0, (size_t)out_bytes, s);
      if (e != cudaSuccess) return fail_cuda(e);
    }
    return TQ_OK;
  }
  if (!Wtq || !Xq) return TQ_ERR_NULL;
  if (!aligned16(Wtq) || !aligned16(Xq)) return TQ_ERR_ALIGN;
  if (overlap(out, out_bytes, Wtq, tq_repacked_bytes(rows, cols)) ||
      overlap(out, out_bytes, Xq, q8K_bytes(ntok, cols)))
    return TQ_ERR_ALIAS;
  const int64_t need = use_ws ? workspace_bytes(rows, cols, ntok) : 0;
  if (need > 0) {
    if (!ws) return TQ_ERR_NULL;
    if (!aligned16(ws)) return TQ_ERR_ALIGN;
    if (ws_bytes < need) return TQ_ERR_WORKSPACE;
    if (overlap(ws, need, out, out_bytes) || overlap(ws, need, Wtq, tq_repacked_bytes(rows, cols)) ||
        overlap(ws, need, Xq, q8K_bytes(ntok, cols)))
      return TQ_ERR_ALIAS;
  }

  const uint8_t* W = static_cast<const uint8_t*>(Wtq);
  const uint8_t* X = static_cast<const uint8_t*>(Xq);
  int* status = nullptr;
  cudaError_t e = device_status_ptr(&status);
  if (e != cudaSuccess) return fail_cuda(e);
  const int64_t w_bytes = tq_repacked_bytes(rows, cols);
  const bool gemv = ntok <= (use_ws ? kWsGemvMaxTok : gemv_max_tokens());
  if (gemv && need > 0 && gemv_stage_fits(cols, (int)ntok, false)) {
    // 4..8 tokens with a workspace: the activations staged once (see
    // tq_quantize_matmul), from the q8_K blocks
    uint8_t* region = static_cast<uint8_t*>(ws);
    StreamLast prev;
    bool proven = false;
    const bool x_final = stage_input_final(s, Xq, q8K_bytes(ntok, cols), &prev, &proven);
    note_op(s, kOpOther);
    e = launch_gemv_stage(nullptr, X, nullptr, region, cols, (int)ntok, x_final, proven, s);
    if (e != cudaSuccess) return fail_cuda(e);
    note_early_trigger_kernel(s, kOpQuantize, prev, proven, region, need);
    const bool early_w = early_weights_ok(s, Wtq, w_bytes);
    note_op(s, kOpOther);
    e = launch_gemv(W, X, Y, S, rows, cols, (int)ntok, status, early_w, false, s, nullptr, nullptr,
                    region);
    if (e != cudaSuccess) return fail_cuda(e);
    note_kernel(s, kOpGemv, out, out_bytes);
    return TQ_OK;
  }
  const bool early = early_weights_ok(s, Wtq, w_bytes);
  const bool inputs_final =
      gemv && gemv_inputs_final(s, Xq, q8K_bytes(ntok, cols), Wtq, w_bytes);
  note_op(s, kOpOther);
  if (gemv) {
    e = launch_gemv(W, X, Y, S, rows, cols, (int)ntok, status, early, inputs_final, s);
    if (e == cudaSuccess) {
      note_kernel(s, kOpGemv, out, out_bytes);
      return TQ_OK;
    }
    if (e != cudaErrorNotSupported) return fail_cuda(e);
    // activations too large for the GEMV's shared memory: tensor-core path
  }
  // up to kWsGemvMaxTok tokens a workspace is sized for the staged GEMV, not
  // for the tensor cores
  if (need > 0 && ntok > kWsGemvMaxTok)
    e = launch_gemm_tc_ws(W, X, Y, S, rows, cols, ntok, static_cast<uint8_t*>(ws), status, s);
  else
    e = launch_gemm_tc(W, X, Y, S, rows, cols, ntok, status, s);
  if (e != cudaSuccess) return fail_cuda(e);
  note_kernel(s, kOpMatmul, out, out_bytes, ws, need);
  return TQ_OK;
}

}  // namespace

void record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

int ws_gemv_max_tokens() { return kWsGemvMaxTok; }

namespace {
std::atomic<int64_t> g_debug_stall_ns{0};
}  // namespace

int64_t take_debug_stall() {
  if (g_debug_stall_ns.load(std::memory_order_relaxed) == 0) return 0;   // the usual case
  return g_debug_stall_ns.exchange(0);
}

cudaError_t ensure_dynamic_smem(const void* kernel, int bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(dev, kernel);
  auto it = g_smem_optin.find(key);
  if (it != g_smem_optin.end() && it->second >= bytes) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (bytes > optin) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  g_smem_optin[key] = optin;
  return cudaSuccess;
}

cudaError_t device_limits(DeviceLimits* out) {
  static DeviceLimits limits[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceLimits& l = limits[dev];
  if (l.sms == 0) {
    int optin = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    l.optin_smem = optin;
    l.sms = sms;
  }
  *out = l;
  return cudaSuccess;
}

cudaError_t resident_ctas(const void* kernel, int threads, size_t smem, int* out) {
  static std::map<std::tuple<int, const void*, int, size_t>, int> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(dev, kernel, threads, smem);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  cache[key] = n;
  *out = n;
  return cudaSuccess;
}

}  // namespace tq

using namespace tq;

extern "C" {

int tq_quantize_q8K(const float* X, void* Xq, int64_t ntok, int64_t cols, void* stream) {
  if (ntok < 0 || cols < 0 || cols % kQK != 0) return TQ_ERR_SHAPE;
  if (ntok == 0 || cols == 0) return TQ_OK;
  if (!X || !Xq) return TQ_ERR_NULL;
  if (!aligned16(X) || !aligned16(Xq)) return TQ_ERR_ALIGN;
  if (overlap(X, ntok * cols * 4, Xq, q8K_bytes(ntok, cols))) return TQ_ERR_ALIAS;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  note_op(s, kOpOther);
  cudaError_t e = launch_quantize_q8K(X, static_cast<uint8_t*>(Xq), ntok * (cols / kQK), s);
  if (e != cudaSuccess) return fail_cuda(e);
  note_kernel(s, kOpQuantize, Xq, q8K_bytes(ntok, cols));
  return TQ_OK;
}

int64_t tq_repacked_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % kGroup != 0) return -1;
  return (rows + kTileRows - 1) / kTileRows * (cols / kGroup) * kTileBytes;
}

int tq_repack(const void* Wpq2, void* Wtq, int64_t rows, int64_t cols, void* stream) {
  if (rows < 0 || cols < 0 || cols % kGroup != 0) return TQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return TQ_OK;
  if (!Wpq2 || !Wtq) return TQ_ERR_NULL;
  if (!aligned16(Wpq2) || !aligned16(Wtq)) return TQ_ERR_ALIGN;
  if (overlap(Wpq2, rows * (cols / kGroup) * kPq2Bytes, Wtq, tq_repacked_bytes(rows, cols)))
    return TQ_ERR_ALIAS;
  note_op(static_cast<cudaStream_t>(stream), kOpOther);
  cudaError_t e = launch_repack(static_cast<const uint8_t*>(Wpq2), static_cast<uint8_t*>(Wtq),
                                rows, cols, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TQ_OK : fail_cuda(e);
}

int64_t tq_ptq1_0_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % kGroup != 0) return -1;
  return rows * (cols / kGroup) * kPtq1Bytes;
}

int tq_repack_ptq1_0(const void* Wpt, void* Wtq, int64_t rows, int64_t cols, void* stream) {
  if (rows < 0 || cols < 0 || cols % kGroup != 0) return TQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return TQ_OK;
  if (!Wpt || !Wtq) return TQ_ERR_NULL;
  if (!aligned16(Wpt) || !aligned16(Wtq)) return TQ_ERR_ALIGN;
  if (overlap(Wpt, tq_ptq1_0_bytes(rows, cols), Wtq, tq_repacked_bytes(rows, cols)))
    return TQ_ERR_ALIAS;
  note_op(static_cast<cudaStream_t>(stream), kOpOther);
  cudaError_t e = launch_repack_ptq1(static_cast<const uint8_t*>(Wpt), static_cast<uint8_t*>(Wtq),
                                     rows, cols, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TQ_OK : fail_cuda(e);
}

int64_t tq_ptq1_0_stream_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % kGroup != 0) return -1;
  return (rows + kTileRows - 1) / kTileRows * (cols / kGroup) * kTq1TileBytes;
}

int tq_repack_ptq1_0_stream(const void* Wpt, void* Wt1, int64_t rows, int64_t cols,
                            void* stream) {
  if (rows < 0 || cols < 0 || cols % kGroup != 0) return TQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return TQ_OK;
  if (!Wpt || !Wt1) return TQ_ERR_NULL;
  if (!aligned16(Wpt) || !aligned16(Wt1)) return TQ_ERR_ALIGN;
  if (overlap(Wpt, tq_ptq1_0_bytes(rows, cols), Wt1, tq_ptq1_0_stream_bytes(rows, cols)))
    return TQ_ERR_ALIAS;
  note_op(static_cast<cudaStream_t>(stream), kOpOther);
  cudaError_t e = launch_repack_ptq1_stream(static_cast<const uint8_t*>(Wpt),
                                            static_cast<uint8_t*>(Wt1), rows, cols,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TQ_OK : fail_cuda(e);
}

int tq_unrepack(const void* Wtq, void* Wpq2, int64_t rows, int64_t cols, void* stream) {
  if (rows < 0 || cols < 0 || cols % kGroup != 0) return TQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return TQ_OK;
  if (!Wpq2 || !Wtq) return TQ_ERR_NULL;
  if (!aligned16(Wpq2) || !aligned16(Wtq)) return TQ_ERR_ALIGN;
  if (overlap(Wpq2, rows * (cols / kGroup) * kPq2Bytes, Wtq, tq_repacked_bytes(rows, cols)))
    return TQ_ERR_ALIAS;
  note_op(static_cast<cudaStream_t>(stream), kOpOther);
  cudaError_t e = launch_unrepack(static_cast<const uint8_t*>(Wtq), static_cast<uint8_t*>(Wpq2),
                                  rows, cols, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TQ_OK : fail_cuda(e);
}

int tq_matmul(const void* Wtq, const void* Xq, float* Y, int64_t rows, int64_t cols,
              int64_t ntok, void* stream) {
  return matmul_impl(Wtq, Xq, Y, nullptr, rows, cols, ntok, nullptr, 0, false, stream);
}

int tq_matmul_groupsums(const void* Wtq, const void* Xq, int32_t* S, int64_t rows,
                        int64_t cols, int64_t ntok, void* stream) {
  return matmul_impl(Wtq, Xq, nullptr, S, rows, cols, ntok, nullptr, 0, false, stream);
}

namespace {
int matmul_ptq1_stream(const void* Wt1, const void* Xq, float* Y, int32_t* S, int64_t rows,
                       int64_t cols, int64_t ntok, void* stream) {
  if (rows < 0 || cols < 0 || ntok < 0 || cols % kQK != 0) return TQ_ERR_SHAPE;
  if (rows == 0 || ntok == 0) return TQ_OK;
  void* out = Y ? (void*)Y : (void*)S;
  if (!out) return TQ_ERR_NULL;
  const int64_t out_bytes = Y ? ntok * rows * 4 : ntok * rows * (cols / kGroup) * 4;
  if (!aligned4(out)) return TQ_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cols == 0) {
    if (Y) {
      note_op(s, kOpOther);
      cudaError_t e = cudaMemsetAsync(Y, 0, (size_t)out_bytes, s);
      if (e != cudaSuccess) return fail_cuda(e);
    }
    return TQ_OK;
  }
  if (!Wt1 || !Xq) return TQ_ERR_NULL;
  if (!aligned16(Wt1) || !aligned16(Xq)) return TQ_ERR_ALIGN;
  const int64_t w_bytes = tq_ptq1_0_stream_bytes(rows, cols);
  if (overlap(out, out_bytes, Wt1, w_bytes) || overlap(out, out_bytes, Xq, q8K_bytes(ntok, cols)))
    return TQ_ERR_ALIAS;
  if (ntok > 0x7fffffff) return TQ_ERR_SHAPE;
  int* status = nullptr;
  cudaError_t e = device_status_ptr(&status);
  if (e != cudaSuccess) return fail_cuda(e);
  const bool early = early_weights_ok(s, Wt1, w_bytes);
  note_op(s, kOpOther);
  e = launch_gemv_ptq1(static_cast<const uint8_t*>(Wt1), static_cast<const uint8_t*>(Xq), Y, S,
                       rows, cols, (int)ntok, status, early, s);
  if (e != cudaSuccess) return fail_cuda(e);
  note_kernel(s, kOpMatmul, out, out_bytes);
  return TQ_OK;
}
}  // namespace

int tq_matmul_ptq1_0_stream(const void* Wt1, const void* Xq, float* Y, int64_t rows, int64_t cols,
                            int64_t ntok, void* stream) {
  return matmul_ptq1_stream(Wt1, Xq, Y, nullptr, rows, cols, ntok, stream);
}

int tq_matmul_ptq1_0_stream_groupsums(const void* Wt1, const void* Xq, int32_t* S, int64_t rows,
                                      int64_t cols, int64_t ntok, void* stream) {
  return matmul_ptq1_stream(Wt1, Xq, nullptr, S, rows, cols, ntok, stream);
}

int64_t tq_matmul_workspace_bytes(int64_t rows, int64_t cols, int64_t ntok) {
  if (rows < 0 || cols < 0 || ntok < 0 || cols % kQK != 0) return -1;
  return workspace_bytes(rows, cols, ntok);
}

int tq_matmul_ws(const void* Wtq, const void* Xq, float* Y, int64_t rows, int64_t cols,
                 int64_t ntok, void* workspace, int64_t workspace_bytes, void* stream) {
  return matmul_impl(Wtq, Xq, Y, nullptr, rows, cols, ntok, workspace, workspace_bytes, true,
                     stream);
}

int tq_matmul_groupsums_ws(const void* Wtq, const void* Xq, int32_t* S, int64_t rows,
                           int64_t cols, int64_t ntok, void* workspace, int64_t workspace_bytes,
                           void* stream) {
  return matmul_impl(Wtq, Xq, nullptr, S, rows, cols, ntok, workspace, workspace_bytes, true,
                     stream);
}

int tq_quantize_matmul(const void* Wtq, const float* X, void* Xq, float* Y, int64_t rows,
                       int64_t cols, int64_t ntok, void* workspace, int64_t workspace_bytes,
                       void* stream) {
  if (rows < 0 || cols < 0 || ntok < 0 || cols % kQK != 0) return TQ_ERR_SHAPE;
  if (rows == 0 || ntok == 0) return TQ_OK;
  if (cols == 0) return tq_matmul_ws(Wtq, Xq, Y, rows, cols, ntok, workspace, workspace_bytes, stream);
  // every check of the calls below, before anything is enqueued
  if (!X || !Xq || !Y || !Wtq) return TQ_ERR_NULL;
  if (!aligned16(X) || !aligned16(Xq) || !aligned16(Wtq) || !aligned4(Y)) return TQ_ERR_ALIGN;
  const int64_t x_bytes = ntok * cols * 4, y_bytes = ntok * rows * 4;
  const int64_t xq_bytes = q8K_bytes(ntok, cols), w_bytes = tq_repacked_bytes(rows, cols);
  if (overlap(X, x_bytes, Xq, xq_bytes) || overlap(Y, y_bytes, Wtq, w_bytes) ||
      overlap(Y, y_bytes, Xq, xq_bytes) || overlap(Y, y_bytes, X, x_bytes) ||
      overlap(Xq, xq_bytes, Wtq, w_bytes))
    return TQ_ERR_ALIAS;
  const int64_t need = tq::workspace_bytes(rows, cols, ntok);
  if (need > 0) {
    if (!workspace) return TQ_ERR_NULL;
    if (!aligned16(workspace)) return TQ_ERR_ALIGN;
    if (workspace_bytes < need) return TQ_ERR_WORKSPACE;
    if (overlap(workspace, need, Y, y_bytes) || overlap(workspace, need, Wtq, w_bytes) ||
        overlap(workspace, need, Xq, xq_bytes) || overlap(workspace, need, X, x_bytes))
      return TQ_ERR_ALIAS;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ntok <= kWsGemvMaxTok) {
    int* status = nullptr;
    cudaError_t e = device_status_ptr(&status);
    if (e != cudaSuccess) return fail_cuda(e);
    if (need > 0 && gemv_stage_fits(cols, (int)ntok, true)) {
      // 4..8 tokens: one kernel quantizes X, writes Xq and stages the GEMV's
      // activations in the workspace; the GEMV loads them
      uint8_t* region = static_cast<uint8_t*>(workspace);
      StreamLast prev;
      bool proven = false;
      const bool x_final = stage_input_final(s, X, x_bytes, &prev, &proven);
      note_op(s, kOpOther);
      e = launch_gemv_stage(X, nullptr, static_cast<uint8_t*>(Xq), region, cols, (int)ntok, x_final,
                            proven, s);
      if (e != cudaSuccess) return fail_cuda(e);
      note_early_trigger_kernel(s, kOpQuantize, prev, proven, Xq, xq_bytes, region, need);
      const bool early_w = early_weights_ok(s, Wtq, w_bytes);
      note_op(s, kOpOther);
      e = launch_gemv(static_cast<const uint8_t*>(Wtq), nullptr, Y, nullptr, rows, cols, (int)ntok,
                      status, early_w, false, s, nullptr, nullptr, region);
      if (e != cudaSuccess) return fail_cuda(e);
      note_kernel(s, kOpGemv, Y, y_bytes);
      return TQ_OK;
    }
    const bool early = early_weights_ok(s, Wtq, w_bytes);
    const bool inputs_final = gemv_inputs_final(s, X, x_bytes, Wtq, w_bytes);
    note_op(s, kOpOther);
    e = launch_gemv(static_cast<const uint8_t*>(Wtq), nullptr, Y, nullptr, rows, cols, (int)ntok,
                    status, early, inputs_final, s, X, static_cast<uint8_t*>(Xq));
    if (e == cudaSuccess) {
      note_kernel(s, kOpGemv, Y, y_bytes, Xq, xq_bytes);
      return TQ_OK;
    }
    if (e != cudaErrorNotSupported) {
      note_op(s, kOpOther);
      return fail_cuda(e);
    }
    // activations too large for the GEMV's shared memory: the separate calls
  }
  if (need > 0 && ntok > kWsGemvMaxTok) {
    // one kernel quantizes and packs the workspace, then the tensor-core kernel
    int* status = nullptr;
    cudaError_t e = device_status_ptr(&status);
    if (e != cudaSuccess) return fail_cuda(e);
    note_op(s, kOpOther);
    e = launch_quantize_gemm_tc_ws(X, static_cast<uint8_t*>(Xq), static_cast<const uint8_t*>(Wtq),
                                   Y, rows, cols, ntok, static_cast<uint8_t*>(workspace), status, s);
    if (e != cudaSuccess) return fail_cuda(e);
    note_kernel(s, kOpMatmul, Y, y_bytes, Xq, xq_bytes, workspace, need);
    return TQ_OK;
  }
  int rc = tq_quantize_q8K(X, Xq, ntok, cols, stream);
  if (rc != TQ_OK) return rc;
  return tq_matmul_ws(Wtq, Xq, Y, rows, cols, ntok, workspace, workspace_bytes, stream);
}

int tq_matmul_host(const void* Wtq, const float* X_host, float* X, void* Xq, float* Y,
                   float* Y_host, int64_t rows, int64_t cols, int64_t ntok, void* workspace,
                   int64_t workspace_bytes, void* stream) {
  if (rows < 0 || cols < 0 || ntok < 0 || cols % kQK != 0) return TQ_ERR_SHAPE;
  if (rows == 0 || ntok == 0) return TQ_OK;
  // every check of the calls below, before anything is enqueued
  if (!X_host || !Y_host || !X || !Xq || !Y || !Wtq) return TQ_ERR_NULL;
  if (!aligned16(X) || !aligned16(Xq) || !aligned16(Wtq) || !aligned4(Y)) return TQ_ERR_ALIGN;
  const int64_t x_bytes = ntok * cols * 4, y_bytes = ntok * rows * 4;
  const int64_t xq_bytes = q8K_bytes(ntok, cols), w_bytes = tq_repacked_bytes(rows, cols);
  if (overlap(X, x_bytes, Xq, xq_bytes) || overlap(Y, y_bytes, Wtq, w_bytes) ||
      overlap(Y, y_bytes, Xq, xq_bytes) || overlap(Y, y_bytes, X, x_bytes))
    return TQ_ERR_ALIAS;
  const int64_t need = tq::workspace_bytes(rows, cols, ntok);
  if (need > 0) {
    if (!workspace) return TQ_ERR_NULL;
    if (!aligned16(workspace)) return TQ_ERR_ALIGN;
    if (workspace_bytes < need) return TQ_ERR_WORKSPACE;
    if (overlap(workspace, need, Y, y_bytes) || overlap(workspace, need, Wtq, w_bytes) ||
        overlap(workspace, need, Xq, xq_bytes))
      return TQ_ERR_ALIAS;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (x_bytes > 0) {
    const cudaError_t e = cudaMemcpyAsync(X, X_host, (size_t)x_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  const int rc = tq_quantize_matmul(Wtq, X, Xq, Y, rows, cols, ntok, workspace, workspace_bytes,
                                    stream);
  if (rc != TQ_OK) return rc;
  const cudaError_t e = cudaMemcpyAsync(Y_host, Y, (size_t)y_bytes, cudaMemcpyDeviceToHost, s);
  note_op(s, kOpOther);
  return e == cudaSuccess ? TQ_OK : fail_cuda(e);
}

const char* tq_strerror(int code) {
  switch (code) {
    case TQ_OK: return "ok";
    case TQ_ERR_SHAPE: return "bad shape (cols must be a multiple of 256, sizes >= 0)";
    case TQ_ERR_NULL: return "null pointer";
    case TQ_ERR_ALIGN: return "misaligned buffer";
    case TQ_ERR_CUDA: return "CUDA error (see tq_last_cuda_error)";
    case TQ_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case TQ_ERR_ALIAS: return "output buffer overlaps an input";
    case TQ_ERR_WORKSPACE: return "workspace smaller than tq_matmul_workspace_bytes";
    default: return "unknown error";
  }
}

int tq_last_cuda_error(void) { return g_last_cuda_error; }

int tq_device_status(void) {
  int* p = nullptr;
  cudaError_t e = device_status_ptr(&p);
  if (e != cudaSuccess) return fail_cuda(e);
  int v = 0;
  e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  if (v != kDevOk) {
    const int zero = kDevOk;
    e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return v == kDevTimeout ? TQ_ERR_TIMEOUT : TQ_OK;
}

int tq_probe_read_sum(const void* buf, int64_t bytes, uint32_t* out, int early, void* stream) {
  if (bytes < 0 || bytes % 16 != 0) return TQ_ERR_SHAPE;
  if (!out) return TQ_ERR_NULL;
  if (bytes == 0) return TQ_OK;
  if (!buf) return TQ_ERR_NULL;
  if (!aligned16(buf) || !aligned4(out)) return TQ_ERR_ALIGN;
  if (overlap(buf, bytes, out, 4)) return TQ_ERR_ALIAS;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  note_op(s, kOpOther);
  const cudaError_t e = launch_read_sum(buf, bytes, out, early != 0, s);
  return e == cudaSuccess ? TQ_OK : fail_cuda(e);
}

int tq_debug_stall_next_launch(int64_t wait_limit_ns) {
  if (wait_limit_ns < 0) return TQ_ERR_SHAPE;
  g_debug_stall_ns.store(wait_limit_ns);
  return TQ_OK;
}

const char* tq_version(void) { return "0.2.0"; }

}  // extern "C"
