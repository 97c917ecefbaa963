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
constexpr int kPtq1Bytes = TQ_PTQ1_0_BYTES;
constexpr int kQ8KBytes = TQ_Q8K_BYTES;
constexpr int kTileRows = TQ_TILE_ROWS;  // rows per tile of the tq layout
constexpr int kTileBytes = TQ_TILE_BYTES;
constexpr int kTileCodeBytes = 1024;     // code bytes per tile; fp16 scales follow
// ptq1_0 stream layout: the 28-byte ptq1_0 blocks of 32 rows and one group,
// row after row (row l of the tile at byte 28 l)
constexpr int kTq1TileBytes = kTileRows * TQ_PTQ1_0_BYTES;   // 896
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

// ---------------------------------------------------------------- mbarrier / bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbarrier_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbarrier_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One bounded poll: the thread may sleep in hardware up to `hint_ns` for the
// phase to complete (it wakes as soon as it does), so waiting costs no issue
// slots.
__device__ __forceinline__ bool mbarrier_try_wait(uint32_t bar, uint32_t parity,
                                                  uint32_t hint_ns = 20000u) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking check that phase `parity` of an mbarrier has completed: cheaper
// than a suspending try_wait when the phase is usually complete already.
__device__ __forceinline__ bool mbarrier_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with acquire at cluster scope: for barriers that threads of the
// other CTA of a cluster arrive on.
__device__ __forceinline__ bool mbarrier_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbarrier_wait_bounded at cluster scope.
__device__ __forceinline__ bool mbarrier_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                              uint64_t limit_ns) {
  if (mbarrier_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if (mbarrier_try_wait_cluster(bar, parity)) return true;
    if ((it & 15u) == 15u && global_timer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns` of global
// time (checked every 16 polls, with a cap of 2^28 polls). Returns false on
// giving up; the caller records the failure and stops using the barrier.
__device__ __forceinline__ bool mbarrier_wait_bounded(uint32_t bar, uint32_t parity,
                                                      uint64_t limit_ns) {
  if (mbarrier_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if (mbarrier_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && global_timer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// Arm an mbarrier for `bytes` of incoming bulk-copy data (one arrival).
__device__ __forceinline__ void mbarrier_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// L2 policy for data every CTA of a launch reads: keep it.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy for data read once per launch: evict it first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared (TMA), completion counted on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Plain arrival on an mbarrier (release semantics at CTA scope).
__device__ __forceinline__ void mbarrier_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barrier for a subset of the CTA's warps (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- launchers
// Each returns a cudaError_t from the launch (cudaSuccess if nothing ran).

__device__ __forceinline__ uint32_t pack4_s8(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xFF) | ((uint32_t)(b & 0xFF) << 8) | ((uint32_t)(c & 0xFF) << 16) |
         ((uint32_t)(d & 0xFF) << 24);
}

// One warp quantizes one q8_K block of 256 activations; lane l holds values
// 8l .. 8l + 7 in (a, b). Scale: the block's largest magnitude over 127
// (the absolute max as a warp max over float bit patterns, which order like
// non-negative floats); q = round-to-nearest-even(x * (127 / amax)) clamped to
// +-127, with IEEE division and no contraction; an all-zero block gives zeros.
// Out: this lane's 8 values packed as int8 (w0, w1), their sum s8, and the
// block scale d (the same on every lane). The quantizer kernel and the fused
// GEMV staging both use it, so their q8_K bytes are identical.
__device__ __forceinline__ void q8K_warp(const float4 a, const float4 b, uint32_t& w0,
                                         uint32_t& w1, int& s8, float& d) {
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
  if (amax == 0.0f) {   // uniform across the warp
    w0 = w1 = 0u;
    s8 = 0;
    d = 0.0f;
    return;
  }
  const float iscale = __fdiv_rn(127.0f, amax);
  int q[8];
  s8 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int qi = __float2int_rn(__fmul_rn(v[i], iscale));
    qi = max(-127, min(127, qi));
    q[i] = qi;
    s8 += qi;
  }
  w0 = pack4_s8(q[0], q[1], q[2], q[3]);
  w1 = pack4_s8(q[4], q[5], q[6], q[7]);
  d = __fdiv_rn(amax, 127.0f);
}

// Stores one lane's share of a q8_K block quantized by q8K_warp (the warp
// writes the whole 292-byte block at blk).
__device__ __forceinline__ void q8K_store(uint8_t* blk, int lane, uint32_t w0, uint32_t w1, int s8,
                                          float d) {
  const int s16 = s8 + __shfl_xor_sync(0xffffffffu, s8, 1);   // 16 values: lanes 2i, 2i + 1
  uint32_t* qs = reinterpret_cast<uint32_t*>(blk + kQ8KQsOffset) + 2 * lane;
  qs[0] = w0;
  qs[1] = w1;
  if ((lane & 1) == 0) reinterpret_cast<int16_t*>(blk + kQ8KBsumsOffset)[lane >> 1] = (int16_t)s16;
  if (lane == 0) *reinterpret_cast<float*>(blk) = d;
}

cudaError_t launch_quantize_q8K(const float* X, uint8_t* Xq, int64_t nblocks, cudaStream_t s);
cudaError_t launch_repack(const uint8_t* Wpq2, uint8_t* Wtq, int64_t rows, int64_t cols,
                          cudaStream_t s);
cudaError_t launch_unrepack(const uint8_t* Wtq, uint8_t* Wpq2, int64_t rows, int64_t cols,
                            cudaStream_t s);
cudaError_t launch_repack_ptq1(const uint8_t* Wpt, uint8_t* Wtq, int64_t rows, int64_t cols,
                               cudaStream_t s);

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream finishes; it must call pdl_wait_primary()
// before reading that kernel's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// GEMV for 1..16 tokens. Returns cudaErrorNotSupported (without launching)
// when the activations of all tokens do not fit in shared memory.
// early_weights: the kernel enqueued just before on the stream does not write
// Wtq, so weight reads may start before waiting for it.
// inputs_final: the kernel enqueued just before is a GEMV (which lets its
// successor start only after its own wait, so nothing older still runs) and
// none of its outputs overlaps Wtq, Xq or X; the kernel may then read all its
// inputs before waiting for it and wait only before its first global write.
// Every GEMV kernel lets the next kernel start only after its own wait.
// With X non-null the GEMV quantizes the f32 activations X itself (the fused
// form; Xq is then an output, written once, and may be null) instead of
// reading q8_K blocks from Xq.
// With Xs non-null (4..8 tokens, the mma.sync GEMV) the activations come
// staged by launch_gemv_stage into Xs, enqueued just before on s; the kernel
// waits for it, loads the image with one bulk copy, and lets its successor
// start only once that copy has landed.
cudaError_t launch_gemv(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                        int64_t rows, int64_t cols, int ntok, int* dev_status, bool early_weights,
                        bool inputs_final, cudaStream_t s, const float* X = nullptr,
                        uint8_t* Xq_out = nullptr, const uint8_t* Xs = nullptr);

// Bytes of the staged activations of the mma.sync GEMV for ntok tokens (0
// outside 4..8, below 3072 columns, or where that GEMV would need more than
// the 227 KB of shared memory a block may opt in to on sm_103a), and whether
// the staged form runs: it fits on the current device, and the call
// quantizes X (quantizes) or has at least 5120 columns.
int64_t gemv_stage_bytes(int64_t cols, int ntok);
bool gemv_stage_fits(int64_t cols, int ntok, bool quantizes);
// Stages the activations into region (gemv_stage_bytes, 16-byte aligned):
// from the f32 X (quantized, the q8_K blocks written to Xq_out) or from the
// q8_K blocks Xq_in. x_final: the kernel before it on s writes nothing it
// reads (it may then read before waiting; it writes only after the wait).
// early_trigger: its successor may start before its wait (the host then
// checks that successor's early reads against the outputs of the kernel
// before this one too).
cudaError_t launch_gemv_stage(const float* X, const uint8_t* Xq_in, uint8_t* Xq_out,
                              uint8_t* region, int64_t cols, int ntok, bool x_final,
                              bool early_trigger, cudaStream_t s);
int gemv_max_tokens();
// Token counts up to which the workspace forms also run the GEMV (beyond, the
// tensor cores, which need the workspace).
int ws_gemv_max_tokens();

// Tensor-core path for any ntok >= 1 (used for ntok > gemv_max_tokens()).
cudaError_t launch_gemm_tc(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                           int64_t rows, int64_t cols, int64_t ntok, int* dev_status,
                           cudaStream_t s);

// Tensor-core path with a workspace: an activation pre-pass writes e4m3 B
// tiles into `ws` (tc_workspace_bytes(cols, ntok) bytes, 16-byte aligned).
int64_t tc_workspace_bytes(int64_t cols, int64_t ntok);
cudaError_t launch_gemm_tc_ws(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                              int64_t rows, int64_t cols, int64_t ntok, uint8_t* ws,
                              int* dev_status, cudaStream_t s);
// The same from f32 activations: one kernel quantizes them into Xq (q8_K, as
// launch_quantize_q8K) and packs the workspace, then the tensor-core kernel.
cudaError_t launch_quantize_gemm_tc_ws(const float* X, uint8_t* Xq, const uint8_t* Wtq, float* Y,
                                       int64_t rows, int64_t cols, int64_t ntok, uint8_t* ws,
                                       int* dev_status, cudaStream_t s);

// Opt a kernel in to `bytes` of dynamic shared memory on the current device
// (cached per device and kernel).
cudaError_t ensure_dynamic_smem(const void* kernel, int bytes);

// The current device's opt-in shared memory per block and SM count, read from
// the driver once per device.
struct DeviceLimits {
  int optin_smem;
  int sms;
};
cudaError_t device_limits(DeviceLimits* out);

// CTAs of kernel (threads per CTA, dynamic shared memory smem) that fit on one
// SM of the current device, asked of the driver once per device, kernel,
// block size and shared memory size (the answer never changes).
cudaError_t resident_ctas(const void* kernel, int threads, size_t smem, int* out);
// Record e as this host thread's tq_last_cuda_error.
void record_cuda_error(cudaError_t e);

// Read-ceiling probe: adds the buffer's 32-bit words (wrapping) to *out.
cudaError_t launch_read_sum(const void* buf, int64_t bytes, uint32_t* out, bool early,
                            cudaStream_t s);

// ptq1_0 stream layout (see tq_repack_ptq1_0_stream): re-tiling of the file.
cudaError_t launch_repack_ptq1_stream(const uint8_t* Wpt, uint8_t* Wt1, int64_t rows,
                                      int64_t cols, cudaStream_t s);
// GEMV over the ptq1_0 stream layout (1.75 bits per weight streamed and
// decoded in the kernel), any ntok >= 1 in launches of up to 8 tokens.
cudaError_t launch_gemv_ptq1(const uint8_t* Wt1, const uint8_t* Xq, float* Y, int32_t* S,
                             int64_t rows, int64_t cols, int ntok, int* dev_status,
                             bool early_weights, cudaStream_t s);

// Trit n (0..4) of a ptq1_0 code byte b: floor(3 * (b * 3^n mod 256) / 256),
// the code u = w + 1 (the ternary post, "the detour that lost").
__host__ __device__ __forceinline__ uint32_t ptq1_trit(uint32_t b, int n) {
  const uint32_t p3 = n == 0 ? 1u : n == 1 ? 3u : n == 2 ? 9u : n == 3 ? 27u : 81u;
  return (((b * p3) & 0xFFu) * 3u) >> 8;
}

// Test facility (tq_debug_stall_next_launch): the wait limit in ns that the
// next matmul kernel launched takes for its stalled first CTA, or 0 if none is
// pending; taking it clears it.
int64_t take_debug_stall();

}  // namespace tq
