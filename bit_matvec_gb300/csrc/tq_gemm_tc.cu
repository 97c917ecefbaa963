// tq_gemm_tc.cu -- ternary x q8_K product for many tokens on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// With many tokens a loaded weight is reused by all of them and instruction
// count, not the bus, bounds the work (ternary post, "prefill wants a
// different shape"). The pages use the CPU's int8 matrix instruction; here
// the contraction runs as tcgen05.mma kind::f16 with f32 accumulation, which
// is exact for this problem: w in {-1, 0, 1} and q in [-127, 127] are exact
// f16 values, each product is exact in f32, and every partial sum of a
// 128-weight group is an integer of magnitude <= 16256 < 2^24. (GB300's int8
// tensor rate is a small fraction of its f16 rate, so f16 is the faster exact
// route.)
//
// Per CTA: M = 128 weight rows (four 32-row tiles) x N = 64 tokens (zero
// padded; post, "the leftovers": pad, run one pass, store only the real
// outputs). For each 128-weight group g:
//   1. each thread unpacks its row's 128 codes straight to f16 w = u - 1 and
//      writes them to shared memory in the UMMA K-major no-swizzle layout;
//      threads also convert the group's int8 activations of all 64 tokens;
//   2. one thread issues 8 MMAs (K = 16 each) into a TMEM accumulator and
//      commits them to an mbarrier;
//   3. every thread reads its row of the accumulator (exact group sums) with
//      tcgen05.ld and applies d_w[r][g] * d_x[t][g/2] in f32.
// Each group's sum stays separate because the weight scale changes from
// group to group.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kM = 128;       // rows per CTA = UMMA M
constexpr int kN = 64;        // tokens per CTA = UMMA N
constexpr int kThreads = 128;
constexpr int kTilesPerCta = kM / kTileRows;
constexpr uint32_t kTmemCols = 64;  // one f32 accumulator of 128 lanes x 64 columns

// UMMA canonical K-major layout without swizzle: a core matrix is 8 rows x 16
// bytes stored as 128 contiguous bytes; LBO = distance between core matrices
// along K, SBO = distance between 8-row groups. A group (128 f16 along K) is
// 16 core matrices per 8-row group.
constexpr uint32_t kLBO = 128;
constexpr uint32_t kSBO = 16 * 128;
constexpr int kABytes = kM * kGroup * 2;   // 32 KB
constexpr int kBBytes = kN * kGroup * 2;   // 16 KB
constexpr int kSmemBytes = kABytes + kBBytes + kN * 4 + 16;

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s; an MMA group takes microseconds

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Shared-memory matrix descriptor: start >> 4 (bits 0-13), LBO >> 4 (16-29),
// SBO >> 4 (32-45), the constant 0b001 at bits 46-48, no swizzle (61-63 = 0).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(kLBO >> 4) << 16) |
         ((uint64_t)(kSBO >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after kWaitLimitNs of global time (or 2^30 polls).
__device__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return false;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}

// 16 consecutive f32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Codes of slot s (bits 2s..2s+1 of two bytes, placed in the low byte of each
// 16-bit half) -> f16 pair of w = u - 1. OR-ing 0x6400 (1024.0) makes the half
// 1024 + u * 4^s exactly; one FMA by 4^-s minus (1024 * 4^-s + 1) gives u - 1.
template <int s>
__device__ __forceinline__ uint32_t codes_to_w(uint32_t x) {
  const uint32_t v = (x & (0x00030003u << (2 * s))) | 0x64006400u;
  const float sc = 1.0f / (float)(1 << (2 * s));
  const __half2 m = __float2half2_rn(sc);
  const __half2 b = __float2half2_rn(-(1024.0f * sc + 1.0f));
  return h2_bits(__hfma2(bits_h2(v), m, b));
}

// int8 x4 -> two f16 pairs (exact): bias to u8, place under exponent 0x64
// (1024 + byte), subtract 1152.
__device__ __forceinline__ void s8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const __half2 off = __float2half2_rn(1152.0f);
  lo = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x5150)), off));
  hi = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x5352)), off));
}

struct TcArgs {
  const uint8_t* Wtq;
  const uint8_t* Xq;
  float* Y;
  int32_t* S;
  int* status;
  int64_t rows;
  int64_t ntok;
  int ngroups;
  int nblk;
  int nrb;
};

template <bool kGroupSums>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sA = smem;
  uint8_t* sB = smem + kABytes;
  float* sdx = reinterpret_cast<float*>(smem + kABytes + kBBytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sdx + kN);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar_a = smem_addr(bar);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(bar_a, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // this thread's weight row and its activation duty
  const int64_t rb = (int64_t)blockIdx.x * kTilesPerCta + warp;
  const int64_t row = rb * kTileRows + lane;
  const uint8_t* tiles = a.Wtq + rb * a.ngroups * kTileBytes;
  const bool row_tile_ok = rb < a.nrb;
  const int n_local = tid & (kN - 1);          // token converted by this thread
  const int k_half = tid >> 6;                 // which 64 activations of the group
  const int64_t tok = (int64_t)blockIdx.y * kN + n_local;
  const bool tok_ok = tok < a.ntok;
  const uint32_t a_row_off = (uint32_t)((tid >> 3) * kSBO + (tid & 7) * 16);
  const uint32_t b_row_off = (uint32_t)((n_local >> 3) * kSBO + (n_local & 7) * 16);

  float y[kN];
#pragma unroll
  for (int n = 0; n < kN; ++n) y[n] = 0.0f;
  bool failed = false;

  for (int g = 0; g < a.ngroups; ++g) {
    // ---- 1a. weights of this row -> f16 w in A (row tid, K-major)
    uint32_t wv[8];
    uint16_t sbits = 0;
    if (row_tile_ok) {
      const uint8_t* tile = tiles + (int64_t)g * kTileBytes;
      const uint4 lo = ldg_stream_v4(tile + lane * 16);
      const uint4 hi = ldg_stream_v4(tile + 512 + lane * 16);
      sbits = ldg_u16(tile + kTileCodeBytes + lane * 2);
      wv[0] = lo.x; wv[1] = lo.y; wv[2] = lo.z; wv[3] = lo.w;
      wv[4] = hi.x; wv[5] = hi.y; wv[6] = hi.z; wv[7] = hi.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) wv[i] = 0x55555555u;  // w = 0
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // word i: weights 16i + 4s + j sit in byte j at bits 2s
      const uint32_t x01 = __byte_perm(wv[i], 0, 0x4140);  // bytes 0,1 -> low byte of each half
      const uint32_t x23 = __byte_perm(wv[i], 0, 0x4342);  // bytes 2,3
      const uint4 c0 = make_uint4(codes_to_w<0>(x01), codes_to_w<0>(x23), codes_to_w<1>(x01),
                                  codes_to_w<1>(x23));       // k = 16i .. 16i+7
      const uint4 c1 = make_uint4(codes_to_w<2>(x01), codes_to_w<2>(x23), codes_to_w<3>(x01),
                                  codes_to_w<3>(x23));       // k = 16i+8 .. 16i+15
      *reinterpret_cast<uint4*>(sA + a_row_off + (2 * i) * kLBO) = c0;
      *reinterpret_cast<uint4*>(sA + a_row_off + (2 * i + 1) * kLBO) = c1;
    }

    // ---- 1b. activations: token n_local, k = 64*k_half .. +63 -> f16 in B
    {
      uint32_t q[16];
      if (tok_ok) {
        const uint8_t* blk = a.Xq + (tok * a.nblk + (g >> 1)) * kQ8KBytes;
        const uint32_t* src =
            reinterpret_cast<const uint32_t*>(blk + kQ8KQsOffset + (g & 1) * 128 + k_half * 64);
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = __ldg(src + i);
        if (k_half == 0) sdx[n_local] = __ldg(reinterpret_cast<const float*>(blk));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = 0u;
        if (k_half == 0) sdx[n_local] = 0.0f;
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // 8 activations per core-matrix row
        uint4 h;
        s8x4_to_h2x2(q[2 * c], h.x, h.y);
        s8x4_to_h2x2(q[2 * c + 1], h.z, h.w);
        *reinterpret_cast<uint4*>(sB + b_row_off + (k_half * 8 + c) * kLBO) = h;
      }
    }
    // generic-proxy smem writes -> visible to the tensor core (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    // ---- 2. one thread issues the group's 8 MMAs (K = 16 each)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_addr(sA), b0 = smem_addr(sB);
#pragma unroll
      for (int kk = 0; kk < kGroup / 16; ++kk)
        mma_f16(tmem, smem_desc(a0 + kk * 2 * kLBO), smem_desc(b0 + kk * 2 * kLBO), kIdesc,
                kk > 0 ? 1u : 0u);
      mma_commit(bar_a);
    }

    // ---- 3. wait for the accumulator, then scale and accumulate in f32
    const bool ok = mbar_wait_bounded(bar_a, (uint32_t)(g & 1));
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();
    const float dw = __half2float(__ushort_as_half(sbits));
#pragma unroll
    for (int c = 0; c < kN / 16; ++c) {
      float acc[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c * 16, acc);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = c * 16 + j;
        if (kGroupSums) {
          const int64_t t = (int64_t)blockIdx.y * kN + n;
          if (row_tile_ok && row < a.rows && t < a.ntok)
            a.S[(t * a.rows + row) * a.ngroups + g] = __float2int_rn(acc[j]);
        } else {
          y[n] = fmaf(dw * sdx[n], acc[j], y[n]);
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // all TMEM reads and sA/sB/sdx reads done before the next group
  }

  if (failed && tid == 0) atomicExch(a.status, kDevTimeout);
  if (!failed && !kGroupSums && row_tile_ok && row < a.rows) {
#pragma unroll
    for (int n = 0; n < kN; ++n) {
      const int64_t t = (int64_t)blockIdx.y * kN + n;
      if (t < a.ntok) a.Y[t * a.rows + row] = y[n];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols) : "memory");
  }
}

}  // namespace

cudaError_t launch_gemm_tc(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                           int64_t rows, int64_t cols, int64_t ntok, int* dev_status,
                           cudaStream_t s) {
  if (rows <= 0 || ntok <= 0 || cols <= 0) return cudaSuccess;
  TcArgs a;
  a.Wtq = Wtq;
  a.Xq = Xq;
  a.Y = Y;
  a.S = S;
  a.status = dev_status;
  a.rows = rows;
  a.ntok = ntok;
  a.ngroups = (int)(cols / kGroup);
  a.nblk = (int)(cols / kQK);
  a.nrb = (int)((rows + kTileRows - 1) / kTileRows);
  const int64_t gx = (rows + kM - 1) / kM, gy = (ntok + kN - 1) / kN;
  if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)gx, (unsigned)gy);
  const void* fn = S ? reinterpret_cast<const void*>(&gemm_tc_kernel<true>)
                     : reinterpret_cast<const void*>(&gemm_tc_kernel<false>);
  cudaError_t e = ensure_dynamic_smem(fn, kSmemBytes);
  if (e != cudaSuccess) return e;
  if (S)
    gemm_tc_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(a);
  else
    gemm_tc_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tq
