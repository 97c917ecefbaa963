// tq_gemm_tc.cu -- ternary x q8_K product for many tokens on the 5th-generation
// tensor cores (tcgen05.mma, operands and accumulators in tensor memory).
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
// One CTA computes 128 weight rows x 64 tokens (tokens zero-padded; ternary
// post, "the leftovers": pad, run one pass, store only the real outputs).
// Each 128-weight group g flows through a 3-stage ring:
//   - 8 converter warps load the group's codes (16 bytes per row-half per
//     thread) and unpack them straight to f16 w = u - 1: (code & mask) | 0x6400
//     is 1024 + u*4^s, one HFMA2 by 4^-s takes off the 1024 and the 1. The
//     result goes into tensor memory with tcgen05.st as the MMA's A operand
//     (lane = row), so A never touches shared memory. They also convert the
//     group's int8 activations of the 64 tokens to f16 into shared memory in
//     the UMMA K-major layout (the B operand). Loads for group g+1 are in
//     flight while group g is converted.
//   - one thread issues 8 MMAs (M=128, N=64, K=16) into the stage's TMEM
//     accumulator and commits them to an mbarrier.
//   - 8 epilogue warps read the accumulator (exact group sums) with
//     tcgen05.ld and apply d_w[r][g] * d_x[t][g/2] in f32.
// Each group's sum stays separate because the weight scale changes from
// group to group; the ring lets conversion, MMA and epilogue of consecutive
// groups overlap.
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

using namespace tc;

constexpr int kM = 128;          // weight rows per CTA (UMMA M)
constexpr int kN = 64;           // tokens per CTA (UMMA N)
constexpr int kStages = 3;
constexpr int kConvWarps = 8;    // converters: warp w -> rows 32*(w%4).., k half w/4
constexpr int kEpiWarps = 8;     // epilogue: warp w -> rows 32*(w%4).., tokens 32*(w/4)..
constexpr int kMmaWarp = kConvWarps + kEpiWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kTilesPerCta = kM / kTileRows;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;      // stage s accumulator: columns s*64 ..
constexpr uint32_t kACol = 192;      // stage s A operand: columns 192 + s*64 ..

// UMMA canonical K-major layout without swizzle for B: a core matrix is 8
// tokens x 16 bytes stored as 128 contiguous bytes; LBO = distance between
// core matrices along K, SBO = distance between 8-token groups.
constexpr uint32_t kLBO = 128;
constexpr uint32_t kSBO = 16 * 128;
constexpr int kBBytes = kN * kGroup * 2;   // 16 KB per stage
constexpr int kSmemUsed = kStages * kBBytes + kStages * (kM + kN) * 4 + 3 * kStages * 8 + 16;
// Request enough shared memory that only one CTA fits on an SM: each CTA
// allocates all 512 tensor-memory columns.
constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;

constexpr uint32_t kIdesc = tc::idesc_f16(kM, kN);

constexpr uint64_t kWaitLimitNs = 2000000000ull;

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

// What one converter thread loads for one group.
struct ConvIn {
  uint4 codes;      // 64 weights of its row (half of the group)
  uint32_t scale;   // fp16 bits of d_w (used by the k-half-0 threads)
  uint32_t q[8];    // 32 int8 activations of its token
  float dx;         // q8_K scale of its token's block (k-quarter-0 threads)
};

template <bool kGroupSums>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sB = smem;                                                          // [S][16 KB]
  float* sdw = reinterpret_cast<float*>(smem + kStages * kBBytes);             // [S][128]
  float* sdx = sdw + kStages * kM;                                             // [S][64]
  uint64_t* conv_full = reinterpret_cast<uint64_t*>(sdx + kStages * kN);       // [S]
  uint64_t* mma_done = conv_full + kStages;                                    // [S]
  uint64_t* stage_free = mma_done + kStages;                                   // [S]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stage_free + kStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.ngroups;

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbarrier_init(smem_u32(conv_full + s), kConvWarps * 32);
      mbarrier_init(smem_u32(mma_done + s), 1);
      mbarrier_init(smem_u32(stage_free + s), kEpiWarps * 32);
    }
    mbarrier_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp < kConvWarps) {
    // ---------------- converters
    const int q4 = warp & 3, khalf = warp >> 2;          // row quarter, k half of A
    const int64_t rb = (int64_t)blockIdx.x * kTilesPerCta + q4;
    const bool row_ok = rb < a.nrb;
    const uint8_t* tiles = a.Wtq + rb * G * kTileBytes + khalf * 512 + lane * 16;
    const int ct = warp * 32 + lane;                      // 0..255
    const int n = ct & (kN - 1), kq = ct >> 6;            // token, k quarter of B
    const int64_t tok = (int64_t)blockIdx.y * kN + n;
    const bool tok_ok = tok < a.ntok;
    const uint8_t* xrow = a.Xq + tok * a.nblk * kQ8KBytes;
    const uint32_t b_off = (uint32_t)((n >> 3) * kSBO + (n & 7) * 16);
    const uint32_t a_lane = (uint32_t)(q4 * 32) << 16;

    auto load = [&](int g, ConvIn& in) {
      if (row_ok) {
        const uint8_t* t = tiles + (int64_t)g * kTileBytes;
        in.codes = ldg_stream_v4(t);
        in.scale = khalf == 0 ? ldg_u16(t - khalf * 512 - lane * 16 + kTileCodeBytes + lane * 2) : 0u;
      } else {
        in.codes = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);  // w = 0
        in.scale = 0u;
      }
      if (tok_ok) {
        const uint8_t* blk = xrow + (int64_t)(g >> 1) * kQ8KBytes;
        const uint32_t* src =
            reinterpret_cast<const uint32_t*>(blk + kQ8KQsOffset + (g & 1) * 128 + kq * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) in.q[i] = __ldg(src + i);
        in.dx = kq == 0 ? __ldg(reinterpret_cast<const float*>(blk)) : 0.0f;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) in.q[i] = 0u;
        in.dx = 0.0f;
      }
    };

    ConvIn cur, nxt;
    load(0, cur);
    int s = 0;
    uint32_t ph = 0;
    for (int g = 0; g < G; ++g) {
      if (g + 1 < G) load(g + 1, nxt);
      // stage s is free once the epilogue has drained group g - 3
      if (g >= kStages && !failed &&
          !mbarrier_wait_bounded(smem_u32(stage_free + s), ph ^ 1u, kWaitLimitNs))
        failed = true;
      failed = __any_sync(0xffffffffu, failed);   // tcgen05.st below is warp-wide
      tc_fence_after();
      if (!failed) {
        // A: 64 weights of this row -> 32 f16 pairs in TMEM (columns = k pairs)
        uint32_t wa[32];
        const uint32_t wv[4] = {cur.codes.x, cur.codes.y, cur.codes.z, cur.codes.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          // word i: weights 16i + 4s + j in byte j at bits 2s (k local to this half)
          const uint32_t x01 = __byte_perm(wv[i], 0, 0x4140);
          const uint32_t x23 = __byte_perm(wv[i], 0, 0x4342);
          wa[8 * i + 0] = codes_to_w<0>(x01);
          wa[8 * i + 1] = codes_to_w<0>(x23);
          wa[8 * i + 2] = codes_to_w<1>(x01);
          wa[8 * i + 3] = codes_to_w<1>(x23);
          wa[8 * i + 4] = codes_to_w<2>(x01);
          wa[8 * i + 5] = codes_to_w<2>(x23);
          wa[8 * i + 6] = codes_to_w<3>(x01);
          wa[8 * i + 7] = codes_to_w<3>(x23);
        }
        tmem_st32(tmem + a_lane + kACol + (uint32_t)s * 64 + (uint32_t)khalf * 32, wa);
        // B: 32 activations of token n -> 4 core-matrix rows (8 k each)
        uint8_t* b = sB + s * kBBytes + b_off;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 h;
          s8x4_to_h2x2(cur.q[2 * c], h.x, h.y);
          s8x4_to_h2x2(cur.q[2 * c + 1], h.z, h.w);
          *reinterpret_cast<uint4*>(b + (kq * 4 + c) * kLBO) = h;
        }
        if (khalf == 0) sdw[s * kM + q4 * 32 + lane] = __half2float(__ushort_as_half((unsigned short)cur.scale));
        if (kq == 0) sdx[s * kN + n] = cur.dx;
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbarrier_arrive(smem_u32(conv_full + s));
      cur = nxt;
      if (++s == kStages) { s = 0; ph ^= 1u; }
    }
  } else if (warp < kMmaWarp) {
    // ---------------- epilogue
    const int ew = warp - kConvWarps;
    const int q4 = ew & 3, nhalf = ew >> 2;               // row quarter, token half
    const int64_t row = ((int64_t)blockIdx.x * kTilesPerCta + q4) * kTileRows + lane;
    const int n0 = nhalf * 32;
    const uint32_t acc_lane = (uint32_t)(q4 * 32) << 16;
    float y[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = 0.0f;
    int s = 0;
    uint32_t ph = 0;
    for (int g = 0; g < G; ++g) {
      if (!failed && !mbarrier_wait_bounded(smem_u32(mma_done + s), ph, kWaitLimitNs)) failed = true;
      failed = __any_sync(0xffffffffu, failed);   // tcgen05.ld below is warp-wide
      tc_fence_after();
      if (!failed) {
        uint32_t acc[32];
        tmem_ld32(tmem + acc_lane + kAccCol + (uint32_t)s * 64 + (uint32_t)n0, acc);
        if (kGroupSums) {
          if (row < a.rows) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int64_t t = (int64_t)blockIdx.y * kN + n0 + j;
              if (t < a.ntok) a.S[(t * a.rows + row) * G + g] = __float2int_rn(__uint_as_float(acc[j]));
            }
          }
        } else {
          const float dw = sdw[s * kM + q4 * 32 + lane];
          const float4* dx4 = reinterpret_cast<const float4*>(sdx + s * kN + n0);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 d = dx4[j4];
            y[4 * j4 + 0] = fmaf(dw * d.x, __uint_as_float(acc[4 * j4 + 0]), y[4 * j4 + 0]);
            y[4 * j4 + 1] = fmaf(dw * d.y, __uint_as_float(acc[4 * j4 + 1]), y[4 * j4 + 1]);
            y[4 * j4 + 2] = fmaf(dw * d.z, __uint_as_float(acc[4 * j4 + 2]), y[4 * j4 + 2]);
            y[4 * j4 + 3] = fmaf(dw * d.w, __uint_as_float(acc[4 * j4 + 3]), y[4 * j4 + 3]);
          }
        }
      }
      tc_fence_before();
      mbarrier_arrive(smem_u32(stage_free + s));
      if (++s == kStages) { s = 0; ph ^= 1u; }
    }
    if (!kGroupSums && !failed && row < a.rows) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int64_t t = (int64_t)blockIdx.y * kN + n0 + j;
        if (t < a.ntok) a.Y[t * a.rows + row] = y[j];
      }
    }
  } else if (lane == 0) {
    // ---------------- MMA issuer
    const uint32_t b0 = smem_u32(sB);
    int s = 0;
    uint32_t ph = 0;
    for (int g = 0; g < G; ++g) {
      if (!failed && !mbarrier_wait_bounded(smem_u32(conv_full + s), ph, kWaitLimitNs)) failed = true;
      tc_fence_after();
      if (!failed) {
        const uint32_t d = tmem + kAccCol + (uint32_t)s * 64;
        const uint32_t at = tmem + kACol + (uint32_t)s * 64;
#pragma unroll
        for (int kk = 0; kk < kGroup / 16; ++kk)
          mma_f16_tmem_a(d, at + 8 * kk, smem_desc(b0 + s * kBBytes + kk * 2 * kLBO, kLBO, kSBO), kIdesc,
                         kk > 0 ? 1u : 0u);
      }
      mma_commit(smem_u32(mma_done + s));   // also on failure: keeps the epilogue's phases moving
      if (++s == kStages) { s = 0; ph ^= 1u; }
    }
  }

  if (failed) atomicExch(a.status, kDevTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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
