// tq_gemm_tc_ws.cu -- the tensor-core path with a caller-provided workspace.
//
// Converting the int8 activations to the MMA's f16 B operand is the same work
// for every 128-row tile of the weights; without a workspace each CTA repeats
// it (tq_gemm_tc.cu). Here a pre-pass does it once: act_pack writes, for each
// 64-token tile and each 128-weight group, the 64 x 128 f16 B operand laid out
// exactly as the MMA reads it (UMMA K-major, no swizzle: 16 KB contiguous),
// plus the q8_K block scales. The tensor-core kernel then stages a group with
// one bulk copy for B, four for the weight tiles and one for the scales, and
// its converter warps only unpack weights.
//
// Per CTA (128 weight rows x 64 tokens) and 128-weight group g:
//   - a producer warp stages the group's B tile, four 1088-byte weight tiles
//     and 64 block scales into an 8-slot shared-memory ring (TMA bulk copies,
//     one mbarrier per slot). Issuing a bulk copy can stall while the SM's
//     tensor cores are busy, so no other role issues copies;
//   - 8 converter warps unpack the codes to exact f16 w = u - 1 and store them
//     into tensor memory as the A operand (tcgen05.st), 64 weights per thread;
//   - one thread issues 8 tcgen05.mma kind::f16 (M=128, N=64, K=16) with A in
//     tensor memory and B read straight from the staged slot, accumulating the
//     exact group sums in tensor memory; its commit frees the slot;
//   - 8 epilogue warps tcgen05.ld the sums and apply d_w * d_x in f32.
// The exactness argument is the one of tq_gemm_tc.cu: w and q are exact f16,
// products exact in f32, group sums integers below 2^24.
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

using namespace tc;

constexpr int kM = 128;          // weight rows per CTA (UMMA M)
constexpr int kN = 64;           // tokens per CTA (UMMA N)
constexpr int kStages = 3;       // A operand / accumulator ring in tensor memory
// Staged-input ring depth: the group after next after next... must be in
// flight long enough to cover a bulk copy's latency under load (~2.5 us)
// while the tensor cores take ~0.35 us per group.
#ifndef TQ_TC_IN_STAGES
#define TQ_TC_IN_STAGES 8
#endif
constexpr int kInStages = TQ_TC_IN_STAGES;  // staged-input ring in shared memory
constexpr int kConvWarps = 8;    // converters: warp w -> rows 32*(w%4).., k half w/4
constexpr int kEpiWarps = 8;     // epilogue: warp w -> rows 32*(w%4).., tokens 32*(w/4)..
constexpr int kMmaWarp = kConvWarps + kEpiWarps;
constexpr int kProdWarp = kMmaWarp + 1;
constexpr int kThreads = (kProdWarp + 1) * 32;
constexpr int kTilesPerCta = kM / kTileRows;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;      // stage s accumulator: columns s*64 ..
constexpr uint32_t kACol = 192;      // stage s A operand: columns 192 + s*64 ..

// B tile of one (64-token tile, group): UMMA canonical K-major layout without
// swizzle; a core matrix is 8 tokens x 8 f16 (16 bytes each) stored as 128
// contiguous bytes; LBO = 128 (next 8 k), SBO = 2048 (next 8 tokens).
constexpr uint32_t kLBO = 128;
constexpr uint32_t kSBO = 16 * 128;
constexpr int kBTile = kN * kGroup * 2;                // 16384
constexpr int kDxBytes = kN * 4;                       // scales of one block, 64 tokens
// one staged slot: B tile, 4 weight tiles, block scales
constexpr int kInB = 0;
constexpr int kInW = kBTile;
constexpr int kInDx = kInW + kTilesPerCta * kTileBytes;
constexpr int kInBytes = kInDx + kDxBytes;             // 20992
constexpr int kSmemUsed = kInStages * kInBytes + kStages * (kM + kN) * 4 +
                          (2 * kInStages + 3 * kStages) * 8 + 16;
// Enough shared memory that only one CTA fits on an SM: each CTA allocates
// all 512 tensor-memory columns.
constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
constexpr uint32_t kIdesc = idesc_f16(kM, kN);
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct Layout {
  int64_t ntile;      // 64-token tiles
  int64_t b_bytes;    // ntile * G * 16 KB
  int64_t dx_bytes;   // ntile * nblk * 64 * 4
};

__host__ __device__ inline Layout ws_layout(int64_t cols, int64_t ntok) {
  Layout l;
  l.ntile = (ntok + kN - 1) / kN;
  l.b_bytes = l.ntile * (cols / kGroup) * kBTile;
  l.dx_bytes = l.ntile * (cols / kQK) * kDxBytes;
  return l;
}

// ---------------------------------------------------------------- pre-pass

// One CTA per (group g, token tile): thread t converts token t % 64, k quarter
// t / 64 (32 activations) and writes them as 4 core-matrix rows of 16 bytes.
__global__ void __launch_bounds__(256) act_pack_kernel(const uint8_t* __restrict__ Xq,
                                                       uint8_t* __restrict__ Bt,
                                                       float* __restrict__ Dx, int64_t ntok,
                                                       int ngroups, int nblk) {
  pdl_launch_dependents();
  pdl_wait_primary();   // the q8_K activations come from the previous kernel
  const int g = blockIdx.x;
  const int64_t nt = blockIdx.y;
  const int n = threadIdx.x & (kN - 1), kq = threadIdx.x >> 6;
  const int64_t tok = nt * kN + n;
  uint32_t q[8];
  float d = 0.0f;
  if (tok < ntok) {
    const uint8_t* blk = Xq + (tok * nblk + (g >> 1)) * kQ8KBytes;
    const uint32_t* src =
        reinterpret_cast<const uint32_t*>(blk + kQ8KQsOffset + (g & 1) * kGroup + kq * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __ldg(src + i);
    d = __ldg(reinterpret_cast<const float*>(blk));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0u;   // padded tokens: zero activations, zero scale
  }
  uint8_t* tile = Bt + (nt * ngroups + g) * kBTile + (n >> 3) * kSBO + (n & 7) * 16;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 h;
    s8x4_to_h2x2(q[2 * c], h.x, h.y);
    s8x4_to_h2x2(q[2 * c + 1], h.z, h.w);
    *reinterpret_cast<uint4*>(tile + (kq * 4 + c) * kLBO) = h;
  }
  if (kq == 0 && (g & 1) == 0) Dx[(nt * nblk + (g >> 1)) * kN + n] = d;
}

// ---------------------------------------------------------------- tensor cores

struct WsArgs {
  const uint8_t* Wtq;
  const uint8_t* Bt;
  const float* Dx;
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
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_ws_kernel(const WsArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sIn = smem;                                                         // [4][20992]
  float* sdw = reinterpret_cast<float*>(smem + kInStages * kInBytes);          // [S][128]
  float* sdx = sdw + kStages * kM;                                             // [S][64]
  uint64_t* in_full = reinterpret_cast<uint64_t*>(sdx + kStages * kN);         // [4]
  uint64_t* in_empty = in_full + kInStages;                                    // [4]
  uint64_t* conv_full = in_empty + kInStages;                                  // [S]
  uint64_t* mma_done = conv_full + kStages;                                    // [S]
  uint64_t* stage_free = mma_done + kStages;                                   // [S]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stage_free + kStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.ngroups;
  const int64_t rb0 = (int64_t)blockIdx.x * kTilesPerCta;
  const int64_t nt = blockIdx.y;
  const int64_t tok0 = nt * kN;

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < kInStages; ++i) {
      mbarrier_init(smem_u32(in_full + i), 1);
      // converters have read the weights and scales, and the MMAs have read B
      mbarrier_init(smem_u32(in_empty + i), kConvWarps * 32 + 1);
    }
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

  if (warp == kProdWarp) {
    // ---------------- producer: stage group g into slot g % kInStages
    if (lane == 0) {
      int nvalid = 0;                                     // weight tiles that exist
      for (int q = 0; q < kTilesPerCta; ++q) nvalid += (rb0 + q < a.nrb) ? 1 : 0;
      const uint64_t policy = l2_evict_first_policy();
      pdl_wait_primary();   // the workspace is written by the previous kernel (the pre-pass)
      int i = 0;
      uint32_t ph = 0;
      for (int g = 0; g < G; ++g) {
        // the slot is free once the converters and the MMAs of group g - kInStages are done
        if (g >= kInStages &&
            !mbarrier_wait_bounded(smem_u32(in_empty + i), ph ^ 1u, kWaitLimitNs)) {
          failed = true;
          break;
        }
        uint8_t* st = sIn + i * kInBytes;
        const uint32_t full = smem_u32(in_full + i);
        mbarrier_arrive_expect_tx(full, (uint32_t)(kBTile + nvalid * kTileBytes + kDxBytes));
        bulk_copy_g2s(smem_u32(st + kInB), a.Bt + (nt * G + g) * (int64_t)kBTile, kBTile, full,
                      policy);
        for (int q = 0; q < nvalid; ++q)
          bulk_copy_g2s(smem_u32(st + kInW + q * kTileBytes),
                        a.Wtq + ((rb0 + q) * G + g) * kTileBytes, kTileBytes, full, policy);
        bulk_copy_g2s(smem_u32(st + kInDx), a.Dx + (nt * a.nblk + (g >> 1)) * kN, kDxBytes, full,
                      policy);
        if (++i == kInStages) { i = 0; ph ^= 1u; }
      }
    }
  } else if (warp < kConvWarps) {
    // ---------------- converters
    const int q4 = warp & 3, khalf = warp >> 2;          // row quarter, k half of A
    const bool row_ok = rb0 + q4 < a.nrb;
    const int ct = warp * 32 + lane;                      // 0..255; ct < 64 copies scales
    const uint32_t a_lane = (uint32_t)(q4 * 32) << 16;
    int i = 0, s = 0;
    uint32_t pin = 0, ph = 0;
    for (int g = 0; g < G; ++g) {
      if (!failed && !mbarrier_wait_bounded(smem_u32(in_full + i), pin, kWaitLimitNs)) failed = true;
      const uint8_t* st = sIn + i * kInBytes;
      uint4 codes = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);  // w = 0
      uint32_t scale = 0u;
      float dx = 0.0f;
      if (!failed) {
        if (row_ok) {
          codes = *reinterpret_cast<const uint4*>(st + kInW + q4 * kTileBytes + khalf * 512 + lane * 16);
          if (khalf == 0)
            scale = *reinterpret_cast<const uint16_t*>(st + kInW + q4 * kTileBytes + kTileCodeBytes + lane * 2);
        }
        if (ct < kN) dx = reinterpret_cast<const float*>(st + kInDx)[ct];
      }
      mbarrier_arrive(smem_u32(in_empty + i));
      if (++i == kInStages) { i = 0; pin ^= 1u; }

      // conversion stage s is free once the epilogue has drained group g - 3
      if (g >= kStages && !failed &&
          !mbarrier_wait_bounded(smem_u32(stage_free + s), ph ^ 1u, kWaitLimitNs))
        failed = true;
      failed = __any_sync(0xffffffffu, failed);   // tcgen05.st below is warp-wide
      tc_fence_after();
      if (!failed) {
        uint32_t wa[32];
        const uint32_t wv[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          // word w: weights 16w + 4s + j in byte j at bits 2s (k local to this half)
          const uint32_t x01 = __byte_perm(wv[w], 0, 0x4140);
          const uint32_t x23 = __byte_perm(wv[w], 0, 0x4342);
          wa[8 * w + 0] = codes_to_w<0>(x01);
          wa[8 * w + 1] = codes_to_w<0>(x23);
          wa[8 * w + 2] = codes_to_w<1>(x01);
          wa[8 * w + 3] = codes_to_w<1>(x23);
          wa[8 * w + 4] = codes_to_w<2>(x01);
          wa[8 * w + 5] = codes_to_w<2>(x23);
          wa[8 * w + 6] = codes_to_w<3>(x01);
          wa[8 * w + 7] = codes_to_w<3>(x23);
        }
        tmem_st32(tmem + a_lane + kACol + (uint32_t)s * 64 + (uint32_t)khalf * 32, wa);
        if (khalf == 0) sdw[s * kM + q4 * 32 + lane] = __half2float(__ushort_as_half((unsigned short)scale));
        if (ct < kN) sdx[s * kN + ct] = dx;
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      tc_fence_before();
      mbarrier_arrive(smem_u32(conv_full + s));
      if (++s == kStages) { s = 0; ph ^= 1u; }
    }
  } else if (warp < kMmaWarp) {
    // ---------------- epilogue
    const int ew = warp - kConvWarps;
    const int q4 = ew & 3, nhalf = ew >> 2;               // row quarter, token half
    const int64_t row = (rb0 + q4) * kTileRows + lane;
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
              const int64_t t = tok0 + n0 + j;
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
        const int64_t t = tok0 + n0 + j;
        if (t < a.ntok) a.Y[t * a.rows + row] = y[j];
      }
    }
  } else if (lane == 0) {
    // ---------------- MMA issuer
    int i = 0, s = 0;
    uint32_t ph = 0;
    for (int g = 0; g < G; ++g) {
      if (!failed && !mbarrier_wait_bounded(smem_u32(conv_full + s), ph, kWaitLimitNs)) failed = true;
      tc_fence_after();
      if (!failed) {
        const uint32_t d = tmem + kAccCol + (uint32_t)s * 64;
        const uint32_t at = tmem + kACol + (uint32_t)s * 64;
        const uint32_t b0 = smem_u32(sIn + i * kInBytes + kInB);
#pragma unroll
        for (int kk = 0; kk < kGroup / 16; ++kk)
          mma_f16_tmem_a(d, at + 8 * kk, smem_desc(b0 + kk * 2 * kLBO, kLBO, kSBO), kIdesc,
                         kk > 0 ? 1u : 0u);
      }
      // both commits fire when these MMAs are done (at once if none were issued)
      mma_commit(smem_u32(mma_done + s));
      mma_commit(smem_u32(in_empty + i));
      if (++s == kStages) { s = 0; ph ^= 1u; }
      if (++i == kInStages) i = 0;
    }
  }

  if (failed) atomicExch(a.status, kDevTimeout);
  // After a failure, staged copies may still be in flight: let the last use of
  // each input slot land before shared memory is released.
  if (__syncthreads_or(failed) && warp == kProdWarp && lane == 0) {
    for (int i = 0; i < kInStages && i < G; ++i) {
      const int last = i + (G - 1 - i) / kInStages * kInStages;
      mbarrier_wait_bounded(smem_u32(in_full + i), (uint32_t)((last / kInStages) & 1), kWaitLimitNs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols) : "memory");
  }
}

}  // namespace

int64_t tc_workspace_bytes(int64_t cols, int64_t ntok) {
  const Layout l = ws_layout(cols, ntok);
  return l.b_bytes + l.dx_bytes;
}

cudaError_t launch_gemm_tc_ws(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                              int64_t rows, int64_t cols, int64_t ntok, uint8_t* ws,
                              int* dev_status, cudaStream_t s) {
  if (rows <= 0 || ntok <= 0 || cols <= 0) return cudaSuccess;
  const Layout l = ws_layout(cols, ntok);
  const int G = (int)(cols / kGroup), nblk = (int)(cols / kQK);
  if (l.ntile > 65535) return cudaErrorInvalidConfiguration;
  uint8_t* Bt = ws;
  float* Dx = reinterpret_cast<float*>(ws + l.b_bytes);
  cudaError_t e = launch_pdl(act_pack_kernel, dim3((unsigned)G, (unsigned)l.ntile), dim3(256), 0,
                             s, Xq, Bt, Dx, ntok, G, nblk);
  if (e != cudaSuccess) return e;

  WsArgs a;
  a.Wtq = Wtq;
  a.Bt = Bt;
  a.Dx = Dx;
  a.Y = Y;
  a.S = S;
  a.status = dev_status;
  a.rows = rows;
  a.ntok = ntok;
  a.ngroups = G;
  a.nblk = nblk;
  a.nrb = (int)((rows + kTileRows - 1) / kTileRows);
  const int64_t gx = (rows + kM - 1) / kM;
  if (gx > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)gx, (unsigned)l.ntile);
  if (S) {
    e = ensure_dynamic_smem(reinterpret_cast<const void*>(&gemm_tc_ws_kernel<true>), kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemm_tc_ws_kernel<true>, grid, dim3(kThreads), kSmemBytes, s, a);
  }
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(&gemm_tc_ws_kernel<false>), kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(gemm_tc_ws_kernel<false>, grid, dim3(kThreads), kSmemBytes, s, a);
}

}  // namespace tq
