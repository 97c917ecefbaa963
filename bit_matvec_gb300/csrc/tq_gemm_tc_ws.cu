// tq_gemm_tc_ws.cu -- the tensor-core path with a caller-provided workspace.
//
// Converting the int8 activations to the MMA's f16 B operand is the same work
// for every 128-row tile of the weights; without a workspace each CTA repeats
// it (tq_gemm_tc.cu). Here a pre-pass does it once: act_pack writes, for each
// 64-token tile and each 128-weight group, the f16 B operand laid out exactly
// as the MMA reads it (UMMA K-major, no swizzle), a small correction operand,
// and the q8_K block scales. The tensor-core kernel stages a q8_K block with
// one bulk copy for B, one per 32-row weight tile and one for the scales.
//
// Operands. A weight code u (w = u - 1) at bits 2s..2s+1 of a byte is turned
// into an f16 by one AND: with the exponent field zero, the half is the
// subnormal u * 4^s * 2^-24 (exact; the tensor cores take subnormal f16
// operands exactly). The pre-pass scales each activation by the matching
// 2^(9 - 2s), so every product is u * q * 2^-15 exactly. A sixteen-column
// correction MMA per group adds -2^-15 * sum_k q_k (A = constant -2^-9 and
// -2^-15 columns, B = the sum split as 64 * hi + lo), so the accumulator ends
// at isum * 2^-15 with isum = sum_k (u_k - 1) q_k. Every partial sum is an
// integer multiple of 2^-15 below 2^16 * 2^-15 in magnitude, so the f32
// accumulation is exact; the epilogue scales by d_w * 2^15 * d_x.
//
// Per CTA (128 weight rows x 64 tokens) the work goes one q8_K block (two
// 128-weight groups) at a time:
//   - a producer warp stages the block's two B tiles (one 36 KB bulk copy),
//     the weight tiles of both groups (one 2176-byte copy per 32-row tile:
//     consecutive groups of a tile are adjacent in the repacked layout) and 64
//     block scales into a shared-memory ring. Few large copies: issuing a bulk
//     copy stalls once many are in flight, and no other role issues copies;
//   - 8 converter warps mask the codes of both groups into A and store them
//     into tensor memory (tcgen05.st), 2 x 64 weights per thread;
//   - one thread issues per group 8 tcgen05.mma kind::f16 (M=128, N=64, K=16)
//     with A in tensor memory and B read from the staged slot, plus the
//     correction MMA, into one accumulator per group in tensor memory;
//   - 8 epilogue warps tcgen05.ld both accumulators and add
//     d_x * (d_w0 * acc0 + d_w1 * acc1) in packed f32x2 arithmetic.
// The A operand and the accumulators have separate rings in tensor memory: an
// A stage is free again as soon as its MMAs finish, an accumulator once the
// epilogue has read it.
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

using namespace tc;

constexpr int kM = 128;          // weight rows per CTA (UMMA M)
constexpr int kN = 64;           // tokens per CTA (UMMA N)
constexpr int kGPB = kQK / kGroup;   // groups per q8_K block (2)
constexpr int kAStages = 2;      // A operand ring in tensor memory (one block each)
constexpr int kAccStages = 2;    // accumulator ring in tensor memory (one block each)
// d_w / d_x per block, written by the converters and read by the epilogue: a
// converter at block b has seen the MMAs of b - kAStages finish, which were
// issued after the epilogue released block b - kAStages - kAccStages.
constexpr int kScaleStages = kAStages + kAccStages;
#ifndef TQ_TC_IN_STAGES
#define TQ_TC_IN_STAGES 3
#endif
constexpr int kInStages = TQ_TC_IN_STAGES;  // staged-input ring in shared memory
constexpr int kConvWarps = 8;    // converters: warp w -> rows 32*(w%4).., k half w/4
constexpr int kEpiWarps = 8;     // epilogue: warp w -> rows 32*(w%4).., tokens 32*(w/4)..
constexpr int kMmaWarp = kConvWarps + kEpiWarps;
constexpr int kProdWarp = kMmaWarp + 1;
constexpr int kThreads = (kProdWarp + 1) * 32;
constexpr int kTilesPerCta = kM / kTileRows;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBlkCols = kGPB * kN;             // 128: one block's accumulators (or A)
constexpr uint32_t kAccCol = 0;                      // accumulator stage c: c*128 + gi*64
constexpr uint32_t kACol = kAccStages * kBlkCols;    // A stage a: kACol + a*128 + gi*64
static_assert(kACol + kAStages * kBlkCols <= kTmemCols, "tensor memory overflow");
static_assert(kAStages == kAccStages, "mma_ready pairs A stage b % 2 with accumulator stage b % 2");

// B operands in UMMA canonical K-major layout without swizzle: a core matrix
// is 8 rows x 8 f16 (16 bytes each) stored as 128 contiguous bytes; LBO = 128
// (next 8 k). Main tile: 64 tokens x 128 k, SBO = 2048 (next 8 tokens).
// Correction tile: 64 tokens x 16 k, SBO = 256. The constant correction A
// operand (128 rows x 16 k) uses the layout of the correction tile.
constexpr uint32_t kLBO = 128;
constexpr uint32_t kSBO = 16 * 128;
constexpr uint32_t kSBOc = 2 * 128;
constexpr int kBMain = kN * kGroup * 2;                // 16384
constexpr int kBCorr = kN * 16 * 2;                    // 2048
constexpr int kBTile = kBMain + kBCorr;                // per (token tile, group)
constexpr int kACorrBytes = kM * 16 * 2;               // 4096
constexpr float kProdScale = 32768.0f;                 // products carry 2^-15
constexpr int kDxBytes = kN * 4;                       // scales of one block, 64 tokens
// one staged slot: the block's B tiles, its weight tiles (per 32-row tile both
// groups, adjacent), its block scales
constexpr int kInB = 0;
constexpr int kInW = kGPB * kBTile;
constexpr int kWRun = kGPB * kTileBytes;               // one 32-row tile, both groups
constexpr int kInDx = kInW + kTilesPerCta * kWRun;
constexpr int kInBytes = kInDx + kDxBytes;
static_assert(kInBytes % 16 == 0 && kWRun % 16 == 0, "bulk copies need 16-byte multiples");
constexpr int kSmemUsed = kInStages * kInBytes + kACorrBytes +
                          kScaleStages * (kGPB * kM + kN) * 4 +
                          (2 * kInStages + 2 * kAStages + kAccStages) * 8 + 16;
// Enough shared memory that only one CTA fits on an SM: each CTA allocates
// all 512 tensor-memory columns.
constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
constexpr uint32_t kIdesc = idesc_f16(kM, kN);
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct Layout {
  int64_t ntile;      // 64-token tiles
  int64_t b_bytes;    // ntile * G * 18 KB
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

// f16x2 bits of 2^(9 - 2s), s = 0..3: the activation scale matching slot s.
__device__ __forceinline__ uint32_t slot_scale(int s) {
  return s == 0 ? 0x60006000u : s == 1 ? 0x58005800u : s == 2 ? 0x50005000u : 0x48004800u;
}

__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// One CTA per (group g, token tile): thread t converts token t % 64, k quarter
// t / 64 (32 activations, scaled by 2^(9 - 2s)) and writes them as 4 core-
// matrix rows of 16 bytes; the k-quarter-0 threads also write the token's
// correction row and (for even g) its block scale.
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
  int sq = 0;   // sum of the group's 128 activations
  if (tok < ntok) {
    const uint8_t* blk = Xq + (tok * nblk + (g >> 1)) * kQ8KBytes;
    const uint32_t* src =
        reinterpret_cast<const uint32_t*>(blk + kQ8KQsOffset + (g & 1) * kGroup + kq * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __ldg(src + i);
    d = __ldg(reinterpret_cast<const float*>(blk));
    if (kq == 0) {
      // bsums: 16 int16 after the 256 values, 16 activations each
      const int16_t* bs = reinterpret_cast<const int16_t*>(blk + kQ8KQsOffset + kQK);
#pragma unroll
      for (int i = 0; i < 8; ++i) sq += __ldg(bs + (g & 1) * 8 + i);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0u;   // padded tokens: zero activations, zero scale
  }
  uint8_t* tile = Bt + (nt * ngroups + g) * kBTile;
  uint8_t* row = tile + (n >> 3) * kSBO + (n & 7) * 16;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    // words 2c, 2c+1: k = kq*32 + 8c + 0..7, slots s = (2c) % 4 and (2c + 1) % 4
    uint4 h;
    s8x4_to_h2x2(q[2 * c], h.x, h.y);
    s8x4_to_h2x2(q[2 * c + 1], h.z, h.w);
    const uint32_t m0 = slot_scale((2 * c) & 3), m1 = slot_scale((2 * c + 1) & 3);
    h.x = h2_mul(h.x, m0);
    h.y = h2_mul(h.y, m0);
    h.z = h2_mul(h.z, m1);
    h.w = h2_mul(h.w, m1);
    *reinterpret_cast<uint4*>(row + (kq * 4 + c) * kLBO) = h;
  }
  if (kq == 0) {
    // correction row: k0 = hi, k1 = lo with sq = 64 * hi + lo, 0 <= lo < 64
    const int hi = sq >> 6, lo = sq & 63;
    const uint32_t w0 = (uint32_t)__half_as_ushort(__int2half_rn(hi)) |
                        ((uint32_t)__half_as_ushort(__int2half_rn(lo)) << 16);
    uint8_t* crow = tile + kBMain + (n >> 3) * kSBOc + (n & 7) * 16;
    *reinterpret_cast<uint4*>(crow) = make_uint4(w0, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(crow + kLBO) = make_uint4(0u, 0u, 0u, 0u);
    if ((g & 1) == 0) Dx[(nt * nblk + (g >> 1)) * kN + n] = d;
  }
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

// One group's codes (this thread: one row, 64 weights) -> subnormal f16 A
// values u * 4^s * 2^-24, stored to tensor memory at taddr. Register 8w + 2s + p
// holds weights 16w + 4s + 2p and +1 (k local to this half), the pairs the
// MMA reads from that column.
__device__ __forceinline__ void convert_store(const uint4 codes, uint32_t taddr) {
  uint32_t wa[32];
  const uint32_t wv[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    // word w: weights 16w + 4s + j in byte j at bits 2s
    const uint32_t x01 = __byte_perm(wv[w], 0, 0x4140);
    const uint32_t x23 = __byte_perm(wv[w], 0, 0x4342);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      wa[8 * w + 2 * s + 0] = x01 & (0x00030003u << (2 * s));
      wa[8 * w + 2 * s + 1] = x23 & (0x00030003u << (2 * s));
    }
  }
  tmem_st32(taddr, wa);
}

template <bool kGroupSums>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_ws_kernel(const WsArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sIn = smem;                                                         // [in][slot]
  uint8_t* sAc = smem + kInStages * kInBytes;                                  // [4096]
  float* sdw = reinterpret_cast<float*>(sAc + kACorrBytes);                    // [scale][2][128]
  float* sdx = sdw + kScaleStages * kGPB * kM;                                 // [scale][64]
  uint64_t* in_full = reinterpret_cast<uint64_t*>(sdx + kScaleStages * kN);    // [in]
  uint64_t* in_empty = in_full + kInStages;                                    // [in]
  // mma_ready[s]: the MMAs of block b (stage s = b % 2) may go: the converters
  // have written A(b) and the epilogue has read the accumulators of b - 2 (one
  // barrier, so the issuing thread waits once per block; the epilogue
  // pre-arrives for blocks 0 and 1).
  uint64_t* mma_ready = in_empty + kInStages;                                  // [A]
  uint64_t* a_free = mma_ready + kAStages;                                     // [A]
  uint64_t* mma_done = a_free + kAStages;                                      // [acc]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + kAccStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.ngroups;
  const int nb = G / kGPB;                                // q8_K blocks
  const int64_t rb0 = (int64_t)blockIdx.x * kTilesPerCta;
  const int64_t nt = blockIdx.y;
  const int64_t tok0 = nt * kN;

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid < kM) {
    // constant correction A: row r, k0 = -2^-9, k1 = -2^-15 (subnormal), rest 0
    uint8_t* r = sAc + (tid >> 3) * kSBOc + (tid & 7) * 16;
    *reinterpret_cast<uint4*>(r) = make_uint4(0x82009800u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(r + kLBO) = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (tid == 0) {
    // Consumer warps arrive once per warp (lane 0, after __syncwarp).
    for (int i = 0; i < kInStages; ++i) {
      mbarrier_init(smem_u32(in_full + i), 1);
      // converters have read the slot's weights and scales, the MMAs its B
      mbarrier_init(smem_u32(in_empty + i), kConvWarps + 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbarrier_init(smem_u32(mma_ready + s), kConvWarps + kEpiWarps);
      mbarrier_init(smem_u32(a_free + s), 1);
      mbarrier_init(smem_u32(mma_done + s), 1);
    }
    mbarrier_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp == kProdWarp) {
    // ---------------- producer: stage block j into slot j % kInStages
    if (lane == 0) {
      int nvalid = 0;                                     // weight tiles that exist
      for (int q = 0; q < kTilesPerCta; ++q) nvalid += (rb0 + q < a.nrb) ? 1 : 0;
      const uint64_t policy = l2_evict_first_policy();
      pdl_wait_primary();   // the workspace is written by the previous kernel (the pre-pass)
      int i = 0;
      uint32_t ph = 0;
      for (int j = 0; j < nb; ++j) {
        // the slot is free once the converters and the MMAs of block j - kInStages are done
        if (j >= kInStages &&
            !mbarrier_wait_bounded(smem_u32(in_empty + i), ph ^ 1u, kWaitLimitNs)) {
          failed = true;
          break;
        }
        uint8_t* st = sIn + i * kInBytes;
        const uint32_t full = smem_u32(in_full + i);
        const int g0 = j * kGPB;
        mbarrier_arrive_expect_tx(full, (uint32_t)(kInW + nvalid * kWRun + kDxBytes));
        bulk_copy_g2s(smem_u32(st + kInB), a.Bt + (nt * G + g0) * (int64_t)kBTile, kInW, full,
                      policy);
        for (int q = 0; q < nvalid; ++q)
          bulk_copy_g2s(smem_u32(st + kInW + q * kWRun), a.Wtq + ((rb0 + q) * G + g0) * kTileBytes,
                        kWRun, full, policy);
        bulk_copy_g2s(smem_u32(st + kInDx), a.Dx + (nt * a.nblk + j) * kN, kDxBytes, full,
                      policy);
        if (++i == kInStages) { i = 0; ph ^= 1u; }
      }
    }
  } else if (warp < kConvWarps) {
    // ---------------- converters
    const int q4 = warp & 3, khalf = warp >> 2;          // row quarter, k half of A
    const bool row_ok = rb0 + q4 < a.nrb;
    const int ct = warp * 32 + lane;                      // 0..255; ct < 64 copies scales
    const uint32_t a_base = tmem + ((uint32_t)(q4 * 32) << 16) + kACol + (uint32_t)khalf * 32;
    int i = 0, sa = 0, ss = 0;
    uint32_t pin = 0, pa = 0;
    for (int b = 0; b < nb; ++b) {
      if (!failed && !mbarrier_wait_bounded(smem_u32(in_full + i), pin, kWaitLimitNs)) failed = true;
      const uint8_t* st = sIn + i * kInBytes;
      const uint8_t* tile = st + kInW + q4 * kWRun;
      uint4 c0 = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);  // w = 0
      uint4 c1 = c0;
      uint32_t sc0 = 0u, sc1 = 0u;
      float dx = 0.0f;
      if (!failed) {
        if (row_ok) {
          c0 = *reinterpret_cast<const uint4*>(tile + khalf * 512 + lane * 16);
          c1 = *reinterpret_cast<const uint4*>(tile + kTileBytes + khalf * 512 + lane * 16);
          if (khalf == 0) {
            sc0 = *reinterpret_cast<const uint16_t*>(tile + kTileCodeBytes + lane * 2);
            sc1 = *reinterpret_cast<const uint16_t*>(tile + kTileBytes + kTileCodeBytes + lane * 2);
          }
        }
        if (ct < kN) dx = reinterpret_cast<const float*>(st + kInDx)[ct];
      }
      __syncwarp();
      if (lane == 0) mbarrier_arrive(smem_u32(in_empty + i));
      if (++i == kInStages) { i = 0; pin ^= 1u; }

      // A stage sa is free once the MMAs of block b - kAStages have finished
      if (b >= kAStages && !failed &&
          !mbarrier_wait_bounded(smem_u32(a_free + sa), pa ^ 1u, kWaitLimitNs))
        failed = true;
      failed = __any_sync(0xffffffffu, failed);   // tcgen05.st below is warp-wide
      tc_fence_after();
      if (!failed) {
        const uint32_t ta = a_base + (uint32_t)sa * kBlkCols;
        convert_store(c0, ta);
        convert_store(c1, ta + kN);
        if (khalf == 0) {
          sdw[(ss * kGPB + 0) * kM + q4 * 32 + lane] =
              __half2float(__ushort_as_half((unsigned short)sc0)) * kProdScale;
          sdw[(ss * kGPB + 1) * kM + q4 * 32 + lane] =
              __half2float(__ushort_as_half((unsigned short)sc1)) * kProdScale;
        }
        if (ct < kN) sdx[ss * kN + ct] = dx;
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbarrier_arrive(smem_u32(mma_ready + sa));
      if (++sa == kAStages) { sa = 0; pa ^= 1u; }
      if (++ss == kScaleStages) ss = 0;
    }
  } else if (warp < kMmaWarp) {
    // ---------------- epilogue
    const int ew = warp - kConvWarps;
    const int q4 = ew & 3, nhalf = ew >> 2;               // row quarter, token half
    const int64_t row = (rb0 + q4) * kTileRows + lane;
    const int n0 = nhalf * 32;
    const uint32_t acc_base = tmem + ((uint32_t)(q4 * 32) << 16) + kAccCol + (uint32_t)n0;
    uint64_t y2[16];                                      // tokens n0 + 2p, +1
#pragma unroll
    for (int p = 0; p < 16; ++p) y2[p] = 0ull;
    int c = 0, ss = 0;
    uint32_t pc = 0;
    if (lane == 0) {   // both accumulator stages start free (blocks 0 and 1)
      for (int s = 0; s < kAccStages; ++s) mbarrier_arrive(smem_u32(mma_ready + s));
    }
    for (int b = 0; b < nb; ++b) {
      if (!failed && !mbarrier_wait_bounded(smem_u32(mma_done + c), pc, kWaitLimitNs)) failed = true;
      failed = __any_sync(0xffffffffu, failed);   // tcgen05.ld below is warp-wide
      tc_fence_after();
      if (!failed) {
        const uint32_t tc0 = acc_base + (uint32_t)c * kBlkCols;
        if (kGroupSums) {
#pragma unroll
          for (int gi = 0; gi < kGPB; ++gi) {
            uint32_t acc[32];
            tmem_ld32(tc0 + (uint32_t)gi * kN, acc);
            if (row < a.rows) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int64_t t = tok0 + n0 + j;
                if (t < a.ntok)
                  a.S[(t * a.rows + row) * G + b * kGPB + gi] =
                      __float2int_rn(__uint_as_float(acc[j]) * kProdScale);
              }
            }
          }
        } else {
          const float dw0 = sdw[(ss * kGPB + 0) * kM + q4 * 32 + lane];
          const float dw1 = sdw[(ss * kGPB + 1) * kM + q4 * 32 + lane];
          const uint64_t w0 = f2_packf(dw0, dw0), w1 = f2_packf(dw1, dw1);
          const float4* dx4 = reinterpret_cast<const float4*>(sdx + ss * kN + n0);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t a0[16], a1[16];
            tmem_ld16_nowait(tc0 + (uint32_t)h * 16, a0);
            tmem_ld16_nowait(tc0 + kN + (uint32_t)h * 16, a1);
            tmem_wait_ld();
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 d = dx4[h * 4 + j4];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int j = 4 * j4 + 2 * e;             // token pair n0 + 16h + j, +1
                const uint64_t z = f2_fma(w1, f2_pack(a1[j], a1[j + 1]),
                                          f2_mul(w0, f2_pack(a0[j], a0[j + 1])));
                const uint64_t dxp = e == 0 ? f2_packf(d.x, d.y) : f2_packf(d.z, d.w);
                y2[8 * h + j / 2] = f2_fma(dxp, z, y2[8 * h + j / 2]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbarrier_arrive(smem_u32(mma_ready + c));   // for block b + 2
      if (++c == kAccStages) { c = 0; pc ^= 1u; }
      if (++ss == kScaleStages) ss = 0;
    }
    if (!kGroupSums && !failed && row < a.rows) {
#pragma unroll
      for (int p = 0; p < 16; ++p) {
        const float2 v = f2_unpack(y2[p]);
        const int64_t t = tok0 + n0 + 2 * p;
        if (t < a.ntok) a.Y[t * a.rows + row] = v.x;
        if (t + 1 < a.ntok) a.Y[(t + 1) * a.rows + row] = v.y;
      }
    }
  } else if (lane == 0) {
    // ---------------- MMA issuer
    const uint64_t ac_desc = smem_desc(smem_u32(sAc), kLBO, kSBOc);
    int i = 0, sa = 0, c = 0;
    uint32_t pa = 0;
    for (int b = 0; b < nb; ++b) {
      // A(b) written and the accumulators of block b - 2 read
      if (!failed && !mbarrier_wait_bounded(smem_u32(mma_ready + sa), pa, kWaitLimitNs)) failed = true;
      tc_fence_after();
      if (!failed) {
        const uint32_t d = tmem + kAccCol + (uint32_t)c * kBlkCols;
        const uint32_t at = tmem + kACol + (uint32_t)sa * kBlkCols;
        // Descriptors of this slot, once: the start address field (bits 0-13,
        // address >> 4) then advances by plain adds, as no address passes 2^18.
        const uint32_t b0 = smem_u32(sIn + i * kInBytes + kInB);
        const uint64_t bd0 = smem_desc(b0, kLBO, kSBO);
        const uint64_t cd0 = smem_desc(b0 + kBMain, kLBO, kSBOc);
#pragma unroll
        for (int gi = 0; gi < kGPB; ++gi) {
#pragma unroll
          for (int kk = 0; kk < kGroup / 16; ++kk)
            mma_f16_tmem_a(d + gi * kN, at + gi * kN + 8 * kk,
                           bd0 + (uint64_t)((gi * kBTile + kk * 2 * kLBO) >> 4), kIdesc,
                           kk > 0 ? 1u : 0u);
          mma_f16_ss(d + gi * kN, ac_desc, cd0 + (uint64_t)((gi * kBTile) >> 4), kIdesc, 1u);
        }
      }
      // the commits fire when these MMAs are done (at once if none were issued)
      mma_commit(smem_u32(mma_done + c));
      mma_commit(smem_u32(a_free + sa));
      mma_commit(smem_u32(in_empty + i));
      if (++i == kInStages) i = 0;
      if (++sa == kAStages) { sa = 0; pa ^= 1u; }
      if (++c == kAccStages) c = 0;
    }
  }

  if (failed) atomicExch(a.status, kDevTimeout);
  // After a failure, staged copies may still be in flight: let the last use of
  // each input slot land before shared memory is released.
  if (__syncthreads_or(failed) && warp == kProdWarp && lane == 0) {
    for (int i = 0; i < kInStages && i < nb; ++i) {
      const int last = i + (nb - 1 - i) / kInStages * kInStages;
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
