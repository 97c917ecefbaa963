// tq_gemv.cu -- ternary x q8_K product for 1..16 tokens, bound by the weight
// stream from HBM.
//
// Decode reads every weight once per token batch, so the bus is the limit
// (ternary post, "did it reach the wall?" and "prefill wants a different
// shape"). The kernel streams the repacked weights once for all tokens:
//   - each CTA owns a contiguous range of 32-row tile columns; its weights are
//     one contiguous byte range, streamed through a ring of shared-memory
//     stages with 1-D TMA bulk copies (cp.async.bulk, 16 or more tiles of
//     1088 bytes per copy), each completed on a "full" mbarrier; the last of
//     the warps to release a slot refills it, so no warp waits for another;
//   - the warps (8 for one token, 16 for more) each take tiles of a stage:
//     the same 32 rows, different 128-weight groups. Lane l is row l, so no
//     lane ever needs a cross-lane reduction of dot products; the warps'
//     partial sums of a row are added in shared memory once per tile column,
//     in a fixed order (deterministic output);
//   - the activations of all tokens sit in shared memory; every lane of a warp
//     reads the same 16 bytes at once (a broadcast);
//   - unpacking a 32-bit weight word (16 weights) is one AND per dp4a operand:
//     word & (0x03030303 << 2s) is 4 consecutive weights times 4^s, and slot s
//     accumulates in its own register (post, "the trick with 4 and 16"); the
//     unsigned x signed dp4a takes slot 3 (up to 128) without a shift;
//   - once per 128 weights: dot(u,q) = a0 + a1/4 + a2/16 + a3/64 (exact shifts),
//     minus the sum of the group's activations from the q8_K partial sums turns
//     u back into w (dot(w,y) = dot(u,y) - sum(y)), and one f32 FMA applies
//     d_w * d_x;
//   - launched as a programmatic dependent: when the previous kernel writes no
//     weights, the first weight stages are requested before waiting for it;
//     a GEMV lets the next kernel start only after its own wait, so in a
//     captured chain of GEMVs whose inputs the previous GEMV does not write,
//     the host lets a launch read everything first and wait only before its
//     first store (launch_gemv, defer_wait);
//   - where the activations of all tokens do not fit in shared memory, one
//     launch per half of the tokens.
#include <algorithm>

#include "tq_tcgen05.cuh"

namespace tq {
namespace {

// Compile-time tuning: warps per CTA (one token / more tokens), tiles each
// warp takes from a stage, the deepest ring, the most CTAs on one SM, and
// whether the grid should split the tile columns evenly.
#ifndef TQ_GEMV_WARPS_T1
#define TQ_GEMV_WARPS_T1 8
#endif
#ifndef TQ_GEMV_WARPS
#define TQ_GEMV_WARPS 16
#endif
#ifndef TQ_GEMV_TILES_PER_WARP_T1
#define TQ_GEMV_TILES_PER_WARP_T1 4
#endif
#ifndef TQ_GEMV_TILES_PER_WARP
#define TQ_GEMV_TILES_PER_WARP 2
#endif
#ifndef TQ_GEMV_MAX_STAGES
#define TQ_GEMV_MAX_STAGES 2
#endif
#ifndef TQ_GEMV_CTAS_PER_SM
#define TQ_GEMV_CTAS_PER_SM 2
#endif
#ifndef TQ_GEMV_EVEN_GRID
#define TQ_GEMV_EVEN_GRID 1
#endif

constexpr int kMaxTok = 16;         // tokens the GEMV takes (in one launch up to 8 with dp4a)
constexpr int kMaxDp4aTok = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Per token count: warps (each owns tiles of every stage), stage size, and
// how many CTAs the register budget is planned for.
template <int T>
struct Cfg {
  static constexpr int kWarps = T == 1 ? TQ_GEMV_WARPS_T1 : TQ_GEMV_WARPS;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kTilesPerWarp = T == 1 ? TQ_GEMV_TILES_PER_WARP_T1 : TQ_GEMV_TILES_PER_WARP;
  static constexpr int kStageTiles = kWarps * kTilesPerWarp;
  static constexpr int kStageBytes = kStageTiles * kTileBytes;
  static constexpr int kMinCtas = (T == 1 && kThreads <= 512) ? TQ_GEMV_CTAS_PER_SM : 1;
};

struct GemvArgs {
  const uint8_t* Wtq;
  const uint8_t* Xq;
  float* Y;
  int32_t* S;
  int* status;
  int rows;
  int ngroups;        // cols / 128
  int nblk;           // cols / 256
  int nrb;            // 32-row tile columns
  int stages;         // ring depth
  int early_weights;  // 1: the previous kernel does not write Wtq; prefetch before waiting
  const float* X;     // fused form: f32 activations [T][cols] quantized here (else null)
  uint8_t* Xq_out;    // fused form: where the q8_K blocks are written (may be null)
  int defer;          // the inputs are final when the kernel starts: wait for the
                      // previous kernel only after the first tile column (1) or
                      // after the first ring stage (2), before any global write
  int stall;          // test facility: CTA 0 requests no weight stage, so its
                      // waits expire after stall_ns (tq_debug_stall_next_launch)
  uint64_t stall_ns;
  const uint8_t* Xs = nullptr;  // mma.sync GEMV: the activations already staged by the
                      // staging kernel (the shared-memory image of the f16
                      // rows, group sums and scales), or null to stage here
};

// Fused form: quantizes the T x cols f32 activations block by block (warp per
// q8_K block, q8K_warp, so the bytes equal the quantizer kernel's), four
// blocks per warp whose loads are issued together, and hands each block to
// store(tb, w0, w1, s8, d) on every lane of the warp. CTA 0 also writes the
// q8_K blocks to a.Xq_out, unless the kernel defers its writes (then each CTA
// writes some of them from shared memory after its wait).
template <class Store>
__device__ __forceinline__ void stage_quantize(const GemvArgs& a, int nblocks, int warp,
                                               int nwarps, int lane, Store store) {
  const bool write_xq = a.Xq_out != nullptr && blockIdx.x == 0 && !a.defer;
  for (int tb0 = warp; tb0 < nblocks; tb0 += 4 * nwarps) {
    float4 va[4], vb[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tb = tb0 + c * nwarps;
      if (tb < nblocks) {
        const float4* src = reinterpret_cast<const float4*>(a.X + (int64_t)tb * kQK) + 2 * lane;
        va[c] = __ldg(src);
        vb[c] = __ldg(src + 1);
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tb = tb0 + c * nwarps;
      if (tb < nblocks) {   // warp-uniform
        uint32_t w0, w1;
        int s8;
        float d;
        q8K_warp(va[c], vb[c], w0, w1, s8, d);
        store(tb, w0, w1, s8, d);
        if (write_xq) q8K_store(a.Xq_out + (int64_t)tb * kQ8KBytes, lane, w0, w1, s8, d);
      }
    }
  }
}

// Sum of s8 over the 16 lanes of each half-warp (one 128-value half-block),
// valid on lanes 0 and 16.
__device__ __forceinline__ int half_block_sum(int s8) {
  s8 += __shfl_xor_sync(0xffffffffu, s8, 1);
  s8 += __shfl_xor_sync(0xffffffffu, s8, 2);
  s8 += __shfl_xor_sync(0xffffffffu, s8, 4);
  s8 += __shfl_xor_sync(0xffffffffu, s8, 8);
  return s8;
}

struct GroupCodes {
  uint4 lo, hi;     // weights 0..63 and 64..127 of this lane's row
  uint32_t scale;   // fp16 bits of d_w (low half)
};


template <int T, bool kGroupSums>
__device__ __forceinline__ void group_dot(const GroupCodes& c, int g, const int8_t* sq,
                                          const int* sgsum, const float* sdx, const GemvArgs& a,
                                          int row, float (&y)[T]) {
  const uint32_t wv[8] = {c.lo.x, c.lo.y, c.lo.z, c.lo.w, c.hi.x, c.hi.y, c.hi.z, c.hi.w};
  const float dw = __half2float(__ushort_as_half((unsigned short)c.scale));
  const int cols = a.ngroups * kGroup;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    // activations of group g, token t: 32 words; word 4i+s pairs with slot s of weight word i
    const int4* qa = reinterpret_cast<const int4*>(sq + t * cols + g * kGroup);
    int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int4 q = qa[i];
      a0 = dp4a_us(wv[i] & 0x03030303u, q.x, a0);
      a1 = dp4a_us(wv[i] & 0x0C0C0C0Cu, q.y, a1);
      a2 = dp4a_us(wv[i] & 0x30303030u, q.z, a2);
      a3 = dp4a_us(wv[i] & 0xC0C0C0C0u, q.w, a3);
    }
    const int isum = a0 + (a1 >> 2) + (a2 >> 4) + (a3 >> 6) - sgsum[t * a.ngroups + g];
    if (kGroupSums) {
      if (row < a.rows) a.S[((int64_t)t * a.rows + row) * a.ngroups + g] = isum;
    } else {
      y[t] = fmaf(dw * sdx[t * a.nblk + (g >> 1)], (float)isum, y[t]);
    }
  }
}

// Shared memory: [ring][full bars][red-full bars][red-empty bars][slot counters]
// [q8 values][group sums][scales][partial sums]
struct SmemPlan {
  int64_t ring, bars, counters, sq, sgsum, sdx, red, table, total;
};

// Weight formats the dp4a GEMV streams: the tq tiles (2 bits per weight) or
// the ptq1_0 stream tiles (1.75 bits, decoded in the kernel).
constexpr int kFmtTq = 0;
constexpr int kFmtPtq1 = 1;
template <int F>
__host__ __device__ constexpr int fmt_tile_bytes() { return F == kFmtPtq1 ? kTq1TileBytes : kTileBytes; }

template <int T, int F = kFmtTq>
__host__ __device__ inline SmemPlan plan_smem(int stages, int64_t cols) {
  SmemPlan p;
  const int64_t g = cols / kGroup, b = cols / kQK;
  p.ring = 0;
  p.bars = (int64_t)stages * Cfg<T>::kStageTiles * fmt_tile_bytes<F>();   // full[S], redfull[2], redempty[2]
  p.counters = p.bars + (stages + 4) * 8;                  // int[S] released, int[S] issued
  p.sq = (p.counters + stages * 8 + 15) / 16 * 16;
  p.sgsum = p.sq + T * cols;
  p.sdx = p.sgsum + T * g * 4;
  p.red = p.sdx + T * b * 4;
  p.table = p.red + (int64_t)2 * Cfg<T>::kWarps * T * 32 * 4;
  p.total = p.table + (F == kFmtPtq1 ? 256 * 4 : 0);   // byte -> five 2-bit codes
  return p;
}

// The five trits of every byte value as 2-bit codes, trit n at bits 2n.
__device__ __forceinline__ uint32_t ptq1_codes(uint32_t b) {
  uint32_t v = 0;
#pragma unroll
  for (int n = 0; n < 5; ++n) v |= ptq1_trit(b, n) << (2 * n);
  return v;
}

// One row's ptq1_0 block of a stream tile (28 bytes: fp16 scale, then 26
// code bytes of five weights each) -> the 128 codes as a 2-bit stream, weight
// k at bits 2 (k % 16) of word k / 16, through the 256-entry table; the last
// code byte's two unused trits fall past the stream.
__device__ __forceinline__ void ptq1_decode(const uint8_t* blk, const uint32_t* table,
                                            uint4& lo, uint4& hi, uint32_t& scale) {
  uint32_t bw[kPtq1Bytes / 4];
#pragma unroll
  for (int i = 0; i < kPtq1Bytes / 4; ++i) bw[i] = reinterpret_cast<const uint32_t*>(blk)[i];
  uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
  for (int c = 0; c < kPtq1Bytes - 2; ++c) {
    const uint32_t v = table[(bw[(2 + c) >> 2] >> (8 * ((2 + c) & 3))) & 0xFFu];
    const int bit = 10 * c;
    w[bit >> 5] |= v << (bit & 31);
    if ((bit & 31) > 22 && (bit >> 5) + 1 < 8) w[(bit >> 5) + 1] |= v >> (32 - (bit & 31));
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
  scale = bw[0] & 0xFFFFu;
}

// Four words of 16 int8 activations x0..x15 -> slot-major order: word s holds
// x_s, x_{s+4}, x_{s+8}, x_{s+12}, the activations that a 2-bit stream word's
// slot s (bits 2s of each byte) multiplies.
__device__ __forceinline__ uint4 act_slot_major(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  const uint32_t t0 = __byte_perm(w0, w1, 0x5140), t1 = __byte_perm(w2, w3, 0x5140);
  const uint32_t t2 = __byte_perm(w0, w1, 0x7362), t3 = __byte_perm(w2, w3, 0x7362);
  return make_uint4(__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632),
                    __byte_perm(t2, t3, 0x5410), __byte_perm(t2, t3, 0x7632));
}

template <int T, bool kGroupSums, int F = kFmtTq>
__global__ void __launch_bounds__(Cfg<T>::kThreads, Cfg<T>::kMinCtas) gemv_kernel(const GemvArgs a) {
  constexpr int kConsumers = Cfg<T>::kWarps;
  constexpr int kStageTiles = Cfg<T>::kStageTiles;
  constexpr int kTileB = fmt_tile_bytes<F>();
  constexpr int kStageBytes = kStageTiles * kTileB;
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = a.stages;
  const int cols = a.ngroups * kGroup;
  const SmemPlan pl = plan_smem<T, F>(S, cols);
  uint8_t* ring = smem + pl.ring;                                 // [S][stage]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.bars);  // [S]
  uint64_t* redfull = full + S;                                   // [2]
  uint64_t* redempty = redfull + 2;                               // [2]
  int* released = reinterpret_cast<int*>(smem + pl.counters);    // [S]
  int* issued = released + S;                                    // [S] copies per slot
  int8_t* sq = reinterpret_cast<int8_t*>(smem + pl.sq);           // [T][cols]
  int* sgsum = reinterpret_cast<int*>(smem + pl.sgsum);           // [T][ngroups]
  float* sdx = reinterpret_cast<float*>(smem + pl.sdx);           // [T][nblk]
  float* red = reinterpret_cast<float*>(smem + pl.red);           // [2][kConsumers][T][32]
  uint32_t* table = reinterpret_cast<uint32_t*>(smem + pl.table); // [256] (ptq1_0 stream)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's tile columns, and the bulk copies (stages) that cover them
  const int rb0 = (int)((int64_t)blockIdx.x * a.nrb / gridDim.x);
  const int rb1 = (int)((int64_t)(blockIdx.x + 1) * a.nrb / gridDim.x);
  const int per_rb = (a.ngroups + kStageTiles - 1) / kStageTiles;
  const int nstage = (rb1 - rb0) * per_rb;
  const uint64_t policy = l2_evict_first_policy();
  const bool stalled = a.stall && blockIdx.x == 0;
  const uint64_t lim = stalled ? a.stall_ns : kWaitLimitNs;   // bound of the stream's waits

  // Stage j of this CTA covers tile column rb0 + j / per_rb, groups from
  // (j % per_rb) * kStageTiles; it lands in ring slot j % S. Counters below
  // advance these incrementally (no division in the loop).
  auto issue = [&](int slot, int rb, int st) {
    const int gs = st * kStageTiles;
    const uint32_t bytes = (uint32_t)(min(kStageTiles, a.ngroups - gs) * kTileB);
    const uint32_t bar = smem_u32(full + slot);
    ++issued[slot];   // one thread at a time per slot: the ring protocol orders them
    mbarrier_arrive_expect_tx(bar, bytes);
    bulk_copy_g2s(smem_u32(ring + (size_t)slot * kStageBytes),
                  a.Wtq + ((int64_t)rb * a.ngroups + gs) * kTileB, bytes, bar, policy);
  };
  auto issue_first = [&]() {
    if (stalled) return;
    int rb = rb0, st = 0;
    for (int j = 0; j < min(S, nstage); ++j) {
      issue(j, rb, st);
      if (++st == per_rb) { st = 0; ++rb; }
    }
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbarrier_init(smem_u32(full + i), 1);
      released[i] = 0;
      issued[i] = 0;
    }
    for (int i = 0; i < 2; ++i) {
      mbarrier_init(smem_u32(redfull + i), kConsumers);
      mbarrier_init(smem_u32(redempty + i), T);
    }
    mbarrier_init_fence();
    // When the previous kernel in the stream writes no weights, the first
    // stages go out before waiting for it.
    if (a.early_weights) issue_first();
  }
  // The activations may come from the previous kernel: wait for it first,
  // unless the host has shown they do not (defer). Either way the next kernel
  // is let in only after this kernel's wait, so when it starts, only this
  // kernel can still be running before it.
  if (!a.defer) {
    pdl_wait_primary();
    pdl_launch_dependents();
  }
  if (threadIdx.x == 0 && !a.early_weights) issue_first();

  // Stage q8_K activations, every thread issuing independent loads: qs as a
  // dense int8 [T][cols] array (block tb = t * nblk + b lands at tb * 256), the
  // sum of each 128-value half-block (8 partial sums), and the block scales.
  // The fused form quantizes a.X into the same arrays instead.
  if (a.X) {
    stage_quantize(a, T * a.nblk, warp, kConsumers, lane,
                   [&](int tb, uint32_t w0, uint32_t w1, int s8, float d) {
                     reinterpret_cast<uint2*>(sq + tb * kQK)[lane] = make_uint2(w0, w1);
                     const int hs = half_block_sum(s8);
                     if ((lane & 15) == 0) sgsum[2 * tb + (lane >> 4)] = hs;
                     if (lane == 0) sdx[tb] = d;
                   });
  } else if (F == kFmtPtq1) {
    // 16 activations per thread, stored slot-major for the 2-bit stream words
    const int nc = T * a.nblk * (kQK / 16);
    for (int c = threadIdx.x; c < nc; c += Cfg<T>::kThreads) {
      const int tb = c >> 4, k = c & 15;
      const uint32_t* src =
          reinterpret_cast<const uint32_t*>(a.Xq + (int64_t)tb * kQ8KBytes + kQ8KQsOffset) + 4 * k;
      reinterpret_cast<uint4*>(sq + tb * kQK)[k] =
          act_slot_major(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
    }
    for (int i = threadIdx.x; i < 256; i += Cfg<T>::kThreads) table[i] = ptq1_codes((uint32_t)i);
  } else {
    const int nw = T * a.nblk * (kQK / 4);
#pragma unroll 4
    for (int w = threadIdx.x; w < nw; w += Cfg<T>::kThreads) {
      const int tb = w >> 6, k = w & 63;
      reinterpret_cast<uint32_t*>(sq + tb * kQK)[k] = __ldg(
          reinterpret_cast<const uint32_t*>(a.Xq + (int64_t)tb * kQ8KBytes + kQ8KQsOffset) + k);
    }
  }
  if (!a.X) {
    for (int h = threadIdx.x; h < T * a.nblk * 2; h += Cfg<T>::kThreads) {
      const int tb = h >> 1, half = h & 1;
      const uint8_t* blk = a.Xq + (int64_t)tb * kQ8KBytes;
      const int16_t* bs = reinterpret_cast<const int16_t*>(blk + kQ8KBsumsOffset) + half * 8;
      int sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += __ldg(bs + i);
      sgsum[h] = sum;   // = sgsum[t * ngroups + 2 * b + half]
      if (half == 0) sdx[tb] = __ldg(reinterpret_cast<const float*>(blk));
    }
  }
  __syncthreads();

  // Deferred form: the wait (and the next kernel's start) comes after the
  // first ring stage's or the first tile column's dot products, before any
  // global write; then this CTA's share of the q8_K blocks goes out from the
  // staged copy.
  bool waited = !a.defer;
  auto finish_wait = [&]() {
    pdl_wait_primary();
    pdl_launch_dependents();
    if (a.X && a.Xq_out) {
      for (int tb = blockIdx.x + warp * gridDim.x; tb < T * a.nblk; tb += gridDim.x * kConsumers) {
        const uint2 q = reinterpret_cast<const uint2*>(sq + tb * kQK)[lane];
        const int s8 = __dp4a((int)q.x, 0x01010101, 0) + __dp4a((int)q.y, 0x01010101, 0);
        q8K_store(a.Xq_out + (int64_t)tb * kQ8KBytes, lane, q.x, q.y, s8, sdx[tb]);
      }
    }
    waited = true;
  };

  bool failed = false;
  int j = 0, slot = 0;
  uint32_t phase = 0;
  for (int rb = rb0, i = 0; rb < rb1; ++rb, ++i) {
    const int row = rb * kTileRows + lane;
    float y[T];
#pragma unroll
    for (int t = 0; t < T; ++t) y[t] = 0.0f;
    for (int st = 0; st < per_rb; ++st, ++j) {
      const int gs = st * kStageTiles;
      const int nt = min(kStageTiles, a.ngroups - gs);
      if (!failed && !mbarrier_wait_bounded(smem_u32(full + slot), phase, lim))
        failed = true;
      // this warp's tiles of the stage: warp, warp + 16, ... (spread for short stages)
      GroupCodes c[Cfg<T>::kTilesPerWarp];
#pragma unroll
      for (int u = 0; u < Cfg<T>::kTilesPerWarp; ++u) {
        const int tl = warp + u * kConsumers;
        if (!failed && tl < nt) {
          const uint8_t* tile = ring + (size_t)slot * kStageBytes + tl * kTileB;
          if (F == kFmtPtq1) {
            ptq1_decode(tile + lane * kPtq1Bytes, table, c[u].lo, c[u].hi, c[u].scale);
          } else {
            c[u].lo = *reinterpret_cast<const uint4*>(tile + lane * 16);
            c[u].hi = *reinterpret_cast<const uint4*>(tile + 512 + lane * 16);
            c[u].scale = *reinterpret_cast<const uint16_t*>(tile + kTileCodeBytes + lane * 2);
          }
        }
      }
      __syncwarp();   // the whole warp has read its tile: release the slot
      if (lane == 0) {
        // the last of the warps to release a slot refills it (nobody waits)
        __threadfence_block();
        if (atomicAdd(released + slot, 1) == kConsumers - 1) {
          released[slot] = 0;
          if (!failed && j + S < nstage) {
            int st2 = st + S, rb2 = rb;
            while (st2 >= per_rb) { st2 -= per_rb; ++rb2; }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(slot, rb2, st2);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < Cfg<T>::kTilesPerWarp; ++u) {
        const int tl = warp + u * kConsumers;
        if (!failed && tl < nt) group_dot<T, kGroupSums>(c[u], gs + tl, sq, sgsum, sdx, a, row, y);
      }
      if (++slot == S) { slot = 0; phase ^= 1u; }
      if (!waited && a.defer == 2) finish_wait();
    }
    if (!waited) finish_wait();
    if (!kGroupSums) {
      // The warps' partial sums of each row meet in shared memory; warp
      // (i*T + t) % warps adds those of token t in warp order (deterministic) and
      // stores them. Buffers alternate between tile columns; mbarriers order
      // the writers and the reducers, so no warp waits for all the others.
      const int p = i & 1;
      float* r = red + p * (kConsumers * T * 32);
      if (i >= 2 && !failed &&
          !mbarrier_wait_bounded(smem_u32(redempty + p), (uint32_t)(((i >> 1) - 1) & 1),
                                 lim))
        failed = true;
#pragma unroll
      for (int t = 0; t < T; ++t) r[(warp * T + t) * 32 + lane] = y[t];
      __syncwarp();
      if (lane == 0) mbarrier_arrive(smem_u32(redfull + p));
      const int t = (warp - i * T) & (kConsumers - 1);
      if (t < T) {
        if (!failed && !mbarrier_wait_bounded(smem_u32(redfull + p), (uint32_t)((i >> 1) & 1),
                                              lim))
          failed = true;
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < kConsumers; ++k) s += r[(k * T + t) * 32 + lane];
        if (!failed && row < a.rows) a.Y[(int64_t)t * a.rows + row] = s;
        __syncwarp();
        if (lane == 0) mbarrier_arrive(smem_u32(redempty + p));
      }
    }
  }
  if (!waited) finish_wait();   // a CTA without tile columns
  if (failed && lane == 0) atomicExch(a.status, kDevTimeout);
  // Copies can still be in flight only after a failed wait: then let the last
  // copy requested into each slot land before the CTA's shared memory is
  // released. A slot is refilled only by a warp that saw its previous copy
  // land, so at most that last one can be in flight; it completes phase
  // issued - 1 of the slot's barrier.
  if (__syncthreads_or(failed) && threadIdx.x == 0) {
    for (int sl = 0; sl < S; ++sl)
      if (issued[sl] > 0)
        mbarrier_wait_bounded(smem_u32(full + sl), (uint32_t)((issued[sl] - 1) & 1), kWaitLimitNs);
  }
}

// ---------------------------------------------------------------- 4..16 tokens
//
// With several tokens the dp4a loop pays one dot instruction per 4 weights
// per token. From TQ_GEMV_MMA_MIN_TOK tokens up this variant runs the group
// dot on the tensor cores with the warp-level mma.sync m16n8k16 (f16 in, f32
// out): measured on GB300 it sustains about 600 TFLOP/s, while tcgen05.mma
// takes about 23 ns per instruction for any N <= 64, too slow for 8 token
// columns, and int8 mma.sync runs at about 160 TOP/s. Same stream, same ring,
// same work split; per 32-row tile and group a warp issues 2 x 8 MMAs (two
// 16-row halves, K = 16 each) over 8 token columns (zero beyond ntok).
//   - A (weights) costs one AND per two weights: code bits 2s..2s+1 in the low
//     byte of an f16 half with zero exponent make the subnormal u * 4^s * 2^-24,
//     exact (the tensor cores multiply subnormals exactly);
//   - B (activations) sits in shared memory as f16 q * 2^(9 - 2s), exact, so
//     every product is u * q * 2^-15; partial sums stay integer multiples of
//     2^-15 below 1, exact in f32;
//   - per group: isum = acc * 2^15 - sum(q) (exact), then y += d_w d_x isum.
// Lane layout of one MMA (groupID g8 = lane / 4, q = lane % 4): A rows g8 and
// g8 + 8 of the half, weights 16q + 4s + {0,1} (registers a0, a1) and
// 16q + 4s + {2,3} (a2, a3) of code word q of a 64-weight half c; B token g8,
// the same four activations; C rows g8, g8 + 8, tokens 2q, 2q + 1.

// The tensor-core variant's shape: T's warps, and TPW tiles per warp and stage
// (two, or one where the larger ring and the activations do not fit in
// shared memory). Up to 8 tokens fill the 8 columns of one MMA and the
// activations sit in shared memory as f16 already scaled for their slot;
// 9 to 16 tokens take two MMAs of 8 columns per weight fragment (the weights
// stream once for all of them), and, since 16 rows of f16 activations would
// leave no room for the weight ring, the activations sit there as int8 and
// each B fragment is converted when it is used (exactly).
template <int T, int TPW>
struct MmaCfg {
  static constexpr int kWarps = Cfg<(T > 8 ? 8 : T)>::kWarps;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kTilesPerWarp = TPW;
  static constexpr int kStageTiles = kWarps * TPW;
  static constexpr int kStageBytes = kStageTiles * kTileBytes;
  static constexpr int kNB = (T + 7) / 8;        // 8-column token blocks
  static constexpr bool kI8 = T > 8;             // int8 activations in shared memory
  static constexpr int kReducers = 8 * kNB;      // C positions per lane, one reducing warp each
  static_assert(kReducers <= kWarps, "one reducing warp per C position");
};

struct MmaPlan {
  int64_t ring, bars, counters, sb, sgsum, sdx, red, total;
  int64_t sb_stride;   // bytes per token row of f16 activations (+8: bank spread)
};

template <int T, int TPW>
__host__ __device__ inline MmaPlan plan_mma(int stages, int64_t cols) {
  MmaPlan p;
  const int64_t g = cols / kGroup, b = cols / kQK;
  // bytes per token row; the pad spreads the rows' fragments over the banks
  p.sb_stride = MmaCfg<T, TPW>::kI8 ? cols + 4 : cols * 2 + 8;
  p.ring = 0;
  p.bars = (int64_t)stages * MmaCfg<T, TPW>::kStageBytes;
  p.counters = p.bars + (stages + 5) * 8;                  // int[S] released, int[S] issued
  p.sb = (p.counters + stages * 8 + 15) / 16 * 16;
  p.sgsum = (p.sb + T * p.sb_stride + 15) / 16 * 16;
  p.sdx = p.sgsum + T * g * 4;
  p.red = (p.sdx + T * b * 4 + 15) / 16 * 16;
  p.total = p.red + (int64_t)2 * MmaCfg<T, TPW>::kWarps * MmaCfg<T, TPW>::kReducers * 32 * 4;
  return p;
}

// f16x2 bits of 2^(9 - 2s): the activation scale that matches code slot s.
__device__ __forceinline__ uint32_t mma_slot_scale(int s) {
  return s == 0 ? 0x60006000u : s == 1 ? 0x58005800u : s == 2 ? 0x50005000u : 0x48004800u;
}

__device__ __forceinline__ uint32_t h2_mul_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  // not volatile: a pure register operation the compiler may schedule freely
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 32-row tile x one group on the tensor cores; adds d_w d_x isum into y
// (y[4h + 2r + j]: half h, row g8 + 8r, token 2q + j) or stores isum.
// This lane's share of one 32-row tile and group: code word q of both 64-weight
// halves for rows g8, g8 + 8, g8 + 16, g8 + 24, and the four fp16 scales.
struct MmaCodes {
  uint32_t w[2][2][2];   // [code half][tile half][row g8 / g8 + 8]
  uint32_t sc[2][2];     // [tile half][row]
};

__device__ __forceinline__ void load_mma_codes(const uint8_t* tile, int lane, MmaCodes& m) {
  const int g8 = lane >> 2, q = lane & 3;
#pragma unroll
  for (int ch = 0; ch < 2; ++ch)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int r = 0; r < 2; ++r)
        m.w[ch][h][r] = *reinterpret_cast<const uint32_t*>(tile + ch * 512 + (16 * h + g8 + 8 * r) * 16 + q * 4);
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int r = 0; r < 2; ++r)
      m.sc[h][r] = *reinterpret_cast<const uint16_t*>(tile + kTileCodeBytes + (16 * h + g8 + 8 * r) * 2);
}

// One 32-row tile and group on the tensor cores: adds d_w d_x isum into y
// (y[8nb + 4h + 2r + j]: token block nb, half h, row g8 + 8r, token
// 8nb + 2q + j) or stores isum.
template <int T, bool kGroupSums>
__device__ __forceinline__ void group_mma(const MmaCodes& m, int g, const uint8_t* sb,
                                          int64_t sb_stride, const int* sgsum, const float* sdx,
                                          const GemvArgs& a, int row_base, int lane,
                                          float (&y)[8 * ((T + 7) / 8)]) {
  constexpr int NB = (T + 7) / 8;
  constexpr bool kI8 = T > 8;
  const int g8 = lane >> 2, q = lane & 3;
  // B: token 8nb + g8's activations of this group, as f16 rows in natural k
  // order (up to 8 tokens) or int8 (more)
  const uint8_t* brow[NB];
  bool tok_ok[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int tok = 8 * nb + g8;
    tok_ok[nb] = tok < T;
    brow[nb] = sb + (tok_ok[nb] ? tok : 0) * sb_stride +
               (kI8 ? (int64_t)g * kGroup + q * 16 : (int64_t)g * kGroup * 2 + q * 32);
  }
  float c[NB][2][4] = {};
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {   // 64-weight half of the group (code half)
    uint32_t x01[2][2], x23[2][2];   // [tile half][row g8 / g8 + 8]
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        x01[h][r] = __byte_perm(m.w[ch][h][r], 0, 0x4140);
        x23[h][r] = __byte_perm(m.w[ch][h][r], 0, 0x4342);
      }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t mk = 0x00030003u << (2 * s);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        uint2 bv = make_uint2(0u, 0u);
        if (tok_ok[nb]) {
          if (kI8) {
            // four int8 activations -> two exact f16 pairs, times 2^(9 - 2s)
            uint32_t lo, hi;
            tc::s8x4_to_h2x2(*reinterpret_cast<const uint32_t*>(brow[nb] + ch * 64 + s * 4), lo, hi);
            const uint32_t sc = mma_slot_scale(s);
            bv = make_uint2(h2_mul_rn(lo, sc), h2_mul_rn(hi, sc));
          } else {
            bv = *reinterpret_cast<const uint2*>(brow[nb] + ch * 128 + s * 8);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
          mma16816(c[nb][h], x01[h][0] & mk, x01[h][1] & mk, x23[h][0] & mk, x23[h][1] & mk, bv.x,
                   bv.y);
      }
    }
  }
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    // tokens 8nb + 2q, 8nb + 2q + 1 of this lane
    const int t0 = 8 * nb + 2 * q;
    int sq[2];
    float dx[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const bool ok = t0 + j < T;
      sq[j] = ok ? sgsum[(t0 + j) * a.ngroups + g] : 0;
      dx[j] = ok ? sdx[(t0 + j) * a.nblk + (g >> 1)] : 0.0f;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = row_base + 16 * h + g8 + 8 * r;
        const float dw =
            kGroupSums ? 0.0f : __half2float(__ushort_as_half((unsigned short)m.sc[h][r]));
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float isum = fmaf(c[nb][h][2 * r + j], 32768.0f, (float)(-sq[j]));   // exact
          if (kGroupSums) {
            if (t0 + j < T && row < a.rows)
              a.S[((int64_t)(t0 + j) * a.rows + row) * a.ngroups + g] = __float2int_rn(isum);
          } else {
            float& yy = y[8 * nb + 4 * h + 2 * r + j];
            yy = fmaf(dw * dx[j], isum, yy);
          }
        }
      }
  }
}

template <int T, bool kGroupSums, int TPW>
__global__ void __launch_bounds__(MmaCfg<T, TPW>::kThreads, 1) gemv_mma_kernel(const GemvArgs a) {
  using Mc = MmaCfg<T, TPW>;
  constexpr int kConsumers = Mc::kWarps;
  constexpr int kReducers = Mc::kReducers;
  constexpr int kStageTiles = Mc::kStageTiles;
  constexpr int kStageBytes = Mc::kStageBytes;
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = a.stages;
  const int cols = a.ngroups * kGroup;
  const MmaPlan pl = plan_mma<T, TPW>(S, cols);
  uint8_t* ring = smem + pl.ring;                                 // [S][stage]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.bars);  // [S]
  uint64_t* redfull = full + S;                                   // [2]
  uint64_t* redempty = redfull + 2;                               // [2]
  uint64_t* actfull = redempty + 2;                               // staged activations
  int* released = reinterpret_cast<int*>(smem + pl.counters);    // [S]
  int* issued = released + S;                                    // [S] copies per slot
  uint8_t* sb = smem + pl.sb;                                     // [T][cols] f16 (+8 B)
  int* sgsum = reinterpret_cast<int*>(smem + pl.sgsum);           // [T][ngroups]
  float* sdx = reinterpret_cast<float*>(smem + pl.sdx);           // [T][nblk]
  float* red = reinterpret_cast<float*>(smem + pl.red);           // [2][kConsumers][8][32]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb0 = (int)((int64_t)blockIdx.x * a.nrb / gridDim.x);
  const int rb1 = (int)((int64_t)(blockIdx.x + 1) * a.nrb / gridDim.x);
  const int per_rb = (a.ngroups + kStageTiles - 1) / kStageTiles;
  const int nstage = (rb1 - rb0) * per_rb;
  const uint64_t policy = l2_evict_first_policy();
  const bool stalled = a.stall && blockIdx.x == 0;
  const uint64_t lim = stalled ? a.stall_ns : kWaitLimitNs;   // bound of the stream's waits

  auto issue = [&](int slot, int rb, int st) {
    const int gs = st * kStageTiles;
    const uint32_t bytes = (uint32_t)(min(kStageTiles, a.ngroups - gs) * kTileBytes);
    const uint32_t bar = smem_u32(full + slot);
    ++issued[slot];   // one thread at a time per slot: the ring protocol orders them
    mbarrier_arrive_expect_tx(bar, bytes);
    bulk_copy_g2s(smem_u32(ring + (size_t)slot * kStageBytes),
                  a.Wtq + ((int64_t)rb * a.ngroups + gs) * kTileBytes, bytes, bar, policy);
  };
  auto issue_first = [&]() {
    if (stalled) return;
    int rb = rb0, st = 0;
    for (int j = 0; j < min(S, nstage); ++j) {
      issue(j, rb, st);
      if (++st == per_rb) { st = 0; ++rb; }
    }
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbarrier_init(smem_u32(full + i), 1);
      released[i] = 0;
      issued[i] = 0;
    }
    for (int i = 0; i < 2; ++i) {
      mbarrier_init(smem_u32(redfull + i), kConsumers);
      mbarrier_init(smem_u32(redempty + i), kReducers);
    }
    mbarrier_init(smem_u32(actfull), 1);
    mbarrier_init_fence();
    if (a.early_weights) issue_first();
  }
  if (!a.defer) {   // as in the one-token kernel
    pdl_wait_primary();
    if (!a.Xs) pdl_launch_dependents();
  }
  if (threadIdx.x == 0 && !a.early_weights) issue_first();

  // Activations staged by the staging kernel (which this kernel has waited
  // for): one bulk copy of their shared-memory image. The next kernel may
  // start only once the copy has landed, since it may overwrite the staged
  // region (the next call's staging).
  bool failed = false;
  const int64_t act_bytes = pl.red - pl.sb;
  if (a.Xs) {
    __syncthreads();   // thread 0 has initialized the barriers
    if (threadIdx.x == 0) {
      mbarrier_arrive_expect_tx(smem_u32(actfull), (uint32_t)act_bytes);
      bulk_copy_g2s(smem_u32(sb), a.Xs, (uint32_t)act_bytes, smem_u32(actfull),
                    l2_evict_last_policy());
    }
    if (!mbarrier_wait_bounded(smem_u32(actfull), 0u, lim)) failed = true;
    pdl_launch_dependents();
  }

  // Stage the activations: f16 q * 2^(9 - 2s) (up to 8 tokens) or the int8 q
  // (more) per token row, the sum of each 128-value half-block (8 partial
  // sums), and the block scales. Lane l takes values 8l .. 8l + 7 of a block
  // (slots 2(l & 1) and 2(l & 1) + 1).
  auto put_f16 = [&](int tb, uint32_t v0, uint32_t v1) {
    const int t = tb / a.nblk, b = tb - t * a.nblk;
    if (Mc::kI8) {
      uint32_t* dst = reinterpret_cast<uint32_t*>(sb + t * pl.sb_stride + (int64_t)b * kQK + 8 * lane);
      dst[0] = v0;
      dst[1] = v1;
      return;
    }
    uint32_t h[4];
    tc::s8x4_to_h2x2(v0, h[0], h[1]);
    tc::s8x4_to_h2x2(v1, h[2], h[3]);
    const uint32_t m0 = mma_slot_scale(2 * (lane & 1)), m1 = mma_slot_scale(2 * (lane & 1) + 1);
    uint2* dst = reinterpret_cast<uint2*>(sb + t * pl.sb_stride + ((int64_t)b * kQK + 8 * lane) * 2);
    dst[0] = make_uint2(h2_mul_rn(h[0], m0), h2_mul_rn(h[1], m0));
    dst[1] = make_uint2(h2_mul_rn(h[2], m1), h2_mul_rn(h[3], m1));
  };
  if (a.Xs) {
    // staged already
  } else if (a.X) {
    stage_quantize(a, T * a.nblk, warp, kConsumers, lane,
                   [&](int tb, uint32_t w0, uint32_t w1, int s8, float d) {
                     put_f16(tb, w0, w1);
                     const int hs = half_block_sum(s8);
                     if ((lane & 15) == 0) sgsum[2 * tb + (lane >> 4)] = hs;
                     if (lane == 0) sdx[tb] = d;
                   });
  } else {
    for (int tb = warp; tb < T * a.nblk; tb += kConsumers) {
      const uint8_t* blk = a.Xq + (int64_t)tb * kQ8KBytes;
      const uint32_t* qs = reinterpret_cast<const uint32_t*>(blk + kQ8KQsOffset);
      put_f16(tb, __ldg(qs + 2 * lane), __ldg(qs + 2 * lane + 1));
      int s = lane < 16 ? (int)__ldg(reinterpret_cast<const int16_t*>(blk + kQ8KBsumsOffset) + lane) : 0;
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      if (lane == 0 || lane == 8) sgsum[2 * tb + (lane >> 3)] = s;   // t * ngroups + 2b + half
      if (lane == 0) sdx[tb] = __ldg(reinterpret_cast<const float*>(blk));
    }
  }
  __syncthreads();

  // Deferred form, as in the one-token kernel; the q8_K values come back
  // exactly from their staged f16 copies (q * 2^(9 - 2s), |q| <= 127).
  bool waited = !a.defer;
  auto finish_wait = [&]() {
    pdl_wait_primary();
    pdl_launch_dependents();
    if (a.X && a.Xq_out) {
      const float inv0 = (lane & 1) ? 0.03125f : 0.001953125f;   // 2^-5 : 2^-9
      const float inv1 = (lane & 1) ? 0.125f : 0.0078125f;       // 2^-3 : 2^-7
      for (int tb = blockIdx.x + warp * gridDim.x; tb < T * a.nblk; tb += gridDim.x * kConsumers) {
        const int t = tb / a.nblk, b = tb - t * a.nblk;
        if (Mc::kI8) {   // the int8 values as staged
          const uint32_t* src =
              reinterpret_cast<const uint32_t*>(sb + t * pl.sb_stride + (int64_t)b * kQK + 8 * lane);
          const uint32_t w0 = src[0], w1 = src[1];
          const int s8 = __dp4a((int)w0, 0x01010101, 0) + __dp4a((int)w1, 0x01010101, 0);
          q8K_store(a.Xq_out + (int64_t)tb * kQ8KBytes, lane, w0, w1, s8, sdx[tb]);
          continue;
        }
        const uint2* src =
            reinterpret_cast<const uint2*>(sb + t * pl.sb_stride + ((int64_t)b * kQK + 8 * lane) * 2);
        int q[8];
        int s8 = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint2 v = src[h];
          const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
          const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
          const float inv = h ? inv1 : inv0;
          q[4 * h + 0] = __float2int_rn(f0.x * inv);
          q[4 * h + 1] = __float2int_rn(f0.y * inv);
          q[4 * h + 2] = __float2int_rn(f1.x * inv);
          q[4 * h + 3] = __float2int_rn(f1.y * inv);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) s8 += q[e];
        q8K_store(a.Xq_out + (int64_t)tb * kQ8KBytes, lane, pack4_s8(q[0], q[1], q[2], q[3]),
                  pack4_s8(q[4], q[5], q[6], q[7]), s8, sdx[tb]);
      }
    }
    waited = true;
  };

  int j = 0, slot = 0;
  uint32_t phase = 0;
  for (int rb = rb0, i = 0; rb < rb1; ++rb, ++i) {
    const int row_base = rb * kTileRows;
    float y[kReducers];
#pragma unroll
    for (int e = 0; e < kReducers; ++e) y[e] = 0.0f;
    for (int st = 0; st < per_rb; ++st, ++j) {
      const int gs = st * kStageTiles;
      const int nt = min(kStageTiles, a.ngroups - gs);
      if (!failed && !mbarrier_wait_bounded(smem_u32(full + slot), phase, lim))
        failed = true;
      failed = __any_sync(0xffffffffu, failed);   // mma.sync below is warp-wide
      const uint8_t* stage = ring + (size_t)slot * kStageBytes;
      MmaCodes mc[Mc::kTilesPerWarp];
#pragma unroll
      for (int u = 0; u < Mc::kTilesPerWarp; ++u) {
        const int tl = warp + u * kConsumers;
        if (!failed && tl < nt) load_mma_codes(stage + tl * kTileBytes, lane, mc[u]);
      }
      __syncwarp();   // the whole warp has read its tiles: release the slot
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(released + slot, 1) == kConsumers - 1) {
          released[slot] = 0;
          if (!failed && j + S < nstage) {
            int st2 = st + S, rb2 = rb;
            while (st2 >= per_rb) { st2 -= per_rb; ++rb2; }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(slot, rb2, st2);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < Mc::kTilesPerWarp; ++u) {
        const int tl = warp + u * kConsumers;
        if (!failed && tl < nt)
          group_mma<T, kGroupSums>(mc[u], gs + tl, sb, pl.sb_stride, sgsum, sdx, a, row_base, lane, y);
      }
      if (++slot == S) { slot = 0; phase ^= 1u; }
    }
    if (!waited) finish_wait();
    if (!kGroupSums) {
      // The warps' partial sums of this tile column meet in shared memory;
      // warp (i*R + e) % warps adds C position e (of R = 8 per token block)
      // over the warps in warp order.
      const int p = i & 1;
      float* r = red + p * (kConsumers * kReducers * 32);
      if (i >= 2 && !failed &&
          !mbarrier_wait_bounded(smem_u32(redempty + p), (uint32_t)(((i >> 1) - 1) & 1),
                                 lim))
        failed = true;
#pragma unroll
      for (int e = 0; e < kReducers; ++e) r[(warp * kReducers + e) * 32 + lane] = y[e];
      __syncwarp();
      if (lane == 0) mbarrier_arrive(smem_u32(redfull + p));
      const int e = (warp - i * kReducers) & (kConsumers - 1);
      if (e < kReducers) {
        if (!failed && !mbarrier_wait_bounded(smem_u32(redfull + p), (uint32_t)((i >> 1) & 1),
                                              lim))
          failed = true;
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < kConsumers; ++k) sum += r[(k * kReducers + e) * 32 + lane];
        // e = 8nb + 4h + 2r + j: token block nb, half h, row g8 + 8r, token 2q + j
        const int row = row_base + 16 * ((e >> 2) & 1) + (lane >> 2) + 8 * ((e >> 1) & 1);
        const int t = 8 * (e >> 3) + 2 * (lane & 3) + (e & 1);
        if (!failed && t < T && row < a.rows) a.Y[(int64_t)t * a.rows + row] = sum;
        __syncwarp();
        if (lane == 0) mbarrier_arrive(smem_u32(redempty + p));
      }
    }
  }
  if (!waited) finish_wait();   // a CTA without tile columns
  if (failed && lane == 0) atomicExch(a.status, kDevTimeout);
  if (__syncthreads_or(failed) && threadIdx.x == 0) {   // as in the one-token kernel
    for (int sl = 0; sl < S; ++sl)
      if (issued[sl] > 0)
        mbarrier_wait_bounded(smem_u32(full + sl), (uint32_t)((issued[sl] - 1) & 1), kWaitLimitNs);
    if (a.Xs) mbarrier_wait_bounded(smem_u32(actfull), 0u, kWaitLimitNs);   // the staged copy
  }
}

// The staging kernel of the mma.sync GEMV's workspace forms: the activations
// in the shared-memory image the GEMV would otherwise build in every CTA (f16
// rows of q * 2^(9 - 2s), the half-block sums, the block scales), built once
// in the caller's workspace; each GEMV CTA then loads it with one bulk copy.
// One warp per q8_K block (token t, block b), from the f32 activations
// (quantized exactly as the quantizer kernel does, the q8_K block written to
// Xq_out) or from the q8_K blocks Xq_in. Launched as a programmatic dependent:
// with x_final (the host showed the kernel before it writes nothing this one
// reads) it reads and quantizes before waiting for that kernel; it writes
// only after the wait. It lets its successor (the GEMV, which waits for it
// before reading the image) start at once when early_trigger (the host knows
// the kernel before it and passes its outputs on to the GEMV's early-read
// check), else only after its own wait.
constexpr int kStageWarps = 8;

template <int T>
__global__ void __launch_bounds__(kStageWarps * 32) gemv_stage_kernel(
    const float* __restrict__ X, const uint8_t* __restrict__ Xq_in, uint8_t* __restrict__ Xq_out,
    uint8_t* __restrict__ region, int nblk, int64_t sb_stride, int64_t off_sgsum, int64_t off_sdx,
    int x_final, int early_trigger) {
  const int lane = threadIdx.x & 31;
  const int tb = blockIdx.x * kStageWarps + (threadIdx.x >> 5);
  const bool active = tb < T * nblk;   // warp-uniform
  if (early_trigger) pdl_launch_dependents();
  if (!x_final) {
    pdl_wait_primary();
    if (!early_trigger) pdl_launch_dependents();
  }
  uint32_t w0 = 0u, w1 = 0u;
  int s8 = 0, bs = 0;
  float d = 0.0f;
  if (active) {
    if (X) {
      const float4* src = reinterpret_cast<const float4*>(X + (int64_t)tb * kQK) + 2 * lane;
      q8K_warp(__ldg(src), __ldg(src + 1), w0, w1, s8, d);
    } else {
      const uint8_t* blk = Xq_in + (int64_t)tb * kQ8KBytes;
      const uint32_t* qs = reinterpret_cast<const uint32_t*>(blk + kQ8KQsOffset);
      w0 = __ldg(qs + 2 * lane);
      w1 = __ldg(qs + 2 * lane + 1);
      bs = lane < 16 ? (int)__ldg(reinterpret_cast<const int16_t*>(blk + kQ8KBsumsOffset) + lane) : 0;
      d = __ldg(reinterpret_cast<const float*>(blk));
    }
  }
  if (x_final) {
    pdl_wait_primary();
    if (!early_trigger) pdl_launch_dependents();
  }
  if (!active) return;
  if (X && Xq_out) q8K_store(Xq_out + (int64_t)tb * kQ8KBytes, lane, w0, w1, s8, d);
  const int t = tb / nblk, b = tb - t * nblk;
  uint32_t h[4];
  tc::s8x4_to_h2x2(w0, h[0], h[1]);
  tc::s8x4_to_h2x2(w1, h[2], h[3]);
  const uint32_t m0 = mma_slot_scale(2 * (lane & 1)), m1 = mma_slot_scale(2 * (lane & 1) + 1);
  uint2* dst = reinterpret_cast<uint2*>(region + t * sb_stride + ((int64_t)b * kQK + 8 * lane) * 2);
  dst[0] = make_uint2(h2_mul_rn(h[0], m0), h2_mul_rn(h[1], m0));
  dst[1] = make_uint2(h2_mul_rn(h[2], m1), h2_mul_rn(h[3], m1));
  int* sgsum = reinterpret_cast<int*>(region + off_sgsum);
  if (X) {
    const int hs = half_block_sum(s8);
    if ((lane & 15) == 0) sgsum[2 * tb + (lane >> 4)] = hs;
  } else {
    bs += __shfl_xor_sync(0xffffffffu, bs, 1);
    bs += __shfl_xor_sync(0xffffffffu, bs, 2);
    bs += __shfl_xor_sync(0xffffffffu, bs, 4);
    if (lane == 0 || lane == 8) sgsum[2 * tb + (lane >> 3)] = bs;
  }
  if (lane == 0) reinterpret_cast<float*>(region + off_sdx)[tb] = d;
}

// Where a launch the host allowed to defer its wait (a.defer) waits: never
// for group sums (stored per group); after the first ring stage when a tile
// column takes three or more stages (the dp4a loop only); else after the
// first tile column when every CTA has two or more, so the rest of its stream
// overlaps the previous kernel's end. With a single short column per CTA the
// wait would come at its end and hold back the next kernel's start. Measured
// on GB300 in graph chains at one token: 5120 x 17408 (five stages per
// column, one column per CTA) 11.4 -> 8.2 us waiting after the first stage;
// 32768 x 8192 13.5 us after the first column, 13.8 after the first stage;
// 5120 x 5120 (two stages, one column) slower either way; the mma.sync
// variant slower waiting after a stage.
inline int defer_wait(const GemvArgs& a, bool group_sums, int grid, int stage_tiles,
                      bool after_stage_ok) {
  if (!a.defer || group_sums) return 0;
  const int per_rb = (a.ngroups + stage_tiles - 1) / stage_tiles;
  if (after_stage_ok && per_rb >= 3) return 2;
  return a.nrb >= 2 * grid ? 1 : 0;
}

// A launch about to go takes a pending test stall (tq_debug_stall_next_launch).
inline void take_stall(GemvArgs& a) {
  const int64_t ns = take_debug_stall();
  a.stall = ns > 0 ? 1 : 0;
  a.stall_ns = ns > 0 ? (uint64_t)ns : 0;
}

template <int T, bool G, int TPW>
cudaError_t launch_mma(const GemvArgs& a0, int64_t cols, cudaStream_t s) {
  auto kernel = gemv_mma_kernel<T, G, TPW>;
  GemvArgs a = a0;
  DeviceLimits lim;
  cudaError_t e = device_limits(&lim);
  if (e != cudaSuccess) return e;
  const int optin = lim.optin_smem, nsm = lim.sms;
  int stages = TQ_GEMV_MAX_STAGES;
  while (stages > 2 && plan_mma<T, TPW>(stages, cols).total > optin) --stages;
  const int64_t smem = plan_mma<T, TPW>(stages, cols).total;
  if (smem > optin) return cudaErrorNotSupported;
  a.stages = stages;
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = resident_ctas(reinterpret_cast<const void*>(kernel), MmaCfg<T, TPW>::kThreads, (size_t)smem,
                    &per_sm);
  if (e != cudaSuccess) return e;
  per_sm = max(1, min(per_sm, TQ_GEMV_CTAS_PER_SM));
  int grid = (int)std::min<int64_t>(a.nrb, (int64_t)nsm * per_sm);
#if TQ_GEMV_EVEN_GRID
  if (a.defer)   // as in launch_t
    for (int g = grid; g >= grid - grid / 4 && g >= 1; --g)
      if (a.nrb % g == 0) { grid = g; break; }
#endif
  a.defer = defer_wait(a, G, grid, MmaCfg<T, TPW>::kStageTiles, false);
  take_stall(a);
  return launch_pdl(kernel, dim3(grid), dim3(MmaCfg<T, TPW>::kThreads), (size_t)smem, s, a);
}

template <int T, bool G, int F = kFmtTq>
cudaError_t launch_t(const GemvArgs& a0, int64_t cols, cudaStream_t s) {
  static_assert(T >= 1 && T <= kMaxDp4aTok, "token count");
  auto kernel = gemv_kernel<T, G, F>;
  GemvArgs a = a0;
  DeviceLimits lim;
  cudaError_t e = device_limits(&lim);
  if (e != cudaSuccess) return e;
  const int optin = lim.optin_smem, nsm = lim.sms;
  // deepest ring that fits
  int stages = TQ_GEMV_MAX_STAGES;
  while (stages > 2 && plan_smem<T, F>(stages, cols).total > optin) --stages;
  const int64_t smem = plan_smem<T, F>(stages, cols).total;
  if (smem > optin) return cudaErrorNotSupported;
  a.stages = stages;
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = resident_ctas(reinterpret_cast<const void*>(kernel), Cfg<T>::kThreads, (size_t)smem, &per_sm);
  if (e != cudaSuccess) return e;
  per_sm = max(1, min(per_sm, TQ_GEMV_CTAS_PER_SM));
  int grid = (int)std::min<int64_t>(a.nrb, (int64_t)nsm * per_sm);
#if TQ_GEMV_EVEN_GRID
  // A launch that may read its inputs before the kernel ahead of it ends
  // (a.defer: the host showed they are final) starts its CTAs staggered, as
  // that kernel's CTAs leave: there a grid that splits the tile columns
  // evenly (every CTA the same work), if one exists within the top quarter of
  // the resident capacity, measured faster. A launch that waits for that
  // kernel first starts all its CTAs together, and the SM with the most work
  // sets the pace: there the grid fills every resident slot (uneven columns
  // per CTA, but less on the busiest SM). Measured on GB300 at one token, the
  // full grid against the even split: waiting first 14.07 -> 13.68 us on
  // 32768 x 8192 and 7.07 -> 6.70 on 17408 x 5120; reading early 12.49 ->
  // 12.90 and 6.11 -> 6.96 (so launches that read early keep the even split).
  if (a.defer)
    for (int g = grid; g >= grid - grid / 4 && g >= 1; --g)
      if (a.nrb % g == 0) { grid = g; break; }
#endif
  a.defer = defer_wait(a, G, grid, Cfg<T>::kStageTiles, true);
  take_stall(a);
  return launch_pdl(kernel, dim3(grid), dim3(Cfg<T>::kThreads), (size_t)smem, s, a);
}

// Token count from which the tensor-core variant is used: measured on GB300,
// it matches the dp4a loop at 4 tokens and is up to 1.45x faster above.
#ifndef TQ_GEMV_MMA_MIN_TOK
#define TQ_GEMV_MMA_MIN_TOK 4
#endif

// Tiles per warp and stage of the tensor-core variant: 0 picks by shape;
// 1..3 force a value (where it fits in shared memory).
#ifndef TQ_GEMV_MMA_TPW
#define TQ_GEMV_MMA_TPW 0
#endif

// A tile column's groups run in stages of (warps x TPW) tiles; the last
// stage of each column leaves warps idle when the count does not divide. Of
// two and three tiles per warp, take the one with fewer idle tiles (two on a
// tie): measured on GB300, three is 2-4% faster at 40 groups (5120 columns),
// two 3-10% faster at 64 (8192); four never won.
inline int mma_tiles_per_warp(int ngroups) {
  if (TQ_GEMV_MMA_TPW) return TQ_GEMV_MMA_TPW;
  auto idle = [&](int tpw) {
    const int st = TQ_GEMV_WARPS * tpw;
    return (ngroups + st - 1) / st * st - ngroups;
  };
  return idle(3) < idle(2) ? 3 : 2;
}

template <int T, bool G>
cudaError_t launch_mma_tpw(int tpw, const GemvArgs& a, int64_t cols, cudaStream_t s) {
  switch (tpw) {
    case 1: return launch_mma<T, G, 1>(a, cols, s);
    case 2: return launch_mma<T, G, 2>(a, cols, s);
    default: return launch_mma<T, G, 3>(a, cols, s);
  }
}

template <int T>
cudaError_t launch_tok(const GemvArgs& a, int64_t cols, bool gsum, cudaStream_t s) {
  if constexpr (T >= TQ_GEMV_MMA_MIN_TOK) {
    // above 8 tokens the int8 activations and the wider reduction leave room
    // for two tiles per warp and stage at most
    const int tpw = T > kMaxDp4aTok ? min(2, mma_tiles_per_warp(a.ngroups))
                                    : mma_tiles_per_warp(a.ngroups);
    cudaError_t e = gsum ? launch_mma_tpw<T, true>(tpw, a, cols, s)
                         : launch_mma_tpw<T, false>(tpw, a, cols, s);
    // the ring and the f16 activations did not fit in shared memory: one
    // tile per warp and stage, then the dp4a loop
    if (e == cudaErrorNotSupported && tpw != 1)
      e = gsum ? launch_mma<T, true, 1>(a, cols, s) : launch_mma<T, false, 1>(a, cols, s);
    if (e != cudaErrorNotSupported || a.Xs) return e;   // staged activations: the mma kernel only
  }
  if constexpr (T <= kMaxDp4aTok)
    return gsum ? launch_t<T, true>(a, cols, s) : launch_t<T, false>(a, cols, s);
  else
    return cudaErrorNotSupported;
}

template <bool G>
cudaError_t launch_ptq1_tok(const GemvArgs& a, int64_t cols, int ntok, cudaStream_t s) {
  switch (ntok) {
    case 1: return launch_t<1, G, kFmtPtq1>(a, cols, s);
    case 2: return launch_t<2, G, kFmtPtq1>(a, cols, s);
    case 3: return launch_t<3, G, kFmtPtq1>(a, cols, s);
    case 4: return launch_t<4, G, kFmtPtq1>(a, cols, s);
    case 5: return launch_t<5, G, kFmtPtq1>(a, cols, s);
    case 6: return launch_t<6, G, kFmtPtq1>(a, cols, s);
    case 7: return launch_t<7, G, kFmtPtq1>(a, cols, s);
    default: return launch_t<8, G, kFmtPtq1>(a, cols, s);
  }
}

}  // namespace

int gemv_max_tokens() { return kMaxTok; }

cudaError_t launch_gemv_ptq1(const uint8_t* Wt1, const uint8_t* Xq, float* Y, int32_t* S,
                             int64_t rows, int64_t cols, int ntok, int* dev_status,
                             bool early_weights, cudaStream_t s) {
  if (ntok < 1) return cudaSuccess;
  if (rows > 0x7fffffff / 2 || cols / kGroup > 0x7fffffff / kTq1TileBytes)
    return cudaErrorNotSupported;
  const int nblk = (int)(cols / kQK);
  const int ngroups = (int)(cols / kGroup);
  // launches of up to 8 tokens (each streams the weights once)
  for (int t0 = 0; t0 < ntok; t0 += kMaxDp4aTok) {
    const int n = min(kMaxDp4aTok, ntok - t0);
    GemvArgs a;
    a.Wtq = Wt1;
    a.Xq = Xq + (int64_t)t0 * nblk * kQ8KBytes;
    a.Y = Y ? Y + (int64_t)t0 * rows : nullptr;
    a.S = S ? S + (int64_t)t0 * rows * ngroups : nullptr;
    a.status = dev_status;
    a.rows = (int)rows;
    a.ngroups = ngroups;
    a.nblk = nblk;
    a.nrb = (int)((rows + kTileRows - 1) / kTileRows);
    a.stages = 2;
    // a later chunk follows this function's own GEMV, which writes no weights
    a.early_weights = (early_weights || t0 > 0) ? 1 : 0;
    a.X = nullptr;
    a.Xq_out = nullptr;
    a.defer = 0;
    a.stall = 0;
    a.stall_ns = 0;
    const cudaError_t e = S ? launch_ptq1_tok<true>(a, cols, n, s) : launch_ptq1_tok<false>(a, cols, n, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}


cudaError_t launch_gemv(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                        int64_t rows, int64_t cols, int ntok, int* dev_status, bool early_weights,
                        bool inputs_final, cudaStream_t s, const float* X, uint8_t* Xq_out,
                        const uint8_t* Xs) {
  if (ntok < 1 || ntok > kMaxTok) return cudaErrorNotSupported;
  if (rows > 0x7fffffff / 2 || cols / kGroup > 0x7fffffff / kTileBytes)
    return cudaErrorNotSupported;
  GemvArgs a;
  a.Wtq = Wtq;
  a.Xq = Xq;
  a.Y = Y;
  a.S = S;
  a.status = dev_status;
  a.rows = (int)rows;
  a.ngroups = (int)(cols / kGroup);
  a.nblk = (int)(cols / kQK);
  a.nrb = (int)((rows + kTileRows - 1) / kTileRows);
  a.stages = 2;
  a.early_weights = early_weights || inputs_final ? 1 : 0;
  a.X = X;
  a.Xq_out = Xq_out;
  a.defer = inputs_final ? 1 : 0;
  a.stall = 0;
  a.stall_ns = 0;
  a.Xs = Xs;
  const bool gsum = S != nullptr;
  cudaError_t e;
  switch (ntok) {
    case 1: e = launch_tok<1>(a, cols, gsum, s); break;
    case 2: e = launch_tok<2>(a, cols, gsum, s); break;
    case 3: e = launch_tok<3>(a, cols, gsum, s); break;
    case 4: e = launch_tok<4>(a, cols, gsum, s); break;
    case 5: e = launch_tok<5>(a, cols, gsum, s); break;
    case 6: e = launch_tok<6>(a, cols, gsum, s); break;
    case 7: e = launch_tok<7>(a, cols, gsum, s); break;
    case 8: e = launch_tok<8>(a, cols, gsum, s); break;
    case 9: e = launch_tok<9>(a, cols, gsum, s); break;
    case 10: e = launch_tok<10>(a, cols, gsum, s); break;
    case 11: e = launch_tok<11>(a, cols, gsum, s); break;
    case 12: e = launch_tok<12>(a, cols, gsum, s); break;
    case 13: e = launch_tok<13>(a, cols, gsum, s); break;
    case 14: e = launch_tok<14>(a, cols, gsum, s); break;
    case 15: e = launch_tok<15>(a, cols, gsum, s); break;
    default: e = launch_tok<16>(a, cols, gsum, s); break;
  }
  if (e != cudaErrorNotSupported || ntok == 1 || Xs) return e;
  // The activations of all tokens do not fit in shared memory (long rows:
  // 8 tokens of 17408 columns, 16 of 8192): one launch per half of the tokens, each
  // streaming the weights once, instead of the tensor-core path for a tile
  // of 64 tokens. Every token's inputs and outputs are contiguous rows, and
  // each half's arithmetic is that of a call with those tokens alone. The
  // second half has no more tokens than the first, so it fits whenever the
  // first does (fewer tokens need less shared memory): either both launch or
  // neither does.
  const int n0 = (ntok + 1) / 2;
  e = launch_gemv(Wtq, Xq, Y, S, rows, cols, n0, dev_status, early_weights, inputs_final, s, X,
                  Xq_out);
  if (e != cudaSuccess) return e;
  // the first half's kernel writes no weights and none of the second half's inputs
  return launch_gemv(Wtq, Xq ? Xq + (int64_t)n0 * a.nblk * kQ8KBytes : nullptr,
                     Y ? Y + (int64_t)n0 * rows : nullptr,
                     S ? S + (int64_t)n0 * rows * a.ngroups : nullptr, rows, cols, ntok - n0,
                     dev_status, true, false, s, X ? X + (int64_t)n0 * cols : nullptr,
                     Xq_out ? Xq_out + (int64_t)n0 * a.nblk * kQ8KBytes : nullptr);
}

namespace {

// The staged image's layout (relative to its first byte) for ntok tokens of
// cols columns: the same for every ring depth and tiles per warp.
template <int T>
MmaPlan stage_plan(int64_t cols) { return plan_mma<T, 1>(2, cols); }

// The staged form is planned against the opt-in shared memory of one block
// on sm_103a (227 KB), so whether it applies, and the workspace it needs, are
// functions of the shape alone.
constexpr int64_t kStageSmemLimit = 232448;

// Staging pays where preparing the activations in every CTA costs more than
// the staging kernel's launch: from 3072 columns where the call also
// quantizes X (tq_quantize_matmul), from 5120 where the GEMV only converts
// q8_K blocks to f16, work it does before waiting for the launch before it
// in a chain (measured at 4 to 8 tokens on matrices of 2048 to 17408
// columns). Below, the workspace stays empty and the fused GEMV runs.
#ifndef TQ_GEMV_STAGE_MIN_COLS
#define TQ_GEMV_STAGE_MIN_COLS 3072
#endif
constexpr int64_t kStageMinColsConvert = 5120;

template <int T>
bool stage_fits(int64_t cols) {
  DeviceLimits lim;
  if (device_limits(&lim) != cudaSuccess) return false;
  const int64_t total = stage_plan<T>(cols).total;   // the smallest mma.sync configuration
  return total <= kStageSmemLimit && total <= lim.optin_smem;
}

template <int T>
cudaError_t launch_stage_t(const float* X, const uint8_t* Xq_in, uint8_t* Xq_out, uint8_t* region,
                           int64_t cols, bool x_final, bool early_trigger, cudaStream_t s) {
  const MmaPlan p = stage_plan<T>(cols);
  const int nblk = (int)(cols / kQK);
  const int grid = (T * nblk + kStageWarps - 1) / kStageWarps;
  return launch_pdl(gemv_stage_kernel<T>, dim3(grid), dim3(kStageWarps * 32), 0, s, X, Xq_in,
                    Xq_out, region, nblk, p.sb_stride, p.sgsum - p.sb, p.sdx - p.sb,
                    x_final ? 1 : 0, early_trigger ? 1 : 0);
}

}  // namespace

int64_t gemv_stage_bytes(int64_t cols, int ntok) {
  if (cols <= 0 || cols < TQ_GEMV_STAGE_MIN_COLS || ntok < TQ_GEMV_MMA_MIN_TOK ||
      ntok > kMaxDp4aTok)
    return 0;
  MmaPlan p;
  switch (ntok) {
    case 4: p = stage_plan<4>(cols); break;
    case 5: p = stage_plan<5>(cols); break;
    case 6: p = stage_plan<6>(cols); break;
    case 7: p = stage_plan<7>(cols); break;
    default: p = stage_plan<8>(cols); break;
  }
  return p.total <= kStageSmemLimit ? p.red - p.sb : 0;
}

bool gemv_stage_fits(int64_t cols, int ntok, bool quantizes) {
  if (gemv_stage_bytes(cols, ntok) == 0) return false;
  if (!quantizes && cols < kStageMinColsConvert) return false;
  if (cols / kGroup > 0x7fffffff / kTileBytes) return false;
  switch (ntok) {
    case 4: return stage_fits<4>(cols);
    case 5: return stage_fits<5>(cols);
    case 6: return stage_fits<6>(cols);
    case 7: return stage_fits<7>(cols);
    default: return stage_fits<8>(cols);
  }
}

cudaError_t launch_gemv_stage(const float* X, const uint8_t* Xq_in, uint8_t* Xq_out,
                              uint8_t* region, int64_t cols, int ntok, bool x_final,
                              bool early_trigger, cudaStream_t s) {
  switch (ntok) {
    case 4: return launch_stage_t<4>(X, Xq_in, Xq_out, region, cols, x_final, early_trigger, s);
    case 5: return launch_stage_t<5>(X, Xq_in, Xq_out, region, cols, x_final, early_trigger, s);
    case 6: return launch_stage_t<6>(X, Xq_in, Xq_out, region, cols, x_final, early_trigger, s);
    case 7: return launch_stage_t<7>(X, Xq_in, Xq_out, region, cols, x_final, early_trigger, s);
    case 8: return launch_stage_t<8>(X, Xq_in, Xq_out, region, cols, x_final, early_trigger, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace tq
