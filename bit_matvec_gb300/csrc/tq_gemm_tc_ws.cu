// tq_gemm_tc_ws.cu -- the tensor-core path with a caller-provided workspace.
//
// Turning the int8 activations into the MMA's B operand is the same work for
// every 128-row tile of the weights; without a workspace each CTA repeats it
// (tq_gemm_tc.cu). Here a pre-pass does it once: act_pack writes, for each
// 64-token tile and each 128-weight group, the e4m3 B operand laid out exactly
// as the MMA reads it (UMMA K-major, no swizzle), and per q8_K block the block
// scales and the per-group activation sums (as e4m3 digits). The
// tensor-core kernel stages a q8_K block with one bulk copy for B, one per
// 32-row weight tile and one for the scales and sums.
//
// Operands (kind::f8f6f4, e4m3 x e4m3, f32 accumulate). An int8 activation q
// is 16 * hi + lo with lo = q & 15 in [0, 15] and hi = q >> 4 in [-8, 7]; both
// are exact in e4m3 (four significant bits), and so are lo / 4 and 16 * hi /
// 4. B holds 128 columns per 64-token tile: lo of the 64 tokens, then 16 * hi,
// so one MMA (M = 128, N = 128, K = 32) produces both halves and
// sum_k u q = acc_lo + acc_hi. A weight code u (w = u - 1) at bits 2s..2s+1 of
// a byte becomes an e4m3 byte by one AND (and a shift for s >= 2): bits 0-1
// give the subnormal u * 2^-9, bits 2-3 give u * 4 * 2^-9 (u = 2 sets the
// lowest exponent bit, 2^-6 = 8 * 2^-9). The pre-pass divides B by 4 at the
// k whose A carries the factor 4, so every product is u * lo * 2^-9 or
// u * 16 hi * 2^-9 exactly. Every partial sum is an integer multiple of 2^-9
// below 2^15 in magnitude, so the accumulation is exact and the low plus high
// columns end at sum_k u q * 2^-9. Turning u back into w = u - 1 takes the
// group's activation sum from the q8_K bsums (dot(w, q) = dot(u, q) - sum(q),
// post "the trick with 4 and 16"), in one of two exact ways:
//   - a fifth MMA per group (64-token tiles on single CTAs): B holds the
//     sum's four base-16 digits d0..d3 (d0..d2 in [0, 15], d3 in [-4, 3], all
//     exact in e4m3) at k = 0..3 of each token's low row, A the constants
//     -2^-9 * 16^i, so the accumulator ends at isum * 2^-9 and the epilogue
//     only scales it;
//   - in the epilogue (16- and 32-token tiles, CTA pairs): isum =
//     2^9 * acc - sum(q), one exact f32 FMA per output.
// Both give the same bits. Measured on GB300 (17408 x 5120): at 64 tokens
// the MMA is the cheaper place, 21.1 against 22.5 us, because each epilogue
// warp then handles 32 tokens per group and the epilogue warps share their
// sub-partitions with the MMA-issuing thread; at 16 and 32 tokens the extra
// MMA costs more (17.5 against 16.1 us, 18.6 against 17.9 us).
//
// Per CTA (128 weight rows x 64 tokens) the work goes one q8_K block (two
// 128-weight groups) at a time:
//   - a producer warp stages the block's two B tiles (one 32 KB bulk copy),
//     the weight tiles of both groups (one 2176-byte copy per 32-row tile:
//     consecutive groups of a tile are adjacent in the repacked layout) and
//     the block's scales and sums into a shared-memory ring;
//   - 8 converter warps mask the codes of each group into A and store them
//     into tensor memory (tcgen05.st), 64 weights per thread and group;
//   - one thread issues per group 4 tcgen05.mma (K = 32 each) with A in
//     tensor memory and B read from the staged slot into one accumulator of
//     128 columns per group, plus the digit MMA, and one commit;
//   - epilogue warps, four per 32 tokens of the tile (four of 16 tokens at
//     N = 16), tcgen05.ld each accumulator and add d_x * d_w * isum in
//     packed f32x2 arithmetic.
// The A operands and the accumulators form one ring of three group stages
// (3 x 128 accumulator and 3 x 32 A columns of tensor memory; the digit
// tiles form the same ring in shared memory). The MMAs of group g wait on a
// single barrier: the converters have written A(g) and the digits of g, and
// the epilogue has read the accumulator of g - 3. One commit per group tells both
// the epilogue (accumulator g is complete) and the converters (A stage g is
// free again). Measured on GB300 with clock stamps, the issuing thread sets
// the pace: each commit and each wait costs it more than an MMA does, so the
// group's path has one of each.
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

using namespace tc;

constexpr int kM = 128;            // weight rows per CTA (UMMA M)
constexpr int kK = 32;             // UMMA K of kind::f8f6f4
constexpr int kGPB = kQK / kGroup;     // groups per q8_K block (2)
constexpr int kMmaPerGroup = kGroup / kK;   // 4
constexpr int kConvWarps = 8;    // converters: warp w -> rows 32*(w%4).., k half w/4
// Tokens per epilogue warp, by token tile, and whether the activation sums
// enter through the digit MMA (1) or the epilogue (0) (compile-time tuning).
#ifndef TQ_TC_EPI_TOK_64
#define TQ_TC_EPI_TOK_64 32
#endif
#ifndef TQ_TC_SUM_MMA_64
#define TQ_TC_SUM_MMA_64 1
#endif
#ifndef TQ_TC_SUM_MMA_32
#define TQ_TC_SUM_MMA_32 0
#endif
#ifndef TQ_TC_SUM_MMA_16
#define TQ_TC_SUM_MMA_16 0
#endif
#ifndef TQ_TC_EPI_TOK_32
#define TQ_TC_EPI_TOK_32 32
#endif
constexpr int kTilesPerCta = kM / kTileRows;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACols = kGroup / 4;              // 32 per group: four e4m3 per column
constexpr uint32_t kAccCol = 0;                      // accumulator stage s: s * kNB
// B operand per (token tile, group) in UMMA canonical K-major layout without
// swizzle: 2N rows (row n < N: lo of token n; row N + n: 16 * hi of token n)
// x 128 k, one byte each. A core matrix is 8 rows x 16 bytes stored as 128
// contiguous bytes; LBO = 128 (next 16 k), SBO = 1024 (next 8 rows). The MMA
// for k = 32 kk.. starts kk * 256 bytes in.
constexpr uint32_t kLBO = 128;
constexpr uint32_t kSBO = 8 * 128;
constexpr float kProdScale = 512.0f;                   // products carry 2^-9
// The digit MMA: B per group stage is 2N rows x 32 k (K-major, no swizzle:
// LBO = 128 for the next 16 k, SBO = 256 for the next 8 rows), the digits of
// token n at k = 0..3 of row n, zeros elsewhere; A is one word per row of
// tensor memory, e4m3 -2^-9, -2^-5, -2^-1, -2^3 at k = 0..3.
constexpr uint32_t kSBOs = 2 * 128;
constexpr uint32_t kASumWord = 0xD0B09081u;
constexpr uint32_t kASumCols = 16;                     // one 16-column store per lane quarter
constexpr int kWRun = kGPB * kTileBytes;               // one 32-row tile, both groups
constexpr int kInB = 0;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Everything that depends on the token tile N (16, 32 or 64 tokens per CTA).
// A smaller tile for fewer tokens: a smaller B per group (less to stage and
// to read from L2), fewer accumulator columns for the epilogue to read, and
// room in tensor memory for more group stages.
template <int N, int CG = 1>
struct TcCfg {
  static_assert(N == 16 || N == 32 || N == 64, "token tile");
  static_assert(CG == 1 || CG == 2, "CTAs per MMA");
  static constexpr int kN = N;                         // tokens per CTA
  static constexpr int kNB = 2 * N;                    // UMMA N: low and high parts
  static constexpr bool kSumMma =
      CG == 1 && (N == 64 ? TQ_TC_SUM_MMA_64 : N == 32 ? TQ_TC_SUM_MMA_32 : TQ_TC_SUM_MMA_16) != 0;
  // A + accumulator ring in tensor memory, one group per stage (after it the
  // digit MMA's constant A)
  static constexpr int kStages = (int)((kTmemCols - (kSumMma ? kASumCols : 0u)) / (kNB + kACols));
  // d_w, d_x and the group sums per block, written by the converters and
  // read by the epilogue. A converter writing block b has seen the MMAs of
  // group 2b - kStages finish, which were issued after the epilogue released
  // group 2b - 2 kStages; the epilogue then is past block b - kStages - 1, so
  // a ring of kStages + 1 blocks is never overwritten while read.
  static constexpr int kScaleStages = kStages + 1;
  static constexpr int kInStages = N == 64 ? 3 : N == 32 ? 4 : 6;   // staged-input ring
  // epilogue: warp w -> rows 32*(w%4).., tokens kEpiTok*(w/4).. (a warp reaches
  // only the tensor-memory lanes of its warp index mod 4)
  static constexpr int kEpiTok = N == 64 ? TQ_TC_EPI_TOK_64 : N == 32 ? TQ_TC_EPI_TOK_32 : 16;
  static_assert(kEpiTok % 16 == 0 && N % kEpiTok == 0, "epilogue width");
  static constexpr int kEpiWarps = 4 * (N / kEpiTok);
  static constexpr int kMmaWarp = kConvWarps + kEpiWarps;
  static constexpr int kProdWarp = kMmaWarp + 1;
  static constexpr int kThreads = (kProdWarp + 1) * 32;
  static constexpr uint32_t kAccCols = kNB;
  static constexpr uint32_t kACol = kStages * kAccCols;   // A stage s: kACol + s * 32
  static constexpr uint32_t kASumCol = kACol + kStages * kACols;
  static_assert(kASumCol + (kSumMma ? kASumCols : 0u) <= kTmemCols, "tensor memory overflow");
  static constexpr int kBSumBytes = kSumMma ? kNB * kK : 0;   // digit tile per group stage
  static constexpr int kBTile = kNB * kGroup;
  // per (token tile, block): d_x of N tokens (f32), then per group each
  // token's activation sum: its four e4m3 digits as one word for the digit
  // MMA, else minus the sum as f32 (magnitude at most 16384, exact)
  static constexpr int kSumOff = N;                    // floats
  static constexpr int kDxFloats = N + kGPB * N;
  static constexpr int kDxBytes = kDxFloats * 4;
  // one staged slot: the block's B tiles (with a CTA pair, this CTA's half of
  // each: rows 0..N-1, the low parts, in rank 0; rows N..2N-1 in rank 1), its
  // weight tiles (per 32-row tile both groups, adjacent), its scales and sums
  static constexpr int kBPart = kBTile / CG;
  static constexpr int kInW = kGPB * kBPart;
  static constexpr int kInDx = kInW + kTilesPerCta * kWRun;
  static constexpr int kInBytes = kInDx + kDxBytes;
  static_assert(kInBytes % 16 == 0 && kWRun % 16 == 0 && kInW % 16 == 0 && kDxBytes % 16 == 0,
                "bulk copies need 16-byte multiples");
  // scale ring stage: d_w per group and row (times 2^9 with the digit MMA),
  // then d_x of the block (and minus the sums of each group without it)
  static constexpr int kScaleFloats = kGPB * kM + (kSumMma ? N : kDxFloats);
  static constexpr int kNumBars = 2 * kInStages + 2 * kStages + 1;   // + the failure drain
  static constexpr int kSmemUsed = kInStages * kInBytes + kStages * kBSumBytes +
                                   kScaleStages * kScaleFloats * 4 + kNumBars * 8 + 16;
  // Enough shared memory that only one CTA fits on an SM: each CTA allocates
  // all 512 tensor-memory columns.
  static constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  static constexpr uint32_t kIdesc = idesc_e4m3(kM * CG, kNB);
};

// Local names for the token tile's constants inside a function templated on N.
#define TQ_TC_CFG(N)                                                        \
  TQ_TC_CFG2(N, 1)
#define TQ_TC_CFG2(N, CG)                                                   \
  using Cfg_ = TcCfg<N, CG>;                                                \
  constexpr int kBPart = Cfg_::kBPart;                                      \
  (void)kBPart;                                                             \
  constexpr int kN = Cfg_::kN;                                              \
  constexpr int kNB = Cfg_::kNB;                                            \
  constexpr int kStages = Cfg_::kStages;                                    \
  constexpr int kScaleStages = Cfg_::kScaleStages;                          \
  constexpr int kInStages = Cfg_::kInStages;                                \
  constexpr int kEpiWarps = Cfg_::kEpiWarps;                                \
  constexpr int kEpiTok = Cfg_::kEpiTok;                                    \
  constexpr bool kSumMma = Cfg_::kSumMma;                                   \
  constexpr uint32_t kASumCol = Cfg_::kASumCol;                             \
  constexpr int kBSumBytes = Cfg_::kBSumBytes;                              \
  constexpr int kMmaWarp = Cfg_::kMmaWarp;                                  \
  constexpr int kProdWarp = Cfg_::kProdWarp;                                \
  constexpr int kThreads = Cfg_::kThreads;                                  \
  constexpr uint32_t kAccCols = Cfg_::kAccCols;                             \
  constexpr uint32_t kACol = Cfg_::kACol;                                   \
  constexpr int kBTile = Cfg_::kBTile;                                      \
  constexpr int kSumOff = Cfg_::kSumOff;                                    \
  constexpr int kDxFloats = Cfg_::kDxFloats;                                \
  constexpr int kDxBytes = Cfg_::kDxBytes;                                  \
  constexpr int kInW = Cfg_::kInW;                                          \
  constexpr int kInDx = Cfg_::kInDx;                                        \
  constexpr int kInBytes = Cfg_::kInBytes;                                  \
  constexpr int kScaleFloats = Cfg_::kScaleFloats;                          \
  constexpr uint32_t kIdesc = Cfg_::kIdesc;                                 \
  (void)kN; (void)kNB; (void)kStages; (void)kScaleStages; (void)kInStages;  \
  (void)kEpiWarps; (void)kEpiTok; (void)kSumMma; (void)kASumCol; (void)kBSumBytes; (void)kMmaWarp; (void)kProdWarp; (void)kThreads;          \
  (void)kAccCols; (void)kACol; (void)kBTile; (void)kSumOff; (void)kDxFloats; \
  (void)kDxBytes; (void)kInW; (void)kInDx; (void)kInBytes; (void)kScaleFloats; \
  (void)kIdesc

struct Layout {
  int64_t ntile;      // N-token tiles
  int64_t b_bytes;    // ntile * G * kBTile
  int64_t dx_bytes;   // ntile * nblk * kDxBytes
};

template <int N>
__host__ __device__ inline Layout ws_layout(int64_t cols, int64_t ntok) {
  Layout l;
  l.ntile = (ntok + N - 1) / N;
  l.b_bytes = l.ntile * (cols / kGroup) * TcCfg<N>::kBTile;
  l.dx_bytes = l.ntile * (cols / kQK) * TcCfg<N>::kDxBytes;
  return l;
}

// ---------------------------------------------------------------- pre-pass

// A group's activation sum as the four e4m3 digits the digit MMA reads:
// sq = d0 + 16 d1 + 256 d2 + 4096 d3, d0..d2 in [0, 15], d3 in [-4, 3].
__device__ __forceinline__ uint32_t sum_digits(int sq) {
  return e4m3x2((float)(sq & 15), (float)((sq >> 4) & 15)) |
         (e4m3x2((float)((sq >> 8) & 15), (float)(sq >> 12)) << 16);
}

// The record word of a token's group sum (see TcCfg::kDxFloats).
template <bool kSumMma>
__device__ __forceinline__ uint32_t sum_word(int sq) {
  return kSumMma ? sum_digits(sq) : __float_as_uint((float)(-sq));
}

// One CTA of 4N threads per (group g, token tile): thread t takes token t % N
// and k quarter t / N (32 activations) and writes two 16-byte core-matrix rows
// of the low part and two of the high part; the k-quarter-0 threads also
// write the token's group sum word and (for even g) its block scale.
template <int N, int CG>
__global__ void __launch_bounds__(4 * N) act_pack_kernel(const uint8_t* __restrict__ Xq,
                                                         uint8_t* __restrict__ Bt,
                                                         float* __restrict__ Dx, int64_t ntok,
                                                         int ngroups, int nblk) {
  TQ_TC_CFG2(N, CG);
  pdl_launch_dependents();
  pdl_wait_primary();   // the q8_K activations come from the previous kernel
  const int g = blockIdx.x;
  const int64_t nt = blockIdx.y;
  const int n = threadIdx.x % kN, kq = threadIdx.x / kN;
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
      const int16_t* bs = reinterpret_cast<const int16_t*>(blk + kQ8KBsumsOffset);
#pragma unroll
      for (int i = 0; i < 8; ++i) sq += __ldg(bs + (g & 1) * 8 + i);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0u;   // padded tokens: zero activations, zero scale
  }
  uint8_t* tile = Bt + (nt * ngroups + g) * kBTile;
  uint8_t* row_lo = tile + (n >> 3) * kSBO + (n & 7) * 16;
  uint8_t* row_hi = tile + ((kN + n) >> 3) * kSBO + (n & 7) * 16;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    // words 4c..4c+3: k = kq*32 + 16c + 4w' + j; the A bytes of odd words
    // (bit 2 of k set) carry the factor 4, so those activations take 1/4
    uint4 lo, hi;
    split_e4m3(q[4 * c + 0], 1.0f, lo.x, hi.x);
    split_e4m3(q[4 * c + 1], 0.25f, lo.y, hi.y);
    split_e4m3(q[4 * c + 2], 1.0f, lo.z, hi.z);
    split_e4m3(q[4 * c + 3], 0.25f, lo.w, hi.w);
    *reinterpret_cast<uint4*>(row_lo + (kq * 2 + c) * kLBO) = lo;
    *reinterpret_cast<uint4*>(row_hi + (kq * 2 + c) * kLBO) = hi;
  }
  if (kq == 0) {
    float* rec = Dx + (nt * nblk + (g >> 1)) * kDxFloats;
    reinterpret_cast<uint32_t*>(rec)[kSumOff + (g & 1) * kN + n] = sum_word<kSumMma>(sq);
    if ((g & 1) == 0) rec[n] = d;
  }
}

// Fused form of the quantizer and the pre-pass (tq_quantize_matmul): one warp
// per (token slot, q8_K block) quantizes the f32 activations exactly as the
// quantizer kernel does (q8K_warp), writes the q8_K block, and writes the
// token's e4m3 rows of both groups' B tiles, the group sum words and the
// block scale. Token slots past ntok (the last tile's padding) get zeros.
// Lane l holds values 8l .. 8l + 7: group l / 16, k = 8 (l % 16) .. + 7 of it,
// bit 2 of k clear for the first four and set for the last four.
constexpr int kPackWarps = 8;

template <int N, int CG>
__global__ void __launch_bounds__(kPackWarps * 32) quantize_pack_kernel(
    const float* __restrict__ X, uint8_t* __restrict__ Xq, uint8_t* __restrict__ Bt,
    float* __restrict__ Dx, int64_t ntok, int ngroups, int nblk, int64_t nslots) {
  TQ_TC_CFG2(N, CG);
  pdl_launch_dependents();
  // the workspace and Xq may still be read by the previous kernel in the stream
  pdl_wait_primary();
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * kPackWarps + (threadIdx.x >> 5);
  if (w >= nslots * nblk) return;   // whole warp leaves together
  const int64_t tok = w / nblk;
  const int b = (int)(w - tok * nblk);
  uint32_t w0 = 0u, w1 = 0u;
  int s8 = 0;
  float d = 0.0f;
  if (tok < ntok) {
    const float4* src = reinterpret_cast<const float4*>(X + (tok * nblk + b) * kQK) + 2 * lane;
    q8K_warp(__ldg(src), __ldg(src + 1), w0, w1, s8, d);
    q8K_store(Xq + (tok * nblk + b) * kQ8KBytes, lane, w0, w1, s8, d);
  }
  // group sums: the 16 lanes of each half-warp
  int sq = s8;
  sq += __shfl_xor_sync(0xffffffffu, sq, 1);
  sq += __shfl_xor_sync(0xffffffffu, sq, 2);
  sq += __shfl_xor_sync(0xffffffffu, sq, 4);
  sq += __shfl_xor_sync(0xffffffffu, sq, 8);
  const int64_t nt = tok / kN;
  const int n = (int)(tok - nt * kN), gi = lane >> 4, kl = 8 * (lane & 15);
  uint8_t* tile = Bt + (nt * ngroups + 2 * b + gi) * kBTile;
  uint32_t l0, h0, l1, h1;
  split_e4m3(w0, 1.0f, l0, h0);
  split_e4m3(w1, 0.25f, l1, h1);
  const int off = (kl >> 4) * kLBO + (kl & 15);
  *reinterpret_cast<uint2*>(tile + (n >> 3) * kSBO + (n & 7) * 16 + off) = make_uint2(l0, l1);
  *reinterpret_cast<uint2*>(tile + ((kN + n) >> 3) * kSBO + (n & 7) * 16 + off) = make_uint2(h0, h1);
  float* rec = Dx + (nt * nblk + b) * kDxFloats;
  if ((lane & 15) == 0) reinterpret_cast<uint32_t*>(rec)[kSumOff + gi * kN + n] = sum_word<kSumMma>(sq);
  if (lane == 0) rec[n] = d;
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
  int stall;          // test facility: the first CTA (pair) requests no input, so its
  uint64_t stall_ns;  // waits expire after stall_ns (tq_debug_stall_next_launch)
};

// One group's codes (this thread: one row, the 64 weights of one k half) ->
// 16 A columns of e4m3 bytes. Code word w holds weights 16w + 4s + j (k local
// to the half) in byte j at bits 2s; column 4w + s takes the four weights of
// slot s, k = 16w + 4s + 0..3, as bytes 0..3.
__device__ __forceinline__ void convert_store(const uint4 codes, uint32_t taddr) {
  uint32_t wa[16];
  const uint32_t wv[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t x = wv[w], x4 = wv[w] >> 4;
    wa[4 * w + 0] = x & 0x03030303u;    // u * 2^-9
    wa[4 * w + 1] = x & 0x0c0c0c0cu;    // u * 4 * 2^-9
    wa[4 * w + 2] = x4 & 0x03030303u;
    wa[4 * w + 3] = x4 & 0x0c0c0c0cu;
  }
  tmem_st16(taddr, wa);
}

// CG = 2: the CTAs of a cluster of 2 (consecutive 128-row blocks, one token
// tile) run each MMA as a pair: rank 0 issues 256-row MMAs over both CTAs'
// tensor memory, and each CTA stages only its half of B. The converters and
// epilogues of both CTAs arrive on rank 0's mma_ready; rank 0's commits
// arrive on both CTAs' mma_done and in_empty.
template <int N, int CG, bool kGroupSums>
__global__ void __launch_bounds__(TcCfg<N, CG>::kThreads, 1) gemm_tc_ws_kernel(const WsArgs a) {
  TQ_TC_CFG2(N, CG);
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sIn = smem;                                                         // [in][slot]
  uint8_t* sBSum = smem + kInStages * kInBytes;                                // [stage][digits]
  float* sScale = reinterpret_cast<float*>(sBSum + kStages * kBSumBytes);      // [scale]
  uint64_t* in_full = reinterpret_cast<uint64_t*>(sScale + kScaleStages * kScaleFloats);  // [in]
  uint64_t* in_empty = in_full + kInStages;                                    // [in]
  // mma_ready[s]: the MMAs of group g (stage s = g % 3) may go: the converters
  // have written A(g) (and its digits), and the epilogue has read the
  // accumulator of g - 3 (the epilogue pre-arrives for groups 0..2).
  uint64_t* mma_ready = in_empty + kInStages;                                  // [stage]
  // mma_done[s]: the MMAs of group g are complete: its accumulator is ready
  // for the epilogue, and A (and digit) stage s is free for the converters'
  // group g + 3.
  uint64_t* mma_done = mma_ready + kStages;                                    // [stage]
  uint64_t* drain_bar = mma_done + kStages;   // after a failure: the MMAs issued are done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  // Set by a converter warp that gave up waiting for a slot's copy, before its
  // arrival on the slot's in_empty: the producer then requests no more input.
  // A slot is freed only once every converter has arrived on it (each after
  // seeing the copy land or after setting this flag) and the MMAs that read
  // it are complete, so a slot is never refilled while a copy into it may
  // still be in flight. (The MMA thread sets nothing here: a store on its
  // failure branch made the kernel up to 8 percent slower.)
  volatile int* s_failed = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.ngroups;
  const int nb = G / kGPB;                                // q8_K blocks
  const int64_t rb0 = (int64_t)blockIdx.x * kTilesPerCta;
  const int64_t nt = blockIdx.y;
  const int64_t tok0 = nt * kN;
  // the test stall takes the first CTA (with pairs, the first pair: once one
  // CTA of a pair gives up, the other's waits can fall out of step with the
  // pair's commits and would run to their own limit)
  const bool stalled = a.stall && blockIdx.x < (unsigned)CG && blockIdx.y == 0;
  const uint64_t lim = stalled ? a.stall_ns : kWaitLimitNs;   // bound of the pipeline's waits
  int issued[kInStages] = {};   // producer: copies requested per input slot
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;   // rank 0 issues the MMAs

  if (warp == kMmaWarp) {
    tmem_alloc<CG>(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish<CG>();
  }
  if (tid == 0) {
    // Consumer warps arrive once per warp (lane 0, after __syncwarp).
    for (int i = 0; i < kInStages; ++i) {
      mbarrier_init(smem_u32(in_full + i), 1);
      // the converters have read the slot's weights and scales, and the MMAs
      // that read its B are complete (a commit)
      mbarrier_init(smem_u32(in_empty + i), kConvWarps + 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbarrier_init(smem_u32(mma_ready + s), CG * (kConvWarps + kEpiWarps));
      mbarrier_init(smem_u32(mma_done + s), 1);
    }
    mbarrier_init(smem_u32(drain_bar), 1);
    *s_failed = 0;
    mbarrier_init_fence();
  }
  if (kSumMma) {
    // the digit tiles are zero outside k = 0..3 of rows 0..N-1
    for (int i = tid; i < kStages * kBSumBytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(sBSum)[i] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();   // the peer's barriers are initialized before any arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;
  if (kSumMma) {   // the digit MMA's constant A, one warp per lane quarter
    if (warp < 4) {
      uint32_t r[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) r[j] = j == 0 ? kASumWord : 0u;
      tmem_st16(tmem + ((uint32_t)(warp * 32) << 16) + kASumCol, r);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (warp == kProdWarp) {
    // ---------------- producer: stage block j into slot j % kInStages
    if (lane == 0) {
      int nvalid = 0;                                     // weight tiles that exist
      for (int q = 0; q < kTilesPerCta; ++q) nvalid += (rb0 + q < a.nrb) ? 1 : 0;
      const uint64_t policy = l2_evict_first_policy();
      pdl_wait_primary();   // the workspace is written by the previous kernel (the pre-pass)
      int i = 0;
      uint32_t ph = 0;
      for (int j = 0; j < (stalled ? 0 : nb); ++j) {
        // the slot is free once the converters and the MMAs of block j - kInStages are done
        if (j >= kInStages) {
          if (!mbarrier_wait_bounded(smem_u32(in_empty + i), ph ^ 1u, lim)) {
            failed = true;
            break;
          }
          if (*s_failed) break;
        }
        ++issued[i];
        uint8_t* st = sIn + i * kInBytes;
        const uint32_t full = smem_u32(in_full + i);
        const int g0 = j * kGPB;
        // the activations first (from L2), then the weights (from HBM)
        mbarrier_arrive_expect_tx(full, (uint32_t)(kInW + nvalid * kWRun + kDxBytes));
        if (CG == 1) {
          bulk_copy_g2s(smem_u32(st + kInB), a.Bt + (nt * G + g0) * (int64_t)kBTile, kInW, full,
                        policy);
        } else {
#pragma unroll
          for (int gi = 0; gi < kGPB; ++gi)
            bulk_copy_g2s(smem_u32(st + kInB + gi * kBPart),
                          a.Bt + (nt * G + g0 + gi) * (int64_t)kBTile + rank * kBPart, kBPart, full,
                          policy);
        }
        for (int q = 0; q < nvalid; ++q)
          bulk_copy_g2s(smem_u32(st + kInW + q * kWRun), a.Wtq + ((rb0 + q) * G + g0) * kTileBytes,
                        kWRun, full, policy);
        bulk_copy_g2s(smem_u32(st + kInDx), a.Dx + (nt * a.nblk + j) * kDxFloats, kDxBytes, full,
                      policy);
        if (++i == kInStages) { i = 0; ph ^= 1u; }
      }
    }
  } else if (warp < kConvWarps) {
    // ---------------- converters
    const int q4 = warp & 3, khalf = warp >> 2;          // row quarter, k half of A
    const bool row_ok = rb0 + q4 < a.nrb;
    // thread ct < 192 copies word ct of the block's record (d_x of 64 tokens,
    // then minus the sums of each group's 64 tokens) into the scale ring
    const int ct = warp * 32 + lane;
    const uint32_t a_base = tmem + ((uint32_t)(q4 * 32) << 16) + kACol + (uint32_t)khalf * 16;
    int i = 0, sa = 0, ss = 0, g = 0;
    uint32_t pin = 0, pa = 0;
    for (int b = 0; b < nb; ++b) {
      if (!failed && !mbarrier_wait_bounded(smem_u32(in_full + i), pin, lim)) failed = true;
      failed = __any_sync(0xffffffffu, failed);
      if (failed && lane == 0) *s_failed = 1;   // before this warp's arrival below
      const uint8_t* st = sIn + i * kInBytes;
      const uint8_t* tile = st + kInW + q4 * kWRun;
      uint4 cw[kGPB];
      uint32_t sc[kGPB] = {0u, 0u};
      uint32_t rec = 0u;                                  // d_x bits or a digit word
#pragma unroll
      for (int gi = 0; gi < kGPB; ++gi)
        cw[gi] = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);  // w = 0
      if (!failed) {
        if (row_ok) {
#pragma unroll
          for (int gi = 0; gi < kGPB; ++gi) {
            cw[gi] = *reinterpret_cast<const uint4*>(tile + gi * kTileBytes + khalf * 512 + lane * 16);
            if (khalf == 0)
              sc[gi] = *reinterpret_cast<const uint16_t*>(tile + gi * kTileBytes + kTileCodeBytes +
                                                          lane * 2);
          }
        }
        if (ct < kDxFloats) rec = reinterpret_cast<const uint32_t*>(st + kInDx)[ct];
      }
      __syncwarp();
      if (lane == 0) mbarrier_arrive(smem_u32(in_empty + i));
      if (++i == kInStages) { i = 0; pin ^= 1u; }

#pragma unroll
      for (int gi = 0; gi < kGPB; ++gi) {
        // A stage sa is free once the MMAs of group g - kStages have finished
        if (g >= kStages && !failed &&
            !mbarrier_wait_bounded(smem_u32(mma_done + sa), pa ^ 1u, lim))
          failed = true;
        failed = __any_sync(0xffffffffu, failed);   // tcgen05.st below is warp-wide
        tc_fence_after();
        if (!failed) {
          convert_store(cw[gi], a_base + (uint32_t)sa * kACols);
          if (kSumMma && ct >= kSumOff + gi * kN && ct < kSumOff + (gi + 1) * kN) {
            const int n = ct - kSumOff - gi * kN;   // this group's digits of token n
            *reinterpret_cast<uint32_t*>(sBSum + sa * kBSumBytes + (n >> 3) * kSBOs + (n & 7) * 16) =
                rec;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          }
          if (gi == 0) {
            float* sst = sScale + ss * kScaleFloats;
            if (khalf == 0) {
#pragma unroll
              for (int gj = 0; gj < kGPB; ++gj)
                sst[gj * kM + q4 * 32 + lane] = __half2float(__ushort_as_half((unsigned short)sc[gj])) *
                                                (kSumMma ? kProdScale : 1.0f);
            }
            if (ct < (kSumMma ? kN : kDxFloats)) sst[kGPB * kM + ct] = __uint_as_float(rec);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CG == 1) mbarrier_arrive(smem_u32(mma_ready + sa));
          else mbarrier_arrive_rank(smem_u32(mma_ready + sa), 0u);   // rank 0 issues
        }
        if (++sa == kStages) { sa = 0; pa ^= 1u; }
        ++g;
      }
      if (++ss == kScaleStages) ss = 0;
    }
  } else if (warp < kMmaWarp) {
    // ---------------- epilogue
    const int ew = warp - kConvWarps;
    const int q4 = ew & 3;                                // row quarter
    const int64_t row = (rb0 + q4) * kTileRows + lane;
    const int n0 = (ew >> 2) * kEpiTok;                   // first token
    const uint32_t acc_base = tmem + ((uint32_t)(q4 * 32) << 16) + kAccCol + (uint32_t)n0;
    const uint64_t k512 = f2_packf(kProdScale, kProdScale);
    uint64_t y2[kEpiTok / 2];                             // tokens n0 + 2p, +1
#pragma unroll
    for (int p = 0; p < kEpiTok / 2; ++p) y2[p] = 0ull;
    int sa = 0, ss = 0;
    uint32_t pa = 0;
    if (lane == 0) {   // all accumulator stages start free (groups 0..kStages-1)
      for (int s = 0; s < kStages; ++s) {
        if (CG == 1) mbarrier_arrive(smem_u32(mma_ready + s));
        else mbarrier_arrive_rank(smem_u32(mma_ready + s), 0u);
      }
    }
    for (int b = 0; b < nb; ++b) {
      const float* sst = sScale + ss * kScaleFloats;
      const float4* dx4 = reinterpret_cast<const float4*>(sst + kGPB * kM + n0);
#pragma unroll
      for (int gi = 0; gi < kGPB; ++gi) {
        if (!failed && !mbarrier_wait_bounded(smem_u32(mma_done + sa), pa, lim))
          failed = true;
        failed = __any_sync(0xffffffffu, failed);   // tcgen05.ld below is warp-wide
        tc_fence_after();
        if (!failed) {
          const uint32_t tc0 = acc_base + (uint32_t)sa * kAccCols;
          const float dw = sst[gi * kM + q4 * 32 + lane];
          const uint64_t w2 = f2_packf(dw, dw);
          const float4* nsq4 = reinterpret_cast<const float4*>(sst + kGPB * kM + kSumOff + gi * kN + n0);
#pragma unroll
          for (int h = 0; h < kEpiTok / 16; ++h) {
            uint32_t lo[16], hi[16];
            tmem_ld16_nowait(tc0 + (uint32_t)h * 16, lo);
            tmem_ld16_nowait(tc0 + kN + (uint32_t)h * 16, hi);
            tmem_wait_ld();
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 d = dx4[h * 4 + j4];
              const float4 m = kSumMma ? make_float4(0.f, 0.f, 0.f, 0.f)
                                       : nsq4[h * 4 + j4];          // minus the tokens' sums
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int j = 4 * j4 + 2 * e;             // token pair n0 + 16h + j, +1
                // sum u q * 2^-9, or with the digit MMA isum * 2^-9 (exact)
                const uint64_t z = f2_add(f2_pack(lo[j], lo[j + 1]), f2_pack(hi[j], hi[j + 1]));
                const uint64_t nsq = e == 0 ? f2_packf(m.x, m.y) : f2_packf(m.z, m.w);
                // isum (exact); with the digit MMA d_w carries the 2^9 instead
                const uint64_t is = kSumMma ? (kGroupSums ? f2_mul(z, k512) : z) : f2_fma(z, k512, nsq);
                if (kGroupSums) {
                  if (row < a.rows) {
                    const float2 ii = f2_unpack(is);
                    const int64_t t = tok0 + n0 + 16 * h + j;
                    if (t < a.ntok)
                      a.S[(t * a.rows + row) * G + b * kGPB + gi] = __float2int_rn(ii.x);
                    if (t + 1 < a.ntok)
                      a.S[((t + 1) * a.rows + row) * G + b * kGPB + gi] = __float2int_rn(ii.y);
                  }
                } else {
                  const uint64_t dxp = e == 0 ? f2_packf(d.x, d.y) : f2_packf(d.z, d.w);
                  y2[8 * h + j / 2] = f2_fma(f2_mul(dxp, w2), is, y2[8 * h + j / 2]);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {   // for group g + kStages
          if (CG == 1) mbarrier_arrive(smem_u32(mma_ready + sa));
          else mbarrier_arrive_rank(smem_u32(mma_ready + sa), 0u);
        }
        if (++sa == kStages) { sa = 0; pa ^= 1u; }
      }
      if (++ss == kScaleStages) ss = 0;
    }
    if (!kGroupSums && !failed && row < a.rows) {
#pragma unroll
      for (int p = 0; p < kEpiTok / 2; ++p) {
        const float2 v = f2_unpack(y2[p]);
        const int64_t t = tok0 + n0 + 2 * p;
        if (t < a.ntok) a.Y[t * a.rows + row] = v.x;
        if (t + 1 < a.ntok) a.Y[(t + 1) * a.rows + row] = v.y;
      }
    }
  } else if (lane == 0 && rank == 0) {
    // ---------------- MMA issuer (rank 0 of a pair)
    int i = 0, sa = 0;
    uint32_t pa = 0;
    for (int b = 0; b < nb; ++b) {
      // Descriptor of this slot's B, once: the start address field (bits 0-13,
      // address >> 4) then advances by plain adds, as no address passes 2^18.
      const uint64_t bd0 = smem_desc(smem_u32(sIn + i * kInBytes + kInB), kLBO, kSBO);
      const uint64_t sd0 = smem_desc(smem_u32(sBSum), kLBO, kSBOs);
#pragma unroll
      for (int gi = 0; gi < kGPB; ++gi) {
        // A(g) written and the accumulator of group g - 3 read
        const bool ok = failed || mbarrier_test_wait(smem_u32(mma_ready + sa), pa) ||
                        mbarrier_wait_bounded(smem_u32(mma_ready + sa), pa, lim);
        if (!ok) failed = true;
        tc_fence_after();
        if (!failed) {
          const uint32_t d = tmem + kAccCol + (uint32_t)sa * kAccCols;
          const uint32_t at = tmem + kACol + (uint32_t)sa * kACols;
#pragma unroll
          for (int kk = 0; kk < kMmaPerGroup; ++kk) {
            const uint64_t bd = bd0 + (uint64_t)((gi * kBPart + kk * 2 * kLBO) >> 4);
            if (CG == 1)
              mma_e4m3_tmem_a(d, at + (uint32_t)(kK / 4) * kk, bd, kIdesc, kk > 0 ? 1u : 0u);
            else
              mma_e4m3_tmem_a_pair(d, at + (uint32_t)(kK / 4) * kk, bd, kIdesc, kk > 0 ? 1u : 0u);
          }
          if (kSumMma)   // minus the activation sums: the accumulator ends at isum * 2^-9
            mma_e4m3_tmem_a(d, tmem + kASumCol, sd0 + (uint64_t)((sa * kBSumBytes) >> 4), kIdesc, 1u);
        }
        // the commit fires when these MMAs are done (at once if none were issued)
        if (CG == 1) mma_commit(smem_u32(mma_done + sa));
        else mma_commit_pair(smem_u32(mma_done + sa));
        if (++sa == kStages) { sa = 0; pa ^= 1u; }
      }
      // the slot's B is read once these MMAs are complete
      if (CG == 1) mma_commit(smem_u32(in_empty + i));
      else mma_commit_pair(smem_u32(in_empty + i));
      if (++i == kInStages) i = 0;
    }
  }

  if (failed) atomicExch(a.status, kDevTimeout);
  // After a failure, copies and MMAs may still be in flight: before shared
  // and tensor memory are released, let the last copy requested into each
  // input slot land (the producer refills a slot only after every converter
  // saw its previous copy land, so at most that one is pending; it completes
  // phase issued - 1 of the slot's barrier), and let every MMA issued finish
  // (a commit tracks all of the issuing thread's earlier MMAs).
  // With a pair, rank 0's MMAs write both CTAs' tensor memory: both wait for
  // its final commit (always; a failure in either CTA is not seen by the other).
  const bool any_failed = __syncthreads_or(failed);
  if (any_failed && warp == kProdWarp && lane == 0) {
    for (int i = 0; i < kInStages; ++i)
      if (issued[i] > 0)
        mbarrier_wait_bounded(smem_u32(in_full + i), (uint32_t)((issued[i] - 1) & 1),
                              kWaitLimitNs);
  }
  if ((any_failed || CG == 2) && warp == kMmaWarp && lane == 0) {
    if (rank == 0) {
      if (CG == 1) mma_commit(smem_u32(drain_bar));
      else mma_commit_pair(smem_u32(drain_bar));
    }
    if (CG == 1) mbarrier_wait_bounded(smem_u32(drain_bar), 0u, kWaitLimitNs);
    else mbarrier_wait_bounded_cluster(smem_u32(drain_bar), 0u, kWaitLimitNs);
  }
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();   // no CTA leaves while the other may still signal it
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, kTmemCols);
  }
}

// The token tile for ntok tokens: the smallest of 16, 32, 64 that holds them
// all, 64 above.
inline int tile_tokens(int64_t ntok) { return ntok <= 16 ? 16 : ntok <= 32 ? 32 : 64; }

}  // namespace

int64_t tc_workspace_bytes(int64_t cols, int64_t ntok) {
  Layout l;
  switch (tile_tokens(ntok)) {
    case 16: l = ws_layout<16>(cols, ntok); break;
    case 32: l = ws_layout<32>(cols, ntok); break;
    default: l = ws_layout<64>(cols, ntok); break;
  }
  return l.b_bytes + l.dx_bytes;
}

namespace {

// CTAs per MMA: 2 runs the kernel on clusters of two CTAs whose MMAs span
// both (twice the rows per MMA instruction, half of B staged by each CTA;
// the activation sums then enter in the epilogue). Measured on GB300
// (17408 x 5120): 24.8 / 19.0 / 17.4 us at 64 / 32 / 16 tokens against
// 21.1 / 17.7 / 16.1 us for single CTAs, with identical results: the issuing
// thread then waits on the MMAs themselves (about 150 cycles per 256-row
// MMA), so the halved instruction count does not pay for the cross-CTA
// hand-offs. Off by default; building with TQ_TC_PAIR=1 selects it.
#ifndef TQ_TC_PAIR
#define TQ_TC_PAIR 0
#endif
constexpr int kCtasPerMma = TQ_TC_PAIR ? 2 : 1;

// The tensor-core kernel over a workspace already packed.
template <int N, int CG = kCtasPerMma>
cudaError_t launch_main(const uint8_t* Wtq, float* Y, int32_t* S, int64_t rows, int64_t cols,
                        int64_t ntok, uint8_t* ws, int* dev_status, cudaStream_t s) {
  using C = TcCfg<N, CG>;
  const Layout l = ws_layout<N>(cols, ntok);
  WsArgs a;
  a.Wtq = Wtq;
  a.Bt = ws;
  a.Dx = reinterpret_cast<float*>(ws + l.b_bytes);
  a.Y = Y;
  a.S = S;
  a.status = dev_status;
  a.rows = rows;
  a.ntok = ntok;
  a.ngroups = (int)(cols / kGroup);
  a.nblk = (int)(cols / kQK);
  a.nrb = (int)((rows + kTileRows - 1) / kTileRows);
  const int64_t stall_ns = take_debug_stall();
  a.stall = stall_ns > 0 ? 1 : 0;
  a.stall_ns = stall_ns > 0 ? (uint64_t)stall_ns : 0;
  // a whole number of CTA pairs: a last CTA past the rows runs with no weights
  const int64_t gx = ((rows + kM - 1) / kM + CG - 1) / CG * CG;
  if (gx > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)gx, (unsigned)l.ntile);
  auto kernel = S ? gemm_tc_ws_kernel<N, CG, true> : gemm_tc_ws_kernel<N, CG, false>;
  const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (CG == 1) return launch_pdl(kernel, grid, dim3(C::kThreads), (size_t)C::kSmemBytes, s, a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = (size_t)C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CG;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int N>
cudaError_t launch_ws(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S, int64_t rows,
                      int64_t cols, int64_t ntok, uint8_t* ws, int* dev_status, cudaStream_t s) {
  const Layout l = ws_layout<N>(cols, ntok);
  const int G = (int)(cols / kGroup), nblk = (int)(cols / kQK);
  if (l.ntile > 65535) return cudaErrorInvalidConfiguration;
  cudaError_t e = launch_pdl(act_pack_kernel<N, kCtasPerMma>, dim3((unsigned)G, (unsigned)l.ntile),
                             dim3(4 * N), 0, s, Xq, ws, reinterpret_cast<float*>(ws + l.b_bytes),
                             ntok, G, nblk);
  if (e != cudaSuccess) return e;
  return launch_main<N>(Wtq, Y, S, rows, cols, ntok, ws, dev_status, s);
}

template <int N>
cudaError_t launch_quantize_ws(const float* X, uint8_t* Xq, const uint8_t* Wtq, float* Y,
                               int64_t rows, int64_t cols, int64_t ntok, uint8_t* ws,
                               int* dev_status, cudaStream_t s) {
  const Layout l = ws_layout<N>(cols, ntok);
  const int nblk = (int)(cols / kQK);
  if (l.ntile > 65535) return cudaErrorInvalidConfiguration;
  const int64_t warps = l.ntile * N * nblk;
  const int64_t grid = (warps + kPackWarps - 1) / kPackWarps;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  cudaError_t e = launch_pdl(quantize_pack_kernel<N, kCtasPerMma>, dim3((unsigned)grid), dim3(kPackWarps * 32),
                             0, s, X, Xq, ws, reinterpret_cast<float*>(ws + l.b_bytes), ntok,
                             (int)(cols / kGroup), nblk, l.ntile * N);
  if (e != cudaSuccess) return e;
  return launch_main<N>(Wtq, Y, nullptr, rows, cols, ntok, ws, dev_status, s);
}

}  // namespace

cudaError_t launch_gemm_tc_ws(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                              int64_t rows, int64_t cols, int64_t ntok, uint8_t* ws,
                              int* dev_status, cudaStream_t s) {
  if (rows <= 0 || ntok <= 0 || cols <= 0) return cudaSuccess;
  switch (tile_tokens(ntok)) {
    case 16: return launch_ws<16>(Wtq, Xq, Y, S, rows, cols, ntok, ws, dev_status, s);
    case 32: return launch_ws<32>(Wtq, Xq, Y, S, rows, cols, ntok, ws, dev_status, s);
    default: return launch_ws<64>(Wtq, Xq, Y, S, rows, cols, ntok, ws, dev_status, s);
  }
}

cudaError_t launch_quantize_gemm_tc_ws(const float* X, uint8_t* Xq, const uint8_t* Wtq, float* Y,
                                       int64_t rows, int64_t cols, int64_t ntok, uint8_t* ws,
                                       int* dev_status, cudaStream_t s) {
  if (rows <= 0 || ntok <= 0 || cols <= 0) return cudaSuccess;
  switch (tile_tokens(ntok)) {
    case 16: return launch_quantize_ws<16>(X, Xq, Wtq, Y, rows, cols, ntok, ws, dev_status, s);
    case 32: return launch_quantize_ws<32>(X, Xq, Wtq, Y, rows, cols, ntok, ws, dev_status, s);
    default: return launch_quantize_ws<64>(X, Xq, Wtq, Y, rows, cols, ntok, ws, dev_status, s);
  }
}

}  // namespace tq
