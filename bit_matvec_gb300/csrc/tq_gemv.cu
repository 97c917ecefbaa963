// tq_gemv.cu -- ternary x q8_K product for 1..8 tokens, bound by the weight
// stream from HBM.
//
// Decode reads every weight once per token batch, so the bus is the limit
// (ternary post, "did it reach the wall?" and "prefill wants a different
// shape"). The kernel streams the repacked weights once for all tokens:
//   - a warp owns a 32-row tile column; lane l is row l of the tile, so one
//     16-byte load per lane reads 512 contiguous bytes (64 weights of each of
//     32 rows) and no lane ever needs a cross-lane reduction of dot products;
//   - the activations of all tokens sit in shared memory; every lane of a warp
//     reads the same 16 bytes at once (a broadcast), so activation traffic is
//     1/32 of a per-lane scheme;
//   - unpacking a 32-bit weight word (16 weights) is one AND per dp4a operand:
//     word & (0x03030303 << 2s) is 4 consecutive weights times 4^s, and slot s
//     accumulates in its own register (post, "the trick with 4 and 16"); the
//     unsigned x signed dp4a takes slot 3 (up to 128) without a shift;
//   - once per 128 weights: dot(u,q) = a0 + a1/4 + a2/16 + a3/64 (exact shifts),
//     minus the sum of the group's activations from the q8_K partial sums turns
//     u back into w (dot(w,y) = dot(u,y) - sum(y)), and one f32 FMA applies
//     d_w * d_x;
//   - warps of a CTA split the groups of a tile column; partial results are
//     summed in shared memory in a fixed order (deterministic output).
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxTok = 8;
// Groups per batch of weight loads kept in flight: deep for 1 token (bound
// by the weight stream), shallower when the dot products dominate.
template <int T>
__host__ __device__ constexpr int batch_for() { return T == 1 ? 4 : 2; }

struct GemvArgs {
  const uint8_t* Wtq;
  const uint8_t* Xq;
  float* Y;
  int32_t* S;
  int rows;
  int ngroups;   // cols / 128
  int nblk;      // cols / 256
  int nrb;       // row tiles
  int ksplit;    // warps per row tile
};

struct GroupCodes {
  uint4 lo, hi;     // weights 0..63 and 64..127 of this lane's row
  uint16_t scale;   // fp16 bits of d_w
};

__device__ __forceinline__ void load_group(const uint8_t* tile, int lane, GroupCodes& c) {
  c.lo = ldg_stream_v4(tile + lane * 16);
  c.hi = ldg_stream_v4(tile + 512 + lane * 16);
  c.scale = ldg_u16(tile + kTileCodeBytes + lane * 2);
}

template <int T, bool kGroupSums>
__device__ __forceinline__ void group_dot(const GroupCodes& c, int g, const int8_t* sq,
                                          const int* sgsum, const float* sdx, const GemvArgs& a,
                                          int row, float (&y)[T]) {
  const uint32_t wv[8] = {c.lo.x, c.lo.y, c.lo.z, c.lo.w, c.hi.x, c.hi.y, c.hi.z, c.hi.w};
  const float dw = __half2float(__ushort_as_half(c.scale));
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

template <int T, bool kGroupSums>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int cols = a.ngroups * kGroup;
  int8_t* sq = reinterpret_cast<int8_t*>(smem);                 // [T][cols]
  int* sgsum = reinterpret_cast<int*>(smem + T * cols);          // [T][ngroups]
  float* sdx = reinterpret_cast<float*>(sgsum + T * a.ngroups);  // [T][nblk]
  float* sred = sdx + T * a.nblk;                                // [kWarps][T][32]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_per_cta = kWarps / a.ksplit;
  const int rb = blockIdx.x * tiles_per_cta + warp / a.ksplit;
  const int part = warp % a.ksplit;
  const int g0 = (int)((int64_t)a.ngroups * part / a.ksplit);
  const int g1 = (int)((int64_t)a.ngroups * (part + 1) / a.ksplit);
  const bool active = rb < a.nrb;
  const int row = rb * kTileRows + lane;
  const uint8_t* tiles = a.Wtq + (int64_t)rb * a.ngroups * kTileBytes;

  constexpr int kBatch = batch_for<T>();
  // First batch of weights goes out before the activations are staged.
  GroupCodes cur[kBatch];
  if (active) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (g0 + u < g1) load_group(tiles + (int64_t)(g0 + u) * kTileBytes, lane, cur[u]);
  }

  // Stage q8_K activations: qs as a dense int8 [T][cols] array, the sum of each
  // 128-value half-block (8 partial sums), and the block scales.
  for (int tb = warp; tb < T * a.nblk; tb += kWarps) {
    const int t = tb / a.nblk, b = tb - t * a.nblk;
    const uint8_t* blk = a.Xq + (int64_t)tb * kQ8KBytes;
    const uint32_t* qs = reinterpret_cast<const uint32_t*>(blk + kQ8KQsOffset);
    uint32_t* dst = reinterpret_cast<uint32_t*>(sq + t * cols + b * kQK);
    dst[lane] = __ldg(qs + lane);
    dst[lane + 32] = __ldg(qs + lane + 32);
    int s = lane < 16 ? (int)__ldg(reinterpret_cast<const int16_t*>(blk + kQ8KBsumsOffset) + lane) : 0;
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    if (lane == 0 || lane == 8) sgsum[t * a.ngroups + 2 * b + (lane >> 3)] = s;
    if (lane == 0) sdx[tb] = __ldg(reinterpret_cast<const float*>(blk));
  }
  __syncthreads();

  float y[T];
#pragma unroll
  for (int t = 0; t < T; ++t) y[t] = 0.0f;

  if (active) {
    for (int gb = g0; gb < g1; gb += kBatch) {
      GroupCodes nxt[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (gb + kBatch + u < g1)
          load_group(tiles + (int64_t)(gb + kBatch + u) * kTileBytes, lane, nxt[u]);
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (gb + u < g1) group_dot<T, kGroupSums>(cur[u], gb + u, sq, sgsum, sdx, a, row, y);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) cur[u] = nxt[u];
    }
  }
  if (kGroupSums) return;

  if (a.ksplit > 1) {
#pragma unroll
    for (int t = 0; t < T; ++t) sred[(warp * T + t) * 32 + lane] = y[t];
    __syncthreads();
    if (part != 0) return;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float s = y[t];
      for (int k = 1; k < a.ksplit; ++k) s += sred[((warp + k) * T + t) * 32 + lane];
      y[t] = s;
    }
  }
  if (active && row < a.rows) {
#pragma unroll
    for (int t = 0; t < T; ++t) a.Y[(int64_t)t * a.rows + row] = y[t];
  }
}

template <int T, bool G>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&gemv_kernel<T, G>);
}

template <int T>
cudaError_t launch_t(const GemvArgs& a, dim3 grid, int smem, bool gsum, cudaStream_t s) {
  const void* fn = gsum ? kernel_ptr<T, true>() : kernel_ptr<T, false>();
  cudaError_t e = ensure_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return e;
  if (gsum)
    gemv_kernel<T, true><<<grid, kThreads, smem, s>>>(a);
  else
    gemv_kernel<T, false><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int gemv_max_tokens() { return kMaxTok; }

int64_t gemv_smem_bytes(int64_t cols, int ntok) {
  const int64_t g = cols / kGroup, b = cols / kQK;
  return ntok * cols + ntok * g * 4 + ntok * b * 4 + (int64_t)kWarps * ntok * 32 * 4;
}

cudaError_t launch_gemv(const uint8_t* Wtq, const uint8_t* Xq, float* Y, int32_t* S,
                        int64_t rows, int64_t cols, int ntok, cudaStream_t s) {
  if (ntok < 1 || ntok > kMaxTok) return cudaErrorNotSupported;
  const int64_t smem = gemv_smem_bytes(cols, ntok);
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > optin || rows > 0x7fffffff / 2) return cudaErrorNotSupported;

  GemvArgs a;
  a.Wtq = Wtq;
  a.Xq = Xq;
  a.Y = Y;
  a.S = S;
  a.rows = (int)rows;
  a.ngroups = (int)(cols / kGroup);
  a.nblk = (int)(cols / kQK);
  a.nrb = (int)((rows + kTileRows - 1) / kTileRows);
  // Split the groups of a tile column over more warps until ~2048 warps are
  // busy, keeping at least two groups per warp.
  int ksplit = 1;
  while (ksplit < kWarps && (int64_t)a.nrb * ksplit < 2048 && a.ngroups / (ksplit * 2) >= 2)
    ksplit *= 2;
  a.ksplit = ksplit;
  const int tiles_per_cta = kWarps / ksplit;
  const dim3 grid((unsigned)((a.nrb + tiles_per_cta - 1) / tiles_per_cta));
  const bool gsum = S != nullptr;
  switch (ntok) {
    case 1: return launch_t<1>(a, grid, (int)smem, gsum, s);
    case 2: return launch_t<2>(a, grid, (int)smem, gsum, s);
    case 3: return launch_t<3>(a, grid, (int)smem, gsum, s);
    case 4: return launch_t<4>(a, grid, (int)smem, gsum, s);
    case 5: return launch_t<5>(a, grid, (int)smem, gsum, s);
    case 6: return launch_t<6>(a, grid, (int)smem, gsum, s);
    case 7: return launch_t<7>(a, grid, (int)smem, gsum, s);
    default: return launch_t<8>(a, grid, (int)smem, gsum, s);
  }
}

}  // namespace tq
