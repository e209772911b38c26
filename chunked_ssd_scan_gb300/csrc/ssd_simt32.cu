// fp32 chunked SSD forward for P = N = 64 and R | 64: the chunk states on the CUDA cores and the
// chunk scan on the tensor core.
//
// Same chunk decomposition as the generic path (the serial.rs page's K1..K5, with the rotation
// absorbed into B and C as on the scan.py page), over chunks of 128 rank-fused rows (128 / R
// steps; rows i = t R + r are contiguous in memory, and decays, angles and the causal cut use
// the step i / R of a row):
//   phi kernels         : chunk-start angles (shared with the generic path)
//   simt_state_kernel   : K1 and K3 for one chunk, S_c[p][n] = sum_j exp(cum_end - cum_j) x_j[p] B~_j[n],
//                         as 64 x 64 x 64 block products from shared memory (each of the 256
//                         threads owns a 4 x 4 output block and reads two float4 per k), fp32
//                         FMAs rounding to nearest
//   state_pass          : K4 across chunks (shared with the generic path)
//   tc32_scan           : K2 and K5 on tcgen05 kind::tf32 with split operands (ssd_tc32.cu)
// Exponentials use exp2f on double-float prefix sums, and the rotation uses sincosf on
// double-float angles.  A short last chunk (seqlen not a multiple of the chunk) reads its missing
// steps as zeros (dA = x = B = C = theta = 0).
#include <math.h>

#include "common.cuh"
#include "fp_helpers.cuh"
#include "ssd_internal.h"
#include "chunk_prep.cuh"

namespace ssd {

namespace {

using namespace fp;
using namespace prep;

constexpr int kT64 = 64;                     // tile edge (rows, sources, P and N)
constexpr int kSimtThreads = kPrepThreads;
constexpr int kMaxChunk64 = 512;
constexpr int kTileFloats = kT64 * kT64;

// Owner of the 4 x 4 output block (rows 4 ty.., cols 4 tx..) of a 64 x 64 product: each warp
// covers 4 consecutive ty by 8 consecutive tx, so per k its A reads are 64 contiguous bytes and
// its B reads 128 contiguous bytes -- one shared-memory wavefront each (a 2 x 16 warp shape
// needs three).
__device__ __forceinline__ int tile_tx() {
  return (threadIdx.x & 7) + 8 * ((threadIdx.x >> 5) & 1);
}
__device__ __forceinline__ int tile_ty() {
  return ((threadIdx.x >> 3) & 3) + 4 * (threadIdx.x >> 6);
}

// acc[r][c] += sum_k At[k][4 ty + r] * Bt[k][4 tx + c] over k < 64 (both operands k-major,
// 64 floats per k row).
__device__ __forceinline__ void block_product(const float* __restrict__ At,
                                              const float* __restrict__ Bt, int ty, int tx,
                                              float (&acc)[4][4]) {
#pragma unroll 8
  for (int k = 0; k < kT64; ++k) {
    const float4 a = *reinterpret_cast<const float4*>(At + k * kT64 + 4 * ty);
    const float4 bq = *reinterpret_cast<const float4*>(Bt + k * kT64 + 4 * tx);
    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float2 lo = fma2(make_float2(av[r], av[r]), make_float2(bq.x, bq.y),
                             make_float2(acc[r][0], acc[r][1]));
      const float2 hi = fma2(make_float2(av[r], av[r]), make_float2(bq.z, bq.w),
                             make_float2(acc[r][2], acc[r][3]));
      acc[r][0] = lo.x;
      acc[r][1] = lo.y;
      acc[r][2] = hi.x;
      acc[r][3] = hi.y;
    }
  }
}

// Stages 64 rows (fused rows s0 .. of the chunk) of a B/C tensor turned by -Phi (if theta) into
// dst[row][n]: the 16 lanes of a half-warp read and write one row (coalesced loads,
// conflict-free shared stores).
__device__ void stage_bc64(const GenericParams& p, const float* __restrict__ src, int64_t b,
                           int64_t c, int64_t g, int s0, const float* ang, float* dst) {
  const int tid = threadIdx.x;
  const int R = (int)p.R;
  const int64_t row0 = (b * p.T + c * p.l) * R;   // fused row of the chunk's first step
  const int nvr = steps64(p, b, c) * R;              // real rows of the chunk
  const int ch = tid & 15;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = (tid >> 4) + 16 * r;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (s0 + row < nvr)
      f = __ldg(reinterpret_cast<const float4*>(src + ((row0 + s0 + row) * p.G + g) * kT64) + ch);
    if (p.theta) {
      const float* ar = ang + ((s0 + row) >> rank_shift(p)) * kPairs64 + 2 * ch;
      float s, co;
      sincosf(ar[0], &s, &co);
      const float e0 = co * f.x + s * f.y, o0 = -s * f.x + co * f.y;
      sincosf(ar[1], &s, &co);
      const float e1 = co * f.z + s * f.w, o1 = -s * f.z + co * f.w;
      f = make_float4(e0, o0, e1, o1);
    }
    *reinterpret_cast<float4*>(dst + row * kT64 + 4 * ch) = f;
  }
}

// Stages 64 x rows (fused rows s0 .. of the chunk) into dst[row][p], each row scaled by
// scale[step of the row] if given.
__device__ void stage_x64(const GenericParams& p, int64_t b, int64_t c, int64_t h, int s0,
                          const float* scale, float* dst) {
  const int tid = threadIdx.x;
  const int ch = tid & 15;   // half-warps read and write whole rows
  const int R = (int)p.R;
  const int64_t row0 = (b * p.T + c * p.l) * R;
  const int nvr = steps64(p, b, c) * R;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = (tid >> 4) + 16 * r;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (s0 + row < nvr)
      f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.x) +
                                                ((row0 + s0 + row) * p.H + h) * kT64) +
                ch);
    const float w = scale ? scale[(s0 + row) >> rank_shift(p)] : 1.f;
    *reinterpret_cast<float4*>(dst + row * kT64 + 4 * ch) =
        make_float4(f.x * w, f.y * w, f.z * w, f.w * w);
  }
}

// ---------------------------------------------------------------------------------- K1 + K3
size_t simt_state_smem(int64_t l, bool theta) {
  return sizeof(float) * (2 * kTileFloats + 3 * l + (theta ? l * kPairs64 : 0) + 4);
}

// Raw x and B rows of the chunk's first 64 fused rows into xs[row][p] and bs[row][n] with
// 16-byte cp.async (not waited for); rows past the chunk's real ones are zero-filled.
__device__ void issue_rows64(const GenericParams& p, int64_t b, int64_t c, int64_t h, int64_t g,
                             float* xs, float* bs) {
  const float* xsrc = static_cast<const float*>(p.x);
  const float* bsrc = static_cast<const float*>(p.B);
  const int nvr = steps64(p, b, c) * (int)p.R;
  const int64_t row0 = (b * p.T + c * p.l) * p.R;
  for (int e = threadIdx.x; e < kTileFloats / 4; e += kSimtThreads) {
    const int row = e / (kT64 / 4), q = e % (kT64 / 4);
    const bool real = row < nvr;
    const int64_t r = row0 + (real ? row : 0);
    cp_async16(xs + row * kT64 + 4 * q, xsrc + (r * p.H + h) * kT64 + 4 * q, real ? 16 : 0);
    cp_async16(bs + row * kT64 + 4 * q, bsrc + (r * p.G + g) * kT64 + 4 * q, real ? 16 : 0);
  }
}

__global__ void __launch_bounds__(kSimtThreads) simt_state_kernel(GenericParams p) {
  extern __shared__ __align__(16) float sm64[];
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int l = (int)p.l;
  float* xs = sm64;                        // X~ [j][p] of one 64-step block
  float* bs = xs + kTileFloats;            // B~ [j][n]
  float* cum_hi = bs + kTileFloats;
  float* cum_lo = cum_hi + l;
  float* dec = cum_lo + l;
  float* ang = dec + l;
  float* total = ang + (p.theta ? l * kPairs64 : 0);
  // the first block's raw rows are in flight while the prefix sums and the angles are formed
  issue_rows64(p, b, c, h, g, xs, bs);
  chunk_prefix64(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, steps64(p, b, c), cum_hi, cum_lo,
                 total);
  if (p.theta) {
    chunk_angles64(p, b, c, h, l, ang);   // its wait covers the rows too
  } else {
    __syncthreads();
  }
  for (int t = threadIdx.x; t < l; t += kSimtThreads)
    dec[t] = exp2f((cum_hi[l - 1] - cum_hi[t]) + (cum_lo[l - 1] - cum_lo[t]));
  cp_async_wait_all();
  __syncthreads();
  const int tx = tile_tx(), ty = tile_ty();   // output rows p = 4 ty.., cols n = 4 tx..
  const int rs = rank_shift(p);
  float acc[4][4] = {};
  for (int j0 = 0; j0 < l * (int)p.R; j0 += kT64) {   // fused rows
    if (j0 == 0) {
      // in place: x rows scaled by the decay to the chunk end, B rows turned by -Phi
      for (int e = threadIdx.x; e < kTileFloats / 4; e += kSimtThreads) {
        const int row = e / (kT64 / 4);
        float4* x4 = reinterpret_cast<float4*>(xs) + e;
        const float w = dec[row >> rs];
        const float4 v = *x4;
        *x4 = make_float4(v.x * w, v.y * w, v.z * w, v.w * w);
      }
      if (p.theta) {
        for (int e = threadIdx.x; e < kTileFloats / 2; e += kSimtThreads) {
          const int row = e / kPairs64, k = e % kPairs64;
          float2* b2 = reinterpret_cast<float2*>(bs) + e;
          float sn, co;
          sincosf(ang[(row >> rs) * kPairs64 + k], &sn, &co);
          const float2 v = *b2;
          *b2 = make_float2(co * v.x + sn * v.y, -sn * v.x + co * v.y);
        }
      }
    } else {
      stage_x64(p, b, c, h, j0, dec, xs);
      stage_bc64(p, static_cast<const float*>(p.B), b, c, g, j0, ang, bs);
    }
    __syncthreads();
    block_product(xs, bs, ty, tx, acc);   // S[p][n] += sum_j X~[j][p] B~[j][n]
    __syncthreads();
  }
  float* dst = p.states + ((b * p.nch + c) * p.H + h) * kTileFloats;
#pragma unroll
  for (int r = 0; r < 4; ++r)
    if (SSD_INDEX_OK(p.hdr, (dst - p.states) + (4 * ty + r) * kT64 + 4 * tx + 3,
                     p.batch * p.nch * p.H * kTileFloats, 20))
      *reinterpret_cast<float4*>(dst + (4 * ty + r) * kT64 + 4 * tx) =
          make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  if (threadIdx.x == 0 &&
      SSD_INDEX_OK(p.hdr, (b * p.nch + c) * p.H + h, p.batch * p.nch * p.H, 22))
    p.cend[(b * p.nch + c) * p.H + h] = *total;
}

}  // namespace

cudaError_t fp32_forward(const GenericParams& p, cudaStream_t st) {
  cudaError_t e;
  const bool th = p.theta != nullptr;
  if (p.P != kT64 || p.N != kT64 || p.l * p.R > kMaxChunk64) return cudaErrorInvalidValue;
  if (th && (e = generic_phi(p, st)) != cudaSuccess) return e;
  const size_t s1 = simt_state_smem(p.l, th);
  if ((e = cudaFuncSetAttribute(simt_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)s1)) != cudaSuccess)
    return e;
  const dim3 grid((unsigned)p.nch, (unsigned)p.H, (unsigned)p.batch);
  simt_state_kernel<<<grid, kSimtThreads, s1, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = generic_state_pass(p, st)) != cudaSuccess) return e;
  return tc32_scan(p, st);
}

}  // namespace ssd
