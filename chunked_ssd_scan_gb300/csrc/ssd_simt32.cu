// Register-tiled CUDA-core chunked SSD forward for fp32 I/O with P = N = 64 and R | 64.
//
// Same chunk decomposition as the generic path (the serial.rs page's K1..K5, with the rotation
// absorbed into B and C as on the scan.py page):
//   phi kernels         : chunk-start angles (shared with the generic path)
//   simt_state_kernel   : K1 and K3 for one chunk, S_c[p][n] = sum_j exp(cum_end - cum_j) x_j[p] B~_j[n]
//   state_pass          : K4 across chunks (shared with the generic path)
//   simt_scan_kernel    : K2 and K5 for one chunk, in 64-row tiles:
//                         y_i = sum_{j <= i} exp(cum_i - cum_j) (C~_i . B~_j) x_j + exp(cum_i) C~_i . h_in
// With MIMO rank R the rows are the rank-fused rows i = t R + r (the serial.rs page's K2
// reshape), contiguous in memory, and a chunk is 64 / R steps = 64 rows; decays, angles and
// the causal cut use the step i / R of a row.
// Every contraction is a 64 x 64 x 64 block product from shared memory: each of the 256 threads
// owns a 4 x 4 output block and reads two float4 per k (16 FMAs per 32 bytes of shared memory).
// The tensor core is not used here on purpose: its fp32 accumulation truncates toward zero at
// every MMA, and with slowly decaying states the partial sums are large enough that the bias
// exceeds the fp32 tolerance (1e-4 (1 + |y|)) where y cancels; these kernels accumulate with
// round-to-nearest fp32 FMAs.  Exponentials use exp2f on double-float prefix sums, and the
// rotation uses sincosf on double-float angles.  A short last chunk (seqlen not a multiple of
// 64) reads its missing steps as zeros (dA = x = B = C = theta = 0) and writes no y for them.
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
// 64 floats per k row).  With kSwzA (kSwzB) the 16-byte chunks of At's (Bt's) row k are stored
// permuted, chunk c at c ^ ((k >> 2) & 15): the layouts the masked operand and the transposed
// h_in are written in.
// kmax (a multiple of 8, uniform over the warp) ends the reduction early where the rest of A's
// k rows are known to be zero.
template <bool kSwzA = false, bool kSwzB = false>
__device__ __forceinline__ void block_product(const float* __restrict__ At,
                                              const float* __restrict__ Bt, int ty, int tx,
                                              float (&acc)[4][4], int kmax = kT64) {
#pragma unroll 8
  for (int k = 0; k < kmax; ++k) {
    const int ca = kSwzA ? (ty ^ ((k >> 2) & 15)) : ty;
    const int cb = kSwzB ? (tx ^ ((k >> 2) & 15)) : tx;
    const float4 a = *reinterpret_cast<const float4*>(At + k * kT64 + 4 * ca);
    const float4 bq = *reinterpret_cast<const float4*>(Bt + k * kT64 + 4 * cb);
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

// Stages 64 rows (chunk steps s0 ..) of a B/C tensor turned by -Phi (if theta) into dst, either
// row-major dst[row][n] (transpose = false) or transposed dst[n][row].
__device__ void stage_bc64(const GenericParams& p, const float* __restrict__ src, int64_t b,
                           int64_t c, int64_t g, int s0, const float* ang, float* dst,
                           bool transpose) {
  const int tid = threadIdx.x;
  const int R = (int)p.R;
  const int64_t row0 = (b * p.T + c * p.l) * R;   // fused row of the chunk's first step
  const int nvr = steps64(p, b, c) * R;              // real rows of the chunk
  if (!transpose) {
    // row-major: the 16 lanes of a half-warp read and write one row (coalesced loads,
    // conflict-free shared stores)
    const int ch = tid & 15;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = (tid >> 4) + 16 * r;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 + row < nvr)
        f = __ldg(reinterpret_cast<const float4*>(src + ((row0 + s0 + row) * p.G + g) * kT64) +
                  ch);
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
    return;
  }
  const int row = tid >> 2, q0 = (tid & 3) * 16;   // 4 threads per row, 16 values each
  const bool real = s0 + row < nvr;
  const float4* s4 = reinterpret_cast<const float4*>(
      src + ((row0 + (real ? s0 + row : 0)) * p.G + g) * kT64 + q0);
  float v[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 f = real ? __ldg(s4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    v[4 * q] = f.x;
    v[4 * q + 1] = f.y;
    v[4 * q + 2] = f.z;
    v[4 * q + 3] = f.w;
  }
  if (p.theta) {
    const float* ar = ang + ((s0 + row) >> rank_shift(p)) * kPairs64 + q0 / 2;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float s, co;
      sincosf(ar[k], &s, &co);
      const float a = v[2 * k], bb = v[2 * k + 1];
      v[2 * k] = co * a + s * bb;
      v[2 * k + 1] = -s * a + co * bb;
    }
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) dst[(q0 + k) * kT64 + row] = v[k];
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
      stage_bc64(p, static_cast<const float*>(p.B), b, c, g, j0, ang, bs, false);
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

// ---------------------------------------------------------------------------------- K2 + K5
// smem: C~^T [n][i] of the row tile, h_in^T [n][p], B~^T [n][j] (rewritten as (L o CB)^T [j][i]
// once CB is in registers), x [j][p], prefix sums, angles.
size_t simt_scan_smem(int64_t l, bool theta) {
  return sizeof(float) * (4 * kTileFloats + 2 * l + (theta ? l * kPairs64 : 0));
}

__global__ void __launch_bounds__(kSimtThreads, 3) simt_scan_kernel(GenericParams p) {
  extern __shared__ __align__(16) float sm64[];
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int l = (int)p.l;
  float* ct = sm64;                        // C~^T [n][i]
  float* ht = ct + kTileFloats;            // h_in^T [n][p]
  float* bt = ht + kTileFloats;            // B~^T [n][j], then M^T [j][i]
  float* xs = bt + kTileFloats;            // x [j][p]
  float* cum_hi = xs + kTileFloats;
  float* cum_lo = cum_hi + l;
  float* ang = cum_lo + l;
  // theta and the first x tile are in flight while the prefix sums and h_in are staged
  if (p.theta) issue_theta64(p, b, c, h, l, ang);
  {
    const float* xsrc = static_cast<const float*>(p.x);
    const int nvr = steps64(p, b, c) * (int)p.R;
    const int64_t row0 = (b * p.T + c * p.l) * p.R;
    for (int e = threadIdx.x; e < kTileFloats / 4; e += kSimtThreads) {
      const int row = e / (kT64 / 4), q = e % (kT64 / 4);
      const bool real = row < nvr;   // rows after the real ones are zero-filled
      cp_async16(xs + row * kT64 + 4 * q,
                 xsrc + ((row0 + (real ? row : 0)) * p.H + h) * kT64 + 4 * q, real ? 16 : 0);
    }
  }
  chunk_prefix64(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, steps64(p, b, c), cum_hi, cum_lo,
                 nullptr);
  {
    // h_in [p][n] (written over S by the state pass) -> h^T [n][p] with the 16-byte chunks of
    // row n permuted (chunk c at c ^ ((n >> 2) & 15)): half-warps read whole rows p as float4
    // (coalesced), and the transposed scalar stores of a warp then spread over the bank groups
    const float4* hin = reinterpret_cast<const float4*>(
        p.states + ((b * p.nch + c) * p.H + h) * kTileFloats);
    for (int e = threadIdx.x; e < kTileFloats / 4; e += kSimtThreads) {
      const int pp = e >> 4, q = e & 15;   // row p, n = 4 q .. 4 q + 3
      const float4 v = __ldg(hin + e);
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ht[(4 * q + i) * kT64 + 4 * ((pp >> 2) ^ q) + (pp & 3)] = vv[i];
    }
  }
  if (p.theta) {
    chunk_angles64(p, b, c, h, l, ang, true);
  } else {
    cp_async_wait_all();
    __syncthreads();
  }
  const int tx = tile_tx(), ty = tile_ty();   // rows i = 4 ty.., cols 4 tx..
  const float* Csrc = static_cast<const float*>(p.C);
  const float* Bsrc = static_cast<const float*>(p.B);
  const int R = (int)p.R, rs = rank_shift(p);
  for (int i0 = 0; i0 < l * R; i0 += kT64) {   // fused rows
    stage_bc64(p, Csrc, b, c, g, i0, ang, ct, true);
    __syncthreads();
    float yo[4][4] = {};
    block_product<false, true>(ct, ht, ty, tx, yo);   // Yo[i][p] = sum_n C~[i][n] h[p][n]
    float yd[4][4] = {};
    for (int j0 = 0; j0 <= i0; j0 += kT64) {
      stage_bc64(p, Bsrc, b, c, g, j0, ang, bt, true);
      if (j0 > 0 || i0 > 0) stage_x64(p, b, c, h, j0, nullptr, xs);   // tile 0 was prefetched
      __syncthreads();
      // On the diagonal tile this warp's rows i0 + 16 (w >> 1) .. + 15 see no source row of a
      // later step: its C~B~ block is skipped when every column is such a row (the mask below
      // then writes zeros), and its (L o CB) x product stops at the first such row.
      const bool diag = j0 == i0;
      const int wrow = i0 + 16 * (threadIdx.x >> 6) + 15, wcol = j0 + 32 * ((threadIdx.x >> 5) & 1);
      const bool cb_zero = diag && (wcol >> rs) > (wrow >> rs);
      const int kmax = diag ? min(kT64, (((wrow >> rs) + 1) << rs) - j0) : kT64;
      float cb[4][4] = {};
      if (!cb_zero) block_product(ct, bt, ty, tx, cb);   // CB[i][j] = sum_n C~[i][n] B~[j][n]
      __syncthreads();                     // every read of B~^T done before M^T overwrites it
      // (L o CB)^T: causal cut before the exponential
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int tj = (j0 + 4 * tx + jj) >> rs;   // step of source row j
        float m[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int ti = (i0 + 4 * ty + r) >> rs;
          m[r] = tj <= ti ? exp2f((cum_hi[ti] - cum_hi[tj]) + (cum_lo[ti] - cum_lo[tj])) * cb[r][jj]
                          : 0.f;
        }
        // row 4 tx + jj, chunk ty permuted by the row: per instruction the warp writes 8 rows
        // (consecutive tx) and, in each, the chunks ty ^ tx of 4 consecutive ty, which hit every
        // bank group once per four lanes (conflict-free)
        *reinterpret_cast<float4*>(bt + (4 * tx + jj) * kT64 + 4 * (ty ^ tx)) =
            make_float4(m[0], m[1], m[2], m[3]);
      }
      __syncthreads();
      block_product<true>(bt, xs, ty, tx, yd, kmax);   // Yd[i][p] += sum_j M[i][j] x[j][p]
      if (j0 < i0) __syncthreads();   // the next source tile overwrites B~^T / M^T and x
    }
    const int nvr = steps64(p, b, c) * R;
    const int64_t row0 = (b * p.T + c * p.l) * R;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int si = i0 + 4 * ty + r;
      if (si >= nvr) continue;   // padding row of a short last chunk
      const int ti = si >> rs;
      const float sc = exp2f(cum_hi[ti] + cum_lo[ti]);   // exp(cum of row i's step)
      float* yrow = static_cast<float*>(p.y) + ((row0 + si) * p.H + h) * kT64;
      if (SSD_INDEX_OK(p.hdr, ((row0 + si) * p.H + h) * kT64 + 4 * tx + 3,
                       p.batch * p.T * p.R * p.H * kT64, 21))
      *reinterpret_cast<float4*>(yrow + 4 * tx) =
          make_float4(fmaf(sc, yo[r][0], yd[r][0]), fmaf(sc, yo[r][1], yd[r][1]),
                      fmaf(sc, yo[r][2], yd[r][2]), fmaf(sc, yo[r][3], yd[r][3]));
    }
    // the next row tile restages C~^T, B~^T and x; after the last one the warps that finished
    // their (shorter) masked product early retire without waiting
    if (i0 + kT64 < l * R) __syncthreads();
  }
}

}  // namespace

bool simt32_supported(int64_t P, int64_t N, int64_t R, int64_t l, bool bf16, bool theta) {
  if (bf16 || P != kT64 || N != kT64 || R < 1 || R > kT64 || (kT64 % R) != 0) return false;
  if (l < kT64 || l > kMaxChunk64 || (l % kT64) != 0) return false;
  return simt_state_smem(l, theta) <= 227 * 1024 && simt_scan_smem(l, theta) <= 227 * 1024;
}

cudaError_t simt32_forward(const GenericParams& p, cudaStream_t st, bool tc_scan) {
  cudaError_t e;
  const bool th = p.theta != nullptr;
  if (th && (e = generic_phi(p, st)) != cudaSuccess) return e;
  const size_t s1 = simt_state_smem(p.l, th), s2 = simt_scan_smem(p.l, th);
  if ((e = cudaFuncSetAttribute(simt_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)s1)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(simt_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)s2)) != cudaSuccess)
    return e;
  const dim3 grid((unsigned)p.nch, (unsigned)p.H, (unsigned)p.batch);
  simt_state_kernel<<<grid, kSimtThreads, s1, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = generic_state_pass(p, st)) != cudaSuccess) return e;
  if (tc_scan) return tc32_scan(p, st);
  simt_scan_kernel<<<grid, kSimtThreads, s2, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ssd
