// Generic CUDA-core chunked SSD pipeline (fp32 arithmetic, f32 or bf16 I/O).
//
// It follows the K1..K5 chunk decomposition of the serial.rs page (burn_mamba
// mamba3/ssd/serial.rs) as three launches plus two small rotation launches:
//   phi_chunk_sum / phi_prefix : chunk-start cumulative angles Phi (scan.py page,
//                                cumulative_angles), carried across chunks in fp64 and reduced
//                                to [-pi, pi] before use.
//   chunk_state  (K1 + K3)     : intra-chunk cumsum of dA and the chunk-end state
//                                S_c = sum_i exp(cum_end - cum[i//R]) x_i (outer) B~_i.
//   state_pass   (K4)          : h_in(c+1) = exp(cum_end(c)) h_in(c) + S_c, in place over S,
//                                final state turned back to the physical frame by R(Phi_{T-1}).
//   chunk_scan   (K2 + K5)     : y_i = sum_{j//R <= i//R} exp(cum[i//R]-cum[j//R]) (C~_i.B~_j) x_j
//                                      + exp(cum[i//R]) C~_i . h_in.
// B~ / C~ are B / C turned by -Phi_t (scan.py page, module docstring "THE TRICK": the rotation
// is absorbed into B and C so the scan itself is the plain scalar-decay recurrence).
// The causal mask is applied before the exponential (scan.py page, chunked_scan: masked entries
// are never exponentiated).
//
// This path handles every supported shape; the fused tensor-core kernels take over the shapes
// they implement.  When seqlen is not a multiple of the chunk length the last chunk is short:
// its missing steps read as dA = 0, x = 0 and B = C = theta = 0 (zero padding, which leaves y of
// the real steps and the final state unchanged) and their y is not written.
#include <math.h>

#include "common.cuh"
#include "fp_helpers.cuh"
#include "ssd_internal.h"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kStateRows = 16;   // rows of x/B staged per step in chunk_state
constexpr int kScanRows = 64;    // output rows per chunk_scan block
constexpr int kScanCols = 32;    // source rows per chunk_scan step
constexpr double kTwoPi = 6.283185307179586476925286766559;

// Block-cooperative inclusive cumsum of l values read with stride `stride` (warp 0 does it);
// values at or after nv read as zero.
// The prefix sums are accumulated in fp64 and kept as an unevaluated float pair hi + lo, so that
// the segment sums cum[i] - cum[j] of the decay mask are exact to about one float ulp of the
// difference itself (not of |cum|, which reaches hundreds within a chunk); this is the
// segsum.rs page's difference-of-prefix-sums form with the rounding of the large prefix
// removed.
__device__ void chunk_cumsum(const float* __restrict__ src, int64_t stride, int l, int nv,
                             float* s_hi, float* s_lo) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (l + 31) / 32;
    const int beg = min(l, lane * per);
    const int end = min(l, beg + per);
    double s = 0.0;
    for (int t = beg; t < min(end, nv); ++t) s += (double)__ldg(src + (int64_t)t * stride);
    double incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    double acc = incl - s;
    for (int t = beg; t < end; ++t) {
      if (t < nv) acc += (double)__ldg(src + (int64_t)t * stride);
      const float hi = (float)acc;
      s_hi[t] = hi;
      s_lo[t] = (float)(acc - (double)hi);
    }
  }
}

// exp(cum[i] - cum[j]) from the hi/lo prefix pairs.
__device__ __forceinline__ float seg_exp(const float* hi, const float* lo, int i, int j) {
  return expf((hi[i] - hi[j]) + (lo[i] - lo[j]));
}

// Real steps of chunk c of sequence b: the last chunk may be short, and with per-sequence valid
// lengths the steps from valid_len[b] on are padding (none of them is read).
__device__ __forceinline__ int chunk_steps(const GenericParams& p, int64_t b, int64_t c) {
  return (int)max((int64_t)0, min(p.l, seq_steps(p, b) - c * p.l));
}

// x reduced to [-pi, pi] (fp64 in, fp32 out).
__device__ inline float reduce_two_pi(double a) {
  return (float)(a - kTwoPi * rint(a * (1.0 / kTwoPi)));
}

// Angles Phi_t for every step of the chunk, reduced to [-pi, pi].  The running sum over the
// chunk is carried in fp64 from the fp64 chunk-start angle: an angle error e turns every
// absorbed term by e, so Phi must be accurate to a few float ulps of pi, not of |Phi|.
__device__ void chunk_angles(const GenericParams& p, int64_t b, int64_t c, int64_t h,
                             float* s_ang) {
  const int64_t K = p.N / 2;
  const int nv = chunk_steps(p, b, c);
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
    double acc = p.phi[((b * (p.nch + 1) + c) * p.H + h) * K + k];
    const float* th = p.theta + ((b * p.T + c * p.l) * p.H + h) * K + k;
    for (int64_t t = 0; t < p.l; ++t) {
      if (t < nv) acc += (double)__ldg(th + t * p.H * K);
      s_ang[t * K + k] = reduce_two_pi(acc);
    }
  }
}

// Stage `rows` rows of a B/C tensor (fused row index, rotated by -Phi when theta is given).
template <typename T>
__device__ void stage_bc_rows(const GenericParams& p, const T* __restrict__ src, int64_t b,
                              int64_t c, int64_t g, int64_t row0, int rows, const float* s_ang,
                              float* dst, int ld) {
  const int64_t L = (int64_t)chunk_steps(p, b, c) * p.R;   // real rows of the chunk
  const int64_t N = p.N;
  const int64_t base = ((b * p.T + c * p.l) * p.R) * p.G + g;   // fused row 0, group g
  if (p.theta == nullptr) {
    for (int e = threadIdx.x; e < rows * N; e += blockDim.x) {
      const int r = e / (int)N, n = e % (int)N;
      const int64_t i = row0 + r;
      float v = 0.f;
      if (i < L) v = ld_f32(src + (base + i * p.G) * N + n);
      dst[r * ld + n] = v;
    }
  } else {
    const int K = (int)(N / 2);
    for (int e = threadIdx.x; e < rows * K; e += blockDim.x) {
      const int r = e / K, k = e % K;
      const int64_t i = row0 + r;
      float ev = 0.f, od = 0.f;
      if (i < L) {
        const T* q = src + (base + i * p.G) * N + 2 * k;
        const float a = ld_f32(q), bb = ld_f32(q + 1);
        float s, co;
        sincosf(s_ang[(i / p.R) * K + k], &s, &co);   // turn by -Phi: sin(-x) = -sin(x)
        ev = co * a + s * bb;
        od = -s * a + co * bb;
      }
      dst[r * ld + 2 * k] = ev;
      dst[r * ld + 2 * k + 1] = od;
    }
  }
}

// Per-chunk theta sums: one warp per chunk, lanes over pairs (loads coalesced over the pairs of
// one step), kPhiChunksPerBlock chunks per block; the sum is carried as a double-float (TwoSum)
// pair, which is exact enough for the fp64 chunk sums and avoids a chain of slow fp64 adds.
constexpr int kPhiThreads = 256;
constexpr int kPhiChunksPerBlock = kPhiThreads / 32;

__global__ void __launch_bounds__(kPhiThreads) phi_chunk_sum_kernel(GenericParams p) {
  const int64_t c = (int64_t)blockIdx.x * kPhiChunksPerBlock + threadIdx.x / 32;
  const int64_t h = blockIdx.y, b = blockIdx.z;
  if (c >= p.nch) return;
  const int64_t K = p.N / 2;
  for (int64_t k = threadIdx.x % 32; k < K; k += 32) {
    const float* th = p.theta + ((b * p.T + c * p.l) * p.H + h) * K + k;
    fp::DF s = {0.f, 0.f};
    const int nv = chunk_steps(p, b, c);
    for (int64_t t = 0; t < nv; ++t) s = fp::df_add(s, fp::DF{__ldg(th + t * p.H * K), 0.f});
    const int64_t o = ((b * p.nch + c) * p.H + h) * K + k;
    if (SSD_INDEX_OK(p.hdr, o, p.batch * p.nch * p.H * K, 16))
      p.phisum[o] = (double)s.hi + (double)s.lo;
  }
}

// Chunk-start angles: an exclusive fp64 prefix of the chunk sums per (batch, head, pair),
// reduced to [-pi, pi].  One warp per (batch, head, pair): each lane sums a contiguous run of
// chunks, the lane totals are scanned with shuffles, and each lane then writes its run.
__global__ void phi_prefix_kernel(GenericParams p) {
  const int64_t K = p.N / 2;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (wid >= p.batch * p.H * K) return;   // uniform over the warp
  const int64_t k = wid % K, h = (wid / K) % p.H, b = wid / (K * p.H);
  const double* src = p.phisum + (b * p.nch * p.H + h) * K + k;   // + c * H * K
  double* dst = p.phi + (b * (p.nch + 1) * p.H + h) * K + k;
  const int64_t cs = p.H * K;
  const int64_t per = (p.nch + 31) / 32;
  const int64_t c0 = min((int64_t)lane * per, p.nch), c1 = min(c0 + per, p.nch);
  double run = 0.0;
  for (int64_t c = c0; c < c1; ++c) run += src[c * cs];
  double incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  double acc = incl - run;   // exclusive prefix of this lane's first chunk
  const int64_t phi_elems = p.batch * (p.nch + 1) * p.H * K;
  for (int64_t c = c0; c < c1; ++c) {
    if (SSD_INDEX_OK(p.hdr, (dst - p.phi) + c * cs, phi_elems, 15))
      dst[c * cs] = acc - kTwoPi * rint(acc * (1.0 / kTwoPi));
    acc += src[c * cs];
  }
  if (lane == 31 && SSD_INDEX_OK(p.hdr, (dst - p.phi) + p.nch * cs, phi_elems, 15))
    dst[p.nch * cs] = incl - kTwoPi * rint(incl * (1.0 / kTwoPi));
}

template <typename T, int OPT>
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(GenericParams p) {
  extern __shared__ float smem[];
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int l = (int)p.l, R = (int)p.R, L = l * R;
  const int P = (int)p.P, N = (int)p.N;
  float* s_cum = smem;                       // [l] prefix sums, hi part
  float* s_lo = s_cum + l;                   // [l] prefix sums, lo part
  float* s_dec = s_lo + l;                   // [l]
  float* s_x = s_dec + l;                    // [kStateRows][P]
  float* s_B = s_x + kStateRows * P;         // [kStateRows][N]
  float* s_ang = s_B + kStateRows * N;       // [l][N/2] when theta

  const int Lv = chunk_steps(p, b, c) * R;     // real rows of the chunk
  chunk_cumsum(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, Lv / R, s_cum, s_lo);
  if (p.theta) chunk_angles(p, b, c, h, s_ang);
  __syncthreads();
  const float cum_end = s_cum[l - 1] + s_lo[l - 1];
  for (int t = threadIdx.x; t < l; t += blockDim.x) s_dec[t] = seg_exp(s_cum, s_lo, l - 1, t);

  float acc[OPT];
#pragma unroll
  for (int k = 0; k < OPT; ++k) acc[k] = 0.f;

  const T* xs = static_cast<const T*>(p.x);
  const int64_t xbase = (((b * p.T + c * p.l) * p.R) * p.H + h) * p.P;   // fused row 0
  for (int i0 = 0; i0 < L; i0 += kStateRows) {
    __syncthreads();
    const int rows = min(kStateRows, L - i0);
    for (int e = threadIdx.x; e < kStateRows * P; e += blockDim.x) {
      const int r = e / P, pp = e % P;
      s_x[e] = (r < rows && i0 + r < Lv)
                   ? ld_f32(xs + xbase + (int64_t)(i0 + r) * p.H * p.P + pp)
                   : 0.f;
    }
    stage_bc_rows(p, static_cast<const T*>(p.B), b, c, g, i0, kStateRows, s_ang, s_B, N);
    __syncthreads();
    for (int r = 0; r < rows; ++r) {
      const float w = s_dec[(i0 + r) / R];
#pragma unroll
      for (int k = 0; k < OPT; ++k) {
        const int o = threadIdx.x + k * kThreads;
        if (o < P * N) acc[k] += (w * s_x[r * P + o / N]) * s_B[r * N + o % N];
      }
    }
  }
  float* dst = p.states + ((b * p.nch + c) * p.H + h) * p.P * p.N;
#pragma unroll
  for (int k = 0; k < OPT; ++k) {
    const int o = threadIdx.x + k * kThreads;
    if (o < P * N && SSD_INDEX_OK(p.hdr, (dst - p.states) + o, p.batch * p.nch * p.H * P * N, 10))
      dst[o] = acc[k];
  }
  if (threadIdx.x == 0 &&
      SSD_INDEX_OK(p.hdr, (b * p.nch + c) * p.H + h, p.batch * p.nch * p.H, 11))
    p.cend[(b * p.nch + c) * p.H + h] = cum_end;
}

// One thread carries one state element (or, with rotation, one interleaved pair) of one
// (batch, head) through all chunks; the grid covers every element of every (batch, head), and
// the chunk states are loaded kStatePrefetch chunks ahead of the serial update.
constexpr int kStatePrefetch = 16;

template <bool kPairs>
__global__ void __launch_bounds__(kThreads) state_pass_kernel(GenericParams p) {
  const int64_t PN = p.P * p.N, K = p.N / 2;
  constexpr int W = kPairs ? 2 : 1;
  const int64_t per_bh = PN / W;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.batch * p.H * per_bh) return;
  const int64_t bh = idx / per_bh, q = idx % per_bh;
  const int64_t b = bh / p.H, h = bh % p.H;
  const int64_t off = W * q;
  const int64_t cstride = p.H * PN;              // from chunk c to c + 1 in states
  float* sp = p.states + ((b * p.nch) * p.H + h) * PN + off;
  const float* ce = p.cend + (b * p.nch) * p.H + h;
  float hv[W];
#pragma unroll
  for (int w = 0; w < W; ++w) hv[w] = p.init ? p.init[(b * p.H + h) * PN + off + w] : 0.f;
  for (int64_t c0 = 0; c0 < p.nch; c0 += kStatePrefetch) {
    float sv[kStatePrefetch][W], av[kStatePrefetch];
#pragma unroll
    for (int k = 0; k < kStatePrefetch; ++k) {
      if (c0 + k < p.nch) {
        av[k] = ce[(c0 + k) * p.H];
#pragma unroll
        for (int w = 0; w < W; ++w) sv[k][w] = sp[(c0 + k) * cstride + w];
      }
    }
#pragma unroll
    for (int k = 0; k < kStatePrefetch; ++k) {
      if (c0 + k < p.nch) {
        const float a = expf(av[k]);
#pragma unroll
        for (int w = 0; w < W; ++w) {
          if (SSD_INDEX_OK(p.hdr, (sp - p.states) + (c0 + k) * cstride + w,
                           p.batch * p.nch * p.H * PN, 12))
            sp[(c0 + k) * cstride + w] = hv[w];
          hv[w] = a * hv[w] + sv[k][w];
        }
      }
    }
  }
  if (kPairs) {
    // back to the physical frame: turn the pair by +Phi_{T-1}
    const float ang =
        reduce_two_pi(p.phi[((b * (p.nch + 1) + p.nch) * p.H + h) * K + (off % p.N) / 2]);
    float s, co;
    sincosf(ang, &s, &co);
    const float e = co * hv[0] - s * hv[W - 1], o = s * hv[0] + co * hv[W - 1];
    hv[0] = e;
    hv[W - 1] = o;
  }
  if (p.final_state) {
#pragma unroll
    for (int w = 0; w < W; ++w)
      if (SSD_INDEX_OK(p.hdr, (b * p.H + h) * PN + off + w, p.batch * p.H * PN, 13))
        p.final_state[(b * p.H + h) * PN + off + w] = hv[w];
  }
}

template <typename T, int PPT>
__global__ void __launch_bounds__(kThreads) chunk_scan_kernel(GenericParams p) {
  extern __shared__ float smem[];
  const int l = (int)p.l, R = (int)p.R, L = l * R;
  const int P = (int)p.P, N = (int)p.N;
  const int tiles = (L + kScanRows - 1) / kScanRows;
  const int64_t c = blockIdx.x / tiles;
  const int i0 = (int)(blockIdx.x % tiles) * kScanRows;
  const int64_t h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int ldn = N + 1;
  float* s_cum = smem;                               // [l] prefix sums, hi part
  float* s_lo = s_cum + l;                           // [l] prefix sums, lo part
  float* s_C = s_lo + l;                             // [kScanRows][N+1]
  float* s_h = s_C + kScanRows * ldn;                // [P][N+1]
  float* s_B = s_h + P * ldn;                        // [kScanCols][N+1]
  float* s_x = s_B + kScanCols * ldn;                // [kScanCols][P]
  float* s_M = s_x + kScanCols * P;                  // [kScanRows][kScanCols+1]
  float* s_ang = s_M + kScanRows * (kScanCols + 1);  // [l][N/2] when theta

  const int Lv = chunk_steps(p, b, c) * R;     // real rows of the chunk
  chunk_cumsum(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, Lv / R, s_cum, s_lo);
  if (p.theta) chunk_angles(p, b, c, h, s_ang);
  __syncthreads();

  stage_bc_rows(p, static_cast<const T*>(p.C), b, c, g, i0, kScanRows, s_ang, s_C, ldn);
  const float* hin = p.states + ((b * p.nch + c) * p.H + h) * p.P * p.N;
  for (int e = threadIdx.x; e < P * N; e += blockDim.x) s_h[(e / N) * ldn + e % N] = hin[e];
  __syncthreads();

  const int row = threadIdx.x / 4, pg = threadIdx.x % 4;
  const int i = i0 + row;
  float acc[PPT];
  {
    const float scale = (i < L) ? expf(s_cum[i / R] + s_lo[i / R]) : 0.f;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      const int pp = pg + 4 * k;
      float s = 0.f;
      if (pp < P) {
        for (int n = 0; n < N; ++n) s += s_C[row * ldn + n] * s_h[pp * ldn + n];
      }
      acc[k] = s * scale;
    }
  }

  const T* xs = static_cast<const T*>(p.x);
  const int64_t xbase = (((b * p.T + c * p.l) * p.R) * p.H + h) * p.P;
  const int i_last = min(i0 + kScanRows - 1, L - 1);
  const int j_end = min(L, (i_last / R) * R + R);   // exclusive bound of causal sources
  for (int j0 = 0; j0 < j_end; j0 += kScanCols) {
    __syncthreads();
    stage_bc_rows(p, static_cast<const T*>(p.B), b, c, g, j0, kScanCols, s_ang, s_B, ldn);
    for (int e = threadIdx.x; e < kScanCols * P; e += blockDim.x) {
      const int r = e / P, pp = e % P;
      s_x[e] = (j0 + r < Lv) ? ld_f32(xs + xbase + (int64_t)(j0 + r) * p.H * p.P + pp) : 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kScanRows * kScanCols; e += blockDim.x) {
      const int mr = e / kScanCols, mc = e % kScanCols;
      const int ii = i0 + mr, jj = j0 + mc;
      float m = 0.f;
      if (ii < L && jj < L && (jj / R) <= (ii / R)) {
        float d = 0.f;
        for (int n = 0; n < N; ++n) d += s_C[mr * ldn + n] * s_B[mc * ldn + n];
        m = seg_exp(s_cum, s_lo, ii / R, jj / R) * d;   // masked entries never reach expf
      }
      s_M[mr * (kScanCols + 1) + mc] = m;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      const int pp = pg + 4 * k;
      if (pp < P) {
        float s = 0.f;
        for (int jj = 0; jj < kScanCols; ++jj)
          s += s_M[row * (kScanCols + 1) + jj] * s_x[jj * P + pp];
        acc[k] += s;
      }
    }
  }

  if (i < Lv) {
    T* ys = static_cast<T*>(p.y);
    T* yrow = ys + xbase + (int64_t)i * p.H * p.P;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      const int pp = pg + 4 * k;
      if (pp < P && SSD_INDEX_OK(p.hdr, (yrow - ys) + pp, p.batch * p.T * p.R * p.H * p.P, 14))
        st_from_f32(yrow + pp, acc[k]);
    }
  }
}

template <typename T, int OPT>
cudaError_t launch_state(const GenericParams& p, size_t smem, cudaStream_t st) {
  auto k = chunk_state_kernel<T, OPT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<dim3((unsigned)p.nch, (unsigned)p.H, (unsigned)p.batch), kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

template <typename T, int PPT>
cudaError_t launch_scan(const GenericParams& p, size_t smem, cudaStream_t st) {
  auto k = chunk_scan_kernel<T, PPT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t L = p.l * p.R;
  const int64_t tiles = (L + kScanRows - 1) / kScanRows;
  k<<<dim3((unsigned)(p.nch * tiles), (unsigned)p.H, (unsigned)p.batch), kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_state_dispatch(const GenericParams& p, size_t smem, cudaStream_t st) {
  const int64_t opt = (p.P * p.N + kThreads - 1) / kThreads;
  if (opt <= 1) return launch_state<T, 1>(p, smem, st);
  if (opt <= 2) return launch_state<T, 2>(p, smem, st);
  if (opt <= 4) return launch_state<T, 4>(p, smem, st);
  if (opt <= 8) return launch_state<T, 8>(p, smem, st);
  if (opt <= 16) return launch_state<T, 16>(p, smem, st);
  if (opt <= 32) return launch_state<T, 32>(p, smem, st);
  return launch_state<T, 64>(p, smem, st);
}

template <typename T>
cudaError_t launch_scan_dispatch(const GenericParams& p, size_t smem, cudaStream_t st) {
  const int64_t ppt = (p.P + 3) / 4;
  if (ppt <= 1) return launch_scan<T, 1>(p, smem, st);
  if (ppt <= 2) return launch_scan<T, 2>(p, smem, st);
  if (ppt <= 4) return launch_scan<T, 4>(p, smem, st);
  if (ppt <= 8) return launch_scan<T, 8>(p, smem, st);
  if (ppt <= 16) return launch_scan<T, 16>(p, smem, st);
  return launch_scan<T, 32>(p, smem, st);
}

}  // namespace

size_t generic_state_smem(int64_t l, int64_t P, int64_t N, bool theta) {
  size_t f = 3 * l + kStateRows * P + kStateRows * N + (theta ? l * (N / 2) : 0);
  return f * sizeof(float);
}

size_t generic_scan_smem(int64_t l, int64_t P, int64_t N, bool theta) {
  size_t f = 2 * l + kScanRows * (N + 1) + P * (N + 1) + kScanCols * (N + 1) + kScanCols * P +
             kScanRows * (kScanCols + 1) + (theta ? l * (N / 2) : 0);
  return f * sizeof(float);
}

bool generic_supported(int64_t l, int64_t R, int64_t P, int64_t N, bool theta) {
  if (P > 128 || N > 256 || P * N > 64 * kThreads) return false;
  if (l * R > 4096) return false;
  const size_t lim = 227 * 1024;
  return generic_state_smem(l, P, N, theta) <= lim && generic_scan_smem(l, P, N, theta) <= lim;
}

cudaError_t generic_phi(const GenericParams& p, cudaStream_t st) {
  phi_chunk_sum_kernel<<<dim3((unsigned)((p.nch + kPhiChunksPerBlock - 1) / kPhiChunksPerBlock),
                              (unsigned)p.H, (unsigned)p.batch),
                         kPhiThreads, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = p.batch * p.H * (p.N / 2);
  phi_prefix_kernel<<<(unsigned)((warps * 32 + 127) / 128), 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t generic_state_pass(const GenericParams& p, cudaStream_t st) {
  const int64_t n = p.batch * p.H * p.P * p.N / (p.theta ? 2 : 1);
  const unsigned blocks = (unsigned)((n + kThreads - 1) / kThreads);
  if (p.theta) {
    state_pass_kernel<true><<<blocks, kThreads, 0, st>>>(p);
  } else {
    state_pass_kernel<false><<<blocks, kThreads, 0, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t generic_forward(const GenericParams& p, bool bf16, cudaStream_t st) {
  cudaError_t e;
  if (p.theta && (e = generic_phi(p, st)) != cudaSuccess) return e;
  const bool th = p.theta != nullptr;
  const size_t s1 = generic_state_smem(p.l, p.P, p.N, th);
  e = bf16 ? launch_state_dispatch<__nv_bfloat16>(p, s1, st) : launch_state_dispatch<float>(p, s1, st);
  if (e != cudaSuccess) return e;
  if ((e = generic_state_pass(p, st)) != cudaSuccess) return e;
  const size_t s2 = generic_scan_smem(p.l, p.P, p.N, th);
  return bf16 ? launch_scan_dispatch<__nv_bfloat16>(p, s2, st) : launch_scan_dispatch<float>(p, s2, st);
}

}  // namespace ssd
