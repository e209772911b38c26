// Per-chunk preparation shared by the fp32 chunk kernels with P = N = 64 (the register-tiled
// CUDA-core kernels and the tf32 tensor-core chunk scan): the rank shift of fused rows, the real
// steps of a chunk, the double-float prefix sums of dA (K1) and the rotation angles Phi_t of a
// chunk's steps.  chunk_prefix64 runs on warp 0; issue_theta64 on any block; chunk_angles64
// takes the block size as its template argument (kPrepThreads by default).
#pragma once

#include "common.cuh"
#include "fp_helpers.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace prep {

using namespace fp;

constexpr int kPrepThreads = 256;
constexpr int kPairs64 = 32;                              // N / 2 rotation pairs
constexpr float kLog2e64 = 1.4426950408889634f;
constexpr float kTwoPiHi64 = 6.28318548202514648f;        // float(2 pi)
constexpr float kTwoPiLo64 = -1.7484556000744487e-07f;    // 2 pi - kTwoPiHi64

// log2 of the rank (a power of two dividing 64): row i belongs to step i >> rank_shift.
__device__ __forceinline__ int rank_shift(const GenericParams& p) { return __ffs((int)p.R) - 1; }

// Real steps of chunk c of sequence b (short last chunk; padding past valid_len[b] excluded).
__device__ __forceinline__ int steps64(const GenericParams& p, int64_t b, int64_t c) {
  return (int)max((int64_t)0, min(p.l, seq_steps(p, b) - c * p.l));
}

// log2-scaled double-float prefix sums of dA over steps [0, n) of a chunk, by warp 0 (steps at
// or after nv read as zero): cum_hi/cum_lo[t] is the inclusive sum up to step t; *total
// (natural units) if non-null.  With kShared the steps are read from shared memory (a staged
// copy) instead of through the read-only global path.
template <bool kShared = false>
__device__ inline void chunk_prefix64(const float* __restrict__ src, int64_t stride, int n, int nv,
                               float* cum_hi, float* cum_lo, float* total) {
  auto ld = [&](int t) { return kShared ? src[(int64_t)t * stride] : __ldg(src + (int64_t)t * stride); };
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int per = (n + 31) / 32;
  const int beg = min(n, lane * per), end = min(n, beg + per);
  DF s = {0.f, 0.f};
  for (int t = beg; t < min(end, nv); ++t) s = df_add(s, DF{ld(t), 0.f});
  DF incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const DF v = df_shfl_up(incl, off);
    if (lane >= off) incl = df_add(incl, v);
  }
  const DF last = df_shfl(incl, 31);
  DF acc = df_shfl_up(incl, 1);
  if (lane == 0) acc = DF{0.f, 0.f};
  for (int t = beg; t < end; ++t) {
    if (t < nv) acc = df_add(acc, DF{ld(t), 0.f});
    const float chi = acc.hi * kLog2e64;
    cum_hi[t] = chi;
    cum_lo[t] = fmaf(acc.hi, kLog2e64, -chi) + acc.lo * kLog2e64;
  }
  if (lane == 0 && total) *total = last.hi + last.lo;
}

// Rotation angles Phi_t (inclusive cumulative theta from the chunk-start angle) for steps
// [0, n) and all 32 pairs, reduced to [-pi, pi], into ang[t * 32 + k].  theta is staged into
// `ang` (coalesced); thread (pair k, group gr) then sums its run of consecutive steps as a
// double-float, the group totals of each pair are prefix-summed through shared memory, and
// each thread rewrites its run in place.
// theta rows of steps [0, n) into ang[t * 32 + k] with 16-byte cp.async (not waited for);
// steps after the chunk's real ones are zero-filled (no global read).
__device__ inline void issue_theta64(const GenericParams& p, int64_t b, int64_t c, int64_t h, int n,
                              float* ang) {
  const float* th = p.theta + ((b * p.T + c * p.l) * p.H + h) * kPairs64;
  const int nv = steps64(p, b, c);
  for (int e = threadIdx.x; e < n * (kPairs64 / 4); e += blockDim.x) {
    const int t = e / (kPairs64 / 4), q = e % (kPairs64 / 4);
    const bool real = t < nv;
    cp_async16(ang + t * kPairs64 + 4 * q, th + (int64_t)(real ? t : 0) * p.H * kPairs64 + 4 * q,
               real ? 16 : 0);
  }
}

// With staged = true the theta rows were issued earlier by issue_theta64 (and are waited for
// here).  kThreads = blockDim.x (a multiple of 32).  phi0: the chunk's 32 start angles staged in
// shared memory, or null to read them from p.phi.
template <int kThreads = kPrepThreads>
__device__ inline void chunk_angles64(const GenericParams& p, int64_t b, int64_t c, int64_t h, int n,
                               float* ang, bool staged = false, const double* phi0 = nullptr) {
  __shared__ float part_hi[kThreads], part_lo[kThreads];
  if (!staged) issue_theta64(p, b, c, h, n, ang);
  cp_async_wait_all();
  __syncthreads();
  constexpr int kGroups = kThreads / kPairs64;            // step groups per pair
  const int k = threadIdx.x % kPairs64, gr = threadIdx.x / kPairs64;
  const int per = (n + kGroups - 1) / kGroups;
  const int beg = min(n, gr * per), end = min(n, beg + per);
  DF run = {0.f, 0.f};
  for (int t = beg; t < end; ++t) run = df_add(run, DF{ang[t * kPairs64 + k], 0.f});
  part_hi[threadIdx.x] = run.hi;
  part_lo[threadIdx.x] = run.lo;
  __syncthreads();
  const double a0 = phi0 ? phi0[k]   // in [-pi, pi]
                          : p.phi[((b * (p.nch + 1) + c) * p.H + h) * kPairs64 + k];
  const float s_hi = (float)a0;
  DF acc = {s_hi, (float)(a0 - (double)s_hi)};
  for (int g = 0; g < gr; ++g)
    acc = df_add(acc, DF{part_hi[g * kPairs64 + k], part_lo[g * kPairs64 + k]});
  for (int t = beg; t < end; ++t) {
    acc = df_add(acc, DF{ang[t * kPairs64 + k], 0.f});
    const float q = rintf(acc.hi * 0.15915494309189535f);
    ang[t * kPairs64 + k] = (fmaf(-q, kTwoPiHi64, acc.hi) - q * kTwoPiLo64) + acc.lo;
  }
  __syncthreads();
}

}  // namespace prep
}  // namespace ssd
