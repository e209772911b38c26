// Diagonal-A selective scan (SSM Selective Scan page: problem statement and the parallel-scan
// idea of its approach section), time-segmented so that many (batch, channel, segment) threads
// run at once:
//   ss_segment_kernel<false>: each segment's end state from a zero start, and its summed delta;
//   ss_carry_kernel         : segment-input states, h_in(s+1) = exp(A * sum delta_s) h_in(s) + end_s
//                             (the per-step decays of a segment multiply to exp(A * sum delta));
//   ss_segment_kernel<true> : the recurrence again from the true segment-input state, writing
//                             y = C . h + skip * u.
// Channels d are independent and share B and C, so one thread owns one (b, d, segment) with all
// d_state states in registers; loads of u/delta/y are coalesced over d.
#include <math.h>

#include <algorithm>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "fp_helpers.cuh"
#include "ssd_internal.h"

namespace ssd {

namespace {

constexpr int kSsThreads = 128;
constexpr int64_t kSegLen = 64;


template <int NB, bool kOutput>
__global__ void __launch_bounds__(kSsThreads) ss_segment_kernel(SelectiveScanParams p) {
  const int64_t seg = blockIdx.x, b = blockIdx.z;
  const int64_t d = (int64_t)blockIdx.y * blockDim.x + threadIdx.x;
  if (d >= p.D) return;
  const int N = (int)p.N;
  float a[NB], h[NB];
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    a[n] = (n < N) ? __ldg(p.A + d * p.N + n) : 0.f;
    h[n] = 0.f;
    if (kOutput && n < N) h[n] = p.agg_h[((b * p.nseg + seg) * p.N + n) * p.D + d];
  }
  const float sk = (kOutput && p.skip) ? __ldg(p.skip + d) : 0.f;
  const int64_t t0 = seg * p.seg_len;
  const int64_t t1 = min(p.T, t0 + p.seg_len);
  float sdt = 0.f;
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t row = b * p.T + t;
    const float dt = __ldg(p.delta + row * p.D + d);
    const float uu = __ldg(p.u + row * p.D + d);
    const float du = dt * uu;
    const float* Bt = p.B + row * p.N;
    sdt += dt;
    if (kOutput) {
      const float* Ct = p.C + row * p.N;
      float acc = 0.f;
#pragma unroll
      for (int n = 0; n < NB; ++n) {
        if (n < N) {
          h[n] = expf(dt * a[n]) * h[n] + du * __ldg(Bt + n);
          acc += __ldg(Ct + n) * h[n];
        }
      }
      if (SSD_INDEX_OK(p.hdr, row * p.D + d, p.batch * p.T * p.D, 30)) p.y[row * p.D + d] = acc + sk * uu;
    } else {
#pragma unroll
      for (int n = 0; n < NB; ++n) {
        if (n < N) h[n] = expf(dt * a[n]) * h[n] + du * __ldg(Bt + n);
      }
    }
  }
  if (!kOutput) {
#pragma unroll
    for (int n = 0; n < NB; ++n)
      if (n < N && SSD_INDEX_OK(p.hdr, ((b * p.nseg + seg) * p.N + n) * p.D + d,
                                p.batch * p.nseg * p.N * p.D, 31))
        p.agg_h[((b * p.nseg + seg) * p.N + n) * p.D + d] = h[n];
    if (SSD_INDEX_OK(p.hdr, (b * p.nseg + seg) * p.D + d, p.batch * p.nseg * p.D, 32))
      p.agg_dt[(b * p.nseg + seg) * p.D + d] = sdt;
  }
}

template <int NB>
__global__ void __launch_bounds__(kSsThreads) ss_carry_kernel(SelectiveScanParams p) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.batch * p.D) return;
  const int64_t b = idx / p.D, d = idx % p.D;
  const int N = (int)p.N;
  float a[NB], h[NB];
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    a[n] = (n < N) ? __ldg(p.A + d * p.N + n) : 0.f;
    h[n] = 0.f;
  }
  for (int64_t s = 0; s < p.nseg; ++s) {
    const float sdt = p.agg_dt[(b * p.nseg + s) * p.D + d];
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      if (n < N) {
        float* q = p.agg_h + ((b * p.nseg + s) * p.N + n) * p.D + d;
        const float end = *q;
        if (SSD_INDEX_OK(p.hdr, q - p.agg_h, p.batch * p.nseg * p.N * p.D, 33)) *q = h[n];
        h[n] = expf(a[n] * sdt) * h[n] + end;
      }
    }
  }
}

template <int NB>
cudaError_t launch_nb(const SelectiveScanParams& p, cudaStream_t st) {
  const dim3 grid((unsigned)p.nseg, (unsigned)((p.D + kSsThreads - 1) / kSsThreads),
                  (unsigned)p.batch);
  ss_segment_kernel<NB, false><<<grid, kSsThreads, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ss_carry_kernel<NB><<<(unsigned)((p.batch * p.D + kSsThreads - 1) / kSsThreads), kSsThreads, 0,
                        st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ss_segment_kernel<NB, true><<<grid, kSsThreads, 0, st>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// One-pass selective scan for d_state N = SPL * LPC in {8, 16, 32, 64} and d_model % 4 == 0
// (SPL = 4 states per lane, 8 for N = 16, where fewer lanes per channel means fewer shared-
// memory reads per channel-step: the output pass is bound by them).
// A warp owns 32 / LPC channels d of one batch row; the LPC lanes of a channel each carry SPL
// of its N states, so every exp(delta * A) is evaluated on the special-function unit (2^x with
// A pre-scaled by log2 e) and only segment boundary states go to memory.  T is cut into
// segments (at least kSsMinSeg steps) so that enough warps exist: a state-only pass gives each
// segment's end state from zero, a carry pass chains them, and the output pass runs each
// segment from its true input state.  Every LPC steps the lanes of a channel sum their C . h
// partials with a transpose-reduce (log2 LPC shuffle levels), after which lane l holds y of
// step t0 + l.  The block's delta, u, B and C rows are staged through shared memory in a ring
// of kSsStages stages of SsLayout::kSteps steps (16-byte cp.async, zero-filled past the segment
// and D).
// ------------------------------------------------------------------------------------------------
constexpr int kSsWarps = 4;
// Steps per stage and stages in flight: short stages, four deep (measured on the 4 x 4096 x 512
// x 16 workload: 8 x 4 beat 16 x 2 and 16 x 3 by about 15 %); a stage holds at least one step
// per lane of a channel.
constexpr int kSsStepsMin = 8;
constexpr int kSsStages = 4;
// Time segments: enough to give every SM this many blocks' worth of resident work (the scan is
// latency bound, so more blocks than fit at once still help), each at least kSsMinSeg steps.
constexpr int kSsWaveMult = 2;
constexpr int64_t kSsMinSeg = 128;
// the workspace holds ceil(T / kSegLen) segment states: segments may not be shorter
static_assert(kSsMinSeg >= kSegLen, "segments shorter than the workspace's segment length");


template <int SPL, int LPC>
struct SsLayout {
  static constexpr int kN = SPL * LPC;                   // d_state
  static constexpr int kCpw = 32 / LPC;                  // channels per warp
  static constexpr int kCpb = kCpw * kSsWarps;           // channels per block
  static constexpr int kSteps = LPC > kSsStepsMin ? LPC : kSsStepsMin;   // steps per stage
  static constexpr int kDtFloats = kSteps * kCpb;
  static constexpr int kBFloats = kSteps * kN;
  static constexpr int kStageFloats = 2 * kDtFloats + 2 * kBFloats;
  static constexpr size_t kSmemBytes = sizeof(float) * kStageFloats * kSsStages;
};

// SPL consecutive floats (8 or 16 bytes) from shared memory.
template <int SPL>
__device__ __forceinline__ void ld_states(const float* src, float (&v)[SPL]) {
  if constexpr (SPL % 4 == 0) {
#pragma unroll
    for (int q = 0; q < SPL / 4; ++q) {
      const float4 f = *reinterpret_cast<const float4*>(src + 4 * q);
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
  } else {
    const float2 f = *reinterpret_cast<const float2*>(src);
    v[0] = f.x; v[1] = f.y;
  }
}

// One step of SPL states: h <- exp(A dt) h + (dt u) B, exponentials as 2^(A log2e dt).
template <int SPL>
__device__ __forceinline__ void ss_step(const float (&a)[SPL], float dt, float du,
                                        const float (&bb)[SPL], float (&h)[SPL]) {
#pragma unroll
  for (int j = 0; j < SPL; j += 2) {
    const float2 x = fp::mul2(make_float2(a[j], a[j + 1]), make_float2(dt, dt));
    const float2 e = make_float2(fp::ex2_approx(x.x), fp::ex2_approx(x.y));
    const float2 r =
        fp::fma2(e, make_float2(h[j], h[j + 1]), fp::mul2(make_float2(du, du), make_float2(bb[j], bb[j + 1])));
    h[j] = r.x;
    h[j + 1] = r.y;
  }
}

// kOut = false: the segment's end state from a zero start and its summed delta (segments
// 0 .. nseg-2; no C, no output).  kOut = true: the segment from its true input state (left in
// agg_h by the carry pass) with y.  Lane l of a channel carries states SPL*l .. SPL*l+SPL-1.
// Lane mapping of a block: a warp owns kCpw channels, lane l of a channel its states
// SPL*l .. SPL*l+SPL-1.
template <int SPL, int LPC>
struct SsLane {
  using Lay = SsLayout<SPL, LPC>;
  int cl, l;       // channel within the block, lane within the channel
  int64_t d, dd;   // channel (dd clamped to a valid one)
  bool dv;         // d < D
  __device__ SsLane(const SelectiveScanParams& p, int64_t d0) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    cl = warp * Lay::kCpw + lane / LPC;
    l = lane % LPC;
    d = d0 + cl;
    dv = d < p.D;
    dd = dv ? d : 0;
  }
};

// Steps [t_beg, t_end) of batch row b for the block's channels d0 .. d0 + kCpb - 1, from the
// state h (in registers; h is the end state afterwards).  kOut = false: state only, with the
// summed delta of the lane's channel in sdt_sum.  kOut = true: y of every step too.
template <int SPL, int LPC, bool kOut>
__device__ __forceinline__ void ss_segment(const SelectiveScanParams& p, int64_t b, int64_t d0,
                                           const SsLane<SPL, LPC>& ln, int64_t t_beg,
                                           int64_t t_end, const float (&a)[SPL], float sk,
                                           float (&h)[SPL], float& sdt_sum) {
  using Lay = SsLayout<SPL, LPC>;
  constexpr int kN = Lay::kN, kCpb = Lay::kCpb;
  extern __shared__ __align__(16) float ss_sm[];
  const int64_t T = p.T, D = p.D;
  const int cl = ln.cl, l = ln.l;
  constexpr int kSsSteps = Lay::kSteps;
  const int64_t nst = (t_end - t_beg + kSsSteps - 1) / kSsSteps;

  auto issue = [&](int64_t st) {
    float* sm = ss_sm + (st % kSsStages) * Lay::kStageFloats;
    const int64_t t0 = t_beg + st * kSsSteps;
    constexpr int kDtChunks = kSsSteps * kCpb / 4, kBChunks = kSsSteps * kN / 4;
    for (int c = threadIdx.x; c < kDtChunks; c += 32 * kSsWarps) {
      const int k = c / (kCpb / 4), q = c % (kCpb / 4);
      const int64_t t = t0 + k, dc = d0 + 4 * q;
      const bool ok = t < t_end && dc < D;
      const int64_t off = ok ? (b * T + t) * D + dc : 0;
      cp_async16(sm + k * kCpb + 4 * q, p.delta + off, ok ? 16 : 0);
      cp_async16(sm + Lay::kDtFloats + k * kCpb + 4 * q, p.u + off, ok ? 16 : 0);
    }
    for (int c = threadIdx.x; c < kBChunks; c += 32 * kSsWarps) {
      const int k = c / (kN / 4), q = c % (kN / 4);
      const int64_t t = t0 + k;
      const bool ok = t < t_end;
      const int64_t off = ok ? (b * T + t) * kN + 4 * q : 0;
      cp_async16(sm + 2 * Lay::kDtFloats + k * kN + 4 * q, p.B + off, ok ? 16 : 0);
      if (kOut)
        cp_async16(sm + 2 * Lay::kDtFloats + Lay::kBFloats + k * kN + 4 * q, p.C + off,
                   ok ? 16 : 0);
    }
  };

#pragma unroll 1
  for (int s = 0; s < kSsStages - 1; ++s) {
    if (s < nst) issue(s);
    cp_async_commit();
  }
  float* yp = p.y + b * T * D + ln.dd;
#pragma unroll 1
  for (int64_t st = 0; st < nst; ++st) {
    if (st + kSsStages - 1 < nst) issue(st + kSsStages - 1);
    cp_async_commit();
    cp_async_wait<kSsStages - 1>();
    __syncthreads();
    const float* sm = ss_sm + (st % kSsStages) * Lay::kStageFloats;
    const float* sdt = sm + cl;
    const float* su = sm + Lay::kDtFloats + cl;
    const float* sB = sm + 2 * Lay::kDtFloats + SPL * l;
    const float* sC = sm + 2 * Lay::kDtFloats + Lay::kBFloats + SPL * l;
    const int64_t t0 = t_beg + st * kSsSteps;
    if constexpr (!kOut) {
#pragma unroll
      for (int kk = 0; kk < kSsSteps; ++kk) {
        const float dt = sdt[kk * kCpb], uu = su[kk * kCpb];
        float bb[SPL];
        ld_states<SPL>(sB + kk * kN, bb);
        ss_step<SPL>(a, dt, dt * uu, bb, h);   // zero-filled steps past the segment keep h
        sdt_sum += dt;
      }
    } else {
      // unrolled over the whole stage so one group's reduction overlaps the next group's steps
#pragma unroll
      for (int k0 = 0; k0 < kSsSteps; k0 += LPC) {
        float v[LPC];
#pragma unroll
        for (int k = 0; k < LPC; ++k) {
          const int kk = k0 + k;
          const float dt = sdt[kk * kCpb], uu = su[kk * kCpb];
          float bb[SPL], cc[SPL];
          ld_states<SPL>(sB + kk * kN, bb);
          ld_states<SPL>(sC + kk * kN, cc);
          ss_step<SPL>(a, dt, dt * uu, bb, h);
          // C . h over the lane's states as paired products, the two halves added at the end
          float2 acc = fp::mul2(make_float2(cc[0], cc[1]), make_float2(h[0], h[1]));
#pragma unroll
          for (int j = 2; j < SPL; j += 2)
            acc = fp::fma2(make_float2(cc[j], cc[j + 1]), make_float2(h[j], h[j + 1]), acc);
          v[k] = acc.x + acc.y;
        }
        // transpose-reduce over the LPC lanes of the channel: at the level with lane bit m
        // the lanes with that bit keep the upper half of their values, the others the lower
        // half, and each adds its partner's copy of the half it keeps
#pragma unroll
        for (int m = LPC / 2, cnt = LPC; m >= 1; m >>= 1, cnt >>= 1) {
          const bool up_half = (l & m) != 0;
#pragma unroll
          for (int i = 0; i < cnt / 2; ++i) {
            const float send = up_half ? v[i] : v[i + cnt / 2];
            const float keep = up_half ? v[i + cnt / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
        const int64_t t = t0 + k0 + l;
        if (ln.dv && t < t_end && SSD_INDEX_OK(p.hdr, (yp - p.y) + t * D, p.batch * T * D, 34))
          yp[t * D] = fmaf(sk, su[(k0 + l) * kCpb], v[0]);   // + skip * u
      }
    }
    __syncthreads();   // the stage's buffer is refilled by a later issue
  }
}

// The lane's A row (pre-scaled by log2 e) and skip weight.
template <int SPL, int LPC>
__device__ __forceinline__ void ss_lane_params(const SelectiveScanParams& p,
                                               const SsLane<SPL, LPC>& ln, float (&a)[SPL],
                                               float& sk) {
  constexpr int kN = SsLayout<SPL, LPC>::kN;
  const float kLog2e = 1.4426950408889634f;
#pragma unroll
  for (int j = 0; j < SPL; ++j) a[j] = ln.dv ? p.A[ln.dd * kN + SPL * ln.l + j] * kLog2e : 0.f;
  sk = (ln.dv && p.skip) ? p.skip[ln.dd] : 0.f;
}

template <int SPL, int LPC, bool kOut>
__global__ void __launch_bounds__(32 * kSsWarps) ss_onepass_kernel(SelectiveScanParams p) {
  using Lay = SsLayout<SPL, LPC>;
  constexpr int kN = Lay::kN, kCpb = Lay::kCpb;
  const int64_t groups = (p.D + kCpb - 1) / kCpb;
  const int64_t nrun = kOut ? p.nseg : p.nseg - 1;      // segments this pass covers
  const int64_t seg = blockIdx.x % nrun;
  const int64_t bgrp = blockIdx.x / nrun;
  const int64_t b = bgrp / groups;
  const int64_t d0 = (bgrp % groups) * kCpb;
  const SsLane<SPL, LPC> ln(p, d0);
  const int64_t D = p.D;
  float a[SPL], h[SPL], sk;
  ss_lane_params(p, ln, a, sk);
#pragma unroll
  for (int j = 0; j < SPL; ++j) h[j] = 0.f;
  const int64_t t_beg = seg * p.seg_len, t_end = min(p.T, t_beg + p.seg_len);
  float* agg = p.agg_h + ((b * p.nseg + seg) * kN + SPL * ln.l) * D + ln.dd;   // [b, seg, n, d]
  float sdt_sum = 0.f;
  if (kOut && seg > 0 && ln.dv) {   // segment-input state from the carry pass
#pragma unroll
    for (int j = 0; j < SPL; ++j) h[j] = agg[j * D];
  }
  ss_segment<SPL, LPC, kOut>(p, b, d0, ln, t_beg, t_end, a, sk, h, sdt_sum);
  if (!kOut && ln.dv) {
#pragma unroll
    for (int j = 0; j < SPL; ++j)
      if (SSD_INDEX_OK(p.hdr, (agg - p.agg_h) + j * D, p.batch * p.nseg * kN * D, 35))
        agg[j * D] = h[j];
    if (ln.l == 0 &&
        SSD_INDEX_OK(p.hdr, (b * p.nseg + seg) * D + ln.dd, p.batch * p.nseg * D, 36))
      p.agg_dt[(b * p.nseg + seg) * D + ln.dd] = sdt_sum;
  }
}

// ------------------------------------------------------------------------------------------------
// The same scan in one cooperative launch with a decoupled look-back over time segments: every
// block but the last segment's runs its segment state-only from zero and publishes that end
// state (segment 0: the inclusive state itself), then finds its input state by walking back
// over the published states of earlier segments until it meets an inclusive one
// (h_in(s) = E_{s-1} + D_{s-1} (E_{s-2} + D_{s-2} ( ... I_j))), publishes its own inclusive
// state I_s = D_s h_in(s) + E_s, and runs its segment again with the output.  All blocks are
// resident at once (cooperative launch), and a block only waits for blocks of earlier segments,
// which publish their end states without waiting for anything: every wait ends.  Each wait is
// still bounded (1 s); one that gives up latches SSD_ERR_TIMEOUT and the block goes on from
// what it has.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// The state (1 = end state from zero, 2 = inclusive) a segment published in this call, or 0 if
// nothing was published within the bound.
__device__ int ss_wait_flag(const uint64_t* f, uint64_t epoch) {
  const uint64_t t0 = global_ns();
  for (;;) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    if ((v >> 2) == epoch) return (int)(v & 3u);
    if (global_ns() - t0 > 1000000000ull) return 0;
    __nanosleep(100);
  }
}

__device__ __forceinline__ void ss_publish(uint64_t* f, uint64_t epoch, int state) {
  const uint64_t v = epoch * 4 + (uint64_t)state;
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

template <int SPL, int LPC>
__global__ void __launch_bounds__(32 * kSsWarps) ss_lookback_kernel(SelectiveScanParams p) {
  using Lay = SsLayout<SPL, LPC>;
  constexpr int kN = Lay::kN, kCpb = Lay::kCpb;
  __shared__ int s_state;
  const int64_t groups = (p.D + kCpb - 1) / kCpb;
  const int64_t seg = blockIdx.x % p.nseg;
  const int64_t bgrp = blockIdx.x / p.nseg;
  const int64_t b = bgrp / groups;
  const int64_t d0 = (bgrp % groups) * kCpb;
  const SsLane<SPL, LPC> ln(p, d0);
  const int64_t D = p.D;
  float a[SPL], h[SPL], sk;
  ss_lane_params(p, ln, a, sk);
  const int64_t t_beg = seg * p.seg_len, t_end = min(p.T, t_beg + p.seg_len);
  const bool last = seg == p.nseg - 1;
  // this lane's states of segment s in a [b, nseg, N, D] array
  auto at = [&](float* base, int64_t s) {
    return base + ((b * p.nseg + s) * kN + SPL * ln.l) * D + ln.dd;
  };
  uint64_t* flag = p.flags + bgrp * p.nseg;
  float e_s[SPL], sdt = 0.f;
  if (!last) {
#pragma unroll
    for (int j = 0; j < SPL; ++j) h[j] = 0.f;
    ss_segment<SPL, LPC, false>(p, b, d0, ln, t_beg, t_end, a, sk, h, sdt);
    float* dst = at(seg == 0 ? p.inc_h : p.agg_h, seg);
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
      e_s[j] = h[j];
      if (ln.dv && SSD_INDEX_OK(p.hdr, (dst - p.agg_h) + j * D, 2 * p.batch * p.nseg * kN * D, 38))
        dst[j * D] = h[j];
    }
    if (seg > 0 && ln.dv && ln.l == 0 &&
        SSD_INDEX_OK(p.hdr, (b * p.nseg + seg) * D + ln.dd, p.batch * p.nseg * D, 39))
      p.agg_dt[(b * p.nseg + seg) * D + ln.dd] = sdt;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) ss_publish(flag + seg, p.epoch, seg == 0 ? 2 : 1);
  }
  // input state of the segment
  float hin[SPL];
#pragma unroll
  for (int j = 0; j < SPL; ++j) hin[j] = 0.f;
  if (seg > 0) {
    float acc[SPL], dec[SPL];
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
      acc[j] = 0.f;
      dec[j] = 1.f;
    }
    for (int64_t s = seg - 1; s >= 0; --s) {
      if (threadIdx.x == 0) s_state = ss_wait_flag(flag + s, p.epoch);
      __syncthreads();
      const int state = s_state;
      __syncthreads();
      if (state == 0) {   // gave up: latch and go on from the partial sum
        if (threadIdx.x == 0 && p.hdr) latch_error(p.hdr, SSD_ERR_TIMEOUT, 300 + (int)(s & 63));
#pragma unroll
        for (int j = 0; j < SPL; ++j) hin[j] = acc[j];
        break;
      }
      const float* src = at(state == 2 ? p.inc_h : p.agg_h, s);
#pragma unroll
      for (int j = 0; j < SPL; ++j) acc[j] = fmaf(dec[j], ln.dv ? __ldcg(src + j * D) : 0.f, acc[j]);
      if (state == 2) {
#pragma unroll
        for (int j = 0; j < SPL; ++j) hin[j] = acc[j];
        break;
      }
      const float sd = ln.dv ? __ldcg(p.agg_dt + (b * p.nseg + s) * D + ln.dd) : 0.f;
#pragma unroll
      for (int j = 0; j < SPL; ++j) dec[j] *= fp::ex2_approx(a[j] * sd);
    }
    if (!last) {   // the inclusive state of this segment for later ones
      float* dst = at(p.inc_h, seg);
#pragma unroll
      for (int j = 0; j < SPL; ++j)
        if (ln.dv && SSD_INDEX_OK(p.hdr, (dst - p.agg_h) + j * D, 2 * p.batch * p.nseg * kN * D, 38))
          dst[j * D] = fmaf(fp::ex2_approx(a[j] * sdt), hin[j], e_s[j]);
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) ss_publish(flag + seg, p.epoch, 2);
    }
  }
#pragma unroll
  for (int j = 0; j < SPL; ++j) h[j] = hin[j];
  float unused = 0.f;
  ss_segment<SPL, LPC, true>(p, b, d0, ln, t_beg, t_end, a, sk, h, unused);
}

// Segment-input states for the one-pass path, one thread per (b, state n, d): h_in(0) = 0,
// h_in(s+1) = exp(A[d,n] * sum delta_s) h_in(s) + end_s, written over end_s in place.
__global__ void __launch_bounds__(kSsThreads) ss_carry_states_kernel(SelectiveScanParams p) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.batch * p.N * p.D) return;
  const int64_t d = idx % p.D, n = (idx / p.D) % p.N, b = idx / (p.D * p.N);
  const float a = p.A[d * p.N + n];
  const int64_t sstride = p.N * p.D;            // from segment s to s + 1 in agg_h
  float* q = p.agg_h + ((b * p.nseg) * p.N + n) * p.D + d;
  const float* sd = p.agg_dt + (b * p.nseg) * p.D + d;
  float h = 0.f;
  // 32 segments per round: every load of the round is issued before the first is used and the
  // decays are formed off the chain, so the serial part is one FMA per segment
  constexpr int kRound = 32;
  for (int64_t s0 = 0; s0 + 1 < p.nseg; s0 += kRound) {
    float ev[kRound], dv[kRound];
#pragma unroll
    for (int k = 0; k < kRound; ++k) {
      const bool in = s0 + k + 1 < p.nseg;
      ev[k] = in ? q[(s0 + k) * sstride] : 0.f;
      dv[k] = in ? sd[(s0 + k) * p.D] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kRound; ++k) dv[k] = expf(a * dv[k]);
#pragma unroll
    for (int k = 0; k < kRound; ++k) {
      if (s0 + k + 1 < p.nseg) {
        if (SSD_INDEX_OK(p.hdr, (q - p.agg_h) + (s0 + k) * sstride, p.batch * p.nseg * p.N * p.D, 37))
          q[(s0 + k) * sstride] = h;
        h = dv[k] * h + ev[k];
      }
    }
  }
  if (SSD_INDEX_OK(p.hdr, (q - p.agg_h) + (p.nseg - 1) * sstride, p.batch * p.nseg * p.N * p.D, 37))
    q[(p.nseg - 1) * sstride] = h;
}

// Calls of the look-back form draw distinct epochs, so flags left in a workspace by an earlier
// call never pass for this call's.
std::atomic<uint64_t> g_ss_epoch{0};

// One cooperative launch over as many segments as fit resident at once with the whole grid
// (at least kSsMinSeg steps each); the look-back arrays live in the workspace's segment arrays,
// which are sized for ceil(T / kSegLen) segments (p.nseg): inclusive states after the end
// states, flags after the summed deltas.  Returns cudaErrorNotSupported (nothing launched) when
// the form does not apply, and the caller runs the three-launch form.
template <int SPL, int LPC>
cudaError_t launch_lookback(const SelectiveScanParams& p, cudaStream_t st) {
  using Lay = SsLayout<SPL, LPC>;
  auto kern = ss_lookback_kernel<SPL, LPC>;
  int dev = 0, sms = 0, coop = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return e;
  if (!coop) return cudaErrorNotSupported;
  if (Lay::kSmemBytes > 48 * 1024 &&
      (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Lay::kSmemBytes)) != cudaSuccess)
    return e;
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * kSsWarps,
                                                          Lay::kSmemBytes)) != cudaSuccess)
    return e;
  const int64_t bgroups = (p.D + Lay::kCpb - 1) / Lay::kCpb;   // channel blocks per batch row
  const int64_t groups = p.batch * bgroups;
  int64_t nseg = (int64_t)sms * per_sm / groups;
  nseg = std::min<int64_t>(nseg, p.T / kSsMinSeg);
  if (nseg < 2) return cudaErrorNotSupported;
  int64_t seg_len = (p.T + nseg - 1) / nseg;
  seg_len = (seg_len + Lay::kSteps - 1) / Lay::kSteps * Lay::kSteps;
  nseg = (p.T + seg_len - 1) / seg_len;
  // room in the workspace (p.nseg segments of end states and summed deltas)
  const int64_t flags_floats = 2 * groups * nseg + 2;
  if (2 * nseg > p.nseg || p.batch * nseg * p.D + flags_floats > p.batch * p.nseg * p.D)
    return cudaErrorNotSupported;
  SelectiveScanParams q = p;
  q.seg_len = seg_len;
  q.nseg = nseg;
  q.inc_h = p.agg_h + p.batch * nseg * p.N * p.D;
  const int64_t fo = (p.batch * nseg * p.D + 1) / 2 * 2;   // 8-byte aligned
  q.flags = reinterpret_cast<uint64_t*>(p.agg_dt + fo);
  q.epoch = g_ss_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  void* args[] = {&q};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern),
                                     dim3((unsigned)(groups * nseg)), dim3(32 * kSsWarps), args,
                                     Lay::kSmemBytes, st);
}

template <int SPL, int LPC>
cudaError_t launch_onepass(const SelectiveScanParams& p, cudaStream_t st) {
#ifndef SS_THREE_PASS
  {
    const cudaError_t e = launch_lookback<SPL, LPC>(p, st);
    if (e != cudaErrorNotSupported) return e;
  }
#endif
  using Lay = SsLayout<SPL, LPC>;
  const int64_t groups = p.batch * ((p.D + Lay::kCpb - 1) / Lay::kCpb);
  // Segments of T (each at least 256 steps, a multiple of the staging step) until the output
  // pass fills one wave of resident blocks: one warp per scheduler cannot hide the latency of
  // its serial recurrence, and a second partial wave would idle most SMs.  The extra cost is
  // one more exponential per step of every segment but the last (the state-only pass).
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (Lay::kSmemBytes > 48 * 1024) {
    if ((e = cudaFuncSetAttribute(ss_onepass_kernel<SPL, LPC, false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)Lay::kSmemBytes)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(ss_onepass_kernel<SPL, LPC, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)Lay::kSmemBytes)) != cudaSuccess)
      return e;
  }
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ss_onepass_kernel<SPL, LPC, true>,
                                                          32 * kSsWarps, Lay::kSmemBytes)) !=
      cudaSuccess)
    return e;
  int64_t nseg = std::max<int64_t>(1, (int64_t)sms * std::max(per_sm, 1) * kSsWaveMult / groups);
  nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, p.T / kSsMinSeg));
  int64_t seg_len = (p.T + nseg - 1) / nseg;
  seg_len = (seg_len + Lay::kSteps - 1) / Lay::kSteps * Lay::kSteps;
  SelectiveScanParams q = p;
  q.seg_len = seg_len;
  q.nseg = (p.T + seg_len - 1) / seg_len;   // <= ceil(T / 64): fits the workspace's segment arrays
  if (q.nseg > 1) {
    ss_onepass_kernel<SPL, LPC, false>
        <<<(unsigned)(groups * (q.nseg - 1)), 32 * kSsWarps, Lay::kSmemBytes, st>>>(q);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ss_carry_states_kernel<<<(unsigned)((q.batch * q.N * q.D + kSsThreads - 1) / kSsThreads),
                             kSsThreads, 0, st>>>(q);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  ss_onepass_kernel<SPL, LPC, true>
      <<<(unsigned)(groups * q.nseg), 32 * kSsWarps, Lay::kSmemBytes, st>>>(q);
  return cudaGetLastError();
}

}  // namespace

int64_t ss_segment_length(int64_t) { return kSegLen; }

bool selective_scan_onepass_supported(int64_t batch, int64_t D, int64_t N) {
  if (N != 8 && N != 16 && N != 32 && N != 64) return false;
  if (D % 4 != 0) return false;                      // 16-byte staging of delta / u rows
  const int64_t cpb = 128 / N * kSsWarps;   // channels per block at 4 states per lane (a lower
                                            // bound: more blocks than any SPL launches)
  const int64_t blocks = batch * ((D + cpb - 1) / cpb);
  return blocks <= 0x7fffffffLL;
}

cudaError_t selective_scan_onepass_launch(const SelectiveScanParams& p, cudaStream_t st) {
  switch (p.N) {
    case 8: return launch_onepass<4, 2>(p, st);
    case 16: return launch_onepass<8, 2>(p, st);
    case 32: return launch_onepass<4, 8>(p, st);
    case 64: return launch_onepass<4, 16>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t selective_scan_launch(const SelectiveScanParams& p, cudaStream_t st) {
  if (p.N <= 16) return launch_nb<16>(p, st);
  if (p.N <= 32) return launch_nb<32>(p, st);
  return launch_nb<64>(p, st);
}

}  // namespace ssd

// ------------------------------------------------------------------------------------------------
// Allocation-free selective scan: the same three kernels, with their scratch (segment end states
// and summed deltas) in a fixed device array owned by this library instead of a caller
// workspace.  It exists for callers that cannot allocate device memory -- for example code
// that is handed only its input and output buffers through a fixed plugin interface, or code on
// a path where cudaMalloc (and the device synchronisation it can imply) is not allowed.
// ------------------------------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchFloats = SSD_NOALLOC_SCRATCH_BYTES / sizeof(float);

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once per device (the
// array's name in host code is only a host-side stand-in, never a device address).
cudaError_t noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" ssd_status selective_scan_forward_noalloc(const float* u, const float* delta,
                                                     const float* A, const float* B,
                                                     const float* C, const float* skip, float* y,
                                                     int64_t batch, int64_t seqlen,
                                                     int64_t d_model, int64_t d_state,
                                                     void* stream) {
  if (batch < 1 || seqlen < 1 || d_model < 1 || d_state < 1) return SSD_ERR_INVALID_ARG;
  if (d_state > 64 || batch > 65535 || d_model > ((int64_t)65535 * 128)) return SSD_ERR_UNSUPPORTED;
  if (!u || !delta || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
  const void* ptrs[] = {u, delta, A, B, C, skip, y};
  for (const void* q : ptrs)
    if (q && !ssd::aligned16(q)) return SSD_ERR_INVALID_ARG;
  const int64_t seg = ssd::ss_segment_length(seqlen);
  const int64_t nseg = (seqlen + seg - 1) / seg;
  // scratch: segment end states [b, nseg, N, D] then summed deltas [b, nseg, D]
  if (batch > (int64_t)kNoAllocScratchFloats || nseg > (int64_t)kNoAllocScratchFloats ||
      d_model > (int64_t)kNoAllocScratchFloats)
    return SSD_ERR_UNSUPPORTED;
  const int64_t rows = batch * nseg * d_model;
  if (rows > (int64_t)kNoAllocScratchFloats / (d_state + 1)) return SSD_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return SSD_ERR_CUDA;
  ssd::SelectiveScanParams p{};
  p.u = u;
  p.delta = delta;
  p.A = A;
  p.B = B;
  p.C = C;
  p.skip = skip;
  p.y = y;
  p.batch = batch;
  p.T = seqlen;
  p.D = d_model;
  p.N = d_state;
  p.seg_len = seg;
  p.nseg = nseg;
  p.agg_h = scratch;
  p.agg_dt = scratch + rows * d_state;
  p.hdr = nullptr;
  const cudaError_t e = ssd::selective_scan_launch(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
