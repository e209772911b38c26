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

#include <mutex>

#include "common.cuh"
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
      p.y[row * p.D + d] = acc + sk * uu;
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
      if (n < N) p.agg_h[((b * p.nseg + seg) * p.N + n) * p.D + d] = h[n];
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
        *q = h[n];
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

}  // namespace

int64_t ss_segment_length(int64_t) { return kSegLen; }

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
