// Trapezoidal Mamba-3 forward as one scalar-decay scan with 2R write channels.
//
// The trapezoid (scan.py page, the trapezoidal forward) adds to each step's write gamma_t S_t the
// previous step's write beta_t S_{t-1}, turned by one step less of rotation.  The moments.rs
// page realises it as a single scalar-decay system whose write channel axis is doubled
// ("combined injections"): x^ = [gamma_t x_t, beta_t x_{t-1}] and b^ = [B_t, B_{t-1}], the second
// half shifted one step (its first element from the previous call).  In the physical frame the
// shifted write must be turned by this step's theta, so that after the chunk kernels absorb
// R(-Phi_t) into every channel of step t it carries R(-Phi_{t-1}), one step less:
//     b^[t, R + r] = R(theta_t) B[t-1, r].
// The R output channels read the state after all 2R writes of the step, which is the MIMO rule
// of the chunk kernels once C is given zeros on the extra channels.
//
// These kernels build x^, b^ (per head when theta is given, since the turn is per head) and c^
// as fp32 in the workspace, the generic chunk pipeline runs the expanded problem, and
// trap_compact_y writes the R real output channels back in the I/O dtype.  Scaling and turning
// happen in fp32, so no bf16 rounding of a derived operand enters the result.
#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {

namespace {

constexpr int kTrapThreads = 256;

// x^[b,t,m,h,p], m < 2R: gamma x_t for m < R, beta x_{t-1} (prev_x at t = 0) for m >= R.
template <typename T>
__global__ void __launch_bounds__(kTrapThreads)
    trap_expand_x(const T* __restrict__ x, const float* __restrict__ gamma,
                  const float* __restrict__ beta, const T* __restrict__ prev_x,
                  float* __restrict__ xh, int64_t batch, int64_t Tn, int64_t R, int64_t H,
                  int64_t P) {
  const int64_t n = batch * Tn * 2 * R * H * P;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = idx % P;
    const int64_t h = (idx / P) % H;
    const int64_t m = (idx / (P * H)) % (2 * R);
    const int64_t bt = idx / (P * H * 2 * R);   // b * Tn + t
    const int64_t t = bt % Tn, b = bt / Tn;
    float v;
    if (m < R) {
      v = gamma[bt * H + h] * ld_f32(x + ((bt * R + m) * H + h) * P + p);
    } else {
      const int64_t r = m - R;
      float src = 0.f;
      if (t > 0) {
        src = ld_f32(x + (((bt - 1) * R + r) * H + h) * P + p);
      } else if (prev_x) {
        src = ld_f32(prev_x + ((b * R + r) * H + h) * P + p);
      }
      v = beta[bt * H + h] * src;
    }
    xh[idx] = v;
  }
}

// b^ and c^ [b,t,m,g2,n] over pairs (n = 2k, 2k+1).  g2 runs over heads when theta is given
// (the shifted channel is turned by that head's theta_t) and over groups otherwise.
template <typename T>
__global__ void __launch_bounds__(kTrapThreads)
    trap_expand_bc(const T* __restrict__ B, const T* __restrict__ C,
                   const float* __restrict__ theta, const T* __restrict__ prev_B,
                   float* __restrict__ bh, float* __restrict__ ch, int64_t batch, int64_t Tn,
                   int64_t R, int64_t H, int64_t G, int64_t G2, int64_t N) {
  const int64_t K = (N + 1) / 2;   // pairs (the last one single when N is odd, no theta)
  const int64_t n_all = batch * Tn * 2 * R * G2 * K;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n_all;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = idx % K;
    const int64_t g2 = (idx / K) % G2;
    const int64_t m = (idx / (K * G2)) % (2 * R);
    const int64_t bt = idx / (K * G2 * 2 * R);
    const int64_t t = bt % Tn, b = bt / Tn;
    const int64_t g = theta ? g2 / (H / G) : g2;
    const int64_t n0 = 2 * k;
    const bool two = n0 + 1 < N;
    float b0, b1 = 0.f, c0 = 0.f, c1 = 0.f;
    if (m < R) {
      const int64_t o = ((bt * R + m) * G + g) * N + n0;
      b0 = ld_f32(B + o);
      c0 = ld_f32(C + o);
      if (two) {
        b1 = ld_f32(B + o + 1);
        c1 = ld_f32(C + o + 1);
      }
    } else {
      const int64_t r = m - R;
      const T* src = nullptr;
      if (t > 0) {
        src = B + (((bt - 1) * R + r) * G + g) * N + n0;
      } else if (prev_B) {
        src = prev_B + ((b * R + r) * G + g) * N + n0;
      }
      b0 = src ? ld_f32(src) : 0.f;
      if (two) b1 = src ? ld_f32(src + 1) : 0.f;
      if (theta) {   // turn the pair by +theta_t of head g2
        float s, co;
        sincosf(theta[(bt * H + g2) * (N / 2) + k], &s, &co);
        const float e = co * b0 - s * b1, od = s * b0 + co * b1;
        b0 = e;
        b1 = od;
      }
    }
    const int64_t out = ((bt * 2 * R + m) * G2 + g2) * N + n0;
    bh[out] = b0;
    ch[out] = c0;
    if (two) {
      bh[out + 1] = b1;
      ch[out + 1] = c1;
    }
  }
}

// y[b,t,r,h,p] = y^[b,t,r,h,p] for the R real output channels (r < R of 2R).
template <typename T>
__global__ void __launch_bounds__(kTrapThreads)
    trap_compact_y(const float* __restrict__ yh, T* __restrict__ y, int64_t batch, int64_t Tn,
                   int64_t R, int64_t H, int64_t P) {
  const int64_t n = batch * Tn * R * H * P;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t hp = idx % (H * P);
    const int64_t r = (idx / (H * P)) % R;
    const int64_t bt = idx / (H * P * R);
    st_from_f32(y + idx, yh[(bt * 2 * R + r) * H * P + hp]);
  }
}

unsigned grid_for(int64_t n) {
  const int64_t blocks = (n + kTrapThreads - 1) / kTrapThreads;
  return (unsigned)(blocks < 152 * 16 ? (blocks < 1 ? 1 : blocks) : 152 * 16);
}

template <typename T>
cudaError_t expand_typed(const TrapArgs& a, cudaStream_t st) {
  const int64_t nx = a.batch * a.T * 2 * a.R * a.H * a.P;
  trap_expand_x<T><<<grid_for(nx), kTrapThreads, 0, st>>>(
      static_cast<const T*>(a.x), a.gamma, a.beta, static_cast<const T*>(a.prev_x), a.xh,
      a.batch, a.T, a.R, a.H, a.P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nbc = a.batch * a.T * 2 * a.R * a.G2 * ((a.N + 1) / 2);
  trap_expand_bc<T><<<grid_for(nbc), kTrapThreads, 0, st>>>(
      static_cast<const T*>(a.B), static_cast<const T*>(a.C), a.theta,
      static_cast<const T*>(a.prev_B), a.bh, a.ch, a.batch, a.T, a.R, a.H, a.G, a.G2, a.N);
  return cudaGetLastError();
}

template <typename T>
cudaError_t compact_typed(const TrapArgs& a, cudaStream_t st) {
  const int64_t n = a.batch * a.T * a.R * a.H * a.P;
  trap_compact_y<T><<<grid_for(n), kTrapThreads, 0, st>>>(a.yh, static_cast<T*>(a.y), a.batch,
                                                          a.T, a.R, a.H, a.P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t trap_expand(const TrapArgs& a, bool bf16, cudaStream_t st) {
  return bf16 ? expand_typed<__nv_bfloat16>(a, st) : expand_typed<float>(a, st);
}

cudaError_t trap_compact(const TrapArgs& a, bool bf16, cudaStream_t st) {
  return bf16 ? compact_typed<__nv_bfloat16>(a, st) : compact_typed<float>(a, st);
}

}  // namespace ssd
