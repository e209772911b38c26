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
// as fp32 in the workspace, the chunk kernels run the expanded problem (the register-tiled
// fp32 kernels for P = N = 64, the generic ones otherwise), and
// trap_compact_y writes the R real output channels back in the I/O dtype.  Scaling and turning
// happen in fp32, so no bf16 rounding of a derived operand enters the result.
#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {

namespace {

// One block per step (b, t): nested loops over the channel, the head (or group) rows and the
// row's elements, so no index is recovered by division and the 32 lanes of a row are coalesced.
constexpr int kRowLanes = 32, kRowsPerBlock = 8;

// True if step t of sequence b is padding (t >= valid_len[b], clamped to [0, Tn]).
__device__ __forceinline__ bool pad_step(const int64_t* valid_len, int64_t b, int64_t t,
                                         int64_t Tn) {
  if (valid_len == nullptr) return false;
  const int64_t v = __ldg(valid_len + b);
  return t >= (v < 0 ? 0 : (v > Tn ? Tn : v));
}

unsigned step_blocks(int64_t steps) {
  return (unsigned)(steps < 1 ? 1 : (steps > 0x7fffffff ? 0x7fffffff : steps));
}

// x^[b,t,m,h,:], m < 2R: gamma x_t for m < R, beta x_{t-1} (prev_x at t = 0) for m >= R.
template <typename T>
__global__ void __launch_bounds__(kRowLanes * kRowsPerBlock)
    trap_expand_x(const T* __restrict__ x, const float* __restrict__ gamma,
                  const float* __restrict__ beta, const T* __restrict__ prev_x,
                  float* __restrict__ xh, const int64_t* __restrict__ valid_len,
                  int64_t batch, int64_t Tn, int64_t R, int64_t H, int64_t P, WsHeader* hdr) {
  for (int64_t bt = blockIdx.x; bt < batch * Tn; bt += gridDim.x) {
    const int64_t t = bt % Tn, b = bt / Tn;
    if (pad_step(valid_len, b, t, Tn)) continue;   // padding: never read downstream
    for (int64_t m = 0; m < 2 * R; ++m) {
      for (int64_t h = threadIdx.y; h < H; h += kRowsPerBlock) {
        const T* src = nullptr;
        float w;
        if (m < R) {
          src = x + ((bt * R + m) * H + h) * P;
          w = gamma[bt * H + h];
        } else {
          if (t > 0) {
            src = x + (((bt - 1) * R + (m - R)) * H + h) * P;
          } else if (prev_x) {
            src = prev_x + ((b * R + (m - R)) * H + h) * P;
          }
          w = beta[bt * H + h];
        }
        float* dst = xh + ((bt * 2 * R + m) * H + h) * P;
        for (int64_t p = threadIdx.x; p < P; p += kRowLanes)
          if (SSD_INDEX_OK(hdr, (dst - xh) + p, batch * Tn * 2 * R * H * P, 40))
            dst[p] = src ? w * ld_f32(src + p) : 0.f;
      }
    }
  }
}

// b^ and c^ [b,t,m,g2,:].  g2 runs over heads when theta is given (the shifted channel is turned
// by that head's theta_t) and over groups otherwise.  Lanes walk the interleaved pairs.
template <typename T>
__global__ void __launch_bounds__(kRowLanes * kRowsPerBlock)
    trap_expand_bc(const T* __restrict__ B, const T* __restrict__ C,
                   const float* __restrict__ theta, const T* __restrict__ prev_B,
                   float* __restrict__ bh, float* __restrict__ ch,
                   const int64_t* __restrict__ valid_len, int64_t batch, int64_t Tn, int64_t R,
                   int64_t H, int64_t G, int64_t G2, int64_t N, WsHeader* hdr) {
  const int64_t K = (N + 1) / 2;   // pairs (the last one single when N is odd, no theta)
  const int64_t hpg = H / G;
  for (int64_t bt = blockIdx.x; bt < batch * Tn; bt += gridDim.x) {
    const int64_t t = bt % Tn, b = bt / Tn;
    if (pad_step(valid_len, b, t, Tn)) continue;
    for (int64_t m = 0; m < 2 * R; ++m) {
      for (int64_t g2 = threadIdx.y; g2 < G2; g2 += kRowsPerBlock) {
        const int64_t g = theta ? g2 / hpg : g2;
        const T *bsrc = nullptr, *csrc = nullptr;
        if (m < R) {
          bsrc = B + ((bt * R + m) * G + g) * N;
          csrc = C + ((bt * R + m) * G + g) * N;
        } else if (t > 0) {
          bsrc = B + (((bt - 1) * R + (m - R)) * G + g) * N;
        } else if (prev_B) {
          bsrc = prev_B + ((b * R + (m - R)) * G + g) * N;
        }
        const float* th = (theta && m >= R) ? theta + (bt * H + g2) * (N / 2) : nullptr;
        float* bd = bh + ((bt * 2 * R + m) * G2 + g2) * N;
        float* cd = ch + ((bt * 2 * R + m) * G2 + g2) * N;
        for (int64_t k = threadIdx.x; k < K; k += kRowLanes) {
          const int64_t n0 = 2 * k;
          const bool two = n0 + 1 < N;
          float b0 = bsrc ? ld_f32(bsrc + n0) : 0.f;
          float b1 = (bsrc && two) ? ld_f32(bsrc + n0 + 1) : 0.f;
          if (th) {   // turn the pair by +theta_t of head g2
            float sn, co;
            sincosf(th[k], &sn, &co);
            const float e = co * b0 - sn * b1, od = sn * b0 + co * b1;
            b0 = e;
            b1 = od;
          }
          if (!SSD_INDEX_OK(hdr, (bd - bh) + n0 + (two ? 1 : 0), batch * Tn * 2 * R * G2 * N, 41))
            continue;
          bd[n0] = b0;
          cd[n0] = csrc ? ld_f32(csrc + n0) : 0.f;
          if (two) {
            bd[n0 + 1] = b1;
            cd[n0 + 1] = csrc ? ld_f32(csrc + n0 + 1) : 0.f;
          }
        }
      }
    }
  }
}

// y[b,t,r,h,:] = y^[b,t,r,h,:] for the R real output channels (r < R of 2R).
template <typename T>
__global__ void __launch_bounds__(kRowLanes * kRowsPerBlock)
    trap_compact_y(const float* __restrict__ yh, T* __restrict__ y,
                   const int64_t* __restrict__ valid_len, int64_t batch, int64_t Tn, int64_t R,
                   int64_t H, int64_t P, WsHeader* hdr) {
  for (int64_t bt = blockIdx.x; bt < batch * Tn; bt += gridDim.x) {
    if (pad_step(valid_len, bt / Tn, bt % Tn, Tn)) continue;   // y at padding is not written
    for (int64_t r = 0; r < R; ++r) {
      for (int64_t h = threadIdx.y; h < H; h += kRowsPerBlock) {
        const float* src = yh + ((bt * 2 * R + r) * H + h) * P;
        T* dst = y + ((bt * R + r) * H + h) * P;
        for (int64_t p = threadIdx.x; p < P; p += kRowLanes)
          if (SSD_INDEX_OK(hdr, (dst - y) + p, batch * Tn * R * H * P, 42)) st_from_f32(dst + p, src[p]);
      }
    }
  }
}

template <typename T>
cudaError_t expand_typed(const TrapArgs& a, cudaStream_t st) {
  const dim3 blk(kRowLanes, kRowsPerBlock);
  trap_expand_x<T><<<step_blocks(a.batch * a.T), blk, 0, st>>>(
      static_cast<const T*>(a.x), a.gamma, a.beta, static_cast<const T*>(a.prev_x), a.xh,
      a.valid_len, a.batch, a.T, a.R, a.H, a.P, a.hdr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  trap_expand_bc<T><<<step_blocks(a.batch * a.T), blk, 0, st>>>(
      static_cast<const T*>(a.B), static_cast<const T*>(a.C), a.theta,
      static_cast<const T*>(a.prev_B), a.bh, a.ch, a.valid_len, a.batch, a.T, a.R, a.H, a.G,
      a.G2, a.N, a.hdr);
  return cudaGetLastError();
}

template <typename T>
cudaError_t compact_typed(const TrapArgs& a, cudaStream_t st) {
  trap_compact_y<T><<<step_blocks(a.batch * a.T), dim3(kRowLanes, kRowsPerBlock), 0,
                      st>>>(a.yh, static_cast<T*>(a.y), a.valid_len, a.batch, a.T, a.R, a.H, a.P, a.hdr);
  return cudaGetLastError();
}

// Rows of 16-byte words: copy n words from src (zeros if src is null) to dst, lanes along the row.
__device__ __forceinline__ void copy_row16(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                           int64_t n, WsHeader* hdr, const uint4* base,
                                           int64_t extent, int site) {
  for (int64_t k = threadIdx.x; k < n; k += kRowLanes)
    if (SSD_INDEX_OK(hdr, (dst - base) + k, extent, site))
      dst[k] = src ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
}

// x^, B^, C^ (exact bf16 copies) and the write weights w^ = [gamma_t, beta_t] of step (b, t).
__global__ void __launch_bounds__(kRowLanes * kRowsPerBlock)
    trap_fused_expand_kernel(TrapFusedArgs a) {
  const int64_t Tn = a.T, R = a.R, R2 = 2 * a.R;
  const int64_t xw = a.P / 8, bw = a.N / 8;   // 16-byte words per row
  const uint4* x = static_cast<const uint4*>(a.x);
  const uint4* B = static_cast<const uint4*>(a.B);
  const uint4* C = static_cast<const uint4*>(a.C);
  const uint4* px = static_cast<const uint4*>(a.prev_x);
  const uint4* pB = static_cast<const uint4*>(a.prev_B);
  uint4* xq = static_cast<uint4*>(a.xq);
  uint4* bq = static_cast<uint4*>(a.bq);
  uint4* cq = static_cast<uint4*>(a.cq);
  for (int64_t bt = blockIdx.x; bt < a.batch * Tn; bt += gridDim.x) {
    const int64_t t = bt % Tn, b = bt / Tn;
    if (pad_step(a.valid_len, b, t, Tn)) continue;   // padding: never read downstream
    for (int64_t m = 0; m < R2; ++m) {
      const bool cur = m < R;
      for (int64_t h = threadIdx.y; h < a.H; h += kRowsPerBlock) {
        const uint4* src = cur ? x + ((bt * R + m) * a.H + h) * xw
                               : (t > 0 ? x + (((bt - 1) * R + (m - R)) * a.H + h) * xw
                                        : (px ? px + ((b * R + (m - R)) * a.H + h) * xw : nullptr));
        copy_row16(xq + ((bt * R2 + m) * a.H + h) * xw, src, xw, a.hdr, xq,
                   a.batch * Tn * R2 * a.H * xw, 43);
        if (threadIdx.x == 0 &&
            SSD_INDEX_OK(a.hdr, (bt * R2 + m) * a.H + h, a.batch * Tn * R2 * a.H, 44))
          a.wq[(bt * R2 + m) * a.H + h] = cur ? a.gamma[bt * a.H + h] : a.beta[bt * a.H + h];
      }
      for (int64_t g = threadIdx.y; g < a.G; g += kRowsPerBlock) {
        const uint4* bsrc = cur ? B + ((bt * R + m) * a.G + g) * bw
                                : (t > 0 ? B + (((bt - 1) * R + (m - R)) * a.G + g) * bw
                                         : (pB ? pB + ((b * R + (m - R)) * a.G + g) * bw : nullptr));
        const int64_t bext = a.batch * Tn * R2 * a.G * bw;
        copy_row16(bq + ((bt * R2 + m) * a.G + g) * bw, bsrc, bw, a.hdr, bq, bext, 45);
        copy_row16(cq + ((bt * R2 + m) * a.G + g) * bw,
                   cur ? C + ((bt * R + m) * a.G + g) * bw : nullptr, bw, a.hdr, cq, bext, 46);
      }
    }
  }
}

// y[b, t, r] = y^[b, t, r] for the R real output channels (bf16 rows copied as 16-byte words).
__global__ void __launch_bounds__(kRowLanes * kRowsPerBlock)
    trap_fused_compact_kernel(TrapFusedArgs a) {
  const int64_t Tn = a.T, R = a.R, R2 = 2 * a.R, xw = a.P / 8;
  const uint4* yq = static_cast<const uint4*>(a.yq);
  uint4* y = static_cast<uint4*>(a.y);
  for (int64_t bt = blockIdx.x; bt < a.batch * Tn; bt += gridDim.x) {
    if (pad_step(a.valid_len, bt / Tn, bt % Tn, Tn)) continue;   // y at padding is not written
    for (int64_t r = 0; r < R; ++r)
      for (int64_t h = threadIdx.y; h < a.H; h += kRowsPerBlock)
        copy_row16(y + ((bt * R + r) * a.H + h) * xw, yq + ((bt * R2 + r) * a.H + h) * xw, xw,
                   a.hdr, y, a.batch * Tn * R * a.H * xw, 47);
  }
}

}  // namespace

cudaError_t trap_fused_expand(const TrapFusedArgs& a, cudaStream_t st) {
  trap_fused_expand_kernel<<<step_blocks(a.batch * a.T), dim3(kRowLanes, kRowsPerBlock), 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t trap_fused_compact(const TrapFusedArgs& a, cudaStream_t st) {
  trap_fused_compact_kernel<<<step_blocks(a.batch * a.T), dim3(kRowLanes, kRowsPerBlock), 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t trap_expand(const TrapArgs& a, bool bf16, cudaStream_t st) {
  return bf16 ? expand_typed<__nv_bfloat16>(a, st) : expand_typed<float>(a, st);
}

cudaError_t trap_compact(const TrapArgs& a, bool bf16, cudaStream_t st) {
  return bf16 ? compact_typed<__nv_bfloat16>(a, st) : compact_typed<float>(a, st);
}

}  // namespace ssd
