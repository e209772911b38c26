// Backward of the trapezoidal Mamba-3 forward through its 2R-channel expansion.
//
// The trapezoidal forward (scan.py page, the trapezoidal forward; moments.rs page, combined
// injections) runs as one scan with 2R write channels, x^ = [gamma_t x_t, beta_t x_{t-1}],
// B^ = [B_t, R(theta_t) B_{t-1}] (per head when theta is given), C^ = [C_t, 0].  Its reverse mode
// is the backward of that scan (ssd_chunked_backward on the expanded problem, with dy^ = [dy, 0])
// followed by the chain rule through the expansion:
//   dx_t      = gamma_t dx^[t, r] + beta_{t+1} dx^[t+1, R+r]      dprev_x = beta_0 dx^[0, R+r]
//   dgamma_t  = sum_{r,p} dx^[t, r] x_t                           dbeta_t = sum_{r,p} dx^[t, R+r] x_{t-1}
//   dB_t      = sum over the group's heads of dB^[t, r] + R(theta_{t+1})^T dB^[t+1, R+r]
//   dprev_B   = sum over the group's heads of R(theta_0)^T dB^[0, R+r]
//   dC_t      = sum over the group's heads of dC^[t, r]
//   dtheta_t  = dtheta^_t + sum_r (dB^_1 B^_0 - dB^_0 B^_1)[t, R+r]   (d R(th) v / d th = J R(th) v)
// ddA and dinit are the expanded problem's.
#include <string.h>

#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kLanes = 32, kRows = 8;

unsigned tb_blocks(int64_t n) {
  return (unsigned)(n < 1 ? 1 : (n > 0x7fffffff ? 0x7fffffff : n));
}

// dy^ [b,T,2R,H,P]: dy on the first R channels, zero on the rest.  One block per step.
__global__ void __launch_bounds__(kLanes * kRows)
    tbwd_expand_dy(const float* __restrict__ dy, float* __restrict__ dyh, int64_t steps,
                   int64_t R, int64_t H, int64_t P) {
  for (int64_t bt = blockIdx.x; bt < steps; bt += gridDim.x) {
    for (int64_t m = 0; m < 2 * R; ++m) {
      for (int64_t h = threadIdx.y; h < H; h += kRows) {
        float* dst = dyh + ((bt * 2 * R + m) * H + h) * P;
        const float* src = m < R ? dy + ((bt * R + m) * H + h) * P : nullptr;
        for (int64_t p = threadIdx.x; p < P; p += kLanes) dst[p] = src ? src[p] : 0.f;
      }
    }
  }
}

__device__ __forceinline__ float warp_total(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// dx, dgamma, dbeta (and dprev_x at t = 0) from dx^: one block per step, one warp per head row.
template <typename T>
__global__ void __launch_bounds__(kLanes * kRows)
    tbwd_x_kernel(const T* __restrict__ x, const T* __restrict__ prev_x,
                  const float* __restrict__ gamma, const float* __restrict__ beta,
                  const float* __restrict__ dxh, float* __restrict__ dx,
                  float* __restrict__ dgamma, float* __restrict__ dbeta,
                  float* __restrict__ dprev_x, int64_t batch, int64_t Tn, int64_t R, int64_t H,
                  int64_t P) {
  for (int64_t bt = blockIdx.x; bt < batch * Tn; bt += gridDim.x) {
    const int64_t t = bt % Tn, b = bt / Tn;
    for (int64_t h = threadIdx.y; h < H; h += kRows) {
      const float gm = gamma[bt * H + h];
      const float bn = t + 1 < Tn ? beta[(bt + 1) * H + h] : 0.f;
      float sg = 0.f, sb = 0.f;
      for (int64_t r = 0; r < R; ++r) {
        const float* cur = dxh + ((bt * 2 * R + r) * H + h) * P;             // dx^[t, r]
        const float* sh = dxh + ((bt * 2 * R + R + r) * H + h) * P;          // dx^[t, R+r]
        const float* nxt = t + 1 < Tn ? dxh + (((bt + 1) * 2 * R + R + r) * H + h) * P : nullptr;
        const T* xc = x + ((bt * R + r) * H + h) * P;
        const T* xp = t > 0 ? x + (((bt - 1) * R + r) * H + h) * P
                            : (prev_x ? prev_x + ((b * R + r) * H + h) * P : nullptr);
        float* out = dx + ((bt * R + r) * H + h) * P;
        for (int64_t p = threadIdx.x; p < P; p += kLanes) {
          const float xv = ld_f32(xc + p);
          sg = fmaf(cur[p], xv, sg);
          if (xp) sb = fmaf(sh[p], ld_f32(xp + p), sb);
          out[p] = fmaf(gm, cur[p], nxt ? bn * nxt[p] : 0.f);
          if (t == 0 && dprev_x) dprev_x[((b * R + r) * H + h) * P + p] = beta[bt * H + h] * sh[p];
        }
      }
      sg = warp_total(sg);
      sb = warp_total(sb);
      if (threadIdx.x == 0) {
        dgamma[bt * H + h] = sg;
        dbeta[bt * H + h] = sb;
      }
    }
  }
}

// dB, dC (and dprev_B at t = 0) from dB^, dC^, and the shifted channel's part of dtheta: one block
// per step.  G2 = H (B^ per head) when theta is given, else G2 = G.
__global__ void __launch_bounds__(kLanes * kRows)
    tbwd_bc_kernel(const float* __restrict__ bh, const float* __restrict__ dbh,
                   const float* __restrict__ dch, const float* __restrict__ theta,
                   float* __restrict__ dB, float* __restrict__ dC, float* __restrict__ dtheta,
                   float* __restrict__ dprev_B, int64_t batch, int64_t Tn, int64_t R, int64_t G,
                   int64_t G2, int64_t N) {
  const int64_t K = N / 2, per = G2 / G;   // heads (or 1) per group
  for (int64_t bt = blockIdx.x; bt < batch * Tn; bt += gridDim.x) {
    const int64_t t = bt % Tn, b = bt / Tn;
    if (theta) {   // dtheta_t += sum_r (dB^_1 B^_0 - dB^_0 B^_1) of the shifted channels
      for (int64_t h = threadIdx.y; h < G2; h += kRows) {
        for (int64_t k = threadIdx.x; k < K; k += kLanes) {
          float s = 0.f;
          for (int64_t r = 0; r < R; ++r) {
            const int64_t o = ((bt * 2 * R + R + r) * G2 + h) * N + 2 * k;
            s += dbh[o + 1] * bh[o] - dbh[o] * bh[o + 1];
          }
          dtheta[(bt * G2 + h) * K + k] += s;
        }
      }
    }
    for (int64_t r = 0; r < R; ++r) {
      for (int64_t g = threadIdx.y; g < G; g += kRows) {
        for (int64_t k = threadIdx.x; k < (N + 1) / 2; k += kLanes) {
          const int64_t n0 = 2 * k;
          const bool two = n0 + 1 < N;
          float b0 = 0.f, b1 = 0.f, c0 = 0.f, c1 = 0.f, q0 = 0.f, q1 = 0.f;
          for (int64_t g2 = g * per; g2 < (g + 1) * per; ++g2) {
            const int64_t oc = ((bt * 2 * R + r) * G2 + g2) * N + n0;
            b0 += dbh[oc];
            c0 += dch[oc];
            if (two) {
              b1 += dbh[oc + 1];
              c1 += dch[oc + 1];
            }
            // the shifted channel of the next step (t+1) carries B_t, turned by theta_{t+1};
            // at t = 0 this step's shifted channel carries the previous write
            for (int which = 0; which < 2; ++which) {
              const int64_t bs = which == 0 ? bt + 1 : bt;
              if (which == 0 && t + 1 >= Tn) continue;
              if (which == 1 && (t != 0 || !dprev_B)) continue;
              const int64_t os = ((bs * 2 * R + R + r) * G2 + g2) * N + n0;
              float e0 = dbh[os], e1 = two ? dbh[os + 1] : 0.f;
              if (theta) {   // R(theta)^T = R(-theta)
                float sn, cs;
                sincosf(theta[(bs * G2 + g2) * K + k], &sn, &cs);
                const float f0 = cs * e0 + sn * e1, f1 = cs * e1 - sn * e0;
                e0 = f0;
                e1 = f1;
              }
              if (which == 0) {
                b0 += e0;
                b1 += e1;
              } else {
                q0 += e0;
                q1 += e1;
              }
            }
          }
          const int64_t o = ((bt * R + r) * G + g) * N + n0;
          dB[o] = b0;
          dC[o] = c0;
          if (two) {
            dB[o + 1] = b1;
            dC[o + 1] = c1;
          }
          if (t == 0 && dprev_B) {
            const int64_t op = ((b * R + r) * G + g) * N + n0;
            dprev_B[op] = q0;
            if (two) dprev_B[op + 1] = q1;
          }
        }
      }
    }
  }
}

// Workspace after the 256-byte header: the expanded problem (x^, B^, C^ fp32, as the forward
// builds them), dy^, its gradients dx^, dB^, dC^ (and dtheta^), then the inner backward's own
// workspace.
struct TbwdLayout {
  size_t xh = 0, bh = 0, ch = 0, dyh = 0, dxh = 0, dbh = 0, dch = 0, dth = 0, inner = 0,
         inner_bytes = 0, total = 0;
};

ssd_shape tbwd_expanded(const ssd_shape* s) {
  ssd_shape e = *s;
  e.mimo_rank = 2 * s->mimo_rank;
  e.io_dtype = SSD_F32;
  if (s->has_theta) e.ngroups = s->nheads;
  return e;
}

ssd_status tbwd_status(const ssd_shape* s) {
  const ssd_status st = shape_status(s);
  if (st != SSD_OK) return st;
  if (s->mimo_rank > (int64_t(1) << 30)) return SSD_ERR_UNSUPPORTED;
  const ssd_shape e = tbwd_expanded(s);
  return ssd_backward_workspace_bytes(&e) == 0 ? SSD_ERR_UNSUPPORTED : SSD_OK;
}

TbwdLayout tbwd_layout(const ssd_shape* s) {
  const ssd_shape e = tbwd_expanded(s);
  const size_t steps = (size_t)(s->batch * s->seqlen), R2 = (size_t)e.mimo_rank;
  const size_t xs = sizeof(float) * steps * R2 * (size_t)(s->nheads * s->headdim);
  const size_t bs = sizeof(float) * steps * R2 * (size_t)(e.ngroups * s->dstate);
  TbwdLayout L;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kWsAlign);
    return at;
  };
  L.xh = take(xs);
  L.bh = take(bs);
  L.ch = take(bs);
  L.dyh = take(xs);
  L.dxh = take(xs);
  L.dbh = take(bs);
  L.dch = take(bs);
  if (s->has_theta) L.dth = take(sizeof(float) * steps * (size_t)(s->nheads * (s->dstate / 2)));
  L.inner_bytes = ssd_backward_workspace_bytes(&e);
  L.inner = take(L.inner_bytes);
  L.total = off;
  return L;
}

bool a16(const void* q) { return q == nullptr || aligned16(q); }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_trapezoidal_backward_workspace_bytes(const ssd_shape* shape) {
  if (tbwd_status(shape) != SSD_OK) return 0;
  return tbwd_layout(shape).total;
}

ssd_status ssd_trapezoidal_backward(
    const ssd_shape* shape, const void* x, const float* dA, const void* B, const void* C,
    const float* gamma, const float* beta, const float* theta, const void* prev_x,
    const void* prev_B, const float* init_state, const float* dy, const float* dfinal, float* dx,
    float* ddA, float* dB, float* dC, float* dgamma, float* dbeta, float* dtheta, float* dinit,
    float* dprev_x, float* dprev_B, void* workspace, size_t workspace_bytes, void* stream) {
  const ssd_status vs = tbwd_status(shape);
  if (vs != SSD_OK) return vs;
  if (!x || !dA || !B || !C || !gamma || !beta || !dy || !dx || !ddA || !dB || !dC || !dgamma ||
      !dbeta)
    return SSD_ERR_INVALID_ARG;
  const bool rot = shape->has_theta != 0;
  if (rot != (theta != nullptr) || rot != (dtheta != nullptr)) return SSD_ERR_INVALID_ARG;
  if ((prev_x == nullptr) != (prev_B == nullptr)) return SSD_ERR_INVALID_ARG;
  if (!prev_x && (dprev_x || dprev_B)) return SSD_ERR_INVALID_ARG;
  const void* ptrs[] = {x,  dA, B,   C,   gamma,  beta,  theta,  prev_x, prev_B, init_state,
                        dy, dfinal, dx, ddA, dB, dC, dgamma, dbeta, dtheta, dinit, dprev_x, dprev_B};
  for (const void* q : ptrs)
    if (!a16(q)) return SSD_ERR_INVALID_ARG;
  const TbwdLayout lay = tbwd_layout(shape);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0 ||
      workspace_bytes < lay.total)
    return SSD_ERR_WORKSPACE;
  const ssd_shape e = tbwd_expanded(shape);
  char* ws = static_cast<char*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = shape->io_dtype == SSD_BF16;
  const int64_t steps = shape->batch * shape->seqlen, R = shape->mimo_rank, H = shape->nheads;
  const int64_t P = shape->headdim, N = shape->dstate, G = shape->ngroups, G2 = e.ngroups;
  float* xh = reinterpret_cast<float*>(ws + lay.xh);
  float* bh = reinterpret_cast<float*>(ws + lay.bh);
  float* ch = reinterpret_cast<float*>(ws + lay.ch);
  float* dyh = reinterpret_cast<float*>(ws + lay.dyh);
  float* dxh = reinterpret_cast<float*>(ws + lay.dxh);
  float* dbh = reinterpret_cast<float*>(ws + lay.dbh);
  float* dch = reinterpret_cast<float*>(ws + lay.dch);
  float* dth = rot ? reinterpret_cast<float*>(ws + lay.dth) : nullptr;

  TrapArgs t;
  memset(&t, 0, sizeof(t));
  t.x = x;
  t.B = B;
  t.C = C;
  t.prev_x = prev_x;
  t.prev_B = prev_B;
  t.gamma = gamma;
  t.beta = beta;
  t.theta = theta;
  t.xh = xh;
  t.bh = bh;
  t.ch = ch;
  t.batch = shape->batch;
  t.T = shape->seqlen;
  t.R = R;
  t.H = H;
  t.G = G;
  t.G2 = G2;
  t.P = P;
  t.N = N;
  t.hdr = reinterpret_cast<WsHeader*>(ws);   // this call's own header (offset 0)
  if (trap_expand(t, bf16, st) != cudaSuccess) return SSD_ERR_CUDA;
  const dim3 blk(kLanes, kRows);
  tbwd_expand_dy<<<tb_blocks(steps), blk, 0, st>>>(dy, dyh, steps, R, H, P);
  if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;

  // The inner backward's workspace header must be clean like any other: it is this call's own.
  if (cudaMemsetAsync(ws + lay.inner, 0, sizeof(WsHeader), st) != cudaSuccess) return SSD_ERR_CUDA;
  const ssd_status si = ssd_chunked_backward(&e, xh, dA, bh, ch, theta, init_state, dyh, dfinal,
                                             dxh, ddA, dbh, dch, dth, dinit, ws + lay.inner,
                                             lay.inner_bytes, stream);
  if (si != SSD_OK) return si;

  if (bf16) {
    tbwd_x_kernel<__nv_bfloat16><<<tb_blocks(steps), blk, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(prev_x), gamma,
        beta, dxh, dx, dgamma, dbeta, dprev_x, shape->batch, shape->seqlen, R, H, P);
  } else {
    tbwd_x_kernel<float><<<tb_blocks(steps), blk, 0, st>>>(
        static_cast<const float*>(x), static_cast<const float*>(prev_x), gamma, beta, dxh, dx,
        dgamma, dbeta, dprev_x, shape->batch, shape->seqlen, R, H, P);
  }
  if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  if (rot && cudaMemcpyAsync(dtheta, dth, sizeof(float) * (size_t)(steps * H * (N / 2)),
                             cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return SSD_ERR_CUDA;
  tbwd_bc_kernel<<<tb_blocks(steps), blk, 0, st>>>(bh, dbh, dch, theta, dB, dC, dtheta, dprev_B,
                                                    shape->batch, shape->seqlen, R, G, G2, N);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
