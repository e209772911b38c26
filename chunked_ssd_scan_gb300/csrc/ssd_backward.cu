// Backward of the chunked SSD forward (unrotated; CUDA-core fp32), recompute per chunk.
//
// The scan.py page asks for a scan that can train; the moments.rs page's memory model keeps only
// the chunk-boundary states and recomputes inside a chunk.  Three launches:
//   1. bwd_chunk_state_kernel: per chunk both rank-Lr products, the chunk's own end state
//      S_c = sum_i exp(cum_end - cum_i) x_i (outer) B_i and D_c = sum_i exp(cum_i) dy_i (outer) C_i,
//      the part of dL/dh_in(c) that the chunk's own outputs contribute;
//   2. bwd_carry_kernel: the carry across chunks both ways, h_in(c) forward (K4) and
//      G_c = dL/dh_out(c) backward (G_{nch-1} = dfinal, dL/dh_in(c) = exp(cum_end(c)) G_c + D_c,
//      dinit = dL/dh_in(0));
//   3. bwd_chunk_grad_kernel: per chunk, with L_ij = exp(cum_i - cum_j) below the step diagonal,
//      CB_ij = C_i . B_j and DX_ij = dy_i . x_j:
//        dx_j = sum_i L_ij CB_ij dy_i + exp(cum_end - cum_j) G B_j
//        dB_j = sum_i L_ij DX_ij C_i + exp(cum_end - cum_j) G^T x_j
//        dC_i = sum_j L_ij DX_ij B_j + exp(cum_i) h_in^T dy_i
//      and the gradient of every prefix sum cum_s (from L, exp(cum_i), exp(cum_end - cum_j) and
//      exp(cum_end) h_in), whose suffix sums over the chunk's steps are ddA.
// Rows are rank-fused (i = t R + r, step i / R), 64 per chunk; dB and dC add over the heads of a
// group.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kBwdThreads = 256, kBwdWarps = kBwdThreads / 32;
constexpr int kBwdRows = 64;   // fused rows per chunk
constexpr int kBwdMaxP = 64, kBwdMaxN = 128;

// fp64 inclusive prefix sums of dA over the chunk's steps (warp 0); steps at or after nv are 0.
__device__ void bwd_cumsum(const float* __restrict__ src, int64_t stride, int l, int nv,
                           double* cum) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int per = (l + 31) / 32;
  const int beg = min(l, lane * per), end = min(l, beg + per);
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
    cum[t] = acc;
  }
}

// Real steps of chunk c.
__device__ __forceinline__ int bwd_steps(const GenericParams& p, int64_t c) {
  return (int)min(p.l, p.T - c * p.l);
}

// Register tiles: thread t owns rows t / 16 + 16 a (a < 4) and columns t % 16 + 16 q (q < NQ)
// of a 64 x (16 NQ) output, so one k step loads 4 + NQ values for 4 NQ FMAs and the 16 lanes of
// a half-warp read 16 consecutive floats.
template <int NQ>
constexpr int nq_cols() { return 16 * NQ; }

// Dynamic shared memory of bwd_chunk_state_kernel: the prefix sums, then the scaled x and dy rows
// [Lr][P] and the B and C rows [Lr][N].
size_t bwd_state_smem(int64_t Lr, int64_t P, int64_t N) {
  return kBwdRows * sizeof(double) + sizeof(float) * (size_t)(2 * Lr * P + 2 * Lr * N);
}

// Per chunk (one CTA per (c, h, b)), both rank-Lr products of the chunk:
//   S_c[p][n] = sum_i exp(cum_end - cum_i) x_i[p] B_i[n]   (the chunk's own end state, K3)
//   D_c[p][n] = sum_i exp(cum_i) dy_i[p] C_i[n]             (its outputs' part of dL/dh_in(c))
// and the chunk's total log-decay cum_end.
template <typename T, int NQ>
__global__ void __launch_bounds__(kBwdThreads)
    bwd_chunk_state_kernel(GenericParams p, const float* __restrict__ dy,
                           float* __restrict__ dst) {
  extern __shared__ double bwd_ssm[];
  double* cum = bwd_ssm;                                        // [kBwdRows]
  const int l = (int)p.l, R = (int)p.R, P = (int)p.P, N = (int)p.N, Lr = l * R;
  float* sx = reinterpret_cast<float*>(cum + kBwdRows);        // [Lr][P]
  float* sdy = sx + Lr * P;                                     // [Lr][P]
  float* sB = sdy + Lr * P;                                     // [Lr][N]
  float* sC = sB + Lr * N;                                      // [Lr][N]
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int nv = bwd_steps(p, c), nvr = nv * R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bwd_cumsum(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, nv, cum);
  __syncthreads();
  const double cum_end = cum[l - 1];
  const int64_t row0 = (b * p.T + c * p.l) * R;
  const T* xs = static_cast<const T*>(p.x);
  const T* Bs = static_cast<const T*>(p.B);
  const T* Cs = static_cast<const T*>(p.C);
  for (int i = warp; i < Lr; i += kBwdWarps) {
    const bool real = i < nvr;
    const float wl = expf((float)(cum_end - cum[i / R])), we = expf((float)cum[i / R]);
    const int64_t xo = ((row0 + i) * p.H + h) * P, bo = ((row0 + i) * p.G + g) * N;
    for (int pp = lane; pp < P; pp += 32) {
      sx[i * P + pp] = real ? wl * ld_f32(xs + xo + pp) : 0.f;
      sdy[i * P + pp] = real ? we * __ldg(dy + xo + pp) : 0.f;
    }
    for (int n = lane; n < N; n += 32) {
      sB[i * N + n] = real ? ld_f32(Bs + bo + n) : 0.f;
      sC[i * N + n] = real ? ld_f32(Cs + bo + n) : 0.f;
    }
  }
  __syncthreads();
  const int t16 = threadIdx.x >> 4, l16 = threadIdx.x & 15;
  int pc[4], nc[NQ];
#pragma unroll
  for (int a = 0; a < 4; ++a) pc[a] = min(t16 + 16 * a, P - 1);
#pragma unroll
  for (int q = 0; q < NQ; ++q) nc[q] = min(l16 + 16 * q, N - 1);
  float as[4][NQ], ad[4][NQ];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int q = 0; q < NQ; ++q) as[a][q] = ad[a][q] = 0.f;
  for (int i = 0; i < Lr; ++i) {
    float xv[4], dv[4], bv[NQ], cv[NQ];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      xv[a] = sx[i * P + pc[a]];
      dv[a] = sdy[i * P + pc[a]];
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      bv[q] = sB[i * N + nc[q]];
      cv[q] = sC[i * N + nc[q]];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        as[a][q] = fmaf(xv[a], bv[q], as[a][q]);
        ad[a][q] = fmaf(dv[a], cv[q], ad[a][q]);
      }
  }
  const int64_t so = ((b * p.nch + c) * p.H + h) * (int64_t)P * N;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int pp = t16 + 16 * a;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int n = l16 + 16 * q;
      if (pp < P && n < N) {
        p.states[so + pp * N + n] = as[a][q];
        dst[so + pp * N + n] = ad[a][q];
      }
    }
  }
  if (threadIdx.x == 0) p.cend[(b * p.nch + c) * p.H + h] = (float)cum_end;
}

// Both carries across chunks, one thread per state element of one (b, h), loads kCarryAhead
// chunks ahead of the serial update:
//   forward  (K4): states[c] <- h_in(c),  h_in(c+1) = exp(cend_c) h_in(c) + S_c,  h_in(0) = init
//   backward:      dg[c] <- G_c = dL/dh_in(c+1),  dL/dh_in(c) = exp(cend_c) G_c + D_c,
//                  G_{nch-1} = dfinal, dinit = dL/dh_in(0).
constexpr int kCarryAhead = 16;

__global__ void __launch_bounds__(kBwdThreads, 2)
    bwd_carry_kernel(GenericParams p, const float* __restrict__ dfinal, float* __restrict__ dg,
                     float* __restrict__ dinit) {
  const int64_t PN = p.P * p.N;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.batch * p.H * PN) return;
  const int64_t bh = idx / PN, e = idx % PN;
  const int64_t b = bh / p.H, h = bh % p.H;
  const int64_t cs = p.H * PN;                        // chunk stride
  float* sp = p.states + (b * p.nch * p.H + h) * PN + e;
  float* gp = dg + (b * p.nch * p.H + h) * PN + e;
  const float* ce = p.cend + b * p.nch * p.H + h;
  float hv = p.init ? p.init[idx] : 0.f;
  for (int64_t c0 = 0; c0 < p.nch; c0 += kCarryAhead) {
    float sv[kCarryAhead], av[kCarryAhead];
#pragma unroll
    for (int k = 0; k < kCarryAhead; ++k)
      if (c0 + k < p.nch) {
        sv[k] = sp[(c0 + k) * cs];
        av[k] = ce[(c0 + k) * p.H];
      }
#pragma unroll
    for (int k = 0; k < kCarryAhead; ++k)
      if (c0 + k < p.nch) {
        sp[(c0 + k) * cs] = hv;
        hv = fmaf(expf(av[k]), hv, sv[k]);
      }
  }
  float gv = dfinal ? dfinal[idx] : 0.f;
  for (int64_t c1 = p.nch - 1; c1 >= 0; c1 -= kCarryAhead) {
    float dv[kCarryAhead], av[kCarryAhead];
#pragma unroll
    for (int k = 0; k < kCarryAhead; ++k)
      if (c1 - k >= 0) {
        dv[k] = gp[(c1 - k) * cs];
        av[k] = ce[(c1 - k) * p.H];
      }
#pragma unroll
    for (int k = 0; k < kCarryAhead; ++k)
      if (c1 - k >= 0) {
        gp[(c1 - k) * cs] = gv;
        gv = fmaf(expf(av[k]), gv, dv[k]);
      }
  }
  if (dinit) dinit[idx] = gv;
}

// Dynamic shared memory of bwd_chunk_grad_kernel: per-step prefix sums and four per-row double
// vectors, then x, dy [Lr][P+1], B, C [Lr][N+1], h_in, G [P][N+1] and M, A, W [Lr][Lr+1] (one
// float of padding per row keeps the column walks free of bank conflicts).
size_t bwd_grad_smem(int64_t Lr, int64_t P, int64_t N) {
  const size_t f = 2 * (size_t)(Lr * (P + 1)) + 2 * (size_t)(Lr * (N + 1)) +
                   2 * (size_t)(P * (N + 1)) + 3 * (size_t)(Lr * (Lr + 1));
  return (5 * kBwdRows + kBwdWarps) * sizeof(double) + f * sizeof(float);
}

// Sum over the 16 lanes of a half-warp (every lane of the warp takes part).
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Every gradient of one chunk (one CTA per (c, h, b)); dB and dC are added atomically (the heads
// of a group share them and were zeroed by the caller); dx and ddA are written for real steps.
// The per-row gradients are register-tiled products over the chunk's rows or the state:
//   dx = M^T dy + diag(el) B G^T,  dB = A^T C + diag(el) x G,  dC = A B + diag(e) dy h_in
// with M = L o CB, A = L o DX, el_j = exp(cum_end - cum_j), e_i = exp(cum_i).
template <typename T, int NQ>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_chunk_grad_kernel(GenericParams p, const float* __restrict__ dy,
                          const float* __restrict__ dg, float* __restrict__ dx,
                          float* __restrict__ ddA, float* __restrict__ dB,
                          float* __restrict__ dC) {
  extern __shared__ double bwd_gsm[];
  const int l = (int)p.l, R = (int)p.R, P = (int)p.P, N = (int)p.N, Lr = l * R;
  const int PS = P + 1, NS = N + 1, LS = Lr + 1;
  double* cum = bwd_gsm;               // [l] inclusive prefix sums of dA
  double* roww = cum + kBwdRows;       // [Lr] sum_j W_ij
  double* colw = roww + kBwdRows;      // [Lr] sum_i W_ij
  double* ein = colw + kBwdRows;       // [Lr] exp(cum_i) C_i . (h_in^T dy_i)
  double* qj = ein + kBwdRows;         // [Lr] exp(cum_end - cum_j) x_j . (G B_j)
  double* red = qj + kBwdRows;         // [kBwdWarps] partial sums of <G, h_in>
  float* sx = reinterpret_cast<float*>(red + kBwdWarps);
  float* sdy = sx + Lr * PS;
  float* sB = sdy + Lr * PS;
  float* sC = sB + Lr * NS;
  float* sH = sC + Lr * NS;
  float* sG = sH + P * NS;
  float* sM = sG + P * NS;             // L_ij CB_ij
  float* sA = sM + Lr * LS;            // L_ij DX_ij
  float* sW = sA + Lr * LS;            // L_ij CB_ij DX_ij

  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int nv = bwd_steps(p, c), nvr = nv * R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = (b * p.T + c * p.l) * R;
  const T* xs = static_cast<const T*>(p.x);
  const T* Bs = static_cast<const T*>(p.B);
  const T* Cs = static_cast<const T*>(p.C);

  bwd_cumsum(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, nv, cum);
  for (int i = warp; i < Lr; i += kBwdWarps) {
    const bool real = i < nvr;
    const int64_t xo = ((row0 + i) * p.H + h) * P, bo = ((row0 + i) * p.G + g) * N;
    for (int pp = lane; pp < P; pp += 32) {
      sx[i * PS + pp] = real ? ld_f32(xs + xo + pp) : 0.f;
      sdy[i * PS + pp] = real ? __ldg(dy + xo + pp) : 0.f;
    }
    for (int n = lane; n < N; n += 32) {
      sB[i * NS + n] = real ? ld_f32(Bs + bo + n) : 0.f;
      sC[i * NS + n] = real ? ld_f32(Cs + bo + n) : 0.f;
    }
  }
  const int64_t so = ((b * p.nch + c) * p.H + h) * (int64_t)P * N;
  for (int pp = warp; pp < P; pp += kBwdWarps) {
    for (int n = lane; n < N; n += 32) {
      sH[pp * NS + n] = p.states[so + pp * N + n];
      sG[pp * NS + n] = dg[so + pp * N + n];
    }
  }
  __syncthreads();

  const int t16 = threadIdx.x >> 4, l16 = threadIdx.x & 15;
  // Pairwise products: thread owns rows i = t16 + 16a and columns j = l16 + 16q of the chunk.
  {
    float cb[4][4], dx4[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < 4; ++q) cb[a][q] = dx4[a][q] = 0.f;
    int ri[4], cj[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      ri[a] = min(t16 + 16 * a, Lr - 1);
      cj[a] = min(l16 + 16 * a, Lr - 1);
    }
    for (int n = 0; n < N; ++n) {
      float cv[4], bv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        cv[a] = sC[ri[a] * NS + n];
        bv[a] = sB[cj[a] * NS + n];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) cb[a][q] = fmaf(cv[a], bv[q], cb[a][q]);
    }
    for (int pp = 0; pp < P; ++pp) {
      float dv[4], xv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        dv[a] = sdy[ri[a] * PS + pp];
        xv[a] = sx[cj[a] * PS + pp];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) dx4[a][q] = fmaf(dv[a], xv[q], dx4[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = t16 + 16 * a;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = l16 + 16 * q;
        if (i < Lr && j < Lr) {
          const int si = i / R, sj = j / R;
          const float L = sj <= si ? expf((float)(cum[si] - cum[sj])) : 0.f;
          const float m = L * cb[a][q];
          sM[i * LS + j] = m;
          sA[i * LS + j] = L * dx4[a][q];
          sW[i * LS + j] = m * dx4[a][q];
        }
      }
    }
  }
  __syncthreads();

  const double cum_end = cum[l - 1];
  if (threadIdx.x < Lr) {   // W row sums (four fp32 partials, then fp64)
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < Lr; ++j) s4[j & 3] += sW[threadIdx.x * LS + j];
    roww[threadIdx.x] = ((double)s4[0] + s4[1]) + ((double)s4[2] + s4[3]);
  } else if (threadIdx.x >= 128 && threadIdx.x < 128 + Lr) {   // W column sums
    const int j = threadIdx.x - 128;
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < Lr; ++i) s4[i & 3] += sW[i * LS + j];
    colw[j] = ((double)s4[0] + s4[1]) + ((double)s4[2] + s4[3]);
  }

  int rc[4];   // this thread's rows (clamped for loads)
#pragma unroll
  for (int a = 0; a < 4; ++a) rc[a] = min(t16 + 16 * a, Lr - 1);
  float el[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) el[a] = expf((float)(cum_end - cum[rc[a] / R]));

  // dx [Lr x P]: u = el_j (B G^T)_jp first (Q_j = x_j . u_j), then + (M^T dy)_jp.
  {
    int pc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) pc[q] = min(l16 + 16 * q, P - 1);
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[a][q] = 0.f;
    for (int n = 0; n < N; ++n) {
      float bv[4], gv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) bv[a] = sB[rc[a] * NS + n];
#pragma unroll
      for (int q = 0; q < 4; ++q) gv[q] = sG[pc[q] * NS + n];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(bv[a], gv[q], acc[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float qs = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[a][q] *= el[a];
        if (l16 + 16 * q < P) qs = fmaf(sx[rc[a] * PS + pc[q]], acc[a][q], qs);
      }
      qs = half_warp_sum(qs);
      if (l16 == 0 && t16 + 16 * a < Lr) qj[t16 + 16 * a] = (double)qs;
    }
    for (int i = (t16 / R) * R; i < Lr; ++i) {   // M_ij = 0 before row j's step
      float mv[4], dv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) mv[a] = sM[i * LS + rc[a]];
#pragma unroll
      for (int q = 0; q < 4; ++q) dv[q] = sdy[i * PS + pc[q]];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(mv[a], dv[q], acc[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = t16 + 16 * a;
      if (j < nvr) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int pp = l16 + 16 * q;
          if (pp < P) dx[((row0 + j) * p.H + h) * P + pp] = acc[a][q];
        }
      }
    }
  }

  int nc[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) nc[q] = min(l16 + 16 * q, N - 1);

  // dB [Lr x N]: el_j (x G)_jn, then + (A^T C)_jn.
  {
    float acc[4][NQ];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[a][q] = 0.f;
    for (int pp = 0; pp < P; ++pp) {
      float xv[4], gv[NQ];
#pragma unroll
      for (int a = 0; a < 4; ++a) xv[a] = sx[rc[a] * PS + pp];
#pragma unroll
      for (int q = 0; q < NQ; ++q) gv[q] = sG[pp * NS + nc[q]];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NQ; ++q) acc[a][q] = fmaf(xv[a], gv[q], acc[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[a][q] *= el[a];
    for (int i = (t16 / R) * R; i < Lr; ++i) {   // A_ij = 0 before row j's step
      float av[4], cv[NQ];
#pragma unroll
      for (int a = 0; a < 4; ++a) av[a] = sA[i * LS + rc[a]];
#pragma unroll
      for (int q = 0; q < NQ; ++q) cv[q] = sC[i * NS + nc[q]];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NQ; ++q) acc[a][q] = fmaf(av[a], cv[q], acc[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = t16 + 16 * a;
      if (j < nvr) {
        float* dst = dB + ((row0 + j) * p.G + g) * N;
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (l16 + 16 * q < N) atomicAdd(dst + l16 + 16 * q, acc[a][q]);
      }
    }
  }

  // dC [Lr x N]: e_i (dy h_in)_in first (E_i = C_i . that row), then + (A B)_in.
  {
    float acc[4][NQ];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[a][q] = 0.f;
    for (int pp = 0; pp < P; ++pp) {
      float dv[4], hv[NQ];
#pragma unroll
      for (int a = 0; a < 4; ++a) dv[a] = sdy[rc[a] * PS + pp];
#pragma unroll
      for (int q = 0; q < NQ; ++q) hv[q] = sH[pp * NS + nc[q]];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NQ; ++q) acc[a][q] = fmaf(dv[a], hv[q], acc[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float ei = expf((float)cum[rc[a] / R]);
      float es = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        acc[a][q] *= ei;
        if (l16 + 16 * q < N) es = fmaf(sC[rc[a] * NS + nc[q]], acc[a][q], es);
      }
      es = half_warp_sum(es);
      if (l16 == 0 && t16 + 16 * a < Lr) ein[t16 + 16 * a] = (double)es;
    }
    const int jend = min(Lr, (rc[3] / R + 1) * R);   // A_ij = 0 after row i's step
    for (int j = 0; j < jend; ++j) {
      float av[4], bv[NQ];
#pragma unroll
      for (int a = 0; a < 4; ++a) av[a] = sA[rc[a] * LS + j];
#pragma unroll
      for (int q = 0; q < NQ; ++q) bv[q] = sB[j * NS + nc[q]];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NQ; ++q) acc[a][q] = fmaf(av[a], bv[q], acc[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = t16 + 16 * a;
      if (i < nvr) {
        float* dst = dC + ((row0 + i) * p.G + g) * N;
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (l16 + 16 * q < N) atomicAdd(dst + l16 + 16 * q, acc[a][q]);
      }
    }
  }

  // <G, h_in>, for the chunk-end gradient of exp(cum_end) h_in.
  {
    float s = 0.f;
    for (int pp = warp; pp < P; pp += kBwdWarps)
      for (int n = lane; n < N; n += 32) s = fmaf(sG[pp * NS + n], sH[pp * NS + n], s);
    double d = (double)s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) red[warp] = d;
  }
  __syncthreads();

  // dL/dcum_s, then ddA_t = sum_{s >= t} dL/dcum_s over the chunk's steps.
  if (threadIdx.x == 0) {
    double gh = 0.0, qsum = 0.0;
    for (int w = 0; w < kBwdWarps; ++w) gh += red[w];
    for (int j = 0; j < Lr; ++j) qsum += qj[j];
    double suffix = qsum + exp(cum_end) * gh;   // the chunk-end terms, on the last step
    for (int s = l - 1; s >= 0; --s) {
      for (int r = 0; r < R; ++r) {
        const int i = s * R + r;
        suffix += roww[i] - colw[i] + ein[i] - qj[i];
      }
      if (s < nv) ddA[(b * p.T + c * p.l + s) * p.H + h] = (float)suffix;
    }
  }
}

// Fused rows per backward chunk: 64 / R steps of R rows.
int64_t bwd_chunk_steps(int64_t R) { return R >= kBwdRows ? 1 : kBwdRows / R; }

struct BwdLayout {
  size_t states = 0, cend = 0, dg = 0, total = 0;
};

ssd_status bwd_shape_status(const ssd_shape* s) {
  const ssd_status st = shape_status(s);
  if (st != SSD_OK) return st;
  if (s->has_theta != 0) return SSD_ERR_UNSUPPORTED;
  if (s->mimo_rank > kBwdRows || s->headdim > kBwdMaxP || s->dstate > kBwdMaxN)
    return SSD_ERR_UNSUPPORTED;
  const int64_t l = bwd_chunk_steps(s->mimo_rank), Lr = l * s->mimo_rank;
  const size_t lim = 227 * 1024;
  if (bwd_grad_smem(Lr, s->headdim, s->dstate) > lim ||
      bwd_state_smem(Lr, s->headdim, s->dstate) > lim)
    return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

BwdLayout bwd_layout(const ssd_shape* s) {
  const int64_t l = bwd_chunk_steps(s->mimo_rank);
  const int64_t nch = (s->seqlen + l - 1) / l;
  const size_t st = sizeof(float) * (size_t)(s->batch * nch * s->nheads * s->headdim * s->dstate);
  BwdLayout L;
  size_t off = sizeof(WsHeader);
  L.states = off;
  off = align_up(off + st, kWsAlign);
  L.cend = off;
  off = align_up(off + sizeof(float) * (size_t)(s->batch * nch * s->nheads), kWsAlign);
  L.dg = off;
  off = align_up(off + st, kWsAlign);
  L.total = off;
  return L;
}

bool al16_or_null(const void* q) { return q == nullptr || aligned16(q); }

template <typename T, int NQ>
cudaError_t bwd_launch_nq(const GenericParams& p, const float* dy, const float* dfinal,
                          float* dx, float* ddA, float* dB, float* dC, float* dinit, float* dg,
                          cudaStream_t st) {
  const int64_t Lr = p.l * p.R;
  const dim3 grid((unsigned)p.nch, (unsigned)p.H, (unsigned)p.batch);
  const size_t s1 = bwd_state_smem(Lr, p.P, p.N);
  cudaError_t e = cudaFuncSetAttribute(bwd_chunk_state_kernel<T, NQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e != cudaSuccess) return e;
  bwd_chunk_state_kernel<T, NQ><<<grid, kBwdThreads, s1, st>>>(p, dy, dg);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n = p.batch * p.H * p.P * p.N;
  bwd_carry_kernel<<<(unsigned)((n + kBwdThreads - 1) / kBwdThreads), kBwdThreads, 0, st>>>(
      p, dfinal, dg, dinit);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t s2 = bwd_grad_smem(Lr, p.P, p.N);
  e = cudaFuncSetAttribute(bwd_chunk_grad_kernel<T, NQ>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
  if (e != cudaSuccess) return e;
  bwd_chunk_grad_kernel<T, NQ><<<grid, kBwdThreads, s2, st>>>(p, dy, dg, dx, ddA, dB, dC);
  return cudaGetLastError();
}

// Column tiles of 16 state dims: N <= 16, 32, 64 or 128.
template <typename T>
cudaError_t bwd_launch(const GenericParams& p, const float* dy, const float* dfinal, float* dx,
                       float* ddA, float* dB, float* dC, float* dinit, float* dg,
                       cudaStream_t st) {
  if (p.N <= 16) return bwd_launch_nq<T, 1>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, st);
  if (p.N <= 32) return bwd_launch_nq<T, 2>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, st);
  if (p.N <= 64) return bwd_launch_nq<T, 4>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, st);
  return bwd_launch_nq<T, 8>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, st);
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_backward_workspace_bytes(const ssd_shape* shape) {
  if (bwd_shape_status(shape) != SSD_OK) return 0;
  return bwd_layout(shape).total;
}

ssd_status ssd_chunked_backward(const ssd_shape* shape, const void* x, const float* dA,
                                const void* B, const void* C, const float* init_state,
                                const float* dy, const float* dfinal, float* dx, float* ddA,
                                float* dB, float* dC, float* dinit, void* workspace,
                                size_t workspace_bytes, void* stream) {
  const ssd_status vs = bwd_shape_status(shape);
  if (vs != SSD_OK) return vs;
  if (!x || !dA || !B || !C || !dy || !dx || !ddA || !dB || !dC) return SSD_ERR_INVALID_ARG;
  const void* ptrs[] = {x, dA, B, C, init_state, dy, dfinal, dx, ddA, dB, dC, dinit};
  for (const void* q : ptrs)
    if (!al16_or_null(q)) return SSD_ERR_INVALID_ARG;
  const BwdLayout lay = bwd_layout(shape);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0 ||
      workspace_bytes < lay.total)
    return SSD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = shape->io_dtype == SSD_BF16;

  GenericParams p;
  memset(&p, 0, sizeof(p));
  p.x = x;
  p.dA = dA;
  p.B = B;
  p.C = C;
  p.init = init_state;
  p.batch = shape->batch;
  p.T = shape->seqlen;
  p.H = shape->nheads;
  p.P = shape->headdim;
  p.N = shape->dstate;
  p.G = shape->ngroups;
  p.R = shape->mimo_rank;
  p.l = bwd_chunk_steps(p.R);
  p.nch = (p.T + p.l - 1) / p.l;
  p.states = reinterpret_cast<float*>(ws + lay.states);
  p.cend = reinterpret_cast<float*>(ws + lay.cend);
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  float* dg = reinterpret_cast<float*>(ws + lay.dg);

  const size_t bc = sizeof(float) * (size_t)(p.batch * p.T * p.R * p.G * p.N);
  if (cudaMemsetAsync(dB, 0, bc, st) != cudaSuccess || cudaMemsetAsync(dC, 0, bc, st) != cudaSuccess)
    return SSD_ERR_CUDA;
  const cudaError_t e =
      bf16 ? bwd_launch<__nv_bfloat16>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, st)
           : bwd_launch<float>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, st);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
