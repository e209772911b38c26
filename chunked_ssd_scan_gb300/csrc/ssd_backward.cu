// Backward of the chunked SSD forward (unrotated; CUDA-core fp32), recompute per chunk.
//
// The scan.py page asks for a scan that can train; the moments.rs page's memory model keeps only
// the chunk-boundary states and recomputes inside a chunk.  Here:
//   1. generic_states: the forward chunk-input states h_in(c) (K1, K3, K4; no y), 64 fused rows
//      per chunk;
//   2. bwd_dstate_kernel: per chunk D_c = sum_i exp(cum_i) dy_i (outer) C_i, the part of
//      dL/dh_in(c) that the chunk's own outputs contribute;
//   3. bwd_state_pass_kernel: the reverse of K4 across chunks, G_c = dL/dh_out(c) = dL/dh_in(c+1),
//      G_{nch-1} = dfinal, dL/dh_in(c) = exp(cum_end(c)) G_c + D_c, dinit = dL/dh_in(0);
//   4. bwd_chunk_grad_kernel: per chunk, with L_ij = exp(cum_i - cum_j) below the step diagonal,
//      CB_ij = C_i . B_j and DX_ij = dy_i . x_j:
//        dx_j = sum_i L_ij CB_ij dy_i + exp(cum_end - cum_j) G B_j
//        dB_j = sum_i L_ij DX_ij C_i + exp(cum_end - cum_j) G^T x_j
//        dC_i = sum_j L_ij DX_ij B_j + exp(cum_i) h_in^T dy_i
//      and the gradient of every prefix sum cum_s (from L, exp(cum_i), exp(cum_end - cum_j) and
//      exp(cum_end) h_in), whose suffix sums over the chunk's steps are ddA.
// Rows are rank-fused (i = t R + r, step i / R); dB and dC add over the heads of a group.
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

// Dynamic shared memory of bwd_dstate_kernel: prefix sums, dy rows [Lr][P], C rows [Lr][N].
size_t bwd_dstate_smem(int64_t Lr, int64_t P, int64_t N) {
  return kBwdRows * sizeof(double) + sizeof(float) * (size_t)(Lr * P + Lr * N);
}

// D_c[p][n] = sum_i exp(cum_{i/R}) dy_i[p] C_i[n], written to dst (one CTA per (c, h, b)).
template <typename T>
__global__ void __launch_bounds__(kBwdThreads)
    bwd_dstate_kernel(GenericParams p, const float* __restrict__ dy, float* __restrict__ dst) {
  extern __shared__ double bwd_dsm[];
  double* cum = bwd_dsm;                                       // [kBwdRows]
  const int l = (int)p.l, R = (int)p.R, P = (int)p.P, N = (int)p.N, Lr = l * R;
  float* sdy = reinterpret_cast<float*>(cum + kBwdRows);      // [Lr][P]
  float* sc = sdy + Lr * P;                                    // [Lr][N]
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int nv = bwd_steps(p, c), nvr = nv * R;
  bwd_cumsum(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, nv, cum);
  const int64_t row0 = (b * p.T + c * p.l) * R;
  const T* C = static_cast<const T*>(p.C);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < Lr; i += kBwdWarps) {
    const float* src = dy + ((row0 + i) * p.H + h) * P;
    for (int pp = lane; pp < P; pp += 32) sdy[i * P + pp] = i < nvr ? src[pp] : 0.f;
    const T* cs = C + ((row0 + i) * p.G + g) * N;
    for (int n = lane; n < N; n += 32) sc[i * N + n] = i < nvr ? ld_f32(cs + n) : 0.f;
  }
  __syncthreads();
  for (int i = warp; i < Lr; i += kBwdWarps) {   // fold exp(cum) into the dy rows
    const float w = expf((float)cum[i / R]);
    for (int pp = lane; pp < P; pp += 32) sdy[i * P + pp] *= w;
  }
  __syncthreads();
  float* out = dst + ((b * p.nch + c) * p.H + h) * (int64_t)P * N;
  for (int o = threadIdx.x; o < P * N; o += kBwdThreads) {
    const int pp = o / N, n = o % N;
    float s = 0.f;
    for (int i = 0; i < Lr; ++i) s = fmaf(sdy[i * P + pp], sc[i * N + n], s);
    out[o] = s;
  }
}

// Reverse K4, one thread per state element of one (b, h): G_c = dL/dh_out(c) replaces D_c in
// place; dinit = dL/dh_in(0).
__global__ void __launch_bounds__(kBwdThreads)
    bwd_state_pass_kernel(GenericParams p, const float* __restrict__ dfinal,
                          float* __restrict__ dg, float* __restrict__ dinit) {
  const int64_t PN = p.P * p.N;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.batch * p.H * PN) return;
  const int64_t bh = idx / PN, e = idx % PN;
  const int64_t b = bh / p.H, h = bh % p.H;
  float g = dfinal ? dfinal[idx] : 0.f;
  for (int64_t c = p.nch - 1; c >= 0; --c) {
    float* slot = dg + ((b * p.nch + c) * p.H + h) * PN + e;
    const float d = *slot;
    *slot = g;                                              // G_c
    g = fmaf(expf(p.cend[(b * p.nch + c) * p.H + h]), g, d);   // dL/dh_in(c)
  }
  if (dinit) dinit[idx] = g;
}

// Dynamic shared memory of bwd_chunk_grad_kernel: per-step prefix sums and four per-row double
// vectors, then x, dy [Lr][P+1], B, C [Lr][N+1], h_in, G [P][N+1] and M, A, W [Lr][Lr+1] (one
// float of padding per row keeps the column walks free of bank conflicts).
size_t bwd_grad_smem(int64_t Lr, int64_t P, int64_t N) {
  const size_t f = 2 * (size_t)(Lr * (P + 1)) + 2 * (size_t)(Lr * (N + 1)) +
                   2 * (size_t)(P * (N + 1)) + 3 * (size_t)(Lr * (Lr + 1));
  return (5 * kBwdRows + kBwdWarps) * sizeof(double) + f * sizeof(float);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Every gradient of one chunk (one CTA per (c, h, b)); dB and dC are added atomically (the heads
// of a group share them and were zeroed by the caller); dx and ddA are written for real steps.
template <typename T>
__global__ void __launch_bounds__(kBwdThreads)
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
  for (int e = threadIdx.x; e < P * N; e += kBwdThreads) {
    const int pp = e / N, n = e % N;
    sH[pp * NS + n] = p.states[so + e];
    sG[pp * NS + n] = dg[so + e];
  }
  __syncthreads();

  // Pairwise products: thread (ty, tx) owns rows i = ty + 16a and columns j = tx + 16b.
  {
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    float cb[4][4], dx4[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < 4; ++q) cb[a][q] = dx4[a][q] = 0.f;
    int ri[4], cj[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      ri[a] = min(ty + 16 * a, Lr - 1);
      cj[a] = min(tx + 16 * a, Lr - 1);
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
      const int i = ty + 16 * a;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = tx + 16 * q;
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
  if (threadIdx.x < Lr) {   // W row sums
    double s = 0.0;
    for (int j = 0; j < Lr; ++j) s += (double)sW[threadIdx.x * LS + j];
    roww[threadIdx.x] = s;
  } else if (threadIdx.x >= 128 && threadIdx.x < 128 + Lr) {   // W column sums
    const int j = threadIdx.x - 128;
    double s = 0.0;
    for (int i = 0; i < Lr; ++i) s += (double)sW[i * LS + j];
    colw[j] = s;
  }

  // dx_j = sum_i M_ij dy_i + u_j with u_j = exp(cum_end - cum_j) G B_j; Q_j = x_j . u_j.
  for (int j = warp; j < Lr; j += kBwdWarps) {
    const int sj = j / R;
    const float el = expf((float)(cum_end - cum[sj]));
    float acc[2] = {0.f, 0.f}, u[2] = {0.f, 0.f};
    for (int i = sj * R; i < Lr; ++i) {
      const float m = sM[i * LS + j];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int pp = lane + 32 * k;
        if (pp < P) acc[k] = fmaf(m, sdy[i * PS + pp], acc[k]);
      }
    }
    for (int n = 0; n < N; ++n) {
      const float bv = sB[j * NS + n];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int pp = lane + 32 * k;
        if (pp < P) u[k] = fmaf(sG[pp * NS + n], bv, u[k]);
      }
    }
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int pp = lane + 32 * k;
      if (pp < P) {
        u[k] *= el;
        q = fmaf(sx[j * PS + pp], u[k], q);
        if (j < nvr) dx[((row0 + j) * p.H + h) * P + pp] = acc[k] + u[k];
      }
    }
    q = warp_sum(q);
    if (lane == 0) qj[j] = (double)q;
  }

  // dB_j = sum_i A_ij C_i + exp(cum_end - cum_j) G^T x_j.
  for (int j = warp; j < Lr; j += kBwdWarps) {
    const int sj = j / R;
    const float el = expf((float)(cum_end - cum[sj]));
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, v[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = sj * R; i < Lr; ++i) {
      const float a = sA[i * LS + j];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = lane + 32 * k;
        if (n < N) acc[k] = fmaf(a, sC[i * NS + n], acc[k]);
      }
    }
    for (int pp = 0; pp < P; ++pp) {
      const float xv = sx[j * PS + pp];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = lane + 32 * k;
        if (n < N) v[k] = fmaf(sG[pp * NS + n], xv, v[k]);
      }
    }
    if (j < nvr) {
      float* dst = dB + ((row0 + j) * p.G + g) * N;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = lane + 32 * k;
        if (n < N) atomicAdd(dst + n, fmaf(el, v[k], acc[k]));
      }
    }
  }

  // dC_i = sum_j A_ij B_j + exp(cum_i) h_in^T dy_i; E_i = exp(cum_i) C_i . (h_in^T dy_i).
  for (int i = warp; i < Lr; i += kBwdWarps) {
    const int si = i / R, jend = (si + 1) * R;
    const float ei = expf((float)cum[si]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, v[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < jend; ++j) {
      const float a = sA[i * LS + j];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = lane + 32 * k;
        if (n < N) acc[k] = fmaf(a, sB[j * NS + n], acc[k]);
      }
    }
    for (int pp = 0; pp < P; ++pp) {
      const float dv = sdy[i * PS + pp];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = lane + 32 * k;
        if (n < N) v[k] = fmaf(sH[pp * NS + n], dv, v[k]);
      }
    }
    float e = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int n = lane + 32 * k;
      if (n < N) {
        v[k] *= ei;
        e = fmaf(sC[i * NS + n], v[k], e);
      }
    }
    if (i < nvr) {
      float* dst = dC + ((row0 + i) * p.G + g) * N;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = lane + 32 * k;
        if (n < N) atomicAdd(dst + n, acc[k] + v[k]);
      }
    }
    e = warp_sum(e);
    if (lane == 0) ein[i] = (double)e;
  }

  // <G, h_in>, for the chunk-end gradient of exp(cum_end) h_in.
  {
    double s = 0.0;
    for (int e = threadIdx.x; e < P * N; e += kBwdThreads) {
      const int pp = e / N, n = e % N;
      s += (double)sG[pp * NS + n] * (double)sH[pp * NS + n];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) red[warp] = s;
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
      bwd_dstate_smem(Lr, s->headdim, s->dstate) > lim ||
      !generic_supported(l, s->mimo_rank, s->headdim, s->dstate, false))
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

template <typename T>
cudaError_t bwd_launch(const GenericParams& p, const float* dy, const float* dfinal, float* dx,
                       float* ddA, float* dB, float* dC, float* dinit, float* dg,
                       cudaStream_t st) {
  const int64_t Lr = p.l * p.R;
  const dim3 grid((unsigned)p.nch, (unsigned)p.H, (unsigned)p.batch);
  const size_t s1 = bwd_dstate_smem(Lr, p.P, p.N);
  cudaError_t e = cudaFuncSetAttribute(bwd_dstate_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e != cudaSuccess) return e;
  bwd_dstate_kernel<T><<<grid, kBwdThreads, s1, st>>>(p, dy, dg);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n = p.batch * p.H * p.P * p.N;
  bwd_state_pass_kernel<<<(unsigned)((n + kBwdThreads - 1) / kBwdThreads), kBwdThreads, 0, st>>>(
      p, dfinal, dg, dinit);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t s2 = bwd_grad_smem(Lr, p.P, p.N);
  e = cudaFuncSetAttribute(bwd_chunk_grad_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)s2);
  if (e != cudaSuccess) return e;
  bwd_chunk_grad_kernel<T><<<grid, kBwdThreads, s2, st>>>(p, dy, dg, dx, ddA, dB, dC);
  return cudaGetLastError();
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
  if (generic_states(p, bf16, st) != cudaSuccess) return SSD_ERR_CUDA;
  const cudaError_t e =
      bf16 ? bwd_launch<__nv_bfloat16>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, st)
           : bwd_launch<float>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, st);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
