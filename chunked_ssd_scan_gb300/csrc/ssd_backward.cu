// Backward of the chunked SSD forward (CUDA-core fp32), recompute per chunk.
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
// group.  With the rotation the same three kernels run in chunk-local frames (the rotation
// section below), around angle, staging and chain-rule kernels.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kBwdThreads = 256, kBwdWarps = kBwdThreads / 32;
constexpr int kBwdRows = 64;   // fused rows per chunk
constexpr int kBwdMaxP = 64, kBwdMaxN = 128;
constexpr int kRowsPerWarp = kBwdRows / kBwdWarps;

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

// Column tiles of the state axis: NQ values per thread, as HH runs of VW consecutive columns
// (n = VW l16 + r + 16 VW hh for lane l16 of a half-warp), so one shared-memory load moves VW
// floats and a half-warp reads 16 VW consecutive floats of a row.
template <int NQ>
struct ColTile {
  static constexpr int VW = NQ < 4 ? NQ : 4;
  static constexpr int HH = NQ / VW;
};

template <int V>
__device__ __forceinline__ void lds_vec(const float* src, float* out) {
  if constexpr (V == 4) {
    const float4 v = *reinterpret_cast<const float4*>(src);
    out[0] = v.x;
    out[1] = v.y;
    out[2] = v.z;
    out[3] = v.w;
  } else if constexpr (V == 2) {
    const float2 v = *reinterpret_cast<const float2*>(src);
    out[0] = v.x;
    out[1] = v.y;
  } else {
    out[0] = *src;
  }
}

template <int V>
__device__ __forceinline__ void atomic_add_vec(float* dst, const float* v) {
  if constexpr (V == 4) {
    atomicAdd(reinterpret_cast<float4*>(dst), make_float4(v[0], v[1], v[2], v[3]));
  } else if constexpr (V == 2) {
    atomicAdd(reinterpret_cast<float2*>(dst), make_float2(v[0], v[1]));
  } else {
    atomicAdd(dst, v[0]);
  }
}

template <int V>
__device__ __forceinline__ void st_vec(float* dst, const float* v) {
  if constexpr (V == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  } else if constexpr (V == 2) {
    *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
  } else {
    *dst = v[0];
  }
}

// First column of run hh of lane l16, clamped so the loaded run stays inside the row (columns
// past N are masked by the caller).
template <int NQ>
__device__ __forceinline__ int col0(int l16, int hh, int NR) {
  constexpr int VW = ColTile<NQ>::VW;
  return min(VW * l16 + 16 * VW * hh, NR - VW);
}

__host__ __device__ inline int round4(int v) { return (v + 3) & ~3; }

// Dynamic shared memory of bwd_chunk_state_kernel: the prefix sums, then the scaled x and dy rows
// [Lr][P4] and the B and C rows [Lr][N4] (P4, N4: P, N rounded up to 4, zero-padded).
size_t bwd_state_smem(int64_t Lr, int64_t P, int64_t N) {
  return kBwdRows * sizeof(double) +
         sizeof(float) * (size_t)(2 * Lr * round4((int)P) + 2 * Lr * round4((int)N));
}

// Per chunk (one CTA per (c, h, b)), both rank-Lr products of the chunk:
//   S_c[p][n] = sum_i exp(cum_end - cum_i) x_i[p] B_i[n]   (the chunk's own end state, K3)
//   D_c[p][n] = sum_i exp(cum_i) dy_i[p] C_i[n]             (its outputs' part of dL/dh_in(c))
// and the chunk's total log-decay cum_end.  Thread (t16, l16) owns rows p = 4 t16 + a and the
// column tile of l16.
template <typename TX, typename TBC, int NQ>
__global__ void __launch_bounds__(kBwdThreads, 2)
    bwd_chunk_state_kernel(GenericParams p, const float* __restrict__ dy,
                           float* __restrict__ dst) {
  constexpr int VW = ColTile<NQ>::VW, HH = ColTile<NQ>::HH;
  extern __shared__ double bwd_ssm[];
  double* cum = bwd_ssm;                                        // [kBwdRows]
  const int l = (int)p.l, R = (int)p.R, P = (int)p.P, N = (int)p.N, Lr = l * R;
  const int P4 = round4(P), N4 = round4(N);
  float* sx = reinterpret_cast<float*>(cum + kBwdRows);        // [Lr][P4]
  float* sdy = sx + Lr * P4;                                    // [Lr][P4]
  float* sB = sdy + Lr * P4;                                    // [Lr][N4]
  float* sC = sB + Lr * N4;                                     // [Lr][N4]
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int nv = bwd_steps(p, c), nvr = nv * R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = (b * p.T + c * p.l) * R;
  const TX* xs = static_cast<const TX*>(p.x);
  const TBC* Bs = static_cast<const TBC*>(p.B);
  const TBC* Cs = static_cast<const TBC*>(p.C);
  {
    // each warp stages its 8 rows i = warp + 8 k: every global load first (before the prefix
    // sums are waited for), then the scaled stores
    float xr[kRowsPerWarp][2], dr[kRowsPerWarp][2], br[kRowsPerWarp][4], cr[kRowsPerWarp][4];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int i = warp + kBwdWarps * k;
      const bool real = i < nvr;
      const int64_t xo = ((row0 + i) * p.H + h) * P, bo = ((row0 + i) * p.G + g) * N;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int pp = lane + 32 * u;
        const bool v = real && pp < P;
        xr[k][u] = v ? ld_f32(xs + xo + pp) : 0.f;
        dr[k][u] = v ? __ldg(dy + xo + pp) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int n = lane + 32 * u;
        const bool v = real && n < N;
        br[k][u] = v ? ld_f32(Bs + bo + n) : 0.f;
        cr[k][u] = v ? ld_f32(Cs + bo + n) : 0.f;
      }
    }
    bwd_cumsum(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, nv, cum);
    __syncthreads();
    const double cum_end = cum[l - 1];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int i = warp + kBwdWarps * k;
      if (i >= Lr) continue;
      const float wl = expf((float)(cum_end - cum[i / R])), we = expf((float)cum[i / R]);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int pp = lane + 32 * u;
        if (pp < P4) {
          sx[i * P4 + pp] = wl * xr[k][u];
          sdy[i * P4 + pp] = we * dr[k][u];
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int n = lane + 32 * u;
        if (n < N4) {
          sB[i * N4 + n] = br[k][u];
          sC[i * N4 + n] = cr[k][u];
        }
      }
    }
  }
  __syncthreads();
  const int t16 = threadIdx.x >> 4, l16 = threadIdx.x & 15;
  const int p0 = min(4 * t16, P4 - 4);
  int n0[HH];
#pragma unroll
  for (int hh = 0; hh < HH; ++hh) n0[hh] = col0<NQ>(l16, hh, N4);
  float as[4][NQ], ad[4][NQ];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int q = 0; q < NQ; ++q) as[a][q] = ad[a][q] = 0.f;
  for (int i = 0; i < Lr; ++i) {
    float xv[4], dv[4], bv[NQ], cv[NQ];
    lds_vec<4>(sx + i * P4 + p0, xv);
    lds_vec<4>(sdy + i * P4 + p0, dv);
#pragma unroll
    for (int hh = 0; hh < HH; ++hh) {
      lds_vec<VW>(sB + i * N4 + n0[hh], bv + hh * VW);
      lds_vec<VW>(sC + i * N4 + n0[hh], cv + hh * VW);
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
    const int pp = p0 + a;
    if (pp >= P || p0 != 4 * t16) continue;
#pragma unroll
    for (int hh = 0; hh < HH; ++hh) {
      const int n = n0[hh];
      if (n != VW * l16 + 16 * VW * hh || n >= N) continue;   // a clamped (duplicate) run
      st_vec<VW>(p.states + so + pp * N + n, as[a] + hh * VW);
      st_vec<VW>(dst + so + pp * N + n, ad[a] + hh * VW);
    }
  }
  if (threadIdx.x == 0) p.cend[(b * p.nch + c) * p.H + h] = (float)cum[l - 1];
}

// The carries across chunks, one thread per state element of one (b, h) and direction (the
// first b H P N threads forward, the rest backward), loading kCarryAhead chunks ahead of the
// serial update:
//   forward  (K4): states[c] <- h_in(c),  h_in(c+1) = exp(cend_c) h_in(c) + S_c,  h_in(0) = init,
//                  gfin <- the final state (when asked for)
//   backward:      dg[c] <- G_c = dL/dh_in(c+1),  dL/dh_in(c) = exp(cend_c) G_c + D_c,
//                  G_{nch-1} = dfinal, dinit = dL/dh_in(0).
constexpr int kCarryAhead = 16;

__global__ void __launch_bounds__(kBwdThreads)
    bwd_carry_kernel(GenericParams p, const float* __restrict__ dfinal, float* __restrict__ dg,
                     float* __restrict__ dinit, float* __restrict__ gfin) {
  const int64_t PN = p.P * p.N, n_el = p.batch * p.H * PN;
  int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= 2 * n_el) return;
  const bool back = idx >= n_el;
  if (back) idx -= n_el;
  const int64_t bh = idx / PN, e = idx % PN;
  const int64_t b = bh / p.H, h = bh % p.H;
  const int64_t cs = p.H * PN;                        // chunk stride
  float* vp = (back ? dg : p.states) + (b * p.nch * p.H + h) * PN + e;
  const float* ce = p.cend + b * p.nch * p.H + h;
  float v = back ? (dfinal ? dfinal[idx] : 0.f) : (p.init ? p.init[idx] : 0.f);
  for (int64_t k0 = 0; k0 < p.nch; k0 += kCarryAhead) {
    float sv[kCarryAhead], av[kCarryAhead];
#pragma unroll
    for (int k = 0; k < kCarryAhead; ++k)
      if (k0 + k < p.nch) {
        const int64_t c = back ? p.nch - 1 - (k0 + k) : k0 + k;
        sv[k] = vp[c * cs];
        av[k] = ce[c * p.H];
      }
#pragma unroll
    for (int k = 0; k < kCarryAhead; ++k)
      if (k0 + k < p.nch) {
        const int64_t c = back ? p.nch - 1 - (k0 + k) : k0 + k;
        vp[c * cs] = v;
        v = fmaf(expf(av[k]), v, sv[k]);
      }
  }
  if (back && dinit) dinit[idx] = v;
  if (!back && gfin) gfin[idx] = v;   // the state after the last chunk
}

// Shared-memory row strides of bwd_chunk_grad_kernel: the row length rounded up to 4 plus 4, so
// rows start 16-byte aligned and the 8 lanes of a 16-byte load phase that read 8 different rows
// hit 8 different bank groups.
__host__ __device__ inline int bwd_stride(int len) { return round4(len) + 4; }

// Dynamic shared memory of bwd_chunk_grad_kernel: per-step prefix sums, four per-row double
// vectors and the warp partials of <G, h_in>, the warps' partial column sums of W, then x, dy
// [Lr][P], B, C [Lr][N], h_in, G [P][N] and M, A [Lr][Lr] at the strides above.
size_t bwd_grad_smem(int64_t Lr, int64_t P, int64_t N) {
  const size_t PS = bwd_stride((int)P), NS = bwd_stride((int)N), LS = bwd_stride((int)Lr);
  const size_t f = kBwdWarps * kBwdRows + 2 * (size_t)Lr * PS + 2 * (size_t)Lr * NS +
                   2 * (size_t)P * NS + 2 * (size_t)Lr * LS;
  return (5 * kBwdRows + kBwdWarps) * sizeof(double) + f * sizeof(float);
}

// Sum over the 16 lanes of a half-warp (every lane of the warp takes part).
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// acc[a][q] += sum_k U[ri[a]][k] V[cj[q]][k] over the row length K4 (rows at stride S, read 4 k at
// a time).  With kTri the blocks q > a (entirely above the step diagonal) are skipped.
template <bool kTri>
__device__ __forceinline__ void pair_products(const float* U, const float* V, int S, int K4,
                                              const int (&ri)[4], const int (&cj)[4],
                                              float (&acc)[4][4]) {
  for (int k0 = 0; k0 < K4; k0 += 4) {
    float uv[4][4], vv[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      lds_vec<4>(U + ri[a] * S + k0, uv[a]);
      lds_vec<4>(V + cj[a] * S + k0, vv[a]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (!kTri || q <= a) acc[a][q] = fmaf(uv[a][k], vv[q][k], acc[a][q]);
  }
}

// Every gradient of one chunk (one CTA per (c, h, b)); dB and dC are added atomically (the heads
// of a group share them and were zeroed by the caller); dx and ddA are written for real steps.
// The per-row gradients are register-tiled products over the chunk's rows or the state:
//   dx = M^T dy + diag(el) B G^T,  dB = A^T C + diag(el) x G,  dC = A B + diag(e) dy h_in
// with M = L o CB, A = L o DX, el_j = exp(cum_end - cum_j), e_i = exp(cum_i).  Thread
// (t16, l16) owns output rows 4 t16 + a (a < 4) and, along P, columns l16 + 16 q, along N the
// column tile of l16 (ColTile); products whose reduction runs along a row load 4 k at a time.
template <typename TX, typename TBC, int NQ>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_chunk_grad_kernel(GenericParams p, const float* __restrict__ dy,
                          const float* __restrict__ dg, float* __restrict__ dx,
                          float* __restrict__ ddA, float* __restrict__ dB,
                          float* __restrict__ dC) {
  constexpr int VW = ColTile<NQ>::VW, HH = ColTile<NQ>::HH;
  extern __shared__ double bwd_gsm[];
  const int l = (int)p.l, R = (int)p.R, P = (int)p.P, N = (int)p.N, Lr = l * R;
  const int P4 = round4(P), N4 = round4(N);
  const int PS = bwd_stride(P), NS = bwd_stride(N), LS = bwd_stride(Lr);
  double* cum = bwd_gsm;               // [l] inclusive prefix sums of dA
  double* roww = cum + kBwdRows;       // [Lr] sum_j W_ij, W = M o DX
  double* colw = roww + kBwdRows;      // [Lr] sum_i W_ij
  double* ein = colw + kBwdRows;       // [Lr] exp(cum_i) C_i . (h_in^T dy_i)
  double* qj = ein + kBwdRows;         // [Lr] exp(cum_end - cum_j) x_j . (G B_j)
  double* red = qj + kBwdRows;         // [kBwdWarps] partial sums of <G, h_in>
  float* colp = reinterpret_cast<float*>(red + kBwdWarps);   // [kBwdWarps][kBwdRows]
  float* sx = colp + kBwdWarps * kBwdRows;
  float* sdy = sx + Lr * PS;
  float* sB = sdy + Lr * PS;
  float* sC = sB + Lr * NS;
  float* sH = sC + Lr * NS;
  float* sG = sH + P * NS;
  float* sM = sG + P * NS;             // L_ij CB_ij
  float* sA = sM + Lr * LS;            // L_ij DX_ij

  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (p.H / p.G);
  const int nv = bwd_steps(p, c), nvr = nv * R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = (b * p.T + c * p.l) * R;
  const TX* xs = static_cast<const TX*>(p.x);
  const TBC* Bs = static_cast<const TBC*>(p.B);
  const TBC* Cs = static_cast<const TBC*>(p.C);

  bwd_cumsum(p.dA + (b * p.T + c * p.l) * p.H + h, p.H, l, nv, cum);
  // Rows first (group 0: dy by async copy), then h_in and G (group 1), which are needed only
  // after the pairwise products and land while those are computed.  Pads are zeroed.
  {
    // each warp stages its 8 rows i = warp + 8 k: every global load first, then the stores
    float xr[kRowsPerWarp][2], br[kRowsPerWarp][4], cr[kRowsPerWarp][4];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int i = warp + kBwdWarps * k;
      const bool real = i < nvr;
      const int64_t xo = ((row0 + i) * p.H + h) * P, bo = ((row0 + i) * p.G + g) * N;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int pp = lane + 32 * u;
        const bool v = real && pp < P;
        xr[k][u] = v ? ld_f32(xs + xo + pp) : 0.f;
        if (v) cp_async4(sdy + i * PS + pp, dy + xo + pp);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int n = lane + 32 * u;
        const bool v = real && n < N;
        br[k][u] = v ? ld_f32(Bs + bo + n) : 0.f;
        cr[k][u] = v ? ld_f32(Cs + bo + n) : 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int i = warp + kBwdWarps * k;
      if (i >= Lr) continue;
      const bool real = i < nvr;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int pp = lane + 32 * u;
        if (pp < P4) {
          sx[i * PS + pp] = xr[k][u];
          if (!(real && pp < P)) sdy[i * PS + pp] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int n = lane + 32 * u;
        if (n < N4) {
          sB[i * NS + n] = br[k][u];
          sC[i * NS + n] = cr[k][u];
        }
      }
      for (int j = Lr + lane; j < LS; j += 32) {   // M and A past the chunk's rows read as zero
        sM[i * LS + j] = 0.f;
        sA[i * LS + j] = 0.f;
      }
    }
  }
  cp_async_commit();
  const int64_t so = ((b * p.nch + c) * p.H + h) * (int64_t)P * N;
  for (int pp = warp; pp < P; pp += kBwdWarps) {
    for (int n = lane; n < N4; n += 32) {
      if (n < N) {
        cp_async4(sH + pp * NS + n, p.states + so + pp * N + n);
        cp_async4(sG + pp * NS + n, dg + so + pp * N + n);
      } else {
        sH[pp * NS + n] = 0.f;
        sG[pp * NS + n] = 0.f;
      }
    }
  }
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();

  const int t16 = threadIdx.x >> 4, l16 = threadIdx.x & 15;
  // Pairwise products: rows i = t16 + 16a, columns j = l16 + 16q of the chunk; M, A and the
  // row and column sums of W.
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
    // with R | 16 the 16-row blocks hold whole steps, so the blocks above the diagonal are zero
    if ((16 % R) == 0) {
      pair_products<true>(sC, sB, NS, N4, ri, cj, cb);
      pair_products<true>(sdy, sx, PS, P4, ri, cj, dx4);
    } else {
      pair_products<false>(sC, sB, NS, N4, ri, cj, cb);
      pair_products<false>(sdy, sx, PS, P4, ri, cj, dx4);
    }
    float rs[4] = {0.f, 0.f, 0.f, 0.f}, cs[4] = {0.f, 0.f, 0.f, 0.f};
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
          const float w = m * dx4[a][q];
          rs[a] += w;
          cs[q] += w;
        }
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float r = half_warp_sum(rs[a]);
      if (l16 == 0 && t16 + 16 * a < Lr) roww[t16 + 16 * a] = (double)r;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float v = cs[q] + __shfl_xor_sync(0xffffffffu, cs[q], 16);   // both half-warps
      if (lane < 16 && l16 + 16 * q < Lr) colp[warp * kBwdRows + l16 + 16 * q] = v;
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  const double cum_end = cum[l - 1];
  if (threadIdx.x < Lr) {   // W column sums over the warps' partials
    double sacc = 0.0;
    for (int w = 0; w < kBwdWarps; ++w) sacc += (double)colp[w * kBwdRows + threadIdx.x];
    colw[threadIdx.x] = sacc;
  }

  const int r0 = 4 * t16;   // this thread's output rows r0 + a (clamped for loads)
  int rc[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) rc[a] = min(r0 + a, Lr - 1);
  // 16-byte aligned start of the 4 rows' columns of M and A; only a thread whose rows all lie
  // past the chunk (outputs discarded) is moved back inside the row
  const int ra = min(r0, LS - 4);
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
    for (int n = 0; n < N4; n += 4) {
      float bv[4][4], gv[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a) lds_vec<4>(sB + rc[a] * NS + n, bv[a]);
#pragma unroll
      for (int q = 0; q < 4; ++q) lds_vec<4>(sG + pc[q] * NS + n, gv[q]);
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(bv[a][k], gv[q][k], acc[a][q]);
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
      if (l16 == 0 && r0 + a < Lr) qj[r0 + a] = (double)qs;
    }
    for (int i = (r0 / R) * R; i < Lr; ++i) {   // M_ij = 0 before row j's step
      float mv[4], dv[4];
      lds_vec<4>(sM + i * LS + ra, mv);
#pragma unroll
      for (int q = 0; q < 4; ++q) dv[q] = sdy[i * PS + pc[q]];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(mv[a], dv[q], acc[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = r0 + a;
      if (j < nvr) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int pp = l16 + 16 * q;
          if (pp < P) dx[((row0 + j) * p.H + h) * P + pp] = acc[a][q];
        }
      }
    }
  }

  int n0[HH];
  bool nown[HH];   // the run is this lane's own (not a clamped duplicate) and inside N
#pragma unroll
  for (int hh = 0; hh < HH; ++hh) {
    n0[hh] = col0<NQ>(l16, hh, N4);
    nown[hh] = n0[hh] == VW * l16 + 16 * VW * hh && n0[hh] < N;
  }

  // dB [Lr x N]: el_j (x G)_jn, then + (A^T C)_jn.
  {
    float acc[4][NQ];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[a][q] = 0.f;
    for (int pp = 0; pp < P4; pp += 4) {
      float xv[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a) lds_vec<4>(sx + rc[a] * PS + pp, xv[a]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (pp + k >= P) break;
        float gv[NQ];
#pragma unroll
        for (int hh = 0; hh < HH; ++hh) lds_vec<VW>(sG + (pp + k) * NS + n0[hh], gv + hh * VW);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int q = 0; q < NQ; ++q) acc[a][q] = fmaf(xv[a][k], gv[q], acc[a][q]);
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[a][q] *= el[a];
    for (int i = (r0 / R) * R; i < Lr; ++i) {   // A_ij = 0 before row j's step
      float av[4], cv[NQ];
      lds_vec<4>(sA + i * LS + ra, av);
#pragma unroll
      for (int hh = 0; hh < HH; ++hh) lds_vec<VW>(sC + i * NS + n0[hh], cv + hh * VW);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < NQ; ++q) acc[a][q] = fmaf(av[a], cv[q], acc[a][q]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = r0 + a;
      if (j < nvr) {
        float* dst = dB + ((row0 + j) * p.G + g) * N;
#pragma unroll
        for (int hh = 0; hh < HH; ++hh)
          if (nown[hh]) atomic_add_vec<VW>(dst + n0[hh], acc[a] + hh * VW);
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
    for (int pp = 0; pp < P4; pp += 4) {
      float dv[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a) lds_vec<4>(sdy + rc[a] * PS + pp, dv[a]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (pp + k >= P) break;
        float hv[NQ];
#pragma unroll
        for (int hh = 0; hh < HH; ++hh) lds_vec<VW>(sH + (pp + k) * NS + n0[hh], hv + hh * VW);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int q = 0; q < NQ; ++q) acc[a][q] = fmaf(dv[a][k], hv[q], acc[a][q]);
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float ei = expf((float)cum[rc[a] / R]);
      float cv[NQ];
#pragma unroll
      for (int hh = 0; hh < HH; ++hh) lds_vec<VW>(sC + rc[a] * NS + n0[hh], cv + hh * VW);
      float es = 0.f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        acc[a][q] *= ei;
        if (nown[q / VW]) es = fmaf(cv[q], acc[a][q], es);
      }
      es = half_warp_sum(es);
      if (l16 == 0 && r0 + a < Lr) ein[r0 + a] = (double)es;
    }
    const int jend = min(Lr, (rc[3] / R + 1) * R);   // A_ij = 0 after row i's step
    for (int j0 = 0; j0 < jend; j0 += 4) {
      float av[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a) lds_vec<4>(sA + rc[a] * LS + j0, av[a]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (j0 + k >= jend) break;
        float bv[NQ];
#pragma unroll
        for (int hh = 0; hh < HH; ++hh) lds_vec<VW>(sB + (j0 + k) * NS + n0[hh], bv + hh * VW);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int q = 0; q < NQ; ++q) acc[a][q] = fmaf(av[a][k], bv[q], acc[a][q]);
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = r0 + a;
      if (i < nvr) {
        float* dst = dC + ((row0 + i) * p.G + g) * N;
#pragma unroll
        for (int hh = 0; hh < HH; ++hh)
          if (nown[hh]) atomic_add_vec<VW>(dst + n0[hh], acc[a] + hh * VW);
      }
    }
  }

  // <G, h_in>, for the chunk-end gradient of exp(cum_end) h_in.
  {
    float sacc = 0.f;
    for (int pp = warp; pp < P; pp += kBwdWarps)
      for (int n = lane; n < N; n += 32) sacc = fmaf(sG[pp * NS + n], sH[pp * NS + n], sacc);
    double d = (double)sacc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) red[warp] = d;
  }
  __syncthreads();

  // dL/dcum_s, then ddA_t = sum_{s >= t} dL/dcum_s over the chunk's steps: warp 0, lane k
  // holds steps 2k and 2k + 1 (l <= 64), and a shuffle scan forms the suffix sums.
  if (warp == 0) {
    double gh = 0.0, qsum = 0.0;
#pragma unroll
    for (int w = 0; w < kBwdWarps; ++w) gh += red[w];
    for (int j = lane; j < Lr; j += 32) qsum += qj[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) qsum += __shfl_xor_sync(0xffffffffu, qsum, off);
    double d2[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int st = 2 * lane + k;
      double v = 0.0;
      if (st < l) {
        for (int r = 0; r < R; ++r) {
          const int i = st * R + r;
          v += roww[i] - colw[i] + ein[i] - qj[i];
        }
        if (st == l - 1) v += qsum + exp(cum_end) * gh;   // the chunk-end terms
      }
      d2[k] = v;
    }
    // suffix sums: first over the lanes above (inclusive scan from the top), then within a lane
    double tot = d2[0] + d2[1], incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double v = __shfl_down_sync(0xffffffffu, incl, off);
      if (lane + off < 32) incl += v;
    }
    const double above = incl - tot;   // steps 2 lane + 2 and later
    const double s1 = above + d2[1], s0 = s1 + d2[0];
    const int64_t base = (b * p.T + c * p.l) * p.H + h;
    if (2 * lane < nv) ddA[base + (int64_t)(2 * lane) * p.H] = (float)s0;
    if (2 * lane + 1 < nv) ddA[base + (int64_t)(2 * lane + 1) * p.H] = (float)s1;
  }
}

// ---------------------------------------------------------------------------------------------
// Rotation, in chunk-local frames.  Within chunk c let phi_t be the sum of theta over the chunk's
// steps up to t (zero before the chunk).  The rotated recurrence is then, inside the chunk, the
// plain one on B^ = R(-phi_t) B and C^ = R(-phi_t) C (per head) for the state g_t = R(-phi_t) h_t
// (scan.py page, THE TRICK, restarted at every chunk), entered with the physical h_in(c) and left
// by h_in(c+1) = R(phi_end) g_end.  The plain chunk kernels run on B^, C^; the carry turns by
// phi_end at each chunk boundary (backward: G^_c = R(-phi_end) dL/dh_in(c+1), dfinal entering
// physical).  The chain rule then gives
//   dB = R(phi) dB^, dC = R(phi) dC^ (summed over the heads of a group);
//   dL/dphi_t = sum over the step's rows of (dB^_0 B^_1 - dB^_1 B^_0 + dC^_0 C^_1 - dC^_1 C^_0),
//               plus, at the chunk's last step, sum_p (G^_1 g_0 - G^_0 g_1) with g = g_end
//   (d R(-phi) v / d phi = -J R(-phi) v and d R(phi) v / d phi = J R(phi) v, J the quarter turn);
//   dtheta_t = sum of dL/dphi over the steps t .. chunk end.
// Every dtheta is a sum over one chunk at most: angles never grow past a chunk's sum and no sum
// runs over the whole sequence (whose terms cancel far below their size).
constexpr int kRotLanes = 32, kRotRows = 8;

unsigned bwd_blocks(int64_t n) {
  return (unsigned)(n < 1 ? 1 : (n > 0x7fffffff ? 0x7fffffff : n));
}

// Chunk-local angles phi_t: one thread per (batch, chunk, head, pair), pairs fastest.
__global__ void __launch_bounds__(kBwdThreads)
    bwd_phi_local_kernel(GenericParams p, float* __restrict__ phiL) {
  const int64_t K = p.N / 2;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.batch * p.nch * p.H * K) return;
  const int64_t k = idx % K, h = (idx / K) % p.H, c = (idx / (K * p.H)) % p.nch;
  const int64_t b = idx / (K * p.H * p.nch);
  const int nv = bwd_steps(p, c);
  const int64_t t0 = b * p.T + c * p.l;
  double acc = 0.0;
  for (int t = 0; t < nv; ++t) {
    const int64_t o = ((t0 + t) * p.H + h) * K + k;
    acc += (double)__ldg(p.theta + o);
    phiL[o] = (float)acc;
  }
}

// B^ = R(-phi_t) B and C^ = R(-phi_t) C per head, fp32: one block per step.
template <typename T>
__global__ void __launch_bounds__(kRotLanes * kRotRows)
    bwd_rot_bc_kernel(const T* __restrict__ B, const T* __restrict__ C,
                      const float* __restrict__ phiL, float* __restrict__ Bt,
                      float* __restrict__ Ct, int64_t steps, int64_t R, int64_t H, int64_t G,
                      int64_t N) {
  const int64_t K = N / 2, hpg = H / G;
  for (int64_t bt = blockIdx.x; bt < steps; bt += gridDim.x) {
    for (int64_t r = 0; r < R; ++r) {
      for (int64_t h = threadIdx.y; h < H; h += kRotRows) {
        const int64_t src = ((bt * R + r) * G + h / hpg) * N, dst = ((bt * R + r) * H + h) * N;
        for (int64_t k = threadIdx.x; k < K; k += kRotLanes) {
          float sn, cs;
          sincosf(phiL[(bt * H + h) * K + k], &sn, &cs);
          const float b0 = ld_f32(B + src + 2 * k), b1 = ld_f32(B + src + 2 * k + 1);
          const float c0 = ld_f32(C + src + 2 * k), c1 = ld_f32(C + src + 2 * k + 1);
          Bt[dst + 2 * k] = cs * b0 + sn * b1;
          Bt[dst + 2 * k + 1] = cs * b1 - sn * b0;
          Ct[dst + 2 * k] = cs * c0 + sn * c1;
          Ct[dst + 2 * k + 1] = cs * c1 - sn * c0;
        }
      }
    }
  }
}

// The carries with the turn at each chunk boundary, one thread per state pair (b, h, p, k) and
// direction (forward first), loading kCarryAhead chunks ahead:
//   forward:  states[c] <- h_in(c),  h_in(c+1) = R(phi_end) (exp(cend_c) h_in(c) + S_c),
//             gfin <- h_in(nch) (the final state)
//   backward: dg[c] <- G^_c = R(-phi_end) v,  v <- exp(cend_c) G^_c + D_c  from v = dfinal,
//             dinit <- v.
__global__ void __launch_bounds__(kBwdThreads)
    bwd_carry_rot_kernel(GenericParams p, const float* __restrict__ phiL,
                         const float* __restrict__ dfinal, float* __restrict__ dg,
                         float* __restrict__ dinit, float* __restrict__ gfin) {
  const int64_t K = p.N / 2, PK = p.P * K, n_pr = p.batch * p.H * PK;
  int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= 2 * n_pr) return;
  const bool back = idx >= n_pr;
  if (back) idx -= n_pr;
  const int64_t k = idx % K, pp = (idx / K) % p.P, bh = idx / PK;
  const int64_t b = bh / p.H, h = bh % p.H;
  const int64_t PN = p.P * p.N, cs = p.H * PN;          // chunk stride of states / dg
  const int64_t e0 = (bh * p.P + pp) * p.N + 2 * k;     // element of the pair in [b,H,P,N]
  float* vp = (back ? dg : p.states) + (b * p.nch * p.H + h) * PN + pp * p.N + 2 * k;
  const float* ce = p.cend + b * p.nch * p.H + h;
  const float* init = back ? dfinal : p.init;
  float v0 = init ? init[e0] : 0.f, v1 = init ? init[e0 + 1] : 0.f;
  for (int64_t k0 = 0; k0 < p.nch; k0 += kCarryAhead) {
    float s0[kCarryAhead], s1[kCarryAhead], av[kCarryAhead], ph[kCarryAhead];
#pragma unroll
    for (int q = 0; q < kCarryAhead; ++q)
      if (k0 + q < p.nch) {
        const int64_t c = back ? p.nch - 1 - (k0 + q) : k0 + q;
        s0[q] = vp[c * cs];
        s1[q] = vp[c * cs + 1];
        av[q] = ce[c * p.H];
        const int64_t tl = b * p.T + c * p.l + bwd_steps(p, c) - 1;   // the chunk's last step
        ph[q] = phiL[(tl * p.H + h) * K + k];
      }
#pragma unroll
    for (int q = 0; q < kCarryAhead; ++q)
      if (k0 + q < p.nch) {
        const int64_t c = back ? p.nch - 1 - (k0 + q) : k0 + q;
        const float a = expf(av[q]);
        float sn, co;
        sincosf(ph[q], &sn, &co);
        if (back) {
          const float g0 = co * v0 + sn * v1, g1 = co * v1 - sn * v0;   // R(-phi_end) v
          vp[c * cs] = g0;
          vp[c * cs + 1] = g1;
          v0 = fmaf(a, g0, s0[q]);
          v1 = fmaf(a, g1, s1[q]);
        } else {
          vp[c * cs] = v0;
          vp[c * cs + 1] = v1;
          const float w0 = fmaf(a, v0, s0[q]), w1 = fmaf(a, v1, s1[q]);
          v0 = co * w0 - sn * w1;                                        // R(phi_end) w
          v1 = sn * w0 + co * w1;
        }
      }
  }
  if (back) {
    if (dinit) {
      dinit[e0] = v0;
      dinit[e0 + 1] = v1;
    }
  } else {
    gfin[e0] = v0;
    gfin[e0 + 1] = v1;
  }
}

// The chunk-end term of dL/dphi: sum_p (G^_1 g_0 - G^_0 g_1) with G^ = dg[c] and
// g = g_end(c) = R(-phi_end) h_in(c+1) (the final state for the last chunk); one thread per
// (batch, chunk, head, pair).
__global__ void __launch_bounds__(kBwdThreads)
    bwd_chunk_end_kernel(GenericParams p, const float* __restrict__ phiL,
                         const float* __restrict__ dg, const float* __restrict__ gfin,
                         float* __restrict__ eterm) {
  const int64_t K = p.N / 2;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.batch * p.nch * p.H * K) return;
  const int64_t k = idx % K, h = (idx / K) % p.H, c = (idx / (K * p.H)) % p.nch;
  const int64_t b = idx / (K * p.H * p.nch);
  const int64_t tl = b * p.T + c * p.l + bwd_steps(p, c) - 1;
  float sn, co;
  sincosf(phiL[(tl * p.H + h) * K + k], &sn, &co);
  const int64_t PN = p.P * p.N;
  const float* gh = dg + ((b * p.nch + c) * p.H + h) * PN + 2 * k;
  const float* hn = (c + 1 < p.nch) ? p.states + ((b * p.nch + c + 1) * p.H + h) * PN + 2 * k
                                    : gfin + (b * p.H + h) * PN + 2 * k;
  double e = 0.0;
  for (int64_t pp = 0; pp < p.P; ++pp) {
    const float h0 = hn[pp * p.N], h1 = hn[pp * p.N + 1];
    const float g0 = co * h0 + sn * h1, g1 = co * h1 - sn * h0;   // R(-phi_end) h_in(c+1)
    e += (double)(gh[pp * p.N + 1] * g0 - gh[pp * p.N] * g1);
  }
  eterm[idx] = (float)e;
}

// Per step (one block): dB and dC per group from the heads' dB^, dC^ turned back by +phi, and
// the step's dL/dphi per (head, pair) into dphi.
__global__ void __launch_bounds__(kRotLanes * kRotRows)
    bwd_rot_grad_kernel(const float* __restrict__ Bt, const float* __restrict__ Ct,
                        const float* __restrict__ dBt, const float* __restrict__ dCt,
                        const float* __restrict__ phiL, float* __restrict__ dB,
                        float* __restrict__ dC, float* __restrict__ dphi, int64_t steps,
                        int64_t R, int64_t H, int64_t G, int64_t N) {
  const int64_t K = N / 2, hpg = H / G;
  for (int64_t bt = blockIdx.x; bt < steps; bt += gridDim.x) {
    for (int64_t h = threadIdx.y; h < H; h += kRotRows) {
      for (int64_t k = threadIdx.x; k < K; k += kRotLanes) {
        float s = 0.f;
        for (int64_t r = 0; r < R; ++r) {
          const int64_t o = ((bt * R + r) * H + h) * N + 2 * k;
          s += dBt[o] * Bt[o + 1] - dBt[o + 1] * Bt[o] + dCt[o] * Ct[o + 1] - dCt[o + 1] * Ct[o];
        }
        dphi[(bt * H + h) * K + k] = s;
      }
    }
    for (int64_t r = 0; r < R; ++r) {
      for (int64_t g = threadIdx.y; g < G; g += kRotRows) {
        for (int64_t k = threadIdx.x; k < K; k += kRotLanes) {
          float b0 = 0.f, b1 = 0.f, c0 = 0.f, c1 = 0.f;
          for (int64_t h = g * hpg; h < (g + 1) * hpg; ++h) {
            float sn, cs;
            sincosf(phiL[(bt * H + h) * K + k], &sn, &cs);
            const int64_t o = ((bt * R + r) * H + h) * N + 2 * k;
            const float e0 = dBt[o], e1 = dBt[o + 1], f0 = dCt[o], f1 = dCt[o + 1];
            b0 += cs * e0 - sn * e1;
            b1 += sn * e0 + cs * e1;
            c0 += cs * f0 - sn * f1;
            c1 += sn * f0 + cs * f1;
          }
          const int64_t o = ((bt * R + r) * G + g) * N + 2 * k;
          dB[o] = b0;
          dB[o + 1] = b1;
          dC[o] = c0;
          dC[o + 1] = c1;
        }
      }
    }
  }
}

// dtheta_t = the chunk-end term plus dL/dphi over the steps t .. chunk end (fp64), one thread per
// (batch, chunk, head, pair).
__global__ void __launch_bounds__(kBwdThreads)
    bwd_dtheta_kernel(GenericParams p, const float* __restrict__ dphi,
                      const float* __restrict__ eterm, float* __restrict__ dtheta) {
  const int64_t K = p.N / 2;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.batch * p.nch * p.H * K) return;
  const int64_t k = idx % K, h = (idx / K) % p.H, c = (idx / (K * p.H)) % p.nch;
  const int64_t b = idx / (K * p.H * p.nch);
  const int nv = bwd_steps(p, c);
  const int64_t t0 = b * p.T + c * p.l;
  double acc = (double)eterm[idx];
  for (int t = nv - 1; t >= 0; --t) {
    const int64_t o = ((t0 + t) * p.H + h) * K + k;
    acc += (double)dphi[o];
    dtheta[o] = (float)acc;
  }
}

// Fused rows per backward chunk: 64 / R steps of R rows.
int64_t bwd_chunk_steps(int64_t R) { return R >= kBwdRows ? 1 : kBwdRows / R; }

struct BwdLayout {
  size_t states = 0, cend = 0, dg = 0;
  // rotation only
  size_t phiL = 0, Bt = 0, Ct = 0, dBt = 0, dCt = 0, gfin = 0, dphi = 0, eterm = 0;
  size_t total = 0;
};

ssd_status bwd_shape_status(const ssd_shape* s) {
  const ssd_status st = shape_status(s);
  if (st != SSD_OK) return st;
  if (s->mimo_rank > kBwdRows || s->headdim > kBwdMaxP || s->dstate > kBwdMaxN ||
      (s->dstate % 4) != 0)
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
  const size_t b = (size_t)s->batch, T = (size_t)s->seqlen, R = (size_t)s->mimo_rank;
  const size_t H = (size_t)s->nheads, P = (size_t)s->headdim, N = (size_t)s->dstate, K = N / 2;
  const size_t st = sizeof(float) * b * (size_t)nch * H * P * N;
  BwdLayout L;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kWsAlign);
    return at;
  };
  L.states = take(st);
  L.cend = take(sizeof(float) * b * (size_t)nch * H);
  L.dg = take(st);
  if (s->has_theta) {
    L.phiL = take(sizeof(float) * b * T * H * K);
    const size_t bc = sizeof(float) * b * T * R * H * N;
    L.Bt = take(bc);
    L.Ct = take(bc);
    L.dBt = take(bc);
    L.dCt = take(bc);
    L.gfin = take(sizeof(float) * b * H * P * N);
    L.dphi = take(sizeof(float) * b * T * H * K);
    L.eterm = take(sizeof(float) * b * (size_t)nch * H * K);
  }
  L.total = off;
  return L;
}

bool al16_or_null(const void* q) { return q == nullptr || aligned16(q); }

// The three launches; with chunk-local angles phiL the carry turns at every chunk boundary.
template <typename TX, typename TBC, int NQ>
cudaError_t bwd_launch_nq(const GenericParams& p, const float* dy, const float* dfinal,
                          float* dx, float* ddA, float* dB, float* dC, float* dinit, float* dg,
                          const float* phiL, float* gfin, cudaStream_t st) {
  const int64_t Lr = p.l * p.R;
  const dim3 grid((unsigned)p.nch, (unsigned)p.H, (unsigned)p.batch);
  const size_t s1 = bwd_state_smem(Lr, p.P, p.N);
  cudaError_t e = cudaFuncSetAttribute(bwd_chunk_state_kernel<TX, TBC, NQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e != cudaSuccess) return e;
  bwd_chunk_state_kernel<TX, TBC, NQ><<<grid, kBwdThreads, s1, st>>>(p, dy, dg);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (phiL) {
    const int64_t n = p.batch * p.H * p.P * p.N;   // two directions x N/2 pairs
    bwd_carry_rot_kernel<<<(unsigned)((n + kBwdThreads - 1) / kBwdThreads), kBwdThreads, 0,
                           st>>>(p, phiL, dfinal, dg, dinit, gfin);
  } else {
    const int64_t n = 2 * p.batch * p.H * p.P * p.N;
    bwd_carry_kernel<<<(unsigned)((n + kBwdThreads - 1) / kBwdThreads), kBwdThreads, 0, st>>>(
        p, dfinal, dg, dinit, gfin);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t s2 = bwd_grad_smem(Lr, p.P, p.N);
  e = cudaFuncSetAttribute(bwd_chunk_grad_kernel<TX, TBC, NQ>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
  if (e != cudaSuccess) return e;
  bwd_chunk_grad_kernel<TX, TBC, NQ><<<grid, kBwdThreads, s2, st>>>(p, dy, dg, dx, ddA, dB, dC);
  return cudaGetLastError();
}

// Column tiles of 16 state dims: N <= 16, 32, 64 or 128.
template <typename TX, typename TBC>
cudaError_t bwd_launch(const GenericParams& p, const float* dy, const float* dfinal, float* dx,
                       float* ddA, float* dB, float* dC, float* dinit, float* dg,
                       const float* phiL, float* gfin, cudaStream_t st) {
  if (p.N <= 16)
    return bwd_launch_nq<TX, TBC, 1>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, phiL, gfin, st);
  if (p.N <= 32)
    return bwd_launch_nq<TX, TBC, 2>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, phiL, gfin, st);
  if (p.N <= 64)
    return bwd_launch_nq<TX, TBC, 4>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, phiL, gfin, st);
  return bwd_launch_nq<TX, TBC, 8>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, phiL, gfin, st);
}

// The rotated backward: chunk-local angles and B^, C^, the plain chunk kernels on them with the
// turning carry, then dB, dC turned back and dtheta from per-chunk sums.
cudaError_t bwd_rotated(GenericParams p, const ssd_shape* s, const BwdLayout& lay, char* ws,
                        const float* dy, const float* dfinal, float* dx, float* ddA, float* dB,
                        float* dC, float* dtheta, float* dinit, float* dg, cudaStream_t st) {
  const int64_t K = p.N / 2, steps = p.batch * p.T;
  float* phiL = reinterpret_cast<float*>(ws + lay.phiL);
  float* Bt = reinterpret_cast<float*>(ws + lay.Bt);
  float* Ct = reinterpret_cast<float*>(ws + lay.Ct);
  float* dBt = reinterpret_cast<float*>(ws + lay.dBt);
  float* dCt = reinterpret_cast<float*>(ws + lay.dCt);
  float* gfin = reinterpret_cast<float*>(ws + lay.gfin);
  float* dphi = reinterpret_cast<float*>(ws + lay.dphi);
  float* eterm = reinterpret_cast<float*>(ws + lay.eterm);
  const int64_t nk = p.batch * p.nch * p.H * K;
  const unsigned gk = bwd_blocks((nk + kBwdThreads - 1) / kBwdThreads);
  bwd_phi_local_kernel<<<gk, kBwdThreads, 0, st>>>(p, phiL);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 blk(kRotLanes, kRotRows);
  if (s->io_dtype == SSD_BF16) {
    bwd_rot_bc_kernel<__nv_bfloat16><<<bwd_blocks(steps), blk, 0, st>>>(
        static_cast<const __nv_bfloat16*>(p.B), static_cast<const __nv_bfloat16*>(p.C), phiL, Bt,
        Ct, steps, p.R, p.H, p.G, p.N);
  } else {
    bwd_rot_bc_kernel<float><<<bwd_blocks(steps), blk, 0, st>>>(
        static_cast<const float*>(p.B), static_cast<const float*>(p.C), phiL, Bt, Ct, steps, p.R,
        p.H, p.G, p.N);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t bc = sizeof(float) * (size_t)(steps * p.R * p.H * p.N);
  if ((e = cudaMemsetAsync(dBt, 0, bc, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dCt, 0, bc, st)) != cudaSuccess) return e;
  GenericParams q = p;   // the chunk-local plain problem: fp32 B^, C^, one group per head
  q.B = Bt;
  q.C = Ct;
  q.G = p.H;
  q.theta = nullptr;
  e = s->io_dtype == SSD_BF16
          ? bwd_launch<__nv_bfloat16, float>(q, dy, dfinal, dx, ddA, dBt, dCt, dinit, dg, phiL,
                                             gfin, st)
          : bwd_launch<float, float>(q, dy, dfinal, dx, ddA, dBt, dCt, dinit, dg, phiL, gfin, st);
  if (e != cudaSuccess) return e;
  bwd_chunk_end_kernel<<<gk, kBwdThreads, 0, st>>>(p, phiL, dg, gfin, eterm);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_rot_grad_kernel<<<bwd_blocks(steps), blk, 0, st>>>(Bt, Ct, dBt, dCt, phiL, dB, dC, dphi,
                                                          steps, p.R, p.H, p.G, p.N);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_dtheta_kernel<<<gk, kBwdThreads, 0, st>>>(p, dphi, eterm, dtheta);
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
                                const void* B, const void* C, const float* theta,
                                const float* init_state, const float* dy, const float* dfinal,
                                float* dx, float* ddA, float* dB, float* dC, float* dtheta,
                                float* dinit, void* workspace, size_t workspace_bytes,
                                void* stream) {
  const ssd_status vs = bwd_shape_status(shape);
  if (vs != SSD_OK) return vs;
  if (!x || !dA || !B || !C || !dy || !dx || !ddA || !dB || !dC) return SSD_ERR_INVALID_ARG;
  const bool rot = shape->has_theta != 0;
  if (rot != (theta != nullptr) || rot != (dtheta != nullptr)) return SSD_ERR_INVALID_ARG;
  const void* ptrs[] = {x, dA, B, C, theta, init_state, dy, dfinal, dx, ddA, dB, dC, dtheta, dinit};
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
  p.theta = theta;
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

  cudaError_t e;
  if (rot) {
    e = bwd_rotated(p, shape, lay, ws, dy, dfinal, dx, ddA, dB, dC, dtheta, dinit, dg, st);
  } else {
    const size_t bc = sizeof(float) * (size_t)(p.batch * p.T * p.R * p.G * p.N);
    if (cudaMemsetAsync(dB, 0, bc, st) != cudaSuccess ||
        cudaMemsetAsync(dC, 0, bc, st) != cudaSuccess)
      return SSD_ERR_CUDA;
    e = bf16 ? bwd_launch<__nv_bfloat16, __nv_bfloat16>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg,
                                                        nullptr, nullptr, st)
             : bwd_launch<float, float>(p, dy, dfinal, dx, ddA, dB, dC, dinit, dg, nullptr,
                                        nullptr, st);
  }
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
