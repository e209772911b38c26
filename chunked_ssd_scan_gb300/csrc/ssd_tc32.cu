// fp32 chunk scan (K2 + K5) on the tensor core: tcgen05.mma kind::tf32 for fp32 I/O with
// P = N = 64, one CTA per chunk of 128 rank-fused rows (128 / R steps) of one (batch, head).
//
// The chunk's outputs (the serial.rs page's K2 and K5, the rotation absorbed into B and C as on
// the scan.py page):
//   y_i = e^{cum_i} C~_i . h_in  +  sum_{j <= i} e^{cum_i - cum_j} (C~_i . B~_j) x_j
// with h_in the state entering the chunk (written by the K4 pass over the chunk states).
//
// Precision.  The tensor core multiplies tf32 (10 explicit mantissa bits) and accumulates in
// fp32 with truncation toward zero at every step, so one tf32 product of fp32 data, or a long
// chain of them in one accumulator, misses the fp32 gate |got - ref| <= 1e-4 (1 + |ref|).  Here
// every fp32 operand is split into a tf32 high part (rounded) and the fp32 remainder (read as
// tf32), each pair takes three products (hi.hi + hi.lo + lo.hi), and an accumulator spans one
// 32-deep K block only: the K blocks land in separate TMEM accumulators whose sum the CUDA cores
// form in fp32, round to nearest.  A CPU model of exactly this arithmetic meets the gate with
// about half of it to spare on slowly decaying inputs with an initial state.
//
// Per chunk:
//   staging   C~, B~ (turned by -Phi_t) and h_in as tf32 hi / lo, K-major with 128-byte swizzle
//   phase 1   CB = C~ B~^T  M128 N128 K64: 2 K blocks x 3 products x 4 MMAs, TMEM cols 0..255
//             Yo = C~ h^T   M128 N64  K64: 2 x 3 x 4, TMEM cols 256..383
//   CUDA      Yo blocks summed into registers; CB blocks summed, the causal decay mask applied
//             (exponent of the step difference, causal cut first), split into hi / lo and
//             written back over the CB columns (hi 0..127, lo 128..255): the A operand of
//             phase 2; x^T split into hi / lo in shared memory over C~
//   phase 2   Yd = (L o CB) x  M128 N64 K128: 4 x 3 x 4 from TMEM (TS), TMEM cols 256..511
//   CUDA      y_i = e^{cum_i} Yo_i + the Yd blocks, stored per row
// A short chunk (the sequence's real steps end inside it) reads its missing rows as zeros and
// writes no y there.
#include <math.h>

#include <algorithm>

#include "chunk_prep.cuh"
#include "common.cuh"
#include "fp_helpers.cuh"
#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {

namespace {

using namespace prep;
using namespace tc;

constexpr int kRows = 128;                       // fused rows per chunk = MMA M
constexpr int kD = 64;                           // P = N
constexpr int kThreads = 512;                    // 16 warps: 4 per TMEM lane quarter
constexpr uint32_t kOpBytes = kRows * kD * 4;    // one 128 x 64 fp32 operand: 32 KB
constexpr uint32_t kAtom128 = kRows * 128;       // a 32-column atom of a 128-row operand
constexpr uint32_t kAtom64 = kD * 128;           // a 32-column atom of a 64-row operand
constexpr uint32_t kOffCHi = 0;
constexpr uint32_t kOffCLo = kOffCHi + kOpBytes;
constexpr uint32_t kOffBHi = kOffCLo + kOpBytes;
constexpr uint32_t kOffBLo = kOffBHi + kOpBytes;
constexpr uint32_t kOffXHi = 0;                  // phase 2: x^T [p][j] over C~ (free by then)
constexpr uint32_t kOffXLo = kOffXHi + kOpBytes;
constexpr uint32_t kOffHHi = kOffBLo + kOpBytes; // h_in [p][n]
constexpr uint32_t kOffHLo = kOffHHi + kOpBytes / 2;
constexpr uint32_t kOffAng = kOffHLo + kOpBytes / 2;           // angles [step][pair]
constexpr uint32_t kOffCum = kOffAng + kRows * kPairs64 * 4;   // cum_hi, cum_lo [step]
constexpr uint32_t kOffXRaw = kOffCum + 2 * kRows * 4;         // raw x rows [j][p]
// raw C, B and h_in rows land in the B~ hi, B~ lo and h lo buffers before staging
constexpr uint32_t kOffPhi0 = kOffXRaw + kOpBytes;             // the 32 chunk-start angles
constexpr uint32_t kOffDA = kOffPhi0 + kPairs64 * 8;            // dA of the chunk's steps
constexpr uint32_t kOffBar = kOffDA + kRows * 4;                // 2 mbarriers + TMEM base
constexpr uint32_t kSmemUsed = kOffBar + 32;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;              // the base is aligned up to 1 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColCB = 0;                   // CB K blocks 0, 1; then (L o CB) hi, lo
constexpr uint32_t kColYo = 256;                 // Yo K blocks 0, 1
constexpr uint32_t kColYd = 256;                 // Yd K blocks 0..3 (after Yo is read)
constexpr uint64_t kWaitNs = 2000000000ull;      // bounded MMA waits: 2 s

// Byte offset of element (row, k) of a K-major fp32 operand with `rows` rows: 32-column atoms
// of rows x 128 bytes, 128-byte swizzle inside each atom (the layout the descriptors name).
__device__ __forceinline__ uint32_t kmaj_off(uint32_t rows, uint32_t row, uint32_t k) {
  return (k >> 5) * rows * 128u + sw128_off32(row, k & 31u);
}

// tf32 high part of v (round to nearest, ties away: the cvt's rounding) and the remainder.
__device__ __forceinline__ float tf32_hi(float v) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
  return __uint_as_float(r);
}

__device__ __forceinline__ void store_split(uint8_t* hi, uint8_t* lo, float4 v) {
  const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
  *reinterpret_cast<float4*>(hi) = h;
  *reinterpret_cast<float4*>(lo) = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
}

__device__ __forceinline__ float comp(const float4& v, int e) {
  return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

// Tile u of the grid-stride loop: chunk c fastest, then head h, then batch b.
struct Tile {
  int64_t c, h, b;
};
__device__ __forceinline__ Tile tile_of(const GenericParams& p, int64_t u) {
  Tile t;
  t.c = u % p.nch;
  const int64_t r = u / p.nch;
  t.h = r % p.H;
  t.b = r / p.H;
  return t;
}

// cp.async copies of tile t's dA, chunk-start angles and theta, raw C rows (into the B~ hi
// buffer), raw B rows (into the B~ lo buffer) and h_in (into the h lo buffer), rows past the
// chunk's real ones zero-filled.  Their buffers are free once the previous tile's phase-1
// products completed and its prefix sums and angles were formed.
__device__ void issue_main(const GenericParams& p, const Tile& t, uint8_t* smem, float* ang) {
  const int R = (int)p.R;
  const int64_t g = t.h / (p.H / p.G);
  const int nv = steps64(p, t.b, t.c);
  const int nvr = nv * R;
  const int64_t row0 = (t.b * p.T + t.c * p.l) * R;
  const float* dA = p.dA + (t.b * p.T + t.c * p.l) * p.H + t.h;
  for (int k = threadIdx.x; k < nv; k += kThreads)
    cp_async4(smem + kOffDA + 4 * k, dA + (int64_t)k * p.H);
  if (p.theta) {
    issue_theta64(p, t.b, t.c, t.h, (int)p.l, ang);
    const double* ph = p.phi + ((t.b * (p.nch + 1) + t.c) * p.H + t.h) * kPairs64;
    for (int k = threadIdx.x; k < kPairs64 / 2; k += kThreads)
      cp_async16(smem + kOffPhi0 + 16 * k, ph + 2 * k, 16);
  }
  const float* Cg = static_cast<const float*>(p.C);
  const float* Bg = static_cast<const float*>(p.B);
  for (int e = threadIdx.x; e < kRows * kD / 4; e += kThreads) {
    const int row = e >> 4, q4 = e & 15;
    const bool real = row < nvr;
    const int64_t r = row0 + (real ? row : 0);
    cp_async16(smem + kOffBHi + 16 * e, Cg + (r * p.G + g) * kD + 4 * q4, real ? 16 : 0);
    cp_async16(smem + kOffBLo + 16 * e, Bg + (r * p.G + g) * kD + 4 * q4, real ? 16 : 0);
  }
  const float* hin = p.states + ((t.b * p.nch + t.c) * p.H + t.h) * (kD * kD);
  for (int e = threadIdx.x; e < kD * kD / 4; e += kThreads)
    cp_async16(smem + kOffHLo + 16 * e, hin + 4 * e, 16);
}

// cp.async copies of tile t's raw x rows; their buffer is free once the previous tile's x^T
// was formed.
__device__ void issue_x(const GenericParams& p, const Tile& t, uint8_t* smem) {
  const int R = (int)p.R;
  const int nvr = steps64(p, t.b, t.c) * R;
  const int64_t row0 = (t.b * p.T + t.c * p.l) * R;
  const float* Xg = static_cast<const float*>(p.x);
  for (int e = threadIdx.x; e < kRows * kD / 4; e += kThreads) {
    const int row = e >> 4, q4 = e & 15;
    const bool real = row < nvr;
    cp_async16(smem + kOffXRaw + 16 * e, Xg + ((row0 + (real ? row : 0)) * p.H + t.h) * kD + 4 * q4,
               real ? 16 : 0);
  }
}

// One CTA per SM walks the tiles u = blockIdx.x, + gridDim.x, ...; the copies of tile u + grid
// are issued while tile u's mask, x^T, phase 2 and output run, so the loads of one tile overlap
// the arithmetic of the previous one.
__global__ void __launch_bounds__(kThreads, 1) tc32_scan_kernel(GenericParams p, int64_t ntiles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* ang = reinterpret_cast<float*>(smem + kOffAng);
  float* cum_hi = reinterpret_cast<float*>(smem + kOffCum);
  float* cum_lo = cum_hi + kRows;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);        // MMA phases
  uint64_t* drain = bar + 1;                                          // abort path
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffBar + 16);

  const int l = (int)p.l;                        // steps per chunk (128 / R)
  const int R = (int)p.R, rs = rank_shift(p);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3, cw = warp >> 2;        // TMEM lane quarter; column quarter of the warp
  const int i = 32 * q + lane;                   // the row this thread reads out
  const int ti = i >> rs;
  const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;

  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  int64_t u = blockIdx.x;
  if (u < ntiles) {
    const Tile t = tile_of(p, u);
    issue_main(p, t, smem, ang);
    issue_x(p, t, smem);
  }
  cp_async_commit();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  constexpr uint32_t id_n128 = idesc_tf32(128, 128, 0, 0);
  constexpr uint32_t id_n64 = idesc_tf32(128, 64, 0, 0);
  constexpr uint32_t dh = sdesc_sw128_hi(1024);
  bool ok = true;
  for (; u < ntiles; u += gridDim.x) {
    const Tile t = tile_of(p, u);
    const int64_t nx = u + gridDim.x;
    const int nvr = steps64(p, t.b, t.c) * R;          // real fused rows of the chunk
    const int64_t row0 = (t.b * p.T + t.c * p.l) * R;  // fused row of the chunk's first step
    // prefix sums of dA (warp 0) and the rotation angles, from this tile's staged copies
    cp_async_wait_all();
    __syncthreads();
    chunk_prefix64<true>(reinterpret_cast<const float*>(smem + kOffDA), 1, l, steps64(p, t.b, t.c),
                         cum_hi, cum_lo, nullptr);
    if (p.theta) {
      chunk_angles64<kThreads>(p, t.b, t.c, t.h, l, ang, true,
                               reinterpret_cast<const double*>(smem + kOffPhi0));
    } else {
      __syncthreads();
    }

    // ---------------------------------------------------------------- staging
    {
      // C~ and B~: the half-warps of a row read it whole; both are turned by the same angle.
      // All raw values are read into registers before the first hi / lo store overwrites them.
      constexpr int kRowStep = kThreads / 16;   // rows per pass of the block
      const int ch = threadIdx.x & 15;   // k = 4 ch .. 4 ch + 3 (rotation pairs 2 ch, 2 ch + 1)
      float4 cv[kRows / kRowStep], bv[kRows / kRowStep], hv[kD / kRowStep];
#pragma unroll
      for (int r = 0; r < kRows / kRowStep; ++r) {
        const int e = threadIdx.x + kThreads * r;   // row (threadIdx.x >> 4) + kRowStep r
        cv[r] = *reinterpret_cast<const float4*>(smem + kOffBHi + 16 * e);
        bv[r] = *reinterpret_cast<const float4*>(smem + kOffBLo + 16 * e);
      }
#pragma unroll
      for (int r = 0; r < kD / kRowStep; ++r)
        hv[r] = *reinterpret_cast<const float4*>(smem + kOffHLo + 16 * (threadIdx.x + kThreads * r));
      __syncthreads();
#pragma unroll
      for (int r = 0; r < kRows / kRowStep; ++r) {
        const int row = (threadIdx.x >> 4) + kRowStep * r;
        float4 cr = cv[r], br = bv[r];
        if (p.theta) {
          const float* ar = ang + (row >> rs) * kPairs64 + 2 * ch;
          float s0, c0, s1, c1;
          sincosf(ar[0], &s0, &c0);
          sincosf(ar[1], &s1, &c1);
          cr = make_float4(c0 * cr.x + s0 * cr.y, -s0 * cr.x + c0 * cr.y, c1 * cr.z + s1 * cr.w,
                           -s1 * cr.z + c1 * cr.w);
          br = make_float4(c0 * br.x + s0 * br.y, -s0 * br.x + c0 * br.y, c1 * br.z + s1 * br.w,
                           -s1 * br.z + c1 * br.w);
        }
        const uint32_t o = kmaj_off(kRows, row, 4 * ch);
        store_split(smem + kOffCHi + o, smem + kOffCLo + o, cr);
        store_split(smem + kOffBHi + o, smem + kOffBLo + o, br);
      }
      // h_in [p][n] is K-major for Yo as it stands (rows p, K = n)
#pragma unroll
      for (int r = 0; r < kD / kRowStep; ++r) {
        const int pp = (threadIdx.x >> 4) + kRowStep * r;
        const uint32_t o = kmaj_off(kD, pp, 4 * ch);
        store_split(smem + kOffHHi + o, smem + kOffHLo + o, hv[r]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---------------------------------------------------------------- phase 1: CB, Yo
    if (warp == 1) {
      const uint32_t c_lo[2] = {sdesc_sw128_lo(smem_u32(smem + kOffCHi), 0),
                                sdesc_sw128_lo(smem_u32(smem + kOffCLo), 0)};
      const uint32_t b_lo[2] = {sdesc_sw128_lo(smem_u32(smem + kOffBHi), 0),
                                sdesc_sw128_lo(smem_u32(smem + kOffBLo), 0)};
      const uint32_t h_lo[2] = {sdesc_sw128_lo(smem_u32(smem + kOffHHi), 0),
                                sdesc_sw128_lo(smem_u32(smem + kOffHLo), 0)};
      // products (hi, lo), (lo, hi), (hi, hi) in this order (A part pr == 1, B part pr == 0):
      // the two small correction products go in first, so the accumulator truncates at their
      // magnitude and only the last four steps truncate at the block's own
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int pr = 0; pr < 3; ++pr)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t ko = (kb * kAtom128 + ks * 32) >> 4;
            mma_ss_we_tf32(tmem + kColCB + kb * 128, c_lo[pr == 1] + ko, dh, b_lo[pr == 0] + ko,
                           dh, id_n128, (pr | ks) != 0);
          }
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int pr = 0; pr < 3; ++pr)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t ka = (kb * kAtom128 + ks * 32) >> 4;
            const uint32_t kh = (kb * kAtom64 + ks * 32) >> 4;
            mma_ss_we_tf32(tmem + kColYo + kb * 64, c_lo[pr == 1] + ka, dh, h_lo[pr == 0] + kh,
                           dh, id_n64, (pr | ks) != 0);
          }
      mma_commit_elect(bar);
    }
    ok = mbar_wait_bounded(bar, 0, kWaitNs);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    tc_fence_after();

    // ---------------------------------------------------------------- Yo, mask, x^T
    float yo[16];   // Yo of row i, columns p = 16 cw .. 16 cw + 15
    {
      float a0[16], a1[16];
      tmem_ld16(tmem + lane_addr + kColYo + 16 * cw, a0);
      tmem_ld16(tmem + lane_addr + kColYo + 64 + 16 * cw, a1);
      tmem_ld_wait();
      reg_tie(a0);
      reg_tie(a1);
#pragma unroll
      for (int k = 0; k < 16; ++k) yo[k] = a0[k] + a1[k];
    }
    // the mask of columns j = 32 cw .. 32 cw + 31, 16 at a time; 2^x on the special-function
    // unit (relative error ~2^-22, results below 2^-126 flushed to zero: far below the gate)
    const float chi = cum_hi[ti], clo = cum_lo[ti];
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int j0 = 32 * cw + 16 * hb;
      uint32_t mh[16], ml[16];
      if ((j0 >> rs) > ((32 * q + 31) >> rs)) {   // every column after every row's step
#pragma unroll
        for (int k = 0; k < 16; ++k) mh[k] = ml[k] = 0u;
      } else {
        float v0[16], v1[16];
        tmem_ld16(tmem + lane_addr + kColCB + j0, v0);
        tmem_ld16(tmem + lane_addr + kColCB + 128 + j0, v1);
        tmem_ld_wait();
        reg_tie(v0);
        reg_tie(v1);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int tj = (j0 + k) >> rs;
          const float m = tj <= ti
                              ? fp::ex2_approx((chi - cum_hi[tj]) + (clo - cum_lo[tj])) *
                                    (v0[k] + v1[k])
                              : 0.f;
          const float mhi = tf32_hi(m);
          mh[k] = __float_as_uint(mhi);
          ml[k] = __float_as_uint(m - mhi);
        }
      }
      tmem_st16u(tmem + lane_addr + kColCB + j0, mh);
      tmem_st16u(tmem + lane_addr + kColCB + 128 + j0, ml);
    }
    // x^T [p][j] hi / lo from the raw rows (the warp's task: rows 16 jg .. 16 jg + 15, columns
    // 32 ph .. 32 ph + 31; lane: 4 rows from 4 jc, columns 4 cq ..): per store the 8 lanes of a
    // quarter warp cover 4 j chunks x 2 p rows of different parity, i.e. 8 distinct swizzled
    // chunk positions (conflict-free)
    {
      const int jc = lane & 3, jg = warp & 7, cq = 8 * (warp >> 3) + (lane >> 2);
      float4 xr[4];   // rows 16 jg + 4 jc + r, columns 4 cq .. 4 cq + 3
#pragma unroll
      for (int r = 0; r < 4; ++r)
        xr[r] = *reinterpret_cast<const float4*>(smem + kOffXRaw +
                                                 16 * ((16 * jg + 4 * jc + r) * (kD / 4) + cq));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 v =
            make_float4(comp(xr[0], e), comp(xr[1], e), comp(xr[2], e), comp(xr[3], e));
        const uint32_t o = kmaj_off(kD, 4 * cq + e, 16 * jg + 4 * jc);
        store_split(smem + kOffXHi + o, smem + kOffXLo + o, v);
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the next tile's inputs: phase 1 read B~ and h_in, staging read the angles, the raw x rows
    // were transposed; these copies overlap phase 2, the output and the next prefix sums
    if (nx < ntiles) {
      const Tile tn = tile_of(p, nx);
      issue_main(p, tn, smem, ang);
      issue_x(p, tn, smem);
    }
    cp_async_commit();

    // ---------------------------------------------------------------- phase 2: Yd
    if (warp == 1) {
      const uint32_t x_lo[2] = {sdesc_sw128_lo(smem_u32(smem + kOffXHi), 0),
                                sdesc_sw128_lo(smem_u32(smem + kOffXLo), 0)};
#pragma unroll
      for (int kb = 0; kb < 4; ++kb)
#pragma unroll
        for (int pr = 0; pr < 3; ++pr)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts_we_tf32(tmem + kColYd + kb * 64,
                           tmem + kColCB + (pr == 1 ? 128 : 0) + kb * 32 + ks * 8,
                           x_lo[pr == 0] + ((kb * kAtom64 + ks * 32) >> 4), dh, id_n64,
                           (pr | ks) != 0);
      mma_commit_elect(bar);
    }
    ok = mbar_wait_bounded(bar, 1, kWaitNs);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    tc_fence_after();
    {
      float yd[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) yd[k] = 0.f;
#pragma unroll
      for (int kb = 0; kb < 4; kb += 2) {
        float a0[16], a1[16];
        tmem_ld16(tmem + lane_addr + kColYd + kb * 64 + 16 * cw, a0);
        tmem_ld16(tmem + lane_addr + kColYd + (kb + 1) * 64 + 16 * cw, a1);
        tmem_ld_wait();
        reg_tie(a0);
        reg_tie(a1);
#pragma unroll
        for (int k = 0; k < 16; ++k) yd[k] = (yd[k] + a0[k]) + a1[k];
      }
      if (i < nvr) {
        const float sc = exp2f(chi + clo);   // e^{cum of row i's step}
        const int64_t yoff = ((row0 + i) * p.H + t.h) * kD + 16 * cw;
        if (SSD_INDEX_OK(p.hdr, yoff + 15, p.batch * p.T * p.R * p.H * kD, 24)) {
          float4* y4 = reinterpret_cast<float4*>(static_cast<float*>(p.y) + yoff);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            y4[k] = make_float4(fmaf(sc, yo[4 * k], yd[4 * k]),
                                fmaf(sc, yo[4 * k + 1], yd[4 * k + 1]),
                                fmaf(sc, yo[4 * k + 2], yd[4 * k + 2]),
                                fmaf(sc, yo[4 * k + 3], yd[4 * k + 3]));
        }
      }
    }
    // this tile's TMEM columns and cum arrays are read; the next tile may overwrite them
    tc_fence_before();
    __syncthreads();
  }
  if (!ok) {
    // a bounded wait gave up: latch it, then wait (bounded again) until every MMA issued so
    // far has completed before TMEM is released
    if (threadIdx.x == 0 && p.hdr) latch_error(p.hdr, SSD_ERR_TIMEOUT, 25);
    if (warp == 1) mma_commit_elect(drain);
    if (!mbar_wait_bounded(drain, 0, kWaitNs) && threadIdx.x == 0 && p.hdr)
      latch_error(p.hdr, SSD_ERR_TIMEOUT, 26);
  }
  cp_async_wait_all();   // no copy may still be landing in shared memory at exit
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool tc32_supported(int64_t P, int64_t N, int64_t R, bool bf16) {
  return !bf16 && P == kD && N == kD && R >= 1 && R <= 64 && (kRows % R) == 0;
}

int64_t tc32_chunk_len(int64_t R) { return kRows / R; }

cudaError_t tc32_scan(const GenericParams& p, cudaStream_t st) {
  if (p.P != kD || p.N != kD || p.l * p.R != kRows) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc32_scan_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int64_t ntiles = p.nch * p.H * p.batch;
  const unsigned grid = (unsigned)std::min<int64_t>(ntiles, std::max(sms, 1));
  if (grid == 0) return cudaSuccess;
  tc32_scan_kernel<<<grid, kThreads, kSmemAlloc, st>>>(p, ntiles);
  return cudaGetLastError();
}

}  // namespace ssd
