// Fused tcgen05/TMEM chunked SSD forward for bf16 I/O (sm_103a).
//
// One CTA owns one (batch, head) sequence and walks it in tiles of 128 rank-fused rows
// (fused row i = t*R + r, as in the serial.rs page's K2 reshape), carrying the state on chip
// from tile to tile, so the inter-chunk state of K4 never goes to HBM.  Per tile:
//   K1  tile-local inclusive cumsum of dA (fp64-accumulated, kept as hi+lo floats)
//   K2  CB = C B^T                                   tcgen05.mma  M128 N128 K128 -> TMEM
//   K5a Mcb = (L o CB) with L[i,j] = exp(cum[i/R]-cum[j/R]) for j/R <= i/R, else 0
//       (mask applied before the exponential; segsum.rs / scan.py pages), bf16 -> SMEM
//       Yd = Mcb X                                   tcgen05.mma  M128 N64  K128 -> TMEM
//   K3  S^T = (dec o B)^T X,  dec_i = exp(cum_last - cum[i/R])
//                                                    tcgen05.mma  M128 N64  K128 -> TMEM
//   K5b Yo = C h_in                                  tcgen05.mma  M128 N64  K128 -> TMEM
//       y  = Yd + exp(cum[i/R]) Yo  -> bf16 -> global
//   K4  h_out = exp(cum_last) h_in + S               (fp32, in registers)
// The serial.rs page runs K1..K5 per chunk with the K4 loop across chunks; a 128-row tile is a
// sub-block of a chunk, and the part of a chunk's 1-semiseparable mask below a tile's diagonal
// block has rank one (exp(cum_i - cum_j) = exp(cum_i) exp(-cum_j)), which is exactly what the
// tile-boundary state carries.  The result is the same recurrence for every chunk_len.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner),
// warps 2-5 "mask group" (K1, mask, dec o B), warps 6-9 "state group" (K4, h_in for K5b,
// output).  Operands are staged by TMA in 128-byte swizzled layouts; the two stages of x/B/C
// are double-buffered.  Every wait is bounded; a wait that gives up latches SSD_ERR_TIMEOUT in
// the workspace header and the CTA stops issuing work.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {

namespace {

using namespace tc;

constexpr int kTileRows = 128;
constexpr int kP = 64;
constexpr int kN = 128;
constexpr int kThreadsFused = 320;
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait before giving up

// Shared-memory map (offsets from a 1024-aligned base).
constexpr uint32_t kXBytes = kTileRows * kP * 2;          // 16 KB per stage
constexpr uint32_t kBCBytes = kTileRows * kN * 2;         // 32 KB per stage (two 64-col blocks)
constexpr uint32_t kOffX = 0;                              // 2 stages (x, then dec o x hi part)
constexpr uint32_t kOffXlo = kOffX + 2 * kXBytes;          // dec o x, lo part
constexpr uint32_t kOffB = kOffXlo + kXBytes;              // 2 stages
constexpr uint32_t kOffC = kOffB + 2 * kBCBytes;           // 2 stages
constexpr uint32_t kOffHhi = kOffC + 2 * kBCBytes;         // h_in, hi part  [N rows][P]
constexpr uint32_t kOffHlo = kOffHhi + kN * kP * 2;        // h_in, lo part
constexpr uint32_t kOffDA = kOffHlo + kN * kP * 2;         // 2 stages x 128 steps x 4 floats
constexpr uint32_t kDABytes = kTileRows * 16;
constexpr uint32_t kOffInfo = kOffDA + 2 * kDABytes;       // per-stage tile info
struct TileInfo {
  float cum_hi[kTileRows];   // log2-scaled prefix sum of dA at fused row j (step j/R), hi part
  float cum_lo[kTileRows];   // ... lo part (hi + lo carries ~48 bits)
  float expcum[kTileRows];   // exp(cum) at fused row j
  float dec[kTileRows];      // exp(cum_last - cum) at fused row j
  float etile;               // exp(cum_last)
  float pad[31];
};
constexpr uint32_t kOffBar = kOffInfo + 2 * sizeof(TileInfo);
constexpr uint32_t kSmemUsed = kOffBar + 256;
constexpr uint32_t kSmemAlloc = kSmemUsed;
static_assert(kSmemAlloc <= 232448, "exceeds the 227 KB shared-memory limit per CTA");

// TMEM columns (128 lanes x 512 columns of 32 bit).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColCB = 0;      // CB fp32 [0,128); after masking, (L o CB) hi part packed
                                    // two bf16 per column in [0,64)
constexpr uint32_t kColMlo = 128;   // (L o CB) lo part, packed, [128,192)
constexpr uint32_t kColYd = 192;    // Yd  [192,256)
constexpr uint32_t kColYo = 256;    // Yo from h_hi [256,320) and from h_lo [320,384)
constexpr uint32_t kColS = 384;     // S^T from (dec o x)_hi [384,448) and _lo [448,512)

struct Bars {
  uint64_t full[2], empty[2], info_ready[2];
  uint64_t cb_full, eg0_done, xs_ready, yd_full, yd_empty, yo_full, yo_empty, s_full, s_empty,
      hb_full;
};
static_assert(sizeof(Bars) + 8 <= 256, "barrier block");

struct FusedArgs {
  const float* init;
  float* final_state;
  __nv_bfloat16* y;
  WsHeader* hdr;
  int32_t T, R, H, G, ntiles, steps;   // steps = time steps per tile (128 / R)
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         WsHeader* hdr, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    uint64_t t1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (t1 - t0 > kWaitNs) {
      *abort = 1;
      if (hdr) latch_error(hdr, SSD_ERR_TIMEOUT, site);
      return false;
    }
  }
}

// 2^x on the special-function unit (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi): two bf16 terms carry ~16 mantissa bits.
// Packs the pair (a, b) of each into one 32-bit word (a in the low half).
__device__ __forceinline__ void split_pack(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Double-float arithmetic (unevaluated sum hi + lo of two floats), from Knuth's TwoSum: the
// prefix sums of dA reach |cum| ~ 10^3 within a tile, and the mask needs cum_i - cum_j to a
// few float ulps of the difference, not of |cum|.  fp64 is avoided on purpose (very slow here).
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float err = (a - (s - bb)) + (b - bb);
  return {s, err};
}
__device__ __forceinline__ DF df_add(DF x, DF y) {
  DF s = two_sum(x.hi, y.hi);
  const float e = s.lo + x.lo + y.lo;
  const float hi = s.hi + e;
  return {hi, e - (hi - s.hi)};
}
__device__ __forceinline__ DF df_shfl_up(DF v, int off) {
  return {__shfl_up_sync(0xffffffffu, v.hi, off), __shfl_up_sync(0xffffffffu, v.lo, off)};
}

__global__ void __launch_bounds__(kThreadsFused, 1)
    ssd_fused_bf16_kernel(FusedArgs a, const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_b,
                          const __grid_constant__ CUtensorMap tm_c,
                          const __grid_constant__ CUtensorMap tm_da) {
  // The dynamic shared window is declared 1024-byte aligned (required by the 128-byte swizzle
  // atoms) and addressed directly, so every access stays a shared-memory access.
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  TileInfo* info = reinterpret_cast<TileInfo*>(smem + kOffInfo);
  uint32_t& s_tmem = *reinterpret_cast<uint32_t*>(smem + kOffBar + sizeof(Bars));
  int& s_abort = *reinterpret_cast<int*>(smem + kOffBar + sizeof(Bars) + 4);
  if ((smem_u32(smem) & 1023u) != 0) {   // never expected; refuse rather than mis-swizzle
    if (threadIdx.x == 0 && a.hdr) latch_error(a.hdr, SSD_ERR_CUDA, 99);
    return;
  }

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int seq = blockIdx.x;                 // (b, h)
  const int b = seq / a.H, h = seq % a.H;
  const int g = h / (a.H / a.G);
  const int R = a.R, steps = a.steps, nt = a.ntiles;
  const int row_base = b * a.T * R;           // fused row of (b, t=0, r=0)
  volatile int* abort = &s_abort;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 5);        // MMA commit + the four state-group warps
      mbar_init(&bars->info_ready[s], 1);
    }
    mbar_init(&bars->cb_full, 1);
    mbar_init(&bars->eg0_done, 4);
    mbar_init(&bars->xs_ready, 4);
    mbar_init(&bars->yd_full, 1);
    mbar_init(&bars->yd_empty, 4);
    mbar_init(&bars->yo_full, 1);
    mbar_init(&bars->yo_empty, 4);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_empty, 4);
    mbar_init(&bars->hb_full, 4);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
    tma_prefetch_desc(&tm_da);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (warp)
    const uint32_t tx = kXBytes + 2 * kBCBytes + 16u * steps;
    for (int t = 0; t < nt; ++t) {
      const int s = t & 1;
      if (t >= 2 && !wait_bar(&bars->empty[s], ((t - 2) >> 1) & 1, abort, a.hdr, 1)) break;
      mbar_arrive_expect_tx_elect(&bars->full[s], tx);
      const int row = row_base + t * kTileRows;
      tma_load_3d_elect(smem + kOffX + s * kXBytes, &tm_x, &bars->full[s], 0, h, row);
      tma_load_3d_elect(smem + kOffB + s * kBCBytes, &tm_b, &bars->full[s], 0, g, row);
      tma_load_3d_elect(smem + kOffB + s * kBCBytes + kBCBytes / 2, &tm_b, &bars->full[s], 64, g,
                        row);
      tma_load_3d_elect(smem + kOffC + s * kBCBytes, &tm_c, &bars->full[s], 0, g, row);
      tma_load_3d_elect(smem + kOffC + s * kBCBytes + kBCBytes / 2, &tm_c, &bars->full[s], 64, g,
                        row);
      tma_load_2d_elect(smem + kOffDA + s * kDABytes, &tm_da, &bars->full[s], h & ~3,
                        b * a.T + t * steps);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (warp)
    // Per tile t the issue order is  Yd_t, CB_{t+1}, Yo_t, K3_t.  CB_{t+1} overwrites the TMEM
    // columns that Yd_t reads as its A operand; MMAs issued by one thread execute in order.
    const uint32_t id_cb = idesc_bf16(128, 128, 0, 0);
    const uint32_t id_yd = idesc_bf16(128, 64, 0, 1);
    const uint32_t id_k3 = idesc_bf16(128, 128, 1, 1);
    const uint32_t id_yo = idesc_bf16(128, 128, 0, 1);
    const uint32_t sXlo = smem_u32(smem + kOffXlo);
    const uint32_t sHhi = smem_u32(smem + kOffHhi);
    auto issue_cb = [&](int t) {
      const int s = t & 1;
      const uint32_t sB = smem_u32(smem + kOffB + s * kBCBytes);
      const uint32_t sC = smem_u32(smem + kOffC + s * kBCBytes);
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * (kBCBytes / 2) + (ks & 3) * 32;
        mma_bf16_elect(tmem + kColCB, sdesc_sw128(sC + off, 0, 1024),
                       sdesc_sw128(sB + off, 0, 1024), id_cb, ks > 0);
      }
      mma_commit_elect(&bars->cb_full);
    };
    bool ok = wait_bar(&bars->full[0], 0, abort, a.hdr, 2);
    if (ok) issue_cb(0);
    for (int t = 0; ok && t < nt; ++t) {
      const int s = t & 1;
      const uint32_t sB = smem_u32(smem + kOffB + s * kBCBytes);
      const uint32_t sC = smem_u32(smem + kOffC + s * kBCBytes);
      const uint32_t sX = smem_u32(smem + kOffX + s * kXBytes);
      // Yd = (L o CB)_hi x + (L o CB)_lo x   (A from TMEM; K = 2 x 128)
      if (!wait_bar(&bars->eg0_done, t & 1, abort, a.hdr, 3)) break;
      if (t >= 1 && !wait_bar(&bars->yd_empty, (t - 1) & 1, abort, a.hdr, 4)) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {
        const uint32_t acol = (ks < 8 ? kColCB : kColMlo) + (ks & 7) * 8;
        mma_bf16_ts_elect(tmem + kColYd, tmem + acol, sdesc_sw128(sX + (ks & 7) * 2048, 0, 1024),
                          id_yd, ks > 0);
      }
      mma_commit_elect(&bars->yd_full);
      // CB of the next tile
      if (t + 1 < nt) {
        if (!wait_bar(&bars->full[(t + 1) & 1], ((t + 1) >> 1) & 1, abort, a.hdr, 5)) break;
        issue_cb(t + 1);
      }
      // Yo = C [h_hi | h_lo]   (N = 128: the two halves are summed by the state group)
      if (!wait_bar(&bars->hb_full, t & 1, abort, a.hdr, 7)) break;
      if (t >= 1 && !wait_bar(&bars->yo_empty, (t - 1) & 1, abort, a.hdr, 8)) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t offa = (ks >> 2) * (kBCBytes / 2) + (ks & 3) * 32;
        mma_bf16_elect(tmem + kColYo, sdesc_sw128(sC + offa, 0, 1024),
                       sdesc_sw128(sHhi + ks * 2048, kOffHlo - kOffHhi, 1024), id_yo, ks > 0);
      }
      mma_commit_elect(&bars->yo_full);
      // K3: S^T = B^T [(dec o x)_hi | (dec o x)_lo]   (A = B as MN-major: M = state index)
      if (!wait_bar(&bars->xs_ready, t & 1, abort, a.hdr, 10)) break;
      if (t >= 1 && !wait_bar(&bars->s_empty, (t - 1) & 1, abort, a.hdr, 6)) break;
      tc_fence_after();
      const uint32_t lbo_x = sXlo - sX;   // distance from the hi block (in place of x) to lo
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma_bf16_elect(tmem + kColS, sdesc_sw128(sB + ks * 2048, kBCBytes / 2, 1024),
                       sdesc_sw128(sX + ks * 2048, lbo_x, 1024), id_k3, ks > 0);
      }
      mma_commit_elect(&bars->s_full);
      if (t + 2 < nt) mma_commit_elect(&bars->empty[s]);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------------ mask group (warps 2-5)
    const int q = warp & 3;                 // TMEM lane quarter
    const int i = q * 32 + lane;            // tile row owned by this thread
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    for (int t = 0; t < nt; ++t) {
      const int s = t & 1;
      if (!wait_bar(&bars->full[s], (t >> 1) & 1, abort, a.hdr, 11)) break;
      TileInfo& ti = info[s];
      // K1: tile-local inclusive cumsum of dA over `steps` time steps (warp 2 only), in
      // double-float, stored per fused row (expanded over the R ranks of each step)
      if (warp == 2) {
        const float* dA = reinterpret_cast<const float*>(smem + kOffDA + s * kDABytes);
        const int per = (steps + 31) / 32;
        const int beg = min(steps, lane * per), end = min(steps, beg + per);
        DF sum = {0.f, 0.f};
        for (int k = beg; k < end; ++k) sum = df_add(sum, DF{dA[k * 4 + (h & 3)], 0.f});
        DF incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const DF v = df_shfl_up(incl, off);
          if (lane >= off) incl = df_add(incl, v);
        }
        const DF last = {__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
        DF acc = df_shfl_up(incl, 1);   // exclusive prefix of this lane's first step
        if (lane == 0) acc = DF{0.f, 0.f};
        for (int k = beg; k < end; ++k) {
          acc = df_add(acc, DF{dA[k * 4 + (h & 3)], 0.f});
          const float c = acc.hi + acc.lo;
          const float d = (last.hi - acc.hi) + (last.lo - acc.lo);
          // log2-scaled copy for the mask: (hi, lo) * log2(e) as a double-float
          const float l2e = 1.4426950408889634f;
          const float chi = acc.hi * l2e;
          const float clo = fmaf(acc.hi, l2e, -chi) + acc.lo * l2e;
          const float ec = exp2f(c * l2e), ed = exp2f(d * l2e);
          for (int r = 0; r < R; ++r) {
            const int j = k * R + r;
            ti.cum_hi[j] = chi;
            ti.cum_lo[j] = clo;
            ti.expcum[j] = ec;
            ti.dec[j] = ed;
          }
        }
        if (lane == 0) ti.etile = exp2f((last.hi + last.lo) * 1.4426950408889634f);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->info_ready[s]);
      } else if (!wait_bar(&bars->info_ready[s], (t >> 1) & 1, abort, a.hdr, 12)) {
        break;
      }
      // mask: (L o CB)[i][j] = exp(cum[i/R] - cum[j/R]) CB[i][j] for j/R <= i/R, else 0,
      // split into bf16 hi + lo and written back to TMEM as the A operand of Yd
      if (!wait_bar(&bars->cb_full, t & 1, abort, a.hdr, 13)) break;
      tc_fence_after();
      // row i may see columns j < jlim (steps up to its own); the warp needs columns < ncols
      const int jlim = (i / R + 1) * R;
      const int ncols = min(kTileRows, ((q * 32 + 31) / R + 1) * R);
      const float chi = ti.cum_hi[i], clo = ti.cum_lo[i];
#pragma unroll 1
      for (int h0 = 0; h0 < kTileRows; h0 += 32) {
        float v[32];
        if (h0 < ncols) {
          tmem_ld32(tmem + lane_addr + kColCB + h0, v);
          tmem_ld_wait();
        }
#pragma unroll
        for (int c = 0; c < 32; c += 16) {
          const int c0 = h0 + c;
          uint32_t hi[8], lo[8];
          if (c0 >= ncols) {
#pragma unroll
            for (int k = 0; k < 8; ++k) hi[k] = lo[k] = 0u;
          } else {
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
              const int j = c0 + k;
              const float2 ch = *reinterpret_cast<const float2*>(&ti.cum_hi[j]);
              const float2 cl = *reinterpret_cast<const float2*>(&ti.cum_lo[j]);
              // mask before the exponential: future columns get exponent -inf (-> 0)
              const float e0 = (j < jlim) ? (chi - ch.x) + (clo - cl.x) : -INFINITY;
              const float e1 = (j + 1 < jlim) ? (chi - ch.y) + (clo - cl.y) : -INFINITY;
              split_pack(ex2_approx(e0) * v[c + k], ex2_approx(e1) * v[c + k + 1], hi[k / 2],
                         lo[k / 2]);
            }
          }
          // columns [c0/2, c0/2+8) were read in this or an earlier step: safe to overwrite
          tmem_st8(tmem + lane_addr + kColCB + c0 / 2, hi);
          tmem_st8(tmem + lane_addr + kColMlo + c0 / 2, lo);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->eg0_done);
      // dec o x, split: hi in place of x (after Yd_t has read x), lo in its own buffer
      if (!wait_bar(&bars->yd_full, t & 1, abort, a.hdr, 14)) break;
      {
        const float w = ti.dec[i];
        uint8_t* xrow = smem + kOffX + s * kXBytes;
        uint8_t* xlo = smem + kOffXlo;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint32_t off = sw128_off16(i, ch * 8);
          uint4* p = reinterpret_cast<uint4*>(xrow + off);
          const uint4 u = *p;
          const float2 f0 = unpack_bf16(u.x), f1 = unpack_bf16(u.y), f2 = unpack_bf16(u.z),
                       f3 = unpack_bf16(u.w);
          uint4 uh, ul;
          split_pack(f0.x * w, f0.y * w, uh.x, ul.x);
          split_pack(f1.x * w, f1.y * w, uh.y, ul.y);
          split_pack(f2.x * w, f2.y * w, uh.z, ul.z);
          split_pack(f3.x * w, f3.y * w, uh.w, ul.w);
          *p = uh;
          *reinterpret_cast<uint4*>(xlo + off) = ul;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->xs_ready);
    }
  } else {
    // ------------------------------------------------------------------ state group (warps 6-9)
    const int q = warp & 3;
    const int n = q * 32 + lane;            // state row (and output row) owned by this thread
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    float hst[kP];
    const size_t st_base = (size_t)seq * kP * kN;
#pragma unroll
    for (int p = 0; p < kP; ++p) hst[p] = a.init ? a.init[st_base + (size_t)p * kN + n] : 0.f;
    uint8_t* hbhi = smem + kOffHhi;
    uint8_t* hblo = smem + kOffHlo;
    auto write_hb = [&]() {
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint4 uh, ul;
        split_pack(hst[ch * 8 + 0], hst[ch * 8 + 1], uh.x, ul.x);
        split_pack(hst[ch * 8 + 2], hst[ch * 8 + 3], uh.y, ul.y);
        split_pack(hst[ch * 8 + 4], hst[ch * 8 + 5], uh.z, ul.z);
        split_pack(hst[ch * 8 + 6], hst[ch * 8 + 7], uh.w, ul.w);
        const uint32_t off = sw128_off16(n, ch * 8);
        *reinterpret_cast<uint4*>(hbhi + off) = uh;
        *reinterpret_cast<uint4*>(hblo + off) = ul;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->hb_full);
    };
    write_hb();
    for (int t = 0; t < nt; ++t) {
      const int s = t & 1;
      TileInfo& ti = info[s];
      // output: y = Yd + exp(cum[i/R]) (Yo_hi + Yo_lo)
      if (!wait_bar(&bars->yo_full, t & 1, abort, a.hdr, 21)) break;
      if (!wait_bar(&bars->yd_full, t & 1, abort, a.hdr, 22)) break;
      tc_fence_after();
      const float sc = ti.expcum[n];
      __nv_bfloat16* yrow = a.y + ((size_t)(row_base + t * kTileRows + n) * a.H + h) * kP;
#pragma unroll 1
      for (int c = 0; c < kP; c += 16) {
        float vd[16], vh[16], vl[16];
        tmem_ld16(tmem + lane_addr + kColYd + c, vd);
        tmem_ld16(tmem + lane_addr + kColYo + c, vh);
        tmem_ld16(tmem + lane_addr + kColYo + 64 + c, vl);
        tmem_ld_wait();
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          pk[k] = pack_bf16(fmaf(sc, vh[2 * k] + vl[2 * k], vd[2 * k]),
                            fmaf(sc, vh[2 * k + 1] + vl[2 * k + 1], vd[2 * k + 1]));
        uint4* dst = reinterpret_cast<uint4*>(yrow + c);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->yd_empty);
        mbar_arrive(&bars->yo_empty);
      }
      // K4: h <- exp(cum_last) h + S_hi + S_lo
      if (!wait_bar(&bars->s_full, t & 1, abort, a.hdr, 20)) break;
      tc_fence_after();
      const float e = ti.etile;
#pragma unroll
      for (int c = 0; c < kP; c += 16) {
        float sh[16], sl[16];
        tmem_ld16(tmem + lane_addr + kColS + c, sh);
        tmem_ld16(tmem + lane_addr + kColS + 64 + c, sl);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) hst[c + k] = fmaf(e, hst[c + k], sh[k] + sl[k]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->s_empty);
        if (t + 2 < nt) mbar_arrive(&bars->empty[s]);
      }
      if (t + 1 < nt) write_hb();   // Yo_t has already consumed h_in(t) (yo_full waited above)
    }
    if (a.final_state && !*abort) {
#pragma unroll
      for (int p = 0; p < kP; ++p) a.final_state[st_base + (size_t)p * kN + n] = hst[p];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t rank, const void* base,
              const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
              CUtensorMapSwizzle sw) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, rank, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fused_bf16_supported(int64_t T, int64_t H, int64_t P, int64_t N, int64_t R, int64_t l,
                          bool bf16, bool theta) {
  if (!bf16 || theta) return false;
  if (P != kP || N != kN) return false;
  if (R < 1 || R > 32 || (kTileRows % R) != 0) return false;
  if (H % 4 != 0) return false;                      // dA tile loads use 16-byte boxes
  if ((T * R) % kTileRows != 0) return false;
  (void)l;
  return true;
}

cudaError_t fused_bf16_forward(const GenericParams& p, cudaStream_t st) {
  const int64_t rows = p.batch * p.T * p.R;
  CUtensorMap mx, mb, mc, mda;
  {
    cuuint64_t dims[3] = {(cuuint64_t)p.P, (cuuint64_t)p.H, (cuuint64_t)rows};
    cuuint64_t str[2] = {(cuuint64_t)p.P * 2, (cuuint64_t)p.H * p.P * 2};
    cuuint32_t box[3] = {64, 1, kTileRows};
    if (!make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.x, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.G, (cuuint64_t)rows};
    cuuint64_t str[2] = {(cuuint64_t)p.N * 2, (cuuint64_t)p.G * p.N * 2};
    cuuint32_t box[3] = {64, 1, kTileRows};
    if (!make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.B, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (!make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.C, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const int steps = (int)(kTileRows / p.R);
  {
    cuuint64_t dims[2] = {(cuuint64_t)p.H, (cuuint64_t)(p.batch * p.T)};
    cuuint64_t str[1] = {(cuuint64_t)p.H * 4};
    cuuint32_t box[2] = {4, (cuuint32_t)steps};
    if (!make_map(&mda, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.dA, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  FusedArgs a;
  a.init = p.init;
  a.final_state = p.final_state;
  a.y = static_cast<__nv_bfloat16*>(p.y);
  a.hdr = p.hdr;
  a.T = (int32_t)p.T;
  a.R = (int32_t)p.R;
  a.H = (int32_t)p.H;
  a.G = (int32_t)p.G;
  a.ntiles = (int32_t)(p.T * p.R / kTileRows);
  a.steps = steps;
  cudaError_t e = cudaFuncSetAttribute(ssd_fused_bf16_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  ssd_fused_bf16_kernel<<<(unsigned)(p.batch * p.H), kThreadsFused, kSmemAlloc, st>>>(a, mx, mb,
                                                                                     mc, mda);
  return cudaGetLastError();
}

}  // namespace ssd
