// Fused tcgen05/TMEM chunked SSD forward for bf16 I/O (sm_103a).
//
// One CTA owns one (batch, head) sequence (or a time segment of one) and walks it in tiles of
// 128 rank-fused rows (fused row i = t*R + r, as in the serial.rs page's K2 reshape), carrying
// the state on chip from tile to tile, so the inter-chunk state of K4 never goes to HBM.  Per
// tile:
//   K1  tile-local inclusive cumsum of dA (fp32 over warp shuffles), decay factors
//   K2  CB = C B^T                                       tcgen05.mma, both from shared memory
//   K5a (L o CB), L[i,j] = exp(cum[i/R] - cum[j/R]) for j/R <= i/R else 0, split into bf16
//       hi + lo and written back to TMEM;  Yd = (L o CB) x     tcgen05.mma, A from TMEM
//   K3  S^T = B^T (dec o x), dec_i = exp(cum_last - cum[i/R]), (dec o x) split hi + lo
//   K5b Yo = C h_in, h_in split hi + lo;  y = Yd + exp(cum[i/R]) Yo -> bf16 -> TMA store
//   K4  h_out = exp(cum_last) h_in + S^T in fp32 registers of the state warps
// The serial.rs page runs K1..K5 per chunk with the K4 loop across chunks; a 128-row tile is a
// sub-block of a chunk, and the part of a chunk's 1-semiseparable mask below a tile's diagonal
// block has rank one (exp(cum_i - cum_j) = exp(cum_i) exp(-cum_j)), which is exactly what the
// tile-boundary state carries.  The result is the same recurrence for every chunk_len.
// Inside a tile the same structure is used once more: below the diagonal 32 x 32 blocks of L
// are rank one, L[i,j] = exp(cum_i - cum_ref) exp(cum_ref - cum_j) with cum_ref taken at the
// end of the column block, so only the diagonal blocks need one exponential per element.
//
// Operands that are products of inputs ((L o CB), dec o x and h_in) are carried as two bf16
// terms (hi + lo, ~16 mantissa bits): one bf16 rounding of them is far too coarse for the
// 2e-2 (1 + |y|) bound when decay is slow and y cancels.  Products of two bf16 inputs are exact
// in the fp32 accumulators.  Every wait is bounded; a wait that gives up latches
// SSD_ERR_TIMEOUT in the workspace header and the CTA stops issuing work, drains the TMA loads
// and MMAs it issued, and frees its TMEM.
//
// Ragged sequences: when seqlen * R is not a multiple of 128 the last tile is partial.  The
// tensor maps carry the batch as their own dimension, so TMA fills the rows past the end of a
// sequence with zeros (x = B = C = 0), K1 reads dA = 0 there, and the TMA store writes no y
// there: zero padding, which leaves y of the real steps and the final state unchanged.
//
// Time segments: with fewer sequences than SMs, each sequence is cut into segments run by
// separate CTAs.  The same kernel in its state-only form (kPre: K1, dec o x, K3 and K4; no C,
// CB, mask, Yd, Yo or output) gives the end states of pieces of the sequence before its last
// segment, fused_seg_carry_kernel chains them into every segment's true initial state, and the
// full form then runs all segments in parallel, writing every y once.  The state-only pieces
// are a whole number of times shorter than the segments, so that this pass, which costs about a
// third of the full one per tile, still fills the SMs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "fp_helpers.cuh"
#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {

namespace {

using namespace tc;
using namespace fp;

constexpr int kTileRows = 128;
constexpr int kP = 64;
constexpr int kN = 128;
constexpr long long kWaitCycles = 4000000000ll;   // per wait before giving up (~2 s at 2 GHz)
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kXBytes = kTileRows * kP * 2;          // 16 KB per stage
constexpr uint32_t kBCBytes = kTileRows * kN * 2;         // 32 KB per stage (two 64-col blocks)
constexpr int kInfoSlots = 4;                             // K1 runs up to this many tiles ahead
struct TileInfo {
  float cum_hi[kTileRows];   // log2-scaled prefix sum of dA at fused row j
  float qf[kTileRows];       // exp(cum_ref(block of j) - cum_j) (times w_j), cum_ref at the
                             // block's end
  float w[kTileRows];        // write weight of fused row j (with per-row weights only)
  float last_hi;             // log2-scaled total of the tile
  float etile;               // exp(cum_last)
  int monotone;              // 1 if every dA of the tile is <= 0 (factorized mask is safe)
  float pad[29];
};
// the rows are read as float4 from every slot of the ring
static_assert(sizeof(TileInfo) % 16 == 0, "TileInfo slots must keep 16-byte alignment");
constexpr uint32_t kTmemCols = 512;

struct FusedArgs {
  const float* dA;
  const float* init;
  float* final_state;
  __nv_bfloat16* y;
  WsHeader* hdr;
  int32_t T, R, H, G, ntiles, steps;   // steps = time steps per tile (128 / R)
  // Time segments: each (batch, head) sequence is cut into nseg segments of seg_tiles tiles
  // (the last may be shorter), each run by its own CTA.  The state-only pre-pass cuts the
  // tiles before the last segment into npre pieces of pre_tiles tiles (pre_tiles divides
  // seg_tiles) and writes each piece's end state (from the true initial state for piece 0,
  // from zero otherwise) to seg_end and its decay exp(sum dA) to seg_decay; a carry pass chains
  // them into the true initial state of every segment (seg_init).
  int32_t nseg, seg_tiles, npre, pre_tiles;
  const float* seg_init;   // [b*H*nseg][P][N] (segment 0 unused: it starts from init)
  float* seg_end;          // [b*H*npre][P][N]
  float* seg_decay;        // [b*H*npre]
  // Per-sequence valid lengths [batch] (device, may be null): steps from valid_len[b] on are
  // padding.  Tiles wholly inside it are not run (a segment past the end still runs one, so
  // that it hands its state through); in the tile that straddles the end, K1 reads zero decay,
  // the pad rows of x and B are zeroed in shared memory before any product reads them (so any
  // pad contents, NaN included, stay out of the result) and y is stored for real rows only.
  const int64_t* valid_len;
  // Per fused row write weights [b][T * R][H] (device, may be null): row i's write x_i (x) B_i
  // enters the state and every later output scaled by w_i.  They are folded into the column
  // factors of the mask and into (dec o x), so x and B stay exact bf16 operands (the
  // trapezoidal form runs on this kernel this way, its gamma and beta as the weights).
  const float* wrow;
  // element counts of the outputs (index checks of the debug build)
  int64_t y_elems, st_elems, seqs;
};

// The loop of a wait that did not complete at once, kept out of line: the kernels wait at many
// sites, and inlining this at each of them multiplies the code the warps must fetch.
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           WsHeader* hdr, int site) {
  // bounded in cycles of this SM's clock, which only moves forward
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort = 1;
      if (hdr) latch_error(hdr, SSD_ERR_TIMEOUT, site);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         WsHeader* hdr, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, abort, hdr, site);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi): two bf16 terms carry ~16 mantissa bits.
// Packs the pair (v.x, v.y) of each into one 32-bit word (v.x in the low half).
__device__ __forceinline__ void split2(float2 v, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(v.x, v.y);
  const float2 r = sub2(v, unpack_bf16(hi));
  lo = pack_bf16(r.x, r.y);
}

// One 32-column block cb of the masked operand for the calling thread's row (w = its CB
// values): below the diagonal block and with a monotone tile the factorized form
// exp(cum_i - cum_ref) * qf_j, else one exponential per element with the causal cut at jlim.
template <bool kW>
__device__ __forceinline__ void mask_block(const TileInfo& ti, int cb, bool exact, float chi,
                                           int jlim, const float (&w)[32],
                                           uint32_t (&hi)[16], uint32_t (&lo)[16]) {
  if (!exact) {
    const int ref = cb * 32 + 31;
    const float r = ex2_approx(chi - ti.cum_hi[ref]);
    const float2 rr = make_float2(r, r);
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
      const float4 qq = *reinterpret_cast<const float4*>(&ti.qf[cb * 32 + k]);
      split2(mul2(make_float2(w[k], w[k + 1]), mul2(make_float2(qq.x, qq.y), rr)), hi[k / 2],
             lo[k / 2]);
      split2(mul2(make_float2(w[k + 2], w[k + 3]), mul2(make_float2(qq.z, qq.w), rr)),
             hi[k / 2 + 1], lo[k / 2 + 1]);
    }
  } else {
    const float2 ch2 = make_float2(chi, chi);
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
      const int j = cb * 32 + k;
      const float4 ch = *reinterpret_cast<const float4*>(&ti.cum_hi[j]);
      const float2 e0 = sub2(ch2, make_float2(ch.x, ch.y));
      const float2 e1 = sub2(ch2, make_float2(ch.z, ch.w));
      // future columns (j >= jlim) are cut after the exponential, which may overflow there
      float2 l0 = make_float2(j < jlim ? ex2_approx(e0.x) : 0.f,
                              j + 1 < jlim ? ex2_approx(e0.y) : 0.f);
      float2 l1 = make_float2(j + 2 < jlim ? ex2_approx(e1.x) : 0.f,
                              j + 3 < jlim ? ex2_approx(e1.y) : 0.f);
      if constexpr (kW) {   // the column's write weight
        const float4 wj = *reinterpret_cast<const float4*>(&ti.w[j]);
        l0 = mul2(l0, make_float2(wj.x, wj.y));
        l1 = mul2(l1, make_float2(wj.z, wj.w));
      }
      split2(mul2(make_float2(w[k], w[k + 1]), l0), hi[k / 2], lo[k / 2]);
      split2(mul2(make_float2(w[k + 2], w[k + 3]), l1), hi[k / 2 + 1], lo[k / 2 + 1]);
    }
  }
}

// K1 for one warp: reads dA straight from global memory (one tile ahead, into registers) and
// publishes each tile's prefix sums and decay factors into a ring of kInfoSlots slots.
template <bool kW>
__device__ __forceinline__ void k1_warp(const FusedArgs& a, TileInfo* info, uint64_t* info_ready,
                                        uint64_t* info_empty, volatile int* abort, int b, int h,
                                        int tbase, int nt, int Tb, int lane) {
  const int R = a.R, steps = a.steps;
  const int per = (steps + 31) / 32;                 // steps per lane (<= 4)
  const int beg = min(steps, lane * per), end = min(steps, beg + per);
  const float* dsrc = a.dA + ((size_t)b * a.T + (size_t)tbase * steps) * a.H + h;
  float dnext[4];
  auto load_tile = [&](int t) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      dnext[k] = (beg + k < end && (tbase + t) * steps + beg + k < Tb)
                     ? __ldg(dsrc + (size_t)(t * steps + beg + k) * a.H)
                     : 0.f;
  };
  // per-row write weights: rows lane + 32 k of the tile, one tile ahead
  const float* wsrc = kW ? a.wrow + (size_t)b * a.T * R * a.H + h : nullptr;
  float wnext[4], wcur[4];
  auto load_w = [&](int t) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = (tbase + t) * kTileRows + lane + 32 * k;
      wnext[k] = row < Tb * R ? __ldg(wsrc + (size_t)row * a.H) : 0.f;
    }
  };
  load_tile(0);
  if constexpr (kW) load_w(0);
  for (int t = 0; t < nt; ++t) {
    float dcur[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) dcur[k] = dnext[k];
    if (t + 1 < nt) load_tile(t + 1);
    if constexpr (kW) {
#pragma unroll
      for (int k = 0; k < 4; ++k) wcur[k] = wnext[k];
      if (t + 1 < nt) load_w(t + 1);
    }
    // fp32 prefix sums: within a 128-row tile |cum| stays far below the range where fp32
    // rounding would show at the bf16 output's precision
    float sum = 0.f;
    int pos = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      pos |= (dcur[k] > 0.f);
      sum += dcur[k];
    }
    float incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const float last = __shfl_sync(0xffffffffu, incl, 31);
    float acc = __shfl_up_sync(0xffffffffu, incl, 1);   // exclusive prefix of the lane's first step
    if (lane == 0) acc = 0.f;
    const int monotone = __all_sync(0xffffffffu, pos == 0);
    const int slot = t % kInfoSlots;
    if (t >= kInfoSlots &&
        !wait_bar(&info_empty[slot], ((t - kInfoSlots) / kInfoSlots) & 1, abort, a.hdr, 11))
      break;
    TileInfo& ti = info[slot];
    float chv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc += dcur[k];   // dcur is 0 past the lane's steps
      chv[k] = acc * kLog2e;
    }
    // with R in {1, 2, 4} the lane's steps cover exactly the rows 4 lane .. 4 lane + 3 (row
    // 4 lane + m belongs to the lane's step m / R): one 16-byte store
    const bool quad = R == 1 || R == 2 || R == 4;
    float4 c4 = make_float4(chv[0], chv[0], chv[0], chv[0]);
    if (R == 1) c4 = make_float4(chv[0], chv[1], chv[2], chv[3]);
    if (R == 2) c4 = make_float4(chv[0], chv[0], chv[1], chv[1]);
    if (quad) {
      *reinterpret_cast<float4*>(&ti.cum_hi[4 * lane]) = c4;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (beg + k < end)
          for (int r = 0; r < R; ++r) ti.cum_hi[(beg + k) * R + r] = chv[k];
    }
    if (lane == 0) {
      const float lhi = last * kLog2e;
      ti.last_hi = lhi;
      ti.etile = ex2_approx(lhi);
      ti.monotone = monotone;
    }
    // qf of the rank-one blocks: the reference of column block c is its last fused row
    if (!kW && quad) {
      // the reference row 32 (lane / 8) + 31 of the lane's rows is row 3 of lane 8 (lane / 8) + 7
      const float cref = __shfl_sync(0xffffffffu, c4.w, (lane & ~7) | 7);
      *reinterpret_cast<float4*>(&ti.qf[4 * lane]) =
          make_float4(ex2_approx(cref - c4.x), ex2_approx(cref - c4.y), ex2_approx(cref - c4.z),
                      ex2_approx(cref - c4.w));
    } else if constexpr (kW) {   // times the column's write weight
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = lane + 32 * k;
        const int ref = (e >> 5) * 32 + 31;
        ti.qf[e] = wcur[k] * ex2_approx(ti.cum_hi[ref] - ti.cum_hi[e]);
        ti.w[e] = wcur[k];
      }
    } else {
      __syncwarp();
#pragma unroll
      for (int e = lane; e < kTileRows; e += 32) {
        const int ref = (e >> 5) * 32 + 31;
        ti.qf[e] = ex2_approx(ti.cum_hi[ref] - ti.cum_hi[e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&info_ready[slot]);
  }
}

// ============================================================================================
// Full forward pass (one CTA per (batch, head) sequence or time segment of one).
//
// Per 128-row tile t the tensor core runs, in this order,
//   Yo_t     = C_t h_t^T                      A = C_t (TMEM), B = [h_hi ; h_lo]   (K = 2 x 128)
//   K3_t     = B_t^T [(dec o x)_hi ; lo]      A = B_t (MN-major smem)             (K = 2 x 128)
//   CB_{t+1} = C_{t+1} B_{t+1}^T              both K-major in smem, into mask buffer (t+1) & 1
//   Yd_t    += (L o CB)_t x_t                 A = (L o CB) hi/lo (TMEM)           (K = 2 x 128)
// where Yd_t starts from e^{cum_i} Yo_t, written into its accumulator by the out warps, so y_t
// is one accumulator.  The mask of tile t+1 is computed while Yd_t, Yo_{t+1} and K3_{t+1} run
// (two mask buffers), which gives the element-wise mask about one tile of tensor work to hide
// behind.  The CUDA cores, around the tensor core:
//   state warps  h_{t+1} = e^{cum_last} h_t + S_t in registers (the K4 step, fp32), written as
//                bf16 hi/lo rows for Yo_{t+1}; the state never leaves the SM
//   mask warps   (dec o x)_t into its own buffer, then the mask of tile t in place over CB_t
//   out warps    e^{cum_i} Yo_t into the Yd accumulator; C_{t+1} from its shared-memory tile
//                into TMEM; y_t -> bf16 -> the tile's x slot -> TMA store
// The state recurrence never passes through the tensor core (K3 starts from zero).
//
// kPre = true is the state-only pre-pass of a sequence cut into time segments: per tile only
// K1, (dec o x), K3 and the state step (no C, CB, mask, Yo, Yd or y).  Piece j (of the npre
// pieces that cover the first nseg - 1 segments) runs from the true initial state when j = 0 and
// from zero otherwise, and writes its end state and its decay product exp(sum dA);
// fused_seg_carry_kernel turns those into every segment's true initial state for the full pass.
// ============================================================================================

constexpr int kThreads = 512;
constexpr int kXSlots = 3;                                  // x ring (a slot also stages y_t)
constexpr uint32_t kOffX = 0;
constexpr uint32_t kOffB = kOffX + kXSlots * kXBytes;        // two B stages
constexpr uint32_t kOffC = kOffB + 2 * kBCBytes;             // one C slot (copied into TMEM)
constexpr uint32_t kOffDxHi = kOffC + kBCBytes;              // (dec o x) hi  [rows][P]
constexpr uint32_t kOffDxLo = kOffDxHi + kXBytes;            // (dec o x) lo
constexpr uint32_t kOffHHi = kOffDxLo + kXBytes;             // h^T hi [N rows][P]
constexpr uint32_t kOffHLo = kOffHHi + kXBytes;              // h^T lo
constexpr uint32_t kOffInfo = kOffHLo + kXBytes;
constexpr uint32_t kOffBar = kOffInfo + kInfoSlots * sizeof(TileInfo);
constexpr uint32_t kSmem = kOffBar + 512;
static_assert(kSmem <= 232448, "exceeds the 227 KB shared-memory limit per CTA");
static_assert(kOffInfo % 1024 == 0, "operand buffers must stay 1024-byte aligned");

// TMEM columns (128 lanes x 512 columns of 32 bit)
constexpr uint32_t kColM = 0;      // two buffers of 128: CB fp32, rewritten as (L o CB) hi/lo
                                   // per 32-column block (16 hi then 16 lo columns)
constexpr uint32_t kColYd = 256;   // y accumulator: e^{cum_i} Yo_t, then + Yd_t
constexpr uint32_t kColYo = 320;   // C h^T
constexpr uint32_t kColS = 384;    // B^T (dec o x) (hi and lo stacked along K)
constexpr uint32_t kColC = 448;    // C: 128 bf16 of the state axis, two per column

// The MMA warp waits on few barriers (a wait costs a few hundred cycles of latency even when its
// phase has completed, and the issuing thread runs only a few MMAs ahead of the tensor core),
// and tests each of them before issuing the product before it:
//   yo_go(t)     state warps wrote h_t; out warps read Yo_{t-1} and copied C_t into TMEM
//   k3_go(t)     (dec o x)_t written; state warps read S_{t-1}
//   c_full, b_full  CB_t reads C_t and B_t straight from shared memory (with valid lengths:
//                cb_go(t), which the out warps arrive on once B_t's pad rows are zero)
//   m_ready[b]   the mask of the tile in mask buffer b is in TMEM
//   y_pre(t)     e^{cum_i} Yo_t written into the y accumulator (after y_{t-1} was read)
// x_t needs no wait of its own: the (dec o x) warps waited for it before arriving on k3_go(t),
// and Yd_t is issued after K3_t.  Barriers whose next phase can complete before a waiter has
// seen the current one (CB_{t+1} and the mask of tile t+1 may both finish before Yd_t is
// issued) come in pairs, one per mask buffer.
struct Bars {
  uint64_t x_full[kXSlots], x_empty[kXSlots], b_full[2], b_empty[2];
  uint64_t c_full, cb_go;
  uint64_t info_ready[kInfoSlots], info_empty[kInfoSlots];
  uint64_t cb_full[2], m_ready[2], yd_full, yo_full, s_full;
  uint64_t yo_go, k3_go, y_pre, drain;
};
static_assert(sizeof(Bars) + 16 <= 512, "barrier block");

// Mask blocks [cb0, cb1) of the tile's rows in quarter q = warp % 4 (the diagonal block q is
// exact, the ones below it factorized), blocks [cb1, zero_end) set to zero.  Five warps share the
// 1 + 2 + 3 + 4 blocks of the causal tile.
struct MaskShare {
  int cb0, cb1, zero_end;
};
__device__ __forceinline__ MaskShare mask_share(int warp) {
  switch (warp) {
    case 4: return {0, 1, 4};
    case 5: return {0, 2, 4};
    case 6: return {0, 3, 4};
    case 7: return {2, 4, 4};
    case 3: return {0, 2, 2};
    default: return {0, 0, 0};
  }
}
constexpr int kMaskWarps = 5;

// (dec o x) work units (32 rows x 16 columns; 16 per tile) of the warps that compute it.  In the
// full pass most go to sub-partition 0 (the least mask work) and none to sub-partition 2 (three
// mask blocks and K1); the pre-pass has no mask, so there the five mask warps share them evenly.
template <bool kPre>
__device__ __forceinline__ int2 dx_units(int warp) {
  if constexpr (kPre) {
    switch (warp) {
      case 4: return make_int2(0, 4);
      case 5: return make_int2(4, 7);
      case 6: return make_int2(7, 10);
      case 7: return make_int2(10, 13);
      case 3: return make_int2(13, 16);
      default: return make_int2(0, 0);
    }
  } else {
    switch (warp) {
      case 4: return make_int2(0, 7);
      case 5: return make_int2(7, 12);
      case 7: return make_int2(12, 14);
      case 3: return make_int2(14, 16);
      default: return make_int2(0, 0);
    }
  }
}
// warps with (dec o x) units (each arrives on k3_go, and in the pre-pass on x_empty)
template <bool kPre>
constexpr int kDxWarps = kPre ? 5 : 4;

template <bool kPre, bool kW>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_fused_bf16_kernel(FusedArgs a, const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_b,
                          const __grid_constant__ CUtensorMap tm_c,
                          const __grid_constant__ CUtensorMap tm_y) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  TileInfo* info = reinterpret_cast<TileInfo*>(smem + kOffInfo);
  uint32_t& s_tmem = *reinterpret_cast<uint32_t*>(smem + kOffBar + sizeof(Bars));
  int& s_abort = *reinterpret_cast<int*>(smem + kOffBar + sizeof(Bars) + 4);
  int& s_keep_tmem = *reinterpret_cast<int*>(smem + kOffBar + sizeof(Bars) + 8);
  if ((smem_u32(smem) & 1023u) != 0) {   // never expected; refuse rather than mis-swizzle
    if (threadIdx.x == 0 && a.hdr) latch_error(a.hdr, SSD_ERR_CUDA, 99);
    return;
  }

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const int nrun = kPre ? a.npre : a.nseg;       // segments (pieces) run per sequence
  const int seq = blockIdx.x / nrun;             // (b, h)
  const int seg = blockIdx.x % nrun;
  const int span = kPre ? a.pre_tiles : a.seg_tiles;
  const int end_tile = kPre ? (a.nseg - 1) * a.seg_tiles : a.ntiles;
  const int b = seq / a.H, h = seq % a.H;
  const int g = h / (a.H / a.G);
  const int R = a.R;
  const int tbase = seg * span;
  const int seg_row = tbase * kTileRows;
  int Tb = a.T;   // real steps of the sequence
  if (a.valid_len) {
    const int64_t v = a.valid_len[b];
    Tb = (int)(v < 0 ? 0 : (v > a.T ? a.T : v));
  }
  const int vrows = Tb * R;   // real fused rows of the sequence
  const int nt = max(1, min(min(end_tile - tbase, span),
                            (vrows - seg_row + kTileRows - 1) / kTileRows));
  // the out warps zero B's pad rows and, in the pre-pass, gate K3 on that
  const bool zero_b = a.valid_len != nullptr;
  volatile int* abort = &s_abort;

  if (threadIdx.x == 0) {
    s_abort = 0;
    s_keep_tmem = 0;
    for (int s = 0; s < kXSlots; ++s) {
      mbar_init(&bars->x_full[s], 1);
      // out warps once their y store has read the slot (the pre-pass: the (dec o x) warps)
      mbar_init(&bars->x_empty[s], kPre ? kDxWarps<true> : 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->b_full[s], 1);
      mbar_init(&bars->b_empty[s], 1);     // a state warp once K3 of the tile is done
      // CB_t done (MMA commit) and C_t held in TMEM (out warps): the mask may start and C_t's
      // shared-memory slot is free
      mbar_init(&bars->cb_full[s], 5);
      mbar_init(&bars->m_ready[s], kMaskWarps);
    }
    mbar_init(&bars->c_full, 1);
    mbar_init(&bars->cb_go, 4);            // out warps: B of the tile landed, pad rows zeroed
    for (int k = 0; k < kInfoSlots; ++k) {
      mbar_init(&bars->info_ready[k], 1);
      mbar_init(&bars->info_empty[k], kPre ? 4 : 8);   // state warps (and out warps)
    }
    mbar_init(&bars->yd_full, 1);
    mbar_init(&bars->yo_full, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->yo_go, 8);            // 4 state warps + 4 out warps
    // (dec o x) warps + 4 state warps (+ 4 out warps zeroing B's pad rows in the pre-pass)
    mbar_init(&bars->k3_go, kDxWarps<kPre> + 4 + (kPre && zero_b ? 4 : 0));
    mbar_init(&bars->y_pre, 4);            // out warps
    mbar_init(&bars->drain, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
    tma_prefetch_desc(&tm_y);
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
    // ------------------------------------------------------------------ TMA producer
    // Per tile: C (one slot, freed once the out warps hold it in registers), B (two stages,
    // freed by K3), x (three slots, freed once y of the tile has been stored from the slot).
    int nc = 0, nb = 0, nx = 0;   // tiles whose C, B, x loads were issued
    for (int t = 0; t < nt; ++t) {
      const int row = seg_row + t * kTileRows;   // rows past the sequence's end read as zeros
      if (!kPre) {   // the pre-pass needs no C
        if (t >= 1 &&
            !wait_bar(&bars->cb_full[(t - 1) & 1], ((t - 1) >> 1) & 1, abort, a.hdr, 31))
          break;
        mbar_arrive_expect_tx_elect(&bars->c_full, kBCBytes);
        tma_load_4d_elect(smem + kOffC, &tm_c, &bars->c_full, 0, g, row, b);
        tma_load_4d_elect(smem + kOffC + kBCBytes / 2, &tm_c, &bars->c_full, 64, g, row, b);
        nc = t + 1;
      }
      const int sb = t & 1;
      if (t >= 2 && !wait_bar(&bars->b_empty[sb], ((t - 2) >> 1) & 1, abort, a.hdr, 32)) break;
      mbar_arrive_expect_tx_elect(&bars->b_full[sb], kBCBytes);
      tma_load_4d_elect(smem + kOffB + sb * kBCBytes, &tm_b, &bars->b_full[sb], 0, g, row, b);
      tma_load_4d_elect(smem + kOffB + sb * kBCBytes + kBCBytes / 2, &tm_b, &bars->b_full[sb], 64,
                        g, row, b);
      nb = t + 1;
      const int sx = t % kXSlots;
      if (t >= kXSlots &&
          !wait_bar(&bars->x_empty[sx], ((t - kXSlots) / kXSlots) & 1, abort, a.hdr, 33))
        break;
      mbar_arrive_expect_tx_elect(&bars->x_full[sx], kXBytes);
      tma_load_4d_elect(smem + kOffX + sx * kXBytes, &tm_x, &bars->x_full[sx], 0, h, row, b);
      nx = t + 1;
      if (t + 3 < nt) {   // pull a later tile into L2 so its load later finds it there
        const int r3 = row + 3 * kTileRows;
        tma_prefetch_l2_4d_elect(&tm_x, 0, h, r3, b);
        tma_prefetch_l2_4d_elect(&tm_b, 0, g, r3, b);
        tma_prefetch_l2_4d_elect(&tm_b, 64, g, r3, b);
        if (!kPre) {
          tma_prefetch_l2_4d_elect(&tm_c, 0, g, r3, b);
          tma_prefetch_l2_4d_elect(&tm_c, 64, g, r3, b);
        }
      }
    }
    // Drain: no TMA load may still be writing this CTA's shared memory when it exits.  In a
    // normal run every load has been waited for by its consumer and these return at once.
    // Slot s of an n-slot ring received the loads of tiles s, s + n, ... below the issued count;
    // waiting for the parity of the last of them covers all of them.
    bool drained = true;
    for (int s = 0; s < kXSlots; ++s) {
      const int k = nx > s ? (nx - 1 - s) / kXSlots + 1 : 0;
      if (k > 0) drained &= mbar_wait_bounded(&bars->x_full[s], (k - 1) & 1, 2000000000ull);
    }
    for (int s = 0; s < 2; ++s) {
      const int k = nb > s ? (nb - 1 - s) / 2 + 1 : 0;
      if (k > 0) drained &= mbar_wait_bounded(&bars->b_full[s], (k - 1) & 1, 2000000000ull);
    }
    if (nc > 0) drained &= mbar_wait_bounded(&bars->c_full, (nc - 1) & 1, 2000000000ull);
    if (!drained && lane == 0 && a.hdr) latch_error(a.hdr, SSD_ERR_TIMEOUT, 91);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and one elected lane issues each MMA; descriptors are
    // precomputed 32-bit words plus constant offsets (a start-address step of s bytes adds
    // s >> 4 to the low word).
    constexpr uint32_t id_cb = idesc_bf16(128, 128, 0, 0);   // TS: A = C, B = B tile K-major
    constexpr uint32_t id_n64 = idesc_bf16(128, 64, 0, 1);   // TS: A in TMEM, B MN-major
    constexpr uint32_t id_k3 = idesc_bf16(128, 64, 1, 1);    // SS: A = B tile MN-major
    constexpr uint32_t dhi = sdesc_sw128_hi(1024);
    const uint32_t hlo = sdesc_sw128_lo(smem_u32(smem + kOffHHi), 0);
    const uint32_t dxlo = sdesc_sw128_lo(smem_u32(smem + kOffDxHi), 0);
    const uint32_t blo0 = sdesc_sw128_lo(smem_u32(smem + kOffB), 0);             // K-major
    const uint32_t bmlo0 = sdesc_sw128_lo(smem_u32(smem + kOffB), kBCBytes / 2);  // MN-major
    const uint32_t xlo0 = sdesc_sw128_lo(smem_u32(smem + kOffX), 0);
    const uint32_t clo0 = sdesc_sw128_lo(smem_u32(smem + kOffC), 0);             // K-major
    const uint32_t tC = tmem + kColC;
    // A product's barrier is tested (non-blocking) before the previous product is issued; only
    // if that test failed does the warp block on it afterwards.
    auto gate = [&](uint32_t probed, uint64_t* bar, uint32_t parity, int site) -> bool {
      if (!probed && !wait_bar(bar, parity, abort, a.hdr, site)) return false;
      return true;
    };
    // CB_t = C_t B_t^T with both operands K-major in shared memory (SS at N = 128 runs as fast
    // as TS), so it waits only for the two TMA loads; C_t's slot is released by this commit and
    // by the out warps once they hold C_t in TMEM for Yo_t
    auto issue_cb = [&](int t) {
      const uint32_t bl = blo0 + (t & 1) * (kBCBytes >> 4);
      const uint32_t dm = tmem + kColM + (t & 1) * 128;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t ko = ((ks >> 2) * (kBCBytes / 2) + (ks & 3) * 32) >> 4;
        mma_ss_we(dm, clo0 + ko, dhi, bl + ko, dhi, id_cb, ks > 0);
      }
      mma_commit_elect(&bars->cb_full[t & 1]);
    };
    // CB_t's inputs: probed without blocking, then waited for
    auto probe_cb = [&](int t) -> uint32_t {
      if (zero_b) return mbar_test_wait(&bars->cb_go, t & 1);
      return mbar_test_wait(&bars->c_full, t & 1) &&
             mbar_test_wait(&bars->b_full[t & 1], (t >> 1) & 1);
    };
    auto gate_cb = [&](uint32_t probed, int t) -> bool {
      if (probed) return true;
      if (zero_b) return wait_bar(&bars->cb_go, t & 1, abort, a.hdr, 35);
      return wait_bar(&bars->c_full, t & 1, abort, a.hdr, 35) &&
             wait_bar(&bars->b_full[t & 1], (t >> 1) & 1, abort, a.hdr, 37);
    };
    if constexpr (kPre) {
      // K3 only; B_t is waited for here (in the full pass the out warps wait for it)
      for (int t = 0; t < nt; ++t) {
        const int sb = t & 1;
        if (!gate(0, &bars->b_full[sb], (t >> 1) & 1, 34)) break;
        if (!gate(0, &bars->k3_go, t & 1, 38)) break;
        tc_fence_after();
        const uint32_t al = bmlo0 + sb * (kBCBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < 16; ++ks)
          mma_ss_we(tmem + kColS, al + (ks & 7) * (2048 >> 4), dhi,
                    dxlo + (((ks < 8 ? 0u : kOffDxLo - kOffDxHi) + (ks & 7) * 2048) >> 4), dhi,
                    id_k3, ks > 0);
        mma_commit_elect(&bars->s_full);
      }
    } else {
    uint32_t p_yo = mbar_test_wait(&bars->yo_go, 0);
    bool ok = gate_cb(0, 0);
    if (ok) {
      tc_fence_after();
      issue_cb(0);
    }
    for (int t = 0; ok && t < nt; ++t) {
      const int sb = t & 1;
      // Yo_t = C_t [h_hi ; h_lo]
      const uint32_t p_k3 = mbar_test_wait(&bars->k3_go, t & 1);
      if (!gate(p_yo, &bars->yo_go, t & 1, 36)) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 16; ++ks)
        mma_ts_we(tmem + kColYo, tC + (ks & 7) * 8,
                  hlo + (((ks < 8 ? 0u : kOffHLo - kOffHHi) + (ks & 7) * 2048) >> 4), dhi, id_n64,
                  ks > 0);
      mma_commit_elect(&bars->yo_full);
      // K3_t = B_t^T [(dec o x)_hi ; (dec o x)_lo]
      const uint32_t p_cb = t + 1 < nt ? probe_cb(t + 1) : 1u;
      if (!gate(p_k3, &bars->k3_go, t & 1, 38)) break;
      tc_fence_after();
      {
        const uint32_t al = bmlo0 + sb * (kBCBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < 16; ++ks)
          mma_ss_we(tmem + kColS, al + (ks & 7) * (2048 >> 4), dhi,
                    dxlo + (((ks < 8 ? 0u : kOffDxLo - kOffDxHi) + (ks & 7) * 2048) >> 4), dhi,
                    id_k3, ks > 0);
      }
      mma_commit_elect(&bars->s_full);
      // CB of the next tile, into the other mask buffer
      const uint32_t p_m = mbar_test_wait(&bars->m_ready[sb], (t >> 1) & 1);
      const uint32_t p_pre = mbar_test_wait(&bars->y_pre, t & 1);
      if (t + 1 < nt) {
        if (!gate_cb(p_cb, t + 1)) break;
        tc_fence_after();
        issue_cb(t + 1);
      }
      // Yd_t += (L o CB)_hi x + (L o CB)_lo x onto e^{cum_i} Yo_t
      p_yo = t + 1 < nt ? mbar_test_wait(&bars->yo_go, (t + 1) & 1) : 1u;
      if (!gate(p_m, &bars->m_ready[sb], (t >> 1) & 1, 40)) break;
      if (!gate(p_pre, &bars->y_pre, t & 1, 41)) break;
      tc_fence_after();
      {
        const uint32_t xl = xlo0 + (t % kXSlots) * (kXBytes >> 4);
        const uint32_t am = tmem + kColM + sb * 128;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const int kk = ks & 7;
          const uint32_t acol = (kk >> 1) * 32 + (kk & 1) * 8 + (ks < 8 ? 0 : 16);
          mma_ts_we(tmem + kColYd, am + acol, xl + kk * (2048 >> 4), dhi, id_n64, 1);
        }
      }
      mma_commit_elect(&bars->yd_full);
    }
    }
    // Drain: every MMA issued has completed before TMEM is freed.
    mma_commit_elect(&bars->drain);
    if (!mbar_wait_bounded(&bars->drain, 0, 2000000000ull) && lane == 0) {
      s_keep_tmem = 1;   // MMAs may still write TMEM: leave it allocated
      if (a.hdr) latch_error(a.hdr, SSD_ERR_TIMEOUT, 92);
    }
  } else if (warp == 2) {
    k1_warp<kW>(a, info, bars->info_ready, bars->info_empty, abort, b, h, tbase, nt, Tb, lane);
  } else {
    const int q = warp & 3;                 // TMEM lane quarter == SM sub-partition
    const int i = q * 32 + lane;            // tile row / state row of this thread
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    if (warp == 3 || (warp >= 4 && warp < 8)) {
      // ---------------------------------------------------------------- mask warps
      const int jlim = (i / R + 1) * R;     // columns j < jlim are at or before row i's step
      const MaskShare ms = mask_share(warp);
      const int2 du = dx_units<kPre>(warp);
      const bool has_dx = du.y > du.x;
      // (dec o x)_t split into hi and lo (own buffers; x_t stays for Yd_t).
      auto dec_x = [&](int t) -> bool {
        const int slot = t % kInfoSlots;
        const TileInfo& ti = info[slot];
        if (!wait_bar(&bars->info_ready[slot], (t / kInfoSlots) & 1, abort, a.hdr, 45))
          return false;
        if (!wait_bar(&bars->x_full[t % kXSlots], (t / kXSlots) & 1, abort, a.hdr, 46))
          return false;
        if (t >= 1 && !wait_bar(&bars->s_full, (t - 1) & 1, abort, a.hdr, 47)) return false;
        uint8_t* xs = smem + kOffX + (t % kXSlots) * kXBytes;
        uint8_t* dhi = smem + kOffDxHi;
        uint8_t* dlo = smem + kOffDxLo;
        const int lim = vrows - (seg_row + t * kTileRows);   // rows from lim on are padding
#pragma unroll 1
        for (int u = du.x; u < du.y; ++u) {
          const int row = (u >> 2) * 32 + lane, c0 = (u & 3) * 16;
          if (row >= lim) {   // pad row: zero in x (for Yd) and in (dec o x)
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t o0 = sw128_off16(row, c0), o1 = sw128_off16(row, c0 + 8);
            *reinterpret_cast<uint4*>(xs + o0) = z;
            *reinterpret_cast<uint4*>(xs + o1) = z;
            *reinterpret_cast<uint4*>(dhi + o0) = z;
            *reinterpret_cast<uint4*>(dhi + o1) = z;
            *reinterpret_cast<uint4*>(dlo + o0) = z;
            *reinterpret_cast<uint4*>(dlo + o1) = z;
            continue;
          }
          float wd = ex2_approx(ti.last_hi - ti.cum_hi[row]);
          if constexpr (kW) wd *= ti.w[row];
          const float2 w2 = make_float2(wd, wd);
          const uint32_t o0 = sw128_off16(row, c0), o1 = sw128_off16(row, c0 + 8);
          const uint4 v0 = *reinterpret_cast<const uint4*>(xs + o0);
          const uint4 v1 = *reinterpret_cast<const uint4*>(xs + o1);
          uint4 h0, l0, h1, l1;
          split2(mul2(unpack_bf16(v0.x), w2), h0.x, l0.x);
          split2(mul2(unpack_bf16(v0.y), w2), h0.y, l0.y);
          split2(mul2(unpack_bf16(v0.z), w2), h0.z, l0.z);
          split2(mul2(unpack_bf16(v0.w), w2), h0.w, l0.w);
          split2(mul2(unpack_bf16(v1.x), w2), h1.x, l1.x);
          split2(mul2(unpack_bf16(v1.y), w2), h1.y, l1.y);
          split2(mul2(unpack_bf16(v1.z), w2), h1.z, l1.z);
          split2(mul2(unpack_bf16(v1.w), w2), h1.w, l1.w);
          *reinterpret_cast<uint4*>(dhi + o0) = h0;
          *reinterpret_cast<uint4*>(dhi + o1) = h1;
          *reinterpret_cast<uint4*>(dlo + o0) = l0;
          *reinterpret_cast<uint4*>(dlo + o1) = l1;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->k3_go);
        return true;
      };
      // Mask blocks of tile t for this thread's row, in place over CB_t (mask buffer t & 1).
      auto mask_part = [&](int t) -> bool {
        const int slot = t % kInfoSlots;
        const TileInfo& ti = info[slot];
        if (!wait_bar(&bars->info_ready[slot], (t / kInfoSlots) & 1, abort, a.hdr, 43))
          return false;
        if (!wait_bar(&bars->cb_full[t & 1], (t >> 1) & 1, abort, a.hdr, 44)) return false;
        tc_fence_after();
        const uint32_t mb = tmem + lane_addr + kColM + (t & 1) * 128;
        const bool fact_ok = ti.monotone != 0;
        const float chi = ti.cum_hi[i];
#pragma unroll 1
        for (int cb = ms.cb0; cb < ms.cb1; ++cb) {
          float w[32];
          tmem_ld32(mb + cb * 32, w);
          tmem_ld_wait();
          reg_tie(w);
          uint32_t hi[16], lo[16];
          mask_block<kW>(ti, cb, cb == q || !fact_ok, chi, jlim, w, hi, lo);
          tmem_st16u(mb + cb * 32, hi);
          tmem_st16u(mb + cb * 32 + 16, lo);
        }
        if (ms.cb1 < ms.zero_end) {
          uint32_t z[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) z[k] = 0u;
#pragma unroll 1
          for (int cb = ms.cb1; cb < ms.zero_end; ++cb) {
            tmem_st16u(mb + cb * 32, z);
            tmem_st16u(mb + cb * 32 + 16, z);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->m_ready[t & 1]);
        return true;
      };
      for (int t = 0; t < nt; ++t) {
        if (has_dx && !dec_x(t)) break;
        if (kPre) {
          // x_t has no other reader in the pre-pass
          if (has_dx && lane == 0) mbar_arrive(&bars->x_empty[t % kXSlots]);
          continue;
        }
        if (!mask_part(t)) break;
      }
    } else if (warp < 12) {
      // ---------------------------------------------------------------- state warps
      // Thread = state row n = i; h^T[n][0..63] in registers across the whole sequence.
      const size_t st_base = (size_t)seq * kP * kN;
      const size_t seg_base = ((size_t)seq * nrun + seg) * kP * kN;
      // initial state: the call's for segment 0; the carried one for later segments of the full
      // pass; zero for later segments of the pre-pass
      const float* init0 = seg == 0 ? (a.init ? a.init + st_base : nullptr)
                                    : (kPre ? nullptr : a.seg_init + seg_base);
      float seg_decay = 1.f;   // pre-pass: product of the tiles' exp(cum_last)
      float hv[kP];
#pragma unroll
      for (int p = 0; p < kP; ++p) hv[p] = init0 ? init0[(size_t)p * kN + i] : 0.f;
      if (lane == 0) mbar_arrive(&bars->k3_go);   // the S accumulator is free for K3_0
      // t = -1 publishes h_0; iteration t folds S_t into the state and publishes h_{t+1}
      for (int t = -1; t < nt; ++t) {
        if (t >= 0) {
          const int slot = t % kInfoSlots;
          if (!wait_bar(&bars->info_ready[slot], (t / kInfoSlots) & 1, abort, a.hdr, 48)) break;
          if (!wait_bar(&bars->s_full, t & 1, abort, a.hdr, 49)) break;
          tc_fence_after();
          if (warp == 8 && lane == 0) mbar_arrive(&bars->b_empty[t & 1]);   // K3_t read B_t
          const float e = info[slot].etile;
          const float2 e2 = make_float2(e, e);
          seg_decay *= e;
#pragma unroll
          for (int c = 0; c < kP; c += 32) {
            float sv[32];
            tmem_ld32(tmem + lane_addr + kColS + c, sv);
            tmem_ld_wait();
            reg_tie(sv);
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const float2 v = fma2(e2, make_float2(hv[c + k], hv[c + k + 1]),
                                    make_float2(sv[k], sv[k + 1]));
              hv[c + k] = v.x;
              hv[c + k + 1] = v.y;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (t + 1 < nt) mbar_arrive(&bars->k3_go);   // S_t read: K3_{t+1} may go
            mbar_arrive(&bars->info_empty[slot]);
          }
          if (t + 1 == nt) break;
          if (kPre) continue;   // the pre-pass has no Yo
          // Yo_t has read h_t from the operand buffer (it was issued before K3_t)
          if (!wait_bar(&bars->yo_full, t & 1, abort, a.hdr, 50)) break;
        } else if (kPre) {
          continue;
        }
        // h^T row n as bf16 hi and lo rows of the Yo operand
        uint8_t* hhi = smem + kOffHHi;
        uint8_t* hlo = smem + kOffHLo;
#pragma unroll
        for (int k = 0; k < kP; k += 8) {
          uint4 uh, ul;
          split2(make_float2(hv[k], hv[k + 1]), uh.x, ul.x);
          split2(make_float2(hv[k + 2], hv[k + 3]), uh.y, ul.y);
          split2(make_float2(hv[k + 4], hv[k + 5]), uh.z, ul.z);
          split2(make_float2(hv[k + 6], hv[k + 7]), uh.w, ul.w);
          const uint32_t off = sw128_off16(i, k);
          *reinterpret_cast<uint4*>(hhi + off) = uh;
          *reinterpret_cast<uint4*>(hlo + off) = ul;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->yo_go);
      }
      if (kPre) {   // the segment's end state and decay for the carry pass
        if (!*abort) {
#pragma unroll
          for (int p = 0; p < kP; ++p)
            if (SSD_INDEX_OK(a.hdr, seg_base + (size_t)p * kN + i, a.seqs * a.npre * kP * kN, 3))
              a.seg_end[seg_base + (size_t)p * kN + i] = hv[p];
          if (warp == 8 && lane == 0 &&
              SSD_INDEX_OK(a.hdr, (size_t)seq * nrun + seg, a.seqs * a.npre, 4))
            a.seg_decay[(size_t)seq * nrun + seg] = seg_decay;
        }
      } else if (a.final_state && seg == a.nseg - 1 && !*abort) {
#pragma unroll
        for (int p = 0; p < kP; ++p)
          if (SSD_INDEX_OK(a.hdr, st_base + (size_t)p * kN + i, a.st_elems, 2))
            a.final_state[st_base + (size_t)p * kN + i] = hv[p];
      }
    } else {
      // ---------------------------------------------------------------- out warps
      // Row i of B_t zeroed when it is padding (both 64-column halves of the stage).
      auto zero_b_pad = [&](int t) {
        if (i < vrows - (seg_row + t * kTileRows)) return;
        uint8_t* bs = smem + kOffB + (t & 1) * kBCBytes;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(bs + blk * (kBCBytes / 2) + sw128_off16(i, c * 8)) = z;
      };
      if constexpr (kPre) {
        // K3_t waits for these warps once B_t's pad rows are zero; tile t is taken up only
        // after K3_{t-1} completed, so no arrival runs a phase ahead
        for (int t = 0; zero_b && t < nt; ++t) {
          if (t >= 1 && !wait_bar(&bars->s_full, (t - 1) & 1, abort, a.hdr, 56)) break;
          if (!wait_bar(&bars->b_full[t & 1], (t >> 1) & 1, abort, a.hdr, 57)) break;
          zero_b_pad(t);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->k3_go);
        }
      }
      if constexpr (!kPre) {   // the pre-pass has no output
        // Per tile: e^{cum_i} Yo_t into the y accumulator; C_{t+1} into TMEM once Yo_t has read
        // C_t; then y_t = the accumulator after Yd_t -> bf16 -> the tile's x slot -> TMA store.
        auto copy_c = [&](int t) -> bool {
          if (!wait_bar(&bars->c_full, t & 1, abort, a.hdr, 51)) return false;
          const uint8_t* cs = smem + kOffC;
  #pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            uint32_t w[32];
  #pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v = *reinterpret_cast<const uint4*>(cs + blk * (kBCBytes / 2) +
                                                              sw128_off16(i, c * 8));
              w[c * 4 + 0] = v.x;
              w[c * 4 + 1] = v.y;
              w[c * 4 + 2] = v.z;
              w[c * 4 + 3] = v.w;
            }
            tmem_st32u(tmem + lane_addr + kColC + blk * 32, w);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->cb_full[t & 1]);
          tmem_st_wait();
          tc_fence_before();
          if (zero_b) {   // CB_t waits for B_t's pad rows to be zero
            if (!wait_bar(&bars->b_full[t & 1], (t >> 1) & 1, abort, a.hdr, 55)) return false;
            if (vrows - (seg_row + t * kTileRows) < kTileRows) {
              zero_b_pad(t);
              fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->cb_go);
          }
          return true;
        };
        // t = -1 only copies C_0 (no Yo to read before tile 0)
        for (int t = -1; t < nt; ++t) {
          if (t < 0) {
            if (!copy_c(0)) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->yo_go);
            continue;
          }
          const int slot = t % kInfoSlots;
          if (!wait_bar(&bars->info_ready[slot], (t / kInfoSlots) & 1, abort, a.hdr, 54)) break;
          if (!wait_bar(&bars->yo_full, t & 1, abort, a.hdr, 52)) break;
          tc_fence_after();
          const TileInfo& ti = info[slot];
          {
            // e^{cum_i} Yo_t into the y accumulator (y_{t-1} was read in the previous iteration)
            const float sc = ex2_approx(ti.cum_hi[i]);
            const float2 sc2 = make_float2(sc, sc);
  #pragma unroll
            for (int c = 0; c < kP; c += 32) {
              float vo[32];
              tmem_ld32(tmem + lane_addr + kColYo + c, vo);
              tmem_ld_wait();
              reg_tie(vo);
              uint32_t vu[32];
  #pragma unroll
              for (int k = 0; k < 32; k += 2) {
                const float2 v = mul2(sc2, make_float2(vo[k], vo[k + 1]));
                vu[k] = __float_as_uint(v.x);
                vu[k + 1] = __float_as_uint(v.y);
              }
              tmem_st32u(tmem + lane_addr + kColYd + c, vu);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->y_pre);
          }
          if (t + 1 < nt) {   // Yo_t read and C_{t+1} in TMEM: Yo_{t+1} may go
            if (!copy_c(t + 1)) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->yo_go);
          }
          if (!wait_bar(&bars->yd_full, t & 1, abort, a.hdr, 53)) break;
          tc_fence_after();
          uint8_t* ys = smem + kOffX + (t % kXSlots) * kXBytes;   // x_t is no longer needed
          // a quarter of whole real rows goes out by TMA from the slot; one that reaches the
          // end of the real rows is stored row by row from registers (real rows only)
          const int qrow = seg_row + t * kTileRows + q * 32;   // first fused row of the quarter
          const int vq = vrows - qrow;
          __nv_bfloat16* yrow = a.y + (((size_t)b * a.T * R + qrow + lane) * a.H + h) * kP;
  #pragma unroll
          for (int c = 0; c < kP; c += 32) {
            float vy[32];
            tmem_ld32(tmem + lane_addr + kColYd + c, vy);
            tmem_ld_wait();
            reg_tie(vy);
            uint32_t pk[16];
  #pragma unroll
            for (int k = 0; k < 16; ++k) pk[k] = pack_bf16(vy[2 * k], vy[2 * k + 1]);
            if (vq >= 32) {
  #pragma unroll
              for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4*>(ys + sw128_off16(i, c + 8 * k)) =
                    make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            } else if (lane < vq) {
  #pragma unroll
              for (int k = 0; k < 4; ++k)
                if (SSD_INDEX_OK(a.hdr, (yrow - a.y) + c + 8 * k + 7, a.y_elems, 1))
                *reinterpret_cast<uint4*>(yrow + c + 8 * k) =
                    make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            }
          }
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars->info_empty[slot]);
            if (vq >= 32) {
              tma_store_4d(&tm_y, ys + q * 4096, 0, h, qrow, b);
              bulk_commit_group();
            }
            // the store of the previous tile has read its slot: hand it back to the producer
            if (t >= 1) {
              if (vq >= 32)
                bulk_wait_group_read<1>();
              else
                bulk_wait_group_read<0>();
              mbar_arrive(&bars->x_empty[(t - 1) % kXSlots]);
            }
          }
          __syncwarp();
        }
        if (lane == 0) {
          bulk_wait_group<0>();   // every y store complete before the CTA exits
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1 && !s_keep_tmem) {
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
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, dt, rank, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded tensor maps of the last few distinct (pointers, shape) keys per host thread: a call
// with the same buffers skips the three encodes.
struct MapKey {
  const void *x, *B, *C, *y;
  int64_t batch, T, H, G, R, P, N;
  bool operator==(const MapKey& o) const {
    return x == o.x && B == o.B && C == o.C && y == o.y && batch == o.batch && T == o.T &&
           H == o.H && G == o.G && R == o.R && P == o.P && N == o.N;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap mx, mb, mc, my;
  bool valid = false;
};
constexpr int kMapCacheSize = 4;

// Maps over [batch][T * R fused rows][heads or groups][P or N]: the batch is a dimension of
// its own so that a tile running past the end of a sequence reads zeros, not the next one.
bool encode_maps(const GenericParams& p, MapEntry& m) {
  const int64_t rows = p.T * p.R;
  {
    cuuint64_t dims[4] = {(cuuint64_t)p.P, (cuuint64_t)p.H, (cuuint64_t)rows, (cuuint64_t)p.batch};
    cuuint64_t str[3] = {(cuuint64_t)p.P * 2, (cuuint64_t)p.H * p.P * 2,
                         (cuuint64_t)rows * p.H * p.P * 2};
    cuuint32_t box[4] = {64, 1, kTileRows, 1};
    if (!make_map(&m.mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.x, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    // y has x's layout; each out warp stores its 32 rows of a tile
    cuuint32_t ybox[4] = {64, 1, 32, 1};
    if (!make_map(&m.my, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.y, dims, str, ybox,
                  CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  }
  cuuint64_t dims[4] = {(cuuint64_t)p.N, (cuuint64_t)p.G, (cuuint64_t)rows, (cuuint64_t)p.batch};
  cuuint64_t str[3] = {(cuuint64_t)p.N * 2, (cuuint64_t)p.G * p.N * 2,
                       (cuuint64_t)rows * p.G * p.N * 2};
  cuuint32_t box[4] = {64, 1, kTileRows, 1};
  return make_map(&m.mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.B, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&m.mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.C, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

const MapEntry* cached_maps(const GenericParams& p) {
  thread_local MapEntry cache[kMapCacheSize];
  thread_local int next = 0;
  const MapKey key{p.x, p.B, p.C, p.y, p.batch, p.T, p.H, p.G, p.R, p.P, p.N};
  for (auto& m : cache)
    if (m.valid && m.key == key) return &m;
  MapEntry& m = cache[next];
  next = (next + 1) % kMapCacheSize;
  m.valid = false;
  if (!encode_maps(p, m)) return nullptr;
  m.key = key;
  m.valid = true;
  return &m;
}

// The kernel's dynamic shared-memory limit is raised once per device.
cudaError_t ensure_smem_attribute() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  const void* kernels[] = {reinterpret_cast<const void*>(ssd_fused_bf16_kernel<false, false>),
                           reinterpret_cast<const void*>(ssd_fused_bf16_kernel<true, false>),
                           reinterpret_cast<const void*>(ssd_fused_bf16_kernel<false, true>),
                           reinterpret_cast<const void*>(ssd_fused_bf16_kernel<true, true>)};
  for (const void* k : kernels)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// True initial state of every segment after the first, one thread per (sequence, state element):
// piece 0 of the pre-pass started from the true state, later ones from zero, so after piece j
// h = end_0 (j = 0) or decay_j h + end_j; at the end of every per = seg_tiles / pre_tiles pieces
// that is the initial state of the next segment.
__global__ void fused_seg_carry_kernel(FusedArgs a, int64_t elems) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= elems) return;
  constexpr int64_t kPN = (int64_t)kP * kN;
  const int64_t seq = idx / kPN, e = idx % kPN;
  float* init = const_cast<float*>(a.seg_init);
  const int per = a.seg_tiles / a.pre_tiles;   // pieces per segment
  float hcur = 0.f;
  for (int j = 0; j < a.npre; ++j) {
    const float end = a.seg_end[(seq * a.npre + j) * kPN + e];
    hcur = j == 0 ? end : fmaf(a.seg_decay[seq * a.npre + j], hcur, end);
    const int64_t o = (seq * a.nseg + (j + 1) / per) * kPN + e;
    if ((j + 1) % per == 0 && SSD_INDEX_OK(a.hdr, o, a.seqs * a.nseg * kPN, 5)) init[o] = hcur;
  }
}

// Segments per sequence: enough CTAs to cover the SMs when there are fewer sequences than SMs
// (each segment keeps at least four tiles).
// Tiles of 128 fused rows per sequence (the last may be partial).
int64_t fused_tiles(int64_t T, int64_t R) { return (T * R + kTileRows - 1) / kTileRows; }

struct SegPlan {
  int ntiles, nseg, seg_tiles, npre, pre_tiles;
};

// Segments per sequence: enough CTAs to cover the SMs when there are fewer sequences than SMs
// (each segment keeps at least four tiles); then the state-only pieces: each segment before the
// last is cut into the largest number k of equal pieces (k divides seg_tiles, each piece keeps
// at least four tiles) with seqs * (nseg - 1) * k CTAs still within one wave.
SegPlan fused_plan(int64_t batch, int64_t T, int64_t H, int64_t R) {
  SegPlan pl;
  pl.ntiles = (int)fused_tiles(T, R);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  const int64_t seqs = std::max<int64_t>(batch * H, 1);
  int64_t n = sms / seqs;
  n = std::min<int64_t>(n, pl.ntiles / 4);
  n = std::min<int64_t>(n, 16);
  pl.nseg = (int)std::max<int64_t>(n, 1);
  pl.seg_tiles = (pl.ntiles + pl.nseg - 1) / pl.nseg;
  pl.nseg = (pl.ntiles + pl.seg_tiles - 1) / pl.seg_tiles;   // no empty segment
  int k = 1;
  if (pl.nseg > 1) {
    const int64_t pre_seqs = seqs * (pl.nseg - 1);
    for (int c = 2; c <= 16; ++c)
      if (pl.seg_tiles % c == 0 && pl.seg_tiles / c >= 4 && pre_seqs * c <= sms) k = c;
  }
  pl.pre_tiles = pl.seg_tiles / k;
  pl.npre = (pl.nseg - 1) * k;
  return pl;
}

}  // namespace

size_t fused_bf16_workspace_bytes(int64_t batch, int64_t T, int64_t H, int64_t R) {
  const SegPlan pl = fused_plan(batch, T, H, R);
  size_t bytes = sizeof(WsHeader);
  if (pl.nseg > 1) {
    const size_t seqs = (size_t)batch * H;
    bytes += seqs * (pl.nseg + pl.npre) * kP * kN * sizeof(float) +
             align_up(seqs * pl.npre * sizeof(float), 256);
  }
  return bytes;
}

bool fused_bf16_supported(int64_t T, int64_t H, int64_t P, int64_t N, int64_t R, int64_t l,
                          bool bf16, bool theta) {
  if (!bf16 || theta) return false;
  if (P != kP || N != kN) return false;
  if (R < 1 || R > 32 || (kTileRows % R) != 0) return false;
  if (H % 4 != 0) return false;                      // dA tile loads use 16-byte boxes
  (void)T;
  (void)l;
  return true;
}

cudaError_t fused_bf16_forward(const GenericParams& p, cudaStream_t st) {
  const MapEntry* m = cached_maps(p);
  if (!m) return cudaErrorInvalidValue;
  const int steps = (int)(kTileRows / p.R);
  FusedArgs a;
  a.dA = p.dA;
  a.init = p.init;
  a.final_state = p.final_state;
  a.y = static_cast<__nv_bfloat16*>(p.y);
  a.hdr = p.hdr;
  a.valid_len = p.valid_len;
  a.wrow = p.wrow;
  a.seqs = p.batch * p.H;
  a.y_elems = p.batch * p.T * p.R * p.H * p.P;
  a.st_elems = a.seqs * p.P * p.N;
  a.T = (int32_t)p.T;
  a.R = (int32_t)p.R;
  a.H = (int32_t)p.H;
  a.G = (int32_t)p.G;
  const SegPlan pl = fused_plan(p.batch, p.T, p.H, p.R);
  a.ntiles = pl.ntiles;
  a.steps = steps;
  a.nseg = pl.nseg;
  a.seg_tiles = pl.seg_tiles;
  a.npre = pl.npre;
  a.pre_tiles = pl.pre_tiles;
  // workspace after the header: segment initial states, piece end states, piece decays
  char* ws = reinterpret_cast<char*>(p.hdr);
  const size_t seqs_z = (size_t)p.batch * p.H;
  const size_t init_bytes = seqs_z * a.nseg * kP * kN * sizeof(float);
  const size_t end_bytes = seqs_z * a.npre * kP * kN * sizeof(float);
  a.seg_init = reinterpret_cast<const float*>(ws + sizeof(WsHeader));
  a.seg_end = reinterpret_cast<float*>(ws + sizeof(WsHeader) + init_bytes);
  a.seg_decay = reinterpret_cast<float*>(ws + sizeof(WsHeader) + init_bytes + end_bytes);
  cudaError_t e = ensure_smem_attribute();
  if (e != cudaSuccess) return e;
  const unsigned seqs = (unsigned)(p.batch * p.H);
  if (a.nseg > 1) {
    if (a.wrow)
      ssd_fused_bf16_kernel<true, true><<<seqs * a.npre, kThreads, kSmem, st>>>(
          a, m->mx, m->mb, m->mc, m->my);
    else
      ssd_fused_bf16_kernel<true, false><<<seqs * a.npre, kThreads, kSmem, st>>>(
          a, m->mx, m->mb, m->mc, m->my);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t elems = (int64_t)seqs * kP * kN;
    fused_seg_carry_kernel<<<(unsigned)((elems + 255) / 256), 256, 0, st>>>(a, elems);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.wrow)
    ssd_fused_bf16_kernel<false, true><<<seqs * a.nseg, kThreads, kSmem, st>>>(
        a, m->mx, m->mb, m->mc, m->my);
  else
    ssd_fused_bf16_kernel<false, false><<<seqs * a.nseg, kThreads, kSmem, st>>>(
        a, m->mx, m->mb, m->mc, m->my);
  return cudaGetLastError();
}

int fused_bf16_launches(int64_t batch, int64_t T, int64_t H, int64_t R) {
  return fused_plan(batch, T, H, R).nseg > 1 ? 3 : 1;
}

}  // namespace ssd
