// Rotation variants of the Mamba-3 SSD forward: a partial rotation over the first rope_dim state
// dimensions, and the split-halves pairing (k, k + rope_dim/2) instead of the interleaved
// (2k, 2k+1) (moments.rs page, RotationSeq::Angle { rope_dim, rotate_pairwise }).
//
// Both reduce to the interleaved full-width rotation of ssd_chunked_forward:
//   - the state axis can be reordered freely (y = C . h does not see the order), and the order
//     d -> 2d, d + rope_dim/2 -> 2d + 1 (d < rope_dim/2) turns the split halves into interleaved
//     pairs; B, C and the initial state are reordered on the way in and the final state back;
//   - angles past rope_dim/2 are zero, which turns nothing.
// So the call reorders B/C (only for the split halves), pads theta to dstate/2 angles in the
// workspace, and runs the chunked forward on them.
#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kLanes = 32, kRows = 8;

// New position of state dimension d (identity for the interleaved pairing).
__device__ __forceinline__ int64_t rot_pos(int64_t d, int64_t half, bool halves) {
  if (!halves || d >= 2 * half) return d;
  return d < half ? 2 * d : 2 * (d - half) + 1;
}

// dst[row][rot_pos(d)] = src[row][d] for rows of N values (B and C, one block per step).
template <typename T>
__global__ void __launch_bounds__(kLanes * kRows)
    rot_reorder_bc(const T* __restrict__ B, const T* __restrict__ C, T* __restrict__ Bo,
                   T* __restrict__ Co, int64_t steps, int64_t rows_per_step, int64_t N,
                   int64_t half) {
  for (int64_t s = blockIdx.x; s < steps; s += gridDim.x) {
    for (int64_t r = threadIdx.y; r < rows_per_step; r += kRows) {
      const int64_t base = (s * rows_per_step + r) * N;
      for (int64_t d = threadIdx.x; d < N; d += kLanes) {
        const int64_t o = base + rot_pos(d, half, true);
        Bo[o] = B[base + d];
        Co[o] = C[base + d];
      }
    }
  }
}

// theta [steps][K] -> [steps][N/2] with zeros past K.
__global__ void __launch_bounds__(kLanes * kRows)
    rot_pad_theta(const float* __restrict__ th, float* __restrict__ out, int64_t rows, int64_t K,
                  int64_t K2) {
  for (int64_t r = (int64_t)blockIdx.x * kRows + threadIdx.y; r < rows;
       r += (int64_t)gridDim.x * kRows) {
    for (int64_t k = threadIdx.x; k < K2; k += kLanes)
      out[r * K2 + k] = k < K ? th[r * K + k] : 0.f;
  }
}

// States [rows][N]: forward (dst[rot_pos(d)] = src[d]) or back (dst[d] = src[rot_pos(d)]).
__global__ void __launch_bounds__(kLanes * kRows)
    rot_reorder_state(const float* __restrict__ src, float* __restrict__ dst, int64_t rows,
                      int64_t N, int64_t half, bool back) {
  for (int64_t r = (int64_t)blockIdx.x * kRows + threadIdx.y; r < rows;
       r += (int64_t)gridDim.x * kRows) {
    for (int64_t d = threadIdx.x; d < N; d += kLanes) {
      const int64_t q = rot_pos(d, half, true);
      if (back) {
        dst[r * N + d] = src[r * N + q];
      } else {
        dst[r * N + q] = src[r * N + d];
      }
    }
  }
}

unsigned blocks_for(int64_t n) {
  return (unsigned)(n < 1 ? 1 : (n > 0x7fffffff ? 0x7fffffff : n));
}

struct RotLayout {
  size_t inner = 0, bo = 0, co = 0, th = 0, init = 0, fin = 0, total = 0;
};

bool rot_args_ok(const ssd_shape* s, int64_t rope_dim, int32_t halves) {
  if (!s || s->has_theta != 1) return false;
  if (rope_dim < 0 || rope_dim > s->dstate || (rope_dim % 2) != 0) return false;
  return halves == 0 || halves == 1;
}

RotLayout rot_layout(const ssd_shape* s, size_t inner) {
  const size_t e = s->io_dtype == SSD_BF16 ? 2 : 4;
  const size_t bc = e * (size_t)(s->batch * s->seqlen * s->mimo_rank * s->ngroups * s->dstate);
  const size_t st = sizeof(float) * (size_t)(s->batch * s->nheads * s->headdim * s->dstate);
  RotLayout L;
  L.inner = inner;
  size_t off = align_up(inner, kWsAlign);
  L.bo = off;
  off = align_up(off + bc, kWsAlign);
  L.co = off;
  off = align_up(off + bc, kWsAlign);
  L.th = off;
  const size_t th = sizeof(float) * (size_t)(s->batch * s->seqlen * s->nheads * (s->dstate / 2));
  off = align_up(off + th, kWsAlign);
  L.init = off;
  off = align_up(off + st, kWsAlign);
  L.fin = off;
  off = align_up(off + st, kWsAlign);
  L.total = off;
  return L;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_rotation_variant_workspace_bytes(const ssd_shape* shape, int64_t rope_dim,
                                            int32_t halves) {
  if (!rot_args_ok(shape, rope_dim, halves)) return 0;
  const size_t inner = ssd_chunked_workspace_bytes(shape);
  if (inner == 0) return 0;
  return rot_layout(shape, inner).total;
}

ssd_status ssd_rotation_variant_forward(const ssd_shape* shape, int64_t rope_dim,
                                        int32_t halves, const void* x, const float* dA,
                                        const void* B, const void* C, const float* theta,
                                        const float* init_state, void* y, float* final_state,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  const ssd_status vs = shape_status(shape);
  if (vs != SSD_OK) return vs;
  if (!rot_args_ok(shape, rope_dim, halves)) return SSD_ERR_INVALID_ARG;
  const size_t inner = ssd_chunked_workspace_bytes(shape);
  if (!x || !dA || !B || !C || !theta || !y) return SSD_ERR_INVALID_ARG;
  const RotLayout lay = rot_layout(shape, inner);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0 ||
      workspace_bytes < lay.total)
    return SSD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t N = shape->dstate, rd = rope_dim > 0 ? rope_dim : N, half = rd / 2;
  const bool bf16 = shape->io_dtype == SSD_BF16;
  const dim3 blk(kLanes, kRows);

  const void *Bu = B, *Cu = C;
  const float* init_u = init_state;
  float* fin_u = final_state;
  if (halves) {   // reorder the state axis so the split halves become interleaved pairs
    const int64_t steps = shape->batch * shape->seqlen;
    const int64_t rows = shape->mimo_rank * shape->ngroups;
    if (bf16) {
      rot_reorder_bc<__nv_bfloat16><<<blocks_for(steps), blk, 0, st>>>(
          static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C),
          reinterpret_cast<__nv_bfloat16*>(ws + lay.bo),
          reinterpret_cast<__nv_bfloat16*>(ws + lay.co), steps, rows, N, half);
    } else {
      rot_reorder_bc<float><<<blocks_for(steps), blk, 0, st>>>(
          static_cast<const float*>(B), static_cast<const float*>(C),
          reinterpret_cast<float*>(ws + lay.bo), reinterpret_cast<float*>(ws + lay.co), steps,
          rows, N, half);
    }
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
    Bu = ws + lay.bo;
    Cu = ws + lay.co;
    const int64_t srows = shape->batch * shape->nheads * shape->headdim;
    if (init_state) {
      rot_reorder_state<<<blocks_for((srows + kRows - 1) / kRows), blk, 0, st>>>(
          init_state, reinterpret_cast<float*>(ws + lay.init), srows, N, half, false);
      if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
      init_u = reinterpret_cast<const float*>(ws + lay.init);
    }
    if (final_state) fin_u = reinterpret_cast<float*>(ws + lay.fin);
  }
  const float* th_u = theta;
  if (half != N / 2) {   // zero angles past rope_dim / 2
    const int64_t rows = shape->batch * shape->seqlen * shape->nheads;
    rot_pad_theta<<<blocks_for((rows + kRows - 1) / kRows), blk, 0, st>>>(
        theta, reinterpret_cast<float*>(ws + lay.th), rows, half, N / 2);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
    th_u = reinterpret_cast<const float*>(ws + lay.th);
  }
  const ssd_status sc = ssd_chunked_forward(shape, x, dA, Bu, Cu, th_u, init_u, y, fin_u,
                                            workspace, lay.inner, stream);
  if (sc != SSD_OK) return sc;
  if (halves && final_state) {
    const int64_t srows = shape->batch * shape->nheads * shape->headdim;
    rot_reorder_state<<<blocks_for((srows + kRows - 1) / kRows), blk, 0, st>>>(
        fin_u, final_state, srows, N, half, true);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  }
  return SSD_OK;
}

}  // extern "C"
