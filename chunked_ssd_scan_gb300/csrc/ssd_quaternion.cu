// Quaternion rotation of the Mamba-3 SSD forward (moments.rs page, RotationSeq::Quaternion
// { cum_bshj4 }: the cumulative unit quaternion Q_t per (batch, step, head) and block j of four
// state dimensions).  Block j of the state, read as the quaternion h[4j] + h[4j+1] i +
// h[4j+2] j + h[4j+3] k, is turned at every step by left multiplication with the step
// quaternion Q_t Q_{t-1}^*, so the turns up to step t compose to Q_t.
//
// Left multiplication by a unit quaternion is an orthogonal map whose transpose is left
// multiplication by the conjugate, so the rotation absorbs into B and C exactly as the angle
// form does (scan.py page, "THE TRICK"): with g_t = Q_t^* h_t (block-wise),
//   g_t = exp(dA_t) g_{t-1} + x_t (Q_t^* B_t),   y_t = (Q_t^* C_t) . g_t,   h_{T-1} = Q_{T-1} g.
// The call turns B and C per head into fp32 copies in the workspace (the turned values are not
// bf16-exact, so bf16 x is widened and y narrowed around an fp32 problem), runs
// ssd_chunked_forward on that problem (one B/C group per head, no angles) and turns the final
// state back by Q_{T-1}.
#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 256;

// o = q v for quaternions (w, x, y, z) = w + x i + y j + z k.
__device__ __forceinline__ float4 qmul(float4 q, float4 v) {
  return make_float4(q.x * v.x - q.y * v.y - q.z * v.z - q.w * v.w,
                     q.x * v.y + q.y * v.x + q.z * v.w - q.w * v.z,
                     q.x * v.z - q.y * v.w + q.z * v.x + q.w * v.y,
                     q.x * v.w + q.y * v.z - q.z * v.y + q.w * v.x);
}

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return make_float4(p[0], p[1], p[2], p[3]);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  return make_float4(__bfloat162float(p[0]), __bfloat162float(p[1]), __bfloat162float(p[2]),
                     __bfloat162float(p[3]));
}

// Bt[b,t,r,h,4k..4k+3] = Q[b,t,h,k]^* B[b,t,r,g(h),4k..4k+3], and the same for C.  One thread
// per (b, t, r, h, k).
template <typename T>
__global__ void __launch_bounds__(kThreads)
    quat_turn_bc(const T* __restrict__ B, const T* __restrict__ C, const float* __restrict__ Q,
                 float* __restrict__ Bt, float* __restrict__ Ct, int64_t batch, int64_t Tl,
                 int64_t R, int64_t H, int64_t G, int64_t N) {
  const int64_t K = N / 4;
  const int64_t total = batch * Tl * R * H * K;
  for (int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * kThreads) {
    const int64_t k = idx % K;
    const int64_t h = (idx / K) % H;
    const int64_t r = (idx / (K * H)) % R;
    const int64_t bt = idx / (K * H * R);   // b * Tl + t
    const int64_t g = h / (H / G);
    const float4 q = *reinterpret_cast<const float4*>(Q + ((bt * H + h) * K + k) * 4);
    const float4 qc = make_float4(q.x, -q.y, -q.z, -q.w);
    const int64_t src = ((bt * R + r) * G + g) * N + 4 * k;
    const int64_t dst = ((bt * R + r) * H + h) * N + 4 * k;
    *reinterpret_cast<float4*>(Bt + dst) = qmul(qc, load4(B + src));
    *reinterpret_cast<float4*>(Ct + dst) = qmul(qc, load4(C + src));
  }
}

// final[b,h,p,4k..4k+3] = Q[b,T-1,h,k] g[b,h,p,4k..4k+3].  One thread per (b, h, p, k).
__global__ void __launch_bounds__(kThreads)
    quat_turn_final(const float* __restrict__ g, const float* __restrict__ Q,
                    float* __restrict__ fin, int64_t batch, int64_t Tl, int64_t H, int64_t P,
                    int64_t N) {
  const int64_t K = N / 4;
  const int64_t total = batch * H * P * K;
  for (int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * kThreads) {
    const int64_t k = idx % K;
    const int64_t bh = idx / (K * P);   // b * H + h
    const int64_t b = bh / H, h = bh % H;
    const float4 q =
        *reinterpret_cast<const float4*>(Q + (((b * Tl + Tl - 1) * H + h) * K + k) * 4);
    const int64_t o = (idx / K) * N + 4 * k;
    *reinterpret_cast<float4*>(fin + o) = qmul(q, *reinterpret_cast<const float4*>(g + o));
  }
}

__global__ void __launch_bounds__(kThreads)
    widen_bf16(const __nv_bfloat16* __restrict__ src, float* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kThreads)
    dst[i] = __bfloat162float(src[i]);
}

__global__ void __launch_bounds__(kThreads)
    narrow_bf16(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kThreads)
    dst[i] = __float2bfloat16_rn(src[i]);
}

unsigned grid_for(int64_t n) {
  const int64_t blocks = (n + kThreads - 1) / kThreads;
  return (unsigned)(blocks < 1 ? 1 : (blocks > 65535 * 16 ? 65535 * 16 : blocks));
}

// The fp32 problem the call runs: one B/C group per head, no angles.
ssd_shape inner_shape(const ssd_shape* s) {
  ssd_shape e = *s;
  e.io_dtype = SSD_F32;
  e.ngroups = s->nheads;
  e.has_theta = 0;
  return e;
}

struct QuatLayout {
  size_t inner = 0, bt = 0, ct = 0, x32 = 0, y32 = 0, g = 0, total = 0;
};

QuatLayout quat_layout(const ssd_shape* s) {
  QuatLayout L;
  const ssd_shape e = inner_shape(s);
  L.inner = ssd_chunked_workspace_bytes(&e);
  if (L.inner == 0) return L;
  const size_t rows = (size_t)(s->batch * s->seqlen * s->mimo_rank * s->nheads);
  size_t off = align_up(L.inner, kWsAlign);
  L.bt = off;
  off = align_up(off + sizeof(float) * rows * s->dstate, kWsAlign);
  L.ct = off;
  off = align_up(off + sizeof(float) * rows * s->dstate, kWsAlign);
  if (s->io_dtype == SSD_BF16) {
    L.x32 = off;
    off = align_up(off + sizeof(float) * rows * s->headdim, kWsAlign);
    L.y32 = off;
    off = align_up(off + sizeof(float) * rows * s->headdim, kWsAlign);
  }
  L.g = off;
  off = align_up(off + sizeof(float) * (size_t)(s->batch * s->nheads * s->headdim * s->dstate),
                 kWsAlign);
  L.total = off;
  return L;
}

bool quat_shape_ok(const ssd_shape* s) {
  return s && s->has_theta == 0 && s->dstate % 4 == 0;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_quaternion_workspace_bytes(const ssd_shape* shape) {
  if (!quat_shape_ok(shape) || shape_status(shape) != SSD_OK) return 0;
  return quat_layout(shape).total;
}

ssd_status ssd_quaternion_forward(const ssd_shape* shape, const void* x, const float* dA,
                                  const void* B, const void* C, const float* qcum,
                                  const float* init_state, void* y, float* final_state,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const ssd_status vs = shape_status(shape);
  if (vs != SSD_OK) return vs;
  if (!quat_shape_ok(shape)) return SSD_ERR_INVALID_ARG;
  if (!x || !dA || !B || !C || !qcum || !y) return SSD_ERR_INVALID_ARG;
  // qcum is read and the final state written as float4
  if (!aligned16(qcum) || (final_state && !aligned16(final_state))) return SSD_ERR_INVALID_ARG;
  const QuatLayout lay = quat_layout(shape);
  if (lay.total == 0) return SSD_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0 ||
      workspace_bytes < lay.total)
    return SSD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = shape->io_dtype == SSD_BF16;
  const int64_t b = shape->batch, T = shape->seqlen, R = shape->mimo_rank, H = shape->nheads,
                G = shape->ngroups, P = shape->headdim, N = shape->dstate;
  float* Bt = reinterpret_cast<float*>(ws + lay.bt);
  float* Ct = reinterpret_cast<float*>(ws + lay.ct);
  const int64_t turns = b * T * R * H * (N / 4);
  if (bf16) {
    quat_turn_bc<__nv_bfloat16><<<grid_for(turns), kThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), qcum, Bt, Ct,
        b, T, R, H, G, N);
  } else {
    quat_turn_bc<float><<<grid_for(turns), kThreads, 0, st>>>(
        static_cast<const float*>(B), static_cast<const float*>(C), qcum, Bt, Ct, b, T, R, H, G,
        N);
  }
  if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  const int64_t nx = b * T * R * H * P;
  const void* xu = x;
  void* yu = y;
  if (bf16) {
    widen_bf16<<<grid_for(nx), kThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                  reinterpret_cast<float*>(ws + lay.x32), nx);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
    xu = ws + lay.x32;
    yu = ws + lay.y32;
  }
  float* g = reinterpret_cast<float*>(ws + lay.g);
  const ssd_shape e = inner_shape(shape);
  const ssd_status sc = ssd_chunked_forward(&e, xu, dA, Bt, Ct, nullptr, init_state, yu,
                                            final_state ? g : nullptr, workspace, lay.inner,
                                            stream);
  if (sc != SSD_OK) return sc;
  if (bf16) {
    narrow_bf16<<<grid_for(nx), kThreads, 0, st>>>(reinterpret_cast<const float*>(yu),
                                                   static_cast<__nv_bfloat16*>(y), nx);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  }
  if (final_state) {
    quat_turn_final<<<grid_for(b * H * P * (N / 4)), kThreads, 0, st>>>(g, qcum, final_state, b,
                                                                         T, H, P, N);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  }
  return SSD_OK;
}

}  // extern "C"
