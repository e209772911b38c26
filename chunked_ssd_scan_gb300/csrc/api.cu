// C ABI of the library: argument validation, workspace layout and kernel launches.
// Declarations and the contract of every entry point are in include/ssdscan.h.
#include <string.h>

#include "common.cuh"
#include "ssd_internal.h"

using namespace ssd;

namespace {

constexpr int64_t kMaxElems = (int64_t)1 << 40;

struct SsdLayout {
  size_t states = 0, cend = 0, phi = 0, phisum = 0, total = 0;
};

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > kMaxElems / a) return false;
  *out = a * b;
  return true;
}

ssd_status check_shape(const ssd_shape* s) {
  if (!s) return SSD_ERR_INVALID_ARG;
  if (s->batch < 1 || s->seqlen < 1 || s->nheads < 1 || s->headdim < 1 || s->dstate < 1 ||
      s->ngroups < 1 || s->mimo_rank < 1 || s->chunk_len < 1)
    return SSD_ERR_INVALID_ARG;
  if (s->nheads % s->ngroups != 0) return SSD_ERR_INVALID_ARG;
  if (s->io_dtype != SSD_F32 && s->io_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
  if (s->has_theta != 0 && s->has_theta != 1) return SSD_ERR_INVALID_ARG;
  if (s->has_theta && (s->dstate % 2) != 0) return SSD_ERR_INVALID_ARG;
  int64_t t;
  if (!mul_ok(s->batch, s->seqlen, &t) || !mul_ok(t, s->mimo_rank, &t) ||
      !mul_ok(t, s->nheads, &t) || !mul_ok(t, s->headdim, &t))
    return SSD_ERR_INVALID_ARG;
  if (!mul_ok(s->batch, s->seqlen, &t) || !mul_ok(t, s->mimo_rank, &t) ||
      !mul_ok(t, s->ngroups, &t) || !mul_ok(t, s->dstate, &t))
    return SSD_ERR_INVALID_ARG;
  if (!mul_ok(s->batch, s->nheads, &t) || !mul_ok(t, s->headdim, &t) || !mul_ok(t, s->dstate, &t))
    return SSD_ERR_INVALID_ARG;
  if (s->batch > 65535 || s->nheads > 65535) return SSD_ERR_UNSUPPORTED;   // grid limits
  if (!generic_supported(s->chunk_len, s->mimo_rank, s->headdim, s->dstate, s->has_theta != 0))
    return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

int32_t pick_variant(const ssd_shape* s) {
  if (fused_bf16_supported(s->seqlen, s->nheads, s->headdim, s->dstate, s->mimo_rank,
                           s->chunk_len, s->io_dtype == SSD_BF16, s->has_theta != 0))
    return SSD_VARIANT_TC_BF16;
  if (tc32_supported(s->headdim, s->dstate, s->mimo_rank, s->io_dtype == SSD_BF16))
    return SSD_VARIANT_TC_TF32;
  return SSD_VARIANT_GENERIC;
}

// Chunk length the kernels tile time by.  The decomposition is exact for any chunk length, so
// this is a tiling choice: the fp32 path with the tensor-core chunk scan uses 128 rank-fused
// rows (128 / R steps, one MMA tile), every other path the caller's chunk_len.
int64_t kernel_chunk_len(const ssd_shape* s) {
  return pick_variant(s) == SSD_VARIANT_TC_TF32 ? tc32_chunk_len(s->mimo_rank) : s->chunk_len;
}

// Workspace of the chunk pipeline run with chunks of l steps.
SsdLayout chunk_layout(const ssd_shape* s, int64_t l) {
  SsdLayout L;
  const int64_t nch = (s->seqlen + l - 1) / l;   // the last chunk may be short
  size_t off = sizeof(WsHeader);
  L.states = off;
  off = align_up(off + sizeof(float) * (size_t)(s->batch * nch * s->nheads * s->headdim * s->dstate),
                 kWsAlign);
  L.cend = off;
  off = align_up(off + sizeof(float) * (size_t)(s->batch * nch * s->nheads), kWsAlign);
  if (s->has_theta) {
    L.phi = off;
    off = align_up(off + sizeof(double) * (size_t)(s->batch * (nch + 1) * s->nheads * (s->dstate / 2)),
                   kWsAlign);
    L.phisum = off;
    off = align_up(off + sizeof(double) * (size_t)(s->batch * nch * s->nheads * (s->dstate / 2)),
                   kWsAlign);
  }
  L.total = off;
  return L;
}

SsdLayout ssd_layout(const ssd_shape* s) {
  if (pick_variant(s) == SSD_VARIANT_TC_BF16) {   // the fused kernel keeps its state on chip
    SsdLayout L;
    L.total = fused_bf16_workspace_bytes(s->batch, s->seqlen, s->nheads, s->mimo_rank);
    return L;
  }
  return chunk_layout(s, kernel_chunk_len(s));
}

bool al16(const void* p) { return p == nullptr || aligned16(p); }

// The trapezoidal form runs as this expanded problem: 2R fp32 write channels, B/C per head when
// theta is given (the shifted channel is turned by each head's own angle).
ssd_shape trap_expanded(const ssd_shape* s) {
  ssd_shape e = *s;
  e.mimo_rank = 2 * s->mimo_rank;
  e.io_dtype = SSD_F32;
  if (s->has_theta) e.ngroups = s->nheads;
  return e;
}

struct TrapLayout {
  SsdLayout inner;   // the generic pipeline's buffers (offsets from the workspace start)
  size_t xh = 0, bh = 0, ch = 0, yh = 0, total = 0;
  // the bf16 tensor-core form: the fused kernel's workspace first, then x^, B^, C^, w^, y^
  bool fused = false;
  size_t xq = 0, bq = 0, cq = 0, wq = 0, yq = 0;
};

// bf16 without rotation on a shape the fused kernel takes at 2R channels: the trapezoid runs
// there, with gamma and beta as per-row write weights.
bool trap_fused(const ssd_shape* s) {
  return s->io_dtype == SSD_BF16 && !s->has_theta && s->mimo_rank <= 16 &&
         fused_bf16_supported(s->seqlen, s->nheads, s->headdim, s->dstate, 2 * s->mimo_rank,
                              s->chunk_len, true, false);
}

ssd_status check_trap_shape(const ssd_shape* s) {
  ssd_status st = check_shape(s);
  if (st != SSD_OK) return st;
  if (s->mimo_rank > (int64_t(1) << 30)) return SSD_ERR_UNSUPPORTED;
  if (trap_fused(s)) return SSD_OK;
  const ssd_shape e = trap_expanded(s);
  if ((st = check_shape(&e)) != SSD_OK) return st;
  const int32_t v = pick_variant(&e);
  return (v == SSD_VARIANT_GENERIC || v == SSD_VARIANT_TC_TF32) ? SSD_OK : SSD_ERR_UNSUPPORTED;
}

TrapLayout trap_layout(const ssd_shape* s) {
  TrapLayout L;
  if (trap_fused(s)) {
    L.fused = true;
    const size_t rows = (size_t)(s->batch * s->seqlen * 2 * s->mimo_rank);
    size_t off = align_up(fused_bf16_workspace_bytes(s->batch, s->seqlen, s->nheads,
                                                     2 * s->mimo_rank),
                          kWsAlign);
    L.xq = off;
    off = align_up(off + 2 * rows * s->nheads * s->headdim, kWsAlign);
    L.bq = off;
    off = align_up(off + 2 * rows * s->ngroups * s->dstate, kWsAlign);
    L.cq = off;
    off = align_up(off + 2 * rows * s->ngroups * s->dstate, kWsAlign);
    L.wq = off;
    off = align_up(off + sizeof(float) * rows * s->nheads, kWsAlign);
    L.yq = off;
    off = align_up(off + 2 * rows * s->nheads * s->headdim, kWsAlign);
    L.total = off;
    return L;
  }
  const ssd_shape e = trap_expanded(s);
  L.inner = ssd_layout(&e);
  const size_t xs = sizeof(float) * (size_t)(e.batch * e.seqlen * e.mimo_rank * e.nheads * e.headdim);
  const size_t bs = sizeof(float) * (size_t)(e.batch * e.seqlen * e.mimo_rank * e.ngroups * e.dstate);
  size_t off = align_up(L.inner.total, kWsAlign);
  L.xh = off;
  off = align_up(off + xs, kWsAlign);
  L.bh = off;
  off = align_up(off + bs, kWsAlign);
  L.ch = off;
  off = align_up(off + bs, kWsAlign);
  L.yh = off;
  off = align_up(off + xs, kWsAlign);
  L.total = off;
  return L;
}

}  // namespace

namespace ssd {
ssd_status shape_status(const ssd_shape* s) { return check_shape(s); }
}  // namespace ssd

extern "C" {

size_t ssd_chunked_workspace_bytes(const ssd_shape* shape) {
  if (check_shape(shape) != SSD_OK) return 0;
  return ssd_layout(shape).total;   // ssd_chunked_forward_tf32 runs the same layout
}

int32_t ssd_chunked_launches(const ssd_shape* shape) {
  if (check_shape(shape) != SSD_OK) return 0;
  const int32_t v = pick_variant(shape);
  if (v == SSD_VARIANT_TC_BF16)
    return fused_bf16_launches(shape->batch, shape->seqlen, shape->nheads, shape->mimo_rank);
  return 3 + (shape->has_theta ? 2 : 0);
}

int32_t ssd_chunked_variant(const ssd_shape* shape) {
  if (check_shape(shape) != SSD_OK) return SSD_VARIANT_NONE;
  return pick_variant(shape);
}

}  // extern "C"

namespace {

// The forward entry points; valid_len is null for ssd_chunked_forward, and tf32 (the
// ssd_chunked_forward_tf32 entry) insists on the fp32 path with the tensor-core chunk scan
// instead of falling back to the generic pipeline for other shapes.
ssd_status chunked_forward(const ssd_shape* shape, const void* x, const float* dA, const void* B,
                           const void* C, const float* theta, const int64_t* valid_len,
                           const float* init_state, void* y, float* final_state, void* workspace,
                           size_t workspace_bytes, void* stream, bool tf32 = false) {
  const ssd_status sc = check_shape(shape);
  if (sc != SSD_OK) return sc;
  if (tf32 && !tc32_supported(shape->headdim, shape->dstate, shape->mimo_rank,
                              shape->io_dtype == SSD_BF16))
    return SSD_ERR_UNSUPPORTED;
  if (!x || !dA || !B || !C || !y) return SSD_ERR_INVALID_ARG;
  if ((shape->has_theta != 0) != (theta != nullptr)) return SSD_ERR_INVALID_ARG;
  if (!al16(x) || !al16(dA) || !al16(B) || !al16(C) || !al16(y) || !al16(theta) ||
      !al16(init_state) || !al16(final_state))
    return SSD_ERR_INVALID_ARG;
  const int64_t l = tf32 ? tc32_chunk_len(shape->mimo_rank) : kernel_chunk_len(shape);
  const SsdLayout lay = tf32 ? chunk_layout(shape, l) : ssd_layout(shape);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0 ||
      workspace_bytes < lay.total)
    return SSD_ERR_WORKSPACE;

  char* ws = static_cast<char*>(workspace);
  GenericParams p;
  memset(&p, 0, sizeof(p));
  p.x = x;
  p.dA = dA;
  p.B = B;
  p.C = C;
  p.theta = theta;
  p.init = init_state;
  p.y = y;
  p.final_state = final_state;
  p.batch = shape->batch;
  p.T = shape->seqlen;
  p.H = shape->nheads;
  p.P = shape->headdim;
  p.N = shape->dstate;
  p.G = shape->ngroups;
  p.R = shape->mimo_rank;
  p.l = l;
  p.nch = (shape->seqlen + p.l - 1) / p.l;   // the last chunk may be short
  p.states = reinterpret_cast<float*>(ws + lay.states);
  p.cend = reinterpret_cast<float*>(ws + lay.cend);
  p.phi = theta ? reinterpret_cast<double*>(ws + lay.phi) : nullptr;
  p.phisum = theta ? reinterpret_cast<double*>(ws + lay.phisum) : nullptr;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.valid_len = valid_len;
  cudaError_t e;
  const int32_t variant = tf32 ? SSD_VARIANT_TC_TF32 : pick_variant(shape);
  if (variant == SSD_VARIANT_TC_BF16) {
    e = fused_bf16_forward(p, static_cast<cudaStream_t>(stream));
  } else if (variant == SSD_VARIANT_TC_TF32) {
    e = fp32_forward(p, static_cast<cudaStream_t>(stream));
  } else {
    e = generic_forward(p, shape->io_dtype == SSD_BF16, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

extern "C" {

ssd_status ssd_chunked_forward(const ssd_shape* shape, const void* x, const float* dA,
                               const void* B, const void* C, const float* theta,
                               const float* init_state, void* y, float* final_state,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return chunked_forward(shape, x, dA, B, C, theta, nullptr, init_state, y, final_state,
                         workspace, workspace_bytes, stream);
}

ssd_status ssd_chunked_forward_varlen(const ssd_shape* shape, const void* x, const float* dA,
                                      const void* B, const void* C, const float* theta,
                                      const int64_t* valid_len, const float* init_state, void* y,
                                      float* final_state, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (!valid_len || reinterpret_cast<uintptr_t>(valid_len) % alignof(int64_t) != 0)
    return SSD_ERR_INVALID_ARG;
  return chunked_forward(shape, x, dA, B, C, theta, valid_len, init_state, y, final_state,
                         workspace, workspace_bytes, stream);
}

ssd_status ssd_chunked_forward_tf32(const ssd_shape* shape, const void* x, const float* dA,
                                    const void* B, const void* C, const float* theta,
                                    const int64_t* valid_len, const float* init_state, void* y,
                                    float* final_state, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (valid_len && reinterpret_cast<uintptr_t>(valid_len) % alignof(int64_t) != 0)
    return SSD_ERR_INVALID_ARG;
  return chunked_forward(shape, x, dA, B, C, theta, valid_len, init_state, y, final_state,
                         workspace, workspace_bytes, stream, true);
}

int32_t ssd_trapezoidal_variant(const ssd_shape* shape) {
  if (check_trap_shape(shape) != SSD_OK) return SSD_VARIANT_NONE;
  if (trap_fused(shape)) return SSD_VARIANT_TC_BF16;
  const ssd_shape e = trap_expanded(shape);
  return pick_variant(&e);
}

size_t ssd_trapezoidal_workspace_bytes(const ssd_shape* shape) {
  if (check_trap_shape(shape) != SSD_OK) return 0;
  return trap_layout(shape).total;
}

}  // extern "C"

namespace {

ssd_status trapezoidal_forward(const ssd_shape* shape, const void* x, const float* dA,
                               const void* B, const void* C, const float* gamma,
                               const float* beta, const float* theta, const void* prev_x,
                               const void* prev_B, const int64_t* valid_len,
                               const float* init_state, void* y, float* final_state,
                               void* workspace, size_t workspace_bytes, void* stream) {
  const ssd_status sc = check_trap_shape(shape);
  if (sc != SSD_OK) return sc;
  if (!x || !dA || !B || !C || !gamma || !beta || !y) return SSD_ERR_INVALID_ARG;
  if ((shape->has_theta != 0) != (theta != nullptr)) return SSD_ERR_INVALID_ARG;
  if ((prev_x == nullptr) != (prev_B == nullptr)) return SSD_ERR_INVALID_ARG;
  if (!al16(x) || !al16(dA) || !al16(B) || !al16(C) || !al16(y) || !al16(theta) ||
      !al16(gamma) || !al16(beta) || !al16(init_state) || !al16(final_state))
    return SSD_ERR_INVALID_ARG;
  const TrapLayout lay = trap_layout(shape);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0 ||
      workspace_bytes < lay.total)
    return SSD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = shape->io_dtype == SSD_BF16;
  if (lay.fused) {
    if (!al16(prev_x) || !al16(prev_B)) return SSD_ERR_INVALID_ARG;   // copied as 16-byte words
    TrapFusedArgs f;
    memset(&f, 0, sizeof(f));
    f.x = x;
    f.B = B;
    f.C = C;
    f.prev_x = prev_x;
    f.prev_B = prev_B;
    f.gamma = gamma;
    f.beta = beta;
    f.y = y;
    f.xq = ws + lay.xq;
    f.bq = ws + lay.bq;
    f.cq = ws + lay.cq;
    f.wq = reinterpret_cast<float*>(ws + lay.wq);
    f.yq = ws + lay.yq;
    f.valid_len = valid_len;
    f.batch = shape->batch;
    f.T = shape->seqlen;
    f.R = shape->mimo_rank;
    f.H = shape->nheads;
    f.G = shape->ngroups;
    f.P = shape->headdim;
    f.N = shape->dstate;
    f.hdr = reinterpret_cast<WsHeader*>(ws);
    if (trap_fused_expand(f, st) != cudaSuccess) return SSD_ERR_CUDA;
    GenericParams p;
    memset(&p, 0, sizeof(p));
    p.x = f.xq;
    p.dA = dA;
    p.B = f.bq;
    p.C = f.cq;
    p.init = init_state;
    p.y = f.yq;
    p.final_state = final_state;
    p.batch = shape->batch;
    p.T = shape->seqlen;
    p.H = shape->nheads;
    p.P = shape->headdim;
    p.N = shape->dstate;
    p.G = shape->ngroups;
    p.R = 2 * shape->mimo_rank;
    p.l = shape->chunk_len;
    p.nch = (shape->seqlen + p.l - 1) / p.l;
    p.hdr = reinterpret_cast<WsHeader*>(ws);
    p.valid_len = valid_len;
    p.wrow = f.wq;
    if (fused_bf16_forward(p, st) != cudaSuccess) return SSD_ERR_CUDA;
    return trap_fused_compact(f, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  }
  const ssd_shape e = trap_expanded(shape);

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
  t.y = y;
  t.xh = reinterpret_cast<float*>(ws + lay.xh);
  t.bh = reinterpret_cast<float*>(ws + lay.bh);
  t.ch = reinterpret_cast<float*>(ws + lay.ch);
  t.yh = reinterpret_cast<float*>(ws + lay.yh);
  t.batch = shape->batch;
  t.T = shape->seqlen;
  t.R = shape->mimo_rank;
  t.H = shape->nheads;
  t.G = shape->ngroups;
  t.G2 = e.ngroups;
  t.P = shape->headdim;
  t.N = shape->dstate;
  t.valid_len = valid_len;
  t.hdr = reinterpret_cast<WsHeader*>(ws);
  if (trap_expand(t, bf16, st) != cudaSuccess) return SSD_ERR_CUDA;

  GenericParams p;
  memset(&p, 0, sizeof(p));
  p.x = t.xh;
  p.dA = dA;
  p.B = t.bh;
  p.C = t.ch;
  p.theta = theta;
  p.init = init_state;
  p.y = t.yh;
  p.final_state = final_state;
  p.batch = e.batch;
  p.T = e.seqlen;
  p.H = e.nheads;
  p.P = e.headdim;
  p.N = e.dstate;
  p.G = e.ngroups;
  p.R = e.mimo_rank;
  p.l = kernel_chunk_len(&e);
  p.nch = (e.seqlen + p.l - 1) / p.l;
  p.states = reinterpret_cast<float*>(ws + lay.inner.states);
  p.cend = reinterpret_cast<float*>(ws + lay.inner.cend);
  p.phi = theta ? reinterpret_cast<double*>(ws + lay.inner.phi) : nullptr;
  p.phisum = theta ? reinterpret_cast<double*>(ws + lay.inner.phisum) : nullptr;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.valid_len = valid_len;
  const cudaError_t ce = pick_variant(&e) == SSD_VARIANT_TC_TF32 ? fp32_forward(p, st)
                                                                  : generic_forward(p, false, st);
  if (ce != cudaSuccess) return SSD_ERR_CUDA;
  return trap_compact(t, bf16, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

extern "C" {

ssd_status ssd_trapezoidal_forward(const ssd_shape* shape, const void* x, const float* dA,
                                   const void* B, const void* C, const float* gamma,
                                   const float* beta, const float* theta, const void* prev_x,
                                   const void* prev_B, const float* init_state, void* y,
                                   float* final_state, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  return trapezoidal_forward(shape, x, dA, B, C, gamma, beta, theta, prev_x, prev_B, nullptr,
                             init_state, y, final_state, workspace, workspace_bytes, stream);
}

ssd_status ssd_trapezoidal_forward_varlen(const ssd_shape* shape, const void* x,
                                          const float* dA, const void* B, const void* C,
                                          const float* gamma, const float* beta,
                                          const float* theta, const void* prev_x,
                                          const void* prev_B, const int64_t* valid_len,
                                          const float* init_state, void* y, float* final_state,
                                          void* workspace, size_t workspace_bytes,
                                          void* stream) {
  if (!valid_len || reinterpret_cast<uintptr_t>(valid_len) % alignof(int64_t) != 0)
    return SSD_ERR_INVALID_ARG;
  return trapezoidal_forward(shape, x, dA, B, C, gamma, beta, theta, prev_x, prev_B, valid_len,
                             init_state, y, final_state, workspace, workspace_bytes, stream);
}

size_t selective_scan_workspace_bytes(int64_t batch, int64_t seqlen, int64_t d_model,
                                      int64_t d_state) {
  if (batch < 1 || seqlen < 1 || d_model < 1 || d_state < 1 || d_state > 64) return 0;
  int64_t t;
  if (!mul_ok(batch, seqlen, &t) || !mul_ok(t, d_model, &t)) return 0;
  const int64_t seg = ss_segment_length(seqlen);
  const int64_t nseg = (seqlen + seg - 1) / seg;
  size_t off = sizeof(WsHeader);
  off = align_up(off + sizeof(float) * (size_t)(batch * nseg * d_state * d_model), kWsAlign);
  off = align_up(off + sizeof(float) * (size_t)(batch * nseg * d_model), kWsAlign);
  return off;
}

ssd_status selective_scan_forward(const float* u, const float* delta, const float* A,
                                  const float* B, const float* C, const float* skip, float* y,
                                  int64_t batch, int64_t seqlen, int64_t d_model,
                                  int64_t d_state, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (batch < 1 || seqlen < 1 || d_model < 1 || d_state < 1) return SSD_ERR_INVALID_ARG;
  if (d_state > 64 || batch > 65535 || d_model > ((int64_t)65535 * 128)) return SSD_ERR_UNSUPPORTED;
  int64_t t;
  if (!mul_ok(batch, seqlen, &t) || !mul_ok(t, d_model, &t)) return SSD_ERR_INVALID_ARG;
  if (!u || !delta || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
  if (!al16(u) || !al16(delta) || !al16(A) || !al16(B) || !al16(C) || !al16(skip) || !al16(y))
    return SSD_ERR_INVALID_ARG;
  const size_t need = selective_scan_workspace_bytes(batch, seqlen, d_model, d_state);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0 ||
      workspace_bytes < need)
    return SSD_ERR_WORKSPACE;
  SelectiveScanParams p;
  memset(&p, 0, sizeof(p));
  p.u = u;
  p.delta = delta;
  p.A = A;
  p.B = B;
  p.C = C;
  p.skip = skip;
  p.y = y;
  p.batch = batch;
  p.T = seqlen;
  p.D = d_model;
  p.N = d_state;
  p.seg_len = ss_segment_length(seqlen);
  p.nseg = (seqlen + p.seg_len - 1) / p.seg_len;
  char* ws = static_cast<char*>(workspace);
  size_t off = sizeof(WsHeader);
  p.agg_h = reinterpret_cast<float*>(ws + off);
  off = align_up(off + sizeof(float) * (size_t)(batch * p.nseg * d_state * d_model), kWsAlign);
  p.agg_dt = reinterpret_cast<float*>(ws + off);
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  const cudaError_t e = selective_scan_onepass_supported(batch, d_model, d_state)
                            ? selective_scan_onepass_launch(p, static_cast<cudaStream_t>(stream))
                            : selective_scan_launch(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_workspace_status(void* workspace, void* stream, int64_t* detail) {
  if (detail) *detail = 0;
  if (!workspace) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SSD_ERR_CUDA;
  if (h.error != 0) {
    if (detail) *detail = h.detail;
    const int64_t zero[2] = {0, 0};
    if (cudaMemcpy(workspace, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return SSD_ERR_CUDA;
    return static_cast<ssd_status>(h.error);
  }
  return SSD_OK;
}

const char* ssd_status_string(ssd_status status) {
  switch (status) {
    case SSD_OK: return "SSD_OK";
    case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG";
    case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA";
    case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE";
    case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT";
    case SSD_ERR_INDEX: return "SSD_ERR_INDEX";
  }
  return "SSD_ERR_UNKNOWN";
}

int32_t ssd_abi_version(void) { return 1; }

}  // extern "C"
