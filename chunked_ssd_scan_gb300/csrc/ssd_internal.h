// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ssdscan.h"

namespace ssd {

struct WsHeader;

// Arguments of the generic CUDA-core chunk pipeline.
struct GenericParams {
  const void* x;
  const float* dA;
  const void* B;
  const void* C;
  const float* theta;
  const float* init;
  void* y;
  float* final_state;
  int64_t batch, T, H, P, N, G, R, l, nch;
  float* states;    // [b, nch, H, P, N]: chunk states, overwritten with chunk-input states
  float* cend;      // [b, nch, H]: chunk-end cumulative log-decay
  double* phi;      // [b, nch+1, H, N/2]: chunk-start angles (mod 2 pi); the last one is Phi_{T-1}
  double* phisum;   // [b, nch, H, N/2]: per-chunk angle sums
  WsHeader* hdr;
  // Per-sequence valid lengths [batch] (device, may be null): steps t >= valid_len[b] are
  // padding, read as zero decay, zero input and no turn; y there is not written.
  const int64_t* valid_len;
  // Per fused row write weights [b, T*R, H] f32 (device, may be null; tensor-core kernel only):
  // row i's write enters the state and every later output scaled by w_i.
  const float* wrow;
};

#ifdef __CUDACC__
// Real steps of sequence b: valid_len[b] clamped to [0, T], or T without valid lengths.
__device__ __forceinline__ int64_t seq_steps(const GenericParams& p, int64_t b) {
  if (p.valid_len == nullptr) return p.T;
  const int64_t v = __ldg(p.valid_len + b);
  return v < 0 ? 0 : (v > p.T ? p.T : v);
}
#endif

size_t generic_state_smem(int64_t l, int64_t P, int64_t N, bool theta);
size_t generic_scan_smem(int64_t l, int64_t P, int64_t N, bool theta);
bool generic_supported(int64_t l, int64_t R, int64_t P, int64_t N, bool theta);
cudaError_t generic_forward(const GenericParams& p, bool bf16, cudaStream_t st);
// Pieces of the generic path shared with the fp32 tensor-core path: chunk-start angles
// (phi, phisum) and the K4 pass over chunks (states -> h_in in place, final state).
cudaError_t generic_phi(const GenericParams& p, cudaStream_t st);
cudaError_t generic_state_pass(const GenericParams& p, cudaStream_t st);
// fp32 I/O with P = N = 64 and R a power of two up to 64, over chunks of 128 fused rows
// (p.l * p.R = 128): the chunk states on the CUDA cores (K1, K3), the K4 pass, and the chunk
// scan (K2 + K5) as tcgen05 kind::tf32 products with split operands and 32-deep K blocks.
bool tc32_supported(int64_t P, int64_t N, int64_t R, bool bf16);
int64_t tc32_chunk_len(int64_t R);
cudaError_t fp32_forward(const GenericParams& p, cudaStream_t st);
cudaError_t tc32_scan(const GenericParams& p, cudaStream_t st);

// Host-side validation of an SSD shape (the ssd_chunked_* rules).
ssd_status shape_status(const ssd_shape* s);

// Trapezoidal form: the 2R-channel expansion around the generic pipeline.
struct TrapArgs {
  const void *x, *B, *C, *prev_x, *prev_B;   // I/O dtype
  const float *gamma, *beta, *theta;
  void* y;                                    // I/O dtype, R channels
  float *xh, *bh, *ch, *yh;                   // workspace: the expanded problem (fp32, 2R channels)
  int64_t batch, T, R, H, G, G2, P, N;        // G2: groups of the expanded B/C (H when theta)
  const int64_t* valid_len;                   // [batch] device, or null (no padding)
  WsHeader* hdr;                              // error word (index checks of the debug build)
};
cudaError_t trap_expand(const TrapArgs& a, bool bf16, cudaStream_t st);
cudaError_t trap_compact(const TrapArgs& a, bool bf16, cudaStream_t st);

// Trapezoidal form on the bf16 tensor-core kernel (no theta): the 2R channels hold exact bf16
// copies (x^ = [x_t, x_{t-1}], B^ = [B_t, B_{t-1}], C^ = [C_t, 0]) and gamma / beta become the
// kernel's per-row write weights.
struct TrapFusedArgs {
  const void *x, *B, *C, *prev_x, *prev_B;   // bf16
  const float *gamma, *beta;
  void* y;                                    // bf16, R channels
  void *xq, *bq, *cq, *yq;                    // workspace, bf16, 2R channels
  float* wq;                                  // workspace [b, T, 2R, H]
  const int64_t* valid_len;
  int64_t batch, T, R, H, G, P, N;
  WsHeader* hdr;
};
cudaError_t trap_fused_expand(const TrapFusedArgs& a, cudaStream_t st);
cudaError_t trap_fused_compact(const TrapFusedArgs& a, cudaStream_t st);

// Selective scan.
struct SelectiveScanParams {
  const float* u;
  const float* delta;
  const float* A;
  const float* B;
  const float* C;
  const float* skip;
  float* y;
  int64_t batch, T, D, N;
  int64_t seg_len, nseg;
  float* agg_h;     // [b, nseg, N, D]: segment-local end states, then segment-input states
  float* agg_dt;    // [b, nseg, D]: summed delta per segment
  WsHeader* hdr;
  // One-launch look-back form (set by its launcher): inclusive states [b, nseg, N, D] and one
  // flag per (channel block, segment), tagged with the call's epoch.
  float* inc_h;
  uint64_t* flags;
  uint64_t epoch;
};

int64_t ss_segment_length(int64_t T);

// Fused tcgen05 kernel for bf16 I/O.
bool fused_bf16_supported(int64_t T, int64_t H, int64_t P, int64_t N, int64_t R, int64_t l,
                          bool bf16, bool theta);
cudaError_t fused_bf16_forward(const GenericParams& p, cudaStream_t st);
// Workspace bytes of the fused kernel (header plus, when sequences are cut into time segments,
// the segment states) and its launches per call.
size_t fused_bf16_workspace_bytes(int64_t batch, int64_t T, int64_t H, int64_t R);
int fused_bf16_launches(int64_t batch, int64_t T, int64_t H, int64_t R);
cudaError_t selective_scan_launch(const SelectiveScanParams& p, cudaStream_t st);
// Single-kernel path for d_state in {8, 16, 32, 64} (no workspace use beyond the header).
bool selective_scan_onepass_supported(int64_t batch, int64_t D, int64_t N);
cudaError_t selective_scan_onepass_launch(const SelectiveScanParams& p, cudaStream_t st);

}  // namespace ssd
