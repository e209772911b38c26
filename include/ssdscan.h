/*
 * ssdscan.h -- C ABI of the GB300 (sm_103a) chunked SSD scan and diagonal-A selective scan.
 *
 * Every function is extern "C", takes plain pointers and integer sizes, throws nothing, and
 * returns an ssd_status (or a size / string).  Pointers named as device pointers must be
 * device-accessible memory of the current CUDA device; the caller owns every buffer.  Compute
 * entry points are asynchronous on the given stream (a cudaStream_t passed as void*, NULL for
 * the legacy default stream) and never synchronise the device; they allocate no device memory.
 *
 * Sources of the operations (web pages, cited by title and section):
 *  - serial.rs (burn_mamba mamba3/ssd/serial.rs): the SSD chunk pipeline K1..K5 on rank-fused
 *    tensors -- K1 intra-chunk cumsum of dA, K2 C.B^T, K3 chunk states from pre-scaled V,
 *    K4 sequential state passing, K5 y = (L o CB) V + exp(cumA) C h_in.
 *  - segsum.rs (burn_mamba modules/misc/segsum.rs): the stable segment sum behind the causal mask.
 *  - scan.py (steertts mamba3/scan.py): cumulative angles Phi_t = sum_{s<=t} theta_s and the
 *    pairwise rotation rotate_by; the data-dependent rotation is absorbed into B and C.
 *  - SSM Selective Scan (LeetGPU write-up): the diagonal-A selective scan with skip term.
 *
 * Layouts (row-major, contiguous, innermost index last):
 *   x, y          [batch, seqlen, mimo_rank, nheads, headdim]     io dtype
 *   dA            [batch, seqlen, nheads]                         f32  (log-decay dt*A)
 *   B, C          [batch, seqlen, mimo_rank, ngroups, dstate]     io dtype
 *   theta         [batch, seqlen, nheads, dstate/2]               f32
 *   init_state    [batch, nheads, headdim, dstate]                f32
 *   final_state   [batch, nheads, headdim, dstate]                f32
 * Head h reads B/C group h / (nheads/ngroups).  x, B, C and y share io_dtype (f32 or bf16).
 */
#ifndef SSDSCAN_H
#define SSDSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ssd_status {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad divisibility, misalignment */
  SSD_ERR_UNSUPPORTED = 2, /* valid arguments outside what the kernels implement             */
  SSD_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed                    */
  SSD_ERR_WORKSPACE = 4,   /* workspace missing, misaligned or smaller than required         */
  SSD_ERR_TIMEOUT = 5,     /* a device-side wait gave up (latched in the workspace)          */
  SSD_ERR_INDEX = 6        /* index-checked build only: a kernel skipped an access outside its
                              buffer (latched in the workspace, detail = the access's site)   */
} ssd_status;

typedef enum ssd_dtype { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

typedef struct ssd_shape {
  int64_t batch;     /* b >= 1                                                   */
  int64_t seqlen;    /* T >= 1                                                   */
  int64_t nheads;    /* H >= 1                                                   */
  int64_t headdim;   /* P                                                        */
  int64_t dstate;    /* N (even when theta is given)                             */
  int64_t ngroups;   /* G, divides H                                             */
  int64_t mimo_rank; /* R >= 1; the fused chunk length is L = chunk_len * R      */
  int64_t chunk_len; /* l >= 1; need not divide T (the last chunk is then short) */
  int32_t io_dtype;  /* ssd_dtype of x, B, C and y                               */
  int32_t has_theta; /* 1 when theta will be passed (changes the workspace size) */
} ssd_shape;

/* Kernel families that ssd_chunked_forward may run for a shape. */
typedef enum ssd_kernel_variant {
  SSD_VARIANT_NONE = 0,    /* shape not supported                                    */
  SSD_VARIANT_GENERIC = 1, /* CUDA-core fp32 chunk pipeline (any supported shape)    */
  SSD_VARIANT_TC_BF16 = 2, /* fused tcgen05/TMEM kernel, bf16 operands, fp32 accum.  */
  SSD_VARIANT_TILED_F32 = 3, /* not returned by this library: the all-CUDA-core fp32 path that
                                SSD_VARIANT_TC_TF32 replaced (value kept for the ABI)        */
  SSD_VARIANT_TC_TF32 = 4    /* fp32, P = N = 64, R | 64: CUDA-core chunk states + K4 pass, the
                                chunk scan as tcgen05 kind::tf32 (split operands, 32-deep K
                                blocks)                                                      */
} ssd_kernel_variant;

/*
 * Bytes of device workspace ssd_chunked_forward needs for `shape` (0 if the shape is invalid).
 * The workspace must be 256-byte aligned.  Its contents need no initialisation: every call
 * resets what it uses, on the stream, before reading it.  One workspace must not be used by
 * two calls that can run concurrently.
 */
size_t ssd_chunked_workspace_bytes(const ssd_shape* shape);

/* Which kernel family ssd_chunked_forward will use for `shape` (SSD_VARIANT_NONE if none). */
int32_t ssd_chunked_variant(const ssd_shape* shape);

/*
 * Kernel launches one ssd_chunked_forward call makes for `shape` on the current device (0 if
 * the shape is not supported); for profiling and launch accounting.  The fused kernel cuts
 * sequences into time segments when there are fewer (batch, head) sequences than SMs, which
 * adds a state-only pre-pass and a carry launch.
 */
int32_t ssd_chunked_launches(const ssd_shape* shape);

/*
 * Chunked SSD forward scan (serial.rs: ssd_serial and K1..K5; scan.py: rotation absorption).
 *
 * Per (batch b, head h), with g = h / (H/G), Phi_t = sum_{s<=t} theta[b,s,h,:]:
 *   state_{-1} = init_state[b,h] (zeros if init_state is NULL)
 *   state_t    = exp(dA[b,t,h]) * Rot(theta_t) state_{t-1} + sum_r x[b,t,r,h,:] (outer) B[b,t,r,g,:]
 *   y[b,t,r,h,:] = state_t . C[b,t,r,g,:]                   (sum over dstate)
 *   final_state[b,h] = state_{T-1}  (physical frame: rotations applied, not the absorbed frame)
 * Rot(theta) turns each interleaved pair (2k, 2k+1) of the dstate axis by +theta[...,k].
 * x is the pre-scaled value (no dt factor) and no skip term is added, as in K3/K5.
 * The result equals the sequential recurrence above for any chunk_len; chunk_len sets how the
 * kernels tile time (K1..K5 granularity).  When it does not divide seqlen the last chunk is short
 * (scan.py page, chunked_scan): the kernels treat its missing steps as zero padding (dA = 0,
 * x = 0; moments.rs page: a pad step is an identity decay with a zero write, so the state passes
 * through unchanged), which leaves y of the real steps and the final state exactly those of the
 * unpadded recurrence, and write no y there.
 *
 * Arguments: x, B, C, y are device pointers of io_dtype; dA, theta, init_state, final_state are
 * device f32.  theta may be NULL only if shape->has_theta == 0 (and must be non-NULL otherwise);
 * init_state and final_state may be NULL.  x, B, C, y, dA, final_state must be 16-byte aligned.
 * workspace: device memory of at least ssd_chunked_workspace_bytes(shape), 256-byte aligned; its
 * first 256 bytes (the error header) must be zero before the first call (ssd_workspace_status
 * clears them again after reporting an error; the rest is scratch).
 * stream: cudaStream_t as void*.
 * Errors: INVALID_ARG / UNSUPPORTED / WORKSPACE are detected on the host before any launch and
 * leave every output untouched; CUDA reports a failed launch.  Device-side waits that give up
 * are latched in the workspace and reported by ssd_workspace_status.
 */
ssd_status ssd_chunked_forward(const ssd_shape* shape, const void* x, const float* dA,
                               const void* B, const void* C, const float* theta,
                               const float* init_state, void* y, float* final_state,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * ssd_chunked_forward for sequences of different real lengths in one padded batch (moments.rs
 * page: the valid-length mask of state_moments_phys and the pad rules of its module header).
 * valid_len: device int64 [batch], 8-byte aligned, non-NULL; each value is read clamped to
 * [0, seqlen].  Steps t >= valid_len[b] are padding and are treated as the page's zero pads:
 * dA = 0 (identity decay), no write (x and B taken as zero), no rotation (theta taken as zero).
 * So y at the real steps equals that of ssd_chunked_forward on the sequence cut at its length,
 * final_state[b] is the state at step valid_len[b] - 1 (init_state when the length is 0), and
 * y is not written at pad steps.  The inputs at pad steps may hold anything, NaN included:
 * the CUDA-core kernels do not read them, and the tensor-core kernel, which loads whole tiles,
 * zeroes the pad rows of x and B on chip before any product reads them.
 * Other arguments, workspace size, asynchrony and errors as for ssd_chunked_forward (a NULL or
 * misaligned valid_len is INVALID_ARG).
 */
ssd_status ssd_chunked_forward_varlen(const ssd_shape* shape, const void* x, const float* dA,
                                      const void* B, const void* C, const float* theta,
                                      const int64_t* valid_len, const float* init_state, void* y,
                                      float* final_state, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * The fp32 path with the chunk scan on the tensor core, which ssd_chunked_forward itself runs
 * for fp32 I/O with headdim = dstate = 64 and mimo_rank a power of two up to 64
 * (SSD_VARIANT_TC_TF32); this entry returns UNSUPPORTED for any other shape or dtype instead of
 * falling back to the generic CUDA-core pipeline.  The chunk scan (the serial.rs page's K2 and
 * K5: CB = C B^T, the decay mask, (L o CB) x and C h_in, the scan.py page's rotation absorbed
 * into B and C) runs as tcgen05.mma kind::tf32 over chunks of 128 fused rows (128 / mimo_rank
 * steps, whatever chunk_len says: the result does not depend on it).  Every fp32 operand is
 * split into a tf32 high part and its remainder and each pair takes three products (hi.lo,
 * lo.hi, then hi.hi), accumulated in TMEM over one 32-deep K block at a time and summed in fp32
 * round-to-nearest, so the tensor core's truncating accumulation stays within the fp32 gate
 * 1e-4 (1 + |y|).  K1 and K3 (chunk states) run as fp32 FMAs on the CUDA cores, K4 as the state
 * pass.  valid_len: NULL, or as for ssd_chunked_forward_varlen.  Other arguments, the workspace
 * size, asynchrony and errors as for ssd_chunked_forward.
 */
ssd_status ssd_chunked_forward_tf32(const ssd_shape* shape, const void* x, const float* dA,
                                    const void* B, const void* C, const float* theta,
                                    const int64_t* valid_len, const float* init_state, void* y,
                                    float* final_state, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* Bytes of device workspace ssd_trapezoidal_forward needs for `shape` (0 if unsupported). */
size_t ssd_trapezoidal_workspace_bytes(const ssd_shape* shape);

/*
 * Which kernel family ssd_trapezoidal_forward runs for `shape` (SSD_VARIANT_NONE if none):
 * SSD_VARIANT_TC_BF16 for bf16 I/O without rotation when the fused tensor-core kernel takes the
 * shape at 2·mimo_rank channels (P = 64, N = 128, 2R dividing 128 and at most 32, nheads % 4 = 0),
 * otherwise the family of the fp32 2R-channel expansion (TC_TF32 or GENERIC).
 */
int32_t ssd_trapezoidal_variant(const ssd_shape* shape);

/*
 * Trapezoidal Mamba-3 SSD forward (scan.py page, the trapezoidal forward; moments.rs page,
 * combined injections).  Per (batch b, head h), g = h / (H/G), with the step write
 * S_t = sum_r x[b,t,r,h,:] (outer) B[b,t,r,g,:]:
 *   h_t = Rot(theta_t) (exp(dA[b,t,h]) h_{t-1} + beta[b,t,h] S_{t-1}) + gamma[b,t,h] S_t
 *   y[b,t,r,h,:] = h_t . C[b,t,r,g,:];   final_state[b,h] = h_{T-1}
 * i.e. the beta term carries the previous step's write, turned by one step less of the
 * cumulative rotation than the gamma term.  S_{-1} = sum_r prev_x[b,r,h,:] (outer) prev_B[b,r,g,:]
 * (the last step of the previous call, for streaming) or zero when prev_x and prev_B are NULL.
 * h_{-1} = init_state (zeros if NULL); final_state may be NULL.
 * Arguments: as ssd_chunked_forward, plus gamma and beta (device f32 [batch, seqlen, nheads]) and
 * prev_x [batch, mimo_rank, nheads, headdim], prev_B [batch, mimo_rank, ngroups, dstate] (device,
 * io_dtype; both or neither).  The shape is the caller's (R = mimo_rank output and write
 * channels); the library runs it as one scalar-decay scan with 2R write channels
 * (x^ = [gamma x_t, beta x_{t-1}], B^ = [B_t, Rot(theta_t) B_{t-1}]) built in fp32 in the
 * workspace, on the CUDA-core chunk pipeline; for bf16 without rotation on a shape the fused
 * tensor-core kernel takes (ssd_trapezoidal_variant), the 2R channels are exact bf16 copies
 * (x^ = [x_t, x_{t-1}], B^ = [B_t, B_{t-1}], C^ = [C_t, 0]) and gamma, beta enter that kernel as
 * per-row write weights, so no product of two inputs is rounded to bf16.  Errors, asynchrony
 * and the workspace header as for ssd_chunked_forward; UNSUPPORTED when the expanded shape
 * exceeds the kernels' limits.  With the tensor-core form prev_x and prev_B must be 16-byte
 * aligned.
 */
ssd_status ssd_trapezoidal_forward(const ssd_shape* shape, const void* x, const float* dA,
                                   const void* B, const void* C, const float* gamma,
                                   const float* beta, const float* theta, const void* prev_x,
                                   const void* prev_B, const float* init_state, void* y,
                                   float* final_state, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * ssd_trapezoidal_forward with per-sequence valid lengths, under the rules of
 * ssd_chunked_forward_varlen (moments.rs page: zero pads carry the state through unchanged;
 * the chunk carry is read at the last real step).  Steps t >= valid_len[b] are padding: no
 * decay, no gamma or beta write, no turn, no y written; final_state[b] is h at step
 * valid_len[b] - 1.  Inputs at pad steps are not read.  Workspace, asynchrony and errors as for
 * ssd_trapezoidal_forward.
 */
ssd_status ssd_trapezoidal_forward_varlen(const ssd_shape* shape, const void* x,
                                          const float* dA, const void* B, const void* C,
                                          const float* gamma, const float* beta,
                                          const float* theta, const void* prev_x,
                                          const void* prev_B, const int64_t* valid_len,
                                          const float* init_state, void* y, float* final_state,
                                          void* workspace, size_t workspace_bytes,
                                          void* stream);

/* Bytes of device workspace ssd_rotation_variant_forward needs (0 if unsupported/invalid). */
size_t ssd_rotation_variant_workspace_bytes(const ssd_shape* shape, int64_t rope_dim,
                                            int32_t halves);

/*
 * Rotation variants of the rotated SSD forward (moments.rs page, RotationSeq::Angle with
 * rope_dim and rotate_pairwise; the page names them without defining them, so the plain
 * reading): the rotation turns only the first rope_dim state dimensions (0 = all of dstate;
 * even, <= dstate), with theta [batch, seqlen, nheads, rope_dim/2], and angle k turns the pair
 * (2k, 2k+1) when halves == 0 (rotate_pairwise, the ssd_chunked_forward convention) or
 * (k, k + rope_dim/2) when halves == 1.  Dimensions past rope_dim follow the unrotated
 * recurrence.  shape->has_theta must be 1.  Everything else (layouts, asynchrony, errors, the
 * workspace header) as ssd_chunked_forward, which it runs after reordering the state axis of
 * B, C and init_state in the workspace (halves only) and padding theta with zero angles
 * (rope_dim < dstate only); final_state is reordered back.
 */
ssd_status ssd_rotation_variant_forward(const ssd_shape* shape, int64_t rope_dim,
                                        int32_t halves, const void* x, const float* dA,
                                        const void* B, const void* C, const float* theta,
                                        const float* init_state, void* y, float* final_state,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace ssd_quaternion_forward needs (0 if the shape is invalid or
 * unsupported: has_theta must be 0 and dstate a multiple of 4). */
size_t ssd_quaternion_workspace_bytes(const ssd_shape* shape);

/*
 * Quaternion rotation of the rotated SSD forward (moments.rs page, RotationSeq::Quaternion
 * { cum_bshj4 }; named there, not defined, read plainly): qcum [batch, seqlen, nheads,
 * dstate/4, 4] f32 holds the cumulative unit quaternion Q_t = (w, x, y, z) of every 4-dimension
 * block of the state axis.  Block j of the state, the quaternion h[4j] + h[4j+1] i + h[4j+2] j
 * + h[4j+3] k, is turned at step t (before the decay and the write, as the angle rotation) by
 * left multiplication with Q_t Q_{t-1}^* (Q_{-1} = 1); with Q = cos(Phi) + i sin(Phi) this is
 * the interleaved angle rotation with both pairs of a block turned alike.  init_state and
 * final_state are in the physical frame.  shape->has_theta must be 0 and dstate % 4 == 0;
 * qcum and final_state 16-byte aligned.  Runs as B and C turned by Q_t^* per head into fp32 in
 * the workspace, ssd_chunked_forward on that fp32 problem (one group per head), and the final
 * state turned back by Q_{T-1}.  Layouts of x, dA, B, C, y, the states, asynchrony, errors and
 * the workspace header as ssd_chunked_forward.
 */
ssd_status ssd_quaternion_forward(const ssd_shape* shape, const void* x, const float* dA,
                                  const void* B, const void* C, const float* qcum,
                                  const float* init_state, void* y, float* final_state,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace ssd_chunked_backward needs for `shape` (0 if unsupported). */
size_t ssd_backward_workspace_bytes(const ssd_shape* shape);

/*
 * Reverse mode of the SSD forward (scan.py page: a scan that can be trained, its verify()
 * differentiating the rotated Mamba-3 scan; the moments.rs page's memory model of keeping
 * chunk-boundary states and recomputing inside a chunk).  For the loss
 * L = <dy, y> + <dfinal, final_state> of ssd_chunked_forward on the same inputs it writes
 *   dx [b,T,R,H,P] = dL/dx,  ddA [b,T,H] = dL/ddA,  dB, dC [b,T,R,G,N] = dL/dB, dL/dC (summed over
 *   the heads of a group),  dtheta [b,T,H,N/2] = dL/dtheta (has_theta = 1 only; NULL otherwise),
 *   dinit [b,H,P,N] = dL/dinit_state (may be NULL: not written).
 * dy [b,T,R,H,P] and dfinal [b,H,P,N] (NULL = zero) are device f32; x, B, C in io_dtype as for
 * the forward; dA, theta, init_state (NULL = zeros) f32; every gradient is device f32.  All
 * pointers 16-byte aligned, outputs not aliasing inputs.  theta and dtheta are given exactly when
 * shape->has_theta is 1.  The call recomputes the chunk-input states (64 fused rows per chunk,
 * i.e. 64/R steps, whatever shape->chunk_len says; seqlen need not be a multiple), carries
 * dL/dstate backwards across chunks, and forms each chunk's gradients from its 64 x 64 pairwise
 * products, all in fp32 on CUDA cores with the in-chunk log-decay sums in fp64.  With the
 * rotation it runs that per chunk on B^ = R(-phi)B, C^ = R(-phi)C per head in the workspace
 * (phi the angle accumulated since the chunk's start), turns the state at each chunk boundary,
 * turns dB^, dC^ back and forms dtheta from sums over one chunk plus a chunk-end term.
 * Limits: mimo_rank <= 64, headdim <= 64, dstate <= 128 and a multiple of 4 (else UNSUPPORTED).
 * dB and dC are zeroed by the call and, without the rotation, accumulated atomically, so their
 * low bits can vary between runs when H/G > 1.  Asynchrony, workspace and errors as
 * ssd_chunked_forward.
 */
ssd_status ssd_chunked_backward(const ssd_shape* shape, const void* x, const float* dA,
                                const void* B, const void* C, const float* theta,
                                const float* init_state, const float* dy, const float* dfinal,
                                float* dx, float* ddA, float* dB, float* dC, float* dtheta,
                                float* dinit, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Bytes of device workspace ssd_trapezoidal_backward needs for `shape` (0 if unsupported). */
size_t ssd_trapezoidal_backward_workspace_bytes(const ssd_shape* shape);

/*
 * Reverse mode of ssd_trapezoidal_forward (scan.py page: the trapezoidal forward, and a scan that
 * can be trained).  For the loss L = <dy, y> + <dfinal, final_state> on the same inputs it writes
 *   dx, ddA, dB, dC, dinit as ssd_chunked_backward; dgamma, dbeta [b,T,H] = dL/dgamma, dL/dbeta;
 *   dtheta [b,T,H,N/2] (has_theta = 1 only; NULL otherwise); dprev_x [b,R,H,P], dprev_B [b,R,G,N]
 *   = dL/dprev_x, dL/dprev_B (only when prev_x/prev_B are given; may be NULL).
 * Arguments as ssd_trapezoidal_forward plus dy [b,T,R,H,P] and dfinal [b,H,P,N] (NULL = zero),
 * device f32; every gradient is device f32 and 16-byte aligned; dinit may be NULL.  The call
 * builds the forward's 2R-channel expansion in the workspace, runs ssd_chunked_backward on it
 * (dy on the first R channels) and takes the gradients back through the expansion.  Limits: those
 * of ssd_chunked_backward for 2R channels (2R <= 64, headdim <= 64, dstate <= 128 and a multiple
 * of 4), else UNSUPPORTED.  Asynchrony, workspace and errors as ssd_chunked_forward.
 */
ssd_status ssd_trapezoidal_backward(
    const ssd_shape* shape, const void* x, const float* dA, const void* B, const void* C,
    const float* gamma, const float* beta, const float* theta, const void* prev_x,
    const void* prev_B, const float* init_state, const float* dy, const float* dfinal, float* dx,
    float* ddA, float* dB, float* dC, float* dgamma, float* dbeta, float* dtheta, float* dinit,
    float* dprev_x, float* dprev_B, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace selective_scan_forward needs (0 if the sizes are invalid). */
size_t selective_scan_workspace_bytes(int64_t batch, int64_t seqlen, int64_t d_model,
                                      int64_t d_state);

/*
 * Diagonal-A selective scan (SSM Selective Scan page, problem statement), all f32:
 *   h_{-1} = 0;  h_t[n] = exp(delta[b,t,d] A[d,n]) h_{t-1}[n] + delta[b,t,d] B[b,t,n] u[b,t,d]
 *   y[b,t,d] = sum_n C[b,t,n] h_t[n] + skip[d] u[b,t,d]
 * Layouts: u, delta, y [batch, seqlen, d_model]; A [d_model, d_state]; B, C [batch, seqlen,
 * d_state]; skip [d_model] (NULL = no skip term).  All device pointers, 16-byte aligned.
 * 1 <= d_state <= 64.  Same asynchrony, workspace and error rules as ssd_chunked_forward.
 */
ssd_status selective_scan_forward(const float* u, const float* delta, const float* A,
                                  const float* B, const float* C, const float* skip, float* y,
                                  int64_t batch, int64_t seqlen, int64_t d_model,
                                  int64_t d_state, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* Size of the fixed device scratch array behind selective_scan_forward_noalloc. */
#define SSD_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * Allocation-free variant of selective_scan_forward.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory (for example code that receives
 * only its input and output buffers through a fixed plugin interface, or code on a path where
 * cudaMalloc and the device synchronisation it can imply are not allowed).  It computes the same
 * function as selective_scan_forward but always on the segmented three-kernel path (per-segment
 * states, a carry pass, the output pass), whereas selective_scan_forward takes a one-pass kernel
 * for d_state in {8, 16, 32, 64} with d_model % 4 == 0; the two agree within the fp32 parity
 * bound |got - ref| <= 1e-4 (1 + |ref|), not bit for bit.  It takes no workspace: its scratch
 * lives in one fixed device array of SSD_NOALLOC_SCRATCH_BYTES (16 MiB) inside this library,
 * which every GPU that loads the library holds until the process exits.
 *   - Limit: (d_state + 1) * batch * ceil(seqlen / 64) * d_model floats must fit the array
 *     (the 4 x 4096 x 512 x 16 workload uses 8.9 MB); larger sizes return SSD_ERR_UNSUPPORTED
 *     before any launch.  Other argument errors are reported as in selective_scan_forward.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current, and the library keeps that address for the rest of the process;
 *     make that first call before any stream capture, and do not use this entry point after a
 *     cudaDeviceReset of that device (the kept address would belong to the destroyed context).
 *   - All calls on a device share the one array and it keeps the last call's contents.  Nothing
 *     in it has to start at zero (every call writes its scratch before reading it), but calls
 *     that can overlap on the GPU (different streams, or concurrent host threads) race on it and
 *     must be serialised by the caller.
 *   - It never calls cudaMalloc, cudaFree or any allocating routine.
 */
ssd_status selective_scan_forward_noalloc(const float* u, const float* delta, const float* A,
                                          const float* B, const float* C, const float* skip,
                                          float* y, int64_t batch, int64_t seqlen,
                                          int64_t d_model, int64_t d_state, void* stream);

/*
 * Reads (and clears) the device-side error word of a workspace after synchronising `stream`.
 * Returns SSD_OK, or SSD_ERR_TIMEOUT if a device wait of an earlier call on this workspace gave
 * up, or SSD_ERR_CUDA if the read itself failed.  *detail (if non-NULL) receives the
 * device-recorded detail word (0 when none).
 */
ssd_status ssd_workspace_status(void* workspace, void* stream, int64_t* detail);

/*
 * Failure-path self-test (the pages have no counterpart).  Launches one thread on `stream` that
 * waits on a device barrier nothing arrives on, for at most wait_ns nanoseconds (1 .. 1e8), and
 * then latches SSD_ERR_TIMEOUT with detail 900 in the workspace header, exactly as a pipeline
 * wait of the forward kernels does when it gives up.  ssd_workspace_status then reports it.
 * workspace: device memory of at least 256 bytes, 256-byte aligned, header zeroed (as for every
 * workspace before its first use).  Returns SSD_ERR_WORKSPACE / SSD_ERR_INVALID_ARG for bad
 * arguments (nothing launched), SSD_ERR_CUDA if the launch failed, else SSD_OK.
 */
ssd_status ssd_wait_selftest(void* workspace, size_t workspace_bytes, uint64_t wait_ns,
                             void* stream);

/* Human-readable name of a status code (static storage). */
const char* ssd_status_string(ssd_status status);

/* ABI version of this library (incremented on incompatible changes). */
int32_t ssd_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSDSCAN_H */
