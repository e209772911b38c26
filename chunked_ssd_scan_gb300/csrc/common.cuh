// Shared device/host helpers of the ssdscan library (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssdscan.h"

namespace ssd {

// ----------------------------------------------------------------------------------------------
// Workspace header: the first 256 bytes of every workspace.  Kernels latch device-side errors
// here instead of trapping.
// ----------------------------------------------------------------------------------------------
struct WsHeader {
  int32_t error;     // 0 = ok, otherwise an ssd_status value latched by a kernel
  int32_t pad0;
  int64_t detail;    // kernel-specific detail word of the first latched error
  uint32_t reserved[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header must be 256 bytes");

constexpr size_t kWsAlign = 256;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Latch the first error of a call into the workspace header (never traps).
__device__ inline void latch_error(WsHeader* hdr, int32_t code, int64_t detail) {
  if (atomicCAS(&hdr->error, 0, code) == 0) {
    hdr->detail = detail;
  }
}

// Index checks of the debug build (compiled with SSD_INDEX_CHECKS): an output access whose
// element index lies outside its buffer is skipped and SSD_ERR_INDEX is latched with the
// access's site number as detail.  In the normal build the check is the constant true.
#ifdef SSD_INDEX_CHECKS
__device__ inline bool index_ok(WsHeader* hdr, int64_t idx, int64_t extent, int site) {
  if (idx >= 0 && idx < extent) return true;
  if (hdr) latch_error(hdr, SSD_ERR_INDEX, site);
  return false;
}
#define SSD_INDEX_OK(hdr, idx, extent, site) ::ssd::index_ok((hdr), (int64_t)(idx), (int64_t)(extent), (site))
#else
#define SSD_INDEX_OK(hdr, idx, extent, site) true
#endif

// Load one element of an I/O tensor as fp32.
template <typename T>
__device__ __forceinline__ float ld_f32(const T* p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void st_from_f32(T* p, float v);
template <>
__device__ __forceinline__ void st_from_f32<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_from_f32<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 16-byte global->shared copy; src_bytes 0 writes zeros without reading.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}
// 4-byte asynchronous global -> shared copy (no alignment beyond 4 bytes needed).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

}  // namespace ssd
