// Bounded-wait self-test: one thread waits on an mbarrier that nothing ever arrives on, for at
// most wait_ns, and then latches SSD_ERR_TIMEOUT in the workspace header -- the same give-up
// path every pipeline wait of the fused kernels takes.  It lets the failure path be exercised
// on a GPU without faulting or hanging it.
#include "common.cuh"
#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

constexpr int64_t kSelftestDetail = 900;
constexpr uint64_t kSelftestMaxNs = 100000000ull;   // 100 ms

__global__ void wait_selftest_kernel(WsHeader* hdr, uint64_t wait_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  tc::fence_mbar_init();
  if (!tc::mbar_wait_bounded(&bar, 0, wait_ns)) latch_error(hdr, SSD_ERR_TIMEOUT, kSelftestDetail);
}

}  // namespace
}  // namespace ssd

extern "C" ssd_status ssd_wait_selftest(void* workspace, size_t workspace_bytes, uint64_t wait_ns,
                                        void* stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % ssd::kWsAlign) != 0 ||
      workspace_bytes < sizeof(ssd::WsHeader))
    return SSD_ERR_WORKSPACE;
  if (wait_ns == 0 || wait_ns > ssd::kSelftestMaxNs) return SSD_ERR_INVALID_ARG;
  ssd::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<ssd::WsHeader*>(workspace), wait_ns);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
