// Failure-detection hook for the bounded device waits.
//
// The tensor-core kernels wait on mbarriers (fed by TMA or by tensor-core
// commits) and on tile flags raised by other CTAs; each wait gives up after a
// fixed time, records a timeout in its translation unit's device error word
// and lets the kernel return, so a producer that never comes leaves the CUDA
// context usable and shows up as GDN_ERR_DEVICE_TIMEOUT on the host.  The
// kernel here runs those same two waits, from the same header, on things that
// never complete, so that tests can exercise the path without faulting the GPU.
#include <cuda_runtime.h>

#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

// A flag that no code raises.
__device__ int g_never_raised = 0;

__global__ void __launch_bounds__(32) wait_timeout_hook_kernel() {
  if (threadIdx.x != 0) return;
  __shared__ alignas(8) unsigned long long bar;
  const uint32_t b = ptx::smem_u32(&bar);
  ptx::mbar_init(b, 1);  // one arrival expected; nobody arrives
  ptx::fence_mbar_init();
  ptx::mbar_wait(b, 0);                 // phase 0 never completes: gives up after the limit
  ptx::wait_flag(&g_never_raised, 1);   // the flag stays 0: gives up after the limit
}

}  // namespace

cudaError_t launch_wait_timeout_hook(cudaStream_t stream) {
  wait_timeout_hook_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

int wait_hook_device_error(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, ptx::g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int z = 0;
    if (cudaMemcpyToSymbol(ptx::g_device_error, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace gdn
