// gdn_prefill_noalloc: the prefill for callers that cannot allocate device
// memory.
//
// gdn_prefill needs a device workspace that its caller allocates.  Some
// callers cannot do that: code that runs while a CUDA graph is being captured
// (where a cudaMalloc would break or synchronise the capture), plug-ins that
// receive raw device pointers from a host application but own no allocator,
// and latency-critical paths that must not pay for cudaMalloc's implicit
// device synchronisation.  This entry point instead uses a fixed scratch
// array that lives in the library image itself (one per GPU that loads the
// library, held until the process exits).  It allocates nothing.
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.cuh"

namespace {

// The scratch array (GDN_NOALLOC_SCRATCH_BYTES, 256-byte aligned).  Host code
// must not pass this name to a kernel: on the host it is only a stand-in for
// the device symbol, whose device address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per
// device (with that device current).  Returns nullptr on failure.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int gdn_prefill_noalloc(const void* q, const void* k, const void* v, const void* g,
                                   const void* beta, const float* state_in, float* state_out,
                                   void* y, int B, int T, int Hk, int Hv, int Dk, int Dv,
                                   int chunk, int dtype, void* stream) {
  // gdn_prefill_workspace_bytes returns 0 for any argument gdn_prefill would
  // reject; gdn_prefill itself then reports which one.
  const size_t need = gdn_prefill_workspace_bytes(B, T, Hk, Hv, Dk, Dv, chunk, dtype);
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_NOALLOC_LIMIT;
  void* scratch = scratch_address();
  if (!scratch) return GDN_ERR_CUDA;
  return gdn_prefill(q, k, v, g, beta, state_in, state_out, y, B, T, Hk, Hv, Dk, Dv, chunk,
                     dtype, scratch, (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}
