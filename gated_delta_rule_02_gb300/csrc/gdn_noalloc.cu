// gdn_prefill_noalloc: the prefill for callers that cannot allocate device
// memory.
//
// gdn_prefill needs a device workspace that its caller allocates.  Some
// callers cannot do that: plug-ins that are handed raw device pointers by a
// host application but own no allocator (and must not grab memory behind the
// host's pool), and latency-critical paths that must not pay for cudaMalloc's
// implicit device synchronisation.  This entry point instead uses a fixed
// scratch array that lives in the library image itself (one copy per CUDA
// context that loads the library's kernels, held until that context is
// destroyed).  It allocates nothing.
#include <cuda.h>

#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.cuh"

namespace {

// The scratch array (GDN_NOALLOC_SCRATCH_BYTES, 256-byte aligned).  Host code
// must not pass this name to a kernel: on the host it is only a stand-in for
// the device symbol, whose device address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_scratch[GDN_NOALLOC_SCRATCH_BYTES];

// A __device__ array has one copy per CUDA context, so its address is looked
// up once per context (with that context current) and remembered under the
// context's unique ID; a context created later, even at a recycled handle
// value, gets an ID of its own and its own lookup.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static DriverFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return fns;
}

constexpr int kMaxContexts = 64;
std::mutex g_setup_mutex;
unsigned long long g_ctx_id[kMaxContexts] = {};
void* g_ctx_addr[kMaxContexts] = {};
int g_ctx_count = 0;

// Device address of g_scratch in the current context.  Returns nullptr if it
// cannot be determined (no context, driver entry points missing, or more than
// kMaxContexts contexts have used this entry point).
void* scratch_address() {
  const DriverFns& fns = driver_fns();
  if (!fns.get_current || !fns.get_id) return nullptr;
  CUcontext ctx = nullptr;
  if (fns.get_current(&ctx) != CUDA_SUCCESS) return nullptr;
  if (ctx == nullptr) {
    // No context is current on this thread yet: this runtime call binds the
    // current device's primary context (its result is looked up again below).
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
    if (fns.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
  }
  unsigned long long id = 0;
  if (fns.get_id(ctx, &id) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  for (int i = 0; i < g_ctx_count; ++i)
    if (g_ctx_id[i] == id) return g_ctx_addr[i];
  if (g_ctx_count == kMaxContexts) return nullptr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return nullptr;
  g_ctx_id[g_ctx_count] = id;
  g_ctx_addr[g_ctx_count] = p;
  ++g_ctx_count;
  return p;
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
