// The C ABI of libgdn.so (declared in include/gdn.h): argument checking and
// dispatch.  Every check runs on the host before anything is enqueued, so a
// rejected call leaves every output untouched.
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.cuh"

namespace gdn {
TmapEncodeFn tmap_encoder() {
  static TmapEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TmapEncodeFn>(p);
  });
  return fn;
}
}  // namespace gdn

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Size limits, checked in 64-bit before any product is formed in int: the
// kernels index heads (B*Hv, times up to 16 row tiles or chunk counts) and
// tokens (B*T) with 32-bit grid and TMA coordinates.
constexpr long long kMaxHeads = 1LL << 20;          // B*Hv
constexpr long long kMaxTokens = (1LL << 31) - 1;   // B*T
constexpr long long kMaxHeadChunks = 1LL << 24;     // B*Hv*ceil(T/16)

int check_common(int B, int T, int Hk, int Hv, int Dk, int Dv, int dtype) {
  if (B <= 0 || T <= 0 || Hk <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0) return GDN_ERR_INVALID;
  if (Hv % Hk != 0) return GDN_ERR_INVALID;
  if (!gdn::head_dim_ok(Dk) || !gdn::head_dim_ok(Dv)) return GDN_ERR_UNSUPPORTED;
  const long long heads = (long long)B * Hv;
  if (heads > kMaxHeads || (long long)B * T > kMaxTokens ||
      heads * (((long long)T + 15) / 16) > kMaxHeadChunks)
    return GDN_ERR_UNSUPPORTED;
  if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F16)
    return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// Option bits the library understands (GDN_OPT_* in include/gdn.h).
constexpr int kKnownOptions = GDN_OPT_TILED_HEADS | GDN_OPT_LOG_GATE | GDN_OPT_L2NORM_QK;
static_assert(GDN_OPT_TILED_HEADS == gdn::kOptTiledHeads && GDN_OPT_LOG_GATE == gdn::kOptLogGate &&
                  GDN_OPT_L2NORM_QK == gdn::kOptL2NormQK,
              "option bits");

int check_pointers(const void* const* ptrs, int n) {
  for (int i = 0; i < n; ++i)
    if (ptrs[i] == nullptr) return GDN_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (!aligned16(ptrs[i])) return GDN_ERR_ALIGNMENT;
  return GDN_OK;
}
// The tensor-core prefill serves 16-bit inputs (bf16, fp16) with the head size
// it is built for.
bool use_tc(int Dk, int Dv, int dtype) {
  return (dtype == GDN_DTYPE_BF16 || dtype == GDN_DTYPE_F16) && Dk == gdn::kHeadDim &&
         Dv == gdn::kHeadDim;
}
}  // namespace

extern "C" {

size_t gdn_prefill_workspace_bytes(int B, int T, int Hk, int Hv, int Dk, int Dv,
                                   int chunk, int dtype) {
  if (check_common(B, T, Hk, Hv, Dk, Dv, dtype) != GDN_OK) return 0;
  if (chunk != 16 && chunk != 32 && chunk != 64) return 0;
  if (T <= gdn::kShortT) return 0;  // the short-T sequential kernel needs none
  if (use_tc(Dk, Dv, dtype)) return gdn::prefill_tc_workspace_bytes(B, T, Hv);
  if (gdn::mma_path_applies(Dk, Dv, dtype, T)) return gdn::prefill_mma_workspace_bytes(B, T, Hv);
  if (gdn::mma256_path_applies(Dk, Dv, dtype, T))
    return gdn::prefill_mma256_workspace_bytes(B, T, Hv);
  return gdn::prefill_simt_workspace_bytes(B, T, Hv, chunk, Dk, Dv);
}

int gdn_prefill_ex(const void* q, const void* k, const void* v, const void* g,
                   const void* beta, const float* state_in, float* state_out, void* y,
                   int B, int T, int Hk, int Hv, int Dk, int Dv, int chunk, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream, int options) {
  int st = check_common(B, T, Hk, Hv, Dk, Dv, dtype);
  if (st != GDN_OK) return st;
  if (options & ~kKnownOptions) return GDN_ERR_UNSUPPORTED;
  if (chunk != 16 && chunk != 32 && chunk != 64) return GDN_ERR_UNSUPPORTED;
  const void* req[] = {q, k, v, g, beta, state_out, y};
  st = check_pointers(req, 7);
  if (st != GDN_OK) return st;
  if (state_in && !aligned16(state_in)) return GDN_ERR_ALIGNMENT;
  const size_t need = gdn_prefill_workspace_bytes(B, T, Hk, Hv, Dk, Dv, chunk, dtype);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_ALIGNMENT;
  }
  gdn::PrefillArgs a{q, k, v, g, beta, state_in, state_out, y, B, T, Hk, Hv, chunk,
                     dtype, options, Dk, Dv, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream)};
  cudaError_t e = T <= gdn::kShortT                       ? gdn::launch_prefill_short(a)
                  : use_tc(Dk, Dv, dtype)                ? gdn::launch_prefill_tc(a)
                  : gdn::mma_path_applies(Dk, Dv, dtype, T) ? gdn::launch_prefill_mma(a)
                  : gdn::mma256_path_applies(Dk, Dv, dtype, T) ? gdn::launch_prefill_mma256(a)
                                                         : gdn::launch_prefill_simt(a);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_prefill(const void* q, const void* k, const void* v, const void* g,
                const void* beta, const float* state_in, float* state_out, void* y,
                int B, int T, int Hk, int Hv, int Dk, int Dv, int chunk, int dtype,
                void* workspace, size_t workspace_bytes, void* stream) {
  return gdn_prefill_ex(q, k, v, g, beta, state_in, state_out, y, B, T, Hk, Hv, Dk, Dv, chunk,
                        dtype, workspace, workspace_bytes, stream, 0);
}

int gdn_decode_step_ex(const void* q, const void* k, const void* v, const void* g,
                       const void* beta, const float* state_in, float* state_out,
                       void* y, int B, int Hk, int Hv, int Dk, int Dv, int dtype,
                       void* stream, int options) {
  int st = check_common(B, 1, Hk, Hv, Dk, Dv, dtype);
  if (st != GDN_OK) return st;
  if (options & ~kKnownOptions) return GDN_ERR_UNSUPPORTED;
  const void* req[] = {q, k, v, g, beta, state_in, state_out, y};
  st = check_pointers(req, 8);
  if (st != GDN_OK) return st;
  gdn::DecodeArgs a{q, k, v, g, beta, state_in, state_out, y, B, Hk, Hv, dtype, options,
                    Dk, Dv, static_cast<cudaStream_t>(stream)};
  cudaError_t e = gdn::launch_decode(a);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_decode_step(const void* q, const void* k, const void* v, const void* g,
                    const void* beta, const float* state_in, float* state_out,
                    void* y, int B, int Hk, int Hv, int Dk, int Dv, int dtype,
                    void* stream) {
  return gdn_decode_step_ex(q, k, v, g, beta, state_in, state_out, y, B, Hk, Hv, Dk, Dv, dtype,
                            stream, 0);
}

int gdn_device_status(int clear) {
  // Each translation unit with bounded waits has its own device error word.
  if (cudaDeviceSynchronize() != cudaSuccess) return GDN_ERR_CUDA;
  const int a = gdn::prefill_tc_device_error(clear != 0);
  const int b = gdn::wait_hook_device_error(clear != 0);
  const int c = gdn::short_tc_device_error(clear != 0);
  const int d = gdn::prefill_mma_device_error(clear != 0);
  const int f = gdn::prefill_mma256_device_error(clear != 0);
  if (a < 0 || b < 0 || c < 0 || d < 0 || f < 0) return GDN_ERR_CUDA;
  return (a || b || c || d || f) ? GDN_ERR_DEVICE_TIMEOUT : GDN_OK;
}

int gdn_selftest_wait_timeout(void* stream) {
  const cudaError_t e = gdn::launch_wait_timeout_hook(static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID: return "invalid argument (null pointer, size <= 0 or Hv % Hk != 0)";
    case GDN_ERR_UNSUPPORTED: return "unsupported shape, chunk, dtype or option (Dk, Dv in {64, 128, 256}, chunk 16/32/64, f32/bf16/f16; B*Hv <= 2^20, B*T < 2^31, B*Hv*ceil(T/16) <= 2^24)";
    case GDN_ERR_ALIGNMENT: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case GDN_ERR_WORKSPACE: return "workspace missing or smaller than gdn_prefill_workspace_bytes()";
    case GDN_ERR_CUDA: return "CUDA launch error";
    case GDN_ERR_DEVICE_TIMEOUT: return "a device-side wait gave up (bounded wait timed out)";
    case GDN_ERR_NOALLOC_LIMIT:
      return "problem needs more scratch than gdn_prefill_noalloc's fixed buffer (GDN_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown status";
  }
}

}  // extern "C"
