// Internal interface between the C ABI (gdn_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace gdn {

// Head sizes: the tcgen05 prefill and the tensor-core short-T kernel are built
// for Dk = Dv = kHeadDim, the warp-level MMA prefills for 64/64 and 256/256;
// the decode, sequential short-T and fp32 SIMT kernels take Dk and Dv from
// {64, 128, 256}.
constexpr int kHeadDim = 128;
__host__ __device__ constexpr bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

// Input conventions selected by the options word of the *_ex entry points
// (same bits as GDN_OPT_* in include/gdn.h).
constexpr int kOptTiledHeads = 1;  // key head of value head hv is hv % Hk (else hv / (Hv/Hk))
constexpr int kOptLogGate = 2;     // g holds log-decays; the decay is exp(g)
constexpr int kOptL2NormQK = 4;    // every q and k row is used as x / |x|

__host__ __device__ __forceinline__ int key_head(int hv, int Hk, int Hv, int opts) {
  return (opts & kOptTiledHeads) ? hv % Hk : hv / (Hv / Hk);
}
// 1/|x| from a row's sum of squares (a zero row stays zero).
__device__ __forceinline__ float inv_norm(float sumsq) { return rsqrtf(fmaxf(sumsq, 1e-30f)); }

// Normalise `rows` fp32 rows of n <= 256 values (row stride `ld` floats) in
// shared memory, one warp per row; all `nthreads` threads of the block call this.
__device__ __forceinline__ void l2norm_rows_f32(float* s, int rows, int n, int ld, int tid,
                                                int nthreads) {
  const int lane = tid & 31;
  for (int r = tid >> 5; r < rows; r += nthreads >> 5) {
    float* row = s + r * ld;
    float ss = 0.f;
    for (int e = lane; e < n; e += 32) ss = fmaf(row[e], row[e], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float f = inv_norm(ss);
    for (int e = lane; e < n; e += 32) row[e] *= f;
  }
}

// The multiplicative decay from a stored gate value.
__device__ __forceinline__ float decay_of(float gate, int opts) {
  return (opts & kOptLogGate) ? exp2f(gate * 1.4426950408889634f) : gate;
}

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* beta;
  const float* state_in;  // may be nullptr (zero initial state)
  float* state_out;
  void* y;
  int B, T, Hk, Hv, chunk, dtype;
  int options;  // kOpt* bits
  int Dk, Dv;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* beta;
  const float* state_in;
  float* state_out;
  void* y;
  int B, Hk, Hv, dtype;
  int options;  // kOpt* bits
  int Dk, Dv;
  cudaStream_t stream;
};

// fp32 SIMT chunked path (any dtype and head size; serves fp32 inputs and the
// head pairs the tensor-core paths do not take).
size_t prefill_simt_workspace_bytes(int B, int T, int Hv, int chunk, int Dk, int Dv);
cudaError_t launch_prefill_simt(const PrefillArgs& a);

// tcgen05 chunked path (bf16 or fp16 inputs): prep + scan launches.
size_t prefill_tc_workspace_bytes(int B, int T, int Hv);
cudaError_t launch_prefill_tc(const PrefillArgs& a);
// Reads (and optionally clears) the tensor-core kernels' device error word;
// -1 if it cannot be read.
int prefill_tc_device_error(bool clear);
cudaError_t launch_wait_timeout_hook(cudaStream_t stream);
int wait_hook_device_error(bool clear);

// Short sequences (T <= kShortT): the sequential rule with the state on chip,
// no workspace.
constexpr int kShortT = 32;
cudaError_t launch_prefill_short(const PrefillArgs& a);
// The same on the tensor cores, one chunk per head (16-bit inputs, Dk = Dv =
// kHeadDim); launch_prefill_short routes there when short_tc_applies.
bool short_tc_applies(const PrefillArgs& a);
cudaError_t launch_prefill_short_tc(const PrefillArgs& a);
int short_tc_device_error(bool clear);

// Chunked prefill on warp-level tensor-core MMAs for 16-bit inputs with Dk =
// Dv = 64 and T > kShortT: a prep launch over every (head, chunk) and a scan
// launch over heads, through a workspace of prefill_mma_workspace_bytes.
bool mma_path_applies(int Dk, int Dv, int dtype, int T);
size_t prefill_mma_workspace_bytes(int B, int T, int Hv);
cudaError_t launch_prefill_mma(const PrefillArgs& a);
int prefill_mma_device_error(bool clear);
// The same for Dk = Dv = 256: the state of a head over four CTAs of 64 value
// rows, keys split over warp pairs.
bool mma256_path_applies(int Dk, int Dv, int dtype, int T);
size_t prefill_mma256_workspace_bytes(int B, int T, int Hv);
cudaError_t launch_prefill_mma256(const PrefillArgs& a);
int prefill_mma256_device_error(bool clear);

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry
// point (nullptr if unavailable).
typedef CUresult (*TmapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
TmapEncodeFn tmap_encoder();

// Streaming single-step decode.
cudaError_t launch_decode(const DecodeArgs& a);

// ---------------------------------------------------------------------------
// Small device helpers shared by the kernel files.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) {
  return __float2half_rn(x);
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Four consecutive elements widened to fp32 (16-byte / 8-byte aligned loads).
__device__ __forceinline__ void load4(const float* p, float* out) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  out[0] = t.x; out[1] = t.y; out[2] = t.z; out[3] = t.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* out) {
  const uint2 t = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&t.x);
  const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&t.y);
  const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
  out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
}
__device__ __forceinline__ void load4(const __half* p, float* out) {
  const uint2 t = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&t.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&t.y));
  out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
}

}  // namespace gdn
