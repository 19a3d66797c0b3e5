// Single-step decode: one token of every (b, hv) through the gated delta rule,
// streaming the fp32 state exactly once (read + write, in place allowed).
//
// Per value row r of S (every row evolves on its own):
//     x = S[r]·k,  z = S[r]·q                (one pass over the row)
//     d = beta (v_r - g x)
//     S[r] <- g S[r] + d k
//     y_r = (g z + d (k·q)) / sqrt(Dk)      (= S_new[r]·q / sqrt(Dk))
// (ferrox-core `gdn_chunk.rs`, "The algebra", one row; the post-update
// output of metaltile-std `gated_delta_wy.rs`, Algorithm step 6.)
//
// Layout on the GPU: one CTA of four warps per (b, hv) head; each warp owns
// Dv/4 rows.  Eight lanes share a row (the row-packing idea of the MLX PR
// "Pack gated_delta_seq: 8 value rows per SIMD-group", re-derived for 32-wide
// warps and 16-byte loads): lane `sub` of a row holds the float4s sub, sub+8,
// sub+16, ... of it (Dk/32 of them), so one warp-wide 16-byte load covers four
// whole rows of Dk = 128 and the two dot products reduce over 3 shuffle levels.
// Dk (64, 128 or 256) is a template parameter, Dv a runtime one.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 128;

__device__ __forceinline__ float4 ld_state(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st_state(float* p, float4 v) {
  __stcg(reinterpret_cast<float4*>(p), v);
}

// G = row groups (of four rows per warp) kept in flight per iteration.
template <typename T, int DK, int G>
__global__ void __launch_bounds__(kDecodeThreads)
decode_kernel(const T* __restrict__ q, const T* __restrict__ k,
              const T* __restrict__ v, const T* __restrict__ g,
              const T* __restrict__ beta, const float* state_in,
              float* state_out, T* __restrict__ y, int Hk, int Hv, int Dv, int opts,
              float scale) {
  constexpr int D = DK;
  constexpr int NJ = DK / 32;  // float4s of a row per lane
  const int bh = blockIdx.x;
  const int b = bh / Hv;
  const int hv = bh - b * Hv;
  const int hk = key_head(hv, Hk, Hv, opts);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int rg = lane >> 3;   // row within a group of four
  const int sub = lane & 7;   // lane within the row

  const T* kp = k + ((size_t)b * Hk + hk) * D;
  const T* qp = q + ((size_t)b * Hk + hk) * D;
  float kr[4 * NJ], qr[4 * NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    load4(kp + 4 * sub + 32 * j, kr + 4 * j);
    load4(qp + 4 * sub + 32 * j, qr + 4 * j);
  }
  if (opts & kOptL2NormQK) {  // the eight lanes of a row hold the whole vectors
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int i = 0; i < 4 * NJ; ++i) {
      sk = fmaf(kr[i], kr[i], sk);
      sq = fmaf(qr[i], qr[i], sq);
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      sk += __shfl_xor_sync(0xffffffffu, sk, off);
      sq += __shfl_xor_sync(0xffffffffu, sq, off);
    }
    const float fk = inv_norm(sk), fq = inv_norm(sq);
#pragma unroll
    for (int i = 0; i < 4 * NJ; ++i) {
      kr[i] *= fk;
      qr[i] *= fq;
    }
  }
  float kq = 0.f;
#pragma unroll
  for (int i = 0; i < 4 * NJ; ++i) kq = fmaf(kr[i], qr[i], kq);
  kq += __shfl_xor_sync(0xffffffffu, kq, 1);
  kq += __shfl_xor_sync(0xffffffffu, kq, 2);
  kq += __shfl_xor_sync(0xffffffffu, kq, 4);

  const float gt = decay_of(to_f32(g[bh]), opts);
  const float bt = to_f32(beta[bh]);
  const float* Sin = state_in + (size_t)bh * Dv * D;
  float* Sout = state_out + (size_t)bh * Dv * D;
  const T* vp = v + (size_t)bh * Dv;
  T* yp = y + (size_t)bh * Dv;
  const int wrows = Dv / 4;  // rows per warp

#pragma unroll 1
  for (int it = 0; it < wrows / (4 * G); ++it) {
    const int row0 = warp * wrows + it * 4 * G + rg;  // this lane's row in group gi: row0 + 4*gi
    float4 s[G][NJ];
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        s[gi][j] = ld_state(Sin + (size_t)(row0 + 4 * gi) * D + 4 * (sub + 8 * j));
    float vr[G];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) vr[gi] = to_f32(vp[row0 + 4 * gi]);

    float x[G], z[G];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      float xa = 0.f, za = 0.f;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        xa = fmaf(s[gi][j].x, kr[4 * j + 0], xa);
        xa = fmaf(s[gi][j].y, kr[4 * j + 1], xa);
        xa = fmaf(s[gi][j].z, kr[4 * j + 2], xa);
        xa = fmaf(s[gi][j].w, kr[4 * j + 3], xa);
        za = fmaf(s[gi][j].x, qr[4 * j + 0], za);
        za = fmaf(s[gi][j].y, qr[4 * j + 1], za);
        za = fmaf(s[gi][j].z, qr[4 * j + 2], za);
        za = fmaf(s[gi][j].w, qr[4 * j + 3], za);
      }
      x[gi] = xa;
      z[gi] = za;
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1)
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        x[gi] += __shfl_xor_sync(0xffffffffu, x[gi], off);
        z[gi] += __shfl_xor_sync(0xffffffffu, z[gi], off);
      }

#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const int row = row0 + 4 * gi;
      const float d = bt * (vr[gi] - gt * x[gi]);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        float4 o;
        o.x = fmaf(gt, s[gi][j].x, d * kr[4 * j + 0]);
        o.y = fmaf(gt, s[gi][j].y, d * kr[4 * j + 1]);
        o.z = fmaf(gt, s[gi][j].z, d * kr[4 * j + 2]);
        o.w = fmaf(gt, s[gi][j].w, d * kr[4 * j + 3]);
        st_state(Sout + (size_t)row * D + 4 * (sub + 8 * j), o);
      }
      if (sub == 0) yp[row] = from_f32<T>(fmaf(gt, z[gi], d * kq) * scale);
    }
  }
}

template <typename T, int DK>
cudaError_t launch_decode_t(const DecodeArgs& a) {
  // Two row groups in flight, one at Dk = 256 (registers).
  constexpr int G = DK == 256 ? 1 : 2;
  const float scale = 1.0f / sqrtf((float)DK);
  dim3 grid(a.B * a.Hv);
  decode_kernel<T, DK, G><<<grid, kDecodeThreads, 0, a.stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k),
      static_cast<const T*>(a.v), static_cast<const T*>(a.g),
      static_cast<const T*>(a.beta), a.state_in, a.state_out,
      static_cast<T*>(a.y), a.Hk, a.Hv, a.Dv, a.options, scale);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode_dk(const DecodeArgs& a) {
  if (a.Dk == 64) return launch_decode_t<T, 64>(a);
  if (a.Dk == 256) return launch_decode_t<T, 256>(a);
  return launch_decode_t<T, 128>(a);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a) {
  if (a.dtype == 0) return launch_decode_dk<float>(a);
  if (a.dtype == 2) return launch_decode_dk<__half>(a);
  return launch_decode_dk<__nv_bfloat16>(a);
}

}  // namespace gdn
