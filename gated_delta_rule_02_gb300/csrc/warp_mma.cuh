// Warp-level tensor-core helpers shared by the kernels that keep a state
// tile in accumulator registers: mma.sync m16n8k16 (16-bit inputs, fp32
// accumulation), ldmatrix / stmatrix lane addressing, and the blockwise
// inverse of a unit lower-triangular matrix.  Inline PTX from the public ISA.
#pragma once

#include <type_traits>

#include "gdn_internal.cuh"

namespace gdn {
namespace wm {

__device__ __forceinline__ uint32_t s_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Two fp32 values rounded into one register of 16-bit pairs (low first).
template <typename E>
__device__ __forceinline__ uint32_t pk(float a, float b);
template <>
__device__ __forceinline__ uint32_t pk<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pk<__half>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
// The two values of a 16-bit pair register, widened.
template <typename E>
__device__ __forceinline__ float2 unpk(uint32_t r);
template <>
__device__ __forceinline__ float2 unpk<__nv_bfloat16>(uint32_t r) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r));
}
template <>
__device__ __forceinline__ float2 unpk<__half>(uint32_t r) {
  return __half22float2(*reinterpret_cast<const __half2*>(&r));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm2(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm2t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
// D (+)= A B, m16n8k16, 16-bit in, fp32 accumulate.  Fragments (g = lane / 4,
// c = lane % 4): A rows g, g+8 x cols 2c, 2c+1 and 8+2c, 9+2c; B rows 2c, 2c+1
// and 8+2c, 9+2c of column g; D (g, 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1).
// Two accumulator tiles side by side, packed to 16 bits, are one A fragment.
template <typename E>
__device__ __forceinline__ void mma(float* d, const uint32_t* a, const uint32_t* b) {
  if constexpr (std::is_same_v<E, __half>) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
}
__device__ __forceinline__ void stsm4t(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr),
               "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
// ldmatrix lane addresses (row-major 16-bit array, `ld` elements per row):
// A (m16 x k16) at (r0, c0); B (k16 x n8) from an [n][k] array (rows n0..,
// cols k0..); B from a [k][n] array (rows k0.., cols n0..), transposing.
template <typename E>
__device__ __forceinline__ uint32_t a_addr(const E* base, int ld, int r0, int c0, int lane) {
  return s_u32(base + (r0 + (lane & 15)) * ld + c0 + 8 * (lane >> 4));
}
template <typename E>
__device__ __forceinline__ uint32_t bnk_addr(const E* base, int ld, int n0, int k0, int lane) {
  return s_u32(base + (n0 + (lane & 7)) * ld + k0 + 8 * ((lane >> 3) & 1));
}
template <typename E>
__device__ __forceinline__ uint32_t bkn_addr(const E* base, int ld, int k0, int n0, int lane) {
  return s_u32(base + (k0 + (lane & 15)) * ld + n0);
}
// A (m16 x k16) of the transpose of a [k][m] array (rows k0.., cols m0..).
template <typename E>
__device__ __forceinline__ uint32_t at_addr(const E* base, int ld, int k0, int m0, int lane) {
  return s_u32(base + (k0 + (lane & 7) + 8 * (lane >> 4)) * ld + m0 + 8 * ((lane >> 3) & 1));
}

// Rows of 64 16-bit values (128 bytes) under the 128-byte swizzle of a TMA box
// whose base is 1024-byte aligned: byte offset of element (r, c), its 16-byte
// chunk c / 8 stored at chunk ^ (r % 8).
__device__ __forceinline__ uint32_t sw64(int r, int c) {
  return r * 128 + ((((c >> 3) ^ (r & 7))) << 4) + ((c & 7) << 1);
}
// The same four lane addressings as above, in such rows at shared address base.
__device__ __forceinline__ uint32_t sw_a(uint32_t base, int r0, int c0, int lane) {
  return base + sw64(r0 + (lane & 15), c0 + 8 * (lane >> 4));
}
__device__ __forceinline__ uint32_t sw_bnk(uint32_t base, int n0, int k0, int lane) {
  return base + sw64(n0 + (lane & 7), k0 + 8 * ((lane >> 3) & 1));
}
__device__ __forceinline__ uint32_t sw_bkn(uint32_t base, int k0, int n0, int lane) {
  return base + sw64(k0 + (lane & 15), n0);
}
__device__ __forceinline__ uint32_t sw_at(uint32_t base, int k0, int m0, int lane) {
  return base + sw64(k0 + (lane & 7) + 8 * (lane >> 4), m0 + 8 * ((lane >> 3) & 1));
}

// Blockwise inverse of a unit lower-triangular TC x TC matrix I + L (L
// strictly lower, fp32 rows of LD floats).  First the diagonal 8 x 8 blocks by
// forward substitution, a lane a column (lane l < TC: column l % 8 of block
// l / 8; the caller runs it on one warp); the entries above each diagonal
// block are zeroed.
template <int TC, int LD>
__device__ __forceinline__ void inverse_diag_blocks(const float (*lm)[LD], float (*tl)[LD],
                                                    int lane) {
  if (lane < TC) {
    const int o = lane & ~7, c = lane & 7;
    float x[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float a = (r == c) ? 1.f : 0.f;
#pragma unroll
      for (int s2 = 0; s2 < r; ++s2) a = fmaf(-lm[o + r][o + s2], x[s2], a);
      x[r] = a;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) tl[o + r][o + c] = x[r];
    for (int r = 0; r < o; ++r) tl[r][o + c] = 0.f;
  }
}
// Then, doubling the block size B: for every diagonal 2B x 2B block at (o, o),
// o = 2B p, whose B x B diagonal blocks T11, T22 are in tl, its lower-left
// block T21 = -T22 (L21 T11) (M = L21 T11 through the scratch array mt).
// All NTHR threads of the block call it.
template <int B, int TC, int NTHR, int LD>
__device__ __forceinline__ void combine_blocks(const float (*lm)[LD], float (*tl)[LD],
                                               float (*mt)[LD], int tid) {
  constexpr int kEl = (TC / (2 * B)) * B * B;
  for (int e = tid; e < kEl; e += NTHR) {
    const int p = e / (B * B), i = (e / B) % B, j = e % B, o = 2 * B * p;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < B; ++k) acc = fmaf(lm[o + B + i][o + k], tl[o + k][o + j], acc);
    mt[o + B + i][o + j] = acc;
  }
  __syncthreads();
  for (int e = tid; e < kEl; e += NTHR) {
    const int p = e / (B * B), i = (e / B) % B, j = e % B, o = 2 * B * p;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < B; ++k) acc = fmaf(tl[o + B + i][o + B + k], mt[o + B + k][o + j], acc);
    tl[o + B + i][o + j] = -acc;
  }
  __syncthreads();
}

}  // namespace wm
}  // namespace gdn
