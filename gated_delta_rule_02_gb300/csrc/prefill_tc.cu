// Chunked prefill on the tcgen05 tensor cores (bf16 inputs, fp32 state).
//
// The method is the chunked Woodbury-Young form of metaltile-std
// `gated_delta_wy.rs` (module docs, "Algorithm", steps 1-9), with the decay
// ratios formed as products (ferrox-core `gdn_chunk.rs`, "The algebra").  It is
// split in two launches:
//
// prep_tc_kernel, one CTA per (b, hv, 64-token tile), every tile in parallel.
// A tile holds 64/C chunks; all C x C matrices are block diagonal by chunk.
//   G1  [K;Q] K^T                      -> KK^T, QK^T          (steps 3, 6-prep)
//   gates: G_t (chunk-local prefix products), Gam[t][j] = g_{j+1}..g_t
//   T_L = (I + L)^-1,  L[t][j] = beta_j KK^T[t][j]          (step 4)
//   T_A = (I + A)^-1,  A[t][j] = beta_t Gam[t][j] KK^T[t][j] (step 5)
//       both by blocked forward substitution (16 x 16 diagonal blocks).
//   G2  [T_L 0; 0 T_A diag(beta)] [K; V]  -> P = T_L K, U = T_A (beta V)
//   G3  [diag(G) M 0; 0 Gam.QK^T] [P; U]  -> the state-free part of step 7
//       (M[t][i] = beta_i QK^T[t][i], i <= t) and y_local (step 6)
//   and writes to the workspace, per tile, in bf16:
//     A1 = per chunk [Pt; Qh], Pt = G_C beta P  (step 9),  Qh = G Q - G M P (step 7)
//     UY = [Ut; Yloc],         Ut = Gam[C-1][.] U          (step 9)
//   plus G_C (fp32) per chunk.
// scan_tc_kernel, one CTA per (b, hv, tile of R value rows); S (R x 128, fp32)
// lives in registers, one column per thread, and as a bf16 MMA operand in
// shared memory.  Per chunk:
//   MMA1  D1 = [Pt; Qh] S^T            -> S Pt^T and S Qh^T
//         W = Ut - S Pt^T;  y = (S Qh^T + Yloc) / sqrt(Dk)            (steps 7-8)
//   MMA2  D2 = K^T W^T                  S <- G_C S + (W K)           (step 9)
// A warp-specialised TMA producer double-buffers the tile operands.
#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

#include <mutex>

namespace gdn {
namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kTile = 64;   // tokens per tile
constexpr int kD = kHeadDim;
constexpr int kLdC = 65;    // padded fp32 row stride of the 64 x 64 matrices

// ------------------------------- workspace --------------------------------
struct WsLayout {
  size_t a1, uy, gc, total;
};
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline WsLayout ws_layout(int BH, int NT) {
  WsLayout w;
  const size_t tiles = (size_t)BH * NT;
  w.a1 = 0;
  w.uy = align256(tiles * 128 * kD * sizeof(bf16));
  w.gc = w.uy + align256(tiles * 128 * kD * sizeof(bf16));
  w.total = w.gc + align256(tiles * 4 * sizeof(float));
  return w;
}

// ------------------------------ smem helpers -------------------------------
// 128B-swizzled K-major tile of bf16 with 64 columns per 128-byte row: byte
// offset of element (row, col), col < 64.
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + (col & 7) * 2;
}
// Row `row` of an MN-major operand whose rows are 2*R bytes (R bf16), with the
// matching swizzle (R = 16: 32B, 32: 64B, 64: 128B); 16-byte chunk `ch`.
template <int R>
__device__ __forceinline__ uint32_t mn_row_chunk(int row, int ch) {
  constexpr int kRowBytes = 2 * R;
  constexpr int kMask = kRowBytes / 16 - 1;
  return row * kRowBytes + ((ch ^ ((row * kRowBytes >> 7) & kMask)) << 4);
}
template <int R>
__host__ __device__ constexpr uint32_t mn_layout() {
  return R == 16 ? kSw32 : (R == 32 ? kSw64 : kSw128);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void unpack8(uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    float2 p = __bfloat1622float2(h);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// ============================================================================
// prep kernel
// ============================================================================
constexpr int kPrepThreads = 256;
// shared-memory map (bytes from the 1024-aligned base)
constexpr uint32_t kOffKQ = 0;               // [K;Q] 2 halves x 128 rows x 128 B
constexpr uint32_t kOffV = 32 * 1024;        // V   2 halves x 64 rows x 128 B
constexpr uint32_t kOffA = 48 * 1024;        // A2 then A3: 2 halves x 128 rows x 128 B
constexpr uint32_t kOffB3 = 80 * 1024;       // [P; U] MN-major, 2 atoms x 128 rows x 128 B
constexpr uint32_t kOffF = 112 * 1024;       // fp32 area
constexpr int kMatF = 64 * kLdC;             // floats per 64 x 64 padded matrix
constexpr uint32_t kPrepSmem = kOffF + (5 * kMatF + 6 * 256 + 4 * 64) * 4 + 1024;

struct PrepF {            // fp32 views into the fp32 area
  float *kk, *qk, *gam, *tl, *ta, *z0, *z1, *g, *b, *gpre, *gsuf;
};

// Inverse of the unit lower-triangular (I + X), X strictly lower and block
// diagonal by chunk, by blocked forward substitution with 16 x 16 diagonal
// blocks; 128 threads (`u` = 0..127) cooperate, `bar` is their named barrier.
//   diagonal blocks: T_ii = (I + X_ii)^-1, one column per thread
//   block row i > 0: Z_ij = sum_{k=j}^{i-1} X_ik T_kj,  T_ij = -T_ii Z_ij
template <int C, typename XF>
__device__ void invert_unit_lower(XF X, float* Tm, float* Z, int u, int bar) {
  // zero the blocks above the diagonal
  for (int idx = u; idx < 64 * 64; idx += 128) {
    const int r = idx >> 6, c = idx & 63;
    if ((c >> 4) > (r >> 4)) Tm[r * kLdC + c] = 0.f;
  }
  if (u < 64) {
    const int bi = u >> 4, jj = u & 15, base = bi * 16;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = (r == jj) ? 1.f : 0.f;
#pragma unroll
      for (int s = 0; s < r; ++s) acc = fmaf(-X(base + r, base + s), x[s], acc);
      x[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Tm[(base + r) * kLdC + base + jj] = x[r];
  }
  named_bar_sync(bar, 128);
  if (C == 16) {
    for (int idx = u; idx < 64 * 64; idx += 128) {
      const int r = idx >> 6, c = idx & 63;
      if ((c >> 4) < (r >> 4)) Tm[r * kLdC + c] = 0.f;
    }
    named_bar_sync(bar, 128);
    return;
  }
  for (int bi = 1; bi < 4; ++bi) {
    // Z_{bi, bj} for bj < bi: bi * 256 outputs
    for (int idx = u; idx < bi * 256; idx += 128) {
      const int bj = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
      float acc = 0.f;
      for (int k = bj; k < bi; ++k)
#pragma unroll
        for (int s = 0; s < 16; ++s)
          acc = fmaf(X(bi * 16 + r, k * 16 + s), Tm[(k * 16 + s) * kLdC + bj * 16 + c], acc);
      Z[idx] = acc;
    }
    named_bar_sync(bar, 128);
    for (int idx = u; idx < bi * 256; idx += 128) {
      const int bj = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < 16; ++s)
        acc = fmaf(Tm[(bi * 16 + r) * kLdC + bi * 16 + s], Z[bj * 256 + s * 16 + c], acc);
      Tm[(bi * 16 + r) * kLdC + bj * 16 + c] = -acc;
    }
    named_bar_sync(bar, 128);
  }
}

template <int C>
__global__ void __launch_bounds__(kPrepThreads, 1)
prep_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_v, const bf16* __restrict__ g,
               const bf16* __restrict__ beta, bf16* __restrict__ wsA1, bf16* __restrict__ wsUY,
               float* __restrict__ wsGC, int T, int Hk, int Hv, int NT) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~(uintptr_t)1023);
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_base_sh;
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);

  float* fa = reinterpret_cast<float*>(sm + kOffF);
  PrepF f;
  f.kk = fa; f.qk = fa + kMatF; f.gam = fa + 2 * kMatF; f.tl = fa + 3 * kMatF;
  f.ta = fa + 4 * kMatF; f.z0 = fa + 5 * kMatF; f.z1 = f.z0 + 3 * 256;
  f.g = f.z1 + 3 * 256; f.b = f.g + 64; f.gpre = f.b + 64; f.gsuf = f.gpre + 64;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int tile = blockIdx.x, bh = blockIdx.y;
  const int b = bh / Hv, hv = bh - b * Hv, hk = hv / (Hv / Hk);
  const int t0 = tile * kTile;
  const size_t tile_id = (size_t)bh * NT + tile;

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tD1 = tmem, tD2 = tmem + 64, tD3 = tmem + 192;

  if (tid == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_v);
    mbar_expect_tx(bar_tma, 6 * 8192);
    tma_load_4d(sbase + kOffKQ, &tm_k, bar_tma, 0, hk, t0, b);
    tma_load_4d(sbase + kOffKQ + 16384, &tm_k, bar_tma, 64, hk, t0, b);
    tma_load_4d(sbase + kOffKQ + 8192, &tm_q, bar_tma, 0, hk, t0, b);
    tma_load_4d(sbase + kOffKQ + 24576, &tm_q, bar_tma, 64, hk, t0, b);
    tma_load_4d(sbase + kOffV, &tm_v, bar_tma, 0, hv, t0, b);
    tma_load_4d(sbase + kOffV + 8192, &tm_v, bar_tma, 64, hv, t0, b);
  }

  // Gates of the tile's tokens; padded tokens take g = 1, beta = 0.
  if (tid < 64) {
    const int tok = t0 + tid;
    const bool valid = tok < T;
    const size_t gi = ((size_t)b * T + tok) * Hv + hv;
    f.g[tid] = valid ? __bfloat162float(g[gi]) : 1.f;
    f.b[tid] = valid ? __bfloat162float(beta[gi]) : 0.f;
  }
  __syncthreads();
  if (tid < 64) {
    const int t = tid, cs = (t / C) * C, ce = cs + C - 1;
    float pre = 1.f;
    for (int i = cs; i <= t; ++i) pre *= f.g[i];
    float suf = 1.f;
    for (int i = t + 1; i <= ce; ++i) suf *= f.g[i];
    f.gpre[t] = pre;
    f.gsuf[t] = suf;
    float* row = f.gam + t * kLdC;
    for (int j = 0; j < 64; ++j) row[j] = 0.f;
    float r = 1.f;
    row[t] = 1.f;
    for (int j = t - 1; j >= cs; --j) {
      r *= f.g[j + 1];
      row[j] = r;
    }
  }

  bool ok = mbar_wait(bar_tma, 0);
  // G1: D1[128 x 64] = [K; Q] K^T.
  if (ok && tid == 0) {
    tc_fence_after();
    const uint32_t id1 = idesc_bf16(128, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t a = sbase + kOffKQ + (kk >> 2) * 16384 + (kk & 3) * 32;
      mma_bf16_ss(tD1, smem_desc(a, 16, 1024, kSw128), smem_desc(a, 16, 1024, kSw128), id1,
                  kk > 0);
    }
    mma_commit(bar_mma);
  }
  ok = ok && mbar_wait(bar_mma, 0);
  tc_fence_after();
  if (ok && tid < 128) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float* dst = tid < 64 ? f.kk + tid * kLdC : f.qk + (tid - 64) * kLdC;
#pragma unroll
    for (int c = 0; c < 64; c += 16) {
      float v[16];
      tmem_ld16(tD1 + lane_base + c, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) dst[c + j] = v[j];
    }
  }
  ok = __syncthreads_and(ok);

  // Steps 4 and 5: the two triangular inverses, one per 128-thread group.
  if (ok) {
    const float* kk = f.kk;
    const float* gam = f.gam;
    const float* bb = f.b;
    if (tid < 128) {
      auto XL = [=](int t, int j) { return j / C == t / C ? bb[j] * kk[t * kLdC + j] : 0.f; };
      invert_unit_lower<C>(XL, f.tl, f.z0, tid, 1);
    } else {
      auto XA = [=](int t, int j) { return bb[t] * gam[t * kLdC + j] * kk[t * kLdC + j]; };
      invert_unit_lower<C>(XA, f.ta, f.z1, tid - 128, 2);
    }
  }
  __syncthreads();

  // A2 = [T_L 0; 0 T_A diag(beta)] (K-major, 128B swizzle).
  if (ok) {
    for (int idx = tid; idx < 128 * 16; idx += kPrepThreads) {
      const int row = idx >> 4, ch = idx & 15, col0 = ch * 8;
      float v[8];
      const bool top = row < 64;
      const int t = row & 63;
      const bool live = top ? (col0 < 64) : (col0 >= 64);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = (col0 + e) & 63;
        v[e] = !live ? 0.f : (top ? f.tl[t * kLdC + c] : f.ta[t * kLdC + c] * f.b[c]);
      }
      st_shared_v4(sbase + kOffA + (col0 >> 6) * 16384 + sw128(row, col0 & 63), pack8(v));
    }
    fence_proxy_async();
  }
  ok = __syncthreads_and(ok);

  // G2: D2[128 x 128] = A2 [K; V]  (B MN-major: tokens are the reduction).
  if (ok && tid == 0) {
    tc_fence_after();
    const uint32_t id2 = idesc_bf16(128, 128, false, true);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t a = sbase + kOffA + (kk >> 2) * 16384 + (kk & 3) * 32;
      const uint64_t bdesc =
          kk < 4 ? smem_desc(sbase + kOffKQ + kk * 2048, 16384, 1024, kSw128)
                 : smem_desc(sbase + kOffV + (kk - 4) * 2048, 8192, 1024, kSw128);
      mma_bf16_ss(tD2, smem_desc(a, 16, 1024, kSw128), bdesc, id2, kk > 0);
    }
    mma_commit(bar_mma);
  }
  ok = ok && mbar_wait(bar_mma, 1);
  tc_fence_after();

  if (ok && tid < 128) {
    // Rows of D2: P (lanes 0..63) and U (lanes 64..127) -> B3 (bf16) and the
    // workspace rows Pt = G_C beta P and Ut = Gam[C-1][.] U.
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int m = tid & 63;
    const int c = m / C;
    const int brow = tid;  // B3 K-row: P rows 0..63, U rows 64..127
    float scale;
    bf16* gdst;
    if (tid < 64) {
      scale = f.gpre[c * C + C - 1] * f.b[m];
      gdst = wsA1 + (tile_id * 128 + 2 * C * c + (m % C)) * kD;
    } else {
      scale = f.gsuf[m];
      gdst = wsUY + (tile_id * 128 + m) * kD;
    }
#pragma unroll
    for (int col = 0; col < 128; col += 16) {
      float v[16];
      tmem_ld16(tD2 + lane_base + col, v);
      tmem_wait_ld();
      const uint4 raw0 = pack8(v), raw1 = pack8(v + 8);
      const int atom = col >> 6, cc = col & 63;
      st_shared_v4(sbase + kOffB3 + atom * 16384 + sw128(brow, cc), raw0);
      st_shared_v4(sbase + kOffB3 + atom * 16384 + sw128(brow, cc + 8), raw1);
      float w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = v[j] * scale;
      *reinterpret_cast<uint4*>(gdst + col) = pack8(w);
      *reinterpret_cast<uint4*>(gdst + col + 8) = pack8(w + 8);
    }
  } else if (ok) {
    // A3 = [diag(G) M 0; 0 Gam.QK^T] with M[t][i] = beta_i QK^T[t][i], i <= t.
    for (int idx = tid - 128; idx < 128 * 16; idx += 128) {
      const int row = idx >> 4, ch = idx & 15, col0 = ch * 8;
      const bool top = row < 64;
      const int t = row & 63;
      const bool live = top ? (col0 < 64) : (col0 >= 64);
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = (col0 + e) & 63;
        const bool causal = j <= t && j / C == t / C;  // same chunk, j <= t
        float val = 0.f;
        if (live && causal)
          val = top ? f.gpre[t] * f.b[j] * f.qk[t * kLdC + j]
                    : f.gam[t * kLdC + j] * f.qk[t * kLdC + j];
        v[e] = val;
      }
      st_shared_v4(sbase + kOffA + (col0 >> 6) * 16384 + sw128(row, col0 & 63), pack8(v));
    }
  }
  if (ok) fence_proxy_async();
  ok = __syncthreads_and(ok);

  // G3: D3[128 x 128] = A3 [P; U].
  if (ok && tid == 0) {
    tc_fence_after();
    const uint32_t id3 = idesc_bf16(128, 128, false, true);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t a = sbase + kOffA + (kk >> 2) * 16384 + (kk & 3) * 32;
      const uint64_t bdesc = smem_desc(sbase + kOffB3 + kk * 2048, 16384, 1024, kSw128);
      mma_bf16_ss(tD3, smem_desc(a, 16, 1024, kSw128), bdesc, id3, kk > 0);
    }
    mma_commit(bar_mma);
  }
  ok = ok && mbar_wait(bar_mma, 0);
  tc_fence_after();

  if (ok && tid < 128) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int m = tid & 63;
    const int c = m / C;
    const bool top = tid < 64;
    bf16* gdst = top ? wsA1 + (tile_id * 128 + 2 * C * c + C + (m % C)) * kD
                     : wsUY + (tile_id * 128 + 64 + m) * kD;
    const float gm = f.gpre[m];
#pragma unroll
    for (int col = 0; col < 128; col += 16) {
      float v[16];
      tmem_ld16(tD3 + lane_base + col, v);
      tmem_wait_ld();
      if (top) {  // Qh = G q - D3
        const int half = col >> 6, cc = col & 63;
        float q[16];
        unpack8(ld_shared_v4(sbase + kOffKQ + half * 16384 + 8192 + sw128(m, cc)), q);
        unpack8(ld_shared_v4(sbase + kOffKQ + half * 16384 + 8192 + sw128(m, cc + 8)), q + 8);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = gm * q[j] - v[j];
      }
      *reinterpret_cast<uint4*>(gdst + col) = pack8(v);
      *reinterpret_cast<uint4*>(gdst + col + 8) = pack8(v + 8);
    }
  }
  if (ok && tid < 64 / C) wsGC[tile_id * 4 + tid] = f.gpre[tid * C + C - 1];

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ============================================================================
// scan kernel
// ============================================================================
constexpr int kScanThreads = 160;  // warp 0: TMA producer; warps 1..4: compute
constexpr int kStages = 2;

template <int R>
struct ScanSmem {
  static constexpr uint32_t kA1 = 32 * 1024;
  static constexpr uint32_t kK = 16 * 1024;
  static constexpr uint32_t kUY = 2 * 64 * 2 * R;
  static constexpr uint32_t kStage = ((kA1 + kK + kUY) + 1023) & ~1023u;
  static constexpr uint32_t kS = 128 * 2 * R;  // S operand: 128 K-rows x R
  static constexpr uint32_t kW = 64 * 2 * R;   // W operand: up to 64 K-rows x R
  static constexpr uint32_t kOffS = kStages * kStage;
  static constexpr uint32_t kOffW = kOffS + ((kS + 1023) & ~1023u);
  static constexpr uint32_t kTotal = kOffW + ((kW + 1023) & ~1023u) + 1024;
};

template <int C, int R>
__global__ void __launch_bounds__(kScanThreads, 1)
scan_tc_kernel(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_uy, const float* __restrict__ wsGC,
               const float* state_in, float* state_out, bf16* __restrict__ y, int T, int Hk,
               int Hv, int NT, float scale) {
  using SM = ScanSmem<R>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~(uintptr_t)1023);
  __shared__ uint64_t bars[2 * kStages + 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, bh = blockIdx.y;
  const int b = bh / Hv, hv = bh - b * Hv, hk = hv / (Hv / Hk);
  const int r0 = tile * R;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[kStages + s]); };
  const uint32_t bar_mma = smem_u32(&bars[2 * kStages]);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(bar_mma, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 2 * R < 32 ? 32 : 2 * R);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tD1 = tmem, tD2 = tmem + R;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      prefetch_tmap(&tm_a1);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_uy);
      for (int n = 0; n < NT; ++n) {
        const int s = n % kStages;
        if (n >= kStages && !mbar_wait(empty_bar(s), ((n / kStages) - 1) & 1)) break;
        const uint32_t st = sbase + s * SM::kStage;
        const int row = (int)(((size_t)bh * NT + n) * 128);
        mbar_expect_tx(full_bar(s), SM::kA1 + SM::kK + SM::kUY);
        tma_load_2d(st, &tm_a1, full_bar(s), 0, row);
        tma_load_2d(st + 16384, &tm_a1, full_bar(s), 64, row);
        tma_load_4d(st + SM::kA1, &tm_k, full_bar(s), 0, hk, n * kTile, b);
        tma_load_4d(st + SM::kA1 + 8192, &tm_k, full_bar(s), 64, hk, n * kTile, b);
        tma_load_2d(st + SM::kA1 + SM::kK, &tm_uy, full_bar(s), r0, row);
        tma_load_2d(st + SM::kA1 + SM::kK + 64 * 2 * R, &tm_uy, full_bar(s), r0, row + 64);
      }
    }
    return;
  }

  // ------------------------------- compute --------------------------------
  const int L = ((warp & 3) << 5) | lane;  // TMEM lane = value-column index of S
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const bool issuer = (warp == 1 && lane == 0);
  const size_t sidx = ((size_t)bh * kD + r0) * kD + L;
  float s[R];
#pragma unroll
  for (int r = 0; r < R; ++r) s[r] = state_in ? state_in[sidx + (size_t)r * kD] : 0.f;

  auto write_rows = [&](uint32_t base, int row, const float* v) {
#pragma unroll
    for (int ch = 0; ch < R / 8; ++ch)
      st_shared_v4(base + mn_row_chunk<R>(row, ch), pack8(v + 8 * ch));
  };
  const uint32_t sS = sbase + SM::kOffS, sW = sbase + SM::kOffW;
  write_rows(sS, L, s);
  fence_proxy_async();
  named_bar_sync(1, 128);

  const uint32_t id1 = idesc_bf16(128, R, false, true);
  const uint32_t id2 = idesc_bf16(128, R, true, true);
  constexpr uint32_t kMnLay = mn_layout<R>();
  constexpr uint32_t kRowBytes = 2 * R;
  uint32_t mma_phase = 0;
  bool ok = true;

  for (int n = 0; n < NT && ok; ++n) {
    const int st_i = n % kStages;
    const uint32_t st = sbase + st_i * SM::kStage;
    const uint32_t stK = st + SM::kA1, stU = st + SM::kA1 + SM::kK, stY = stU + 64 * 2 * R;
    ok = mbar_wait(full_bar(st_i), (n / kStages) & 1);
    if (!ok) break;
    for (int c = 0; c < kTile / C; ++c) {
      const int tok0 = n * kTile + c * C;
      if (tok0 >= T) break;
      const float Gc = wsGC[((size_t)bh * NT + n) * 4 + c];
      if (issuer) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a = st + (kk >> 2) * 16384 + (2 * C * c) * 128 + (kk & 3) * 32;
          const uint64_t bd = smem_desc(sS + kk * 16 * kRowBytes, 0, 8 * kRowBytes, kMnLay);
          mma_bf16_ss(tD1, smem_desc(a, 16, 1024, kSw128), bd, id1, kk > 0);
        }
        mma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, mma_phase)) { abort_sh = 1; }
      mma_phase ^= 1;
      tc_fence_after();
      float d[R];
#pragma unroll
      for (int j = 0; j < R; j += 16) tmem_ld16(tD1 + lane_base + j, d + j);
      tmem_wait_ld();
      if (L < C) {
        // W = Ut - S Pt^T for this chunk's token L.
        const uint32_t urow = stU + (c * C + L) * kRowBytes;
        float w[R];
#pragma unroll
        for (int ch = 0; ch < R / 8; ++ch) {
          float u8[8];
          unpack8(ld_shared_v4(urow + ch * 16), u8);
#pragma unroll
          for (int e = 0; e < 8; ++e) w[ch * 8 + e] = u8[e] - d[ch * 8 + e];
        }
        write_rows(sW, L, w);
      } else if (L < 2 * C) {
        const int tl = L - C;
        if (tok0 + tl < T) {
          const uint32_t yrow = stY + (c * C + tl) * kRowBytes;
          bf16* yp = y + (((size_t)b * T + tok0 + tl) * Hv + hv) * kD + r0;
#pragma unroll
          for (int ch = 0; ch < R / 8; ++ch) {
            float y8[8];
            unpack8(ld_shared_v4(yrow + ch * 16), y8);
#pragma unroll
            for (int e = 0; e < 8; ++e) y8[e] = (y8[e] + d[ch * 8 + e]) * scale;
            *reinterpret_cast<uint4*>(yp + ch * 8) = pack8(y8);
          }
        }
      }
      tc_fence_before();
      fence_proxy_async();
      named_bar_sync(1, 128);
      if (abort_sh) { ok = false; break; }
      if (issuer) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
          const uint32_t a = stK + (c * C + 16 * kk) * 128;
          const uint64_t bd = smem_desc(sW + kk * 16 * kRowBytes, 0, 8 * kRowBytes, kMnLay);
          mma_bf16_ss(tD2, smem_desc(a, 8192, 1024, kSw128), bd, id2, kk > 0);
        }
        mma_commit(bar_mma);
      }
      if (!mbar_wait(bar_mma, mma_phase)) { abort_sh = 1; }
      mma_phase ^= 1;
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < R; j += 16) tmem_ld16(tD2 + lane_base + j, d + j);
      tmem_wait_ld();
#pragma unroll
      for (int r = 0; r < R; ++r) s[r] = fmaf(Gc, s[r], d[r]);
      write_rows(sS, L, s);
      tc_fence_before();
      fence_proxy_async();
      named_bar_sync(1, 128);
      if (abort_sh) { ok = false; break; }
    }
    if (issuer) mma_commit(empty_bar(st_i));  // stage free once its MMAs finish
  }

  if (ok) {
#pragma unroll
    for (int r = 0; r < R; ++r) state_out[sidx + (size_t)r * kD] = s[r];
  }
  tc_fence_before();
  named_bar_sync(1, 128);
  if (warp == 1) tmem_dealloc(tmem, 2 * R < 32 ? 32 : 2 * R);
}

// ============================================================================
// host side
// ============================================================================
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [B, T, H, 128] bf16 -> box {64 cols, 1 head, 64 tokens, 1 batch}, 128B swizzle.
bool make_bthd_map(CUtensorMap* m, const void* base, int B, int T, int H) {
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2,
                                 (cuuint64_t)T * H * kD * 2};
  const cuuint32_t box[4] = {64, 1, kTile, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [rows, 128] bf16 2-D view of a workspace region.
bool make_rows_map(CUtensorMap* m, const void* base, size_t rows, int box_cols, int box_rows,
                   bool swizzle) {
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kScanRows = 32;

template <int C>
cudaError_t launch_c(const PrefillArgs& a) {
  const int NT = (a.T + kTile - 1) / kTile;
  const int BH = a.B * a.Hv;
  const WsLayout w = ws_layout(BH, NT);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  bf16* wsA1 = reinterpret_cast<bf16*>(ws + w.a1);
  bf16* wsUY = reinterpret_cast<bf16*>(ws + w.uy);
  float* wsGC = reinterpret_cast<float*>(ws + w.gc);

  if (!encode_fn()) return cudaErrorNotSupported;
  CUtensorMap tk, tq, tv, ta1, tuy;
  if (!make_bthd_map(&tk, a.k, a.B, a.T, a.Hk) || !make_bthd_map(&tq, a.q, a.B, a.T, a.Hk) ||
      !make_bthd_map(&tv, a.v, a.B, a.T, a.Hv) ||
      !make_rows_map(&ta1, wsA1, (size_t)BH * NT * 128, 64, 128, true) ||
      !make_rows_map(&tuy, wsUY, (size_t)BH * NT * 128, kScanRows, 64, false))
    return cudaErrorInvalidValue;

  cudaError_t e = cudaFuncSetAttribute(prep_tc_kernel<C>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
  if (e != cudaSuccess) return e;
  using SM = ScanSmem<kScanRows>;
  e = cudaFuncSetAttribute(scan_tc_kernel<C, kScanRows>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kTotal);
  if (e != cudaSuccess) return e;

  prep_tc_kernel<C><<<dim3(NT, BH), kPrepThreads, kPrepSmem, a.stream>>>(
      tk, tq, tv, static_cast<const bf16*>(a.g), static_cast<const bf16*>(a.beta), wsA1, wsUY,
      wsGC, a.T, a.Hk, a.Hv, NT);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float scale = 1.0f / sqrtf((float)kD);
  scan_tc_kernel<C, kScanRows><<<dim3(kD / kScanRows, BH), kScanThreads, SM::kTotal, a.stream>>>(
      ta1, tk, tuy, wsGC, a.state_in, a.state_out, static_cast<bf16*>(a.y), a.T, a.Hk, a.Hv, NT,
      scale);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_tc_workspace_bytes(int B, int T, int Hv) {
  return ws_layout(B * Hv, (T + kTile - 1) / kTile).total;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a) {
  switch (a.chunk) {
    case 16: return launch_c<16>(a);
    case 32: return launch_c<32>(a);
    default: return launch_c<64>(a);
  }
}

int prefill_tc_device_error(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, ptx::g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int z = 0;
    cudaMemcpyToSymbol(ptx::g_device_error, &z, sizeof(int));
  }
  return v;
}

}  // namespace gdn
