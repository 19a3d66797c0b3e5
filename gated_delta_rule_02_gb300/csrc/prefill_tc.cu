// Chunked prefill on the tcgen05 tensor cores (bf16 inputs, fp32 state).
//
// The method is the chunked Woodbury-Young form of metaltile-std
// `gated_delta_wy.rs` (module docs, "Algorithm", steps 1-9), with the decay
// ratios formed as products (ferrox-core `gdn_chunk.rs`, "The algebra").  Two
// roles share a workspace:
//
// prep (prep_role): the state-free work of one 64-token tile of one (b, hv)
// head; every tile independent.  A tile holds 64/C chunks; all C x C matrices
// are block diagonal by chunk.
//   G1  [K;Q] K^T                      -> KK^T, QK^T          (steps 3, 6-prep)
//   gates: G_t (chunk-local prefix products), Gam[t][j] = g_{j+1}..g_t
//   T_L = (I + L)^-1,  L[t][j] = beta_j KK^T[t][j]          (step 4), by blocked
//       forward substitution; step 5 needs no second inverse:
//       (I + A)^-1 diag(beta) = diag(beta) (Gam . T_L),  A[t][j] = beta_t Gam[t][j] KK^T[t][j]
//   G2  [T_L; diag(beta)(Gam . T_L)] [K | V]  -> P = T_L K, U = (I + A)^-1 (beta V)
//   G3  [diag(G) M 0; 0 Gam.QK^T] [P; U]  -> the state-free part of step 7
//       (M[t][i] = beta_i QK^T[t][i], i <= t) and y_local (step 6)
//   and writes, per tile, in bf16: to the workspace A1 = per chunk [Pt; Qh] with
//   Pt = G_C beta P (step 9), Qh = G Q - G M P (step 7), and Ut = Gam[C-1][.] U
//   (step 9), plus G_C (fp32) per chunk; y_local / sqrt(Dk) straight into y.
// scan (scan_role128): one CTA per (b, hv) carries S (128 x 128, fp32) through
// the chunks.  Step 9 is regrouped as S <- G_C S - S M + N with M = Pt^T K and
// N = Ut^T K, so per chunk only the product with M waits for the state:
//   D  = K^T Ut + (-M^T) S^T;  S <- G_C S + D^T                       (step 9)
//   Y^T = S Qh^T;  y += Y / sqrt(Dk)  (TMA reduction)                 (steps 7-8)
// M^T = K^T Pt is formed a chunk ahead on the tensor cores.
//
// Launches: fused_prefill_kernel runs both roles in one cooperative launch
// (prep publishes each tile through a flag, the scan waits for it); for many
// heads, prep_tc_kernel then scan_head_kernel in stream order.
#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"

#include <algorithm>
#include <mutex>

namespace gdn {
namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kTile = 64;   // tokens per tile
constexpr int kD = kHeadDim;

// ------------------------------- workspace --------------------------------
struct WsLayout {
  size_t a1, u, gc, flags, total;
};
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline WsLayout ws_layout(int BH, int NT) {
  WsLayout w;
  const size_t tiles = (size_t)BH * NT;
  w.a1 = 0;
  w.u = align256(tiles * 128 * kD * sizeof(bf16));
  w.gc = w.u + align256(tiles * kTile * kD * sizeof(bf16));
  w.flags = w.gc + align256(tiles * 4 * sizeof(float));
  w.total = w.flags + align256(tiles * sizeof(int));
  return w;
}

// ------------------------------ smem helpers -------------------------------
// 128B-swizzled K-major tile of bf16 with 64 columns per 128-byte row: byte
// offset of element (row, col), col < 64.
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + (col & 7) * 2;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
// 16 consecutive floats from a 16-byte-aligned shared address.
__device__ __forceinline__ void ld16f(const float* p, float* o) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = *reinterpret_cast<const float4*>(p + 4 * i);
    o[4 * i] = f.x; o[4 * i + 1] = f.y; o[4 * i + 2] = f.z; o[4 * i + 3] = f.w;
  }
}
// 16-byte store through a generic pointer into shared memory: unlike the asm
// form it lets the compiler schedule the surrounding shared loads freely.
__device__ __forceinline__ void st_sm16(uint8_t* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
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

// x / |x| for row `row` of a bf16 tile whose rows are split in two 128B-swizzled
// 64-column halves `half_stride` bytes apart; the calling thread takes half
// `half` and its lane partner (lane ^ 1) the other half.
__device__ __forceinline__ void l2norm_row_sw128(uint8_t* base, int half_stride, int row,
                                                 int half) {
  uint8_t* hb = base + half * half_stride;
  float ss = 0.f;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    float v[8];
    unpack8(*reinterpret_cast<const uint4*>(hb + sw128(row, 8 * ch)), v);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  const float f = inv_norm(ss);
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint4* p = reinterpret_cast<uint4*>(hb + sw128(row, 8 * ch));
    float v[8];
    unpack8(*p, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] *= f;
    *p = pack8(v);
  }
}

// ============================================================================
// prep kernel
// ============================================================================
// The prep kernel is persistent: one CTA per SM holds two independent groups
// of eight warps, each with its own shared-memory map, 256 TMEM columns and
// mbarriers, each looping over tiles.
constexpr int kPrepGroups = 2;
constexpr int kPrepGroupThreads = 256;
constexpr int kPrepThreads = kPrepGroups * kPrepGroupThreads;
constexpr int kPrepIo = 4;  // I/O threads per group (lane 0 of warps 4-7)
// Shared-memory map of one group (bytes from its 1024-aligned base).
constexpr uint32_t kOffKQ = 0;        // [K;Q]: 2 halves x (64 K rows + 64 Q rows) x 128 B
constexpr uint32_t kOffV = 32768;     // V: 2 halves x 64 rows x 128 B
constexpr uint32_t kOffA3 = 49152;    // A3 (128 rows x 64 K-cols, one 128B half)
constexpr uint32_t kOffB = 65536;     // X | T_L | Z (fp32) during the inverse; then A2 over X;
                                      // then P, U (bf16, MN-major, 16 KB each)
constexpr int kLdX = 68;
constexpr uint32_t kOffTL = kOffB + 64 * kLdX * 4;
constexpr uint32_t kOffZ = kOffTL + 64 * kLdX * 4;       // 32 x 32 fp32
constexpr uint32_t kOffSmall = kOffZ + 32 * 32 * 4;      // per-token scalars
constexpr int kLdGd = 20;                                 // row stride of the in-block ratios
constexpr uint32_t kPrepGroupSmem = (kOffSmall + (64 * 6 + 256 + 4 + 64 * kLdGd) * 4 + 1023) & ~1023u;
constexpr uint32_t kPrepSmem = kPrepGroups * kPrepGroupSmem + 1024;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Warp-level 16 x 8 x 8 tf32 MMA (fp32 accumulate): the inverse's block
// products are too small for tcgen05 (M >= 64) and too latency-sensitive for
// scalar FMAs.  Fragment layout (g = lane / 4, t = lane % 4):
//   A 16 x 8 row-major: a0 (g, t) a1 (g+8, t) a2 (g, t+4) a3 (g+8, t+4)
//   B  8 x 8:           b0 (t, g) b1 (t+4, g)
//   D 16 x 8:           d0 (g, 2t) d1 (g, 2t+1) d2 (g+8, 2t) d3 (g+8, 2t+1)
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, const uint32_t* bb) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(bb[0]), "r"(bb[1]));
}
// D(16 x 8) = A[ra.., ca..](16 x K) * B[rb.., cb..](K x 8), fp32 row-major
// operands with row strides lda, ldb; K a multiple of 8.
template <int K>
__device__ __forceinline__ void warp_gemm_16x8(float* d, const float* A, int lda, const float* Bm,
                                               int ldb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  d[0] = d[1] = d[2] = d[3] = 0.f;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 8) {
    const uint32_t a[4] = {to_tf32(A[g * lda + k0 + t]), to_tf32(A[(g + 8) * lda + k0 + t]),
                           to_tf32(A[g * lda + k0 + t + 4]),
                           to_tf32(A[(g + 8) * lda + k0 + t + 4])};
    const uint32_t bb[2] = {to_tf32(Bm[(k0 + t) * ldb + g]), to_tf32(Bm[(k0 + t + 4) * ldb + g])};
    mma_tf32(d, a, bb);
  }
}
__device__ __forceinline__ void warp_store_16x8(float* D, int ldd, const float* d, int lane,
                                                float sign) {
  const int g = lane >> 2, t = lane & 3;
  D[g * ldd + 2 * t] = sign * d[0];
  D[g * ldd + 2 * t + 1] = sign * d[1];
  D[(g + 8) * ldd + 2 * t] = sign * d[2];
  D[(g + 8) * ldd + 2 * t + 1] = sign * d[3];
}

// T = (I + X)^-1 for X strictly lower triangular and block diagonal by chunk
// (zero across chunks), by blocked forward substitution:
//   16 x 16 diagonal blocks   T_ii = (I + X_ii)^-1       (one column per thread)
//   32 x 32 blocks (C >= 32)  T_10 = -T_11 X_10 T_00      (per 16-block pair)
//   64 x 64 (C = 64)          T_BA = -T_BB X_BA T_AA      (32-block halves)
// The block products run on warp-level tf32 MMAs; the group's 256 threads call
// this (u = thread index in the group, sync = the group's barrier).
template <int C, typename Sync>
__device__ void invert_unit_lower(const float* X, float* Tm, float* Zs, int u, Sync sync) {
  for (int idx = u; idx < 64 * 64; idx += kPrepGroupThreads) {
    const int r = idx >> 6, c = idx & 63;
    if ((c >> 4) > (r >> 4) || (c / C) != (r / C)) Tm[r * kLdX + c] = 0.f;
  }
  if (u < 64) {
    const int base = (u >> 4) * 16, jj = u & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float a0 = (r == jj) ? 1.f : 0.f, a1 = 0.f;
      const float* xr = X + (base + r) * kLdX + base;
#pragma unroll
      for (int s = 0; s + 1 < r; s += 2) {
        a0 = fmaf(-xr[s], x[s], a0);
        a1 = fmaf(-xr[s + 1], x[s + 1], a1);
      }
      if (r & 1) a0 = fmaf(-xr[r - 1], x[r - 1], a0);
      x[r] = a0 + a1;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Tm[(base + r) * kLdX + base + jj] = x[r];
  }
  sync();
  const int w = u >> 5, lane = u & 31;
  if constexpr (C >= 32) {
    // Pairs (0,1) and (2,3): warp w < 4 handles pair w/2, columns 8*(w%2)..
    float d[4];
    const int p = (w >> 1) & 1, nt = w & 1;
    const int r0 = (2 * p + 1) * 16, c0 = 2 * p * 16;
    if (w < 4) {
      warp_gemm_16x8<16>(d, X + r0 * kLdX + c0, kLdX, Tm + c0 * kLdX + c0 + nt * 8, kLdX, lane);
      warp_store_16x8(Zs + p * 256 + nt * 8, 16, d, lane, 1.f);
    }
    sync();
    if (w < 4) {
      warp_gemm_16x8<16>(d, Tm + r0 * kLdX + r0, kLdX, Zs + p * 256 + nt * 8, 16, lane);
      warp_store_16x8(Tm + r0 * kLdX + c0 + nt * 8, kLdX, d, lane, -1.f);
    }
    sync();
  }
  if constexpr (C == 64) {
    // M = X[32:64][0:32] T[0:32][0:32], then T[32:64][0:32] = -T[32:64][32:64] M;
    // warp w computes the 16 x 8 tile (w/4, w%4) of each.
    float d[4];
    const int mt = w >> 2, nt = w & 3;
    warp_gemm_16x8<32>(d, X + (32 + mt * 16) * kLdX, kLdX, Tm + nt * 8, kLdX, lane);
    warp_store_16x8(Zs + mt * 16 * 32 + nt * 8, 32, d, lane, 1.f);
    sync();
    warp_gemm_16x8<32>(d, Tm + (32 + mt * 16) * kLdX + 32, kLdX, Zs + nt * 8, 32, lane);
    warp_store_16x8(Tm + (32 + mt * 16) * kLdX + nt * 8, kLdX, d, lane, -1.f);
    sync();
  }
}

// Everything the prep work needs (the tensor maps are kernel parameters).
struct PrepParams {
  const bf16* k;  // the raw inputs, for L2 prefetches
  const bf16* q;
  const bf16* v;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_a1s;
  const CUtensorMap* tm_us;
  const bf16* g;
  const bf16* beta;
  float* wsGC;
  int T, Hk, Hv, NT, BH;
  int opts;  // kOpt* bits
  // y_loc / sqrt(Dk) goes straight to y ([B, T, Hv, 128], 64-token boxes); the
  // scan then adds Qh S^T / sqrt(Dk) to it.
  const CUtensorMap* tm_y;
  float yscale;
};

// The prep work of one CTA (both groups): CTA `cta_rank` of `n_ctas` doing prep.
// With `flags`, each finished tile (b*Hv + hv, n) is published by raising
// flags[(b*Hv + hv) * NT + n] to kPrepIo: each I/O thread adds 1 once its own
// stores of the tile are in memory.
template <int C>
__device__ __forceinline__ void prep_role(const PrepParams& P, uint8_t* smem_raw, int cta_rank,
                                          int n_ctas, int* flags) {
  const int T = P.T, Hk = P.Hk, Hv = P.Hv, NT = P.NT, BH = P.BH, opts = P.opts;
  const bf16* __restrict__ g = P.g;
  const bf16* __restrict__ beta = P.beta;
  float* __restrict__ wsGC = P.wsGC;
  __shared__ uint64_t bars[kPrepGroups][4];
  __shared__ uint32_t tmem_base_sh;
  __shared__ float carry_sh[kPrepGroups];
  __shared__ int abort_sh[kPrepGroups];
  const int grp = threadIdx.x / kPrepGroupThreads;
  const int tid = threadIdx.x % kPrepGroupThreads, warp = tid >> 5;  // within the group
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~(uintptr_t)1023) +
                grp * kPrepGroupSmem;
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar_tma = smem_u32(&bars[grp][0]), bar_mma = smem_u32(&bars[grp][1]);
  // G2 and G3 completions of the P stream (bar_p) and of the U stream (bar_u):
  // two per tile each, so the first wait of a tile is on parity 0, the second on 1.
  const uint32_t bar_p = smem_u32(&bars[grp][2]), bar_u = smem_u32(&bars[grp][3]);
  // Named barriers of the group: the whole group, its gate warps (0-3) and the
  // two warps of the prefix sum.
  const int sync_id = 1 + 2 * grp, gates_id = 2 + 2 * grp, carry_id = 5 + grp;
  // Warps 0, 1, 4, 5 (TMEM lanes 0-63: X, later the P stream) and warps 2, 3, 6,
  // 7 (lanes 64-127: the U stream).
  const int pstream_id = 7 + grp, ustream_id = 9 + grp;
  const bool pstream = (warp & 3) < 2;
  float* X = reinterpret_cast<float*>(sm + kOffB);               // 64 x 68 fp32
  float* TL = reinterpret_cast<float*>(sm + kOffTL);             // 64 x 68 fp32
  float* Zs = reinterpret_cast<float*>(sm + kOffZ);              // 32 x 32 fp32
  float* lam = reinterpret_cast<float*>(sm + kOffSmall);         // chunk-local sum of log2 g
  float* bta = lam + 64;
  float* gsuf = bta + 64;   // g_{t+1} ... g_{chunk end}
  float* gpw = gsuf + 64;   // G_t = g_{chunk start} ... g_t
  float* sfac = gpw + 64;   // 2^(lam[end of t's 16-block] - lam_t)
  float* rfac = sfac + 64;  // [64][4]: 2^(lam_t - lam[end of block b]), b before t's block
  float* gc = rfac + 256;   // G at each chunk's end
  float* gdiag = gc + 4;    // [64][kLdGd]: Gam[t][j] for j in t's 16-block, j <= t
  auto gsync = [&]() { named_bar_sync(sync_id, kPrepGroupThreads); };
  // Group-wide AND of ok (sticky: a group that failed a wait stops).
  auto gsync_and = [&](bool v) {
    if (!v) abort_sh[grp] = 1;
    gsync();
    return abort_sh[grp] == 0;
  };

  if (threadIdx.x == 0) {
    for (int q = 0; q < kPrepGroups; ++q) {
      for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[q][i]), 1);
      abort_sh[q] = 0;
    }
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(&tmem_base_sh), 256 * kPrepGroups);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh + 256 * grp;

  // Tiles in chunk-major order (every head's tile n before any head's n+1);
  // group gid takes gid, gid + ngroups, ...
  const int total = BH * NT;
  const int ngroups = n_ctas * kPrepGroups;
  const int gid = cta_rank * kPrepGroups + grp;
  auto head_of = [&](int lin) { return lin % BH; };
  auto tile_of = [&](int lin) { return lin / BH; };
  // The group's TMA traffic is spread over four threads (lane 0 of warps 4-7),
  // since one thread issues these instructions slowly.  I/O thread `io`
  // owns one 64-column half: io 0/1 load K and Q half io and store the Pt and
  // Qh halves staged over K; io 2/3 load V half io-2 and store the Ut and y_loc
  // halves staged over V.  Each waits for its own stores before reloading the
  // region they read.  io 0 posts the byte count of the whole tile.
  const int io = (warp >= 4 && (tid & 31) == 0) ? warp - 4 : -1;
  // K and V of tile `lin` (io 0 also posts the byte count of K, Q and V) ...
  auto load_kv = [&](int lin) {
    const int bh = head_of(lin), n = tile_of(lin);
    const int b = bh / Hv, hv = bh - b * Hv, hk = key_head(hv, Hk, Hv, opts), t0 = n * kTile;
    if (io == 0) mbar_expect_tx(bar_tma, 6 * 8192);
    if (io < 2) tma_load_4d(sbase + kOffKQ + io * 16384, P.tm_k, bar_tma, 64 * io, hk, t0, b);
    else tma_load_4d(sbase + kOffV + (io - 2) * 8192, P.tm_v, bar_tma, 64 * (io - 2), hv, t0, b);
  };
  // ... and its Q (io 0 and 1).
  auto load_q = [&](int lin) {
    const int bh = head_of(lin), n = tile_of(lin);
    const int b = bh / Hv, hv = bh - b * Hv, hk = key_head(hv, Hk, Hv, opts), t0 = n * kTile;
    if (io < 2) tma_load_4d(sbase + kOffKQ + io * 16384 + 8192, P.tm_q, bar_tma, 64 * io, hk, t0, b);
  };
  // Gate and beta of token `tid` of a tile, read one tile ahead into registers
  // as raw bf16 bits (converted when used, so the load is not waited for here).
  // Padded tokens: decay 1 (gate 1.0, or log-gate 0.0), beta 0.
  const uint16_t g_pad = (opts & kOptLogGate) ? 0x0000 : 0x3f80;
  uint16_t g_next = g_pad, b_next = 0;
  auto load_gates = [&](int lin) {
    g_next = g_pad;
    b_next = 0;
    if (tid < 64 && lin < total) {
      const int bh = head_of(lin), n = tile_of(lin);
      const int b = bh / Hv, hv = bh - b * Hv, tok = n * kTile + tid;
      if (tok < T) {
        const size_t gi = ((size_t)b * T + tok) * Hv + hv;
        b_next = reinterpret_cast<const uint16_t*>(beta)[gi];
        g_next = reinterpret_cast<const uint16_t*>(g)[gi];
      }
    }
  };
  auto bits_to_f32 = [](uint16_t x) { return __uint_as_float((uint32_t)x << 16); };
  if (gid < total && io >= 0) {
    prefetch_tmap(io < 2 ? P.tm_k : P.tm_v);
    if (io < 2) prefetch_tmap(P.tm_q);
    load_kv(gid);
    load_q(gid);
  }
  load_gates(gid);

  bool ok = true;
  bool tma_pending = gid < total;  // a load phase was issued and not yet waited for
  // Publishing: each I/O thread adds 1 to a tile's flag once all of its stores
  // of the tile are in memory, so the flag reaches kPrepIo when the whole tile
  // is.  It does so after the next tile's loads have landed (they were issued
  // after these stores), when the wait for the stores is normally over.
  size_t unpublished = ~(size_t)0;
  auto publish = [&]() {
    if (unpublished != ~(size_t)0) {
      bulk_wait_all();
      fence_proxy_async_global();
      red_release_gpu_add(flags + unpublished, 1);
      unpublished = ~(size_t)0;
    }
  };
  int it = 0;
  for (int lin = gid; lin < total && ok; lin += ngroups, ++it) {
  const size_t tile_id = (size_t)head_of(lin) * NT + tile_of(lin);
  const int next = lin + ngroups;
  const float gv_cur = bits_to_f32(g_next), bt_cur = bits_to_f32(b_next);
  load_gates(next);
  // Warm L2 with the next tile's K, Q and V rows: warps 2-7 (u = tid - 64), one
  // 256-byte token row of one tensor per thread, as plain prefetches that leave
  // the TMA unit free.  Issued while those warps wait for the inverse's first
  // stage, which only warps 0-1 work on.
  auto prefetch_next = [&]() {
    const int u = tid - 64;
    if (next >= total || u < 0 || u >= 3 * kTile) return;
    const int nbh = head_of(next), nb = nbh / Hv, nhv = nbh - nb * Hv;
    const int nhk = key_head(nhv, Hk, Hv, opts), tok = tile_of(next) * kTile + (u & (kTile - 1));
    if (tok < T) {
      const int which = u / kTile;  // 0: K, 1: Q, 2: V
      const bf16* base = which == 0 ? P.k : (which == 1 ? P.q : P.v);
      const int heads = which == 2 ? Hv : Hk, hh = which == 2 ? nhv : nhk;
      const char* row = reinterpret_cast<const char*>(base + (((size_t)nb * T + tok) * heads + hh) * kD);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(row) : "memory");
      asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 128) : "memory");
    }
  };

  // Gates (step 2).  Padded tokens take g = 1, beta = 0.  Decay products are
  // carried as chunk-local prefix sums lam of log2 g: G_t = 2^lam_t and
  // Gam[t][j] = 2^(lam_t - lam_j) (j <= t) -- never a quotient, so a vanishing
  // product underflows to 0.  Gam is used factored per 16-token block b:
  // across 16-token blocks, Gam[t][j] = rfac[t][b(j)] * sfac[j] with the
  // block end as the split point, so both factors are products of decays (<= 1);
  // inside a block it is 2^(lam_t - lam_j) directly.  Warps 0-1 form the
  // prefix sums (one token per thread); warps 0-3 then derive the tables (two
  // threads per token).
  if (tid < 64) {
    const int t = tid, lane = tid & 31;
    bta[t] = bt_cur;  // padded tokens: g = 1, beta = 0
    // log2 of the decay (clamped: a vanishing decay underflows the products to 0)
    float l = fmaxf((opts & kOptLogGate) ? gv_cur * 1.4426950408889634f : lg2(gv_cur), -1000.f);
    constexpr int kSeg = C < 32 ? C : 32;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, l, off);
      if ((lane % kSeg) >= off) l += y;
    }
    if constexpr (C == 64) {
      if (tid == 31) carry_sh[grp] = l;
      named_bar_sync(carry_id, 64);
      if (tid >= 32) l += carry_sh[grp];
    }
    lam[t] = l;
  }
  if (tid < 128) {
    named_bar_sync(gates_id, 128);
    const int t = tid >> 1, p = tid & 1;
    const float l = lam[t];
    const int tb = t & ~15, tt = t & 15;
    float* gd = gdiag + t * kLdGd + 8 * p;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = 8 * p + e;  // in-block ratios (entries past t are never read)
      gd[e] = j <= tt ? ex2(l - lam[tb + j]) : 0.f;
    }
    const int ce = (t / C) * C + C - 1, cs = (t / C) * C;
    const float lend = lam[ce];
    if (p == 0) {
      gsuf[t] = ex2(lend - l);
      gpw[t] = ex2(l);
      sfac[t] = ex2(lam[(t | 15)] - l);
    } else {
#pragma unroll
      for (int bb = 0; bb < 4; ++bb)
        rfac[t * 4 + bb] = (bb * 16 >= cs && bb < (t >> 4)) ? ex2(l - lam[bb * 16 + 15]) : 0.f;
      if (t == ce) gc[t / C] = ex2(lend);
    }
  }

  ok = mbar_wait(bar_tma, it & 1);
  tma_pending = false;
  if (ok && io >= 0) publish();
  if (opts & kOptL2NormQK) {  // rows 0-63 of each half are K, 64-127 Q
    if (ok) l2norm_row_sw128(sm + kOffKQ, 16384, tid >> 1, tid & 1);
    fence_proxy_async();
    gsync();
  }
  // G1: D[128 x 64] = [K; Q] K^T  (TMEM columns 0..63), issued outside the gate
  // warps (lane 1 of warp 4).  The previous tile's last stores must have read A3 and X, which
  // this tile rewrites after G1.
  if (io >= 0) bulk_wait_read_all();
  if (ok && tid == 129) {
    tc_fence_after();
    const uint32_t id1 = idesc_bf16(128, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t a = sbase + kOffKQ + (kk >> 2) * 16384 + (kk & 3) * 32;
      mma_bf16_ss(tmem, smem_desc(a, 16, 1024, kSw128), smem_desc(a, 16, 1024, kSw128), id1,
                  kk > 0);
    }
    mma_commit(bar_mma);
  }
  ok = gsync_and(ok);  // also publishes the gate scalars
  ok = ok && mbar_wait(bar_mma, it & 1);  // G1 completes once per tile
  tc_fence_after();
  if (ok) {
    // Row t of KK^T (TMEM lanes 0..63) -> row t of X = L (step 4):
    //   X[t][j] = beta_j KK^T[t][j], j < t in t's chunk.
    // Row t of QK^T (lanes 64..127) -> rows t and 64+t of
    //   A3 = [diag(G) M; Gam . QK^T], M[t][i] = beta_i QK^T[t][i], i <= t (steps 6, 7).
    // Warps w and w+4 share TMEM lane quadrant w % 4 and take 32 columns each.
    const int q4 = warp & 3, lrow = q4 * 32 + (tid & 31);
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int t = lrow & 63;
    const int cs = (t / C) * C, bt = t >> 4;
    const float gt = gpw[t];
    const int cbeg = (warp >> 2) * 32;
    float vv[2][16];  // both 16-column blocks, one TMEM round trip
    tmem_ld16(tmem + lane_base + cbeg, vv[0]);
    tmem_ld16(tmem + lane_base + cbeg + 16, vv[1]);
    tmem_wait_ld();
#pragma unroll
    for (int c0 = cbeg; c0 < cbeg + 32; c0 += 16) {
      const float* v = vv[(c0 - cbeg) >> 4];
      // A 16-column block lies wholly inside or outside t's chunk (16 | C); it
      // is before, on or after t's own 16-block.
      const int cb = c0 >> 4, tt = t & 15;
      const bool live = c0 >= cs && cb <= bt, diag = cb == bt;
      float b16[16];
      ld16f(bta + c0, b16);
      if (lrow < 64) {
        float o[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = (live && (!diag || e < tt)) ? b16[e] * v[e] : 0.f;
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(X + t * kLdX + c0 + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
      } else {
        float top[16], bot[16], gam[16];
        if (diag) {
          ld16f(gdiag + t * kLdGd, gam);
        } else {
          ld16f(sfac + c0, gam);
          const float rb = rfac[t * 4 + cb];
#pragma unroll
          for (int e = 0; e < 16; ++e) gam[e] *= rb;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const bool keep = live && (!diag || e <= tt);
          top[e] = keep ? gt * b16[e] * v[e] : 0.f;
          bot[e] = keep ? gam[e] * v[e] : 0.f;
        }
        st_sm16(sm, kOffA3 + sw128(t, c0), pack8(top));
        st_sm16(sm, kOffA3 + sw128(t, c0 + 8), pack8(top + 8));
        st_sm16(sm, kOffA3 + sw128(64 + t, c0), pack8(bot));
        st_sm16(sm, kOffA3 + sw128(64 + t, c0 + 8), pack8(bot + 8));
      }
    }
  }
  // Step 4: T_L = (I + L)^-1.  Step 5 needs no second inverse:
  // (I + A)^-1 diag(beta) = diag(beta) (Gam . T_L) for A[t][j] = beta_t Gam[t][j] KK^T[t][j].
  // The inverse's first stage (warps 0-1) needs only X, written by warps 0, 1, 4
  // and 5; the A3 builders (warps 2, 3, 6, 7) finish meanwhile and meet the
  // group at the inverse's first barrier.  The inverse runs (on whatever X
  // holds) even after a failed wait, so every thread passes the same barriers;
  // ok is made uniform after it.
  if (pstream) named_bar_sync(pstream_id, 128);
  prefetch_next();
  invert_unit_lower<C>(X, TL, Zs, tid, gsync);

  // A2 = [T_L; diag(beta) (Gam . T_L)]: 128 rows x 64 K-cols, K-major 128B swizzle.
  // Thread: 8 columns (col0..col0+7) of T_L rows r0 and r0+32, written as rows
  // t and 64+t of A2.
  if (ok) {
    const int col0 = (tid & 7) * 8, r0 = tid >> 3, bj = col0 >> 4;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = r0 + 32 * i;
      const float4 a = *reinterpret_cast<const float4*>(TL + t * kLdX + col0);
      const float4 c4 = *reinterpret_cast<const float4*>(TL + t * kLdX + col0 + 4);
      float v[8] = {a.x, a.y, a.z, a.w, c4.x, c4.y, c4.z, c4.w};
      st_sm16(sm, kOffB + sw128(t, col0), pack8(v));
      // T_L is zero above the diagonal and across chunks (rfac is 0 there too).
      float f[8];
      const float bt = bta[t];
      if (bj < (t >> 4)) {
        const float rb = bt * rfac[t * 4 + bj];
        const float4 s0 = *reinterpret_cast<const float4*>(sfac + col0);
        const float4 s1 = *reinterpret_cast<const float4*>(sfac + col0 + 4);
        f[0] = s0.x * rb; f[1] = s0.y * rb; f[2] = s0.z * rb; f[3] = s0.w * rb;
        f[4] = s1.x * rb; f[5] = s1.y * rb; f[6] = s1.z * rb; f[7] = s1.w * rb;
      } else {
        const float* gd = gdiag + t * kLdGd + (col0 & 15);
        const float4 s0 = *reinterpret_cast<const float4*>(gd);
        const float4 s1 = *reinterpret_cast<const float4*>(gd + 4);
        f[0] = s0.x * bt; f[1] = s0.y * bt; f[2] = s0.z * bt; f[3] = s0.w * bt;
        f[4] = s1.x * bt; f[5] = s1.y * bt; f[6] = s1.z * bt; f[7] = s1.w * bt;
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = (col0 + e <= t) ? f[e] : 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] *= f[e];
      st_sm16(sm, kOffB + sw128(64 + t, col0), pack8(v));
    }
    fence_proxy_async();
  }
  ok = gsync_and(ok);

  // From G2 on the tile runs as two streams that meet again before the last
  // stores: the P stream (warps 0, 1, 4, 5: TMEM lanes 0..63; P, Pt, G M P, Qh;
  // io 0 and 1) and the U stream (warps 2, 3, 6, 7: lanes 64..127; U, Ut,
  // y_loc; io 2 and 3), each with its own barrier and MMA completion barrier.
  // G2 (thread 0): D2b = A2 V (cols 128..255; rows 64..127 = U = T_A (beta V))
  // first, committed to bar_u, then D2a = A2 K (cols 0..127; rows 0..63 =
  // P = T_L K), committed to bar_p.
  if (ok && tid == 0) {
    tc_fence_after();
    const uint32_t id2 = idesc_bf16(128, 128, false, true);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ad = smem_desc(sbase + kOffB + kk * 32, 16, 1024, kSw128);
      mma_bf16_ss(tmem + 128, ad, smem_desc(sbase + kOffV + kk * 2048, 8192, 1024, kSw128), id2,
                  kk > 0);
    }
    mma_commit(bar_u);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ad = smem_desc(sbase + kOffB + kk * 32, 16, 1024, kSw128);
      mma_bf16_ss(tmem, ad, smem_desc(sbase + kOffKQ + kk * 2048, 16384, 1024, kSw128), id2,
                  kk > 0);
    }
    mma_commit(bar_p);
  }
  const uint32_t bar_s = pstream ? bar_p : bar_u;
  const int stream_id = pstream ? pstream_id : ustream_id;
  ok = ok && mbar_wait(bar_s, 0);
  tc_fence_after();

  // Epilogue thread: row t of its stream (TMEM lane (warp % 4) * 32 + lane),
  // columns cbeg .. cbeg+63 (warps w and w+4 share a lane quadrant).
  auto epi_t = [&]() { return ((warp & 3) * 32 + (tid & 31)) & 63; };
  auto epi_src = [&]() {
    return tmem + ((uint32_t)((warp & 3) * 32) << 16) + (pstream ? 0 : 128);
  };
  if (ok) {
    const int t = epi_t(), cbeg = (warp >> 2) * 64;
    const uint32_t src = epi_src();
    // P rows (lanes 0..63) and U rows (lanes 64..127): bf16 into the G3 operand
    // B3 = [P; U] and, scaled, into the workspace: Pt = G_C beta P (step 9),
    // Ut = Gam[C-1][.] U.  Staging: Pt over K, Ut over V (each stream's G2 has
    // read them), as 128B-swizzled 64-column halves stored below with TMA.
    const uint32_t bdst = kOffB + (pstream ? 0 : 16384);
    const float scale = pstream ? gc[t / C] * bta[t] : gsuf[t];
    const uint32_t stage = pstream ? kOffKQ : kOffV;
    const uint32_t half_stride = pstream ? 16384 : 8192;
#pragma unroll
    for (int c2 = cbeg; c2 < cbeg + 64; c2 += 32) {
      float vv[2][16];  // two 16-column blocks per TMEM round trip
      tmem_ld16(src + c2, vv[0]);
      tmem_ld16(src + c2 + 16, vv[1]);
      tmem_wait_ld();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int col = c2 + 16 * hh;
        float* v = vv[hh];
        const uint32_t atom = bdst + (col >> 6) * 8192;
        st_sm16(sm, atom + sw128(t, col & 63), pack8(v));
        st_sm16(sm, atom + sw128(t, (col & 63) + 8), pack8(v + 8));
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] *= scale;
        const uint32_t hs = stage + (col >> 6) * half_stride;
        st_sm16(sm, hs + sw128(t, col & 63), pack8(v));
        st_sm16(sm, hs + sw128(t, (col & 63) + 8), pack8(v + 8));
      }
    }
    fence_proxy_async();
  }
  tc_fence_before();  // this stream's TMEM reads precede its G3
  named_bar_sync(stream_id, 128);
  if (ok && io >= 0) {
    const int row0 = (int)(tile_id * 128);
    if (io < 2) {
#pragma unroll
      for (int c = 0; c < 64 / C; ++c)  // Pt rows of chunk c, half io
        tma_store_2d(P.tm_a1s, sbase + kOffKQ + io * 16384 + c * C * 128, 64 * io,
                     row0 + 2 * C * c);
    } else {
      tma_store_2d(P.tm_us, sbase + kOffV + (io - 2) * 8192, 64 * (io - 2),
                   (int)(tile_id * kTile));  // Ut rows
    }
    bulk_commit();
  }
  // G3 per stream: D3a = A3 P (thread 0; cols 0..127, rows 0..63 = G M P) and
  // D3b = A3 U (thread 64; cols 128..255, rows 64..127 = y_loc).
  if (ok && (tid == 0 || tid == 64)) {
    tc_fence_after();
    const uint32_t id3 = idesc_bf16(128, 128, false, true);
    const uint32_t boff = pstream ? 0 : 16384;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ad = smem_desc(sbase + kOffA3 + kk * 32, 16, 1024, kSw128);
      mma_bf16_ss(tmem + (pstream ? 0 : 128), ad,
                  smem_desc(sbase + kOffB + boff + kk * 2048, 8192, 1024, kSw128), id3, kk > 0);
    }
    mma_commit(bar_s);
  }
  ok = ok && mbar_wait(bar_s, 1);
  tc_fence_after();

  if (ok) {
    // Staging over this stream's half of B3 (read only by its own G3): Qh by
    // the P stream, y_loc / sqrt(Dk) by the U stream.
    const int t = epi_t(), cbeg = (warp >> 2) * 64;
    const uint32_t src = epi_src();
    const uint32_t stage = kOffB + (pstream ? 0 : 16384);
    const float gt = gpw[t];
#pragma unroll
    for (int c2 = cbeg; c2 < cbeg + 64; c2 += 32) {
      float vv[2][16];  // two 16-column blocks per TMEM round trip
      tmem_ld16(src + c2, vv[0]);
      tmem_ld16(src + c2 + 16, vv[1]);
      tmem_wait_ld();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int col = c2 + 16 * hh;
        float* v = vv[hh];
        if (pstream) {  // Qh = G q - G M P  (step 7, state-free part)
          const uint8_t* qa = sm + kOffKQ + (col >> 6) * 16384 + 8192;
          float q[16];
          unpack8(*reinterpret_cast<const uint4*>(qa + sw128(t, col & 63)), q);
          unpack8(*reinterpret_cast<const uint4*>(qa + sw128(t, (col & 63) + 8)), q + 8);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = gt * q[j] - v[j];
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] *= P.yscale;
        }
        const uint32_t hs = stage + (col >> 6) * 8192;
        st_sm16(sm, hs + sw128(t, col & 63), pack8(v));
        st_sm16(sm, hs + sw128(t, (col & 63) + 8), pack8(v + 8));
      }
    }
  }
  if (ok && tid < 64 / C) wsGC[tile_id * 4 + tid] = gc[tid];
  if (ok) fence_proxy_async();
  ok = gsync_and(ok);
  if (ok && io >= 0) {
    const int row0 = (int)(tile_id * 128);
    if (io < 2) {
#pragma unroll
      for (int c = 0; c < 64 / C; ++c)  // Qh rows of chunk c, half io
        tma_store_2d(P.tm_a1s, sbase + kOffB + io * 8192 + c * C * 128, 64 * io,
                     row0 + 2 * C * c + C);
    } else {  // y_loc / sqrt(Dk) into y (rows past T are clipped)
      const int h = io - 2, bh = head_of(lin), b = bh / Hv;
      tma_store_4d(P.tm_y, sbase + kOffB + 16384 + h * 8192, 64 * h, bh - b * Hv,
                   tile_of(lin) * kTile, b);
    }
    bulk_commit();
  }
  if (io >= 0) {
    // The next tile's K, Q and V are loaded once this thread's stores of Pt
    // or Ut (staged in K and V) have read them; Q was last read by the
    // epilogue above.  The Qh / y_loc staging is waited for before the next G1.
    bulk_wait_read<1>();
    if (ok && next < total) {
      load_kv(next);
      load_q(next);
      tma_pending = true;
    }
    if (ok && flags) unpublished = tile_id;
  }
  // No group barrier here: ok is uniform since the last one, and the next
  // tile's gate tables are free (their last reader was the epilogue above), so
  // the gate warps start on the next tile while the I/O threads issue its loads.
  }  // tile loop

  if (io >= 0) {
    if (ok) publish();
    bulk_wait_read_all();  // shared memory must outlive the last stores' reads
  }
  // A group that stopped early lets its last prefetch land before the CTA exits.
  if (io == 0 && tma_pending) mbar_wait(bar_tma, it & 1);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tmem_base_sh, 256 * kPrepGroups);
}

template <int C>
__global__ void __launch_bounds__(kPrepThreads, 1)
prep_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a1s,
               const __grid_constant__ CUtensorMap tm_us, const __grid_constant__ CUtensorMap tm_y,
               const bf16* kin, const bf16* qin, const bf16* vin, const bf16* __restrict__ g,
               const bf16* __restrict__ beta, float* __restrict__ wsGC, int T, int Hk, int Hv,
               int NT, int BH, int opts, float scale) {
  extern __shared__ uint8_t smem_raw[];
  const PrepParams P{kin, qin, vin, &tm_k, &tm_q, &tm_v, &tm_a1s, &tm_us, g, beta, wsGC,
                     T, Hk, Hv, NT, BH, opts, &tm_y, scale};
  prep_role<C>(P, smem_raw, blockIdx.x, gridDim.x, nullptr);
}

// ============================================================================
// fused prefill: prep and scan in one cooperative launch
// ============================================================================
// One CTA per SM.  CTAs 0 .. BH-1 each run the scan of one (b, hv) head over
// all 128 value rows; the others run prep_role in both of their groups and
// publish every finished tile through a flag in the workspace.  A scan CTA
// waits for a tile's flag before loading it, so the scan of chunk n overlaps
// the prep of later chunks.  Prep never waits for the scan and the launch is
// cooperative (every CTA resident), so each wait ends.
//
// The scan role is the chunk update of scan_tc_kernel at R = 128:
//   D = K^T Ut;  D += (-M^T) S^T;  Y = Qh S^T;  S <- G_C S + D^T,
// with M^T = K^T Pt of chunk j+1 and D = K^T Ut of chunk j issued while the
// state group finishes chunk j-1.  One S operand buffer: the state group
// overwrites it only after Y of the chunk has completed.
constexpr int kFusedThreads = kPrepThreads;  // 16 warps

// Two rings of tile buffers: the MN ring (Pt, K, Ut: read by K^T [Pt | Ut],
// released as soon as those products finish; two stages) and the Q ring (Qh,
// later the staging of y; released after the y reduction has read it; three
// stages, since it is held longer).
struct Scan128Smem {
  static constexpr uint32_t kOffP = 0;              // Pt, 2 x 64 rows x 128 B
  static constexpr uint32_t kOffK = 16384;          // K,  2 x 64 rows x 128 B
  static constexpr uint32_t kOffU = 32768;          // Ut, 2 x 64 rows x 128 B
  static constexpr uint32_t kMN = 49152;
  static constexpr uint32_t kQ = 16384;             // Qh, 2 x 64 rows x 128 B
  static constexpr int kStagesMN = 2;
  static constexpr int kStagesQ = 3;
  static constexpr uint32_t kOffQ = kStagesMN * kMN;
  static constexpr uint32_t kOffS = kOffQ + kStagesQ * kQ;   // S operand: 2 x 128 k-rows x 128 B

  static constexpr uint32_t kOffGC = kOffS + 32768;          // G_C per Q stage (fp32 x 4)
  static constexpr uint32_t kTotal = kOffGC + kStagesQ * 16 + 1024;
};
constexpr uint32_t kFusedSmem = Scan128Smem::kTotal > kPrepSmem ? Scan128Smem::kTotal : kPrepSmem;

enum : int {
  kQFullMN = 0,
  kQEmptyMN = kQFullMN + Scan128Smem::kStagesMN,  // MMA commit
  kQFullQ = kQEmptyMN + Scan128Smem::kStagesMN,
  kQEmptyQ = kQFullQ + Scan128Smem::kStagesQ,     // 257: state group + the y-reducing thread
  kQKNorm = kQEmptyQ + Scan128Smem::kStagesQ,     // 128: K rows of the MN stage normalised
  kQDs = kQKNorm + Scan128Smem::kStagesMN,
  kQY,
  kQM,                 // [2]
  kQSop = kQM + 2,     // 256
  kQDsFree,            // 256
  kQMt,                // [2] 128
  kQYFree = kQMt + 2,  // 128
  kQYStaged,           // 128: Y of the chunk staged for the reduction
  kQDN,                // D = K^T Ut of the chunk issued and complete
  kQFin,               // 2: both issuers' last products complete
  kNumQBars
};

template <int C>
__device__ __forceinline__ void scan_role128(const CUtensorMap* tm_a1c, const CUtensorMap* tm_k,
                                             const CUtensorMap* tm_uy, const CUtensorMap* tm_yred,
                                             const float* wsGC, const int* flags,
                                             const float* state_in, float* state_out, int T,
                                             int Hk, int Hv, int NT, int bh, int opts,
                                             float scale, uint8_t* smem_raw) {
  using SM = Scan128Smem;
  constexpr int kCt = kTile / C;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~(uintptr_t)1023);
  __shared__ uint64_t qbars[kNumQBars];
  __shared__ uint32_t qtmem_sh;
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = bh / Hv, hv = bh - b * Hv, hk = key_head(hv, Hk, Hv, opts);
  const int NC = (T + C - 1) / C;
  auto bar = [&](int i) { return smem_u32(&qbars[i]); };

  if (tid == 0) {
    for (int s = 0; s < SM::kStagesMN; ++s) {
      mbar_init(bar(kQFullMN + s), 1);
      mbar_init(bar(kQEmptyMN + s), 1);
      mbar_init(bar(kQKNorm + s), 128);
    }
    for (int s = 0; s < SM::kStagesQ; ++s) {
      mbar_init(bar(kQFullQ + s), 1);
      mbar_init(bar(kQEmptyQ + s), 257);
    }
    mbar_init(bar(kQDs), 1);
    mbar_init(bar(kQY), 1);
    mbar_init(bar(kQM), 1);
    mbar_init(bar(kQM + 1), 1);
    mbar_init(bar(kQSop), 256);
    mbar_init(bar(kQDsFree), 256);
    mbar_init(bar(kQMt), 128);
    mbar_init(bar(kQMt + 1), 128);
    mbar_init(bar(kQYFree), 128);
    mbar_init(bar(kQYStaged), 128);
    mbar_init(bar(kQDN), 1);
    mbar_init(bar(kQFin), 2);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&qtmem_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = qtmem_sh;
  const uint32_t tD = tmem, tY = tmem + 384;
  auto tM = [&](int x) { return tmem + 128 + 128 * x; };  // fp32 M^T; cols 0-63 then -M^T bf16
  const uint32_t sS = sbase + SM::kOffS;
  auto ring_mn = [&](int j) { return (j / kCt) % SM::kStagesMN; };
  auto ring_q = [&](int j) { return (j / kCt) % SM::kStagesQ; };
  auto mn_addr = [&](int j) { return sbase + ring_mn(j) * SM::kMN; };
  auto q_addr = [&](int j) { return sbase + SM::kOffQ + ring_q(j) * SM::kQ; };
  auto last_of_tile = [&](int j) { return (j % kCt) == kCt - 1 || j == NC - 1; };
  auto wait_mn = [&](int j) {
    const int n = j / kCt;
    return mbar_wait(bar(kQFullMN + n % SM::kStagesMN), (n / SM::kStagesMN) & 1);
  };
  // With L2-normalised keys the aux group rewrites each K tile first.
  const bool knorm = (opts & kOptL2NormQK) != 0;
  auto wait_knorm = [&](int j) {
    const int n = j / kCt;
    return mbar_wait(bar(kQKNorm + n % SM::kStagesMN), (n / SM::kStagesMN) & 1);
  };
  auto wait_q = [&](int j) {
    const int n = j / kCt;
    return mbar_wait(bar(kQFullQ + n % SM::kStagesQ), (n / SM::kStagesQ) & 1);
  };

  if ((warp == 0 || warp == 14) && lane == 0) {
    // ---------------------- producers (MN ring, Q ring) ----------------------
    const bool mn = warp == 0;
    const int full0 = mn ? kQFullMN : kQFullQ, empty0 = mn ? kQEmptyMN : kQEmptyQ;
    prefetch_tmap(tm_a1c);
    if (mn) {
      prefetch_tmap(tm_k);
      prefetch_tmap(tm_uy);
    }
    const int stages = mn ? SM::kStagesMN : SM::kStagesQ;
    int n = 0;
    for (; n < NT; ++n) {
      const int s = n % stages;
      if (n >= stages && !mbar_wait(bar(empty0 + s), ((n / stages) - 1) & 1)) break;
      const size_t tid_ws = (size_t)bh * NT + n;
      if (flags) {
        if (!wait_flag(flags + tid_ws, kPrepIo)) break;
        fence_proxy_async_global();
      }
      const uint32_t fb = bar(full0 + s);
      const int row = (int)(tid_ws * 128);
      if (mn) {
        const uint32_t st = sbase + s * SM::kMN;
        mbar_expect_tx(fb, SM::kMN);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = 0; c < kCt; ++c)  // Pt rows of chunk c
            tma_load_2d(st + SM::kOffP + h * 8192 + c * C * 128, tm_a1c, fb, 64 * h,
                        row + 2 * C * c);
          tma_load_4d(st + SM::kOffK + h * 8192, tm_k, fb, 64 * h, hk, n * kTile, b);
          tma_load_2d(st + SM::kOffU + h * 8192, tm_uy, fb, 64 * h, (int)(tid_ws * kTile));
        }
      } else {
        const uint32_t st = sbase + SM::kOffQ + s * SM::kQ;
        mbar_expect_tx(fb, SM::kQ + 16);
        bulk_load(sbase + SM::kOffGC + 16 * s, wsGC + tid_ws * 4, 16, fb);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = 0; c < kCt; ++c)  // Qh rows of chunk c
            tma_load_2d(st + h * 8192 + c * C * 128, tm_a1c, fb, 64 * h, row + 2 * C * c + C);
        }
      }
    }
    for (int m = (n > stages ? n - stages : 0); m < n; ++m)
      mbar_wait(bar(full0 + m % stages), (m / stages) & 1);
  } else if (warp == 1 || warp == 15) {
    // ---------------------------- MMA issuers ----------------------------
    // Two threads issue the products, so that the serial one is not queued
    // behind the others: warp 1 issues D += (-M^T) S^T only; warp 15 issues
    // Y^T = S Qh^T (which needs only the chunk-start state), M^T of the next
    // chunk and D = K^T Ut of the next chunk.  They are ordered through
    // mbarriers: D_S(j) waits for D_N(j) (same accumulator); D_N(j+1) waits
    // until the state group has read D(j); M^T(j+1) overwrites the TMEM operand
    // of D_S(j-1), complete once the S operand of chunk j is written.
    if (lane == 0) {
      const uint32_t id_kt = idesc_bf16(128, 128, true, true);   // K^T x (Pt | Ut)
      const uint32_t id_s = idesc_bf16(128, 128, false, true);   // (-M^T) x S^T
      const uint32_t id_y = idesc_bf16(128, C, true, false);     // S x Qh^T (rows v, cols t)
      // Descriptor bases (per ring stage via a byte offset; see SmemDesc).
      const SmemDesc d_mn_mn = smem_desc_base(sbase, 8192, 1024, kSw128);   // MN-major, 64-row halves
      const SmemDesc d_s = smem_desc_base(sS, 16384, 1024, kSw128);         // S operand
      const SmemDesc d_q = smem_desc_base(sbase + SM::kOffQ, 16, 1024, kSw128);  // Qh, K-major
      bool ok = true;
      if (warp == 1) {
        for (int j = 0; j < NC && ok; ++j) {
          // D += (-M^T) S^T   (the serial step), on D = K^T Ut of the chunk
          if (!(ok = mbar_wait(bar(kQDN), j & 1))) break;
          if (!(ok = mbar_wait(bar(kQSop), j & 1))) break;
          if (!(ok = mbar_wait(bar(kQMt + (j & 1)), (j >> 1) & 1))) break;
          tc_fence_after();
          const uint32_t ta = tM(j & 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(tD, ta + 8 * kk, smem_desc_at(d_s, kk * 2048), id_s, 1);
          mma_commit(bar(kQDs));
        }
      } else {
        // M^T of chunk j into tM(j & 1), once its tile's MN buffers have landed.
        auto issue_mt = [&](int j) {
          if (j % kCt == 0) {
            if (!(knorm ? wait_knorm(j) : wait_mn(j))) return false;
            tc_fence_after();
          }
          const uint32_t off = ring_mn(j) * SM::kMN + (j % kCt) * C * 128;
#pragma unroll
          for (int kk = 0; kk < C / 16; ++kk)
            mma_bf16_ss(tM(j & 1), smem_desc_at(d_mn_mn, off + SM::kOffK + kk * 2048),
                        smem_desc_at(d_mn_mn, off + SM::kOffP + kk * 2048), id_kt, kk > 0);
          mma_commit(bar(kQM + (j & 1)));
          return true;
        };
        // D = K^T Ut of chunk j into tD (after M^T(j): its MN buffers have landed).
        auto issue_dn = [&](int j) {
          tc_fence_after();
          const uint32_t off = ring_mn(j) * SM::kMN + (j % kCt) * C * 128;
#pragma unroll
          for (int kk = 0; kk < C / 16; ++kk)
            mma_bf16_ss(tD, smem_desc_at(d_mn_mn, off + SM::kOffK + kk * 2048),
                        smem_desc_at(d_mn_mn, off + SM::kOffU + kk * 2048), id_kt, kk > 0);
          mma_commit(bar(kQDN));
          // The tile's MN buffers are free once its last products finish.
          if (last_of_tile(j)) mma_commit(bar(kQEmptyMN + ring_mn(j)));
        };
        if (NC > 0) {
          ok = issue_mt(0);
          if (ok) issue_dn(0);
        }
        for (int j = 0; j < NC && ok; ++j) {
          const int c = j % kCt;
          // Y^T = S Qh^T (A = the S operand read MN-major, B = Qh rows): the state
          // group rewrites S once it completes.
          if (!(ok = mbar_wait(bar(kQSop), j & 1))) break;
          if (c == 0 && !(ok = wait_q(j))) break;
          if (j > 0 && !(ok = mbar_wait(bar(kQYFree), (j - 1) & 1))) break;
          tc_fence_after();
          const uint32_t qoff = ring_q(j) * SM::kQ + c * C * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tY, smem_desc_at(d_s, kk * 2048),
                        smem_desc_at(d_q, qoff + (kk >> 2) * 8192 + (kk & 3) * 32), id_y, kk > 0);
          mma_commit(bar(kQY));
          if (j + 1 < NC) {
            // M^T of chunk j+1, converted by the aux group while chunk j finishes.
            if (!(ok = issue_mt(j + 1))) break;
            // D = K^T Ut of chunk j+1 once chunk j's D has been read.
            if (!(ok = mbar_wait(bar(kQDsFree), j & 1))) break;
            issue_dn(j + 1);
          }
        }
      }
      mma_commit(bar(kQFin));
      mbar_wait(bar(kQFin), 0);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 10) {
    // ----------------------------- state group ----------------------------
    // Thread = TMEM lane k (key column); value rows 64h .. 64h+63.
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int L = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const size_t sidx = ((size_t)bh * kD + 64 * h) * kD + L;
    bool ok = true;
    float s[64];
#pragma unroll
    for (int r = 0; r < 64; ++r) s[r] = state_in ? state_in[sidx + (size_t)r * kD] : 0.f;
    auto write_op = [&]() {
      uint8_t* row = sm + SM::kOffS + h * 16384;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) st_sm16(row, sw128(L, 8 * ch), pack8(s + 8 * ch));
      fence_proxy_async();
      mbar_arrive(bar(kQSop));
    };
    write_op();
    for (int j = 0; j < NC; ++j) {
      const int c = j % kCt;
      if (c == 0 && !(ok = wait_q(j))) break;
      const float Gc = ld_shared_f32(sbase + SM::kOffGC + 16 * ring_q(j) + 4 * c);
      if (last_of_tile(j)) mbar_arrive(bar(kQEmptyQ + ring_q(j)));
      if (!(ok = mbar_wait(bar(kQDs), j & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float d[32];
        tmem_ld32(tD + lane_base + 64 * h + 32 * half, d);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < 32; ++r) s[32 * half + r] = fmaf(Gc, s[32 * half + r], d[r]);
      }
      tc_fence_before();
      mbar_arrive(bar(kQDsFree));
      if (j + 1 < NC) {
        // Y of chunk j still reads the S operand.
        if (!(ok = mbar_wait(bar(kQY), j & 1))) break;
        write_op();
      }
    }
    if (ok) {
#pragma unroll
      for (int r = 0; r < 64; ++r) state_out[sidx + (size_t)r * kD] = s[r];
    }
  } else if (warp >= 10 && warp < 14) {
    // ------------------------------ aux group -----------------------------
    const int qd = warp & 3;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    bool ok = true;
    auto convert = [&](int j) {
      if (!mbar_wait(bar(kQM + (j & 1)), (j >> 1) & 1)) return false;
      tc_fence_after();
      const uint32_t tb = tM(j & 1) + lane_base;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v[64];
        tmem_ld32(tb + 64 * hh, v);
        tmem_ld32(tb + 64 * hh + 32, v + 32);
        tmem_wait_ld();
        uint32_t p[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) p[i] = pack_bf16x2(-v[2 * i], -v[2 * i + 1]);
        tmem_st32(tb + 32 * hh, p);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kQMt + (j & 1)));
      return true;
    };
    // Normalise the K rows of the tile holding chunk j (64 rows, two threads
    // per row), then release it to the issuer.
    const int atid = tid - 320;  // 0..127 in the aux group
    auto normalise_k = [&](int j) {
      if (!wait_mn(j)) return false;
      l2norm_row_sw128(sm + (mn_addr(j) - sbase) + SM::kOffK, 8192, atid >> 1, atid & 1);
      fence_proxy_async();
      mbar_arrive(bar(kQKNorm + ring_mn(j)));
      return true;
    };
    if (knorm && NC > 0) ok = normalise_k(0);
    if (ok && NC > 0) ok = convert(0);
    for (int j = 0; j < NC && ok; ++j) {
      const int c = j % kCt;
      if (knorm && j + 1 < NC && (j + 1) % kCt == 0 && !(ok = normalise_k(j + 1))) break;
      if (j + 1 < NC && !(ok = convert(j + 1))) break;
      // Y^T: lane v (value row), columns t < C.  Y / sqrt(Dk) goes, as bf16 and
      // transposed, into this chunk's Qh rows (dead once Y is complete) and is
      // added to y (which holds y_loc / sqrt(Dk)) by a TMA reduction.
      const int v = 32 * qd + lane;
      const uint32_t qst = q_addr(j);
      uint8_t* hbase = sm + (qst - sbase) + (v >> 6) * 8192;
      const int vv = v & 63;
      if (!(ok = mbar_wait(bar(kQY), j & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int t0 = 0; t0 < C; t0 += 32) {
        float d[32];
        if constexpr (C >= 32) {
          tmem_ld32(tY + lane_base + t0, d);
        } else {
          tmem_ld16(tY + lane_base + t0, d);
        }
        tmem_wait_ld();
        if (t0 + 32 >= C) {
          tc_fence_before();
          mbar_arrive(bar(kQYFree));
        }
#pragma unroll
        for (int i = 0; i < (C < 32 ? C : 32); ++i) {
          const int row = c * C + t0 + i;
          const uint32_t off = row * 128 + ((((vv >> 3) ^ (row & 7))) << 4) + (vv & 7) * 2;
          *reinterpret_cast<bf16*>(hbase + off) = __float2bfloat16_rn(d[i] * scale);
        }
      }
      fence_proxy_async();
      mbar_arrive(bar(kQYStaged));
      if (warp == 10 && lane == 0) {
        if (!(ok = mbar_wait(bar(kQYStaged), j & 1))) break;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          tma_reduce_add_4d(tm_yred, qst + hh * 8192 + c * C * 128, 64 * hh, hv, j * C, b);
        bulk_commit();
        bulk_wait_read_all();  // the Q buffers may be refilled once the reduction has read them
        if (last_of_tile(j)) mbar_arrive(bar(kQEmptyQ + ring_q(j)));
      }
    }
    if (warp == 10 && lane == 0) bulk_wait_all();
  }
  // the idle lanes of warps 0 and 14 have no scan work
  tc_fence_before();
  if (warp != 0 && warp != 14) named_bar_sync(1, kFusedThreads - 64);
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int C>
__global__ void __launch_bounds__(kFusedThreads, 1)
fused_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_a1s,
                     const __grid_constant__ CUtensorMap tm_us,
                     const __grid_constant__ CUtensorMap tm_y,
                     const __grid_constant__ CUtensorMap tm_yred, const bf16* kin,
                     const bf16* qin, const bf16* vin, const bf16* __restrict__ g,
                     const bf16* __restrict__ beta, float* __restrict__ wsGC, int* flags,
                     const float* state_in, float* state_out, int T, int Hk, int Hv, int NT,
                     int BH, int opts, float scale) {
  extern __shared__ uint8_t smem_raw[];
  if ((int)blockIdx.x < BH) {
    scan_role128<C>(&tm_a1s, &tm_k, &tm_us, &tm_yred, wsGC, flags, state_in, state_out, T, Hk,
                    Hv, NT, blockIdx.x, opts, scale, smem_raw);
  } else {
    const PrepParams P{kin, qin, vin, &tm_k, &tm_q, &tm_v, &tm_a1s, &tm_us, g, beta, wsGC,
                       T, Hk, Hv, NT, BH, opts, &tm_y, scale};
    prep_role<C>(P, smem_raw, blockIdx.x - BH, gridDim.x - BH, flags);
  }
}

// The scan alone (after prep_tc_kernel in stream order): one CTA per head.
template <int C>
__global__ void __launch_bounds__(kFusedThreads, 1)
scan_head_kernel(const __grid_constant__ CUtensorMap tm_a1s, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_us,
                 const __grid_constant__ CUtensorMap tm_yred, const float* __restrict__ wsGC,
                 const float* state_in, float* state_out, int T, int Hk, int Hv, int NT,
                 int opts, float scale) {
  extern __shared__ uint8_t smem_raw[];
  scan_role128<C>(&tm_a1s, &tm_k, &tm_us, &tm_yred, wsGC, nullptr, state_in, state_out, T, Hk,
                  Hv, NT, blockIdx.x, opts, scale, smem_raw);
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
bool make_bthd_map(CUtensorMap* m, const void* base, int B, int T, int H, int box_t = kTile) {
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2,
                                 (cuuint64_t)T * H * kD * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_t, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [rows, 128] bf16 2-D view of a workspace region.  Swizzled boxes use the
// swizzle whose span equals the box row (box_cols * 2 bytes: 32, 64 or 128).
bool make_rows_map(CUtensorMap* m, const void* base, size_t rows, int box_cols, int box_rows,
                   bool swizzle) {
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle)
    sw = box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                        : (box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// Streaming multiprocessors of the current device (cached per device).
int num_sms() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

template <int C>
cudaError_t launch_c(const PrefillArgs& a) {
  const int NT = (a.T + kTile - 1) / kTile;
  const int BH = a.B * a.Hv;
  const WsLayout w = ws_layout(BH, NT);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  bf16* wsA1 = reinterpret_cast<bf16*>(ws + w.a1);
  bf16* wsU = reinterpret_cast<bf16*>(ws + w.u);
  float* wsGC = reinterpret_cast<float*>(ws + w.gc);

  if (!encode_fn()) return cudaErrorNotSupported;
  CUtensorMap tk, tq, tv, ta1s, tus, ty, tyred;
  if (!make_bthd_map(&tk, a.k, a.B, a.T, a.Hk) || !make_bthd_map(&tq, a.q, a.B, a.T, a.Hk) ||
      !make_bthd_map(&tv, a.v, a.B, a.T, a.Hv) ||
      !make_rows_map(&ta1s, wsA1, (size_t)BH * NT * 128, 64, C, true) ||
      !make_rows_map(&tus, wsU, (size_t)BH * NT * kTile, 64, 64, true) ||
      !make_bthd_map(&ty, a.y, a.B, a.T, a.Hv) || !make_bthd_map(&tyred, a.y, a.B, a.T, a.Hv, C))
    return cudaErrorInvalidValue;

  const float scale = 1.0f / sqrtf((float)kD);
  const int sms = num_sms();
  const bf16* k = static_cast<const bf16*>(a.k);
  const bf16* q = static_cast<const bf16*>(a.q);
  const bf16* v = static_cast<const bf16*>(a.v);
  const bf16* g = static_cast<const bf16*>(a.g);
  const bf16* beta = static_cast<const bf16*>(a.beta);
  cudaError_t e;
  // Fused path: one scan CTA per head next to at least two thirds of the SMs
  // doing prep, in one cooperative launch.
  if (3 * BH <= sms) {
    int* flags = reinterpret_cast<int*>(ws + w.flags);
    e = cudaFuncSetAttribute(fused_prefill_kernel<C>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem);
    if (e == cudaSuccess) e = cudaMemsetAsync(flags, 0, (size_t)BH * NT * sizeof(int), a.stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = kFusedSmem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_prefill_kernel<C>, tk, tq, tv, ta1s, tus, ty, tyred, k,
                              q, v, g, beta, wsGC, flags, a.state_in, a.state_out, a.T, a.Hk,
                              a.Hv, NT, BH, a.options, scale);
  }

  // Split path: the persistent prep kernel on every SM, then one scan CTA per head.
  e = cudaFuncSetAttribute(prep_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kPrepSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(scan_head_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Scan128Smem::kTotal);
  if (e != cudaSuccess) return e;
  const int prep_ctas = std::min(sms, (BH * NT + kPrepGroups - 1) / kPrepGroups);
  prep_tc_kernel<C><<<prep_ctas, kPrepThreads, kPrepSmem, a.stream>>>(
      tk, tq, tv, ta1s, tus, ty, k, q, v, g, beta, wsGC, a.T, a.Hk, a.Hv, NT, BH, a.options,
      scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scan_head_kernel<C><<<BH, kFusedThreads, Scan128Smem::kTotal, a.stream>>>(
      ta1s, tk, tus, tyred, wsGC, a.state_in, a.state_out, a.T, a.Hk, a.Hv, NT, a.options,
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
