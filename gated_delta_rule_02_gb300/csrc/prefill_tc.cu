// Chunked prefill on the tcgen05 tensor cores (bf16 or fp16 inputs, fp32 state).
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
//   GW, F1, F2 (coefficient form, below): with P = T_L K and U = (I + A)^-1 (beta V),
//   it writes, per tile, in the input type: to the workspace A1 = per chunk
//   [-Pt; Qh / sqrt(Dk)] with Pt = G_C beta P (step 9), Qh = G Q - G M P (step 7,
//   M[t][i] = beta_i QK^T[t][i], i <= t), and Ut = Gam[C-1][.] U (step 9), plus
//   G_C (fp32) per chunk; y_local / sqrt(Dk) (step 6) straight into y.
// scan (scan_role): one CTA per (b, hv) carries S (128 x 128, fp32) through the
// chunks.  With Z = S Pt^T, step 9 reads S <- G_C S + (Ut^T - Z) K (the
// innovation form of the update: Ut^T K - S Pt^T K), and steps 7-8 y = Y / sqrt(Dk)
// + y_local with Y^T = S Qh^T, so per chunk
//   [-Z | Y^T / sqrt(Dk)] = S A1^T      (S as a 16-bit tensor-memory operand)
//   D2 = Ut^T K + (-Z) K;  S <- G_C S + D2;  y += Y / sqrt(Dk) (TMA reduction)
// and only the first product and (-Z) K wait for the state.
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

// The 16-bit input types the tensor cores take here (kind::f16: A and B of one
// product always share a type, so every operand the kernels build is stored
// in the input type): bf16 and fp16.
template <typename E>
struct ElemT;
template <>
struct ElemT<__nv_bfloat16> {
  static constexpr uint32_t kFmt = 1;        // tcgen05 kind::f16 A/B format field
  static constexpr uint16_t kOne = 0x3f80;   // 1.0
  static constexpr CUtensorMapDataType kTmap = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  __device__ static uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static float2 unpack2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
  __device__ static float bits(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }
  __device__ static __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct ElemT<__half> {
  static constexpr uint32_t kFmt = 0;
  static constexpr uint16_t kOne = 0x3c00;
  static constexpr CUtensorMapDataType kTmap = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  __device__ static uint32_t pack2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static float2 unpack2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
  __device__ static float bits(uint16_t x) { return __half2float(__ushort_as_half(x)); }
  __device__ static __half from(float x) { return __float2half_rn(x); }
};
// Instruction descriptor of a kind::f16 product with A and B of type E.
template <typename E>
__host__ __device__ constexpr uint32_t idesc_e(int M, int N, bool a_mn, bool b_mn) {
  return idesc_kind_f16(M, N, a_mn, b_mn, ElemT<E>::kFmt);
}

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
  w.u = align256(tiles * 128 * kD * 2);  // 16-bit elements
  w.gc = w.u + align256(tiles * kTile * kD * 2);
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
template <typename E>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  return ElemT<E>::pack2(a, b);
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
template <typename E>
__device__ __forceinline__ void unpack8(uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = ElemT<E>::unpack2(w[i]);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}
template <typename E>
__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack2<E>(f[0], f[1]), pack2<E>(f[2], f[3]), pack2<E>(f[4], f[5]),
                    pack2<E>(f[6], f[7]));
}

// x / |x| for row `row` of a 16-bit tile whose rows are split in two
// 128B-swizzled 64-column halves `half_stride` bytes apart; the calling thread
// takes half `half` and its lane partner (lane ^ 1) the other half.
template <typename E>
__device__ __forceinline__ void l2norm_row_sw128(uint8_t* base, int half_stride, int row,
                                                 int half) {
  uint8_t* hb = base + half * half_stride;
  float ss = 0.f;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    float v[8];
    unpack8<E>(*reinterpret_cast<const uint4*>(hb + sw128(row, 8 * ch)), v);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  const float f = inv_norm(ss);
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint4* p = reinterpret_cast<uint4*>(hb + sw128(row, 8 * ch));
    float v[8];
    unpack8<E>(*p, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] *= f;
    *p = pack8<E>(v);
  }
}

// ============================================================================
// prep kernel
// ============================================================================
// The prep kernel is persistent: one CTA per SM holds two independent groups
// of eight warps, each with its own shared-memory map, 256 TMEM columns and
// mbarriers, each looping over tiles.
//
// Per tile (64 tokens of one (b, hv) head; 64 / C chunks, every C x C matrix
// block diagonal by chunk) a group runs, with T_L = (I + L)^-1 and
// T_A = diag(beta) (Gam . T_L) (the second solve of step 5 without a second
// inverse, (I + A)^-1 diag(beta) = diag(beta)(Gam . T_L)):
//   G1  [K; Q] K^T                              -> KK^T, QK^T        (step 3)
//   build  L = beta_j KK^T (strict lower), A3 = [diag(G) M; Gam . QK^T]
//          with M[t][i] = beta_i QK^T[t][i] (i <= t)
//   T_L    16 x 16 diagonal blocks by substitution (fp32), then the 16 -> 32
//          -> 64 merges T_BA = -T_BB (L_BA T_AA) on warp-level bf16 MMAs  (step 4)
//   coefs  cP = -diag(G_C beta) T_L, cU = diag(Gam[C-1][.]) T_A
//   GW  A3 [T_L | T_A]  -> W_M = diag(G) M T_L,  W_Y = (Gam . QK^T) T_A
//   F1  [cP; -W_M / sqrt(Dk)] K -> -Pt = -G_C beta P (step 9),
//                                  (Qh - diag(G) Q) / sqrt(Dk)  (step 7)
//   F2  [cU; W_Y / sqrt(Dk)] V -> Ut = Gam[C-1][.] U (step 9), y_loc / sqrt(Dk) (step 6)
// so every row of the two final products is an output; the epilogue adds
// diag(G) Q / sqrt(Dk) to the Qh rows.
constexpr int kPrepGroups = 2;
constexpr int kPrepGroupThreads = 256;
constexpr int kPrepThreads = kPrepGroups * kPrepGroupThreads;
// A tile's flag counts to kTilePublished: each of the group's two I/O threads
// (lane 0 of warps 2 and 6) adds 1 once its own stores of the tile are in
// global memory.
constexpr int kTilePublished = 2;
// Shared-memory map of one group (bytes from its 1024-aligned base).  The
// bf16 operand blocks X0..X5 are 64 rows x 64 columns, 128B-swizzled (8 KB).
constexpr uint32_t kOffKQ = 0;        // [K;Q]: 2 halves x (64 K rows + 64 Q rows) x 128 B
constexpr uint32_t kOffV = 32768;     // V: 2 halves x 64 rows x 128 B
// Once F1 has read X0, X1 (and GW X2, X3), X0..X3 stage the tile's A1 rows
// ([Pt; Qh] per chunk, 32 KB); once F2 has read X4, X5 and V, they stage y_loc
// and Ut.  Staging blocks hold rows of 128 values as [row][64-column half],
// each 128-byte unit 128B-swizzled, which is the box layout of the 3-D (A1,
// Ut) and 5-D (y) tensor maps the stores use: one TMA store per output.
constexpr uint32_t kOffX0 = 49152;    // cP                 | A1 staging (X0..X3)
constexpr uint32_t kOffX1 = 57344;    // A3 top, then -W_M
constexpr uint32_t kOffX2 = 65536;    // A3 bottom
constexpr uint32_t kOffX3 = 73728;    // T_A
constexpr uint32_t kOffX4 = 81920;    // cU                 | y_loc staging (X4, X5)
constexpr uint32_t kOffX5 = 90112;    // T_L, then W_Y
constexpr uint32_t kOffXd = 98304;    // fp32 [4][16][16]: the diagonal 16 x 16 blocks of L
constexpr int kLd1 = 24;              // bf16 row stride (elements) of the 16-wide scratch
constexpr int kLd2 = 40;              // bf16 row stride of the 32-wide scratch
constexpr uint32_t kOffXl1 = kOffXd + 4096;          // bf16 [2][16][kLd1]: L_10, L_32
constexpr uint32_t kOffXl2 = kOffXl1 + 2 * 16 * kLd1 * 2;  // bf16 [32][kLd2]: L_BA
constexpr uint32_t kOffZs = kOffXl2 + 32 * kLd2 * 2;       // bf16 [32][kLd2] (merge products)
constexpr uint32_t kOffSmall = kOffZs + 32 * kLd2 * 2;     // per-token scalars
constexpr uint32_t kPrepGroupSmem = (kOffSmall + (64 * 9 + 4) * 4 + 1023) & ~1023u;
constexpr uint32_t kPrepSmem = kPrepGroups * kPrepGroupSmem + 1024;
static_assert(kPrepSmem <= 232448, "prep shared memory");

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

// Warp-level m16n8k16 MMA (16-bit inputs, fp32 accumulate) with ldmatrix operand loads:
// the inverse's block products are too small for tcgen05 (M >= 64).
// Fragments (g = lane / 4, c = lane % 4): A 16 x 16 row-major in four 8 x 8
// matrices (rows 0-7 / 8-15 x cols 0-7 / 8-15), B 16 x 8 with b0 = rows 2c,
// 2c+1 of column g and b1 the same 8 rows down, D d0 (g, 2c) d1 (g, 2c+1)
// d2 (g+8, 2c) d3 (g+8, 2c+1).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
template <typename E>
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, const uint32_t* b) {
  if constexpr (ElemT<E>::kFmt == 1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
}
// Lane address of an ldmatrix.x4 A fragment (rows r0.., cols c0..) and of an
// ldmatrix.x2.trans B fragment (rows k0.. of a row-major [k][n] block, cols
// n0..): in a plain row-major 16-bit array of `ld` elements per row ...
__device__ __forceinline__ uint32_t a_frag_addr(uint32_t base, int ld, int r0, int c0, int lane) {
  return base + ((r0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * ld + c0 + 8 * (lane >> 4)) * 2;
}
__device__ __forceinline__ uint32_t b_frag_addr(uint32_t base, int ld, int k0, int n0, int lane) {
  return base + ((k0 + (lane & 15)) * ld + n0) * 2;
}
// ... and in a 128B-swizzled 64-column block (row stride 128 B).
__device__ __forceinline__ uint32_t a_frag_addr_sw(uint32_t base, int r0, int c0, int lane) {
  const int r = r0 + (lane & 7) + 8 * ((lane >> 3) & 1), c = c0 + 8 * (lane >> 4);
  return base + sw128(r, c);
}
__device__ __forceinline__ uint32_t b_frag_addr_sw(uint32_t base, int k0, int n0, int lane) {
  return base + sw128(k0 + (lane & 15), n0);
}
// Writes a 16 x 8 fp32 fragment times `sign` as type E at (r0, c0) of a
// swizzled block / of a row-major array.
template <typename E>
__device__ __forceinline__ void st_frag_sw(uint8_t* blk, int r0, int c0, const float* d, float sign,
                                           int lane) {
  const int g = lane >> 2, c = 2 * (lane & 3);
  *reinterpret_cast<uint32_t*>(blk + sw128(r0 + g, c0 + c)) = pack2<E>(sign * d[0], sign * d[1]);
  *reinterpret_cast<uint32_t*>(blk + sw128(r0 + g + 8, c0 + c)) =
      pack2<E>(sign * d[2], sign * d[3]);
}
template <typename E>
__device__ __forceinline__ void st_frag(uint8_t* arr, int ld, int r0, int c0, const float* d,
                                        int lane) {
  const int g = lane >> 2, c = 2 * (lane & 3);
  *reinterpret_cast<uint32_t*>(arr + ((r0 + g) * ld + c0 + c) * 2) = pack2<E>(d[0], d[1]);
  *reinterpret_cast<uint32_t*>(arr + ((r0 + g + 8) * ld + c0 + c) * 2) = pack2<E>(d[2], d[3]);
}

// Everything the prep work needs (the tensor maps are kernel parameters).
template <typename E>
struct PrepParams {
  const CUtensorMap* tm_k;    // the inputs as [B][T][H][128], box {64, 1, 64, 1}
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_a1o;  // A1 as [rows][2][64] (3-D), box {64, 2, 128}
  const CUtensorMap* tm_uo;   // Ut as [rows][2][64], box {64, 2, 64}
  const CUtensorMap* tm_yo;   // y as [B][T][Hv][2][64] (5-D), box {64, 2, 1, 64, 1}
  const E* g;
  const E* beta;
  float* wsGC;
  int T, Hk, Hv, NT, BH;
  int opts;  // kOpt* bits
  // y_loc / sqrt(Dk) goes straight into y; the scan then adds Qh S^T / sqrt(Dk).
  float yscale;
};

// The prep work of one CTA (both groups): CTA `cta_rank` of `n_ctas` doing prep.
// With `flags`, each finished tile (b*Hv + hv, n) is published by raising
// flags[(b*Hv + hv) * NT + n] to kTilePublished: each I/O thread adds 1 once
// its own stores of the tile are in global memory.
template <int C, typename E>
__device__ __forceinline__ void prep_role(const PrepParams<E>& P, uint8_t* smem_raw, int cta_rank,
                                          int n_ctas, int* flags) {
  const int T = P.T, Hk = P.Hk, Hv = P.Hv, NT = P.NT, BH = P.BH, opts = P.opts;
  const E* __restrict__ g = P.g;
  const E* __restrict__ beta = P.beta;
  float* __restrict__ wsGC = P.wsGC;
  // Per group: K and Q landed (128 cp.async arrivals, stream A), G1, GW, F1, F2,
  // V landed (128 arrivals, stream B) -- each completes once per tile.
  __shared__ uint64_t bars[kPrepGroups][6];
  __shared__ uint32_t tmem_base_sh;
  __shared__ float carry_sh[kPrepGroups];
  __shared__ int abort_sh[kPrepGroups];
  const int grp = threadIdx.x / kPrepGroupThreads;
  const int tid = threadIdx.x % kPrepGroupThreads, warp = tid >> 5, lane = tid & 31;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~(uintptr_t)1023) +
                grp * kPrepGroupSmem;
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar_tma = smem_u32(&bars[grp][0]), bar_g1 = smem_u32(&bars[grp][1]);
  const uint32_t bar_gw = smem_u32(&bars[grp][2]), bar_f1 = smem_u32(&bars[grp][3]);
  const uint32_t bar_f2 = smem_u32(&bars[grp][4]), bar_v = smem_u32(&bars[grp][5]);
  // Named barriers of the group: the whole group, the two warps of the gate
  // prefix sums, the two epilogue streams (warps 0-3: F1; warps 4-7: F2) and the
  // four warps on the KK^T lanes (0, 1, 4, 5).
  const int sync_id = 1 + grp, carry_id = 3 + grp, streamA_id = 5 + grp, streamB_id = 7 + grp;
  const int kk_id = 9 + grp;
  const bool streamA = warp < 4;
  float* Xd = reinterpret_cast<float*>(sm + kOffXd);
  float* lam = reinterpret_cast<float*>(sm + kOffSmall);  // chunk-local sum of log2 g
  float* bta = lam + 64;
  float* gsuf = bta + 64;   // g_{t+1} ... g_{chunk end}
  float* gpw = gsuf + 64;   // G_t = g_{chunk start} ... g_t
  float* sfac = gpw + 64;   // 2^(lam[end of t's 16-block] - lam_t)
  float* rfac = sfac + 64;  // [64][4]: 2^(lam_t - lam[end of block b]), b before t's block, same chunk
  float* gc = rfac + 256;   // G at each chunk's end
  auto gsync = [&]() { named_bar_sync(sync_id, kPrepGroupThreads); };
  // Group-wide AND of ok (sticky: a group that failed a wait stops).
  auto gsync_and = [&](bool v) {
    if (!v) abort_sh[grp] = 1;
    gsync();
    return abort_sh[grp] == 0;
  };

  if (threadIdx.x == 0) {
    for (int q = 0; q < kPrepGroups; ++q) {
      for (int i = 0; i < 6; ++i) mbar_init(smem_u32(&bars[q][i]), 1);
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
  // The two I/O threads issue the TMA copies of the group: io 0 loads K and Q
  // (into the 128B-swizzled operand layout; rows past T read as zeros) and
  // stores the tile's A1 rows, io 1 loads V and stores y_loc and Ut, and each
  // publishes the tile once its stores have landed.  io 0 loads the next
  // tile's K and Q as soon as this tile's F1 and Qh epilogue are done with
  // them (before its stores, so the loads do not queue behind them); io 1
  // loads a tile's V at its start, once the previous Ut store (staged over V)
  // has read it.
  const int io = tid == 64 ? 0 : (tid == 192 ? 1 : -1);
  bool kq_pending = false, v_pending = false;  // loads issued and not yet waited for
  auto load_kq = [&](int lin) {  // io 0
    const int bh = head_of(lin), b = bh / Hv, hv = bh - b * Hv;
    const int hk = key_head(hv, Hk, Hv, opts), t0 = tile_of(lin) * kTile;
    fence_proxy_async();  // earlier generic reads of the buffers, before the copies
    mbar_expect_tx(bar_tma, 32768);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tma_load_4d(sbase + kOffKQ + h * 16384, P.tm_k, bar_tma, 64 * h, hk, t0, b);
      tma_load_4d(sbase + kOffKQ + h * 16384 + 8192, P.tm_q, bar_tma, 64 * h, hk, t0, b);
    }
    kq_pending = true;
  };
  auto load_v = [&](int lin) {  // io 1
    const int bh = head_of(lin), b = bh / Hv, hv = bh - b * Hv, t0 = tile_of(lin) * kTile;
    fence_proxy_async();
    mbar_expect_tx(bar_v, 16384);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      tma_load_4d(sbase + kOffV + h * 8192, P.tm_v, bar_v, 64 * h, hv, t0, b);
    v_pending = true;
  };
  // Gate and beta of token `tid` of a tile, read one tile ahead into registers
  // as raw 16-bit values (converted when used, so the load is not waited for here).
  // Padded tokens: decay 1 (gate 1.0, or log-gate 0.0), beta 0.
  const uint16_t g_pad = (opts & kOptLogGate) ? 0x0000 : ElemT<E>::kOne;
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
  if (io == 0) {
    prefetch_tmap(P.tm_k);
    prefetch_tmap(P.tm_q);
    prefetch_tmap(P.tm_a1o);
  }
  if (io == 1) {
    prefetch_tmap(P.tm_v);
    prefetch_tmap(P.tm_yo);
    prefetch_tmap(P.tm_uo);
  }
  if (gid < total) {
    if (io == 0) load_kq(gid);
    if (io == 1) load_v(gid);
  }
  load_gates(gid);

  bool ok = true;
  // The tile whose stores this I/O thread has issued but not yet published.
  size_t unpublished = ~(size_t)0;
  auto publish = [&]() {
    if (unpublished != ~(size_t)0) {
      bulk_wait_all();
      fence_proxy_async_global();
      if (flags) red_release_gpu_add(flags + unpublished, 1);
      unpublished = ~(size_t)0;
    }
  };
  // TMEM lane quadrant of this warp, its row in a 128-lane accumulator and the
  // token row t of a 64-row half.
  const int q4 = warp & 3, lrow = q4 * 32 + lane, trow = lrow & 63;
  const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
  int it = 0;
  // ok (false once a bounded wait has given up) is made uniform by the first
  // group barrier of each tile, where the loop stops, so every thread passes the
  // same barriers.
  for (int lin = gid; lin < total; lin += ngroups, ++it) {
  const size_t tile_id = (size_t)head_of(lin) * NT + tile_of(lin);
  const int next = lin + ngroups;
  const float gv_cur = ElemT<E>::bits(g_next), bt_cur = ElemT<E>::bits(b_next);
  load_gates(next);
  // Gates (step 2).  Padded tokens take g = 1, beta = 0.  Decay products are
  // carried as chunk-local prefix sums lam of log2 g: G_t = 2^lam_t and
  // Gam[t][j] = 2^(lam_t - lam_j) (j <= t) -- never a quotient, so a vanishing
  // product underflows to 0.  Warps 0-1 form the prefix sums (one token per
  // thread) and the per-token tables.
  if (tid < 64) {
    const int t = tid;
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
    named_bar_sync(carry_id, 64);
    // Per-token tables: G_t, the decay to the chunk's end, and the two
    // factors of Gam across 16-token blocks (both products of decays, <= 1):
    // Gam[t][j] = rfac[t][b(j)] sfac[j] for j in an earlier block b(j).
    const int cs = (t / C) * C, tb = t >> 4;
    gsuf[t] = ex2(lam[cs + C - 1] - l);
    gpw[t] = ex2(l);
    sfac[t] = ex2(lam[t | 15] - l);
#pragma unroll
    for (int bb = 0; bb < 4; ++bb)
      rfac[t * 4 + bb] = (bb < tb && 16 * bb >= cs) ? ex2(l - lam[16 * bb + 15]) : 0.f;
    if ((t % C) == C - 1) gc[t / C] = ex2(l);
  }

  ok = ok && mbar_wait(bar_tma, it & 1);
  kq_pending = false;
  // The previous tile's stores have read their staging (X0..X5, V) before this
  // tile rewrites it.
  if (io >= 0) bulk_wait_read_all();
  if (opts & kOptL2NormQK) {  // rows 0-63 of each half are K, 64-127 Q
    if (ok) l2norm_row_sw128<E>(sm + kOffKQ, 16384, tid >> 1, tid & 1);
    fence_proxy_async();
    gsync();
  }
  ok = gsync_and(ok);  // also publishes the gate scalars
  if (!ok) break;
  // G1: D[128 x 64] = [K; Q] K^T (TMEM columns 0..63), issued by a thread
  // outside the gate warps (lane 1 of warp 4).
  if (tid == 129) {
    tc_fence_after();
    const uint32_t id1 = idesc_e<E>(128, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t a = sbase + kOffKQ + (kk >> 2) * 16384 + (kk & 3) * 32;
      mma_f16_ss(tmem, smem_desc(a, 16, 1024, kSw128), smem_desc(a, 16, 1024, kSw128), id1,
                  kk > 0);
    }
    mma_commit(bar_g1);
  }
  if (io >= 0) publish();        // the previous tile, stored a while ago
  if (io == 1 && it > 0) load_v(lin);  // V for F2, over the previous Ut staging
  ok = ok && mbar_wait(bar_g1, it & 1);
  tc_fence_after();
  // Warps w and w+4 share TMEM lane quadrant w % 4 and take 32 columns each.
  // The warps on the KK^T lanes (0, 1, 4, 5) build L and go on to the
  // inverse's diagonal blocks, which need nothing else; the warps on the QK^T
  // lanes (2, 3, 6, 7) build A3 meanwhile and meet them at the first merge.
  const bool kk_lanes = lrow < 64;
  {
    const int t = trow, cs = (t / C) * C, tb = t >> 4;
    const int cbeg = (warp >> 2) * 32;
    float v[32];
    if (ok) {
      tmem_ld16(tmem + lane_base + cbeg, v);
      tmem_ld16(tmem + lane_base + cbeg + 16, v + 16);
      tmem_wait_ld();
    }
    if (kk_lanes) {
      // Row t of KK^T -> L[t][j] = beta_j KK^T[t][j], j < t in t's chunk: its
      // diagonal 16 x 16 block in fp32 (Xd) and, as bf16, the blocks the merges
      // read (L_10, L_32 in Xl1; L_BA in Xl2).
      if (ok) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int j = cbeg + e;
          v[e] = (j < t && j >= cs) ? bta[j] * v[e] : 0.f;
        }
        if ((tb >> 1) == (cbeg >> 5)) {  // t's diagonal block lies in these 32 columns
          float* xd = Xd + tb * 256 + (t & 15) * 16;
          const bool hi = tb & 1;  // which 16 of the 32 columns (selects keep v in registers)
          float src[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) src[e] = hi ? v[16 + e] : v[e];
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(xd + e) =
                make_float4(src[e], src[e + 1], src[e + 2], src[e + 3]);
        }
        uint8_t* xl1 = sm + kOffXl1;
        if (cbeg == 0 && t >= 16 && t < 32) {  // L_10: rows 16-31, cols 0-15
          uint8_t* row = xl1 + ((t - 16) * kLd1) * 2;
          *reinterpret_cast<uint4*>(row) = pack8<E>(v);
          *reinterpret_cast<uint4*>(row + 16) = pack8<E>(v + 8);
        }
        if (cbeg == 32 && t >= 48) {  // L_32: rows 48-63, cols 32-47
          uint8_t* row = xl1 + ((16 + t - 48) * kLd1) * 2;
          *reinterpret_cast<uint4*>(row) = pack8<E>(v);
          *reinterpret_cast<uint4*>(row + 16) = pack8<E>(v + 8);
        }
        if (cbeg == 0 && t >= 32) {  // L_BA: rows 32-63, cols 0-31
          uint8_t* row = sm + kOffXl2 + ((t - 32) * kLd2) * 2;
#pragma unroll
          for (int e = 0; e < 32; e += 8) *reinterpret_cast<uint4*>(row + 2 * e) = pack8<E>(v + e);
        }
      }
      tc_fence_before();
      named_bar_sync(kk_id, 128);
      // Step 4, T_L = (I + L)^-1 into X5 (bf16, row-major [t][j]): the
      // diagonal 16 x 16 blocks (warps 0, 1), and zeros in the blocks no merge
      // writes (warps 4, 5).  It runs on whatever L holds even after a failed
      // wait, so every thread passes the same barriers.
      uint8_t* x5 = sm + kOffX5;
      if (warp < 4) {
        // block bl, column jj, by forward substitution (fp32)
        const int bl = tid >> 4, jj = tid & 15;
        const float* xd = Xd + bl * 256;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float a0 = (r == jj) ? 1.f : 0.f, a1 = 0.f;
          const float* xr = xd + r * 16;
#pragma unroll
          for (int s = 0; s + 1 < r; s += 2) {
            a0 = fmaf(-xr[s], x[s], a0);
            a1 = fmaf(-xr[s + 1], x[s + 1], a1);
          }
          if (r & 1) a0 = fmaf(-xr[r - 1], x[r - 1], a0);
          x[r] = a0 + a1;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r)
          *reinterpret_cast<E*>(x5 + sw128(16 * bl + r, 16 * bl + jj)) =
              ElemT<E>::from(x[r]);
      } else {
        // above the diagonal, and across chunks (C < 64): 32 16-byte pieces a block
        for (int p = tid - 128; p < 16 * 32; p += 64) {
          const int blk = p >> 5, rb = blk >> 2, cb = blk & 3;
          if (cb > rb || (16 * rb) / C != (16 * cb) / C) {
            const int r = 16 * rb + ((p & 31) >> 1), c = 16 * cb + 8 * (p & 1);
            *reinterpret_cast<uint4*>(x5 + sw128(r, c)) = make_uint4(0, 0, 0, 0);
          }
        }
      }
    } else if (ok) {
      // Row t of QK^T -> rows t of A3 top (X1) and bottom (X2):
      //   diag(G) M and Gam . QK^T,  M[t][i] = beta_i QK^T[t][i], i <= t.
      // Gam inside t's 16-block is 2^(lam_t - lam_j); across blocks it is
      // rfac[t][b] sfac[j].
      const float gt = gpw[t], lt = lam[t];
      float top[32];
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int jb = (cbeg >> 4) + hb;
        const float rb = jb < 4 ? rfac[t * 4 + jb] : 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = cbeg + 16 * hb + e;
          const bool keep = j <= t && j >= cs;
          const float gm = jb == tb ? ex2(lt - lam[j]) : rb * sfac[j];
          top[16 * hb + e] = keep ? gt * bta[j] * v[16 * hb + e] : 0.f;
          v[16 * hb + e] = keep ? gm * v[16 * hb + e] : 0.f;
        }
      }
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        st_sm16(sm, kOffX1 + sw128(t, cbeg + e), pack8<E>(top + e));
        st_sm16(sm, kOffX2 + sw128(t, cbeg + e), pack8<E>(v + e));
      }
      fence_proxy_async();
    }
  }
  tc_fence_before();
  gsync();

  // Step 4, merges of the diagonal blocks of T_L (in X5).
  {
    uint8_t* x5 = sm + kOffX5;
    const uint32_t x5a = sbase + kOffX5, zsa = sbase + kOffZs;
    uint8_t* zs = sm + kOffZs;
    if constexpr (C >= 32) {
      // 16 -> 32: T_R0 = -T_RR (L_R0 T_00) for the block pairs p = 0, 1 (R = 2p+1,
      // 0 = 2p); warp w < 4 takes pair w / 2, output columns 8 (w % 2) ...
      const int p = (warp >> 1) & 1, nh = warp & 1, R = 16 * (2 * p + 1), c0 = 32 * p;
      if (warp < 4) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a[4], bb[2];
        ldsm_x4(a_frag_addr(sbase + kOffXl1, kLd1, 16 * p, 0, lane), a);
        ldsm_x2_trans(b_frag_addr_sw(x5a, c0, c0 + 8 * nh, lane), bb);
        mma_16816<E>(d, a, bb);
        st_frag<E>(zs, kLd1, 16 * p, 8 * nh, d, lane);
      }
      gsync();
      if (warp < 4) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a[4], bb[2];
        ldsm_x4(a_frag_addr_sw(x5a, R, R, lane), a);
        ldsm_x2_trans(b_frag_addr(zsa, kLd1, 16 * p, 8 * nh, lane), bb);
        mma_16816<E>(d, a, bb);
        st_frag_sw<E>(x5, R, c0 + 8 * nh, d, -1.f, lane);
      }
      gsync();
    }
    if constexpr (C == 64) {
      // 32 -> 64: T_BA = -T_BB (L_BA T_AA), A = [0, 32), B = [32, 64); warp w
      // takes the 16 x 8 output tile (w / 4, w % 4) of each product.
      const int mt = warp >> 2, nt = warp & 3;
      {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a[4], bb[2];
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 16) {
          ldsm_x4(a_frag_addr(sbase + kOffXl2, kLd2, 16 * mt, k0, lane), a);
          ldsm_x2_trans(b_frag_addr_sw(x5a, k0, 8 * nt, lane), bb);
          mma_16816<E>(d, a, bb);
        }
        st_frag<E>(zs, kLd2, 16 * mt, 8 * nt, d, lane);
      }
      gsync();
      {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a[4], bb[2];
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 16) {
          ldsm_x4(a_frag_addr_sw(x5a, 32 + 16 * mt, 32 + k0, lane), a);
          ldsm_x2_trans(b_frag_addr(zsa, kLd2, k0, 8 * nt, lane), bb);
          mma_16816<E>(d, a, bb);
        }
        st_frag_sw<E>(x5, 32 + 16 * mt, 8 * nt, d, -1.f, lane);
      }
      gsync();
    }
  }

  // Coefficients, row t, columns 16 cg .. 16 cg + 15 (four threads a row):
  //   T_A = beta_t Gam[t][j] T_L[t][j]      -> X3
  //   cP  = G_C beta_t T_L[t][j]            -> X0
  //   cU  = Gam[C-1][t] T_A[t][j]           -> X4
  // T_L is zero above the diagonal and across chunks, and so is Gam here.
  if (ok) {
    const int t = tid >> 2, c0 = 16 * (tid & 3), cs = (t / C) * C;
    const float bt = bta[t], lt = lam[t], gcp = -gc[t / C] * bt, gs = gsuf[t];
    float tl[16], ta[16], cp[16], cu[16];
    unpack8<E>(*reinterpret_cast<const uint4*>(sm + kOffX5 + sw128(t, c0)), tl);
    unpack8<E>(*reinterpret_cast<const uint4*>(sm + kOffX5 + sw128(t, c0 + 8)), tl + 8);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int j = c0 + e;
      const float gm = (j <= t && j >= cs) ? ex2(lt - lam[j]) : 0.f;
      ta[e] = bt * gm * tl[e];
      cp[e] = gcp * tl[e];
      cu[e] = gs * ta[e];
    }
    st_sm16(sm, kOffX3 + sw128(t, c0), pack8<E>(ta));
    st_sm16(sm, kOffX3 + sw128(t, c0 + 8), pack8<E>(ta + 8));
    st_sm16(sm, kOffX0 + sw128(t, c0), pack8<E>(cp));
    st_sm16(sm, kOffX0 + sw128(t, c0 + 8), pack8<E>(cp + 8));
    st_sm16(sm, kOffX4 + sw128(t, c0), pack8<E>(cu));
    st_sm16(sm, kOffX4 + sw128(t, c0 + 8), pack8<E>(cu + 8));
    fence_proxy_async();
  }
  ok = gsync_and(ok);

  // GW (thread 0): D[128 x 128] = A3 [T_A | T_L]: rows 0-63 x cols 64-127 are
  // W_M = diag(G) M T_L, rows 64-127 x cols 0-63 are W_Y = (Gam . QK^T) T_A.
  if (ok && tid == 0) {
    tc_fence_after();
    const uint32_t idw = idesc_e<E>(128, 128, false, true);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f16_ss(tmem, smem_desc(sbase + kOffX1 + kk * 32, 16, 1024, kSw128),
                  smem_desc(sbase + kOffX3 + kk * 2048, 16384, 1024, kSw128), idw, kk > 0);
    mma_commit(bar_gw);
  }
  ok = ok && mbar_wait(bar_gw, it & 1);
  tc_fence_after();
  if (ok) {
    // -W_M over A3 top (X1), W_Y / sqrt(Dk) over T_L (X5): both operands of GW,
    // which has completed.  32 columns per thread.
    const int t = trow, c0 = (warp >> 2) * 32;
    float v[32];
    const bool top = lrow < 64;
    tmem_ld16(tmem + lane_base + (top ? 64 : 0) + c0, v);
    tmem_ld16(tmem + lane_base + (top ? 64 : 0) + c0 + 16, v + 16);
    tmem_wait_ld();
    const float s = top ? -P.yscale : P.yscale;
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] *= s;
    const uint32_t dst = top ? kOffX1 : kOffX5;
#pragma unroll
    for (int e = 0; e < 32; e += 8) st_sm16(sm, dst + sw128(t, c0 + e), pack8<E>(v + e));
    fence_proxy_async();
  }
  tc_fence_before();
  ok = gsync_and(ok);

  // F1 = [cP; -W_M] K (TMEM columns 0..127), F2 = [cU; W_Y / sqrt(Dk)] V
  // (columns 128..255), issued by thread 0; F1 commits to bar_f1 (stream A),
  // F2 to bar_f2 (stream B: it also covers F1, issued before it).
  if (ok && tid == 0) ok = mbar_wait(bar_v, it & 1);  // V of this tile has landed
  if (io == 1) v_pending = false;  // (thread 0's wait covers it: F2 has read V by the stores)
  if (ok && tid == 0) {
    tc_fence_after();
    const uint32_t idf = idesc_e<E>(128, 128, false, true);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f16_ss(tmem, smem_desc(sbase + kOffX0 + kk * 32, 16, 1024, kSw128),
                  smem_desc(sbase + kOffKQ + kk * 2048, 16384, 1024, kSw128), idf, kk > 0);
    mma_commit(bar_f1);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f16_ss(tmem + 128, smem_desc(sbase + kOffX4 + kk * 32, 16, 1024, kSw128),
                  smem_desc(sbase + kOffV + kk * 2048, 8192, 1024, kSw128), idf, kk > 0);
    mma_commit(bar_f2);
  }
  // A failed V wait on thread 0 leaves F1 / F2 unissued: the others' waits on
  // them then time out as well (bounded), and ok turns false everywhere.
  ok = ok && mbar_wait(streamA ? bar_f1 : bar_f2, it & 1);
  tc_fence_after();
  if (ok) {
    // Epilogue, 128 columns of row t per thread, staged as [row][half]
    // (128-byte units, 128B-swizzled) for one TMA store per output:
    //   warps 0, 1: Pt (F1, lanes 0-63)        -> A1 staging (X0..X3), row a(t)
    //   warps 2, 3: Qh = G_t q_t + F1 (64-127) -> A1 staging, row a(t) + C
    //   warps 4, 5: Ut (F2, lanes 0-63)        -> V, row t
    //   warps 6, 7: y_loc / sqrt(Dk) (F2)      -> X4, X5, row t
    // with a(t) = 2C (t / C) + t mod C, the row of Pt_t in the tile's A1 rows.
    const int t = trow;
    const uint32_t src = tmem + lane_base + (streamA ? 0 : 128);
    const bool top = lrow < 64;
    const float gt = gpw[t] * P.yscale;
    const int srow = streamA ? 2 * C * (t / C) + (t % C) + (top ? 0 : C) : t;
    const uint32_t sbuf = streamA ? kOffX0 : (top ? kOffV : kOffX4);
#pragma unroll
    for (int c2 = 0; c2 < 128; c2 += 32) {
      float v[32];
      tmem_ld16(src + c2, v);
      tmem_ld16(src + c2 + 16, v + 16);
      tmem_wait_ld();
      const int h = c2 >> 6, cc = c2 & 63;
      if (streamA && !top) {
        const uint32_t qsrc = kOffKQ + h * 16384 + 8192;
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float q8[8];
          unpack8<E>(*reinterpret_cast<const uint4*>(sm + qsrc + sw128(t, cc + e)), q8);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[e + i] = fmaf(gt, q8[i], v[e + i]);
        }
      }
#pragma unroll
      for (int e = 0; e < 32; e += 8)
        st_sm16(sm, sbuf + sw128(2 * srow + h, cc + e), pack8<E>(v + e));
    }
    fence_proxy_async();
  }
  if (ok && tid < 64 / C) wsGC[tile_id * 4 + tid] = gc[tid];
  tc_fence_before();  // the next tile's G1 rewrites these TMEM columns
  named_bar_sync(streamA ? streamA_id : streamB_id, 128);
  if (ok) {
    if (io == 0) {
      // K (read by F1) and Q (read by the Qh epilogue) are free: the next
      // tile's come in while this tile's stores drain.
      if (next < total) load_kq(next);
      // A1 rows of the tile (Pt and Qh of each chunk)
      tma_store_3d(P.tm_a1o, sbase + kOffX0, 0, 0, (int)(tile_id * 128));
      bulk_commit();
    } else if (io == 1) {
      const int bh = head_of(lin), b = bh / Hv;
      tma_store_5d(P.tm_yo, sbase + kOffX4, 0, 0, bh - b * Hv, tile_of(lin) * kTile,
                   b);  // y_loc / sqrt(Dk) (rows past T are clipped)
      tma_store_3d(P.tm_uo, sbase + kOffV, 0, 0, (int)(tile_id * kTile));  // Ut
      bulk_commit();
    }
    unpublished = tile_id;
  }
  }  // tile loop

  gsync();
  if (ok && io >= 0) publish();  // the group's last tile
  if (io >= 0) bulk_wait_all();   // shared memory must outlive the stores' reads
  // and every load into it must have landed (loads issued for a tile the loop
  // did not reach after a failed wait)
  if (kq_pending) mbar_wait(bar_tma, it & 1);
  if (v_pending) mbar_wait(bar_v, it & 1);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tmem_base_sh, 256 * kPrepGroups);
}

template <int C, typename E>
__global__ void __launch_bounds__(kPrepThreads, 1)
prep_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a1o,
               const __grid_constant__ CUtensorMap tm_uo, const __grid_constant__ CUtensorMap tm_yo,
               const E* __restrict__ g, const E* __restrict__ beta,
               float* __restrict__ wsGC, int T, int Hk, int Hv, int NT, int BH, int opts,
               float scale) {
  extern __shared__ uint8_t smem_raw[];
  const PrepParams<E> P{&tm_k, &tm_q, &tm_v, &tm_a1o, &tm_uo, &tm_yo, g, beta, wsGC,
                        T, Hk, Hv, NT, BH, opts, scale};
  prep_role<C, E>(P, smem_raw, blockIdx.x, gridDim.x, nullptr);
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
// The scan role carries S through the chunks in the form
//   [Z | Y^T] = S [Pt; Qh]^T           (Z = S Pt^T; Y: step 7)
//   D2 = Ut^T K + (-Z) K               (step 9 regrouped: Ut^T K - S Pt^T K = N - S M)
//   S <- G_C S + D2
//   y += Y / sqrt(Dk)                  (step 8, TMA reduction onto y_loc / sqrt(Dk))
// with S itself held in tensor memory as the 16-bit A operand of the first
// product (lane = value row) and -Z written back beside it as the A operand of
// the last, so per chunk the tensor cores run 8 + 2 C/16 products, only
// 8 + C/16 of them on the serial path, and no state operand passes through
// shared memory.
constexpr int kFusedThreads = kPrepThreads;  // 16 warps

// Shared memory of the scan: a ring of tile stages, each holding the tile's
// A1 rows ([Pt; Qh] per chunk, two 64-column halves of 128 rows), its K rows
// (two halves of 64 rows), its Ut rows (two halves of 64 rows), and the G_C of
// its chunks; and two y staging buffers (chunk parity), each C token rows of
// 128 bytes per 64-column half, the box layout of the y reduction.  A stage is
// free once its chunks' products are done and their G_C has been read.
struct ScanSmem {
  static constexpr uint32_t kOffA1 = 0;
  static constexpr uint32_t kOffK = 32768;
  static constexpr uint32_t kOffU = 49152;
  static constexpr uint32_t kStage = 65536;
  static constexpr int kStages = 3;
  static constexpr uint32_t kOffY = kStages * kStage;     // 2 buffers x 2 halves x 8 KB
  static constexpr uint32_t kOffGC = kOffY + 2 * 16384;  // fp32 x 4 per stage
  static constexpr uint32_t kTotal = kOffGC + kStages * 16 + 1024;
};
static_assert(ScanSmem::kTotal <= 232448, "scan shared memory");
constexpr uint32_t kFusedSmem = ScanSmem::kTotal > kPrepSmem ? ScanSmem::kTotal : kPrepSmem;

enum : int {
  kZFull = 0,                          // [stages] tile landed (TMA transaction count)
  kZEmpty = kZFull + ScanSmem::kStages,  // [stages] 8 state warps (G_C read) + MMA commit
  kZKNorm = kZEmpty + ScanSmem::kStages, // [stages] 4 aux warps: the tile's K rows normalised
  kZD1Full = kZKNorm + ScanSmem::kStages,  // [2] [Z | Y^T] of the chunk complete
  kZD1Free = kZD1Full + 2,             // [2] 8 state warps (Z read) + 4 aux warps (Y read)
  kZD2Full = kZD1Free + 2,             // Ut^T K + (-Z) K of the chunk complete
  kZSReady,                            // 8 state warps: S_j in tensor memory
  kZWReady,                            // 8 state warps: -Z of the chunk in tensor memory
  kZYGo,                               // y of chunk j may be staged (the next chunk's product is issued)
  kZDone,                              // the issuer's last products complete
  kZNumBars
};

// Tensor-memory loads of N (8, 16, 32 or 64) columns and 16-bit pair stores of
// N / 2 columns, chosen at compile time.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float* v) {
  if constexpr (N == 8) {
    tmem_ld8(taddr, v);
  } else if constexpr (N == 16) {
    tmem_ld16(taddr, v);
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 32) tmem_ld32(taddr + i, v + i);
  }
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t* r) {
  if constexpr (N == 4) {
    tmem_st4(taddr, r);
  } else if constexpr (N == 8) {
    tmem_st8(taddr, r);
  } else if constexpr (N == 16) {
    tmem_st16(taddr, r);
  } else {
    tmem_st32(taddr, r);
  }
}

// The scan of head bh (one CTA, 512 threads):
//   warp 0 lane 0   loads tile stages (after the tile's flag, in the fused launch)
//   warp 1 lane 0   issues every product
//   warps 2..9      state group: thread = (value row v, key half h) holds
//                   S[v][64h .. 64h+63] in fp32 registers; writes -Z, updates S
//                   and writes S back to tensor memory as the next A operand.
//   warps 10..13    aux group: stages y of chunk j while the product of chunk
//                   j+1 runs, normalises K tiles (option)
// Tensor memory: [Z | Y^T] double-buffered at columns 0 and 128 (2C columns
// each), D2 at 256 (128 columns), S (16-bit pairs) at 384 (64 columns), -Z
// (16-bit pairs) at 448 (C / 2 columns).
template <int C, typename E>
__device__ __forceinline__ void scan_role(const CUtensorMap* tm_a1c, const CUtensorMap* tm_k,
                                          const CUtensorMap* tm_uc, const CUtensorMap* tm_yred,
                                          const float* wsGC, const int* flags,
                                          const float* state_in, float* state_out, int T,
                                          int Hk, int Hv, int NT, int bh, int opts, float scale,
                                          uint8_t* smem_raw) {
  using SM = ScanSmem;
  constexpr int kCt = kTile / C;  // chunks per tile
  constexpr int kZc = C / 2;      // Z columns of each state thread
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~(uintptr_t)1023);
  __shared__ uint64_t zbars[kZNumBars];
  __shared__ uint32_t tmem_sh;
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = bh / Hv, hv = bh - b * Hv, hk = key_head(hv, Hk, Hv, opts);
  const int NC = (T + C - 1) / C;
  const bool knorm = (opts & kOptL2NormQK) != 0;
  auto bar = [&](int i) { return smem_u32(&zbars[i]); };

  if (tid == 0) {
    for (int s = 0; s < SM::kStages; ++s) {
      mbar_init(bar(kZFull + s), 1);
      mbar_init(bar(kZEmpty + s), 9);
      mbar_init(bar(kZKNorm + s), 4);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kZD1Full + x), 1);
      mbar_init(bar(kZD1Free + x), 12);
    }
    mbar_init(bar(kZD2Full), 1);
    mbar_init(bar(kZSReady), 8);
    mbar_init(bar(kZWReady), 8);
    mbar_init(bar(kZYGo), 1);
    mbar_init(bar(kZDone), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  auto tD1 = [&](int x) { return tmem + 128u * (uint32_t)x; };
  const uint32_t tD2 = tmem + 256, tS = tmem + 384, tW = tmem + 448;
  auto last_of_tile = [&](int j) { return (j % kCt) == kCt - 1 || j == NC - 1; };

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      prefetch_tmap(tm_a1c);
      prefetch_tmap(tm_k);
      prefetch_tmap(tm_uc);
      int n = 0;
      for (; n < NT; ++n) {
        const int s = n % SM::kStages;
        if (n >= SM::kStages && !mbar_wait(bar(kZEmpty + s), ((n / SM::kStages) - 1) & 1)) break;
        const size_t tile = (size_t)bh * NT + n;
        if (flags) {
          if (!wait_flag(flags + tile, kTilePublished)) break;
          fence_proxy_async_global();
        }
        const uint32_t fb = bar(kZFull + s), st = sbase + s * SM::kStage;
        mbar_expect_tx(fb, SM::kStage + 16);
        bulk_load(sbase + SM::kOffGC + 16 * s, wsGC + tile * 4, 16, fb);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tma_load_2d(st + SM::kOffA1 + h * 16384, tm_a1c, fb, 64 * h, (int)(tile * 128));
          tma_load_4d(st + SM::kOffK + h * 8192, tm_k, fb, 64 * h, hk, n * kTile, b);
          tma_load_2d(st + SM::kOffU + h * 8192, tm_uc, fb, 64 * h, (int)(tile * kTile));
        }
      }
      // The stages still in flight land before the CTA ends.
      for (int m = (n > SM::kStages ? n - SM::kStages : 0); m < n; ++m)
        mbar_wait(bar(kZFull + m % SM::kStages), (m / SM::kStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------- issuer -------------------------------
    // Per chunk: [Z | Y^T] = S [Pt; Qh]^T once S_j is in tensor memory;
    // D2 = Ut^T K right after it (D2 of the previous chunk has been read by
    // then); D2 += (-Z) K once -Z is in tensor memory.
    if (lane == 0) {
      const uint32_t id_z = idesc_e<E>(128, 2 * C, false, false);  // S (TMEM) x [Pt; Qh]^T
      const uint32_t id_n = idesc_e<E>(128, 128, true, true);      // Ut^T x K (both MN-major)
      const uint32_t id_w = idesc_e<E>(128, 128, false, true);     // (-Z) (TMEM) x K
      const SmemDesc d_a1 = smem_desc_base(sbase + SM::kOffA1, 16, 1024, kSw128);  // K-major rows
      const SmemDesc d_mn = smem_desc_base(sbase, 8192, 1024, kSw128);  // MN-major 64-col halves
      bool ok = true;
      // The next chunk's tile and [Z | Y^T] buffer, tested (not waited for)
      // while this chunk's -Z is being written, so that once S_j is ready the
      // product is issued without further checks on the serial path.
      bool next_tile_ready = false, next_buf_free = false;
      for (int j = 0; j < NC && ok; ++j) {
        const int c = j % kCt, n = j / kCt, st = n % SM::kStages;
        if (c == 0 && !next_tile_ready &&
            !(ok = mbar_wait_poll(bar(kZFull + st), (n / SM::kStages) & 1)))
          break;
        if (j >= 2 && !next_buf_free &&
            !(ok = mbar_wait_poll(bar(kZD1Free + (j & 1)), ((j >> 1) - 1) & 1)))
          break;
        if (!(ok = mbar_wait_poll(bar(kZSReady), j & 1))) break;
        tc_fence_after();
        const uint32_t aoff = st * SM::kStage + 2 * C * c * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16_ts(tD1(j & 1), tS + 8 * kk,
                     smem_desc_at(d_a1, aoff + (kk >> 2) * 16384 + (kk & 3) * 32), id_z, kk > 0);
        mma_commit(bar(kZD1Full + (j & 1)));
        if (j > 0) mbar_arrive(bar(kZYGo));  // y of chunk j-1 may be staged now
        if (knorm && c == 0 && !(ok = mbar_wait(bar(kZKNorm + st), (n / SM::kStages) & 1))) break;
        tc_fence_after();
        const uint32_t toff = st * SM::kStage + c * C * 128;  // token row c C of the tile
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)
          mma_f16_ss(tD2, smem_desc_at(d_mn, toff + SM::kOffU + kk * 2048),
                     smem_desc_at(d_mn, toff + SM::kOffK + kk * 2048), id_n, kk > 0);
        if (j + 1 < NC) {
          const int n1 = (j + 1) / kCt;
          next_tile_ready = ((j + 1) % kCt != 0) ||
                            mbar_test_wait(bar(kZFull + n1 % SM::kStages), (n1 / SM::kStages) & 1);
          next_buf_free = j + 1 < 2 ||
                          mbar_test_wait(bar(kZD1Free + ((j + 1) & 1)), (((j + 1) >> 1) - 1) & 1);
        }
        if (!(ok = mbar_wait_poll(bar(kZWReady), j & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)
          mma_f16_ts(tD2, tW + 8 * kk, smem_desc_at(d_mn, toff + SM::kOffK + kk * 2048), id_w, 1);
        mma_commit(bar(kZD2Full));
        if (last_of_tile(j)) mma_commit(bar(kZEmpty + st));
        if (j == NC - 1) mbar_arrive(bar(kZYGo));  // y of the last chunk
      }
      // Every product issued has completed before the tensor memory is freed.
      mma_commit(bar(kZDone));
      mbar_wait(bar(kZDone), 0);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 10) {
    // ---------------------------- state group -----------------------------
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int v = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    float* srow_out = state_out + ((size_t)bh * kD + v) * kD + 64 * h;
    float s[64];
    if (state_in) {
      const float4* src = reinterpret_cast<const float4*>(state_in + ((size_t)bh * kD + v) * kD +
                                                          64 * h);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 x = src[i];
        s[4 * i] = x.x;
        s[4 * i + 1] = x.y;
        s[4 * i + 2] = x.z;
        s[4 * i + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) s[i] = 0.f;
    }
    // S (16-bit pairs) into tensor memory, then one arrival per warp.
    auto write_s = [&]() {
      uint32_t p[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) p[i] = pack2<E>(s[2 * i], s[2 * i + 1]);
      tmem_st32(tS + lane_base + 32 * h, p);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kZSReady));
    };
    write_s();
    bool ok = true;
    for (int j = 0; j < NC; ++j) {
      const int c = j % kCt, n = j / kCt, st = n % SM::kStages;
      // -Z (tokens t = c C + h C/2 + i, i < C/2: this thread's columns) to
      // tensor memory as the A operand of D2 += (-Z) K.
      if (c == 0) ok = ok && mbar_wait(bar(kZFull + st), (n / SM::kStages) & 1);
      ok = ok && mbar_wait_poll(bar(kZD1Full + (j & 1)), (j >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      float z[kZc];
      tmem_ld_n<kZc>(tD1(j & 1) + lane_base + kZc * h, z);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kZD1Free + (j & 1)));
      uint32_t w[kZc / 2];
#pragma unroll
      for (int i = 0; i < kZc; i += 2) w[i / 2] = pack2<E>(z[i], z[i + 1]);
      tmem_st_n<kZc / 2>(tW + lane_base + (kZc / 2) * h, w);
      const float gcv = ld_shared_f32(sbase + SM::kOffGC + 16 * st + 4 * c);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kZWReady));
        if (last_of_tile(j)) mbar_arrive(bar(kZEmpty + st));  // done with the stage's G_C
      }
      // S <- G_C S + D2; S_{j+1} to tensor memory as the next A operand.
      ok = mbar_wait_poll(bar(kZD2Full), j & 1);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float d[32];
        tmem_ld32(tD2 + lane_base + 64 * h + 32 * hh, d);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < 32; ++r) s[32 * hh + r] = fmaf(gcv, s[32 * hh + r], d[r]);
      }
      if (j + 1 < NC) write_s();
    }
    if (ok) {
      float4* dst = reinterpret_cast<float4*>(srow_out);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        dst[i] = make_float4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
    }
  } else if (warp >= 10 && warp < 14) {
    // ------------------------------ aux group -----------------------------
    const int q = warp & 3;
    const bool reducer = warp == 10 && lane == 0;
    const int atid = tid - 320;  // 0..127
    bool ok = true;
    for (int j = 0; j < NC; ++j) {
      const int c = j % kCt, n = j / kCt, st = n % SM::kStages;
      // (Only the K normalisation reads the stage; its barrier keeps the stage
      // from being refilled before it is done.)
      if (knorm && c == 0) ok = ok && mbar_wait(bar(kZFull + st), (n / SM::kStages) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (ok && knorm && c == 0) {
        // The tile's K rows as x / |x| (two threads a row), before W K reads them.
        l2norm_row_sw128<E>(sm + st * SM::kStage + SM::kOffK, 8192, atid >> 1, atid & 1);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kZKNorm + st));
      }
      if (ok) ok = mbar_wait(bar(kZYGo), j & 1);
      if (ok) ok = mbar_wait(bar(kZD1Full + (j & 1)), (j >> 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      const uint32_t yoff = SM::kOffY + (j & 1) * 16384;  // this chunk's y staging
      if (ok) {
        tc_fence_after();
        // Y^T (lanes v, columns t; already / sqrt(Dk): Qh is stored scaled) in
        // 16 x 8 fragments: block (lh, cb) covers lanes 32q + 16 lh .. + 15 and
        // tokens 8 cb .. 8 cb + 7.
        constexpr int kCb = C / 8;
        float yv[2][kCb][4];
#pragma unroll
        for (int lh = 0; lh < 2; ++lh)
#pragma unroll
          for (int cb = 0; cb < kCb; ++cb)
            tmem_ld_16x256b(tD1(j & 1) + ((uint32_t)(32 * q + 16 * lh) << 16) + C + 8 * cb,
                            yv[lh][cb]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kZD1Free + (j & 1)));
        // Stored transposed into the y staging (C token rows of 128 bytes per
        // 64-column half): each 8 x 8 block becomes 8 token rows of 8
        // consecutive values (16 bytes).
        const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
        for (int lh = 0; lh < 2; ++lh) {
          const int v0 = 32 * q + 16 * lh + 8 * (mi & 1);
          const uint32_t hbase = sbase + yoff + (v0 >> 6) * 8192;
#pragma unroll
          for (int cb = 0; cb < kCb; cb += 2) {
            const int t = 8 * (cb + (mi >> 1)) + r8;
            const uint32_t addr = hbase + t * 128 + ((((v0 & 63) >> 3) ^ (t & 7)) << 4);
            stmatrix_x4_trans(addr, pack2<E>(yv[lh][cb][0], yv[lh][cb][1]),
                              pack2<E>(yv[lh][cb][2], yv[lh][cb][3]),
                              pack2<E>(yv[lh][cb + 1][0], yv[lh][cb + 1][1]),
                              pack2<E>(yv[lh][cb + 1][2], yv[lh][cb + 1][3]));
          }
        }
        fence_proxy_async();
      }
      // The previous chunk's reduction has read its buffer before any aux
      // thread passes this barrier, so the buffer it wrote this chunk's y into
      // (two chunks back) and the one of the next chunk are free.
      if (reducer) bulk_wait_read_all();
      ok = named_bar_and(3, 128, ok);
      if (!ok) break;
      if (reducer) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          tma_reduce_add_4d(tm_yred, sbase + yoff + hh * 8192, 64 * hh, hv, j * C, b);
        bulk_commit();
      }
      __syncwarp();
    }
    if (reducer) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int C, typename E>
__global__ void __launch_bounds__(kFusedThreads, 1)
fused_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_a1s,
                     const __grid_constant__ CUtensorMap tm_us,
                     const __grid_constant__ CUtensorMap tm_yred,
                     const __grid_constant__ CUtensorMap tm_a1o,
                     const __grid_constant__ CUtensorMap tm_uo,
                     const __grid_constant__ CUtensorMap tm_yo, const E* __restrict__ g,
                     const E* __restrict__ beta, float* __restrict__ wsGC, int* flags,
                     const float* state_in, float* state_out, int T, int Hk, int Hv, int NT,
                     int BH, int opts, float scale) {
  extern __shared__ uint8_t smem_raw[];
  if ((int)blockIdx.x < BH) {
    scan_role<C, E>(&tm_a1s, &tm_k, &tm_us, &tm_yred, wsGC, flags, state_in, state_out, T, Hk,
                    Hv, NT, blockIdx.x, opts, scale, smem_raw);
  } else {
    const PrepParams<E> P{&tm_k, &tm_q, &tm_v, &tm_a1o, &tm_uo, &tm_yo, g, beta, wsGC,
                          T, Hk, Hv, NT, BH, opts, scale};
    prep_role<C, E>(P, smem_raw, blockIdx.x - BH, gridDim.x - BH, flags);
  }
}

// The scan alone (after prep_tc_kernel in stream order): one CTA per head.
template <int C, typename E>
__global__ void __launch_bounds__(kFusedThreads, 1)
scan_head_kernel(const __grid_constant__ CUtensorMap tm_a1s, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_us,
                 const __grid_constant__ CUtensorMap tm_yred, const float* __restrict__ wsGC,
                 const float* state_in, float* state_out, int T, int Hk, int Hv, int NT,
                 int opts, float scale) {
  extern __shared__ uint8_t smem_raw[];
  scan_role<C, E>(&tm_a1s, &tm_k, &tm_us, &tm_yred, wsGC, nullptr, state_in, state_out, T, Hk,
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

// [B, T, H, 128] 16-bit elements of type dt -> box {64 cols, 1 head, 64
// tokens, 1 batch}, 128B swizzle.
bool make_bthd_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int B, int T, int H, int box_t = kTile) {
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2,
                                 (cuuint64_t)T * H * kD * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_t, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, dt, 4, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [rows, 128] 2-D view of a workspace region of 16-bit elements.  Swizzled
// boxes use the swizzle whose span equals the box row (box_cols * 2 bytes: 32,
// 64 or 128).
bool make_rows_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, size_t rows, int box_cols, int box_rows,
                   bool swizzle) {
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle)
    sw = box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                        : (box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  return encode_fn()(m, dt, 2, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// Rows of 128 16-bit values seen as [rows][2 halves][64] (3-D), box {64, 2,
// box_rows}: the box lands in shared memory as [row][half] 128-byte units.
bool make_rows_halves_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, size_t rows, int box_rows) {
  const cuuint64_t dims[3] = {64, 2, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {128, (cuuint64_t)kD * 2};
  const cuuint32_t box[3] = {64, 2, (cuuint32_t)box_rows};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, dt, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [B, T, H, 128] 16-bit elements seen as [B][T][H][2][64] (5-D), box {64, 2,
// 1, 64, 1}.
bool make_bthd_halves_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int B, int T, int H) {
  const cuuint64_t dims[5] = {64, 2, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[4] = {128, (cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2,
                                 (cuuint64_t)T * H * kD * 2};
  const cuuint32_t box[5] = {64, 2, 1, (cuuint32_t)kTile, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return encode_fn()(m, dt, 5, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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

template <int C, typename E>
cudaError_t launch_c(const PrefillArgs& a) {
  const int NT = (a.T + kTile - 1) / kTile;
  const int BH = a.B * a.Hv;
  const WsLayout w = ws_layout(BH, NT);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  E* wsA1 = reinterpret_cast<E*>(ws + w.a1);
  E* wsU = reinterpret_cast<E*>(ws + w.u);
  float* wsGC = reinterpret_cast<float*>(ws + w.gc);

  if (!encode_fn()) return cudaErrorNotSupported;
  CUtensorMap tk, tq, tv, ta1s, tus, tyred, ta1o, tuo, tyo;
  const CUtensorMapDataType dt = ElemT<E>::kTmap;
  if (!make_bthd_map(&tk, dt, a.k, a.B, a.T, a.Hk) ||
      !make_bthd_map(&tq, dt, a.q, a.B, a.T, a.Hk) ||
      !make_bthd_map(&tv, dt, a.v, a.B, a.T, a.Hv) ||
      !make_rows_map(&ta1s, dt, wsA1, (size_t)BH * NT * 128, 64, 128, true) ||
      !make_rows_map(&tus, dt, wsU, (size_t)BH * NT * kTile, 64, 64, true) ||
      !make_bthd_map(&tyred, dt, a.y, a.B, a.T, a.Hv, C) ||
      !make_rows_halves_map(&ta1o, dt, wsA1, (size_t)BH * NT * 128, 128) ||
      !make_rows_halves_map(&tuo, dt, wsU, (size_t)BH * NT * kTile, kTile) ||
      !make_bthd_halves_map(&tyo, dt, a.y, a.B, a.T, a.Hv))
    return cudaErrorInvalidValue;

  const float scale = 1.0f / sqrtf((float)kD);
  const int sms = num_sms();
  const E* g = static_cast<const E*>(a.g);
  const E* beta = static_cast<const E*>(a.beta);
  cudaError_t e;
  // Fused path: one scan CTA per head next to at least two thirds of the SMs
  // doing prep, in one cooperative launch.
  if (3 * BH <= sms) {
    int* flags = reinterpret_cast<int*>(ws + w.flags);
    e = cudaFuncSetAttribute(fused_prefill_kernel<C, E>,
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
    return cudaLaunchKernelEx(&cfg, fused_prefill_kernel<C, E>, tk, tq, tv, ta1s, tus, tyred, ta1o,
                              tuo, tyo, g, beta, wsGC, flags, a.state_in, a.state_out,
                              a.T, a.Hk, a.Hv, NT, BH, a.options, scale);
  }

  // Split path: the persistent prep kernel on every SM, then one scan CTA per head.
  e = cudaFuncSetAttribute(prep_tc_kernel<C, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kPrepSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(scan_head_kernel<C, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ScanSmem::kTotal);
  if (e != cudaSuccess) return e;
  const int prep_ctas = std::min(sms, (BH * NT + kPrepGroups - 1) / kPrepGroups);
  prep_tc_kernel<C, E><<<prep_ctas, kPrepThreads, kPrepSmem, a.stream>>>(
      tk, tq, tv, ta1o, tuo, tyo, g, beta, wsGC, a.T, a.Hk, a.Hv, NT, BH, a.options, scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scan_head_kernel<C, E><<<BH, kFusedThreads, ScanSmem::kTotal, a.stream>>>(
      ta1s, tk, tus, tyred, wsGC, a.state_in, a.state_out, a.T, a.Hk, a.Hv, NT, a.options,
      scale);
  return cudaGetLastError();
}

template <typename E>
cudaError_t launch_e(const PrefillArgs& a) {
  switch (a.chunk) {
    case 16: return launch_c<16, E>(a);
    case 32: return launch_c<32, E>(a);
    default: return launch_c<64, E>(a);
  }
}

}  // namespace

size_t prefill_tc_workspace_bytes(int B, int T, int Hv) {
  return ws_layout(B * Hv, (T + kTile - 1) / kTile).total;
}

// dtype 1 bf16, 2 fp16 (the GDN_DTYPE_* codes).
cudaError_t launch_prefill_tc(const PrefillArgs& a) {
  return a.dtype == 2 ? launch_e<__half>(a) : launch_e<bf16>(a);
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
