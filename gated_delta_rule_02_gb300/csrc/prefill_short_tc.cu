// Short-T prefill on the tensor cores: bf16 or fp16 inputs, Dk = Dv = 128,
// T <= 32.
//
// The whole sequence of a head is one chunk of TC = 16 or 32 tokens (tokens
// past T padded with g = 1, beta = 0, q = k = v = 0; metaltile-std
// `gated_delta_wy.rs`, "Algorithm" steps 1-9, and the chunk-loop precondition
// on padding), computed with the same chunk algebra as the chunked prefill
// (ferrox-core `gdn_chunk.rs`, "The algebra"):
//   KK^T, QK^T;  G_t, Gam[t][j] = 2^(lam_t - lam_j) (chunk-local log2 prefix sums)
//   T_L = (I + L)^-1, L[t][j] = beta_j KK^T[t][j] (j < t), blockwise in fp32;
//   T_A = diag(beta)(Gam . T_L)
//   -Pt = -diag(G_C beta) T_L K;  Qh = (G Q - diag(G) M T_L K) / sqrt(Dk),
//   M[t][i] = beta_i QK^T[t][i] (i <= t);  Ut = diag(Gam_end) T_A V;
//   y_loc = (Gam . QK^T) T_A V / sqrt(Dk)
//   [-Z | Y] = S [-Pt; Qh]^T;  W = Ut^T - Z;  S <- G_C S + W K;  y = Y + y_loc.
// Warp w of a CTA of eight holds value rows 16w .. 16w + 15 of S in fp32
// registers in the layout of an m16n8 MMA accumulator, which is also (two
// tiles at a time, packed to 16 bits) the layout of an m16k16 A operand: S
// feeds the warp-level MMAs straight from its registers, and W K accumulates
// into them.  Each state is read once and written once.
//
// The kernel is persistent, two CTAs an SM, each looping over heads, with the
// data of the next head in flight while one is computed: its tokens as TMA
// boxes into the other half of a double buffer (rows past T are out of the
// tensor and arrive as zeros), its gates in registers, and, once the current
// state has been read into registers, its state as one 64 KB TMA box.  The new
// state leaves from registers by streaming stores.
#include <type_traits>

#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"
#include "warp_mma.cuh"

namespace gdn {
namespace {
using namespace wm;

constexpr int kD = 128;
constexpr int kThr = 256;
constexpr int kRS = 136;  // 16-bit row stride (elements) of the row arrays (272 B)
constexpr int kCS = 40;   // 16-bit row stride of the TC x TC coefficient arrays (80 B)
constexpr int kFS = 33;   // fp32 row stride of the TC x TC fp32 arrays
constexpr int kSmemAlign = 1024;  // the swizzled boxes' alignment

// Every 16-bit array is in the input type E (bf16 or fp16); TC token rows.
template <typename E, int TC>
struct ShortTcSmem {
  // The state of a head, one TMA box, as [group cb of 32 columns][row v][32],
  // the 16-byte chunks c of row v stored at c ^ (v & 7) (the TMA unit's
  // 128-byte swizzle), so that the reads of eight rows at once in the
  // accumulator layout meet every bank twice, the least possible.
  float st[kD * kD];
  // Tokens, double-buffered: [buffer][k, q, v], each one TMA box landing as
  // two halves of TC rows x 64 columns, 128-byte swizzled (see tok_off).
  E tok[2][3][2 * TC * 64];
  E ys[TC][kRS];  // y staging [t][v]
  union {
    struct {
      float lm[TC][kFS], qk[TC][kFS];  // L = KK^T diag(beta), QK^T (then scratch)
      float tlf[TC][kFS];              // T_L in fp32
      E a3t[TC][kCS], a3b[TC][kCS];    // diag(G) M, Gam . QK^T
      E tlb[TC][kCS], tab[TC][kCS];    // T_L, T_A
    } a;                               // until W_M, W_Y are formed
    struct {
      E p[TC][kRS];   // -Pt
      E qh[TC][kRS];  // Qh / sqrt(Dk)
    } b;                                // from then on
  } u;
  E cp[TC][kCS], cu[TC][kCS];  // -diag(G_C beta) T_L, diag(Gam_end) T_A
  E wm[TC][kCS], wy[TC][kCS];  // -W_M / sqrt(Dk), W_Y / sqrt(Dk)
  float lam[TC], gt[TC], bt[TC], gend[TC];
  float gc;
  alignas(8) uint64_t bar_st;      // the state's box landed
  alignas(8) uint64_t bar_tok[2];  // a token buffer's boxes landed
};

// fp32 element (row r, column c) of the swizzled state boxes.
__device__ __forceinline__ int st_index(int r, int c) {
  return (c >> 5) * (kD * 32) + 32 * r + ((((c & 31) >> 2) ^ (r & 7)) << 2) + (c & 3);
}
// Byte offset of element (t, c) in a token array: box c / 64, row t of 128
// bytes, 16-byte chunk (c % 64) / 8 stored at chunk ^ (t % 8).
template <int TC>
__device__ __forceinline__ uint32_t tok_off(int t, int c) {
  return (c >> 6) * (TC * 128) + t * 128 + ((((c & 63) >> 3) ^ (t & 7)) << 4) + ((c & 7) << 1);
}
// TMA tensor loads into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
// ldmatrix lane addresses in a token array at shared address `base`: A (m16 x
// k16) from rows r0.., columns c0..; B (k16 x n8) from rows n0.. (the n
// index), columns k0..; B from rows k0.., columns n0.., transposing; A of the
// transpose from rows k0.., columns m0.., transposing.
template <int TC>
__device__ __forceinline__ uint32_t tok_a(uint32_t base, int r0, int c0, int lane) {
  return base + tok_off<TC>(r0 + (lane & 15), c0 + 8 * (lane >> 4));
}
template <int TC>
__device__ __forceinline__ uint32_t tok_bnk(uint32_t base, int n0, int k0, int lane) {
  return base + tok_off<TC>(n0 + (lane & 7), k0 + 8 * ((lane >> 3) & 1));
}
template <int TC>
__device__ __forceinline__ uint32_t tok_bkn(uint32_t base, int k0, int n0, int lane) {
  return base + tok_off<TC>(k0 + (lane & 15), n0);
}
template <int TC>
__device__ __forceinline__ uint32_t tok_at(uint32_t base, int k0, int m0, int lane) {
  return base + tok_off<TC>(k0 + (lane & 7) + 8 * (lane >> 4), m0 + 8 * ((lane >> 3) & 1));
}

template <typename E, int TC>
__global__ void __launch_bounds__(kThr, 2)
short_tc_kernel(const __grid_constant__ CUtensorMap tm_state,
                const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_v, const E* __restrict__ g,
                const E* __restrict__ beta, const float* state_in, float* state_out,
                E* __restrict__ y, int T, int Hk, int Hv, int nheads, int opts, float scale) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem_base =
      smem_raw + ((kSmemAlign - (s_u32(smem_raw) & (kSmemAlign - 1))) & (kSmemAlign - 1));
  ShortTcSmem<E, TC>& sm = *reinterpret_cast<ShortTcSmem<E, TC>*>(smem_base);
  auto& lm = sm.u.a.lm;
  auto& qk = sm.u.a.qk;
  auto& tlf = sm.u.a.tlf;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;
  constexpr int NT8 = TC / 8;    // n8 tiles over the chunk's tokens
  constexpr int NK16 = TC / 16;  // k16 steps over the chunk's tokens
  const int G = gridDim.x;
  const uint32_t bar_st = s_u32(&sm.bar_st);

  // TMA issue by one thread: the state of head h (one 64 KB box) and the
  // tokens of head h into buffer j (k, q, v: one box each).
  auto load_state = [&](int h) {
    ptx::mbar_expect_tx(bar_st, kD * kD * sizeof(float));
    tma_load_3d(s_u32(sm.st), &tm_state, bar_st, 0, h * kD, 0);
  };
  // Array a (0 k, 1 q, 2 v) of head h's tokens into buffer j; the buffer's
  // barrier expects all three (the k call arms it, before any can land).
  auto load_tokens = [&](int h, int j, int a) {
    const int bj = h / Hv, hvj = h - bj * Hv, hkj = key_head(hvj, Hk, Hv, opts);
    const uint32_t bar = s_u32(&sm.bar_tok[j]);
    const CUtensorMap* m = a == 0 ? &tm_k : (a == 1 ? &tm_q : &tm_v);
    tma_load_5d(s_u32(&sm.tok[j][a][0]), m, bar, 0, 0, 0, a == 2 ? hvj : hkj, bj);
  };
  // The raw gates of head h, lane t of warp 1 token t (widened where used, so
  // that nothing waits for these loads before then).
  auto load_gates = [&](int h, E& gr, E& br) {
    if (lane < T) {
      const int bj = h / Hv, hvj = h - bj * Hv;
      const size_t gi = ((size_t)bj * T + lane) * Hv + hvj;
      gr = g[gi];
      br = beta[gi];
    }
  };

  if (tid == 0) {
    if (state_in) ptx::prefetch_tmap(&tm_state);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_v);
    ptx::mbar_init(bar_st, 1);
    ptx::mbar_init(s_u32(&sm.bar_tok[0]), 1);
    ptx::mbar_init(s_u32(&sm.bar_tok[1]), 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (blockIdx.x >= nheads) return;
  if (tid == 0) {
    ptx::mbar_expect_tx(s_u32(&sm.bar_tok[0]), 6 * TC * 128);
    for (int a = 0; a < 3; ++a) load_tokens(blockIdx.x, 0, a);
    if (state_in) load_state(blockIdx.x);
  }
  E gr = from_f32<E>(1.f), br = from_f32<E>(0.f);
  if (warp == 1) load_gates(blockIdx.x, gr, br);

  // Heads h = blockIdx.x, + G, ...; iteration `it` computes from token buffer
  // it & 1 (its n-th use completes phase n of that buffer's barrier) and from
  // the state box of phase `it`.  The loads for the next head are issued in
  // the middle of the iteration by threads that would otherwise wait.
  int it = 0;
  for (int h = blockIdx.x; h < nheads; h += G, ++it) {
    const int b = h / Hv, hv = h - b * Hv;
    const int jb = it & 1;
    const bool has_next = h + G < nheads;
    E gr_next = gr, br_next = br;
    const uint32_t tk = s_u32(&sm.tok[jb][0][0]), tq = s_u32(&sm.tok[jb][1][0]),
                   tv = s_u32(&sm.tok[jb][2][0]);

    if (warp == 1) {
      // Gates: chunk-local prefix sums of log2 of the decay (padded tokens: 1).
      const float gv = to_f32(gr), bv = to_f32(br);
      float l = lane < T ? ((opts & kOptLogGate) ? gv * 1.4426950408889634f : log2f(gv)) : 0.f;
      l = fmaxf(l, -1000.f);
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, l, off);
        if (lane >= off) l += u;
      }
      const float lend = __shfl_sync(0xffffffffu, l, TC - 1);
      if (lane < TC) {
        sm.lam[lane] = l;
        sm.gt[lane] = exp2f(l);
        sm.bt[lane] = lane < T ? bv : 0.f;
        sm.gend[lane] = exp2f(lend - l);
      }
      if (lane == 0) sm.gc = exp2f(lend);
    }
    // The state into registers: S rows 16w + gq and 16w + gq + 8, columns 8j
    // + 2cq, +1 (j < 16), the accumulator layout of sixteen m16n8 tiles.  A
    // TMA load that never lands (2 s) is recorded in the device error word
    // and the kernel ends (heads not yet written stay unwritten).
    bool ok = ptx::mbar_wait(s_u32(&sm.bar_tok[jb]), (it >> 1) & 1);
    if (state_in) ok = ptx::mbar_wait(bar_st, it & 1) && ok;
    const int r0 = 16 * warp + gq;
    float s[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float2 lo = make_float2(0.f, 0.f), hi = lo;
      if (state_in) {
        lo = *reinterpret_cast<const float2*>(&sm.st[st_index(r0, 8 * j + 2 * cq)]);
        hi = *reinterpret_cast<const float2*>(&sm.st[st_index(r0 + 8, 8 * j + 2 * cq)]);
      }
      s[j][0] = lo.x;
      s[j][1] = lo.y;
      s[j][2] = hi.x;
      s[j][3] = hi.y;
    }
    if (!__syncthreads_and(ok)) return;
    if (opts & kOptL2NormQK) {
      // Every k and q row as x / |x|: a warp a row, four values a lane.
      for (int r = warp; r < 2 * TC; r += kThr / 32) {
        E* row = reinterpret_cast<E*>(
            reinterpret_cast<uint8_t*>(r < TC ? &sm.tok[jb][0][0] : &sm.tok[jb][1][0]) +
            tok_off<TC>(r < TC ? r : r - TC, 4 * lane));
        float x[4], ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[e] = to_f32(row[e]);
          ss = fmaf(x[e], x[e], ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float f = inv_norm(ss);
#pragma unroll
        for (int e = 0; e < 4; ++e) row[e] = from_f32<E>(x[e] * f);
      }
      ptx::fence_proxy_async();  // these writes before the buffer's next TMA fill
      __syncthreads();
    }

    // L = KK^T diag(beta) and QK^T (fp32): tiles (matrix, m16 tile, n8 tile),
    // K = Dk.
    for (int ti = warp; ti < 2 * NK16 * NT8; ti += kThr / 32) {
      const int mat = ti / (NK16 * NT8), rem = ti - mat * NK16 * NT8;
      const int mt = rem / NT8, nt = rem - mt * NT8;
      const uint32_t A = mat ? tq : tk;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        uint32_t a[4], bb[2];
        ldsm4(tok_a<TC>(A, 16 * mt, 16 * kk, lane), a);
        ldsm2(tok_bnk<TC>(tk, 8 * nt, 16 * kk, lane), bb);
        mma<E>(acc, a, bb);
      }
      float(*o)[kFS] = mat ? qk : lm;
      const int c0 = 8 * nt + 2 * cq;
      const float b0 = mat ? 1.f : sm.bt[c0], b1 = mat ? 1.f : sm.bt[c0 + 1];
      o[16 * mt + gq][c0] = acc[0] * b0;
      o[16 * mt + gq][c0 + 1] = acc[1] * b1;
      o[16 * mt + gq + 8][c0] = acc[2] * b0;
      o[16 * mt + gq + 8][c0 + 1] = acc[3] * b1;
    }
    __syncthreads();

    // T_L = (I + L)^-1 by blocks: the diagonal 8 x 8 blocks by forward
    // substitution, lane l column l % 8 of block l / 8; then, doubling the
    // block size b, every lower-left block of a 2b x 2b diagonal block from
    //   T21 = -T22 (L21 T11).
    if (warp == 0) {
      inverse_diag_blocks<TC, kFS>(lm, tlf, lane);
    } else {
      // The next head's loads (sm.st is free: every warp has read its rows),
      // then A3: diag(G) M and Gam . QK^T, masked to j <= t.
      if (has_next) {
        if (tid == kThr - 32) {
          ptx::mbar_expect_tx(s_u32(&sm.bar_tok[jb ^ 1]), 6 * TC * 128);
          load_tokens(h + G, jb ^ 1, 0);
        }
        if (tid == kThr - 64 && state_in) load_state(h + G);
        if (tid == kThr - 96) load_tokens(h + G, jb ^ 1, 1);
        if (tid == kThr - 128) load_tokens(h + G, jb ^ 1, 2);
        if (warp == 1) load_gates(h + G, gr_next, br_next);
      }
      for (int e = tid - 32; e < TC * TC; e += kThr - 32) {
        const int t = e / TC, j = e - t * TC;
        const bool keep = j <= t;
        const float qkv = qk[t][j];
        sm.u.a.a3t[t][j] = from_f32<E>(keep ? sm.gt[t] * sm.bt[j] * qkv : 0.f);
        sm.u.a.a3b[t][j] = from_f32<E>(keep ? exp2f(sm.lam[t] - sm.lam[j]) * qkv : 0.f);
      }
    }
    __syncthreads();
    combine_blocks<8, TC, kThr, kFS>(lm, tlf, qk, tid);
    if constexpr (TC == 32) combine_blocks<16, TC, kThr, kFS>(lm, tlf, qk, tid);
    // T_L, T_A = diag(beta)(Gam . T_L), cP = -diag(G_C beta) T_L and
    // cU = diag(Gam_end) T_A in 16 bits (zero above the diagonal).
    for (int e = tid; e < TC * TC; e += kThr) {
      const int r = e / TC, jj = e - r * TC;
      const bool low = r >= jj;
      const float tl = low ? tlf[r][jj] : 0.f;
      const float ta = low ? sm.bt[r] * exp2f(sm.lam[r] - sm.lam[jj]) * tl : 0.f;
      sm.u.a.tlb[r][jj] = from_f32<E>(tl);
      sm.u.a.tab[r][jj] = from_f32<E>(ta);
      sm.cp[r][jj] = from_f32<E>(-sm.gc * sm.bt[r] * tl);
      sm.cu[r][jj] = from_f32<E>(sm.gend[r] * ta);
    }
    __syncthreads();

    // W_M = A3t T_L and W_Y = A3b T_A, K = TC; stored as -W_M / sqrt(Dk) and
    // W_Y / sqrt(Dk).
    for (int ti = warp; ti < 2 * NK16 * NT8; ti += kThr / 32) {
      const int mat = ti / (NK16 * NT8), rem = ti - mat * NK16 * NT8;
      const int mt = rem / NT8, nt = rem - mt * NT8;
      const E* A = mat ? &sm.u.a.a3b[0][0] : &sm.u.a.a3t[0][0];
      const E* Bm = mat ? &sm.u.a.tab[0][0] : &sm.u.a.tlb[0][0];
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < NK16; ++kk) {
        uint32_t a[4], bb[2];
        ldsm4(a_addr(A, kCS, 16 * mt, 16 * kk, lane), a);
        ldsm2t(bkn_addr(Bm, kCS, 16 * kk, 8 * nt, lane), bb);
        mma<E>(acc, a, bb);
      }
      const float f = mat ? scale : -scale;
      E(*o)[kCS] = mat ? sm.wy : sm.wm;
      *reinterpret_cast<uint32_t*>(&o[16 * mt + gq][8 * nt + 2 * cq]) =
          pk<E>(f * acc[0], f * acc[1]);
      *reinterpret_cast<uint32_t*>(&o[16 * mt + gq + 8][8 * nt + 2 * cq]) =
          pk<E>(f * acc[2], f * acc[3]);
    }
    __syncthreads();

    // -Pt = cP K and Qh = (G Q - W_M K) / sqrt(Dk): M = TC, N = Dk, K = TC.
    for (int ti = warp; ti < 2 * NK16 * (kD / 8); ti += kThr / 32) {
      const int mat = ti / (NK16 * (kD / 8)), rem = ti - mat * NK16 * (kD / 8);
      const int mt = rem / (kD / 8), nt = rem - mt * (kD / 8);
      const E* A = mat ? &sm.wm[0][0] : &sm.cp[0][0];
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < NK16; ++kk) {
        uint32_t a[4], bb[2];
        ldsm4(a_addr(A, kCS, 16 * mt, 16 * kk, lane), a);
        ldsm2t(tok_bkn<TC>(tk, 16 * kk, 8 * nt, lane), bb);
        mma<E>(acc, a, bb);
      }
      const int t0 = 16 * mt + gq, c0 = 8 * nt + 2 * cq;
      if (mat) {
        const uint8_t* qb = reinterpret_cast<const uint8_t*>(&sm.tok[jb][1][0]);
        const E* q0 = reinterpret_cast<const E*>(qb + tok_off<TC>(t0, c0));
        const E* q1 = reinterpret_cast<const E*>(qb + tok_off<TC>(t0 + 8, c0));
        const float g0 = sm.gt[t0] * scale, g1 = sm.gt[t0 + 8] * scale;
        acc[0] = fmaf(g0, to_f32(q0[0]), acc[0]);
        acc[1] = fmaf(g0, to_f32(q0[1]), acc[1]);
        acc[2] = fmaf(g1, to_f32(q1[0]), acc[2]);
        acc[3] = fmaf(g1, to_f32(q1[1]), acc[3]);
      }
      E(*o)[kRS] = mat ? sm.u.b.qh : sm.u.b.p;
      *reinterpret_cast<uint32_t*>(&o[t0][c0]) = pk<E>(acc[0], acc[1]);
      *reinterpret_cast<uint32_t*>(&o[t0 + 8][c0]) = pk<E>(acc[2], acc[3]);
    }
    __syncthreads();

    // ---- the state step, warp w on value rows 16w .. 16w + 15 ----
    // [-Z | Y] = S [-Pt; Qh]^T (A: S from registers, two accumulator tiles per
    // k16 step; B: the rows of -Pt and Qh).
    float zy[2 * NT8][4];
#pragma unroll
    for (int n = 0; n < 2 * NT8; ++n) zy[n][0] = zy[n][1] = zy[n][2] = zy[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      const uint32_t a[4] = {pk<E>(s[2 * kk][0], s[2 * kk][1]), pk<E>(s[2 * kk][2], s[2 * kk][3]),
                             pk<E>(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                             pk<E>(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
      for (int n = 0; n < 2 * NT8; ++n) {
        uint32_t bb[2];
        const E* Bm = n < NT8 ? &sm.u.b.p[0][0] : &sm.u.b.qh[0][0];
        ldsm2(bnk_addr(Bm, kRS, 8 * (n % NT8), 16 * kk, lane), bb);
        mma<E>(zy[n], a, bb);
      }
    }
    // Ut^T = V^T cU^T and y_loc^T = V^T W_Y^T (A: V^T rows of this warp; B: the
    // rows of cU and W_Y), then W = Ut^T - Z and y = Y + y_loc.
    float ut[NT8][4], yl[NT8][4];
#pragma unroll
    for (int n = 0; n < NT8; ++n) {
      ut[n][0] = ut[n][1] = ut[n][2] = ut[n][3] = 0.f;
      yl[n][0] = yl[n][1] = yl[n][2] = yl[n][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < NK16; ++kk) {
      uint32_t a[4];
      ldsm4t(tok_at<TC>(tv, 16 * kk, 16 * warp, lane), a);
#pragma unroll
      for (int n = 0; n < NT8; ++n) {
        uint32_t bu[2], bw[2];
        ldsm2(bnk_addr(&sm.cu[0][0], kCS, 8 * n, 16 * kk, lane), bu);
        ldsm2(bnk_addr(&sm.wy[0][0], kCS, 8 * n, 16 * kk, lane), bw);
        mma<E>(ut[n], a, bu);
        mma<E>(yl[n], a, bw);
      }
    }
    // y (rows v, columns t) staged transposed as [t][v] for the store.
    {
      const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int n = 0; n < NT8; n += 2) {
        const int t = 8 * (n + (mi >> 1)) + r8, vv = 16 * warp + 8 * (mi & 1);
        stsm4t(s_u32(&sm.ys[t][vv]), pk<E>(zy[NT8 + n][0] + yl[n][0], zy[NT8 + n][1] + yl[n][1]),
               pk<E>(zy[NT8 + n][2] + yl[n][2], zy[NT8 + n][3] + yl[n][3]),
               pk<E>(zy[NT8 + n + 1][0] + yl[n + 1][0], zy[NT8 + n + 1][1] + yl[n + 1][1]),
               pk<E>(zy[NT8 + n + 1][2] + yl[n + 1][2], zy[NT8 + n + 1][3] + yl[n + 1][3]));
      }
    }
    // S <- G_C S + W K, W = Ut^T + (-Z) (A: W from registers; B: the rows of K).
    {
      const float gcv = sm.gc;
#pragma unroll
      for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[j][e] *= gcv;
#pragma unroll
      for (int kk = 0; kk < NK16; ++kk) {
        const uint32_t a[4] = {pk<E>(ut[2 * kk][0] + zy[2 * kk][0], ut[2 * kk][1] + zy[2 * kk][1]),
                               pk<E>(ut[2 * kk][2] + zy[2 * kk][2], ut[2 * kk][3] + zy[2 * kk][3]),
                               pk<E>(ut[2 * kk + 1][0] + zy[2 * kk + 1][0],
                                  ut[2 * kk + 1][1] + zy[2 * kk + 1][1]),
                               pk<E>(ut[2 * kk + 1][2] + zy[2 * kk + 1][2],
                                  ut[2 * kk + 1][3] + zy[2 * kk + 1][3])};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint32_t bb[2];
          ldsm2t(tok_bkn<TC>(tk, 16 * kk, 8 * j, lane), bb);
          mma<E>(s[j], a, bb);
        }
      }
    }
    // The new state (streaming stores) and y.
    {
      float* dst = state_out + (size_t)h * kD * kD;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        __stcs(reinterpret_cast<float2*>(dst + r0 * kD + 8 * j + 2 * cq),
               make_float2(s[j][0], s[j][1]));
        __stcs(reinterpret_cast<float2*>(dst + (r0 + 8) * kD + 8 * j + 2 * cq),
               make_float2(s[j][2], s[j][3]));
      }
    }
    __syncthreads();
    for (int i = tid; i < T * 16; i += kThr) {
      const int t = i >> 4, c8 = (i & 15) * 8;
      *reinterpret_cast<uint4*>(y + (((size_t)b * T + t) * Hv + hv) * kD + c8) =
          *reinterpret_cast<const uint4*>(&sm.ys[t][c8]);
    }
    gr = gr_next;
    br = br_next;
    __syncthreads();  // this head's tokens, coefficients and ys are used up
  }
}

// The fp32 states [nheads * 128 rows][128] seen as {32 columns, rows, 4
// column groups} (the groups 128 bytes apart), box {32, 128, 4}: one head,
// landing as [group][row][32], 128-byte swizzle.
bool make_state_map(CUtensorMap* m, const float* base, int nheads) {
  const TmapEncodeFn enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {32, (cuuint64_t)nheads * kD, 4};
  const cuuint64_t strides[2] = {kD * sizeof(float), 32 * sizeof(float)};
  const cuuint32_t box[3] = {32, kD, 4};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && c > 0)
      n = c;
    else
      return 1;
  }
  return n;
}

// Tokens [B, T, H, 128] of 16-bit type dt seen as {64 columns, T, 2 column
// halves, H, B}, box {64, TC, 2, 1, 1}: one head's tokens, landing as
// [half][token][64], 128-byte swizzle; tokens past T read as zeros.
bool make_token_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int B, int T, int H,
                    int tc) {
  const TmapEncodeFn enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t dims[5] = {64, (cuuint64_t)T, 2, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[4] = {(cuuint64_t)H * kD * 2, 128, (cuuint64_t)kD * 2,
                                 (cuuint64_t)T * H * kD * 2};
  const cuuint32_t box[5] = {64, (cuuint32_t)tc, 2, 1, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, dt, 5, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename E, int TC>
cudaError_t launch_tc(const PrefillArgs& a) {
  const int smem = (int)sizeof(ShortTcSmem<E, TC>) + kSmemAlign;
  cudaError_t e = cudaFuncSetAttribute(short_tc_kernel<E, TC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // As many CTAs as fit at once (two an SM at TC = 16), each looping over heads.
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, short_tc_kernel<E, TC>, kThr, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int nheads = a.B * a.Hv;
  const int grid = nheads < per_sm * sm_count() ? nheads : per_sm * sm_count();
  constexpr CUtensorMapDataType dt = std::is_same_v<E, __half> ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tm_s{}, tm_k{}, tm_q{}, tm_v{};
  if (a.state_in && !make_state_map(&tm_s, a.state_in, nheads)) return cudaErrorInvalidValue;
  if (!make_token_map(&tm_k, dt, a.k, a.B, a.T, a.Hk, TC) ||
      !make_token_map(&tm_q, dt, a.q, a.B, a.T, a.Hk, TC) ||
      !make_token_map(&tm_v, dt, a.v, a.B, a.T, a.Hv, TC))
    return cudaErrorInvalidValue;
  short_tc_kernel<E, TC><<<grid, kThr, smem, a.stream>>>(
      tm_s, tm_k, tm_q, tm_v, static_cast<const E*>(a.g), static_cast<const E*>(a.beta),
      a.state_in, a.state_out, static_cast<E*>(a.y), a.T, a.Hk, a.Hv, nheads, a.options,
      1.0f / sqrtf((float)kD));
  return cudaGetLastError();
}
template <typename E>
cudaError_t launch_tc_t(const PrefillArgs& a) {
  return a.T <= 16 ? launch_tc<E, 16>(a) : launch_tc<E, 32>(a);
}

}  // namespace

bool short_tc_applies(const PrefillArgs& a) {
  return (a.dtype == 1 || a.dtype == 2) && a.Dk == kD && a.Dv == kD && a.T <= 32;
}

cudaError_t launch_prefill_short_tc(const PrefillArgs& a) {
  return a.dtype == 2 ? launch_tc_t<__half>(a) : launch_tc_t<__nv_bfloat16>(a);
}

int short_tc_device_error(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, ptx::g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int z = 0;
    if (cudaMemcpyToSymbol(ptx::g_device_error, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace gdn
