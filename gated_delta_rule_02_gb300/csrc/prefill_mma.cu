// Chunked prefill on warp-level tensor-core MMAs for head size 64 (Dk = Dv =
// 64), bf16 or fp16 inputs, T > 32: the tcgen05 tiles are built for 128-wide
// heads, and at 64 the state of a head is small enough for the registers of
// four warps.
//
// Chunks of C = 32 tokens (the last one padded with g = 1, beta = 0, q = k =
// v = 0; metaltile-std `gated_delta_wy.rs`, "Algorithm" steps 1-9, and the
// chunk-loop precondition on padding), the chunk algebra of ferrox-core
// `gdn_chunk.rs`, "The algebra", in the innovation form:
//   prep, every (head, chunk) at once, one CTA each:
//     L = KK^T diag(beta), QK^T;  T_L = (I + L)^-1 (blockwise, fp32);
//     T_A = diag(beta)(Gam . T_L);  cP = -diag(G_C beta) T_L;  cU = diag(Gam_end) T_A;
//     -Pt = cP K;  Qh = (G Q - diag(G) M T_L K) / sqrt(Dk);  Ut = cU V;
//     y_loc = (Gam . QK^T) T_A V / sqrt(Dk)
//   into a workspace block [-Pt; Qh; Ut; K; y_loc] (5C rows of 64) and G_C;
//   scan, one CTA per head, S in registers (warp w < 4: value rows 16w .. 16w
//   + 15 in the m16n8 accumulator layout), chunk after chunk:
//     [-Z | Y] = S [-Pt; Qh]^T;  y = y_loc + Y;  S <- G_C S + (Ut^T - Z) K,
// the workspace blocks coming in by TMA up to three chunks ahead, issued by a
// fifth warp; the four state warps meet no CTA-wide barrier on the way.
#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"
#include "warp_mma.cuh"

namespace gdn {
namespace {

constexpr int kD = 64;            // head size (Dk = Dv)
constexpr int kC = 32;            // chunk
constexpr int kPT = 256;          // prep threads: eight warps
constexpr int kST = 160;          // scan threads: four warps x 16 value rows + a loader warp
constexpr int kFS = kC + 1;       // fp32 row stride of the C x C arrays
constexpr int kCS = kC + 8;       // 16-bit row stride of the C x C arrays (80 B)
constexpr int kYS = kD + 8;       // 16-bit row stride of the y staging (144 B)
constexpr int kBlkRows = 5 * kC;  // workspace rows per chunk: -Pt, Qh, Ut, K, y_loc
constexpr int kBlkBytes = kBlkRows * kD * 2;
constexpr int kStages = 3;        // scan: workspace blocks in flight
constexpr int kAlign = 1024;      // 128-byte swizzled boxes

template <typename E>
struct PrepSmem {
  E tok[3][kC * kD];  // k, q, v: TMA boxes of C rows x 64, 128-byte swizzled (wm::sw64)
  float lm[kC][kFS], qk[kC][kFS];  // L = KK^T diag(beta), QK^T (then scratch)
  float tlf[kC][kFS];              // T_L in fp32
  E a3t[kC][kCS], a3b[kC][kCS];    // diag(G) M, Gam . QK^T
  E tlb[kC][kCS], tab[kC][kCS];    // T_L, T_A
  E cp[kC][kCS], cu[kC][kCS];      // -diag(G_C beta) T_L, diag(Gam_end) T_A
  E w_m[kC][kCS], w_y[kC][kCS];    // -W_M / sqrt(Dk), W_Y / sqrt(Dk)
  float lam[kC], gt[kC], bt[kC], gend[kC];
  float gc;
  alignas(8) uint64_t bar;  // the token boxes landed
};

template <typename E>
struct ScanSmem {
  E stage[kStages][kBlkRows * kD];  // workspace blocks, 128-byte swizzled rows
  E ys[kC][kYS];                    // Y staging [t][v], each warp its 16 columns
  float gcs[kStages];  // G_C of the chunk in each stage (set by the loader)
  alignas(8) uint64_t full[kStages];   // a block landed
  alignas(8) uint64_t empty[kStages];  // the four state warps are done with a stage
};

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  return raw + ((kAlign - (wm::s_u32(raw) & (kAlign - 1))) & (kAlign - 1));
}

// ---------------------------------------------------------------------------
// prep: one CTA per (head, chunk), blockIdx.x = bh * NC + n
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kPT)
mma_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_v, const E* __restrict__ g,
                const E* __restrict__ beta, E* __restrict__ ws, float* __restrict__ wsgc, int T,
                int Hk, int Hv, int NC, int opts, float scale) {
  using namespace wm;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PrepSmem<E>& sm = *reinterpret_cast<PrepSmem<E>*>(aligned_smem(smem_raw));
  const int blk = blockIdx.x, bh = blk / NC, n = blk - bh * NC;
  const int b = bh / Hv, hv = bh - b * Hv, hk = key_head(hv, Hk, Hv, opts), t0 = n * kC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;
  constexpr int NT8 = kC / 8, NK16 = kC / 16;
  const uint32_t bar = s_u32(&sm.bar);
  const uint32_t tk = s_u32(sm.tok[0]), tq = s_u32(sm.tok[1]), tv = s_u32(sm.tok[2]);
  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();  // the barrier is initialised before anyone waits on it
  if (tid == 0) {
    ptx::mbar_expect_tx(bar, 3 * kC * kD * sizeof(E));
    ptx::tma_load_4d(tk, &tm_k, bar, 0, hk, t0, b);  // tokens past T arrive as zeros
    ptx::tma_load_4d(tq, &tm_q, bar, 0, hk, t0, b);
    ptx::tma_load_4d(tv, &tm_v, bar, 0, hv, t0, b);
  }
  if (warp == 0) {
    // Gates: chunk-local prefix sums of log2 of the decay (padded tokens: 1).
    const int t = t0 + lane;
    float l = 0.f, bv = 0.f;
    if (t < T) {
      const size_t gi = ((size_t)b * T + t) * Hv + hv;
      const float gv = to_f32(g[gi]);
      l = (opts & kOptLogGate) ? gv * 1.4426950408889634f : log2f(gv);
      bv = to_f32(beta[gi]);
    }
    l = fmaxf(l, -1000.f);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, l, off);
      if (lane >= off) l += u;
    }
    const float lend = __shfl_sync(0xffffffffu, l, kC - 1);
    sm.lam[lane] = l;
    sm.gt[lane] = exp2f(l);
    sm.bt[lane] = bv;
    sm.gend[lane] = exp2f(lend - l);
    if (lane == 0) {
      sm.gc = exp2f(lend);
      wsgc[blk] = exp2f(lend);
    }
  }
  // A load that never lands (2 s) is recorded in the device error word and
  // the chunk is left unwritten.
  if (!__syncthreads_and(ptx::mbar_wait(bar, 0))) return;
  if (opts & kOptL2NormQK) {
    // Every k and q row as x / |x|: a warp a row, two values a lane.
    for (int r = warp; r < 2 * kC; r += kPT / 32) {
      E* p = reinterpret_cast<E*>(reinterpret_cast<uint8_t*>(r < kC ? sm.tok[0] : sm.tok[1]) +
                                  sw64(r % kC, 2 * lane));
      const float x0 = to_f32(p[0]), x1 = to_f32(p[1]);
      float ss = fmaf(x0, x0, x1 * x1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float f = inv_norm(ss);
      p[0] = from_f32<E>(x0 * f);
      p[1] = from_f32<E>(x1 * f);
    }
    __syncthreads();
  }

  // L = KK^T diag(beta) and QK^T (fp32): tiles (matrix, m16 tile, n8 tile).
  for (int ti = warp; ti < 2 * NK16 * NT8; ti += kPT / 32) {
    const int mat = ti / (NK16 * NT8), rem = ti - mat * NK16 * NT8;
    const int mt = rem / NT8, nt = rem - mt * NT8;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t a[4], bb[2];
      ldsm4(sw_a(mat ? tq : tk, 16 * mt, 16 * kk, lane), a);
      ldsm2(sw_bnk(tk, 8 * nt, 16 * kk, lane), bb);
      mma<E>(acc, a, bb);
    }
    float(*o)[kFS] = mat ? sm.qk : sm.lm;
    const int c0 = 8 * nt + 2 * cq;
    const float b0 = mat ? 1.f : sm.bt[c0], b1 = mat ? 1.f : sm.bt[c0 + 1];
    o[16 * mt + gq][c0] = acc[0] * b0;
    o[16 * mt + gq][c0 + 1] = acc[1] * b1;
    o[16 * mt + gq + 8][c0] = acc[2] * b0;
    o[16 * mt + gq + 8][c0 + 1] = acc[3] * b1;
  }
  __syncthreads();

  // T_L = (I + L)^-1 blockwise; meanwhile A3 = diag(G) M and Gam . QK^T.
  if (warp == 0) {
    inverse_diag_blocks<kC, kFS>(sm.lm, sm.tlf, lane);
  } else {
    for (int e = tid - 32; e < kC * kC; e += kPT - 32) {
      const int t = e / kC, j = e - t * kC;
      const bool keep = j <= t;
      const float qkv = sm.qk[t][j];
      sm.a3t[t][j] = from_f32<E>(keep ? sm.gt[t] * sm.bt[j] * qkv : 0.f);
      sm.a3b[t][j] = from_f32<E>(keep ? exp2f(sm.lam[t] - sm.lam[j]) * qkv : 0.f);
    }
  }
  __syncthreads();
  combine_blocks<8, kC, kPT, kFS>(sm.lm, sm.tlf, sm.qk, tid);
  combine_blocks<16, kC, kPT, kFS>(sm.lm, sm.tlf, sm.qk, tid);
  // T_L, T_A = diag(beta)(Gam . T_L), cP = -diag(G_C beta) T_L and
  // cU = diag(Gam_end) T_A in 16 bits (zero above the diagonal).
  for (int e = tid; e < kC * kC; e += kPT) {
    const int r = e / kC, jj = e - r * kC;
    const bool low = r >= jj;
    const float tl = low ? sm.tlf[r][jj] : 0.f;
    const float ta = low ? sm.bt[r] * exp2f(sm.lam[r] - sm.lam[jj]) * tl : 0.f;
    sm.tlb[r][jj] = from_f32<E>(tl);
    sm.tab[r][jj] = from_f32<E>(ta);
    sm.cp[r][jj] = from_f32<E>(-sm.gc * sm.bt[r] * tl);
    sm.cu[r][jj] = from_f32<E>(sm.gend[r] * ta);
  }
  __syncthreads();

  // W_M = A3t T_L and W_Y = A3b T_A, stored as -W_M / sqrt(Dk), W_Y / sqrt(Dk).
  for (int ti = warp; ti < 2 * NK16 * NT8; ti += kPT / 32) {
    const int mat = ti / (NK16 * NT8), rem = ti - mat * NK16 * NT8;
    const int mt = rem / NT8, nt = rem - mt * NT8;
    const E* A = mat ? &sm.a3b[0][0] : &sm.a3t[0][0];
    const E* Bm = mat ? &sm.tab[0][0] : &sm.tlb[0][0];
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < NK16; ++kk) {
      uint32_t a[4], bb[2];
      ldsm4(a_addr(A, kCS, 16 * mt, 16 * kk, lane), a);
      ldsm2t(bkn_addr(Bm, kCS, 16 * kk, 8 * nt, lane), bb);
      mma<E>(acc, a, bb);
    }
    const float f = mat ? scale : -scale;
    E(*o)[kCS] = mat ? sm.w_y : sm.w_m;
    *reinterpret_cast<uint32_t*>(&o[16 * mt + gq][8 * nt + 2 * cq]) =
        pk<E>(f * acc[0], f * acc[1]);
    *reinterpret_cast<uint32_t*>(&o[16 * mt + gq + 8][8 * nt + 2 * cq]) =
        pk<E>(f * acc[2], f * acc[3]);
  }
  __syncthreads();

  // The block: -Pt = cP K, Qh = (G Q - W_M K) / sqrt(Dk), Ut = cU V, y_loc =
  // W_Y V / sqrt(Dk) (rows 0, C, 2C, 4C; C x 64 each), written from the
  // accumulators; then the chunk's K rows (row 3C), as normalised here.
  E* blkp = ws + (size_t)blk * kBlkRows * kD;
  for (int ti = warp; ti < 4 * NK16 * (kD / 8); ti += kPT / 32) {
    const int mat = ti / (NK16 * (kD / 8)), rem = ti - mat * NK16 * (kD / 8);
    const int mt = rem / (kD / 8), nt = rem - mt * (kD / 8);
    const E* A = mat == 0 ? &sm.cp[0][0]
                          : (mat == 1 ? &sm.w_m[0][0] : (mat == 2 ? &sm.cu[0][0] : &sm.w_y[0][0]));
    const uint32_t Bm = mat < 2 ? tk : tv;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < NK16; ++kk) {
      uint32_t a[4], bb[2];
      ldsm4(a_addr(A, kCS, 16 * mt, 16 * kk, lane), a);
      ldsm2t(sw_bkn(Bm, 16 * kk, 8 * nt, lane), bb);
      mma<E>(acc, a, bb);
    }
    const int tr = 16 * mt + gq, c0 = 8 * nt + 2 * cq;
    if (mat == 1) {
      const uint8_t* qb = reinterpret_cast<const uint8_t*>(sm.tok[1]);
      const E* q0 = reinterpret_cast<const E*>(qb + sw64(tr, c0));
      const E* q1 = reinterpret_cast<const E*>(qb + sw64(tr + 8, c0));
      const float g0 = sm.gt[tr] * scale, g1 = sm.gt[tr + 8] * scale;
      acc[0] = fmaf(g0, to_f32(q0[0]), acc[0]);
      acc[1] = fmaf(g0, to_f32(q0[1]), acc[1]);
      acc[2] = fmaf(g1, to_f32(q1[0]), acc[2]);
      acc[3] = fmaf(g1, to_f32(q1[1]), acc[3]);
    }
    const int row0 = (mat == 3 ? 4 : mat) * kC + tr;
    *reinterpret_cast<uint32_t*>(blkp + (size_t)row0 * kD + c0) = pk<E>(acc[0], acc[1]);
    *reinterpret_cast<uint32_t*>(blkp + (size_t)(row0 + 8) * kD + c0) = pk<E>(acc[2], acc[3]);
  }
  for (int i = tid; i < kC * kD / 8; i += kPT) {
    const int r = i / (kD / 8), c8 = (i % (kD / 8)) * 8;
    *reinterpret_cast<uint4*>(blkp + (size_t)(3 * kC + r) * kD + c8) =
        *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(sm.tok[0]) + sw64(r, c8));
  }
}

// ---------------------------------------------------------------------------
// scan: one CTA per head
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kST)
mma_scan_kernel(const __grid_constant__ CUtensorMap tm_ws, const float* __restrict__ wsgc,
                const float* state_in, float* state_out, E* __restrict__ y, int T, int Hv,
                int NC) {
  using namespace wm;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ScanSmem<E>& sm = *reinterpret_cast<ScanSmem<E>*>(aligned_smem(smem_raw));
  const int bh = blockIdx.x, b = bh / Hv, hv = bh - b * Hv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3, r0 = 16 * warp + gq;
  constexpr int NT8 = kC / 8, NK16 = kC / 16;
  if (tid == 0) {
    ptx::prefetch_tmap(&tm_ws);
    for (int s2 = 0; s2 < kStages; ++s2) {
      ptx::mbar_init(s_u32(&sm.full[s2]), 1);
      ptx::mbar_init(s_u32(&sm.empty[s2]), 4);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();  // the barriers' initialisation
  if (warp == 4) {
    // Loader: chunk n's block into stage n % kStages once the state warps
    // are done with chunk n - kStages there.  A wait that runs out (2 s) is
    // recorded in the device error word; the loads issued land before the
    // CTA ends.
    if (lane == 0) {
      int n = 0;
      for (; n < NC; ++n) {
        const int st = n % kStages;
        if (n >= kStages &&
            !ptx::mbar_wait(s_u32(&sm.empty[st]), ((n / kStages) - 1) & 1))
          break;
        const uint32_t fb = s_u32(&sm.full[st]);
        sm.gcs[st] = __ldg(wsgc + (size_t)bh * NC + n);  // released by the arrival below
        ptx::mbar_expect_tx(fb, kBlkBytes);
        ptx::tma_load_2d(s_u32(sm.stage[st]), &tm_ws, fb, 0, (bh * NC + n) * kBlkRows);
      }
      for (int m = (n > kStages ? n - kStages : 0); m < n; ++m)
        ptx::mbar_wait(s_u32(&sm.full[m % kStages]), (m / kStages) & 1);
    }
    return;
  }
  // S rows r0 and r0 + 8, columns 8j + 2cq, +1 (j < 8): the accumulator layout
  // of eight m16n8 tiles.
  float s[kD / 8][4];
  {
    const float* src = state_in ? state_in + (size_t)bh * kD * kD : nullptr;
#pragma unroll
    for (int j = 0; j < kD / 8; ++j) {
      float2 lo = make_float2(0.f, 0.f), hi = lo;
      if (src) {
        lo = __ldcs(reinterpret_cast<const float2*>(src + r0 * kD + 8 * j + 2 * cq));
        hi = __ldcs(reinterpret_cast<const float2*>(src + (r0 + 8) * kD + 8 * j + 2 * cq));
      }
      s[j][0] = lo.x;
      s[j][1] = lo.y;
      s[j][2] = hi.x;
      s[j][3] = hi.y;
    }
  }
  for (int j = 0; j < NC; ++j) {
    const int st = j % kStages;
    // A block that never lands (2 s) is recorded in the device error word and
    // the head is left unwritten.
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(s_u32(&sm.full[st]), (j / kStages) & 1))) return;
    const float gcv = sm.gcs[st];
    const uint32_t base = s_u32(sm.stage[st]);
    // [-Z | Y] = S [-Pt; Qh]^T: B from rows 0 .. 2C of the block.
    float zy[2 * NT8][4];
#pragma unroll
    for (int nn = 0; nn < 2 * NT8; ++nn) zy[nn][0] = zy[nn][1] = zy[nn][2] = zy[nn][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      const uint32_t a[4] = {pk<E>(s[2 * kk][0], s[2 * kk][1]), pk<E>(s[2 * kk][2], s[2 * kk][3]),
                             pk<E>(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                             pk<E>(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
      for (int nn = 0; nn < 2 * NT8; ++nn) {
        uint32_t bb[2];
        ldsm2(sw_bnk(base, 8 * nn, 16 * kk, lane), bb);
        mma<E>(zy[nn], a, bb);
      }
    }
    // W = Ut^T - Z as A fragments: Ut^T (rows v of this warp, columns t) read
    // transposed from the block's Ut rows, plus the -Z tiles.
    uint32_t wa[NK16][4];
#pragma unroll
    for (int kk = 0; kk < NK16; ++kk) {
      uint32_t u[4];
      ldsm4t(sw_at(base, 2 * kC + 16 * kk, 16 * warp, lane), u);
      const float2 u0 = unpk<E>(u[0]), u1 = unpk<E>(u[1]), u2 = unpk<E>(u[2]),
                   u3 = unpk<E>(u[3]);
      wa[kk][0] = pk<E>(u0.x + zy[2 * kk][0], u0.y + zy[2 * kk][1]);
      wa[kk][1] = pk<E>(u1.x + zy[2 * kk][2], u1.y + zy[2 * kk][3]);
      wa[kk][2] = pk<E>(u2.x + zy[2 * kk + 1][0], u2.y + zy[2 * kk + 1][1]);
      wa[kk][3] = pk<E>(u3.x + zy[2 * kk + 1][2], u3.y + zy[2 * kk + 1][3]);
    }
    // S <- G_C S + W K (B: the block's K rows, transposing).
#pragma unroll
    for (int jn = 0; jn < kD / 8; ++jn)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[jn][e] *= gcv;
#pragma unroll
    for (int kk = 0; kk < NK16; ++kk)
#pragma unroll
      for (int jn = 0; jn < kD / 8; ++jn) {
        uint32_t bb[2];
        ldsm2t(sw_bkn(base, 3 * kC + 16 * kk, 8 * jn, lane), bb);
        mma<E>(s[jn], wa[kk], bb);
      }
    // y = y_loc + Y for this warp's 16 value columns: Y staged transposed as
    // [t][v], then rows t < T written with the block's y_loc rows added.
    {
      const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int nn = 0; nn < NT8; nn += 2) {
        const int t = 8 * (nn + (mi >> 1)) + r8, vv = 16 * warp + 8 * (mi & 1);
        stsm4t(s_u32(&sm.ys[t][vv]), pk<E>(zy[NT8 + nn][0], zy[NT8 + nn][1]),
               pk<E>(zy[NT8 + nn][2], zy[NT8 + nn][3]),
               pk<E>(zy[NT8 + nn + 1][0], zy[NT8 + nn + 1][1]),
               pk<E>(zy[NT8 + nn + 1][2], zy[NT8 + nn + 1][3]));
      }
      __syncwarp();
      const uint8_t* bb8 = reinterpret_cast<const uint8_t*>(sm.stage[st]);
#pragma unroll
      for (int i = lane; i < kC * 2; i += 32) {
        const int t = i >> 1, c8 = 16 * warp + 8 * (i & 1), tt = j * kC + t;
        if (tt < T) {
          const uint4 yl = *reinterpret_cast<const uint4*>(bb8 + sw64(4 * kC + t, c8));
          const uint4 yv = *reinterpret_cast<const uint4*>(&sm.ys[t][c8]);
          const uint32_t* a = reinterpret_cast<const uint32_t*>(&yl);
          const uint32_t* c = reinterpret_cast<const uint32_t*>(&yv);
          uint4 o;
          uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = unpk<E>(a[e]), z = unpk<E>(c[e]);
            op[e] = pk<E>(x.x + z.x, x.y + z.y);
          }
          *reinterpret_cast<uint4*>(y + (((size_t)b * T + tt) * Hv + hv) * kD + c8) = o;
        }
      }
    }
    __syncwarp();  // this warp is done with the stage and its ys columns
    if (lane == 0) ptx::mbar_arrive(s_u32(&sm.empty[st]));
  }
  float* dst = state_out + (size_t)bh * kD * kD;
#pragma unroll
  for (int jn = 0; jn < kD / 8; ++jn) {
    __stcs(reinterpret_cast<float2*>(dst + r0 * kD + 8 * jn + 2 * cq),
           make_float2(s[jn][0], s[jn][1]));
    __stcs(reinterpret_cast<float2*>(dst + (r0 + 8) * kD + 8 * jn + 2 * cq),
           make_float2(s[jn][2], s[jn][3]));
  }
}

// Tokens [B, T, H, 64] of 16-bit type dt, box {64, 1, C, 1}, 128-byte
// swizzle; tokens past T read as zeros.
bool make_token_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int B, int T,
                    int H) {
  const TmapEncodeFn enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2,
                                 (cuuint64_t)T * H * kD * 2};
  const cuuint32_t box[4] = {(cuuint32_t)kD, 1, (cuuint32_t)kC, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// The workspace blocks as rows of 64 16-bit values, box {64, 5C}: one chunk.
bool make_ws_map(CUtensorMap* m, CUtensorMapDataType dt, void* base, size_t rows) {
  const TmapEncodeFn enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kBlkRows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename E>
cudaError_t launch_mma(const PrefillArgs& a) {
  const int NC = (a.T + kC - 1) / kC, BH = a.B * a.Hv;
  const size_t blocks = (size_t)BH * NC;
  E* ws = static_cast<E*>(a.workspace);
  float* wsgc = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + blocks * kBlkBytes);
  constexpr CUtensorMapDataType dt = std::is_same_v<E, __half> ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tm_k{}, tm_q{}, tm_v{}, tm_ws{};
  if (!make_token_map(&tm_k, dt, a.k, a.B, a.T, a.Hk) ||
      !make_token_map(&tm_q, dt, a.q, a.B, a.T, a.Hk) ||
      !make_token_map(&tm_v, dt, a.v, a.B, a.T, a.Hv) ||
      !make_ws_map(&tm_ws, dt, ws, blocks * kBlkRows))
    return cudaErrorInvalidValue;
  const int prep_smem = (int)sizeof(PrepSmem<E>) + kAlign;
  const int scan_smem = (int)sizeof(ScanSmem<E>) + kAlign;
  cudaError_t e = cudaFuncSetAttribute(mma_prep_kernel<E>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, prep_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(mma_scan_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             scan_smem);
  if (e != cudaSuccess) return e;
  const float scale = 1.0f / sqrtf((float)kD);
  mma_prep_kernel<E><<<(unsigned)blocks, kPT, prep_smem, a.stream>>>(
      tm_k, tm_q, tm_v, static_cast<const E*>(a.g), static_cast<const E*>(a.beta), ws, wsgc, a.T,
      a.Hk, a.Hv, NC, a.options, scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mma_scan_kernel<E><<<BH, kST, scan_smem, a.stream>>>(tm_ws, wsgc, a.state_in, a.state_out,
                                                      static_cast<E*>(a.y), a.T, a.Hv, NC);
  return cudaGetLastError();
}

}  // namespace

bool mma_path_applies(int Dk, int Dv, int dtype, int T) {
  return (dtype == 1 || dtype == 2) && Dk == kD && Dv == kD && T > kShortT;
}

size_t prefill_mma_workspace_bytes(int B, int T, int Hv) {
  const size_t blocks = (size_t)B * Hv * ((T + kC - 1) / kC);
  return blocks * kBlkBytes + ((blocks * sizeof(float) + 255) & ~(size_t)255);
}

cudaError_t launch_prefill_mma(const PrefillArgs& a) {
  return a.dtype == 2 ? launch_mma<__half>(a) : launch_mma<__nv_bfloat16>(a);
}

int prefill_mma_device_error(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, ptx::g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int z = 0;
    if (cudaMemcpyToSymbol(ptx::g_device_error, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace gdn
