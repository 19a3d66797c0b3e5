// Chunked prefill on warp-level tensor-core MMAs for head size 256 (Dk = Dv =
// 256), bf16 or fp16 inputs, T > 32.
//
// The chunk algebra of the head-size-64 path (ferrox-core `gdn_chunk.rs`, "The
// algebra", innovation form; chunks of C = 32 padded as metaltile-std
// `gated_delta_wy.rs` pads its last chunk), with the state spread wider: a
// 256 x 256 fp32 state is 256 KB, the whole register file of an SM, so the
// scan of a head runs on four CTAs of 64 value rows each (the rows of S evolve
// independently given the chunk's coefficients), and inside a CTA the 256 keys
// are split over warp pairs:
//   prep, one CTA of sixteen warps per (head, chunk), all at once: L = KK^T
//     diag(beta), QK^T, T_L blockwise, the coefficients, W_M and W_Y, then
//     -Pt = cP K, Qh / sqrt(Dk), Ut = cU V and y_loc / sqrt(Dk) into a workspace
//     block [-Pt; Qh; K; Ut; y_loc] (5C rows of 256) and G_C beside it;
//   scan, CTA (head, quarter q): warp w < 8 holds value rows 64q + 16(w % 4) ..
//     + 15 and keys 128(w / 4) .. + 127 of S in m16n8 accumulator registers;
//     per chunk each warp forms its half-key part of [-Z | Y] = S [-Pt; Qh]^T,
//     the two warps of a row group add them through shared memory, then
//     S[:, own keys] <- G_C S + (Ut^T - Z) K[:, own keys], and the first warp
//     of the pair writes y = y_loc + Y.  A ninth warp brings in, by TMA, each
//     chunk's -Pt, Qh and K rows (all keys) and the quarter's Ut and y_loc
//     columns, two chunks ahead.
#include "gdn_internal.cuh"
#include "sm100_ptx.cuh"
#include "warp_mma.cuh"

namespace gdn {
namespace {

constexpr int kD = 256;           // head size (Dk = Dv)
constexpr int kC = 32;            // chunk
constexpr int kPT = 512;          // prep threads
constexpr int kST = 288;          // scan threads: 8 state warps + a loader warp
constexpr int kFS = kC + 1;       // fp32 row stride of the C x C arrays
constexpr int kCS = kC + 8;       // 16-bit row stride of the C x C arrays (80 B)
constexpr int kYS = 64 + 8;       // 16-bit row stride of the y staging (144 B)
constexpr int kBlkRows = 5 * kC;  // workspace rows per chunk: -Pt, Qh, K, Ut, y_loc
constexpr size_t kBlkElems = (size_t)kBlkRows * kD;
constexpr int kStages = 2;        // scan: chunks in flight
constexpr int kRowsA = 3 * kC;    // stage part A: -Pt, Qh, K rows, every key
constexpr int kBytesA = kRowsA * kD * 2;
constexpr int kBytesB = 2 * kC * 64 * 2;  // part B: Ut, y_loc rows, the quarter's 64 columns
constexpr int kAlign = 1024;

// Rows of 256 16-bit values held as four 64-column segments, segment-major
// ([seg][row][64], 128-byte swizzled rows): byte offset of element (r, c) in
// an array of `rows` rows.
__device__ __forceinline__ uint32_t seg_off(int rows, int r, int c) {
  return (c >> 6) * (rows * 128) + wm::sw64(r, c & 63);
}

template <typename E>
struct PrepSmem {
  E tok[3][kC * kD];  // k, q, v: TMA boxes landing as [seg][t][64]
  float lm[kC][kFS], qk[kC][kFS], tlf[kC][kFS];
  E a3t[kC][kCS], a3b[kC][kCS], tlb[kC][kCS], tab[kC][kCS];
  E cp[kC][kCS], cu[kC][kCS], w_m[kC][kCS], w_y[kC][kCS];
  float lam[kC], gt[kC], bt[kC], gend[kC];
  float gc;
  alignas(8) uint64_t bar;
};

template <typename E>
struct ScanSmem {
  E stage_a[kStages][kRowsA * kD];  // [seg][row][64] of -Pt, Qh, K
  E stage_b[kStages][2 * kC * 64];  // [row][64] of Ut, y_loc (this quarter's columns)
  float xbuf[8][2][32][32];         // partial [-Z | Y] of each warp, by chunk parity
  E ys[kC][kYS];                    // Y staging [t][v] of the four writing warps
  float gcs[kStages];  // G_C of the chunk in each stage (set by the loader)
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
};

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  return raw + ((kAlign - (wm::s_u32(raw) & (kAlign - 1))) & (kAlign - 1));
}

// TMA tensor loads of 3 and 5 dimensions into shared memory, completing on bar.
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

// The two warps of a row group (ids 1..4, 64 threads).
__device__ __forceinline__ void pair_sync(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

// ---------------------------------------------------------------------------
// prep: one CTA per (head, chunk), blockIdx.x = bh * NC + n
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kPT)
mma256_prep_kernel(const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_v, const E* __restrict__ g,
                   const E* __restrict__ beta, E* __restrict__ ws, float* __restrict__ wsgc,
                   int T, int Hk, int Hv, int NC, int opts, float scale) {
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
    tma_load_5d(tk, &tm_k, bar, 0, t0, 0, hk, b);  // tokens past T arrive as zeros
    tma_load_5d(tq, &tm_q, bar, 0, t0, 0, hk, b);
    tma_load_5d(tv, &tm_v, bar, 0, t0, 0, hv, b);
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
    // Every k and q row as x / |x|: a warp a row, eight values (16 bytes) a lane.
    for (int r = warp; r < 2 * kC; r += kPT / 32) {
      uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(r < kC ? sm.tok[0] : sm.tok[1]) +
                                          seg_off(kC, r % kC, 8 * lane));
      uint4 v = *p;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
      float x[8], ss = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f2 = unpk<E>(w[e]);
        x[2 * e] = f2.x;
        x[2 * e + 1] = f2.y;
        ss = fmaf(f2.x, f2.x, fmaf(f2.y, f2.y, ss));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float f = inv_norm(ss);
#pragma unroll
      for (int e = 0; e < 4; ++e) w[e] = pk<E>(x[2 * e] * f, x[2 * e + 1] * f);
      *p = v;
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
      ldsm4((mat ? tq : tk) + seg_off(kC, 16 * mt + (lane & 15), 16 * kk + 8 * (lane >> 4)), a);
      ldsm2(tk + seg_off(kC, 8 * nt + (lane & 7), 16 * kk + 8 * ((lane >> 3) & 1)), bb);
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

  // The block: -Pt = cP K (row 0), Qh = (G Q - W_M K) / sqrt(Dk) (row C),
  // Ut = cU V (row 3C), y_loc = W_Y V / sqrt(Dk) (row 4C), from the
  // accumulators; then the chunk's K rows (row 2C), as normalised here.
  E* blkp = ws + (size_t)blk * kBlkElems;
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
      ldsm2t(Bm + seg_off(kC, 16 * kk + (lane & 15), 8 * nt), bb);
      mma<E>(acc, a, bb);
    }
    const int tr = 16 * mt + gq, c0 = 8 * nt + 2 * cq;
    if (mat == 1) {
      const uint8_t* qb = reinterpret_cast<const uint8_t*>(sm.tok[1]);
      const E* q0 = reinterpret_cast<const E*>(qb + seg_off(kC, tr, c0));
      const E* q1 = reinterpret_cast<const E*>(qb + seg_off(kC, tr + 8, c0));
      const float g0 = sm.gt[tr] * scale, g1 = sm.gt[tr + 8] * scale;
      acc[0] = fmaf(g0, to_f32(q0[0]), acc[0]);
      acc[1] = fmaf(g0, to_f32(q0[1]), acc[1]);
      acc[2] = fmaf(g1, to_f32(q1[0]), acc[2]);
      acc[3] = fmaf(g1, to_f32(q1[1]), acc[3]);
    }
    const int row0 = (mat < 2 ? mat : mat + 1) * kC + tr;
    *reinterpret_cast<uint32_t*>(blkp + (size_t)row0 * kD + c0) = pk<E>(acc[0], acc[1]);
    *reinterpret_cast<uint32_t*>(blkp + (size_t)(row0 + 8) * kD + c0) = pk<E>(acc[2], acc[3]);
  }
  for (int i = tid; i < kC * kD / 8; i += kPT) {
    const int r = i / (kD / 8), c8 = (i % (kD / 8)) * 8;
    *reinterpret_cast<uint4*>(blkp + (size_t)(2 * kC + r) * kD + c8) =
        *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(sm.tok[0]) +
                                        seg_off(kC, r, c8));
  }
}

// ---------------------------------------------------------------------------
// scan: CTA (head bh, quarter qt) = blockIdx.x = 4 bh + qt
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kST, 1)
mma256_scan_kernel(const __grid_constant__ CUtensorMap tm_wa,
                   const __grid_constant__ CUtensorMap tm_wb, const float* __restrict__ wsgc,
                   const float* state_in, float* state_out, E* __restrict__ y, int T, int Hv,
                   int NC) {
  using namespace wm;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ScanSmem<E>& sm = *reinterpret_cast<ScanSmem<E>*>(aligned_smem(smem_raw));
  const int bh = blockIdx.x >> 2, qt = blockIdx.x & 3, b = bh / Hv, hv = bh - b * Hv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;
  const int rg = warp & 3, kh = warp >> 2;  // row group, key half (state warps)
  const int r0 = 64 * qt + 16 * rg + gq;   // this thread's value rows r0, r0 + 8
  constexpr int NT8 = kC / 8, NK16 = kC / 16;
  if (tid == 0) {
    ptx::prefetch_tmap(&tm_wa);
    ptx::prefetch_tmap(&tm_wb);
    for (int s2 = 0; s2 < kStages; ++s2) {
      ptx::mbar_init(s_u32(&sm.full[s2]), 1);
      ptx::mbar_init(s_u32(&sm.empty[s2]), 8);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();  // the barriers' initialisation
  if (warp == 8) {
    // Loader: chunk n's rows into stage n % kStages once the eight state warps
    // are done with chunk n - kStages there.  A wait that runs out (2 s) is
    // recorded in the device error word; the loads issued land before the
    // CTA ends.
    if (lane == 0) {
      int n = 0;
      for (; n < NC; ++n) {
        const int st = n % kStages;
        if (n >= kStages && !ptx::mbar_wait(s_u32(&sm.empty[st]), ((n / kStages) - 1) & 1))
          break;
        const uint32_t fb = s_u32(&sm.full[st]);
        sm.gcs[st] = __ldg(wsgc + (size_t)bh * NC + n);  // released by the arrival below
        const int row = (bh * NC + n) * kBlkRows;
        ptx::mbar_expect_tx(fb, kBytesA + kBytesB);
        tma_load_3d(s_u32(sm.stage_a[st]), &tm_wa, fb, 0, row, 0);
        tma_load_3d(s_u32(sm.stage_b[st]), &tm_wb, fb, 0, row + kRowsA, qt);
      }
      for (int m = (n > kStages ? n - kStages : 0); m < n; ++m)
        ptx::mbar_wait(s_u32(&sm.full[m % kStages]), (m / kStages) & 1);
    }
    return;
  }
  // S rows r0, r0 + 8, keys 128 kh + 8j + 2cq, +1 (j < 16).
  float s[16][4];
  {
    const float* src = state_in ? state_in + (size_t)bh * kD * kD : nullptr;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int c = 128 * kh + 8 * j + 2 * cq;
      float2 lo = make_float2(0.f, 0.f), hi = lo;
      if (src) {
        lo = __ldcs(reinterpret_cast<const float2*>(src + (size_t)r0 * kD + c));
        hi = __ldcs(reinterpret_cast<const float2*>(src + (size_t)(r0 + 8) * kD + c));
      }
      s[j][0] = lo.x;
      s[j][1] = lo.y;
      s[j][2] = hi.x;
      s[j][3] = hi.y;
    }
  }
  for (int j = 0; j < NC; ++j) {
    const int st = j % kStages, par = j & 1;
    // A chunk that never lands (2 s) is recorded in the device error word and
    // the quarter is left unwritten.
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(s_u32(&sm.full[st]), (j / kStages) & 1))) return;
    const float gcv = sm.gcs[st];
    const uint32_t ba = s_u32(sm.stage_a[st]), bb8 = s_u32(sm.stage_b[st]);
    // This warp's key half of [-Z | Y] = S [-Pt; Qh]^T (B: rows 0 .. 2C of part A).
    float zy[2 * NT8][4];
#pragma unroll
    for (int nn = 0; nn < 2 * NT8; ++nn) zy[nn][0] = zy[nn][1] = zy[nn][2] = zy[nn][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t a[4] = {pk<E>(s[2 * kk][0], s[2 * kk][1]), pk<E>(s[2 * kk][2], s[2 * kk][3]),
                             pk<E>(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                             pk<E>(s[2 * kk + 1][2], s[2 * kk + 1][3])};
      const int k0 = 128 * kh + 16 * kk;
#pragma unroll
      for (int nn = 0; nn < 2 * NT8; ++nn) {
        uint32_t bb[2];
        ldsm2(ba + seg_off(kRowsA, 8 * nn + (lane & 7), k0 + 8 * ((lane >> 3) & 1)), bb);
        mma<E>(zy[nn], a, bb);
      }
    }
    // The pair's halves added: each warp posts its part, then reads the other's.
    {
      float* mine = &sm.xbuf[warp][par][0][0];
#pragma unroll
      for (int nn = 0; nn < 2 * NT8; ++nn)
#pragma unroll
        for (int e = 0; e < 4; ++e) mine[(4 * nn + e) * 32 + lane] = zy[nn][e];
      pair_sync(1 + rg);
      const float* other = &sm.xbuf[warp ^ 4][par][0][0];
#pragma unroll
      for (int nn = 0; nn < 2 * NT8; ++nn)
#pragma unroll
        for (int e = 0; e < 4; ++e) zy[nn][e] += other[(4 * nn + e) * 32 + lane];
    }
    // W = Ut^T - Z (Ut^T: rows v of this row group, read transposed from part
    // B's Ut rows), then S[:, own keys] <- G_C S + W K[:, own keys].
    uint32_t wa[NK16][4];
#pragma unroll
    for (int kk = 0; kk < NK16; ++kk) {
      uint32_t u[4];
      ldsm4t(bb8 + sw64(16 * kk + (lane & 7) + 8 * (lane >> 4), 16 * rg + 8 * ((lane >> 3) & 1)),
             u);
      const float2 u0 = unpk<E>(u[0]), u1 = unpk<E>(u[1]), u2 = unpk<E>(u[2]),
                   u3 = unpk<E>(u[3]);
      wa[kk][0] = pk<E>(u0.x + zy[2 * kk][0], u0.y + zy[2 * kk][1]);
      wa[kk][1] = pk<E>(u1.x + zy[2 * kk][2], u1.y + zy[2 * kk][3]);
      wa[kk][2] = pk<E>(u2.x + zy[2 * kk + 1][0], u2.y + zy[2 * kk + 1][1]);
      wa[kk][3] = pk<E>(u3.x + zy[2 * kk + 1][2], u3.y + zy[2 * kk + 1][3]);
    }
#pragma unroll
    for (int jn = 0; jn < 16; ++jn)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[jn][e] *= gcv;
#pragma unroll
    for (int kk = 0; kk < NK16; ++kk)
#pragma unroll
      for (int jn = 0; jn < 16; ++jn) {
        uint32_t bb[2];
        ldsm2t(ba + seg_off(kRowsA, 2 * kC + 16 * kk + (lane & 15), 128 * kh + 8 * jn), bb);
        mma<E>(s[jn], wa[kk], bb);
      }
    // y = y_loc + Y for this row group's 16 value columns (the key-half-0 warp).
    if (kh == 0) {
      const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int nn = 0; nn < NT8; nn += 2) {
        const int t = 8 * (nn + (mi >> 1)) + r8, vv = 16 * rg + 8 * (mi & 1);
        stsm4t(s_u32(&sm.ys[t][vv]), pk<E>(zy[NT8 + nn][0], zy[NT8 + nn][1]),
               pk<E>(zy[NT8 + nn][2], zy[NT8 + nn][3]),
               pk<E>(zy[NT8 + nn + 1][0], zy[NT8 + nn + 1][1]),
               pk<E>(zy[NT8 + nn + 1][2], zy[NT8 + nn + 1][3]));
      }
      __syncwarp();
      const uint8_t* pb = reinterpret_cast<const uint8_t*>(sm.stage_b[st]);
#pragma unroll
      for (int i = lane; i < kC * 2; i += 32) {
        const int t = i >> 1, c8 = 16 * rg + 8 * (i & 1), tt = j * kC + t;
        if (tt < T) {
          const uint4 yl = *reinterpret_cast<const uint4*>(pb + sw64(kC + t, c8));
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
          *reinterpret_cast<uint4*>(y + (((size_t)b * T + tt) * Hv + hv) * kD + 64 * qt + c8) = o;
        }
      }
    }
    __syncwarp();  // this warp is done with the stage (and its ys columns)
    if (lane == 0) ptx::mbar_arrive(s_u32(&sm.empty[st]));
  }
  float* dst = state_out + (size_t)bh * kD * kD;
#pragma unroll
  for (int jn = 0; jn < 16; ++jn) {
    const int c = 128 * kh + 8 * jn + 2 * cq;
    __stcs(reinterpret_cast<float2*>(dst + (size_t)r0 * kD + c), make_float2(s[jn][0], s[jn][1]));
    __stcs(reinterpret_cast<float2*>(dst + (size_t)(r0 + 8) * kD + c),
           make_float2(s[jn][2], s[jn][3]));
  }
}

// Tokens [B, T, H, 256] of 16-bit type dt seen as {64 columns, T, 4 segments,
// H, B}, box {64, C, 4, 1, 1}: one head's chunk, landing as [seg][t][64],
// 128-byte swizzle; tokens past T read as zeros.
bool make_token_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int B, int T,
                    int H) {
  const TmapEncodeFn enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t dims[5] = {64, (cuuint64_t)T, 4, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[4] = {(cuuint64_t)H * kD * 2, 128, (cuuint64_t)kD * 2,
                                 (cuuint64_t)T * H * kD * 2};
  const cuuint32_t box[5] = {64, (cuuint32_t)kC, 4, 1, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, dt, 5, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// The workspace rows of 256 seen as {64 columns, rows, 4 segments}: box {64,
// rows_box, segs_box}, landing as [seg][row][64], 128-byte swizzle.
bool make_ws_map(CUtensorMap* m, CUtensorMapDataType dt, void* base, size_t rows, int rows_box,
                 int segs_box) {
  const TmapEncodeFn enc = tmap_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, 4};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)rows_box, (cuuint32_t)segs_box};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename E>
cudaError_t launch_mma256(const PrefillArgs& a) {
  const int NC = (a.T + kC - 1) / kC, BH = a.B * a.Hv;
  const size_t blocks = (size_t)BH * NC;
  E* ws = static_cast<E*>(a.workspace);
  float* wsgc =
      reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + blocks * kBlkElems * 2);
  constexpr CUtensorMapDataType dt = std::is_same_v<E, __half> ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tm_k{}, tm_q{}, tm_v{}, tm_wa{}, tm_wb{};
  if (!make_token_map(&tm_k, dt, a.k, a.B, a.T, a.Hk) ||
      !make_token_map(&tm_q, dt, a.q, a.B, a.T, a.Hk) ||
      !make_token_map(&tm_v, dt, a.v, a.B, a.T, a.Hv) ||
      !make_ws_map(&tm_wa, dt, ws, blocks * kBlkRows, kRowsA, 4) ||
      !make_ws_map(&tm_wb, dt, ws, blocks * kBlkRows, 2 * kC, 1))
    return cudaErrorInvalidValue;
  const int smem_p = (int)sizeof(PrepSmem<E>) + kAlign;
  const int smem_s = (int)sizeof(ScanSmem<E>) + kAlign;
  cudaError_t e = cudaFuncSetAttribute(mma256_prep_kernel<E>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_p);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(mma256_scan_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_s);
  if (e != cudaSuccess) return e;
  const float scale = 1.0f / sqrtf((float)kD);
  mma256_prep_kernel<E><<<(unsigned)blocks, kPT, smem_p, a.stream>>>(
      tm_k, tm_q, tm_v, static_cast<const E*>(a.g), static_cast<const E*>(a.beta), ws, wsgc, a.T,
      a.Hk, a.Hv, NC, a.options, scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mma256_scan_kernel<E><<<4 * BH, kST, smem_s, a.stream>>>(
      tm_wa, tm_wb, wsgc, a.state_in, a.state_out, static_cast<E*>(a.y), a.T, a.Hv, NC);
  return cudaGetLastError();
}

}  // namespace

bool mma256_path_applies(int Dk, int Dv, int dtype, int T) {
  return (dtype == 1 || dtype == 2) && Dk == kD && Dv == kD && T > kShortT;
}

size_t prefill_mma256_workspace_bytes(int B, int T, int Hv) {
  const size_t blocks = (size_t)B * Hv * ((T + kC - 1) / kC);
  return blocks * kBlkElems * 2 + ((blocks * sizeof(float) + 255) & ~(size_t)255);
}

cudaError_t launch_prefill_mma256(const PrefillArgs& a) {
  return a.dtype == 2 ? launch_mma256<__half>(a) : launch_mma256<__nv_bfloat16>(a);
}

int prefill_mma256_device_error(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, ptx::g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int z = 0;
    if (cudaMemcpyToSymbol(ptx::g_device_error, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace gdn
