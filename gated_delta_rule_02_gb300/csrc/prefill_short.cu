// Short-T prefill: T <= kShortT tokens of every (b, hv) through the sequential
// rule with the state held on chip, read once and written once.
//
// The pages route short sequences to the row-packed sequential kernel rather
// than the chunked form (MLX PR "Pack gated_delta_seq: 8 value rows per
// SIMD-group", Performance, the short-T rows; ferrox-core `gdn_chunk.rs`,
// `DEVICE_ROWS`): below about a chunk of tokens the chunk machinery costs more
// than it saves.  Per value row r of S and token t (every row evolves on its
// own; ferrox-core "The algebra", one row):
//     x = S[r]·k_t,  z = S[r]·q_t
//     d = beta_t (v_t[r] - g_t x)
//     S[r] <- g_t S[r] + d k_t
//     y_t[r] = (g_t z + d (k_t·q_t)) / sqrt(Dk)      (= S_t[r]·q_t / sqrt(Dk))
//
// Layout: one CTA of four warps per (b, hv) head, each warp owning Dv/4 rows,
// eight lanes per row as in the decode kernel (Dk a template parameter, Dv a
// runtime one).  The CTA first stages the T tokens' k, q, v (as fp32), g, beta
// and k·q in shared memory; each warp then takes G row groups (4 rows each) at
// a time through all T tokens with their state in registers.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kShortThreads = 128;

// Two fp32 values in one 64-bit register, for the paired fp32 instructions of
// sm_100 and later (each lane of a pair rounds as the scalar instruction would).
using f32x2 = unsigned long long;
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ float sum2(f32x2 a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
  return lo + hi;
}
// A row slice of four floats as two pairs.
struct Row4 {
  f32x2 a, b;
};
__device__ __forceinline__ Row4 ld_state(const float* p) {
  const ulonglong2 v = __ldcg(reinterpret_cast<const ulonglong2*>(p));
  return Row4{v.x, v.y};
}
__device__ __forceinline__ void st_state(float* p, Row4 v) {
  __stcg(reinterpret_cast<ulonglong2*>(p), make_ulonglong2(v.a, v.b));
}

template <typename T, int DK, int G>
__global__ void __launch_bounds__(kShortThreads)
short_prefill_kernel(const T* __restrict__ q, const T* __restrict__ k,
                     const T* __restrict__ v, const T* __restrict__ g,
                     const T* __restrict__ beta, const float* state_in,
                     float* state_out, T* __restrict__ y, int Tlen, int Hk, int Hv, int Dv,
                     int opts, float scale) {
  constexpr int D = DK;
  constexpr int NJ = DK / 32;  // float4s of a row per lane
  extern __shared__ float4 smem_f4[];
  float* ks = reinterpret_cast<float*>(smem_f4);  // [Tlen][DK]
  float* qs = ks + Tlen * D;                      // [Tlen][DK]
  float* vs = qs + Tlen * D;                      // [Tlen][Dv]
  float* gs = vs + Tlen * Dv;                     // [Tlen]
  float* bs = gs + Tlen;                          // [Tlen]
  float* kqs = bs + Tlen;                         // [Tlen]

  const int bh = blockIdx.x;
  const int b = bh / Hv;
  const int hv = bh - b * Hv;
  const int hk = key_head(hv, Hk, Hv, opts);
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int rg = lane >> 3;   // row within a group of four
  const int sub = lane & 7;   // lane within the row

  // Stage the tokens: warp w takes rows t = w, w+4, ...; lane l loads the
  // elements 4l..4l+3 (+128, ...) of k and q and of v.
  for (int t = warp; t < Tlen; t += kShortThreads / 32) {
    const size_t kq_off = (((size_t)b * Tlen + t) * Hk + hk) * D;
    const size_t v_off = (((size_t)b * Tlen + t) * Hv + hv) * Dv;
    constexpr int NK = (DK + 127) / 128;  // 4-element pieces of a k row per lane
    float kk[NK][4], qq[NK][4];
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int p = 0; p < NK; ++p) {
      const int e = 4 * lane + 128 * p;
      if (e < DK) {
        load4(k + kq_off + e, kk[p]);
        load4(q + kq_off + e, qq[p]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) kk[p][i] = qq[p][i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sk = fmaf(kk[p][i], kk[p][i], sk);
        sq = fmaf(qq[p][i], qq[p][i], sq);
      }
    }
    if (opts & kOptL2NormQK) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
      }
      const float fk = inv_norm(sk), fq = inv_norm(sq);
#pragma unroll
      for (int p = 0; p < NK; ++p)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kk[p][i] *= fk;
          qq[p][i] *= fq;
        }
    }
    float kq = 0.f;
#pragma unroll
    for (int p = 0; p < NK; ++p) {
      const int e = 4 * lane + 128 * p;
      if (e < DK) {
        *reinterpret_cast<float4*>(ks + t * D + e) = make_float4(kk[p][0], kk[p][1], kk[p][2], kk[p][3]);
        *reinterpret_cast<float4*>(qs + t * D + e) = make_float4(qq[p][0], qq[p][1], qq[p][2], qq[p][3]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) kq = fmaf(kk[p][i], qq[p][i], kq);
    }
    for (int e = 4 * lane; e < Dv; e += 128) {
      float vv[4];
      load4(v + v_off + e, vv);
      *reinterpret_cast<float4*>(vs + t * Dv + e) = make_float4(vv[0], vv[1], vv[2], vv[3]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
    if (lane == 0) {
      const size_t gi = ((size_t)b * Tlen + t) * Hv + hv;
      kqs[t] = kq;
      gs[t] = decay_of(to_f32(g[gi]), opts);
      bs[t] = to_f32(beta[gi]);
    }
  }
  __syncthreads();

  const float* Sin = state_in ? state_in + (size_t)bh * Dv * D : nullptr;
  float* Sout = state_out + (size_t)bh * Dv * D;
  const int wrows = Dv / 4;  // rows per warp

  // The registers hold S scaled: S = gam * St, gam the product of the gates since
  // the last renormalisation (the same for every row of the head).  Then
  //     x = gam (St·k),  z = gam (St·q),  gn = gam g_t,
  //     d = beta_t (v_t[r] - gn (St·k)),   y_t[r] = gn (St·q) + d (k_t·q_t),
  //     St <- St + (d / gn) k_t,  gam <- gn,
  // one paired FMA per element pair instead of a multiply and an FMA.  When gn
  // leaves [2^-24, 2^24] (a zero gate included) the registers are brought back
  // to scale, St <- gn St + d k_t, gam <- 1: a branch that is uniform over the
  // CTA, since every row sees the same gates.
#pragma unroll 1
  for (int it = 0; it < wrows / (4 * G); ++it) {
    const int row0 = warp * wrows + it * 4 * G + rg;  // this lane's row in group gi: row0 + 4*gi
    Row4 s[G][NJ];
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        s[gi][j] = Sin ? ld_state(Sin + (size_t)(row0 + 4 * gi) * D + 4 * (sub + 8 * j))
                       : Row4{0ull, 0ull};
    float gam = 1.f;

#pragma unroll 1
    for (int t = 0; t < Tlen; ++t) {
      Row4 kr[NJ], qr[NJ];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(ks + t * D + 4 * (sub + 8 * j));
        const ulonglong2 c = *reinterpret_cast<const ulonglong2*>(qs + t * D + 4 * (sub + 8 * j));
        kr[j] = Row4{a.x, a.y};
        qr[j] = Row4{c.x, c.y};
      }
      const float gt = gs[t], bt = bs[t], kq = kqs[t];
      float x[G], z[G];
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        f32x2 xa = 0ull, za = 0ull;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          xa = fma2(s[gi][j].a, kr[j].a, xa);
          xa = fma2(s[gi][j].b, kr[j].b, xa);
          za = fma2(s[gi][j].a, qr[j].a, za);
          za = fma2(s[gi][j].b, qr[j].b, za);
        }
        x[gi] = sum2(xa);
        z[gi] = sum2(za);
      }
      const float gn = gam * gt;
      T* yt = y + (((size_t)b * Tlen + t) * Hv + hv) * Dv;
      if constexpr (G == 4) {
        // Sum the eight partial dot products of a lane (x and z of four rows)
        // over the row's eight lanes in a transposing butterfly: after it lane
        // `sub` holds the full x[sub] (sub < 4) or z[sub - 4].
        const bool b2 = (sub & 4) != 0, b1 = (sub & 2) != 0, b0 = (sub & 1) != 0;
        float h4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float keep = b2 ? z[i] : x[i], send = b2 ? x[i] : z[i];
          h4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        float h2[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float keep = b1 ? h4[2 + i] : h4[i], send = b1 ? h4[i] : h4[2 + i];
          h2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        const float own = (b0 ? h2[1] : h2[0]) + __shfl_xor_sync(0xffffffffu, b0 ? h2[0] : h2[1], 1);
        const int base = lane & ~7;
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) x[gi] = __shfl_sync(0xffffffffu, own, base | gi);
        // Lane 4 + gi owns z of row gi and stores that row's y.
        const float xo = __shfl_sync(0xffffffffu, own, base | (sub & 3));
        const int ro = row0 + 4 * (sub & 3);
        const float dd = bt * (vs[t * Dv + ro] - gn * xo);
        if (b2) yt[ro] = from_f32<T>(fmaf(gn, own, dd * kq) * scale);
      } else {
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
          const float dd = bt * (vs[t * Dv + row] - gn * x[gi]);
          if (sub == 0) yt[row] = from_f32<T>(fmaf(gn, z[gi], dd * kq) * scale);
        }
      }
      float d[G];
#pragma unroll
      for (int gi = 0; gi < G; ++gi) d[gi] = bt * (vs[t * Dv + row0 + 4 * gi] - gn * x[gi]);
      if (gn >= 0x1p-24f && gn <= 0x1p24f) {
        const float inv = 1.f / gn;
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
          const float c = d[gi] * inv;
          const f32x2 c2 = pack2(c, c);
#pragma unroll
          for (int j = 0; j < NJ; ++j) {  // St <- St + (d / gn) k
            s[gi][j].a = fma2(c2, kr[j].a, s[gi][j].a);
            s[gi][j].b = fma2(c2, kr[j].b, s[gi][j].b);
          }
        }
        gam = gn;
      } else {
        const f32x2 g2 = pack2(gn, gn);
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
          const f32x2 d2 = pack2(d[gi], d[gi]);
#pragma unroll
          for (int j = 0; j < NJ; ++j) {  // St <- gn St + d k
            s[gi][j].a = fma2(g2, s[gi][j].a, mul2(d2, kr[j].a));
            s[gi][j].b = fma2(g2, s[gi][j].b, mul2(d2, kr[j].b));
          }
        }
        gam = 1.f;
      }
    }
    const f32x2 gam2 = pack2(gam, gam);
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        st_state(Sout + (size_t)(row0 + 4 * gi) * D + 4 * (sub + 8 * j),
                 Row4{mul2(gam2, s[gi][j].a), mul2(gam2, s[gi][j].b)});
  }
}

size_t short_smem_bytes(int T, int Dk, int Dv) {
  return (size_t)T * (2 * Dk + Dv + 3) * sizeof(float);
}

template <typename T, int DK>
cudaError_t launch_short_t(const PrefillArgs& a) {
  constexpr int G = DK == 256 ? 1 : 4;  // row groups of a warp in flight (registers)
  const float scale = 1.0f / sqrtf((float)DK);
  const size_t smem = short_smem_bytes(a.T, DK, a.Dv);
  cudaError_t e = cudaFuncSetAttribute(short_prefill_kernel<T, DK, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  short_prefill_kernel<T, DK, G><<<a.B * a.Hv, kShortThreads, smem, a.stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
      static_cast<const T*>(a.g), static_cast<const T*>(a.beta), a.state_in, a.state_out,
      static_cast<T*>(a.y), a.T, a.Hk, a.Hv, a.Dv, a.options, scale);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_short_dk(const PrefillArgs& a) {
  if (a.Dk == 64) return launch_short_t<T, 64>(a);
  if (a.Dk == 256) return launch_short_t<T, 256>(a);
  return launch_short_t<T, 128>(a);
}

}  // namespace

cudaError_t launch_prefill_short(const PrefillArgs& a) {
  if (short_tc_applies(a)) return launch_prefill_short_tc(a);
  if (a.dtype == 0) return launch_short_dk<float>(a);
  if (a.dtype == 2) return launch_short_dk<__half>(a);
  return launch_short_dk<__nv_bfloat16>(a);
}

}  // namespace gdn
