// Chunked prefill on CUDA cores, all arithmetic in fp32.
//
// This is the exact path for fp32 inputs (and a general fallback-free path
// for any dtype).  It follows the chunked Woodbury-Young form of
// metaltile-std `gated_delta_wy.rs` (module docs, "Algorithm", steps 1-9),
// regrouped so that everything that does not depend on the carried state is
// computed once per chunk, in parallel over all chunks, and the sequential
// scan over chunks only touches the state:
//
//   intra kernel, one CTA per (b, hv, chunk n), chunk rows t = 0..C-1:
//     G_t        = g_0 ... g_t                     (step 2, prefix gates)
//     Gam[t][j]  = g_{j+1} ... g_t, j <= t          (step 2, ratios as products:
//                                                    ferrox-core "The algebra")
//     KK^T, QK^T                                    (steps 3, 6-prep)
//     (I + L) P = K,        L[t][j] = beta_j KK^T[t][j], j < t        (step 4)
//     (I + A) U = beta V,   A[t][j] = beta_t Gam[t][j] KK^T[t][j]     (step 5)
//     y_loc[t]  = sum_{j<=t} Gam[t][j] QK^T[t][j] U[j]                (step 6)
//     Qh[t]     = G_t (q_t - sum_{i<=t} beta_i QK^T[t][i] P[i])        (step 7, S-free part)
//     Ph[j]     = G_{C-1} beta_j P[j]                                  (step 9, S-free part)
//     Ut[j]     = Gam[C-1][j] U[j]                                     (step 9)
//   scan kernel, one CTA per (b, hv, tile of R value rows), chunk by chunk:
//     SP = S Ph^T, SQ = S Qh^T
//     y[t]  = (SQ[:, t] + y_loc[t]) / sqrt(Dk)                         (steps 7-8)
//     S    <- G_{C-1} S + (Ut^T - SP) K                               (step 9)
// A last chunk shorter than C is padded with g = 1, beta = 0, q = k = v = 0
// (metaltile-std kernel, chunk-loop precondition), which changes nothing.
// The head sizes Dk, Dv (64, 128 or 256) are runtime values here.  When a
// chunk of C = 64 rows of Dk = Dv = 256 would not fit in shared memory, the
// chunks are split in two (C = 32): the chunk size changes the result only
// by rounding.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;           // value rows of S per scan CTA
constexpr size_t kMaxSmem = 227 * 1024;

// Workspace per (b, hv, chunk): Ph, Qh [C][Dk] then Ut, Yl [C][Dv], fp32;
// followed by G_{C-1} for every (b, hv, chunk).
__host__ __device__ inline size_t chunk_block_floats(int C, int Dk, int Dv) {
  return (size_t)2 * C * (Dk + Dv);
}
size_t intra_smem_bytes(int C, int Dk, int Dv) {
  return sizeof(float) * ((size_t)C * (2 * (Dk + 1) + (Dv + 1)) + 3 * C * (C + 1) + 3 * C);
}
size_t scan_smem_bytes(int C, int Dk) {
  return sizeof(float) * ((size_t)kRows * Dk + 2 * C * (Dk + 1) + (size_t)C * Dk + 3 * C * kRows);
}
// The chunk size the kernels run: the requested one unless its tiles do not fit.
int simt_chunk(int chunk, int Dk, int Dv) {
  while (chunk > 16 && (intra_smem_bytes(chunk, Dk, Dv) > kMaxSmem ||
                        scan_smem_bytes(chunk, Dk) > kMaxSmem))
    chunk /= 2;
  return chunk;
}

template <typename T, int C>
__global__ void __launch_bounds__(kThreads)
intra_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                  const T* __restrict__ v, const T* __restrict__ g,
                  const T* __restrict__ beta, float* __restrict__ ws,
                  float* __restrict__ wsG, int T_, int Hk, int Hv, int N, int Dk, int Dv,
                  int opts) {
  constexpr int LC = C + 1;
  const int ldk = Dk + 1, ldv = Dv + 1;  // padded row strides
  extern __shared__ float sm[];
  float* sK = sm;               // K, then P (in place)
  float* sQ = sK + C * ldk;     // Q, then Qh (in place)
  float* sV = sQ + C * ldk;     // V, then U (in place)
  float* sKK = sV + C * ldv;    // [C][C+1]
  float* sQK = sKK + C * LC;
  float* sGam = sQK + C * LC;
  float* sG = sGam + C * LC;    // [C]
  float* sg = sG + C;
  float* sb = sg + C;

  // One-dimensional grid (chunk fastest): blockIdx.x = n + N bh, so B Hv is not
  // held to the 65535 blocks of a grid's y dimension.
  const int n = blockIdx.x % N;
  const int bh = blockIdx.x / N;
  const int b = bh / Hv;
  const int hv = bh - b * Hv;
  const int hk = key_head(hv, Hk, Hv, opts);
  const int t0 = n * C;
  const int c = min(C, T_ - t0);
  const int tid = threadIdx.x;

  // Step 1: gather, padded to C rows.
  for (int idx = tid; idx < C * Dk; idx += kThreads) {
    const int t = idx / Dk, d = idx % Dk;
    float kv = 0.f, qv = 0.f;
    if (t < c) {
      const size_t tok = (size_t)b * T_ + t0 + t;
      kv = to_f32(k[(tok * Hk + hk) * Dk + d]);
      qv = to_f32(q[(tok * Hk + hk) * Dk + d]);
    }
    sK[t * ldk + d] = kv;
    sQ[t * ldk + d] = qv;
  }
  for (int idx = tid; idx < C * Dv; idx += kThreads) {
    const int t = idx / Dv, d = idx % Dv;
    sV[t * ldv + d] = t < c ? to_f32(v[(((size_t)b * T_ + t0 + t) * Hv + hv) * Dv + d]) : 0.f;
  }
  for (int t = tid; t < C; t += kThreads) {
    const size_t tok = (size_t)b * T_ + t0 + t;
    sg[t] = t < c ? decay_of(to_f32(g[tok * Hv + hv]), opts) : 1.f;
    sb[t] = t < c ? to_f32(beta[tok * Hv + hv]) : 0.f;
  }
  __syncthreads();
  if (opts & kOptL2NormQK) {
    l2norm_rows_f32(sK, c, Dk, ldk, tid, kThreads);
    l2norm_rows_f32(sQ, c, Dk, ldk, tid, kThreads);
    __syncthreads();
  }

  // Step 2: prefix gates and decay ratios, both as products.
  if (tid < C) {
    const int t = tid;
    float acc = 1.f;
    for (int i = 0; i <= t; ++i) acc *= sg[i];
    sG[t] = acc;
    float r = 1.f;
    sGam[t * LC + t] = 1.f;
    for (int j = t - 1; j >= 0; --j) {
      r *= sg[j + 1];
      sGam[t * LC + j] = r;
    }
    for (int j = t + 1; j < C; ++j) sGam[t * LC + j] = 0.f;
  }
  // Step 3 (and 6-prep): KK^T and QK^T.
  for (int idx = tid; idx < C * C; idx += kThreads) {
    const int t = idx % C, j = idx / C;
    float kk = 0.f, qk = 0.f;
    for (int d = 0; d < Dk; ++d) {
      const float kj = sK[j * ldk + d];
      kk = fmaf(sK[t * ldk + d], kj, kk);
      qk = fmaf(sQ[t * ldk + d], kj, qk);
    }
    sKK[t * LC + j] = kk;
    sQK[t * LC + j] = qk;
  }
  __syncthreads();

  // Steps 4 and 5: forward substitution, one column per thread and step, in
  // place.  Threads 0..127 solve (I + L) P = K (columns d, d + 128, ... < Dk),
  // threads 128..255 (I + A) U = beta V (columns < Dv).
  if (tid < 128) {
    for (int d = tid; d < Dk; d += 128) {
      for (int t = 1; t < C; ++t) {
        float acc = sK[t * ldk + d];
        for (int j = 0; j < t; ++j) acc = fmaf(-sb[j] * sKK[t * LC + j], sK[j * ldk + d], acc);
        sK[t * ldk + d] = acc;
      }
    }
  } else {
    for (int d = tid - 128; d < Dv; d += 128) {
      sV[d] = sb[0] * sV[d];
      for (int t = 1; t < C; ++t) {
        const float bt = sb[t];
        float acc = bt * sV[t * ldv + d];
        for (int j = 0; j < t; ++j)
          acc = fmaf(-bt * sGam[t * LC + j] * sKK[t * LC + j], sV[j * ldv + d], acc);
        sV[t * ldv + d] = acc;
      }
    }
  }
  __syncthreads();

  // Steps 6, 7 (state-free part) and 9 (state-free part); write the block.
  float* blk = ws + ((size_t)bh * N + n) * chunk_block_floats(C, Dk, Dv);
  float* wPh = blk;
  float* wQh = blk + C * Dk;
  float* wUt = blk + 2 * C * Dk;
  float* wYl = wUt + C * Dv;
  {
    const float Gc = sG[C - 1];
    if (tid < 128) {
      for (int d = tid; d < Dk; d += 128) {
        for (int t = 0; t < C; ++t) {
          float acc = sQ[t * ldk + d];
          for (int i = 0; i <= t; ++i) acc = fmaf(-sb[i] * sQK[t * LC + i], sK[i * ldk + d], acc);
          wQh[t * Dk + d] = sG[t] * acc;
          wPh[t * Dk + d] = Gc * sb[t] * sK[t * ldk + d];
        }
      }
    } else {
      for (int d = tid - 128; d < Dv; d += 128) {
        for (int t = 0; t < C; ++t) {
          float acc = 0.f;
          for (int j = 0; j <= t; ++j)
            acc = fmaf(sGam[t * LC + j] * sQK[t * LC + j], sV[j * ldv + d], acc);
          wYl[t * Dv + d] = acc;
          wUt[t * Dv + d] = sGam[(C - 1) * LC + t] * sV[t * ldv + d];
        }
      }
    }
    if (tid == 0) wsG[(size_t)bh * N + n] = Gc;
  }
}

template <typename T, int C>
__global__ void __launch_bounds__(kThreads)
scan_simt_kernel(const T* __restrict__ k, const float* __restrict__ ws,
                 const float* __restrict__ wsG, const float* state_in,
                 float* state_out, T* __restrict__ y, int T_, int Hk, int Hv,
                 int N, int Dk, int Dv, int opts, float scale) {
  constexpr int R = kRows;
  const int D = Dk, ldk = Dk + 1;
  extern __shared__ float sm[];
  float* sS = sm;                  // [R][Dk]
  float* sPQ = sS + R * D;         // [2C][Dk + 1]: rows 0..C-1 Ph, C..2C-1 Qh
  float* sK = sPQ + 2 * C * ldk;   // [C][Dk]
  float* sUt = sK + C * D;         // [C][R]
  float* sYl = sUt + C * R;        // [C][R]
  float* sW = sYl + C * R;         // [R][C]

  // One-dimensional grid (row tile fastest): blockIdx.x = tile + (Dv / R) bh.
  const int tiles = Dv / R;
  const int tile = blockIdx.x % tiles;
  const int bh = blockIdx.x / tiles;
  const int b = bh / Hv;
  const int hv = bh - b * Hv;
  const int hk = key_head(hv, Hk, Hv, opts);
  const int r0 = tile * R;
  const int tid = threadIdx.x;
  const size_t sbase = ((size_t)bh * Dv + r0) * D;

  for (int idx = tid; idx < R * D; idx += kThreads)
    sS[idx] = state_in ? state_in[sbase + idx] : 0.f;

  for (int n = 0; n < N; ++n) {
    const int t0 = n * C;
    const int c = min(C, T_ - t0);
    const float* blk = ws + ((size_t)bh * N + n) * chunk_block_floats(C, Dk, Dv);
    __syncthreads();  // previous chunk's readers of sPQ/sK/sW are done
    for (int idx = tid; idx < 2 * C * D; idx += kThreads)
      sPQ[(idx / D) * ldk + idx % D] = blk[idx];
    for (int idx = tid; idx < C * D; idx += kThreads) {
      const int t = idx / D, d = idx % D;
      sK[idx] = t < c ? to_f32(k[(((size_t)b * T_ + t0 + t) * Hk + hk) * D + d]) : 0.f;
    }
    for (int idx = tid; idx < C * R; idx += kThreads) {
      const int t = idx / R, r = idx % R;
      sUt[idx] = blk[2 * C * D + t * Dv + r0 + r];
      sYl[idx] = blk[2 * C * D + C * Dv + t * Dv + r0 + r];
    }
    const float Gc = wsG[(size_t)bh * N + n];
    __syncthreads();
    if (opts & kOptL2NormQK) {
      l2norm_rows_f32(sK, c, D, D, tid, kThreads);
      __syncthreads();
    }

    // [SP | SQ][r][t'] = S[r] . PQ[t'], t' < 2C.
    for (int idx = tid; idx < R * 2 * C; idx += kThreads) {
      const int tp = idx % (2 * C), r = idx / (2 * C);
      float acc = 0.f;
      for (int d = 0; d < D; ++d) acc = fmaf(sS[r * D + d], sPQ[tp * ldk + d], acc);
      if (tp < C) {
        sW[r * C + tp] = sUt[tp * R + r] - acc;
      } else {
        const int t = tp - C;
        if (t < c)
          y[(((size_t)b * T_ + t0 + t) * Hv + hv) * Dv + r0 + r] =
              from_f32<T>((acc + sYl[t * R + r]) * scale);
      }
    }
    __syncthreads();
    // S <- G_{C-1} S + W K.
    for (int idx = tid; idx < R * D; idx += kThreads) {
      const int d = idx % D, r = idx / D;
      float acc = 0.f;
      for (int j = 0; j < C; ++j) acc = fmaf(sW[r * C + j], sK[j * D + d], acc);
      sS[idx] = fmaf(Gc, sS[idx], acc);
    }
  }
  __syncthreads();
  for (int idx = tid; idx < R * D; idx += kThreads) state_out[sbase + idx] = sS[idx];
}

template <typename T, int C>
cudaError_t launch_t(const PrefillArgs& a) {
  const int N = (a.T + C - 1) / C;
  const int BH = a.B * a.Hv;
  // One block per (chunk, head) and per (row tile, head) on a 1-D grid.
  if ((long long)N * BH > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  float* ws = static_cast<float*>(a.workspace);
  float* wsG = ws + (size_t)BH * N * chunk_block_floats(C, a.Dk, a.Dv);
  const size_t smem_i = intra_smem_bytes(C, a.Dk, a.Dv);
  const size_t smem_s = scan_smem_bytes(C, a.Dk);
  cudaError_t e = cudaFuncSetAttribute(intra_simt_kernel<T, C>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_i);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(scan_simt_kernel<T, C>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_s);
  if (e != cudaSuccess) return e;
  intra_simt_kernel<T, C><<<(unsigned)(N * BH), kThreads, smem_i, a.stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k),
      static_cast<const T*>(a.v), static_cast<const T*>(a.g),
      static_cast<const T*>(a.beta), ws, wsG, a.T, a.Hk, a.Hv, N, a.Dk, a.Dv, a.options);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float scale = 1.0f / sqrtf((float)a.Dk);
  scan_simt_kernel<T, C><<<(unsigned)(a.Dv / kRows * BH), kThreads, smem_s, a.stream>>>(
      static_cast<const T*>(a.k), ws, wsG, a.state_in, a.state_out,
      static_cast<T*>(a.y), a.T, a.Hk, a.Hv, N, a.Dk, a.Dv, a.options, scale);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dtype(const PrefillArgs& a) {
  switch (simt_chunk(a.chunk, a.Dk, a.Dv)) {
    case 16: return launch_t<T, 16>(a);
    case 32: return launch_t<T, 32>(a);
    default: return launch_t<T, 64>(a);
  }
}

}  // namespace

size_t prefill_simt_workspace_bytes(int B, int T, int Hv, int chunk, int Dk, int Dv) {
  chunk = simt_chunk(chunk, Dk, Dv);
  const size_t N = ((size_t)T + chunk - 1) / chunk;
  const size_t BH = (size_t)B * Hv;
  size_t bytes = sizeof(float) * (BH * N * chunk_block_floats(chunk, Dk, Dv) + BH * N);
  return (bytes + 255) & ~(size_t)255;
}

cudaError_t launch_prefill_simt(const PrefillArgs& a) {
  if (a.dtype == 0) return launch_dtype<float>(a);
  if (a.dtype == 2) return launch_dtype<__half>(a);
  return launch_dtype<__nv_bfloat16>(a);
}

}  // namespace gdn
