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
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kLd = kHeadDim + 1;   // padded row stride of the [C][128] tiles
constexpr int kRows = 16;           // value rows of S per scan CTA

// Workspace per (b, hv, chunk): Ph, Qh [C][128] then Ut, Yl [C][128], fp32;
// followed by G_{C-1} for every (b, hv, chunk).
__host__ __device__ inline size_t chunk_block_floats(int C) {
  return (size_t)4 * C * kHeadDim;
}

template <typename T, int C>
__global__ void __launch_bounds__(kThreads)
intra_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                  const T* __restrict__ v, const T* __restrict__ g,
                  const T* __restrict__ beta, float* __restrict__ ws,
                  float* __restrict__ wsG, int T_, int Hk, int Hv, int N, int opts) {
  constexpr int D = kHeadDim;
  constexpr int LC = C + 1;
  extern __shared__ float sm[];
  float* sK = sm;               // K, then P (in place)
  float* sQ = sK + C * kLd;     // Q, then Qh (in place)
  float* sV = sQ + C * kLd;     // V, then U (in place)
  float* sKK = sV + C * kLd;    // [C][C+1]
  float* sQK = sKK + C * LC;
  float* sGam = sQK + C * LC;
  float* sG = sGam + C * LC;    // [C]
  float* sg = sG + C;
  float* sb = sg + C;

  const int n = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / Hv;
  const int hv = bh - b * Hv;
  const int hk = key_head(hv, Hk, Hv, opts);
  const int t0 = n * C;
  const int c = min(C, T_ - t0);
  const int tid = threadIdx.x;

  // Step 1: gather, padded to C rows.
  for (int idx = tid; idx < C * D; idx += kThreads) {
    const int t = idx / D, d = idx % D;
    float kv = 0.f, qv = 0.f, vv = 0.f;
    if (t < c) {
      const size_t tok = (size_t)b * T_ + t0 + t;
      kv = to_f32(k[(tok * Hk + hk) * D + d]);
      qv = to_f32(q[(tok * Hk + hk) * D + d]);
      vv = to_f32(v[(tok * Hv + hv) * D + d]);
    }
    sK[t * kLd + d] = kv;
    sQ[t * kLd + d] = qv;
    sV[t * kLd + d] = vv;
  }
  for (int t = tid; t < C; t += kThreads) {
    const size_t tok = (size_t)b * T_ + t0 + t;
    sg[t] = t < c ? decay_of(to_f32(g[tok * Hv + hv]), opts) : 1.f;
    sb[t] = t < c ? to_f32(beta[tok * Hv + hv]) : 0.f;
  }
  __syncthreads();
  if (opts & kOptL2NormQK) {
    l2norm_rows_f32(sK, c, kLd, tid, kThreads);
    l2norm_rows_f32(sQ, c, kLd, tid, kThreads);
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
    for (int d = 0; d < D; ++d) {
      const float kj = sK[j * kLd + d];
      kk = fmaf(sK[t * kLd + d], kj, kk);
      qk = fmaf(sQ[t * kLd + d], kj, qk);
    }
    sKK[t * LC + j] = kk;
    sQK[t * LC + j] = qk;
  }
  __syncthreads();

  // Steps 4 and 5: forward substitution, one column per thread, in place.
  // Threads 0..127 solve (I + L) P = K, threads 128..255 (I + A) U = beta V.
  {
    const int d = tid & (D - 1);
    if (tid < D) {
      for (int t = 1; t < C; ++t) {
        float acc = sK[t * kLd + d];
        for (int j = 0; j < t; ++j) acc = fmaf(-sb[j] * sKK[t * LC + j], sK[j * kLd + d], acc);
        sK[t * kLd + d] = acc;
      }
    } else {
      sV[d] = sb[0] * sV[d];
      for (int t = 1; t < C; ++t) {
        const float bt = sb[t];
        float acc = bt * sV[t * kLd + d];
        for (int j = 0; j < t; ++j)
          acc = fmaf(-bt * sGam[t * LC + j] * sKK[t * LC + j], sV[j * kLd + d], acc);
        sV[t * kLd + d] = acc;
      }
    }
  }
  __syncthreads();

  // Steps 6, 7 (state-free part) and 9 (state-free part); write the block.
  float* blk = ws + ((size_t)bh * N + n) * chunk_block_floats(C);
  float* wPh = blk;
  float* wQh = blk + C * D;
  float* wUt = blk + 2 * C * D;
  float* wYl = blk + 3 * C * D;
  {
    const int d = tid & (D - 1);
    const float Gc = sG[C - 1];
    if (tid < D) {
      for (int t = 0; t < C; ++t) {
        float acc = sQ[t * kLd + d];
        for (int i = 0; i <= t; ++i) acc = fmaf(-sb[i] * sQK[t * LC + i], sK[i * kLd + d], acc);
        wQh[t * D + d] = sG[t] * acc;
        wPh[t * D + d] = Gc * sb[t] * sK[t * kLd + d];
      }
    } else {
      for (int t = 0; t < C; ++t) {
        float acc = 0.f;
        for (int j = 0; j <= t; ++j) acc = fmaf(sGam[t * LC + j] * sQK[t * LC + j], sV[j * kLd + d], acc);
        wYl[t * D + d] = acc;
        wUt[t * D + d] = sGam[(C - 1) * LC + t] * sV[t * kLd + d];
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
                 int N, int opts, float scale) {
  constexpr int D = kHeadDim;
  constexpr int R = kRows;
  extern __shared__ float sm[];
  float* sS = sm;                  // [R][128]
  float* sPQ = sS + R * D;         // [2C][129]: rows 0..C-1 Ph, C..2C-1 Qh
  float* sK = sPQ + 2 * C * kLd;   // [C][128]
  float* sUt = sK + C * D;         // [C][R]
  float* sYl = sUt + C * R;        // [C][R]
  float* sW = sYl + C * R;         // [R][C]

  const int tile = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / Hv;
  const int hv = bh - b * Hv;
  const int hk = key_head(hv, Hk, Hv, opts);
  const int r0 = tile * R;
  const int tid = threadIdx.x;
  const size_t sbase = (size_t)bh * D * D + (size_t)r0 * D;

  for (int idx = tid; idx < R * D; idx += kThreads)
    sS[idx] = state_in ? state_in[sbase + idx] : 0.f;

  for (int n = 0; n < N; ++n) {
    const int t0 = n * C;
    const int c = min(C, T_ - t0);
    const float* blk = ws + ((size_t)bh * N + n) * chunk_block_floats(C);
    __syncthreads();  // previous chunk's readers of sPQ/sK/sW are done
    for (int idx = tid; idx < 2 * C * D; idx += kThreads)
      sPQ[(idx / D) * kLd + idx % D] = blk[idx];
    for (int idx = tid; idx < C * D; idx += kThreads) {
      const int t = idx / D, d = idx % D;
      sK[idx] = t < c ? to_f32(k[(((size_t)b * T_ + t0 + t) * Hk + hk) * D + d]) : 0.f;
    }
    for (int idx = tid; idx < C * R; idx += kThreads) {
      const int t = idx / R, r = idx % R;
      sUt[idx] = blk[2 * C * D + t * D + r0 + r];
      sYl[idx] = blk[3 * C * D + t * D + r0 + r];
    }
    const float Gc = wsG[(size_t)bh * N + n];
    __syncthreads();
    if (opts & kOptL2NormQK) {
      l2norm_rows_f32(sK, c, D, tid, kThreads);
      __syncthreads();
    }

    // [SP | SQ][r][t'] = S[r] . PQ[t'], t' < 2C.
    for (int idx = tid; idx < R * 2 * C; idx += kThreads) {
      const int tp = idx % (2 * C), r = idx / (2 * C);
      float acc = 0.f;
      for (int d = 0; d < D; ++d) acc = fmaf(sS[r * D + d], sPQ[tp * kLd + d], acc);
      if (tp < C) {
        sW[r * C + tp] = sUt[tp * R + r] - acc;
      } else {
        const int t = tp - C;
        if (t < c)
          y[(((size_t)b * T_ + t0 + t) * Hv + hv) * D + r0 + r] =
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

template <int C>
size_t intra_smem_bytes() {
  return sizeof(float) * (3 * C * kLd + 3 * C * (C + 1) + 3 * C);
}
template <int C>
size_t scan_smem_bytes() {
  return sizeof(float) * (kRows * kHeadDim + 2 * C * kLd + C * kHeadDim +
                          2 * C * kRows + kRows * C);
}

template <typename T, int C>
cudaError_t launch_t(const PrefillArgs& a) {
  const int N = (a.T + C - 1) / C;
  const int BH = a.B * a.Hv;
  float* ws = static_cast<float*>(a.workspace);
  float* wsG = ws + (size_t)BH * N * chunk_block_floats(C);
  const size_t smem_i = intra_smem_bytes<C>();
  const size_t smem_s = scan_smem_bytes<C>();
  cudaError_t e = cudaFuncSetAttribute(intra_simt_kernel<T, C>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_i);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(scan_simt_kernel<T, C>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_s);
  if (e != cudaSuccess) return e;
  intra_simt_kernel<T, C><<<dim3(N, BH), kThreads, smem_i, a.stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k),
      static_cast<const T*>(a.v), static_cast<const T*>(a.g),
      static_cast<const T*>(a.beta), ws, wsG, a.T, a.Hk, a.Hv, N, a.options);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float scale = 1.0f / sqrtf((float)kHeadDim);
  scan_simt_kernel<T, C><<<dim3(kHeadDim / kRows, BH), kThreads, smem_s, a.stream>>>(
      static_cast<const T*>(a.k), ws, wsG, a.state_in, a.state_out,
      static_cast<T*>(a.y), a.T, a.Hk, a.Hv, N, a.options, scale);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dtype(const PrefillArgs& a) {
  switch (a.chunk) {
    case 16: return launch_t<T, 16>(a);
    case 32: return launch_t<T, 32>(a);
    default: return launch_t<T, 64>(a);
  }
}

}  // namespace

size_t prefill_simt_workspace_bytes(int B, int T, int Hv, int chunk) {
  const size_t N = ((size_t)T + chunk - 1) / chunk;
  const size_t BH = (size_t)B * Hv;
  size_t bytes = sizeof(float) * (BH * N * chunk_block_floats(chunk) + BH * N);
  return (bytes + 255) & ~(size_t)255;
}

cudaError_t launch_prefill_simt(const PrefillArgs& a) {
  if (a.dtype == 0) return launch_dtype<float>(a);
  if (a.dtype == 2) return launch_dtype<__half>(a);
  return launch_dtype<__nv_bfloat16>(a);
}

}  // namespace gdn
