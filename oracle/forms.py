"""Independent fp64 NumPy restatements of the gated delta rule.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  These exist to pin
the sequential oracle to something other than itself: each is a different
expression of the same recurrence, so a dropped term, a wrong index or a
transposed operand in one of them shows up as a disagreement.

``chunked_wy``    metaltile-std ``gated_delta_wy.rs``, module docs,
                  "Algorithm (per chunk of size C)", steps 1-9: prefix gates,
                  ratio matrix, KK^T, the two unit-lower-triangular solves
                  (I+L)p = K and (I+A)u = beta*V, the local and pass-through
                  outputs and the chunk-end state.
``chunked_single_solve``
                  ferrox-core ``gdn_chunk.rs``, module docs, "The algebra"
                  (the unrolled chunk identities with decay products R[t][u]
                  and no division) and ``delta_chunk``'s forward substitution
                  for the per-row updates d_t.
``product_form``  the closed form obtained by unrolling S_t = g_t S_{t-1}
                  (I - beta_t k_t k_t^T) + beta_t v_t k_t^T into explicit
                  Dk x Dk matrix products.  Cost O(T^2 Dk^3): tiny cases only.

Readings taken where the pages leave a step open:
  * the ratio Gamma[t, j] = G_t / G_j of step 2 is formed as the product
    g_{j+1} ... g_t (ferrox-core "The algebra": products, never quotients),
    which is equal in exact arithmetic and cannot divide by an underflowed
    prefix;
  * a tail chunk shorter than C is padded with g = 1, beta = 0 and zero
    q, k, v rows (metaltile-std kernel, chunk-loop precondition), which
    leaves the recurrence unchanged;
  * the output carries the 1/sqrt(Dk) scale of ferrox-core "The algebra".
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _f64(x):
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _unpack(q, k, v, g, beta, s0):
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    if s0 is None:
        s0 = np.zeros((B, Hv, Dv, Dk))
    return q, k, v, g, beta, _f64(s0), (B, T, Hk, Hv, Dk, Dv)


def _gate_ratios(gc: np.ndarray) -> np.ndarray:
    """Gamma[t, j] = g_{j+1} * ... * g_t for j <= t (1 on the diagonal), 0 above."""
    C = gc.shape[0]
    gam = np.zeros((C, C))
    for t in range(C):
        gam[t, t] = 1.0
        for j in range(t - 1, -1, -1):
            gam[t, j] = gam[t, j + 1] * gc[j + 1]
    return gam


def chunked_wy(q, k, v, g, beta, s0=None, chunk=32, dtype=np.float64):
    """Chunked Woodbury-Young form, steps 1-9 of metaltile-std ``gated_delta_wy.rs``.

    ``dtype`` is the arithmetic type: float64 for the pins; float32 gives the
    fp32 host chunked form the pages time against the sequential one
    (ferrox-core ``gdn_chunk.rs``, ``CHUNK``), used only as a CPU baseline.
    """
    q, k, v, g, beta, s0, (B, T, Hk, Hv, Dk, Dv) = _unpack(q, k, v, g, beta, s0)
    if dtype != np.float64:
        q, k, v, g, beta, s0 = (a.astype(dtype) for a in (q, k, v, g, beta, s0))
    C = chunk
    group = Hv // Hk
    y = np.zeros((B, T, Hv, Dv), dtype=dtype)
    s_out = np.zeros((B, Hv, Dv, Dk), dtype=dtype)
    eye = np.eye(C, dtype=dtype)
    for b in range(B):
        for hv in range(Hv):
            hk = hv // group
            S = s0[b, hv].copy()
            for start in range(0, T, C):
                n = min(C, T - start)
                # Step 1: gather the chunk, padded to C rows with g=1, beta=0.
                Q = np.zeros((C, Dk), dtype=dtype); K = np.zeros((C, Dk), dtype=dtype)
                V = np.zeros((C, Dv), dtype=dtype)
                gc = np.ones(C, dtype=dtype); bc = np.zeros(C, dtype=dtype)
                Q[:n] = q[b, start:start + n, hk]
                K[:n] = k[b, start:start + n, hk]
                V[:n] = v[b, start:start + n, hv]
                gc[:n] = g[b, start:start + n, hv]
                bc[:n] = beta[b, start:start + n, hv]
                # Step 2: prefix gates and their ratios.
                G = np.cumprod(gc)
                gam = _gate_ratios(gc).astype(dtype)
                # Step 3: KK^T.
                kkt = K @ K.T
                # Step 4: (I + L) p = K, L[t, j] = beta_j KK^T[t, j] for j < t.
                L = np.tril(kkt * bc[None, :], -1)
                P = solve_triangular(eye + L, K, lower=True, unit_diagonal=True)
                # Step 5: (I + A) u = beta * V, A[t, j] = beta_t Gamma[t, j] KK^T[t, j].
                A = np.tril(bc[:, None] * gam * kkt, -1)
                U = solve_triangular(eye + A, bc[:, None] * V, lower=True,
                                     unit_diagonal=True)
                # Step 6: y_local[t] = sum_{j<=t} Gamma[t, j] QK^T[t, j] u_j.
                qkt = Q @ K.T
                y_local = np.tril(gam * qkt) @ U
                # Step 7: y_pass[t] = G_t (S0 q_t - sum_{i<=t} beta_i QK^T[t, i] S0 p_i).
                s0p = S @ P.T            # [Dv, C]
                s0q = S @ Q.T            # [Dv, C]
                corr = np.tril(qkt * bc[None, :]) @ s0p.T   # [C, Dv]
                y_pass = G[:, None] * (s0q.T - corr)
                # Step 8: output (with the 1/sqrt(Dk) scale).
                y[b, start:start + n, hv] = ((y_pass + y_local) / dtype(np.sqrt(Dk)))[:n]
                # Step 9: S_end = G_C (S0 - S0 (beta*p)^T K) + sum_j (G_C/G_j) u_j k_j^T.
                S = G[C - 1] * (S - (s0p * bc[None, :]) @ K) + \
                    (U * gam[C - 1][:, None]).T @ K
            s_out[b, hv] = S
    return y, s_out


def chunked_single_solve(q, k, v, g, beta, s0=None, chunk=32):
    """Single-solve chunk form of ferrox-core ``gdn_chunk.rs`` ("The algebra").

    Per chunk it solves for the per-row updates d_t against S0 k_t and the
    decay products R[t][u] = a_{u+1} ... a_t, then reads the outputs and the
    chunk-end state from S0 and the d_t.  A short last chunk is taken as is
    (no padding), as ``delta_chunk`` does.
    """
    q, k, v, g, beta, s0, (B, T, Hk, Hv, Dk, Dv) = _unpack(q, k, v, g, beta, s0)
    group = Hv // Hk
    scale = 1.0 / np.sqrt(Dk)
    y = np.zeros((B, T, Hv, Dv))
    s_out = np.zeros((B, Hv, Dv, Dk))
    for b in range(B):
        for hv in range(Hv):
            hk = hv // group
            S = s0[b, hv].copy()
            for start in range(0, T, chunk):
                c = min(chunk, T - start)
                K = k[b, start:start + c, hk]
                Q = q[b, start:start + c, hk]
                V = v[b, start:start + c, hv]
                a = g[b, start:start + c, hv]
                bt = beta[b, start:start + c, hv]
                R = _gate_ratios(a)          # R[t][u] = a_{u+1} ... a_t
                A = np.cumprod(a)            # A_t = a_1 ... a_t
                m = S @ K.T                  # S0 k_t  [Dv, c]
                n = S @ Q.T                  # S0 q_t  [Dv, c]
                gram = K @ K.T               # k_u . k_t
                qk = Q @ K.T                 # q_t . k_u
                d = np.zeros((c, Dv))
                for t in range(c):
                    pred = A[t] * m[:, t]
                    read = A[t] * n[:, t]
                    for u in range(t):
                        pred = pred + R[t, u] * gram[t, u] * d[u]
                        read = read + R[t, u] * qk[t, u] * d[u]
                    d[t] = bt[t] * (V[t] - pred)
                    y[b, start + t, hv] = (read + qk[t, t] * d[t]) * scale
                S = A[c - 1] * S + (d * R[c - 1][:, None]).T @ K
            s_out[b, hv] = S
    return y, s_out


def product_form(q, k, v, g, beta, s0=None):
    """S_t from explicit Dk x Dk products; tiny sizes only.

    S_t = S_0 M_1 ... M_t + sum_{j<=t} beta_j v_j k_j^T M_{j+1} ... M_t,
    M_i = g_i (I - beta_i k_i k_i^T),  and y_t = S_t q_t / sqrt(Dk).
    """
    q, k, v, g, beta, s0, (B, T, Hk, Hv, Dk, Dv) = _unpack(q, k, v, g, beta, s0)
    group = Hv // Hk
    eye = np.eye(Dk)
    y = np.zeros((B, T, Hv, Dv))
    s_out = np.zeros((B, Hv, Dv, Dk))
    for b in range(B):
        for hv in range(Hv):
            hk = hv // group
            M = [g[b, i, hv] * (eye - beta[b, i, hv] * np.outer(k[b, i, hk], k[b, i, hk]))
                 for i in range(T)]

            def chain(lo, hi):
                out = eye.copy()
                for i in range(lo, hi):
                    out = out @ M[i]
                return out

            for t in range(T):
                St = s0[b, hv] @ chain(0, t + 1)
                for j in range(t + 1):
                    St = St + beta[b, j, hv] * np.outer(v[b, j, hv], k[b, j, hk]) @ \
                        chain(j + 1, t + 1)
                y[b, t, hv] = St @ q[b, t, hk] / np.sqrt(Dk)
                if t == T - 1:
                    s_out[b, hv] = St
    return y, s_out
