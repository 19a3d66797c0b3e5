"""The algebra the CUDA kernels are built on, restated in fp64 NumPy and checked
against the oracle on the CPU (no GPU, no code shared with either side).

Each identity here is one the kernels rely on beyond the plain recurrence:
  * the chunked form of the tensor-core prefill: T_L = (I + L)^-1 with
    L[t][j] = beta_j KK^T[t][j] (j < t); the second solve without a second
    inverse, (I + A)^-1 diag(beta) = diag(beta) (Gam . T_L) for
    A[t][j] = beta_t Gam[t][j] KK^T[t][j]; P = T_L K, U = diag(beta)(Gam . T_L) V;
    Qh = diag(G) Q - diag(G) M P with M[t][i] = beta_i QK^T[t][i] (i <= t);
    y = (S_0 Qh^T + (Gam . QK^T) U) / sqrt(Dk); and the state update regrouped as
    S <- G_C S - S (Pt^T K) + Ut^T K with Pt = G_C diag(beta) P and
    Ut = diag(Gam[C-1][.]) U (metaltile-std gated_delta_wy.rs "Algorithm", steps
    1-9; ferrox-core gdn_chunk.rs "The algebra");
  * the decay table used across 16-token blocks, Gam[t][j] = rfac[t][b(j)] * sfac[j],
    both factors products of decays, and the clamp of log2 g that makes a
    vanishing gate underflow to exact forgetting;
  * the short-T kernel's scaled state, S = gam * St with renormalisation when
    gam * g leaves [2^-24, 2^24], and its output identity y = g z + d (k . q);
  * the warp-level MMA kernels' blockwise inverse (8 x 8 diagonal blocks by
    forward substitution, then T21 = -T22 (L21 T11) doubling the block size) and
    their coefficient form: cP = -G_C diag(beta) T_L, cU = diag(Gam_end) T_A,
    W_M = diag(G) M T_L, W_Y = (Gam . QK^T) T_A, with the innovation-form update
    S <- G_C S + (Ut^T - Z) K.
A ragged tail is padded with g = 1, beta = 0 and zero q, k, v, as the kernels do.
"""
import numpy as np
import pytest

import oracle


def rel_err(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def rand_problem(rng, T, Hk, Hv, Dk, Dv, g_lo=0.3):
    q = rng.standard_normal((1, T, Hk, Dk))
    k = rng.standard_normal((1, T, Hk, Dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, Hv, Dv))
    g = rng.uniform(g_lo, 1.0, (1, T, Hv))
    beta = rng.uniform(0.0, 1.0, (1, T, Hv))
    s0 = rng.standard_normal((1, Hv, Dv, Dk)) * 0.3
    return q, k, v, g, beta, s0


def gate_tables(gc):
    """lam (chunk-local prefix sums of log2 g, clamped), G_t = 2^lam_t and
    Gam[t][j] = 2^(lam_t - lam_j) for j <= t, else 0."""
    lam = np.cumsum(np.maximum(np.log2(np.maximum(gc, 1e-320)), -1000.0))
    C = len(gc)
    gam = np.zeros((C, C))
    for t in range(C):
        for j in range(t + 1):
            gam[t, j] = 2.0 ** (lam[t] - lam[j])
    return lam, 2.0 ** lam, gam


def tc_chunk_model(q, k, v, g, beta, s0, C):
    """One head through the tensor-core kernel's chunk algebra."""
    T, Dk = k.shape
    Dv = v.shape[1]
    n = -(-T // C)
    pad = n * C - T
    q = np.vstack([q, np.zeros((pad, Dk))])
    k = np.vstack([k, np.zeros((pad, Dk))])
    v = np.vstack([v, np.zeros((pad, Dv))])
    g = np.concatenate([g, np.ones(pad)])
    beta = np.concatenate([beta, np.zeros(pad)])
    S = s0.copy()
    ys = []
    for c in range(n):
        sl = slice(c * C, (c + 1) * C)
        Q, K, V, gc, bc = q[sl], k[sl], v[sl], g[sl], beta[sl]
        _, G, gam = gate_tables(gc)
        KK, QK = K @ K.T, Q @ K.T
        L = np.tril(KK * bc[None, :], -1)
        TL = np.linalg.inv(np.eye(C) + L)
        P = TL @ K
        U = (bc[:, None] * (gam * TL)) @ V
        M = np.tril(QK * bc[None, :])
        Qh = G[:, None] * Q - G[:, None] * (M @ P)
        y_loc = (gam * QK) @ U
        ys.append((Qh @ S.T + y_loc) / np.sqrt(Dk))
        GC = G[-1]
        Pt = GC * bc[:, None] * P
        Ut = gam[-1][:, None] * U
        S = GC * S - S @ (Pt.T @ K) + Ut.T @ K
    return np.vstack(ys)[:T], S


@pytest.mark.parametrize("C,T", [(16, 16), (16, 37), (32, 70), (64, 64), (64, 131)])
def test_tensor_core_chunk_algebra_equals_the_rule(C, T):
    rng = np.random.default_rng(1000 + C + T)
    Hk, Hv, Dk, Dv = 1, 2, 16, 12
    q, k, v, g, beta, s0 = rand_problem(rng, T, Hk, Hv, Dk, Dv)
    yo, so = oracle.gdn_sequential(q, k, v, g, beta, s0)
    for hv in range(Hv):
        y, s = tc_chunk_model(q[0, :, 0], k[0, :, 0], v[0, :, hv], g[0, :, hv],
                              beta[0, :, hv], s0[0, hv], C)
        assert rel_err(y, yo[0, :, hv]) < 1e-10
        assert rel_err(s, so[0, hv]) < 1e-10


def test_second_solve_needs_no_second_inverse():
    rng = np.random.default_rng(7)
    C = 24
    K = rng.standard_normal((C, 10))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    gc = rng.uniform(0.2, 1.0, C)
    bc = rng.uniform(0.0, 1.0, C)
    _, _, gam = gate_tables(gc)
    KK = K @ K.T
    TL = np.linalg.inv(np.eye(C) + np.tril(KK * bc[None, :], -1))
    A = np.tril(bc[:, None] * gam * KK, -1)
    lhs = np.linalg.inv(np.eye(C) + A) @ np.diag(bc)
    rhs = np.diag(bc) @ (gam * TL)
    assert np.max(np.abs(lhs - rhs)) < 1e-12


def test_block_factored_decay_table():
    """Across 16-token blocks the kernel uses Gam[t][j] = rfac[t][b(j)] sfac[j] with
    sfac[j] = 2^(lam[end of j's block] - lam_j), rfac[t][b] = 2^(lam_t - lam[end of b]),
    both <= 1; inside a block 2^(lam_t - lam_j)."""
    rng = np.random.default_rng(8)
    gc = rng.uniform(0.05, 1.0, 64)
    gc[40] = 0.0   # a vanishing gate: everything before token 40 is forgotten
    lam, _, gam = gate_tables(gc)
    fact = np.zeros_like(gam)
    for t in range(64):
        for j in range(t + 1):
            bt, bj = t // 16, j // 16
            if bt == bj:
                fact[t, j] = 2.0 ** (lam[t] - lam[j])
            else:
                e = bj * 16 + 15
                sfac, rfac = 2.0 ** (lam[e] - lam[j]), 2.0 ** (lam[t] - lam[e])
                assert sfac <= 1.0 and rfac <= 1.0
                fact[t, j] = rfac * sfac
    assert np.max(np.abs(fact - gam)) < 1e-14
    assert np.all(np.diag(gam) == 1.0)
    # Across the vanishing gate the exponent is below -1000 + 64 * 5: negligible in
    # fp64 and exactly 0 once the power of two is taken in fp32, as the kernel does.
    diff = np.array([[lam[t] - lam[j] for j in range(40)] for t in range(40, 64)])
    assert np.all(diff < -900)
    assert np.all(np.exp2(diff.astype(np.float32)) == np.float32(0.0))


def short_t_model(q, k, v, g, beta, s0):
    """One head through the short-T kernel's scaled-state rule."""
    T, Dk = k.shape
    St, gam = s0.copy(), 1.0
    ys = []
    for t in range(T):
        x, z, kq = St @ k[t], St @ q[t], k[t] @ q[t]
        gn = gam * g[t]
        d = beta[t] * (v[t] - gn * x)
        ys.append((gn * z + d * kq) / np.sqrt(Dk))
        if 2.0 ** -24 <= gn <= 2.0 ** 24:
            St = St + np.outer(d / gn, k[t])
            gam = gn
        else:
            St = gn * St + np.outer(d, k[t])
            gam = 1.0
    return np.array(ys), gam * St


@pytest.mark.parametrize("gates", ["random", "small", "zeros", "ones"])
def test_short_t_scaled_state_equals_the_rule(gates):
    rng = np.random.default_rng(9)
    T, Dk, Dv = 32, 16, 8
    q, k, v, g, beta, s0 = rand_problem(rng, T, 1, 1, Dk, Dv)
    if gates == "small":
        g[:] = 1e-3
    elif gates == "zeros":
        g[0, 1::3, 0] = 0.0
    elif gates == "ones":
        g[:] = 1.0
    yo, so = oracle.gdn_sequential(q, k, v, g, beta, s0)
    y, s = short_t_model(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0], s0[0, 0])
    assert rel_err(y, yo[0, :, 0]) < 1e-12
    assert rel_err(s, so[0, 0]) < 1e-12


def test_two_chunks_compose_into_one_affine_step():
    """A chunk maps the state affinely, S <- S F + N with F = G_C I - Pt^T K and
    N = Ut^T K, so two chunks compose into one step S <- S (F1 F2) + (N1 F2 + N2),
    and both chunks' outputs come from the first chunk's start state:
    [Y_1 | Y_2] = S [Qh_1^T | F1 Qh_2^T] + [0 | N1 Qh_2^T].  Everything but the
    products with S is independent of the state."""
    rng = np.random.default_rng(3)
    C, Dk, Dv, T = 32, 16, 12, 128
    q, k, v, g, beta, s0 = rand_problem(rng, T, 1, 1, Dk, Dv)
    yo, so = oracle.gdn_sequential(q, k, v, g, beta, s0)
    q, k, v, g, beta, s0 = q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0], s0[0, 0]

    def chunk(sl):
        Q, K, V, gc, bc = q[sl], k[sl], v[sl], g[sl], beta[sl]
        _, G, gam = gate_tables(gc)
        KK, QK = K @ K.T, Q @ K.T
        TL = np.linalg.inv(np.eye(C) + np.tril(KK * bc[None, :], -1))
        P, U = TL @ K, (bc[:, None] * (gam * TL)) @ V
        M = np.tril(QK * bc[None, :])
        Qh = G[:, None] * Q - G[:, None] * (M @ P)
        F = G[-1] * np.eye(Dk) - (G[-1] * bc[:, None] * P).T @ K
        N = (gam[-1][:, None] * U).T @ K
        return F, N, Qh, (gam * QK) @ U

    S, ys = s0.copy(), []
    for p in range(T // (2 * C)):
        F1, N1, Q1, y1 = chunk(slice(2 * p * C, (2 * p + 1) * C))
        F2, N2, Q2, y2 = chunk(slice((2 * p + 1) * C, (2 * p + 2) * C))
        Y = S @ np.hstack([Q1.T, F1 @ Q2.T])
        Y[:, C:] += N1 @ Q2.T
        ys.append((Y.T + np.vstack([y1, y2])) / np.sqrt(Dk))
        S = S @ (F1 @ F2) + (N1 @ F2 + N2)
    assert rel_err(np.vstack(ys), yo[0, :, 0]) < 1e-12
    assert rel_err(S, so[0, 0]) < 1e-12


def blockwise_inverse(L):
    """(I + L)^-1 for strictly lower-triangular L of size C (a multiple of 8)
    the way the warp-MMA kernels form it: the 8 x 8 diagonal blocks by forward
    substitution, then, doubling the block size B, every lower-left block of a
    2B x 2B diagonal block from T21 = -T22 (L21 T11)."""
    C = L.shape[0]
    T = np.zeros((C, C))
    for o in range(0, C, 8):
        for c in range(8):
            x = np.zeros(8)
            for r in range(8):
                x[r] = (1.0 if r == c else 0.0) - L[o + r, o:o + r] @ x[:r]
            T[o:o + 8, o + c] = x
    B = 8
    while B < C:
        for o in range(0, C, 2 * B):
            L21 = L[o + B:o + 2 * B, o:o + B]
            T11 = T[o:o + B, o:o + B]
            T22 = T[o + B:o + 2 * B, o + B:o + 2 * B]
            T[o + B:o + 2 * B, o:o + B] = -T22 @ (L21 @ T11)
        B *= 2
    return T


@pytest.mark.parametrize("C", [16, 32, 64])
def test_blockwise_inverse_equals_the_inverse(C):
    rng = np.random.default_rng(40 + C)
    K = rng.standard_normal((C, 24))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    bc = rng.uniform(0.0, 1.0, C)
    L = np.tril((K @ K.T) * bc[None, :], -1)
    ref = np.linalg.inv(np.eye(C) + L)
    assert np.max(np.abs(blockwise_inverse(L) - ref)) < 1e-12 * max(1.0, np.max(np.abs(ref)))


def coefficient_chunk_model(q, k, v, g, beta, s0, C):
    """One head through the coefficient form of the warp-level MMA kernels
    (short-T, head sizes 64 and 256): per chunk cP = -G_C diag(beta) T_L,
    T_A = diag(beta)(Gam . T_L), cU = diag(Gam_end) T_A, W_M = diag(G) M T_L,
    W_Y = (Gam . QK^T) T_A; -Pt = cP K, Qh = (G Q - W_M K) / sqrt(Dk),
    Ut = cU V, y_loc = W_Y V / sqrt(Dk); then [-Z | Y] = S [-Pt; Qh]^T,
    y = Y + y_loc and S <- G_C S + (Ut^T - Z) K."""
    T, Dk = k.shape
    Dv = v.shape[1]
    n = -(-T // C)
    pad = n * C - T
    q = np.vstack([q, np.zeros((pad, Dk))])
    k = np.vstack([k, np.zeros((pad, Dk))])
    v = np.vstack([v, np.zeros((pad, Dv))])
    g = np.concatenate([g, np.ones(pad)])
    beta = np.concatenate([beta, np.zeros(pad)])
    sc = 1.0 / np.sqrt(Dk)
    S = s0.copy()
    ys = []
    for c in range(n):
        sl = slice(c * C, (c + 1) * C)
        Q, K, V, gc, bc = q[sl], k[sl], v[sl], g[sl], beta[sl]
        _, G, gam = gate_tables(gc)
        GC = G[-1]
        KK, QK = K @ K.T, Q @ K.T
        TL = blockwise_inverse(np.tril(KK * bc[None, :], -1))
        TA = bc[:, None] * (gam * TL)
        cP = -GC * bc[:, None] * TL
        cU = gam[-1][:, None] * TA
        WM = (G[:, None] * np.tril(QK * bc[None, :])) @ TL
        WY = (gam * QK) @ TA
        negPt = cP @ K
        Qh = (G[:, None] * Q - WM @ K) * sc
        Ut = cU @ V
        y_loc = (WY @ V) * sc
        negZ, Y = S @ negPt.T, S @ Qh.T
        ys.append(Y.T + y_loc)
        S = GC * S + (Ut.T + negZ) @ K
    return np.vstack(ys)[:T], S


@pytest.mark.parametrize("C,T", [(16, 16), (16, 9), (32, 32), (32, 70), (32, 257)])
def test_warp_mma_coefficient_form_equals_the_rule(C, T):
    rng = np.random.default_rng(2000 + C + T)
    Hk, Hv, Dk, Dv = 1, 2, 16, 12
    q, k, v, g, beta, s0 = rand_problem(rng, T, Hk, Hv, Dk, Dv)
    yo, so = oracle.gdn_sequential(q, k, v, g, beta, s0)
    for hv in range(Hv):
        y, s = coefficient_chunk_model(q[0, :, 0], k[0, :, 0], v[0, :, hv], g[0, :, hv],
                                       beta[0, :, hv], s0[0, hv], C)
        assert rel_err(y, yo[0, :, hv]) < 1e-10
        assert rel_err(s, so[0, hv]) < 1e-10
