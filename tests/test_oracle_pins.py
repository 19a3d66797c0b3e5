"""Pins for the fp64 sequential oracle (CPU only).

The oracle is pinned to things other than itself:
  * two independent chunk forms (metaltile-std ``gated_delta_wy.rs`` steps 1-9,
    ferrox-core ``gdn_chunk.rs`` "The algebra") at several chunk widths and
    chunk-boundary placements (the placements of ferrox-core's
    ``a_chunk_is_the_sequential_recurrence``);
  * the explicit product form on tiny inputs;
  * closed forms and special cases: beta = 0 (pure decay), g = beta = 1 with
    orthonormal keys (the rule stores v_i under k_i and reduces to causal
    linear attention), beta = 1 with unit keys (S_t k_t = v_t for any gate),
    a hand-worked two-token example (tests/golden), one token in closed form
    written as a projection;
  * invariants: GQA grouped map = MHA on repeated heads, linearity in
    (S_0, V), a vanishing gate resets the state, split/resume.
A mutation test plants plausible mistakes in a NumPy copy of the recurrence
and checks that each one is caught by at least one pin by >= 10x its tolerance.
"""
import json
import os

import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from oracle import forms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(rng, B=1, T=7, Hk=1, Hv=2, Dk=8, Dv=6, unit_keys=True, g_lo=0.3,
              s0_scale=0.5):
    q = rng.standard_normal((B, T, Hk, Dk))
    k = rng.standard_normal((B, T, Hk, Dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, Dv))
    g = rng.uniform(g_lo, 1.0, (B, T, Hv))
    beta = rng.uniform(0.0, 1.0, (B, T, Hv))
    s0 = rng.standard_normal((B, Hv, Dv, Dk)) * s0_scale
    return q, k, v, g, beta, s0


def rel_err(a, b):
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b))) / scale)


def orthonormal_keys(rng, T, Dk):
    """T <= Dk orthonormal vectors (rows), from a QR of a Gaussian matrix."""
    qm, _ = np.linalg.qr(rng.standard_normal((Dk, Dk)))
    return qm[:, :T].T.copy()


# --------------------------------------------------------------------------
# Pins written against an implementation ``impl(q,k,v,g,beta,s0)->(y,s)``;
# each returns (error, tolerance).  The oracle must pass all of them; each
# planted mistake must fail at least one by >= 10x.
# --------------------------------------------------------------------------

def pin_chunked_wy(impl):
    rng = np.random.default_rng(11)
    worst = 0.0
    for C, T in [(1, 5), (2, 7), (8, 37), (16, 3), (16, 21), (32, 33), (64, 69)]:
        case = rand_case(rng, B=1, T=T, Hk=1, Hv=2, Dk=8, Dv=6)
        y, s = impl(*case)
        yc, sc = forms.chunked_wy(*case, chunk=C)
        worst = max(worst, rel_err(y, yc), rel_err(s, sc))
    return worst, 1e-10


def pin_single_solve(impl):
    rng = np.random.default_rng(12)
    worst = 0.0
    for C, T in [(4, 9), (8, 8), (8, 17)]:
        case = rand_case(rng, B=2, T=T, Hk=2, Hv=4, Dk=8, Dv=4)
        y, s = impl(*case)
        yc, sc = forms.chunked_single_solve(*case, chunk=C)
        worst = max(worst, rel_err(y, yc), rel_err(s, sc))
    return worst, 1e-10


def pin_product_form(impl):
    rng = np.random.default_rng(13)
    case = rand_case(rng, B=1, T=5, Hk=1, Hv=2, Dk=6, Dv=4, unit_keys=False)
    y, s = impl(*case)
    yp, sp = forms.product_form(*case)
    return max(rel_err(y, yp), rel_err(s, sp)), 1e-11


def pin_beta_zero(impl):
    """beta = 0: no writes, S_T = (prod g) S_0 and y_t = G_t S_0 q_t / sqrt(Dk)."""
    rng = np.random.default_rng(14)
    q, k, v, g, beta, s0 = rand_case(rng, B=2, T=6, Hk=1, Hv=2, Dk=8, Dv=5)
    beta = np.zeros_like(beta)
    y, s = impl(q, k, v, g, beta, s0)
    G = np.cumprod(g, axis=1)                               # [B,T,Hv]
    s_expect = G[:, -1][:, :, None, None] * s0
    s0q = np.einsum("bhvk,btk->bthv", s0, q[:, :, 0, :])    # Hk = 1
    y_expect = G[..., None] * s0q / np.sqrt(q.shape[-1])
    return max(rel_err(s, s_expect), rel_err(y, y_expect)), 1e-13


def pin_orthonormal_store(impl):
    """g = beta = 1, S_0 = 0, orthonormal keys: S_T k_i = v_i for every i."""
    rng = np.random.default_rng(15)
    T, Dk, Dv = 6, 8, 5
    k = orthonormal_keys(rng, T, Dk)[None, :, None, :]
    q = rng.standard_normal((1, T, 1, Dk))
    v = rng.standard_normal((1, T, 1, Dv))
    ones = np.ones((1, T, 1))
    _, s = impl(q, k, v, ones, ones, np.zeros((1, 1, Dv, Dk)))
    recalled = np.einsum("vk,tk->tv", s[0, 0], k[0, :, 0, :])
    return rel_err(recalled, v[0, :, 0, :]), 1e-13


def pin_causal_linear_attention(impl):
    """g = beta = 1, S_0 = 0, orthonormal keys: Y = tril(Q K^T) V / sqrt(Dk)."""
    rng = np.random.default_rng(16)
    T, Dk, Dv = 7, 8, 3
    K = orthonormal_keys(rng, T, Dk)
    Q = rng.standard_normal((T, Dk))
    V = rng.standard_normal((T, Dv))
    ones = np.ones((1, T, 1))
    y, _ = impl(Q[None, :, None], K[None, :, None], V[None, :, None], ones, ones,
                np.zeros((1, 1, Dv, Dk)))
    expect = np.tril(Q @ K.T) @ V / np.sqrt(Dk)
    return rel_err(y[0, :, 0, :], expect), 1e-13


def pin_unit_key_overwrite(impl):
    """beta = 1 and |k_t| = 1 for any gate and S_0: S_t k_t = v_t, and with
    q_t = k_t the output is v_t / sqrt(Dk)."""
    rng = np.random.default_rng(17)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=5, Hk=1, Hv=1, Dk=8, Dv=4)
    beta = np.ones_like(beta)
    q = k.copy()
    y, s = impl(q, k, v, g, beta, s0)
    recalled = s[0, 0] @ k[0, -1, 0]
    err = max(rel_err(recalled, v[0, -1, 0]),
              rel_err(y[0, :, 0, :], v[0, :, 0, :] / np.sqrt(8)))
    return err, 1e-13


def pin_hand_worked(impl):
    with open(os.path.join(GOLDEN, "hand_worked_d2_t2.json")) as f:
        ex = json.load(f)
    arr = {name: np.array(ex["inputs"][name], dtype=np.float64)
           for name in ("q", "k", "v", "g", "beta", "s0")}
    y, s = impl(arr["q"], arr["k"], arr["v"], arr["g"], arr["beta"], arr["s0"])
    err = max(rel_err(y, np.array(ex["expected"]["y"])),
              rel_err(s, np.array(ex["expected"]["s"])))
    return err, 1e-14


def pin_gqa_grouped(impl):
    """Hv/Hk = 3 grouped map equals MHA with each key head repeated 3 times
    in place (hk = hv // 3)."""
    rng = np.random.default_rng(18)
    q, k, v, g, beta, s0 = rand_case(rng, B=2, T=5, Hk=2, Hv=6, Dk=8, Dv=4)
    y, s = impl(q, k, v, g, beta, s0)
    qr, kr = np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2)
    y2, s2 = impl(qr, kr, v, g, beta, s0)
    return max(rel_err(y, y2), rel_err(s, s2)), 1e-14


def pin_linearity(impl):
    """For fixed q, k, g, beta the rule is linear in (S_0, V)."""
    rng = np.random.default_rng(19)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=6, Hk=1, Hv=2, Dk=8, Dv=4)
    y, s = impl(q, k, v, g, beta, s0)
    ya, sa = impl(q, k, v, g, beta, np.zeros_like(s0))
    yb, sb = impl(q, k, np.zeros_like(v), g, beta, s0)
    return max(rel_err(y, ya + yb), rel_err(s, sa + sb)), 1e-13


def pin_vanishing_gate_resets(impl):
    """A gate of 1e-300 at token t0 forgets everything before it: the outputs
    from t0 on equal a run started at t0 from a zero state (ferrox-core
    ``a_vanishing_decay_is_forgetting_and_not_a_division``)."""
    rng = np.random.default_rng(20)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=9, Hk=1, Hv=2, Dk=8, Dv=4)
    t0 = 4
    g[:, t0, :] = 1e-300
    y, s = impl(q, k, v, g, beta, s0)
    g2 = g[:, t0:].copy()
    g2[:, 0, :] = 1.0
    y2, s2 = impl(q[:, t0:], k[:, t0:], v[:, t0:], g2, beta[:, t0:],
                  np.zeros_like(s0))
    ok_finite = np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    err = max(rel_err(y[:, t0:], y2), rel_err(s, s2))
    return (err if ok_finite else np.inf), 1e-13


def pin_split_resume(impl):
    """Running T1 tokens and then T2 from the carried state equals T1+T2."""
    rng = np.random.default_rng(21)
    q, k, v, g, beta, s0 = rand_case(rng, B=1, T=8, Hk=1, Hv=2, Dk=8, Dv=4)
    y, s = impl(q, k, v, g, beta, s0)
    ya, sa = impl(q[:, :3], k[:, :3], v[:, :3], g[:, :3], beta[:, :3], s0)
    yb, sb = impl(q[:, 3:], k[:, 3:], v[:, 3:], g[:, 3:], beta[:, 3:], sa)
    return max(rel_err(y, np.concatenate([ya, yb], axis=1)), rel_err(s, sb)), 1e-14


def pin_one_token_projection(impl):
    """T = 1 in closed form, arranged as a projection: the update is
    S_1 = g S_0 (I - beta k k^T) + beta v k^T (the state decays, its component
    along k is partly removed, and beta v is written along k), y = S_1 q / sqrt(Dk).
    Keys are not normalised, heads are grouped (Hv/Hk = 2)."""
    rng = np.random.default_rng(22)
    q, k, v, g, beta, s0 = rand_case(rng, B=2, T=1, Hk=2, Hv=4, Dk=6, Dv=5, unit_keys=False)
    y, s = impl(q, k, v, g, beta, s0)
    B, _, Hk, Dk = q.shape
    Hv = v.shape[2]
    ys = np.zeros_like(y)
    ss = np.zeros_like(s)
    for b in range(B):
        for hv in range(Hv):
            hk = hv // (Hv // Hk)
            kk, qq, vv = k[b, 0, hk], q[b, 0, hk], v[b, 0, hv]
            gg, bb = g[b, 0, hv], beta[b, 0, hv]
            proj = np.eye(Dk) - bb * np.outer(kk, kk)
            ss[b, hv] = gg * s0[b, hv] @ proj + bb * np.outer(vv, kk)
            ys[b, 0, hv] = ss[b, hv] @ qq / np.sqrt(Dk)
    return max(rel_err(y, ys), rel_err(s, ss)), 1e-13


PINS = [pin_chunked_wy, pin_single_solve, pin_product_form, pin_beta_zero,
        pin_orthonormal_store, pin_causal_linear_attention, pin_unit_key_overwrite,
        pin_hand_worked, pin_gqa_grouped, pin_linearity, pin_vanishing_gate_resets,
        pin_split_resume, pin_one_token_projection]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    err, tol = pin(oracle.gdn_sequential)
    assert err <= tol, f"{pin.__name__}: {err:.3e} > {tol:.0e}"


# --------------------------------------------------------------------------
# Planted mistakes.  A NumPy restatement of the recurrence with switches;
# used only to show that the pins above would catch each mistake.
# --------------------------------------------------------------------------

def _numpy_recurrence(mutation=None):
    def impl(q, k, v, g, beta, s0):
        q, k, v, g, beta, s0 = (np.asarray(a, dtype=np.float64)
                                for a in (q, k, v, g, beta, s0))
        B, T, Hk, Dk = q.shape
        Hv, Dv = v.shape[2], v.shape[3]
        y = np.zeros((B, T, Hv, Dv))
        s_out = np.zeros((B, Hv, Dv, Dk))
        scale = 1.0 if mutation == "no_scale" else 1.0 / np.sqrt(Dk)
        for b in range(B):
            for hv in range(Hv):
                hk = hv % Hk if mutation == "tiled_head_map" else hv // (Hv // Hk)
                S = s0[b, hv].copy()
                for t in range(T):
                    kt, qt, vt = k[b, t, hk], q[b, t, hk], v[b, t, hv]
                    gt, bt = g[b, t, hv], beta[b, t, hv]
                    if mutation == "transposed_state":
                        x = S.T @ kt if Dv == Dk else S @ kt * 0.5
                    else:
                        x = S @ kt
                    if mutation == "no_gate_in_prediction":
                        d = bt * (vt - x)
                    elif mutation == "beta_only_on_v":
                        d = bt * vt - gt * x
                    else:
                        d = bt * (vt - gt * x)
                    S_prev = S
                    if mutation == "gate_after_write":
                        S = gt * (S + np.outer(d, kt))
                    elif mutation == "key_for_query":
                        S = gt * S + np.outer(d, qt)
                    else:
                        S = gt * S + np.outer(d, kt)
                    if mutation == "output_before_update":
                        y[b, t, hv] = S_prev @ qt * scale
                    else:
                        y[b, t, hv] = S @ qt * scale
                s_out[b, hv] = S
        return y, s_out
    return impl


MUTATIONS = ["tiled_head_map", "no_scale", "transposed_state",
             "no_gate_in_prediction", "beta_only_on_v", "gate_after_write",
             "key_for_query", "output_before_update"]


def test_numpy_restatement_passes_every_pin():
    impl = _numpy_recurrence(None)
    for pin in PINS:
        err, tol = pin(impl)
        assert err <= tol * 10, f"{pin.__name__}: {err:.3e}"


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_pins_catch_planted_mistake(mutation):
    impl = _numpy_recurrence(mutation)
    ratios = {}
    for pin in PINS:
        err, tol = pin(impl)
        ratios[pin.__name__] = err / tol
    worst = max(ratios.values())
    assert worst >= 10.0, f"{mutation} slipped through every pin: {ratios}"


def test_decode_steps_equal_prefill():
    """N single steps with the state carried equal one N-token prefill."""
    rng = np.random.default_rng(22)
    q, k, v, g, beta, s0 = rand_case(rng, B=2, T=5, Hk=1, Hv=2, Dk=8, Dv=4)
    y, s = oracle.gdn_sequential(q, k, v, g, beta, s0)
    steps = [a.transpose(1, 0, *range(2, a.ndim))[:, :, None] for a in (q, k, v, g, beta)]
    yd, sd = oracle.gdn_decode_steps(*steps, s0)
    assert rel_err(yd[:, :, 0].transpose(1, 0, 2, 3), y) <= 1e-15
    assert rel_err(sd, s) <= 1e-15


def test_oracle_zero_state_is_none_state():
    rng = np.random.default_rng(23)
    q, k, v, g, beta, s0 = rand_case(rng)
    y1, s1 = oracle.gdn_sequential(q, k, v, g, beta, None)
    y2, s2 = oracle.gdn_sequential(q, k, v, g, beta, np.zeros_like(s0))
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


def test_oracle_golden_regression():
    """The oracle reproduces the fixture written by tests/golden/make_golden.py
    (a script that calls only oracle/), bit for bit up to 1e-14."""
    path = os.path.join(GOLDEN, "oracle_t37_c16.json")
    with open(path) as f:
        fx = json.load(f)
    ins = {n: np.array(fx["inputs"][n]) for n in ("q", "k", "v", "g", "beta", "s0")}
    y, s = oracle.gdn_sequential(**ins)
    assert rel_err(y, np.array(fx["y"])) <= 1e-14
    assert rel_err(s, np.array(fx["s"])) <= 1e-14


@pytest.mark.parametrize("chunk,T", [(32, 37), (64, 70), (16, 129)])
def test_oracle_matches_chunk_forms_at_head_dim_128(chunk, T):
    """The chunk forms agree with the oracle at the library's head size
    (Dk = Dv = 128) on the synthetic input recipe, GQA 2:1, for chunk
    boundaries that fall short of, on and past a chunk multiple."""
    import gdn_inputs
    ins = gdn_inputs.make_inputs(1, T, 1, 2, 128, 128, "f32", seed=77 + T,
                                 u_max=1.0, s0_std=0.1)
    args = [ins[n] for n in ("q", "k", "v", "g", "beta", "s0")]
    y, s = oracle.gdn_sequential(*args)
    yc, sc = forms.chunked_wy(*args, chunk=chunk)
    ys, ss = forms.chunked_single_solve(*args, chunk=chunk)
    for a, b in ((yc, y), (sc, s), (ys, y), (ss, s)):
        assert rel_err(a, b) <= 1e-11


def test_fp32_chunked_form_tracks_the_oracle():
    """The float32 run of the chunked WY form (timed only as a CPU baseline)
    computes the same rule: it agrees with the fp64 sequential oracle to
    float32 rounding on a multi-chunk case with a ragged tail."""
    ins = gdn_inputs.make_inputs(1, 75, 1, 2, 16, 16, torch.float32, seed=12, u_max=0.5,
                                 s0_std=0.1)
    names = ("q", "k", "v", "g", "beta")
    y32, s32 = forms.chunked_wy(*(ins[n] for n in names), ins["s0"], chunk=32,
                                dtype=np.float32)
    assert y32.dtype == np.float32 and s32.dtype == np.float32
    yo, so = oracle.gdn_sequential(*(ins[n] for n in names), ins["s0"])
    assert np.max(np.abs(y32 - yo)) <= 1e-5 * np.max(np.abs(yo))
    assert np.max(np.abs(s32 - so)) <= 1e-5 * np.max(np.abs(so))
