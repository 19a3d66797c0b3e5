"""The seeded synthetic input recipe (CPU): shapes, dtypes and the value
distributions every parity test and the benchmark rely on -- unit q and k
rows, gates exp(-u) with u ~ U(0, u_max) (and the 10% heavy-decay rows of
the long-context workload), beta in (0, 1), the initial state's spread, and
determinism per seed.  Large workloads are checked on a shortened T."""
import math

import pytest
import torch

import gdn_inputs

W = gdn_inputs.WORKLOADS


def small(w):
    return w.scaled(T=min(w.T, 1024))


@pytest.mark.parametrize("name", sorted(W))
def test_shapes_dtypes_and_ranges(name):
    w = small(W[name])
    ins = gdn_inputs.workload_inputs(w, step=0 if w.steps else None)
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.dtype]
    assert ins["q"].shape == ins["k"].shape == (w.B, w.T, w.Hk, w.Dk)
    assert ins["v"].shape == (w.B, w.T, w.Hv, w.Dv)
    assert ins["g"].shape == ins["beta"].shape == (w.B, w.T, w.Hv)
    assert ins["s0"].shape == (w.B, w.Hv, w.Dv, w.Dk) and ins["s0"].dtype == torch.float32
    for n in ("q", "k", "v", "g", "beta"):
        assert ins[n].dtype == dt and ins[n].is_contiguous()
    # unit rows (up to the cast to the workload dtype)
    for n in ("q", "k"):
        norms = ins[n].double().norm(dim=-1)
        atol = {torch.bfloat16: 2e-2, torch.float16: 2e-3}.get(dt, 1e-5)
        assert torch.allclose(norms, torch.ones_like(norms), atol=atol)
    g = ins["g"].double()
    assert g.max() <= 1.0 and g.min() > 0.0
    beta = ins["beta"].double()
    assert beta.min() > 0.0 and beta.max() < 1.0
    if w.heavy_frac == 0.0:
        assert g.min() >= math.exp(-w.u_max) * (1 - 1e-2)


def test_heavy_decay_rows_of_the_long_workload():
    w = W["prefill_t65536"].scaled(T=2048)
    g = gdn_inputs.workload_inputs(w)["g"].double()
    below = (g < math.exp(-w.u_max) * (1 - 1e-2)).double().mean().item()
    # heavy rows draw u ~ U(0, 5): a fraction 0.1 * (5 - 0.1) / 5 of all rows falls
    # below exp(-0.1)
    assert abs(below - 0.1 * (w.heavy_umax - w.u_max) / w.heavy_umax) < 0.01
    assert g.min() >= math.exp(-w.heavy_umax) * (1 - 1e-2)


@pytest.mark.parametrize("name,std", [("prefill_b4_t2048", 0.1), ("decode_b64", 0.1),
                                      ("prefill_t4096", 0.0), ("fp32_t64", 0.1)])
def test_initial_state_spread(name, std):
    w = small(W[name])
    s0 = gdn_inputs.workload_inputs(w, step=0 if w.steps else None)["s0"]
    if std == 0.0:
        assert torch.count_nonzero(s0) == 0
    else:
        assert abs(s0.double().std().item() - std) < 0.05 * std
        assert abs(s0.double().mean().item()) < 0.01


def test_determinism_and_decode_steps():
    w = small(W["prefill_b4_t2048"])
    a, b = gdn_inputs.workload_inputs(w), gdn_inputs.workload_inputs(w)
    for n in a:
        assert torch.equal(a[n], b[n])
    other = gdn_inputs.workload_inputs(w.scaled(seed=w.seed + 1))
    assert not torch.equal(a["v"], other["v"])
    d = W["decode_b64"]
    s1, s2 = gdn_inputs.workload_inputs(d, step=1), gdn_inputs.workload_inputs(d, step=2)
    assert "s0" not in s1 and not torch.equal(s1["q"], s2["q"])
    assert s1["q"].shape == (d.B, 1, d.Hk, d.Dk)
