"""Input conventions of the *_ex entry points (GDN_OPT_*), on every path,
against the oracle fed the equivalent inputs:

- tiled head map (value head hv reads key head hv % Hk): the oracle runs the
  same problem with q and k expanded to one key head per value head;
- log-decay gates (the decay is exp(g)): the oracle gets exp of the stored
  log-gates, taken in fp64;
- L2-normalised q, k: the oracle gets the stored rows divided by their norm
  in fp64 (a zero row stays zero).
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from parity_util import TOL, gpu_prefill, rel_err

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16
TILED, LOGG, L2N = 1, 2, 4


def _oracle_equivalent(ins, options):
    """Inputs for the oracle (grouped heads, multiplicative gates) that define
    the same problem as `ins` read under `options`."""
    out = dict(ins)
    Hk, Hv = ins["q"].shape[2], ins["v"].shape[2]
    if options & TILED:
        idx = torch.tensor([hv % Hk for hv in range(Hv)])
        out["q"] = ins["q"][:, :, idx]
        out["k"] = ins["k"][:, :, idx]
    if options & LOGG:
        out["g"] = torch.exp(ins["g"].double())
    if options & L2N:
        for n in ("q", "k"):
            x = out[n].double()
            nrm = x.norm(dim=-1, keepdim=True)
            out[n] = x / torch.where(nrm > 0, nrm, torch.ones_like(nrm))
    return out


def _with_log_gates(ins):
    out = dict(ins)
    out["g"] = torch.log(ins["g"].double()).to(ins["g"].dtype)
    return out


def _run(ins, options, chunk, dev):
    gins = _with_log_gates(ins) if options & LOGG else ins
    y, s = gpu_prefill(gins, chunk, dev, options=options)
    o = _oracle_equivalent(gins, options)
    yo, so = oracle.gdn_sequential(o["q"], o["k"], o["v"], o["g"], o["beta"], o["s0"])
    return y, s, yo, so


CASES = [
    # (B, T, Hk, Hv, chunk, dtype): the fused tensor-core path, the split
    # launches (B*Hv = 64), the short-T kernel and the fp32 path
    (1, 150, 2, 6, 32, BF16),
    (2, 100, 16, 32, 64, BF16),
    (2, 20, 4, 8, 64, BF16),
    (1, 70, 2, 4, 32, F32),
]


@pytest.mark.parametrize("options", [TILED, LOGG, L2N, TILED | LOGG | L2N])
@pytest.mark.parametrize("B,T,Hk,Hv,chunk,dtype", CASES)
def test_prefill_options(cuda_device, options, B, T, Hk, Hv, chunk, dtype):
    ins = gdn_inputs.make_inputs(B, T, Hk, Hv, 128, 128, dtype, seed=500 + T + Hv,
                                 u_max=0.5, s0_std=0.1)
    y, s, yo, so = _run(ins, options, chunk, cuda_device)
    assert rel_err(y, yo) <= TOL[dtype], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[dtype], rel_err(s, so)


@pytest.mark.parametrize("options", [TILED, LOGG, L2N, TILED | LOGG | L2N])
def test_prefill_options_head_size_64(cuda_device, options):
    """The same conventions on the warp-level tensor-core path (16-bit inputs,
    Dk = Dv = 64), q and k rows of varied length under L2N."""
    ins = gdn_inputs.make_inputs(2, 100, 2, 4, 64, 64, BF16, seed=520, u_max=0.5, s0_std=0.1)
    if options & L2N:
        ins = _unnormalised(ins)
    y, s, yo, so = _run(ins, options, 32, cuda_device)
    assert rel_err(y, yo) <= TOL[BF16], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[BF16], rel_err(s, so)


@pytest.mark.parametrize("options", [TILED | LOGG | L2N])
def test_prefill_options_head_size_256(cuda_device, options):
    """The conventions on the head-size-256 warp-level tensor-core path."""
    ins = gdn_inputs.make_inputs(1, 70, 2, 4, 256, 256, BF16, seed=530, u_max=0.5, s0_std=0.1)
    ins = _unnormalised(ins)
    y, s, yo, so = _run(ins, options, 32, cuda_device)
    assert rel_err(y, yo) <= TOL[BF16], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[BF16], rel_err(s, so)


def test_tiled_differs_from_grouped(cuda_device):
    """The option changes the result (the two maps pair different heads)."""
    ins = gdn_inputs.make_inputs(1, 40, 2, 4, 128, 128, BF16, seed=7, s0_std=0.1)
    y1, s1 = gpu_prefill(ins, 32, cuda_device, options=0)
    y2, s2 = gpu_prefill(ins, 32, cuda_device, options=TILED)
    assert rel_err(y1, y2) > 0.05


def _unnormalised(ins, scale=3.0):
    """q and k rows of varied length (the stored rows are unit length)."""
    out = dict(ins)
    gen = torch.Generator().manual_seed(11)
    for n in ("q", "k"):
        f = 0.25 + scale * torch.rand(ins[n].shape[:-1] + (1,), generator=gen)
        out[n] = (ins[n].double() * f).to(ins[n].dtype)
    return out


@pytest.mark.parametrize("B,T,Hk,Hv,chunk,dtype", CASES)
def test_prefill_l2norm_of_unnormalised_rows(cuda_device, B, T, Hk, Hv, chunk, dtype):
    """Rows of length 0.25..3.25 in, unit rows used; one key row is zero."""
    ins = _unnormalised(gdn_inputs.make_inputs(B, T, Hk, Hv, 128, 128, dtype, seed=700 + T,
                                               u_max=0.5, s0_std=0.1))
    ins["k"][0, T // 2, 0] = 0
    y, s, yo, so = _run(ins, L2N, chunk, cuda_device)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    assert rel_err(y, yo) <= TOL[dtype], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[dtype], rel_err(s, so)


@pytest.mark.parametrize("options", [TILED, LOGG, L2N, TILED | LOGG | L2N])
def test_decode_options(cuda_device, options):
    import gated_delta_rule_02_gb300 as gdn
    B, Hk, Hv = 3, 2, 6
    ins = _unnormalised(gdn_inputs.make_inputs(B, 1, Hk, Hv, 128, 128, BF16,
                                               seed=600 + options, u_max=0.5, s0_std=0.1))
    gins = _with_log_gates(ins) if options & LOGG else ins
    d = {n: t.to(cuda_device) for n, t in gins.items()}
    y = torch.empty((B, 1, Hv, 128), dtype=BF16, device=cuda_device)
    s_out = torch.empty_like(d["s0"])
    gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"], s_out, y,
                        options=options)
    torch.cuda.synchronize(cuda_device)
    o = _oracle_equivalent(gins, options)
    yo, so = oracle.gdn_sequential(o["q"], o["k"], o["v"], o["g"], o["beta"], o["s0"])
    assert rel_err(y.float().cpu().numpy(), yo) <= TOL[BF16]
    assert rel_err(s_out.cpu().numpy(), so) <= TOL[BF16]
