"""Decode parity: single steps through the C ABI against the fp64 oracle,
with the state carried (in place) across steps."""
import numpy as np
import pytest
import torch

import gated_delta_rule_02_gb300 as gdn
import gdn_inputs
import oracle
from parity_util import NAMES, TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


def run_decode(w, dev, steps, batches=None):
    """Run ``steps`` decode steps of workload ``w`` on the GPU, in place.
    Returns per-step y (optionally restricted to batch rows ``batches``),
    the final state, and the oracle's view of the same inputs."""
    s = gdn_inputs.workload_inputs(w, step=0)["s0"].to(dev)
    ys, step_inputs = [], []
    for i in range(steps):
        ins = gdn_inputs.workload_inputs(w, step=i)
        d = to_device(ins, dev)
        y = torch.empty((w.B, 1, w.Hv, w.Dv), dtype=w.torch_dtype, device=dev)
        gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], s, s, y)
        ys.append(y.float().cpu().numpy())
        step_inputs.append(ins)
    torch.cuda.synchronize(dev)
    return np.stack(ys), s.cpu().numpy(), step_inputs


def oracle_decode(w, step_inputs, batches):
    s0 = gdn_inputs.workload_inputs(w, step=0)["s0"][batches]
    stacked = [torch.stack([ins[n][batches] for ins in step_inputs]) for n in NAMES]
    return oracle.gdn_decode_steps(*stacked, s0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("Hk,Hv", [(2, 4), (1, 3), (4, 4)])
def test_decode_small_matches_oracle(cuda_device, dtype, Hk, Hv):
    w = gdn_inputs.Workload("decode_small", B=2, T=1, Hk=Hk, Hv=Hv, Dk=128, Dv=128,
                            dtype="f32" if dtype == torch.float32 else "bf16",
                            chunk=0, u_max=0.1, s0_std=0.1, seed=77, steps=6)
    ys, s, ins = run_decode(w, cuda_device, w.steps)
    batches = list(range(w.B))
    yo, so = oracle_decode(w, ins, batches)
    tol = TOL[dtype]
    for i in range(w.steps):
        assert rel_err(ys[i], yo[i]) <= tol, (i, rel_err(ys[i], yo[i]))
    assert rel_err(s, so) <= tol


def test_decode_full_size_256_steps(cuda_device):
    """The B=64 decode workload, 256 steps at full size with the state
    carried in place; every step's y and the final state of every batch row
    and value head are checked against the oracle."""
    w = gdn_inputs.WORKLOADS["decode_b64"]
    ys, s, ins = run_decode(w, cuda_device, w.steps)
    assert np.all(np.isfinite(ys)) and np.all(np.isfinite(s))
    batches = list(range(w.B))
    yo, so = oracle_decode(w, ins, batches)
    for i in range(w.steps):
        assert rel_err(ys[i], yo[i]) <= TOL[torch.bfloat16], i
    assert rel_err(s, so) <= TOL[torch.bfloat16]
    for b in range(w.B):
        for hv in range(w.Hv):
            assert rel_err(s[b, hv], so[b, hv]) <= TOL[torch.bfloat16], (b, hv)


def test_decode_steps_equal_prefill(cuda_device):
    """N decode steps equal one N-token prefill of the same tokens."""
    ins = gdn_inputs.make_inputs(2, 9, 1, 2, 128, 128, torch.float32, seed=31,
                                 s0_std=0.1)
    d = to_device(ins, cuda_device)
    yp, sp = gdn.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"], chunk=16)
    s = d["s0"].clone()
    ys = []
    for t in range(9):
        sl = {n: d[n][:, t:t + 1].contiguous() for n in NAMES}
        ys.append(gdn.decode_step(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], s))
    yd = torch.cat(ys, dim=1)
    assert rel_err(yd.cpu().numpy(), yp.cpu().numpy()) <= 1e-5
    assert rel_err(s.cpu().numpy(), sp.cpu().numpy()) <= 1e-5


def test_decode_out_of_place_leaves_input(cuda_device):
    ins = gdn_inputs.make_inputs(1, 1, 1, 2, 128, 128, torch.bfloat16, seed=8,
                                 s0_std=0.1)
    d = to_device(ins, cuda_device)
    s_in = d["s0"].clone()
    s_out = torch.empty_like(s_in)
    y = torch.empty((1, 1, 2, 128), dtype=torch.bfloat16, device=cuda_device)
    gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], s_in, s_out, y)
    torch.cuda.synchronize()
    assert torch.equal(s_in, d["s0"])
    yo, so = oracle.gdn_sequential(*(ins[n] for n in NAMES), ins["s0"])
    assert rel_err(s_out.cpu().numpy(), so) <= TOL[torch.bfloat16]
    assert rel_err(y.float().cpu().numpy(), yo) <= TOL[torch.bfloat16]
