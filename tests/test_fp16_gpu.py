"""fp16 inputs (GDN_DTYPE_F16) against the oracle on the same fp16 values:
decode and T <= 32 on the row-packed kernels, longer prefills with 128-wide
heads on the tensor cores (fp16 operands, fp32 accumulation), other head sizes
on the fp32 CUDA-core chunked path."""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from parity_util import TOL, gpu_prefill, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu
F16 = torch.float16


@pytest.mark.parametrize("B,T,Hk,Hv,chunk", [
    (1, 1, 1, 1, 16),
    (2, 20, 2, 6, 32),     # short-T kernel
    (1, 100, 2, 4, 32),    # tensor cores, ragged tail
    (2, 70, 4, 8, 64),
    (1, 33, 1, 2, 16),     # one token past the short-T switch
    (2, 37, 2, 6, 16),     # ragged tail, GQA 3:1, B = 2
    (1, 129, 1, 1, 64),    # 2 chunks + 1 token
    (2, 100, 16, 32, 64),  # B*Hv = 64 heads: the split prep + scan launches
    (1, 150, 8, 48, 32),   # 48 heads, GQA 6:1: the fused launch at its widest
    (1, 1111, 16, 48, 32), # head pair (16, 48), T = 1111
])
def test_prefill_fp16(cuda_device, B, T, Hk, Hv, chunk):
    ins = gdn_inputs.make_inputs(B, T, Hk, Hv, 128, 128, F16, seed=800 + T, u_max=0.5,
                                 s0_std=0.1)
    y, s = gpu_prefill(ins, chunk, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[F16], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[F16], rel_err(s, so)


def test_prefill_fp16_with_options(cuda_device):
    ins = gdn_inputs.make_inputs(1, 60, 2, 4, 128, 128, F16, seed=9, u_max=0.5, s0_std=0.1)
    y, s = gpu_prefill(ins, 32, cuda_device, options=1)  # tiled heads
    idx = torch.tensor([hv % 2 for hv in range(4)])
    o = dict(ins, q=ins["q"][:, :, idx], k=ins["k"][:, :, idx])
    yo, so = oracle_prefill(o)
    assert rel_err(y, yo) <= TOL[F16]
    assert rel_err(s, so) <= TOL[F16]


def test_decode_fp16(cuda_device):
    import gated_delta_rule_02_gb300 as gdn
    B, Hk, Hv = 4, 2, 8
    ins = gdn_inputs.make_inputs(B, 1, Hk, Hv, 128, 128, F16, seed=17, u_max=0.5, s0_std=0.1)
    d = {n: t.to(cuda_device) for n, t in ins.items()}
    y = torch.empty((B, 1, Hv, 128), dtype=F16, device=cuda_device)
    state = d["s0"].clone()
    gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, state, y)
    torch.cuda.synchronize(cuda_device)
    yo, so = oracle.gdn_sequential(*(ins[n] for n in ("q", "k", "v", "g", "beta")), ins["s0"])
    assert rel_err(y.float().cpu().numpy(), yo) <= TOL[F16]
    assert rel_err(state.cpu().numpy(), so) <= TOL[F16]


@pytest.mark.parametrize("options", [2, 4, 6])
def test_prefill_fp16_log_gate_and_l2norm(cuda_device, options):
    """GDN_OPT_LOG_GATE (2) and GDN_OPT_L2NORM_QK (4) on the fp16 tensor-core
    path: the oracle sees exp(g) and the normalised rows."""
    ins = gdn_inputs.make_inputs(1, 140, 2, 4, 128, 128, F16, seed=31 + options, u_max=0.5,
                                 s0_std=0.1)
    dev_in = dict(ins)
    o = dict(ins)
    if options & 2:
        dev_in["g"] = torch.log(ins["g"].double()).to(F16)
        o["g"] = torch.exp(dev_in["g"].double())
    if options & 4:
        gen = torch.Generator().manual_seed(77)
        for n in ("q", "k"):
            raw = (torch.randn(ins[n].shape, generator=gen) * 3.0).to(F16)
            dev_in[n] = raw
            o[n] = raw.double() / raw.double().norm(dim=-1, keepdim=True)
    y, s = gpu_prefill(dev_in, 64, cuda_device, options=options)
    yo, so = oracle_prefill(o)
    assert rel_err(y, yo) <= TOL[F16], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[F16], rel_err(s, so)


def test_prefill_fp16_vanishing_gate(cuda_device):
    """Gates of 1e-7 (near the bottom of fp16's range) underflow the chunk's
    decay products to zero: outputs stay finite and match the oracle."""
    ins = gdn_inputs.make_inputs(1, 70, 1, 2, 128, 128, F16, seed=4, s0_std=0.1)
    ins["g"] = torch.full_like(ins["g"], 1e-7)
    y, s = gpu_prefill(ins, 64, cuda_device)
    yo, so = oracle_prefill(ins)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    assert rel_err(y, yo) <= TOL[F16]
    assert rel_err(s, so) <= TOL[F16]


def test_prefill_fp16_full_size_every_head(cuda_device):
    """The 4096-token, 32-head fp16 workload at full size, in the benchmark's
    launch configuration: every output element, then head by head."""
    w = gdn_inputs.WORKLOADS["prefill_t4096_f16"]
    ins = gdn_inputs.workload_inputs(w)
    y, s = gpu_prefill(ins, w.chunk, cuda_device)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[F16], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[F16], rel_err(s, so)
    for hv in range(w.Hv):
        assert rel_err(y[0, :, hv], yo[0, :, hv]) <= TOL[F16], hv
        assert rel_err(s[0, hv], so[0, hv]) <= TOL[F16], hv
