"""fp16 inputs (GDN_DTYPE_F16): decode and T <= 32 on the row-packed kernels,
longer prefills on the fp32 CUDA-core chunked path, against the oracle on the
same fp16 values."""
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
    (1, 100, 2, 4, 32),    # chunked fp32 path, ragged tail
    (2, 70, 4, 8, 64),
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
