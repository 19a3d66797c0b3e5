"""Head sizes other than 128 (Dk, Dv in {64, 128, 256}): the decode kernel, the
short-T sequential kernel, the warp-level tensor-core chunked paths (16-bit
inputs at Dk = Dv = 64 and at 256) and the fp32 SIMT chunked path (every other
case),
against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_02_gb300 as gdn
import gdn_inputs
import oracle
from parity_util import NAMES, TOL, gpu_prefill, oracle_prefill, rel_err, to_device

pytestmark = pytest.mark.gpu

PAIRS = [(64, 64), (256, 256), (64, 128), (256, 64), (128, 256)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("Dk,Dv", PAIRS)
def test_decode_head_sizes(cuda_device, dtype, Dk, Dv):
    """Four decode steps with the state carried in place."""
    B, Hk, Hv, steps = 2, 2, 4, 4
    ins = gdn_inputs.make_inputs(B, steps, Hk, Hv, Dk, Dv, dtype=dtype, seed=310 + Dk + Dv)
    d = to_device(ins, cuda_device)
    s = d["s0"].clone()
    ys = []
    for t in range(steps):
        y = torch.empty((B, 1, Hv, Dv), dtype=dtype, device=cuda_device)
        gdn.gdn_decode_step(*(d[n][:, t:t + 1].contiguous() for n in NAMES), s, s, y)
        ys.append(y.float().cpu().numpy())
    torch.cuda.synchronize(cuda_device)
    yo, so = oracle_prefill(ins)
    y = np.concatenate(ys, axis=1)
    assert rel_err(y, yo) <= TOL[dtype], rel_err(y, yo)
    assert rel_err(s.cpu().numpy(), so) <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Dk,Dv", PAIRS)
def test_short_prefill_head_sizes(cuda_device, dtype, Dk, Dv):
    """T = 19 (the short-T sequential kernel), state given."""
    ins = gdn_inputs.make_inputs(2, 19, 2, 4, Dk, Dv, dtype=dtype, seed=330 + Dk + Dv)
    y, s = gpu_prefill(ins, 32, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[dtype]
    assert rel_err(s, so) <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Dk,Dv", PAIRS)
@pytest.mark.parametrize("chunk", [16, 64])
def test_chunked_prefill_head_sizes(cuda_device, dtype, Dk, Dv, chunk):
    """T = 100 (several chunks and a ragged tail) on the chunked paths: at Dk =
    Dv = 64 or 256 with 16-bit inputs the warp-level tensor-core ones, else the
    SIMT one (where at Dk = Dv = 256 a chunk of 64 runs as two chunks of 32)."""
    ins = gdn_inputs.make_inputs(1, 100, 2, 4, Dk, Dv, dtype=dtype, seed=350 + Dk + Dv + chunk)
    y, s = gpu_prefill(ins, chunk, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[dtype], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[dtype]


@pytest.mark.parametrize("Dk,Dv", [(64, 64), (256, 128)])
def test_head_sizes_with_l2norm_and_null_state(cuda_device, Dk, Dv):
    """In-kernel L2 normalisation of q and k at other head sizes, zero initial
    state, on both the short and the chunked path."""
    for T in (9, 70):
        ins = gdn_inputs.make_inputs(1, T, 1, 2, Dk, Dv, dtype=torch.float32, seed=370 + T)
        raw = dict(ins)
        for n in ("q", "k"):
            raw[n] = ins[n] * torch.linspace(0.5, 3.0, T)[None, :, None, None]
        y, s = gpu_prefill(raw, 32, cuda_device, state_mode="null", options=gdn.GDN_OPT_L2NORM_QK)
        yo, so = oracle_prefill(ins, zero_state=True)
        assert rel_err(y, yo) <= 1e-4, (T, rel_err(y, yo))
        assert rel_err(s, so) <= 1e-4


MMA_CASES = [
    # (B, T, Hk, Hv, dtype): Dk = Dv = 64, 16-bit inputs, T > 32
    (1, 33, 1, 1, torch.bfloat16),    # one chunk and one token
    (1, 64, 2, 4, torch.bfloat16),    # two whole chunks
    (2, 257, 2, 6, torch.bfloat16),   # GQA 3:1, B = 2, ragged tail
    (1, 1000, 4, 8, torch.float16),
    (3, 95, 1, 2, torch.float16),
    (4, 40, 8, 64, torch.bfloat16),   # 256 heads
]


@pytest.mark.parametrize("B,T,Hk,Hv,dtype", MMA_CASES)
def test_mma_prefill_d64(cuda_device, B, T, Hk, Hv, dtype):
    ins = gdn_inputs.make_inputs(B, T, Hk, Hv, 64, 64, dtype=dtype, seed=390 + T + Hv,
                                 u_max=0.5, s0_std=0.1)
    y, s = gpu_prefill(ins, 32, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[dtype], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[dtype], rel_err(s, so)


@pytest.mark.parametrize("mode", ["null", "inplace"])
def test_mma_prefill_d64_state_modes(cuda_device, mode):
    ins = gdn_inputs.make_inputs(2, 130, 2, 4, 64, 64, dtype=torch.bfloat16, seed=395, s0_std=0.1)
    y, s = gpu_prefill(ins, 64, cuda_device, state_mode=mode)
    yo, so = oracle_prefill(ins, zero_state=(mode == "null"))
    assert rel_err(y, yo) <= TOL[torch.bfloat16]
    assert rel_err(s, so) <= TOL[torch.bfloat16]


MMA256_CASES = [
    # (B, T, Hk, Hv, dtype): Dk = Dv = 256, 16-bit inputs, T > 32 (the head's
    # state over four CTAs, keys split over warp pairs)
    (1, 33, 1, 1, torch.bfloat16),
    (2, 100, 2, 4, torch.bfloat16),
    (1, 257, 1, 3, torch.float16),
]


@pytest.mark.parametrize("B,T,Hk,Hv,dtype", MMA256_CASES)
def test_mma_prefill_d256(cuda_device, B, T, Hk, Hv, dtype):
    ins = gdn_inputs.make_inputs(B, T, Hk, Hv, 256, 256, dtype=dtype, seed=410 + T + Hv,
                                 u_max=0.5, s0_std=0.1)
    y, s = gpu_prefill(ins, 32, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[dtype], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[dtype], rel_err(s, so)


@pytest.mark.parametrize("mode", ["null", "inplace"])
def test_mma_prefill_d256_state_modes(cuda_device, mode):
    ins = gdn_inputs.make_inputs(1, 70, 2, 2, 256, 256, dtype=torch.bfloat16, seed=415,
                                 s0_std=0.1)
    y, s = gpu_prefill(ins, 64, cuda_device, state_mode=mode)
    yo, so = oracle_prefill(ins, zero_state=(mode == "null"))
    assert rel_err(y, yo) <= TOL[torch.bfloat16]
    assert rel_err(s, so) <= TOL[torch.bfloat16]
