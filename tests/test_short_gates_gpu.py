"""Gates at the limits of the short-T kernels.

The sequential short-T kernel (fp32 inputs, head sizes other than 128/128)
keeps each head's state as gam * St, gam the product of the gates since the
last renormalisation, and brings the registers back to scale when gam * g_t
leaves [2^-24, 2^24]; the one-chunk tensor-core kernel (16-bit inputs at
128/128) forms its decays from log2 prefix sums, clamped at -1000 per token.
These cases drive both: long runs of small gates (the product falls below
2^-24 within a few tokens), exact zero gates (a reset of the state), gates of
one (no decay), and a mix, on two of the four heads while the other two keep
the random gates; compared with the fp64 oracle.
"""
import pytest
import torch

import gdn_inputs
from parity_util import TOL, gpu_prefill, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

MIX = [0.9, 0.0, 1.0, 0.5, 0.0, 0.0, 0.95, 1e-4, 1e-3, 0.99, 1e-3, 1e-3, 1.0, 0.0, 0.7, 1e-4]
PATTERNS = {
    "small": lambda T: [1e-3] * T,
    "zeros": lambda T: [0.0 if t % 3 == 1 else 0.8 for t in range(T)],
    "ones": lambda T: [1.0] * T,
    "mix": lambda T: [MIX[t % len(MIX)] for t in range(T)],
}


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("pattern", sorted(PATTERNS))
@pytest.mark.parametrize("T,Dk,Dv", [(16, 128, 128), (5, 128, 128), (32, 64, 64), (11, 256, 128)])
def test_short_prefill_extreme_gates(cuda_device, dtype, pattern, T, Dk, Dv):
    ins = gdn_inputs.make_inputs(2, T, 2, 4, Dk, Dv, dtype=dtype, seed=500 + T + Dk)
    gates = torch.tensor(PATTERNS[pattern](T), dtype=torch.float64).to(dtype)
    ins["g"][:, :, :2] = gates[None, :, None]
    y, s = gpu_prefill(ins, 32, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[dtype], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[dtype], rel_err(s, so)
