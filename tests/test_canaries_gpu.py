"""Canary-guarded outputs: y and the final state are views into larger buffers
whose guard regions before and after hold a sentinel; after each kind of call
the guards must be untouched and the outputs correct.  Every path is covered:
the fused tensor-core prefill (ragged tail), the split tensor-core prefill
(many heads), the short-T kernel, the fp32 chunked path and decode.  A stray
write lands in the guard (inside the same allocation), so it is reported
rather than faulting.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_02_gb300 as gdn
import gdn_inputs
from parity_util import NAMES, TOL, oracle_prefill, rel_err, to_device

pytestmark = pytest.mark.gpu

GUARD = 1024          # elements on each side (>= 2 KB: keeps every view 256-byte aligned)


def guarded(shape, dtype, dev, fill):
    n = int(np.prod(shape))
    buf = torch.full((GUARD + n + GUARD,), fill, dtype=dtype, device=dev)
    return buf, buf[GUARD:GUARD + n].view(shape)


def guards_intact(buf, fill):
    head, tail = buf[:GUARD], buf[-GUARD:]
    ref = torch.full_like(head, fill)
    return torch.equal(head, ref) and torch.equal(tail, ref)


CASES = [  # (B, T, Hk, Hv, dtype, chunk): the path each one takes
    (1, 200, 2, 4, torch.bfloat16, 64),     # fused tensor-core kernel, ragged tail
    (2, 70, 16, 32, torch.bfloat16, 32),    # split tensor-core path (B*Hv > SMs/3)
    (3, 19, 2, 6, torch.bfloat16, 64),      # short-T kernel
    (1, 100, 2, 4, torch.float32, 32),      # fp32 chunked path
]


@pytest.mark.parametrize("B,T,Hk,Hv,dtype,chunk", CASES)
def test_prefill_writes_only_its_outputs(cuda_device, B, T, Hk, Hv, dtype, chunk):
    ins = gdn_inputs.make_inputs(B, T, Hk, Hv, 128, 128, dtype=dtype, seed=600 + T)
    d = to_device(ins, cuda_device)
    ybuf, y = guarded((B, T, Hv, 128), dtype, cuda_device, -7.0)
    sbuf, s = guarded((B, Hv, 128, 128), torch.float32, cuda_device, -7.0)
    nb = gdn.gdn_prefill_workspace_bytes(B, T, Hk, Hv, 128, 128, chunk, dtype)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=cuda_device)
    gdn.gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"], s, y, chunk,
                    workspace=ws if nb else None)
    torch.cuda.synchronize(cuda_device)
    assert guards_intact(ybuf, -7.0) and guards_intact(sbuf, -7.0)
    yo, so = oracle_prefill(ins)
    assert rel_err(y.float().cpu().numpy(), yo) <= TOL[dtype]
    assert rel_err(s.cpu().numpy(), so) <= TOL[dtype]


def test_decode_writes_only_its_outputs(cuda_device):
    B, Hk, Hv = 4, 2, 8
    ins = gdn_inputs.make_inputs(B, 1, Hk, Hv, 128, 128, dtype=torch.bfloat16, seed=650)
    d = to_device(ins, cuda_device)
    ybuf, y = guarded((B, 1, Hv, 128), torch.bfloat16, cuda_device, -7.0)
    sbuf, s = guarded((B, Hv, 128, 128), torch.float32, cuda_device, -7.0)
    gdn.gdn_decode_step(*(d[n] for n in NAMES), d["s0"], s, y)
    torch.cuda.synchronize(cuda_device)
    assert guards_intact(ybuf, -7.0) and guards_intact(sbuf, -7.0)
    yo, so = oracle_prefill(ins)
    assert rel_err(y.float().cpu().numpy(), yo) <= TOL[torch.bfloat16]
    assert rel_err(s.cpu().numpy(), so) <= TOL[torch.bfloat16]
