"""Shared helpers for the parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare them.

Tolerances (max |gpu - oracle| <= tol * max |oracle|, on y and on the final
state): 1e-4 for fp32 inputs and 2e-2 for bf16 inputs; 2e-3 for fp16 inputs (computed
in fp32; y is rounded to fp16, 2^-11 relative).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2, torch.float16: 2e-3}
NAMES = ("q", "k", "v", "g", "beta")


def rel_err(a, ref) -> float:
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(a - ref)) / scale)


def to_device(ins, dev):
    return {n: t.to(dev) for n, t in ins.items() if t is not None}


def gpu_prefill(ins, chunk, dev, state_mode="given", options=0):
    """state_mode: 'given' (s0 -> new state_out), 'null' (state_in = NULL),
    'inplace' (state_in is state_out).  options: GDN_OPT_* bits."""
    import gated_delta_rule_02_gb300 as gdn
    d = to_device(ins, dev)
    B, T, Hk, Dk = d["q"].shape
    Hv, Dv = d["v"].shape[2], d["v"].shape[3]
    y = torch.empty((B, T, Hv, Dv), dtype=d["q"].dtype, device=dev)
    if state_mode == "inplace":
        s_in = s_out = d["s0"].clone()
    else:
        s_in = None if state_mode == "null" else d["s0"]
        s_out = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=dev)
    gdn.gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], s_in, s_out, y, chunk,
                    options=options)
    torch.cuda.synchronize(dev)
    return y.float().cpu().numpy(), s_out.cpu().numpy()


def oracle_prefill(ins, zero_state=False):
    s0 = None if zero_state else ins["s0"]
    return oracle.gdn_sequential(*(ins[n] for n in NAMES), s0)
