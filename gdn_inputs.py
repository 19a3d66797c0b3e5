"""Seeded synthetic inputs for the gated delta rule.

Shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``, and by
both sides of every parity check (the CUDA library and the fp64 oracle).
This module holds none of the method's arithmetic: only the input recipe.

Recipe (per workload, all draws from one ``torch.Generator`` seeded per
workload, generated on the CPU in fp32 and then cast to the workload dtype):
  q, k   ~ N(0, 1), each (b, t, head) row divided by its L2 norm
  v      ~ N(0, 1)
  g      = exp(-u), u ~ U(0, u_max); with ``heavy_frac`` > 0 each (b, t, hv)
           gate independently, with that probability, draws u ~ U(0, heavy_umax)
  beta   = sigmoid(N(0, 1))
  S_0    ~ N(0, s0_std^2) in fp32 (zeros when s0_std == 0)
The oracle reads the values after the cast, widened exactly to fp64.
"""
from __future__ import annotations

import dataclasses

import torch


DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    dtype: str          # "f32", "bf16" or "f16"
    chunk: int
    u_max: float
    s0_std: float
    seed: int
    heavy_frac: float = 0.0
    heavy_umax: float = 5.0
    steps: int = 0      # decode workloads: number of successive T=1 steps

    @property
    def torch_dtype(self):
        return DTYPES[self.dtype]

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The workloads of the benchmark plan, named by what they are.
WORKLOADS = {
    "fp32_t64": Workload("fp32_t64", B=1, T=64, Hk=2, Hv=2, Dk=128, Dv=128,
                         dtype="f32", chunk=32, u_max=0.1, s0_std=0.1, seed=1000),
    "prefill_t4096": Workload("prefill_t4096", B=1, T=4096, Hk=16, Hv=32, Dk=128,
                              Dv=128, dtype="bf16", chunk=64, u_max=0.1,
                              s0_std=0.0, seed=1001),
    "prefill_b4_t2048": Workload("prefill_b4_t2048", B=4, T=2048, Hk=16, Hv=48,
                                 Dk=128, Dv=128, dtype="bf16", chunk=32, u_max=1.0,
                                 s0_std=0.1, seed=1002),
    "decode_b64": Workload("decode_b64", B=64, T=1, Hk=16, Hv=32, Dk=128, Dv=128,
                           dtype="bf16", chunk=0, u_max=0.1, s0_std=0.1,
                           seed=1003, steps=256),
    "prefill_t65536": Workload("prefill_t65536", B=1, T=65536, Hk=16, Hv=32,
                               Dk=128, Dv=128, dtype="bf16", chunk=64, u_max=0.1,
                               s0_std=0.0, seed=1004, heavy_frac=0.1,
                               heavy_umax=5.0),
    # A short multi-token call (the short-T sequential path): 16 tokens for
    # each of 64 sequences, the decode shape; the state (134 MB) dominates.
    "prefill_b64_t16": Workload("prefill_b64_t16", B=64, T=16, Hk=16, Hv=32, Dk=128,
                                Dv=128, dtype="bf16", chunk=64, u_max=0.1,
                                s0_std=0.1, seed=1005),
    # The headline shape with fp16 inputs (the other 16-bit type the tensor
    # cores take).
    "prefill_t4096_f16": Workload("prefill_t4096_f16", B=1, T=4096, Hk=16, Hv=32, Dk=128,
                                  Dv=128, dtype="f16", chunk=64, u_max=0.1,
                                  s0_std=0.0, seed=1006),
    # The headline shape at the other head sizes of the plan (64 and 256).
    "prefill_t4096_d64": Workload("prefill_t4096_d64", B=1, T=4096, Hk=16, Hv=32, Dk=64,
                                  Dv=64, dtype="bf16", chunk=64, u_max=0.1,
                                  s0_std=0.0, seed=1007),
    "prefill_t4096_d256": Workload("prefill_t4096_d256", B=1, T=4096, Hk=16, Hv=32, Dk=256,
                                   Dv=256, dtype="bf16", chunk=64, u_max=0.1,
                                   s0_std=0.0, seed=1008),
}


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def make_inputs(B, T, Hk, Hv, Dk, Dv, dtype=torch.bfloat16, seed=0, u_max=0.1,
                s0_std=0.1, heavy_frac=0.0, heavy_umax=5.0, draw_state=True):
    """One seeded draw of (q, k, v, g, beta, s0) on the CPU.

    Returns a dict of CPU tensors: q, k [B,T,Hk,Dk], v [B,T,Hv,Dv],
    g, beta [B,T,Hv] in ``dtype`` and s0 [B,Hv,Dv,Dk] in fp32 (drawn last,
    so ``draw_state=False`` leaves the other tensors unchanged and omits it).
    """
    if isinstance(dtype, str):
        dtype = DTYPES[dtype]
    gen = torch.Generator().manual_seed(int(seed))
    q = _unit_rows(torch.randn((B, T, Hk, Dk), generator=gen))
    k = _unit_rows(torch.randn((B, T, Hk, Dk), generator=gen))
    v = torch.randn((B, T, Hv, Dv), generator=gen)
    u = torch.rand((B, T, Hv), generator=gen) * u_max
    if heavy_frac > 0.0:
        heavy = torch.rand((B, T, Hv), generator=gen) < heavy_frac
        u = torch.where(heavy, torch.rand((B, T, Hv), generator=gen) * heavy_umax, u)
    g = torch.exp(-u)
    beta = torch.sigmoid(torch.randn((B, T, Hv), generator=gen))
    out = {name: t.to(dtype).contiguous() for name, t in
           (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta))}
    if draw_state:
        if s0_std > 0.0:
            out["s0"] = (torch.randn((B, Hv, Dv, Dk), generator=gen) * s0_std).contiguous()
        else:
            out["s0"] = torch.zeros((B, Hv, Dv, Dk))
    return out


def workload_inputs(w: Workload, step: int | None = None):
    """Inputs of a prefill workload, or of decode step ``step`` of a decode one.

    Decode steps draw fresh, independent inputs per step from seed
    ``w.seed + 7919 * step`` (T = 1); the initial state comes from step 0's
    draw (later steps carry no ``s0``) and is carried by the caller afterwards.
    """
    seed = w.seed if step is None else w.seed + 7919 * step
    return make_inputs(w.B, w.T, w.Hk, w.Hv, w.Dk, w.Dv, w.torch_dtype, seed,
                       w.u_max, w.s0_std, w.heavy_frac, w.heavy_umax,
                       draw_state=not step)
