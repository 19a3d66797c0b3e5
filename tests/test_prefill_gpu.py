"""Prefill parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every case is compared element by element over every output, the large
workloads included: they run at full size in the launch configuration the
benchmark times, and the oracle follows all of their heads.
"""
import numpy as np
import pytest
import torch

import gdn_inputs
from parity_util import TOL, gpu_prefill, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

F32, BF16, F16 = torch.float32, torch.bfloat16, torch.float16

SMALL = [
    # (B, T, Hk, Hv, chunk, dtype, u_max)
    (1, 64, 2, 2, 32, F32, 0.1),     # the fp32 workload, whole
    (1, 1, 1, 1, 16, BF16, 0.1),     # a single token
    (1, 3, 1, 2, 16, BF16, 0.1),     # shorter than one chunk
    (2, 37, 2, 6, 16, BF16, 1.0),    # ragged tail, GQA 3:1, B = 2
    (1, 100, 2, 4, 32, BF16, 0.1),   # several chunks + ragged tail
    (1, 129, 1, 1, 64, BF16, 0.1),   # 2 chunks + 1 token
    (1, 200, 2, 2, 64, F32, 0.5),
    (3, 70, 1, 3, 32, F32, 1.0),
    (1, 64, 1, 2, 64, BF16, 5.0),    # fast decay: G underflows inside a chunk
    (2, 100, 16, 32, 64, BF16, 0.3), # B*Hv = 64 heads: the split prep + scan launches
    (1, 150, 8, 48, 32, BF16, 0.3),  # 48 heads, GQA 6:1: the fused launch at its widest
    (2, 257, 24, 24, 64, BF16, 0.3), # head pair (24, 24), B = 2, T = 4 chunks + 1 token
    (1, 1111, 16, 48, 32, BF16, 0.5),  # head pair (16, 48), T = 1111
    (1, 257, 24, 24, 16, F32, 0.1),
]


@pytest.mark.parametrize("B,T,Hk,Hv,chunk,dtype,u_max", SMALL)
def test_prefill_small_matches_oracle(cuda_device, B, T, Hk, Hv, chunk, dtype, u_max):
    ins = gdn_inputs.make_inputs(B, T, Hk, Hv, 128, 128, dtype, seed=100 + T + Hv,
                                 u_max=u_max, s0_std=0.1)
    y, s = gpu_prefill(ins, chunk, cuda_device)
    yo, so = oracle_prefill(ins)
    tol = TOL[dtype]
    assert rel_err(y, yo) <= tol, rel_err(y, yo)
    assert rel_err(s, so) <= tol, rel_err(s, so)


@pytest.mark.parametrize("mode", ["null", "inplace"])
def test_prefill_state_modes(cuda_device, mode):
    ins = gdn_inputs.make_inputs(1, 45, 1, 2, 128, 128, BF16, seed=5, s0_std=0.1)
    y, s = gpu_prefill(ins, 16, cuda_device, state_mode=mode)
    yo, so = oracle_prefill(ins, zero_state=(mode == "null"))
    assert rel_err(y, yo) <= TOL[BF16]
    assert rel_err(s, so) <= TOL[BF16]


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_prefill_chunk_width_invariance(cuda_device, chunk):
    """A recurrence right at only one chunk width is not the recurrence
    (ferrox-core ``the_device_chunk_matches_this_one``): every width agrees
    with the oracle on the same draw."""
    ins = gdn_inputs.make_inputs(1, 150, 2, 4, 128, 128, BF16, seed=9, u_max=0.3,
                                 s0_std=0.1)
    y, s = gpu_prefill(ins, chunk, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[BF16]
    assert rel_err(s, so) <= TOL[BF16]


def test_prefill_split_resume(cuda_device):
    """prefill(T1) then prefill(T2) from the carried state = prefill(T1+T2)."""
    ins = gdn_inputs.make_inputs(1, 160, 1, 2, 128, 128, F32, seed=21, s0_std=0.1)
    y, s = gpu_prefill(ins, 32, cuda_device)
    a = {n: t[:, :70] if n != "s0" else t for n, t in ins.items()}
    ya, sa = gpu_prefill(a, 32, cuda_device)
    b = {n: t[:, 70:].contiguous() if n != "s0" else torch.from_numpy(sa)
         for n, t in ins.items()}
    yb, sb = gpu_prefill(b, 32, cuda_device)
    assert rel_err(np.concatenate([ya, yb], axis=1), y) <= 1e-5
    assert rel_err(sb, s) <= 1e-5


def test_prefill_is_deterministic(cuda_device):
    ins = gdn_inputs.make_inputs(2, 77, 2, 4, 128, 128, BF16, seed=3, s0_std=0.1)
    y1, s1 = gpu_prefill(ins, 32, cuda_device)
    y2, s2 = gpu_prefill(ins, 32, cuda_device)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


def test_prefill_vanishing_gate_is_finite(cuda_device):
    """Gates of 1e-30 (bf16 keeps its exponent range) underflow the chunk's
    decay products to zero: outputs stay finite and match the oracle
    (ferrox-core ``a_vanishing_decay_is_forgetting_and_not_a_division``)."""
    ins = gdn_inputs.make_inputs(1, 70, 1, 2, 128, 128, BF16, seed=4, s0_std=0.1)
    ins["g"] = torch.full_like(ins["g"], 1e-30)
    y, s = gpu_prefill(ins, 64, cuda_device)
    yo, so = oracle_prefill(ins)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    assert rel_err(y, yo) <= TOL[BF16]
    assert rel_err(s, so) <= TOL[BF16]


SHORT = [
    # (B, T, Hk, Hv, dtype): T <= 32 runs a short-T kernel: 16-bit inputs the
    # one-chunk tensor-core kernel (16 or 32 token rows), fp32 inputs the
    # sequential one
    (1, 1, 1, 1, BF16),
    (2, 7, 2, 6, BF16),     # GQA 3:1
    (3, 16, 4, 8, F32),
    (1, 31, 16, 32, BF16),
    (2, 32, 8, 16, F32),
    (4, 16, 16, 32, BF16),  # a full 16-row chunk, 128 heads
    (2, 17, 2, 4, BF16),    # one token past the 16-row chunk
    (1, 32, 2, 2, BF16),    # a full 32-row chunk
    (2, 16, 2, 4, F16),
    (1, 32, 1, 3, F16),
    (3, 9, 2, 2, F16),
]


@pytest.mark.parametrize("B,T,Hk,Hv,dtype", SHORT)
def test_prefill_short_t_matches_oracle(cuda_device, B, T, Hk, Hv, dtype):
    ins = gdn_inputs.make_inputs(B, T, Hk, Hv, 128, 128, dtype, seed=300 + T + Hv,
                                 u_max=0.5, s0_std=0.1)
    y, s = gpu_prefill(ins, 64, cuda_device)
    yo, so = oracle_prefill(ins)
    # the sequential kernel computes in fp32 throughout: fp32 inputs meet 1e-4
    tol = TOL[dtype]
    assert rel_err(y, yo) <= tol, rel_err(y, yo)
    assert rel_err(s, so) <= tol, rel_err(s, so)


@pytest.mark.parametrize("mode", ["null", "inplace"])
def test_prefill_short_t_state_modes(cuda_device, mode):
    ins = gdn_inputs.make_inputs(1, 20, 2, 4, 128, 128, BF16, seed=8, s0_std=0.1)
    y, s = gpu_prefill(ins, 32, cuda_device, state_mode=mode)
    yo, so = oracle_prefill(ins, zero_state=(mode == "null"))
    assert rel_err(y, yo) <= TOL[BF16]
    assert rel_err(s, so) <= TOL[BF16]


def test_prefill_short_and_chunked_paths_agree(cuda_device):
    """T = 32 (sequential kernel) then one more token, against T = 33 in one
    call (chunked tensor-core path): the same rule on both sides of the switch."""
    ins = gdn_inputs.make_inputs(1, 33, 2, 4, 128, 128, BF16, seed=33, s0_std=0.1)
    y, s = gpu_prefill(ins, 32, cuda_device)
    a = {n: t[:, :32] if n != "s0" else t for n, t in ins.items()}
    ya, sa = gpu_prefill(a, 32, cuda_device)
    b = {n: t[:, 32:].contiguous() if n != "s0" else torch.from_numpy(sa)
         for n, t in ins.items()}
    yb, sb = gpu_prefill(b, 32, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(np.concatenate([ya, yb], axis=1), yo) <= TOL[BF16]
    assert rel_err(sb, so) <= TOL[BF16]
    assert rel_err(y, yo) <= TOL[BF16]
    assert rel_err(s, so) <= TOL[BF16]


FULL = ["prefill_t4096", "prefill_b4_t2048", "prefill_t65536", "prefill_b64_t16",
        "prefill_t4096_d64", "prefill_t4096_d256"]


@pytest.mark.parametrize("name", FULL)
def test_prefill_full_size_every_head(cuda_device, name):
    """The large workloads at full size, in the launch configuration the
    benchmark times, compared element by element over every output: all of
    y and the whole final state, every (b, hv) head (ferrox-core
    ``the_device_chunk_matches_this_one`` checks every output the same way)."""
    w = gdn_inputs.WORKLOADS[name]
    ins = gdn_inputs.workload_inputs(w)
    y, s = gpu_prefill(ins, w.chunk, cuda_device)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    yo, so = oracle_prefill(ins)
    assert y.shape == yo.shape and s.shape == so.shape
    assert rel_err(y, yo) <= TOL[BF16], rel_err(y, yo)
    assert rel_err(s, so) <= TOL[BF16], rel_err(s, so)
    # and head by head, so that a head-local fault cannot hide under the
    # scale of the others
    for b in range(w.B):
        for hv in range(w.Hv):
            assert rel_err(y[b, :, hv], yo[b, :, hv]) <= TOL[BF16], (b, hv)
            assert rel_err(s[b, hv], so[b, hv]) <= TOL[BF16], (b, hv)


def test_no_device_wait_timed_out(cuda_device):
    """No bounded device-side wait gave up during the runs above."""
    import gated_delta_rule_02_gb300 as gdn
    assert gdn.gdn_device_status() == gdn.GDN_OK
