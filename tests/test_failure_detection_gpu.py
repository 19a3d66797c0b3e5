"""Failure detection without a GPU fault.

Every wait inside the tensor-core kernels is bounded: when its producer never
comes (a lost TMA, a tensor-core commit, a prep CTA that never raises a tile
flag), the wait gives up after 2 s, records a timeout in a device error word
and the kernel returns.  gdn_selftest_wait_timeout runs those same two waits
on an mbarrier phase and a flag that nothing completes; the host must then see
GDN_ERR_DEVICE_TIMEOUT from gdn_device_status, be able to clear it, and the
context must stay usable for the next prefill.
"""
import time

import pytest
import torch

import gated_delta_rule_02_gb300 as gdn
import gdn_inputs
from parity_util import TOL, gpu_prefill, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def test_bounded_waits_report_timeout_and_context_survives(cuda_device):
    torch.cuda.synchronize(cuda_device)
    assert gdn.gdn_device_status(clear=True) in (gdn.GDN_OK, gdn.GDN_ERR_DEVICE_TIMEOUT)
    assert gdn.gdn_device_status() == gdn.GDN_OK

    t0 = time.perf_counter()
    gdn.gdn_selftest_wait_timeout(device=cuda_device)
    torch.cuda.synchronize(cuda_device)
    elapsed = time.perf_counter() - t0
    # Two waits of 2 s each ran out; neither returned early, and both ended.
    assert 3.5 <= elapsed <= 60.0, elapsed

    assert gdn.gdn_device_status() == gdn.GDN_ERR_DEVICE_TIMEOUT
    assert gdn.gdn_device_status(clear=True) == gdn.GDN_ERR_DEVICE_TIMEOUT
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert "timed out" in gdn.gdn_status_string(gdn.GDN_ERR_DEVICE_TIMEOUT)

    # The context is intact: the tensor-core prefill still matches the oracle
    # and leaves the error word clear.
    ins = gdn_inputs.make_inputs(1, 200, 2, 4, 128, 128, dtype=torch.bfloat16, seed=901)
    y, s = gpu_prefill(ins, 64, cuda_device)
    yo, so = oracle_prefill(ins)
    assert rel_err(y, yo) <= TOL[torch.bfloat16]
    assert rel_err(s, so) <= TOL[torch.bfloat16]
    assert gdn.gdn_device_status() == gdn.GDN_OK
