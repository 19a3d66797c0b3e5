"""gdn_prefill_noalloc: the prefill for callers that cannot allocate device
memory (plug-ins handed device pointers but no allocator of their own, paths
that cannot take cudaMalloc's implicit synchronisation).  It uses a fixed scratch
buffer built into the library instead of a caller workspace.

This file is collected last on purpose.  The tests call the entry point
directly through the C ABI, twice in a row (the buffer keeps the previous
call's contents), and captured into a CUDA graph and replayed, and check each
result against gdn_prefill with a caller workspace, within the parity
tolerance.  They pass on their own in a fresh process and after the other GPU
tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_delta_rule_02_gb300 as gdn
import gdn_inputs
from parity_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_prefill_matches_workspace_prefill(cuda_device):
    L = gdn.lib()
    B, T, Hk, Hv, chunk = 2, 300, 2, 4, 32            # 40 tiles: inside the fixed buffer
    ins = to_device(gdn_inputs.make_inputs(B, T, Hk, Hv, 128, 128, torch.bfloat16, seed=41,
                                           u_max=0.3, s0_std=0.1), cuda_device)
    y_ref, s_ref = gdn.prefill(ins["q"], ins["k"], ins["v"], ins["g"], ins["beta"], ins["s0"],
                               chunk=chunk)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        y = torch.full_like(y_ref, float("nan"))
        s = torch.full_like(s_ref, float("nan"))
        st = L.gdn_prefill_noalloc(_p(ins["q"]), _p(ins["k"]), _p(ins["v"]), _p(ins["g"]),
                                   _p(ins["beta"]), _p(ins["s0"]), _p(s), _p(y),
                                   B, T, Hk, Hv, 128, 128, chunk, gdn.GDN_DTYPE_BF16, stream)
        assert st == gdn.GDN_OK, gdn.gdn_status_string(st)
        torch.cuda.synchronize()
        yr, sr = y_ref.float().cpu().numpy(), s_ref.cpu().numpy()
        assert rel_err(y.float().cpu().numpy(), yr) <= TOL[torch.bfloat16], call
        assert rel_err(s.cpu().numpy(), sr) <= TOL[torch.bfloat16], call
    assert gdn.gdn_device_status() == gdn.GDN_OK


@pytest.mark.parametrize("B,T,Hk,Hv,chunk,dtype", [
    (1, 300, 2, 4, 32, torch.bfloat16),     # fused tensor-core launch (cooperative)
    (2, 100, 16, 32, 64, torch.bfloat16),   # 64 heads: the split prep + scan launches
    (1, 70, 2, 4, 32, torch.float32),       # fp32 chunked path
    (4, 16, 16, 32, 64, torch.bfloat16),    # short-T tensor-core kernel
])
def test_noalloc_prefill_under_graph_capture(cuda_device, B, T, Hk, Hv, chunk, dtype):
    """The entry point's purpose is use where nothing may allocate, graph
    capture included: one warm-up call, then the call captured into a CUDA
    graph, replayed twice, each replay against the workspace prefill."""
    L = gdn.lib()
    dt = {torch.bfloat16: gdn.GDN_DTYPE_BF16, torch.float32: gdn.GDN_DTYPE_F32}[dtype]
    need = gdn.gdn_prefill_workspace_bytes(B, T, Hk, Hv, 128, 128, chunk, dt)
    assert need <= gdn.GDN_NOALLOC_SCRATCH_BYTES
    ins = to_device(gdn_inputs.make_inputs(B, T, Hk, Hv, 128, 128, dtype, seed=43 + T,
                                           u_max=0.3, s0_std=0.1), cuda_device)
    y_ref, s_ref = gdn.prefill(ins["q"], ins["k"], ins["v"], ins["g"], ins["beta"], ins["s0"],
                               chunk=chunk)
    torch.cuda.synchronize()
    y = torch.empty_like(y_ref)
    s = torch.empty_like(s_ref)

    def call():
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        return L.gdn_prefill_noalloc(_p(ins["q"]), _p(ins["k"]), _p(ins["v"]), _p(ins["g"]),
                                     _p(ins["beta"]), _p(ins["s0"]), _p(s), _p(y),
                                     B, T, Hk, Hv, 128, 128, chunk, dt, stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert call() == gdn.GDN_OK      # warm-up: attributes and lookups set outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        st = call()
    assert st == gdn.GDN_OK, gdn.gdn_status_string(st)
    yr, sr = y_ref.float().cpu().numpy(), s_ref.cpu().numpy()
    for replay in range(2):
        y.fill_(float("nan"))
        s.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert rel_err(y.float().cpu().numpy(), yr) <= TOL[dtype], replay
        assert rel_err(s.cpu().numpy(), sr) <= TOL[dtype], replay
    assert gdn.gdn_device_status() == gdn.GDN_OK


def test_noalloc_rejects_problems_beyond_its_buffer(cuda_device):
    L = gdn.lib()
    need = gdn.gdn_prefill_workspace_bytes(1, 65536, 16, 32, 128, 128, 64, gdn.GDN_DTYPE_BF16)
    assert need > gdn.GDN_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)   # rejected on the host before any use
    st = L.gdn_prefill_noalloc(fake, fake, fake, fake, fake, fake, fake, fake,
                               1, 65536, 16, 32, 128, 128, 64, gdn.GDN_DTYPE_BF16, None)
    assert st == gdn.GDN_ERR_NOALLOC_LIMIT
    assert "GDN_NOALLOC_SCRATCH_BYTES" in gdn.gdn_status_string(st)
