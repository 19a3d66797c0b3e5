"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

The library is built (nvcc cross-compiles for sm_103a without a GPU) and
loaded; every function include/gdn.h declares must be exported, and every
argument check must answer before any CUDA call is made.  The pointers
used here are never dereferenced: every call below is rejected on the host.
"""
import ctypes
import glob
import os
import re

import pytest

import gated_delta_rule_02_gb300 as gdn
from gated_delta_rule_02_gb300 import build as gdn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gdn_build.build()
    return gdn.lib()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("gdn_prefill", "gdn_decode_step", "gdn_status_string",
                     "gdn_prefill_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), f"{name} is declared in include/ but not exported"


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5):
        s = gdn.gdn_status_string(code)
        assert s and s != "unknown status"
    assert gdn.gdn_status_string(-99) == "unknown status"


def test_workspace_bytes(L):
    w = gdn.gdn_prefill_workspace_bytes
    assert w(1, 4096, 16, 32, 128, 128, 64, 1) > 0
    assert w(1, 4096, 16, 32, 128, 128, 64, 1) % 256 == 0
    assert w(1, 4096, 16, 32, 128, 128, 48, 1) == 0      # bad chunk
    assert w(1, 4096, 16, 32, 96, 128, 64, 1) == 0       # unsupported head size
    assert w(1, 4096, 16, 32, 128, 512, 64, 1) == 0
    # 16-bit inputs at Dk = Dv = 64 or 256 run the warp-level MMA paths, always
    # in chunks of 32: a block of 5 x 32 rows (-Pt, Qh, Ut, K, y_loc) per
    # (head, chunk), plus G_C or a flag per chunk
    nc = 4096 // 32
    assert w(1, 4096, 16, 32, 64, 64, 64, 1) == w(1, 4096, 16, 32, 64, 64, 16, 2)
    assert w(1, 4096, 16, 32, 64, 64, 64, 1) >= 32 * nc * 5 * 32 * 64 * 2
    assert w(1, 4096, 16, 32, 256, 256, 64, 1) == w(1, 4096, 16, 32, 256, 256, 32, 2)
    assert w(1, 4096, 16, 32, 256, 256, 64, 1) >= 32 * nc * 5 * 32 * 256 * 2
    # every other head pair, and fp32, runs the SIMT chunked path ...
    assert w(1, 4096, 16, 32, 64, 64, 64, 0) > 0
    assert w(1, 4096, 16, 32, 256, 64, 64, 1) > w(1, 4096, 16, 32, 64, 128, 64, 1) > 0
    # ... where Dk = Dv = 256 with chunk 64 runs as chunks of 32 (shared memory)
    assert w(1, 4096, 16, 32, 256, 256, 64, 0) == w(1, 4096, 16, 32, 256, 256, 32, 0)
    assert w(1, 4096, 16, 32, 128, 128, 64, 0) != w(1, 4096, 16, 32, 128, 128, 32, 0)
    assert w(1, 0, 16, 32, 128, 128, 64, 1) == 0         # empty
    assert w(1, 100, 3, 32, 128, 128, 64, 1) == 0        # Hv % Hk != 0
    # grows with the sequence
    assert w(1, 8192, 16, 32, 128, 128, 64, 1) > w(1, 4096, 16, 32, 128, 128, 64, 1)
    # short sequences run the sequential kernel, which needs no workspace
    assert w(4, 32, 16, 32, 128, 128, 64, 1) == 0
    assert w(4, 32, 16, 32, 128, 128, 64, 0) == 0
    assert w(4, 33, 16, 32, 128, 128, 64, 1) > 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call is rejected first


def prefill_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state_in=FAKE, state_out=FAKE,
             y=FAKE, B=1, T=64, Hk=1, Hv=2, Dk=128, Dv=128, chunk=32, dtype=1,
             workspace=FAKE, ws=1 << 40, stream=None)
    a.update(over)
    return [a[n] for n in ("q", "k", "v", "g", "beta", "state_in", "state_out", "y",
                           "B", "T", "Hk", "Hv", "Dk", "Dv", "chunk", "dtype",
                           "workspace", "ws", "stream")]


@pytest.mark.parametrize("over,expect", [
    (dict(q=None), gdn.GDN_ERR_INVALID),
    (dict(y=None), gdn.GDN_ERR_INVALID),
    (dict(state_out=None), gdn.GDN_ERR_INVALID),
    (dict(B=0), gdn.GDN_ERR_INVALID),
    (dict(T=0), gdn.GDN_ERR_INVALID),
    (dict(T=-5), gdn.GDN_ERR_INVALID),
    (dict(Hk=3, Hv=4), gdn.GDN_ERR_INVALID),
    (dict(Dk=96), gdn.GDN_ERR_UNSUPPORTED),
    (dict(Dv=512), gdn.GDN_ERR_UNSUPPORTED),
    (dict(Dk=32), gdn.GDN_ERR_UNSUPPORTED),
    (dict(chunk=48), gdn.GDN_ERR_UNSUPPORTED),
    (dict(chunk=128), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dtype=7), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dtype=3), gdn.GDN_ERR_UNSUPPORTED),
    (dict(k=FAKE + 4), gdn.GDN_ERR_ALIGNMENT),
    (dict(state_in=FAKE + 8), gdn.GDN_ERR_ALIGNMENT),
    (dict(workspace=None), gdn.GDN_ERR_WORKSPACE),
    (dict(ws=1024), gdn.GDN_ERR_WORKSPACE),
    (dict(workspace=FAKE + 16), gdn.GDN_ERR_ALIGNMENT),
])
def test_prefill_rejects_bad_arguments_on_host(L, over, expect):
    assert L.gdn_prefill(*prefill_args(**over)) == expect


@pytest.mark.parametrize("over,expect", [
    (dict(state_in=None), gdn.GDN_ERR_INVALID),
    (dict(v=None), gdn.GDN_ERR_INVALID),
    (dict(B=0), gdn.GDN_ERR_INVALID),
    (dict(Hk=2, Hv=3), gdn.GDN_ERR_INVALID),
    (dict(Dk=96), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dtype=3), gdn.GDN_ERR_UNSUPPORTED),
    (dict(y=FAKE + 2), gdn.GDN_ERR_ALIGNMENT),
])
def test_decode_rejects_bad_arguments_on_host(L, over, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state_in=FAKE, state_out=FAKE,
             y=FAKE, B=4, Hk=1, Hv=2, Dk=128, Dv=128, dtype=1, stream=None)
    a.update(over)
    args = [a[n] for n in ("q", "k", "v", "g", "beta", "state_in", "state_out", "y",
                           "B", "Hk", "Hv", "Dk", "Dv", "dtype", "stream")]
    assert L.gdn_decode_step(*args) == expect


def test_binding_fails_loudly_without_library(monkeypatch):
    """The binding has no fallback: a missing library is an error."""
    monkeypatch.setattr(gdn, "_lib", None)
    monkeypatch.setattr(gdn, "LIB_PATH", os.path.join(ROOT, "no", "such", "libgdn.so"))
    with pytest.raises(RuntimeError):
        gdn.lib()


@pytest.mark.parametrize("options", [8, 16, -1, 1 << 20])
def test_ex_entry_points_reject_unknown_options(L, options):
    assert L.gdn_prefill_ex(*prefill_args(), options) == gdn.GDN_ERR_UNSUPPORTED
    dec = [FAKE] * 8 + [1, 1, 2, 128, 128, 1, None]
    assert L.gdn_decode_step_ex(*dec, options) == gdn.GDN_ERR_UNSUPPORTED
