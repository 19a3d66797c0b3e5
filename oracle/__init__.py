"""fp64 CPU oracle for the gated delta rule.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this
package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
cpu_baseline / ``--impl reference`` leg do.  It shares no code, header,
table or constant with the CUDA library in ``gated_delta_rule_02_gb300``.

Contents
--------
``gdn_sequential``   the definition: the sequential recurrence in plain C,
                     fp64 (``gdn_seq.c``), parallel over (batch, value head).
``forms``            independent fp64 NumPy restatements used to pin the
                     oracle: the chunked Woodbury-Young form, the
                     single-solve chunk form and the explicit product form.

Every function takes arrays in the library's layouts:
``q, k [B,T,Hk,Dk]``, ``v [B,T,Hv,Dv]``, ``g, beta [B,T,Hv]``,
``s0 [B,Hv,Dv,Dk]`` (or None for a zero state) and returns
``(y [B,T,Hv,Dv], s_final [B,Hv,Dv,Dk])`` in float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_seq.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gdn_seq.c`` into ``_build/liboracle.so`` with gcc + OpenMP.

    Plain ``-O2`` (no ``-ffast-math``, no ``-march=native``): the oracle must
    keep IEEE fp64 semantics and build the same on x86_64 and aarch64.
    """
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_OUT_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.gdn_seq_f64.argtypes = [ctypes.c_int] * 6 + [dp] * 8
            lib.gdn_seq_f64.restype = None
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Widen to a contiguous float64 array (exact for bf16/fp32 inputs)."""
    if hasattr(x, "detach"):  # torch tensor: widen on the CPU
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def gdn_sequential(q, k, v, g, beta, s0=None):
    """The gated delta rule, token by token, in fp64 (the definition).

    Follows ferrox-core ``gdn_chunk.rs`` ("The algebra") with the decay as
    a multiplicative gate g (metaltile-std ``gated_delta_wy.rs``, Algorithm
    step 2) and the output scale 1/sqrt(Dk).  Returns ``(y, s_final)``.
    """
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    assert k.shape == q.shape and v.shape[:2] == (B, T)
    assert g.shape == (B, T, Hv) and beta.shape == (B, T, Hv)
    assert Hv % Hk == 0
    s = np.empty((B, Hv, Dv, Dk), dtype=np.float64)
    y = np.empty((B, T, Hv, Dv), dtype=np.float64)
    if s0 is not None:
        s0 = _f64(s0)
        assert s0.shape == (B, Hv, Dv, Dk)
    lib = _load()
    lib.gdn_seq_f64(B, T, Hk, Hv, Dk, Dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                    _ptr(beta), _ptr(s0) if s0 is not None else None,
                    _ptr(s), _ptr(y))
    return y, s


def gdn_decode_steps(q, k, v, g, beta, s0):
    """``n`` single decode steps, each the T=1 recurrence with S carried.

    Inputs carry a leading step axis: ``q [n,B,1,Hk,Dk]`` and so on;
    returns ``(y [n,B,1,Hv,Dv], s_final)``.
    """
    s = _f64(s0)
    ys = []
    for i in range(len(q)):
        y, s = gdn_sequential(q[i], k[i], v[i], g[i], beta[i], s)
        ys.append(y)
    return np.stack(ys), s


def num_threads() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS or all cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    return os.cpu_count() or 1
