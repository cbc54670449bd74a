"""Test infrastructure only: the fp64 CPU oracle for the KDA forward pass.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The CUDA
library never does, and the two share no code.

* :func:`fwd`   -- the per-token recurrence from the library's own inputs
  (``kda_oracle.c``), the definition the GPU path is checked against.
* :func:`core`  -- the same recurrence from activated alpha/beta (any K, V).
* :func:`gate`  -- the natural-log gate alone.
* :mod:`oracle.chunk_ref` -- an independent chunked (WY) evaluation in numpy,
  used only to pin the per-token oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_SO = os.path.join(_HERE, "libkda_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``libkda_oracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.kda_oracle_fwd.argtypes = [P, P, P, P, P, D, P, P, P, D, P, P, P, I, I, I, I, I, I, I, I]
        lib.kda_oracle_fwd.restype = I
        lib.kda_oracle_core.argtypes = [P, P, P, P, P, D, P, P, P, P, I, I, I, I, I, I, I]
        lib.kda_oracle_core.restype = I
        lib.kda_oracle_gate.argtypes = [P, P, P, D, P, ctypes.c_int64, I, I]
        lib.kda_oracle_gate.restype = I
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def fwd(q, k, v, g, beta, scale, A_log=None, dt_bias=None, lower_bound=-5.0,
        initial_state=None, cu_seqlens=None, nthreads=None, qk_l2norm=False):
    """Per-token fp64 forward.

    ``q, k, v, g``: uint16 bf16 bit patterns ``[B, T, H, K|V]``; ``beta``: uint16
    ``[B, T, H]`` logits; ``A_log`` float32 ``[H]``; ``dt_bias`` float32 ``[H, K]``;
    ``initial_state`` float64 ``[B|N, H, V, K]``; ``cu_seqlens`` int64 ``[N+1]``.
    ``qk_l2norm``: L2-normalise q and k per (token, head), ``x / sqrt(sum x^2 + 1e-6)``.
    Returns ``(out float64 [B,T,H,V], final_state float64 [B|N,H,V,K])``.
    """
    q, k, v, g, beta = (_c(x, np.uint16) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    cu = _c(cu_seqlens, np.int64)
    N = int(cu.shape[0] - 1) if cu is not None else 0
    nseq = N if cu is not None else B
    out = np.zeros((B, T, H, V), np.float64)
    fin = np.zeros((nseq, H, V, K), np.float64)
    init = _c(initial_state, np.float64)
    rc = _load().kda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
                                _ptr(_c(A_log, np.float32)), _ptr(_c(dt_bias, np.float32)),
                                float(lower_bound), _ptr(init), _ptr(fin), _ptr(cu),
                                B, T, H, K, V, N, int(bool(qk_l2norm)), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, fin


def core(q, k, v, alpha, beta, scale, initial_state=None, cu_seqlens=None, nthreads=1):
    """Per-token fp64 recurrence from activated ``alpha`` ``[B,T,H,K]`` and
    ``beta`` ``[B,T,H]`` (all float64). Returns ``(out, final_state)``."""
    q, k, v, alpha, beta = (_c(x, np.float64) for x in (q, k, v, alpha, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    cu = _c(cu_seqlens, np.int64)
    N = int(cu.shape[0] - 1) if cu is not None else 0
    nseq = N if cu is not None else B
    out = np.zeros((B, T, H, V), np.float64)
    fin = np.zeros((nseq, H, V, K), np.float64)
    init = _c(initial_state, np.float64)
    rc = _load().kda_oracle_core(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), float(scale),
                                 _ptr(out), _ptr(init), _ptr(fin), _ptr(cu), B, T, H, K, V, N,
                                 int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, fin


def gate(g, A_log=None, dt_bias=None, lower_bound=-5.0):
    """Natural-log gate ``lower_bound * sigmoid(exp(A_log) (g + dt_bias))``, fp64.
    ``g``: uint16 bf16 bits ``[..., H, K]``."""
    g = _c(g, np.uint16)
    H, K = g.shape[-2], g.shape[-1]
    n_tok = int(g.size // (H * K))
    out = np.zeros(g.shape, np.float64)
    rc = _load().kda_oracle_gate(_ptr(g), _ptr(_c(A_log, np.float32)), _ptr(_c(dt_bias, np.float32)),
                                 float(lower_bound), _ptr(out), n_tok, H, K)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def bf16_bits_to_f64(bits):
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
