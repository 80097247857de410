"""fp64 CPU oracle for the KDA forward prefill -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is the independent checker of the
CUDA path: it shares no code with ``chunked_kda_delta_gb300`` and never reads
a value that the CUDA path produced.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, OpenMP over
(sequence, head) chains); this module compiles it with gcc and marshals numpy
arrays.  Three forms of the same definition are exposed:

* :func:`recurrent` -- the KDA recurrence token by token,
  ``S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T``,
  ``o_t = scale S_t^T q_t``.
* :func:`chunked` -- the chunkwise WY form, chunks of 16 tokens: decayed q/k,
  beta and the WY inverse per chunk (K1), then the state carried from chunk to
  chunk (K2).
* :func:`segmented` -- the segment pipeline: K1 once, per-segment summaries
  (pre_scan), a serial merge of the carries, then K2 per segment (cuLA PR #103,
  "feat(kda/sm90): FlashKDA prefill port + intracard-CP prefill", commit notes).
* :func:`grouped` -- any form over grouped (unequal) head counts, by running every
  output head as a plain head on the tensors it reads.

Every function takes float64 arrays: q, k, g ``[T, H, Dk]``; v ``[T, H, Dv]``;
beta ``[T, H]``; optional ``s0`` ``[N, H, Dk, Dv]``; ``cu_seqlens`` (N+1
offsets, or None for one sequence of length T) and returns ``(out, final)``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_PD = ctypes.POINTER(ctypes.c_double)
_PI64 = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library (gcc, -O2, OpenMP); returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_PD)


def _prep(q, k, v, g, beta, s0, cu_seqlens):
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    beta = np.ascontiguousarray(beta, dtype=np.float64)
    if q.ndim != 3 or k.shape != q.shape or g.shape != q.shape:
        raise ValueError("q, k, g must share shape [T, H, Dk]")
    T, H, Dk = q.shape
    if v.ndim != 3 or v.shape[:2] != (T, H):
        raise ValueError("v must be [T, H, Dv]")
    Dv = v.shape[2]
    if beta.shape != (T, H):
        raise ValueError("beta must be [T, H]")
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must be non-decreasing offsets from 0 to T")
    N = cu.size - 1
    if s0 is not None:
        s0 = np.ascontiguousarray(s0, dtype=np.float64)
        if s0.shape != (N, H, Dk, Dv):
            raise ValueError("initial state must be [N, H, Dk, Dv]")
    return q, k, v, g, beta, s0, cu, (T, H, Dk, Dv, N)


class OracleLib:
    """The oracle's three forms bound to one compiled copy of ``kda_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        common = [ctypes.c_int64, _PI64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  _PD, _PD, _PD, _PD, _PD, ctypes.c_double, _PD, _PD, _PD]
        lib.kda_oracle_recurrent.argtypes = common + [ctypes.c_int]
        lib.kda_oracle_chunked.argtypes = common + [ctypes.c_int64, ctypes.c_int]
        lib.kda_oracle_segmented.argtypes = common + [ctypes.c_int64, ctypes.c_int64,
                                                      ctypes.c_int]
        for f in (lib.kda_oracle_recurrent, lib.kda_oracle_chunked, lib.kda_oracle_segmented):
            f.restype = ctypes.c_int
        lib.kda_oracle_max_threads.restype = ctypes.c_int
        self._lib = lib
        self.path = path

    def max_threads(self) -> int:
        return int(self._lib.kda_oracle_max_threads())

    def _call(self, fn, extra, q, k, v, g, beta, scale, s0, cu_seqlens, n_threads):
        q, k, v, g, beta, s0, cu, (T, H, Dk, Dv, N) = _prep(q, k, v, g, beta, s0, cu_seqlens)
        out = np.zeros((T, H, Dv), dtype=np.float64)
        fin = np.zeros((N, H, Dk, Dv), dtype=np.float64)
        rc = fn(N, cu.ctypes.data_as(_PI64), H, Dk, Dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                _ptr(beta), float(scale), _ptr(s0), _ptr(out), _ptr(fin), *extra,
                int(n_threads))
        if rc != 0:
            raise RuntimeError(f"oracle call failed with code {rc}")
        return out, fin

    def recurrent(self, q, k, v, g, beta, scale, s0=None, cu_seqlens=None, n_threads=0):
        """Token-by-token fp64 recurrence; returns ``(out [T,H,Dv], final [N,H,Dk,Dv])``."""
        return self._call(self._lib.kda_oracle_recurrent, (), q, k, v, g, beta, scale, s0,
                          cu_seqlens, n_threads)

    def chunked(self, q, k, v, g, beta, scale, s0=None, cu_seqlens=None, chunk=16,
                n_threads=0):
        """Chunkwise WY form (``chunk`` rows per block); same result as the recurrence."""
        return self._call(self._lib.kda_oracle_chunked, (int(chunk),), q, k, v, g, beta,
                          scale, s0, cu_seqlens, n_threads)

    def segmented(self, q, k, v, g, beta, scale, s0=None, cu_seqlens=None, chunk=16,
                  seg_len=64, n_threads=0):
        """Segment pipeline (pre_scan -> merge -> per-segment pass); same result."""
        return self._call(self._lib.kda_oracle_segmented, (int(chunk), int(seg_len)), q, k, v,
                          g, beta, scale, s0, cu_seqlens, n_threads)


def default() -> OracleLib:
    """The oracle compiled from ``oracle/kda_oracle.c`` (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
    return _lib


def max_threads() -> int:
    """Number of OpenMP threads the oracle uses by default."""
    return default().max_threads()


def recurrent(*a, **kw):
    return default().recurrent(*a, **kw)


def chunked(*a, **kw):
    return default().chunked(*a, **kw)


def segmented(*a, **kw):
    return default().segmented(*a, **kw)


recurrent.__doc__ = OracleLib.recurrent.__doc__
chunked.__doc__ = OracleLib.chunked.__doc__
segmented.__doc__ = OracleLib.segmented.__doc__


def grouped_heads(ho: int, H: int, Hq: int):
    """(q head, k head, state head) read by output head ``ho`` when q has ``Hq`` heads and
    v, g, beta and the states have ``H`` (one a multiple of the other; k has min(Hq, H)
    heads, the output max(Hq, H)).  Unequal head counts are named as a follow-up in cuLA
    PR #103 (intracard-CP planner notes: GVA); the two directions are read as: more
    state heads than query heads shares each q/k head among H / Hq state heads; more query
    heads than state heads shares each k/v/g/beta head, and its state, among Hq / H query
    heads."""
    if Hq <= H:
        G = H // Hq
        return ho // G, ho // G, ho
    G = Hq // H
    return ho, ho // G, ho // G


def grouped(q, k, v, g, beta, scale, s0=None, cu_seqlens=None, form="recurrent", lib=None,
            **kw):
    """An oracle form over grouped heads: q ``[T, Hq, D]``, k ``[T, min(Hq, H), D]``, v and g
    ``[T, H, D]``, beta ``[T, H]``, s0 ``[N, H, D, D]``.  Every output head is run as an
    ungrouped head on the tensors it reads (:func:`grouped_heads`); returns
    ``(out [T, max(Hq, H), Dv], final [N, H, Dk, Dv])``, the final state of a state head
    taken from the first output head that reads it."""
    lib = lib or default()
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    Hq, H = q.shape[1], v.shape[1]
    if (Hq % H and H % Hq) or k.shape[1] != min(Hq, H) or g.shape != v.shape:
        raise ValueError("head counts must divide one another; k has min(Hq, H) heads")
    Ho = max(Hq, H)
    maps = [grouped_heads(ho, H, Hq) for ho in range(Ho)]
    iq = [m[0] for m in maps]
    ik = [m[1] for m in maps]
    isx = [m[2] for m in maps]
    s0e = None if s0 is None else np.asarray(s0, dtype=np.float64)[:, isx]
    out, fin = getattr(lib, form)(q[:, iq], k[:, ik], v[:, isx], g[:, isx], beta[:, isx], scale,
                                  s0=s0e, cu_seqlens=cu_seqlens, **kw)
    first = [isx.index(hs) for hs in range(H)]
    return out, fin[:, first]
