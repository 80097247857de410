"""Thin Python binding of the KDA C ABI (``include/kda.h``) through ctypes.

Argument marshalling only: tensors are checked for dtype, layout and device,
their pointers and sizes are passed to ``libkda.so`` and every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the
compiled library is missing or the call fails, :class:`KdaError` is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import numpy as np
import torch

from . import build as _build

MODE_SERIAL = 0
MODE_SEGMENT = 1
MODE_AUTO = 2

_STATUS = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARGUMENT", 2: "KDA_ERR_ALIASING",
    3: "KDA_ERR_UNSUPPORTED_DEVICE", 4: "KDA_ERR_OUT_OF_MEMORY", 5: "KDA_ERR_CUDA",
    6: "KDA_ERR_CAPTURE_NEEDS_WARMUP", 7: "KDA_ERR_DEVICE_TIMEOUT",
}

EXPORTED_SYMBOLS = (
    "kda_prefill", "kda_prefill_ex", "kda_prefill_host", "kda_workspace_bytes",
    "kda_get_device_status", "kda_release_workspaces", "kda_status_string",
    "kda_last_error_message", "kda_version", "kda_prefill_segment_noalloc", "kda_plan",
    "kda_plan_varlen", "kda_decode",
)

STATE_F32 = 0
STATE_BF16 = 1
_STATE_DTYPES = {torch.float32: STATE_F32, torch.bfloat16: STATE_BF16}


class KdaError(RuntimeError):
    """A non-OK status from the library (``status`` holds the code)."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class KdaShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seq_len", ctypes.c_int64),
                ("num_seqs", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("num_q_heads", ctypes.c_int32)]


class KdaOptions(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("segment_len", ctypes.c_int32),
                ("wait_limit", ctypes.c_int64), ("debug_flags", ctypes.c_int32),
                ("host_pieces", ctypes.c_int32), ("state_dtype", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None, build_if_missing: bool = False) -> ctypes.CDLL:
    """Load ``libkda.so`` (built by :mod:`chunked_kda_delta_gb300.build`)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            if build_if_missing:
                p = _build.build()
            else:
                raise KdaError(5, f"CUDA library {p} is missing; build it with "
                                  "`python -m chunked_kda_delta_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, u16p, f32p, i32p = (ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p)
        args = [ctypes.POINTER(KdaShape), u16p, u16p, u16p, f32p, u16p, ctypes.c_float,
                f32p, i32p, u16p, f32p, vp]
        lib.kda_prefill.argtypes = args
        lib.kda_prefill_ex.argtypes = args + [ctypes.POINTER(KdaOptions)]
        lib.kda_prefill_host.argtypes = args + [ctypes.POINTER(KdaOptions)]
        lib.kda_prefill_segment_noalloc.argtypes = [
            ctypes.POINTER(KdaShape), u16p, u16p, u16p, f32p, u16p, ctypes.c_float, f32p, u16p,
            f32p, ctypes.c_int32, vp]
        lib.kda_workspace_bytes.argtypes = [ctypes.POINTER(KdaShape), ctypes.POINTER(KdaOptions),
                                            ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_plan_varlen.argtypes = [ctypes.POINTER(KdaShape), vp, ctypes.c_int32,
                                        ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
        lib.kda_plan.argtypes = [ctypes.POINTER(KdaShape), ctypes.c_int32, ctypes.c_int32,
                                 ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
        lib.kda_decode.argtypes = [ctypes.POINTER(KdaShape), u16p, u16p, u16p, f32p, u16p,
                                   ctypes.c_float, vp, vp, ctypes.c_int32, u16p, vp]
        lib.kda_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        lib.kda_release_workspaces.argtypes = [ctypes.c_int32]
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_last_error_message.restype = ctypes.c_char_p
        lib.kda_version.restype = ctypes.c_char_p
        for f in (lib.kda_prefill, lib.kda_prefill_ex, lib.kda_prefill_host,
                  lib.kda_prefill_segment_noalloc, lib.kda_decode,
                  lib.kda_workspace_bytes, lib.kda_get_device_status, lib.kda_plan,
                  lib.kda_release_workspaces):
            f.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(lib, status: int):
    if status != 0:
        raise KdaError(status, lib.kda_last_error_message().decode())


def kda_status_string(status: int) -> str:
    return load_library().kda_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _shape_of(q: torch.Tensor, v: torch.Tensor, cu_seqlens) -> KdaShape:
    """Shape of a call: batch and tokens from q, state heads from v, query heads from q."""
    if q.dim() == 4:
        B, T, Hq, D = q.shape
    elif q.dim() == 3:
        B, (T, Hq, D) = 1, q.shape
    else:
        raise ValueError("q must be [T, H, 128] or [B, T, H, 128]")
    H = v.shape[-2]
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("packed varlen input needs batch 1")
        return KdaShape(1, T, cu_seqlens.numel() - 1, H, D, Hq)
    return KdaShape(B, T, 0, H, D, Hq)


def _out_shape(q: torch.Tensor, v: torch.Tensor):
    """q's shape with max(query heads, state heads) heads."""
    return tuple(q.shape[:-2]) + (max(q.shape[-2], v.shape[-2]), q.shape[-1])


def _check_tensors(q, k, v, g, beta, initial_state, cu_seqlens, device_type,
                   state_dtypes=(torch.float32,)):
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.bfloat16)):
        if t.dtype != dt:
            raise ValueError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device.type != device_type:
            raise ValueError(f"{name} must be on {device_type}")
    if v.shape != g.shape:
        raise ValueError("v and g must share one shape")
    if q.dim() != v.dim() or q.shape[:-2] != v.shape[:-2] or q.shape[-1] != v.shape[-1]:
        raise ValueError("q and v must agree in every dim but heads")
    Hq, H = q.shape[-2], v.shape[-2]
    if Hq < 1 or H < 1 or (Hq % H and H % Hq):
        raise ValueError(f"query heads ({Hq}) and state heads ({H}) must divide one another")
    if k.shape != q.shape[:-2] + (min(Hq, H), q.shape[-1]):
        raise ValueError("k must have min(query heads, state heads) heads")
    if beta.shape != v.shape[:-1]:
        raise ValueError("beta must have v's shape without the last dim")
    if initial_state is not None:
        if initial_state.dtype not in state_dtypes or not initial_state.is_contiguous():
            raise ValueError("initial_state must be contiguous, one of " +
                             ", ".join(str(d) for d in state_dtypes))
        if initial_state.device.type != device_type:
            raise ValueError(f"initial_state must be on {device_type}")
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be contiguous int32")
        if cu_seqlens.device.type != device_type:
            raise ValueError(f"cu_seqlens must be on {device_type}")


def _check_result(name, t, shape, dtype, device_type):
    """A caller-supplied output must be exactly what the library writes: the C ABI takes
    bare pointers and cannot see a short buffer."""
    if t is None:
        return
    if t.dtype != dtype or not t.is_contiguous() or t.device.type != device_type:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor on {device_type}")
    if tuple(t.shape) != tuple(shape) and t.numel() != math.prod(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


DEBUG_STALL_WAIT = 1


def _options(mode, segment_len, wait_limit, debug_flags=0, host_pieces=0,
             state_dtype=torch.float32):
    return KdaOptions(int(mode), int(segment_len), int(wait_limit), int(debug_flags),
                      int(host_pieces), 1 if state_dtype == torch.bfloat16 else 0)


def _state_dtype(state_dtype, *given):
    """The prefill's state type: as asked, else that of the state tensors given, else fp32;
    every given state must have it."""
    ts = [t for t in given if t is not None]
    if state_dtype is None:
        state_dtype = ts[0].dtype if ts else torch.float32
    if state_dtype not in _STATE_DTYPES:
        raise ValueError("state_dtype must be torch.float32 or torch.bfloat16")
    for t in ts:
        if t.dtype != state_dtype:
            raise ValueError(f"states must all be {state_dtype}, got {t.dtype}")
    return state_dtype


def kda_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                beta: torch.Tensor, scale: Optional[float] = None,
                initial_state: Optional[torch.Tensor] = None,
                cu_seqlens: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None,
                final_state: Optional[torch.Tensor] = None,
                stream=None, output_final_state: bool = False,
                mode: int = MODE_SERIAL, segment_len: int = 0, wait_limit: int = 0,
                debug_flags: int = 0, state_dtype: Optional[torch.dtype] = None):
    """KDA forward prefill on CUDA tensors; returns ``(out, final_state)``.

    q, k, v: bf16 ``[T, H, 128]`` (or ``[B, T, H, 128]`` dense); g: fp32 of the
    same shape; beta: bf16 ``[T, H]``; initial_state / final_state: ``[N, H, 128, 128]``
    in fp32 or bf16 (``state_dtype``, else the type of the states given, else fp32; the
    arithmetic is fp32 either way); cu_seqlens: int32 ``[N + 1]`` on the device.  Grouped heads:
    q may have Hq heads, Hq a multiple or a divisor of v's H (k then has min(Hq, H)
    heads, the output max(Hq, H)).  ``out``
    is allocated when not given; ``final_state`` is allocated when
    ``output_final_state`` is set and none is given (pass ``final_state =
    initial_state`` to update in place).  The call is asynchronous on
    ``stream`` (a ``torch.cuda.Stream``, a raw handle, or the current stream).
    """
    lib = load_library()
    sdt = _state_dtype(state_dtype, initial_state, final_state)
    _check_tensors(q, k, v, g, beta, initial_state, cu_seqlens, "cuda", _STATE_DTYPES)
    shape = _shape_of(q, v, cu_seqlens)
    N = shape.num_seqs if cu_seqlens is not None else shape.batch
    if scale is None:
        scale = shape.head_dim ** -0.5
    _check_result("out", out, _out_shape(q, v), torch.bfloat16, "cuda")
    _check_result("final_state", final_state, (N, shape.num_heads, 128, 128), sdt, "cuda")
    if out is None:
        out = torch.empty(_out_shape(q, v), dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, shape.num_heads, shape.head_dim, shape.head_dim),
                                  dtype=sdt, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    opts = _options(mode, segment_len, wait_limit, debug_flags, state_dtype=sdt)
    with torch.cuda.device(q.device):
        st = lib.kda_prefill_ex(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(beta), ctypes.c_float(scale), _ptr(initial_state),
                                _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                ctypes.c_void_p(int(stream)), ctypes.byref(opts))
    _check(lib, st)
    return out, final_state


def kda_prefill_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                     beta: torch.Tensor, scale: Optional[float] = None,
                     initial_state: Optional[torch.Tensor] = None,
                     cu_seqlens: Optional[torch.Tensor] = None,
                     out: Optional[torch.Tensor] = None,
                     final_state: Optional[torch.Tensor] = None,
                     stream=None, output_final_state: bool = False, device=None,
                     mode: int = MODE_SERIAL, segment_len: int = 0, wait_limit: int = 0,
                     host_pieces: int = 0, state_dtype: Optional[torch.dtype] = None):
    """End-to-end prefill on HOST (CPU) tensors: copy in, compute, copy out, synchronise.

    Same arguments as :func:`kda_prefill` but every tensor lives in host memory
    (pinned memory gives full copy bandwidth); ``device`` picks the GPU.  Large serial
    calls stream in ``host_pieces`` pieces (0: the library's choice) so that copies
    and kernels overlap.
    """
    lib = load_library()
    sdt = _state_dtype(state_dtype, initial_state, final_state)
    _check_tensors(q, k, v, g, beta, initial_state, cu_seqlens, "cpu", _STATE_DTYPES)
    shape = _shape_of(q, v, cu_seqlens)
    N = shape.num_seqs if cu_seqlens is not None else shape.batch
    if scale is None:
        scale = shape.head_dim ** -0.5
    _check_result("out", out, _out_shape(q, v), torch.bfloat16, "cpu")
    _check_result("final_state", final_state, (N, shape.num_heads, 128, 128), sdt, "cpu")
    if out is None:
        out = torch.empty(_out_shape(q, v), dtype=q.dtype, pin_memory=q.is_pinned())
    if final_state is None and output_final_state:
        final_state = torch.empty((N, shape.num_heads, shape.head_dim, shape.head_dim),
                                  dtype=sdt, pin_memory=q.is_pinned())
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    opts = _options(mode, segment_len, wait_limit, host_pieces=host_pieces, state_dtype=sdt)
    with torch.cuda.device(dev):
        st = lib.kda_prefill_host(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                  _ptr(beta), ctypes.c_float(scale), _ptr(initial_state),
                                  _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                  ctypes.c_void_p(int(stream)), ctypes.byref(opts))
    _check(lib, st)
    return out, final_state


def kda_workspace_bytes(batch: int, seq_len: int, num_heads: int, mode: int = MODE_SERIAL,
                        segment_len: int = 0, head_dim: int = 128, num_seqs: int = 0,
                        num_q_heads: int = 0) -> int:
    """Device workspace bytes for a problem of this shape in this mode (packed varlen
    when ``num_seqs`` > 0: ``batch`` 1, ``seq_len`` the total tokens)."""
    lib = load_library()
    shape = KdaShape(batch, seq_len, num_seqs, num_heads, head_dim, num_q_heads)
    opts = _options(mode, segment_len, 0)
    n = ctypes.c_size_t(0)
    _check(lib, lib.kda_workspace_bytes(ctypes.byref(shape), ctypes.byref(opts),
                                        ctypes.byref(n)))
    return int(n.value)


def kda_plan(batch: int, seq_len: int, num_heads: int, resident_clusters: int,
             varlen: bool = False, num_seqs: int = 0, head_dim: int = 128, num_q_heads: int = 0):
    """The (mode, segment_len) that ``MODE_AUTO`` picks for this shape on a device holding
    ``resident_clusters`` co-resident clusters.  Host only."""
    lib = load_library()
    shape = KdaShape(batch, seq_len, num_seqs, num_heads, head_dim, num_q_heads)
    mode, seg = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib, lib.kda_plan(ctypes.byref(shape), int(bool(varlen)), int(resident_clusters),
                             ctypes.byref(mode), ctypes.byref(seg)))
    return int(mode.value), int(seg.value)


def kda_plan_varlen(seq_lens, num_heads: int, resident_clusters: int, head_dim: int = 128,
                    num_q_heads: int = 0):
    """The (mode, segment_len) that ``MODE_AUTO`` of :func:`kda_prefill_host` picks for a
    packed batch with these sequence lengths.  Host only."""
    lib = load_library()
    lens = [int(x) for x in seq_lens]
    cu = (ctypes.c_int32 * (len(lens) + 1))(*([0] + list(np.cumsum(lens, dtype=np.int64))))
    shape = KdaShape(1, int(sum(lens)), len(lens), num_heads, head_dim, num_q_heads)
    mode, seg = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib, lib.kda_plan_varlen(ctypes.byref(shape), ctypes.cast(cu, ctypes.c_void_p),
                                    int(resident_clusters), ctypes.byref(mode), ctypes.byref(seg)))
    return int(mode.value), int(seg.value)


def kda_get_device_status(stream=None, device=None) -> int:
    """Synchronise ``stream`` and read-and-clear the device status word (0 = OK)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    code = ctypes.c_int32(0)
    with torch.cuda.device(dev):
        _check(lib, lib.kda_get_device_status(ctypes.c_void_p(int(stream)), ctypes.byref(code)))
    return int(code.value)


def kda_release_workspaces(device: int = -1) -> None:
    """Free the library's workspaces on ``device`` (-1: all devices)."""
    lib = load_library()
    _check(lib, lib.kda_release_workspaces(int(device)))


def kda_prefill_segment_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                                g: torch.Tensor, beta: torch.Tensor, out: torch.Tensor,
                                segment_len: int, scale: Optional[float] = None,
                                initial_state: Optional[torch.Tensor] = None,
                                final_state: Optional[torch.Tensor] = None, stream=None):
    """Segment-parallel prefill with no device allocation (dense input only; grouped heads
    allowed).

    For callers that cannot allocate device memory: the library keeps the segment
    scratch in a fixed 32 MiB device array shared by all calls, so ``out`` (and
    ``final_state`` when wanted) must be passed in.  Shapes needing more than
    B * H * (3 * nseg - 2) = 512 state slots are rejected; calls overlapping on the
    GPU race on the shared array.
    """
    lib = load_library()
    _check_tensors(q, k, v, g, beta, initial_state, None, "cuda")
    shape = _shape_of(q, v, None)
    _check_result("out", out, _out_shape(q, v), torch.bfloat16, "cuda")
    _check_result("final_state", final_state, (shape.batch, shape.num_heads, 128, 128),
                  torch.float32, "cuda")
    if scale is None:
        scale = shape.head_dim ** -0.5
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    with torch.cuda.device(q.device):
        st = lib.kda_prefill_segment_noalloc(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
            ctypes.c_float(scale), _ptr(initial_state), _ptr(out), _ptr(final_state),
            int(segment_len), ctypes.c_void_p(int(stream)))
    _check(lib, st)
    return out, final_state


def kda_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
               beta: torch.Tensor, scale: Optional[float] = None,
               initial_state: Optional[torch.Tensor] = None,
               final_state: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, output_final_state: bool = True,
               state_dtype: Optional[torch.dtype] = None, stream=None):
    """The recurrent decode step on CUDA tensors; returns ``(out, final_state)``.

    q, k, v: bf16 ``[B, H, 128]`` (one token per sequence) or ``[B, T, H, 128]``;
    g: fp32 of v's shape; beta: bf16 ``[B, H]`` or ``[B, T, H]``; grouped heads as in
    :func:`kda_prefill`.  States are
    ``[B, H, 128, 128]`` in fp32 or bf16 (``state_dtype``, else the dtype of the
    state tensors given, else fp32).  Pass ``final_state = initial_state`` to update a
    state cache in place; a new final state is allocated when ``output_final_state``
    is set and none is given.
    """
    lib = load_library()
    single = q.dim() == 3
    if single:
        q, k, v, g = (x.unsqueeze(1) for x in (q, k, v, g))
        beta = beta.unsqueeze(1)
    _check_tensors(q, k, v, g, beta, None, None, "cuda")
    if q.dim() != 4:
        raise ValueError("q must be [B, H, 128] or [B, T, H, 128]")
    B, T, Hq, D = q.shape
    H = v.shape[2]
    given = [t for t in (initial_state, final_state) if t is not None]
    if state_dtype is None:
        state_dtype = given[0].dtype if given else torch.float32
    if state_dtype not in _STATE_DTYPES:
        raise ValueError("state_dtype must be torch.float32 or torch.bfloat16")
    for t in given:
        if t.dtype != state_dtype or not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError(f"states must be contiguous {state_dtype} CUDA tensors")
        if tuple(t.shape) != (B, H, D, D):
            raise ValueError(f"states must be [{B}, {H}, {D}, {D}]")
    if scale is None:
        scale = D ** -0.5
    _check_result("out", out, _out_shape(q, v), torch.bfloat16, "cuda")
    if out is None:
        out = torch.empty(_out_shape(q, v), dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, D, D), dtype=state_dtype, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    shape = KdaShape(B, T, 0, H, D, Hq)
    with torch.cuda.device(q.device):
        st = lib.kda_decode(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                            ctypes.c_float(scale), _ptr(initial_state), _ptr(final_state),
                            _STATE_DTYPES[state_dtype], _ptr(out), ctypes.c_void_p(int(stream)))
    _check(lib, st)
    return (out.squeeze(1) if single else out), final_state
