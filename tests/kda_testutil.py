"""Helpers shared by the tests: oracle runs on (sampled) heads and the tolerance check.

Tolerance (the pages' bar for bf16 output and fp32 final state against a
reference, flashinfer PR #4351 "Correctness": atol = rtol = 1e-2):
    |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|   elementwise.
"""
import numpy as np
import torch

from chunked_kda_delta_gb300.inputs import to_f64_numpy

ATOL = 1e-2
RTOL = 1e-2


def oracle_on_heads(orc, inp, heads, form="recurrent", **kw):
    """Run the oracle on the given head indices of an input dict; returns (out, final)."""
    hs = list(heads)
    sel = lambda t: None if t is None else t[:, hs] if t.dim() >= 2 else t  # noqa: E731
    q = to_f64_numpy(sel(inp["q"]))
    k = to_f64_numpy(sel(inp["k"]))
    v = to_f64_numpy(sel(inp["v"]))
    g = to_f64_numpy(sel(inp["g"]))
    beta = to_f64_numpy(sel(inp["beta"]))
    s0 = inp["initial_state"]
    s0 = None if s0 is None else to_f64_numpy(s0[:, hs])
    cu = inp["cu_seqlens"].cpu().numpy().astype(np.int64)
    fn = getattr(orc, form)
    return fn(q, k, v, g, beta, inp["scale"], s0=s0, cu_seqlens=cu, **kw)


def excess(got, ref):
    """max over elements of |got - ref| - (atol + rtol |ref|); <= 0 means within tolerance."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref) - (ATOL + RTOL * np.abs(ref)))) if got.size else -1.0


def max_abs(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def assert_close(got, ref, what=""):
    e = excess(got, ref)
    assert e <= 0.0, (f"{what}: exceeds atol=rtol=1e-2 by {e:.3e} "
                      f"(max abs diff {max_abs(got, ref):.3e})")


def gpu_out_heads(out: torch.Tensor, heads):
    return to_f64_numpy(out.reshape(-1, out.shape[-2], out.shape[-1])[:, list(heads)])


def gpu_state_heads(st: torch.Tensor, heads):
    return to_f64_numpy(st[:, list(heads)])
