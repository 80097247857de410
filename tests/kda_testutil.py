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


def oracle_grouped(inp, form="recurrent", **kw):
    """The oracle over an input dict with grouped heads (every output head); returns
    (out [T, Ho, 128], final [N, H, 128, 128])."""
    import oracle
    f = lambda n: to_f64_numpy(inp[n])  # noqa: E731
    cu = inp["cu_seqlens"].cpu().numpy().astype(np.int64)
    return oracle.grouped(f("q"), f("k"), f("v"), f("g"), f("beta"), inp["scale"],
                          s0=to_f64_numpy(inp["initial_state"]), cu_seqlens=cu, form=form, **kw)


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


def oracle_grouped_on_heads(orc, inp, out_heads, form="recurrent", **kw):
    """The oracle on selected OUTPUT heads of a grouped input dict: each output head runs as
    a plain head on the q, k and state heads it reads.  Returns (out [T, len, 128],
    final [N, len, 128, 128]) where the final state is that of the head's state head."""
    import oracle
    w = inp["workload"]
    maps = [oracle.grouped_heads(ho, w.num_heads, w.q_heads) for ho in out_heads]
    sel = lambda n, idx: to_f64_numpy(inp[n][:, idx])  # noqa: E731
    iq, ik, isx = ([m[i] for m in maps] for i in range(3))
    s0 = inp["initial_state"]
    cu = inp["cu_seqlens"].cpu().numpy().astype(np.int64)
    return getattr(orc, form)(sel("q", iq), sel("k", ik), sel("v", isx), sel("g", isx),
                              sel("beta", isx), inp["scale"],
                              s0=None if s0 is None else to_f64_numpy(s0[:, isx]),
                              cu_seqlens=cu, **kw)
