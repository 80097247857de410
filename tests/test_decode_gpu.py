"""GPU parity of the recurrent decode step (kda_decode) against the fp64 oracle.

The decode step is the recurrence itself applied to a few tokens of each sequence, so
the oracle's token-by-token form over sequences of those lengths is its definition.
Bar: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| on the bf16 output and on the state
(flashinfer PR #4351 "Correctness").  With bf16 state storage the oracle starts from
the exact upcast of the bf16 initial state, and the stored final state is compared
after its own bf16 rounding (relative 2^-9, inside the bar).
"""
import numpy as np
import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.inputs import WORKLOADS, custom, make_inputs, to_f64_numpy

from kda_testutil import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    K.load_library()


def dense_view(inp, B, T):
    """Inputs of B dense sequences of T tokens as [B, T, H, 128] (beta [B, T, H])."""
    H = inp["workload"].num_heads
    q, k, v, g = (inp[x].view(B, T, H, 128) for x in ("q", "k", "v", "g"))
    return q, k, v, g, inp["beta"].view(B, T, H)


def oracle(orc, inp, s0, heads=None):
    """Oracle over the input's sequences, optionally on a subset of heads, from state s0
    (a torch tensor of any float dtype, upcast exactly, or None)."""
    hs = slice(None) if heads is None else list(heads)
    sel = lambda t: to_f64_numpy(t[:, hs])  # noqa: E731
    s0n = None if s0 is None else sel(s0)
    cu = inp["cu_seqlens"].cpu().numpy().astype(np.int64)
    return orc.recurrent(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(inp["g"]),
                         sel(inp["beta"]), inp["scale"], s0=s0n, cu_seqlens=cu)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,H", [(1, 1), (7, 12), (33, 4)])
def test_single_token(orc, B, H, state_dtype):
    inp = make_inputs(custom([1] * B, H, True, seed=500 + B * 3 + H), DEV)
    s0 = inp["initial_state"].to(state_dtype)
    out, fin = K.kda_decode(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                            initial_state=s0)
    torch.cuda.synchronize()
    assert out.shape == (B, H, 128) and fin.dtype == state_dtype
    o_ref, f_ref = oracle(orc, inp, s0)
    assert_close(to_f64_numpy(out), o_ref, "decode out")
    assert_close(to_f64_numpy(fin), f_ref, "decode state")


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_steps_in_place_match_recurrence(orc, state_dtype):
    """Six one-token calls updating a state cache in place equal six recurrent steps,
    and equal one six-token call."""
    B, T, H = 5, 6, 12
    inp = make_inputs(custom([T] * B, H, True, seed=510), DEV)
    q, k, v, g, beta = dense_view(inp, B, T)
    s0 = inp["initial_state"].to(state_dtype)
    st = s0.clone()
    outs = []
    for t in range(T):
        o, _ = K.kda_decode(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                            g[:, t].contiguous(), beta[:, t].contiguous(), inp["scale"],
                            initial_state=st, final_state=st)
        outs.append(o)
    o_multi, f_multi = K.kda_decode(q, k, v, g, beta, inp["scale"], initial_state=s0)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle(orc, inp, s0)
    o_steps = torch.stack(outs, dim=1).reshape(B * T, H, 128)
    assert_close(to_f64_numpy(o_steps), o_ref, "stepped out")
    assert_close(to_f64_numpy(st), f_ref, "stepped state")
    assert_close(to_f64_numpy(o_multi.reshape(B * T, H, 128)), o_ref, "multi-token out")
    assert_close(to_f64_numpy(f_multi), f_ref, "multi-token state")
    # the same arithmetic per token, and the same storage rounding (fp32: none beyond the
    # arithmetic; bf16: after every token in both forms): bit-equal
    assert torch.equal(o_steps, o_multi.reshape(B * T, H, 128)) and torch.equal(st, f_multi)


def test_decode_continues_prefill(orc):
    """Prefill of 100 tokens, then two decode steps: the recurrence over 102 tokens."""
    H, L = 8, 102
    inp = make_inputs(custom([L], H, True, seed=520), DEV)
    x = {n: inp[n] for n in ("q", "k", "v", "g", "beta")}
    _, st = K.kda_prefill(*(x[n][:100] for n in ("q", "k", "v", "g", "beta")),
                          scale=inp["scale"], initial_state=inp["initial_state"],
                          output_final_state=True)
    outs = []
    for t in (100, 101):
        o, _ = K.kda_decode(*(x[n][t:t + 1].contiguous() for n in ("q", "k", "v", "g", "beta")),
                            scale=inp["scale"], initial_state=st, final_state=st)
        outs.append(o)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle(orc, inp, inp["initial_state"])
    assert_close(to_f64_numpy(torch.cat(outs)), o_ref[100:], "decode after prefill out")
    assert_close(to_f64_numpy(st), f_ref, "decode after prefill state")


def test_zero_tokens_copies_or_zeroes_state():
    B, H = 3, 5
    z = torch.empty(B, 0, H, 128, device=DEV, dtype=torch.bfloat16)
    zg = torch.empty(B, 0, H, 128, device=DEV, dtype=torch.float32)
    zb = torch.empty(B, 0, H, device=DEV, dtype=torch.bfloat16)
    for dt in (torch.float32, torch.bfloat16):
        s0 = torch.randn(B, H, 128, 128, device=DEV).to(dt)
        _, fin = K.kda_decode(z, z, z, zg, zb, 0.1, initial_state=s0)
        _, fin0 = K.kda_decode(z, z, z, zg, zb, 0.1, state_dtype=dt)
        torch.cuda.synchronize()
        assert torch.equal(fin, s0)
        assert torch.count_nonzero(fin0) == 0 and fin0.dtype == dt


def test_no_initial_state_is_zero_state(orc):
    inp = make_inputs(custom([1] * 9, 3, False, seed=530), DEV)
    out, fin = K.kda_decode(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"])
    torch.cuda.synchronize()
    o_ref, f_ref = oracle(orc, inp, None)
    assert_close(to_f64_numpy(out), o_ref, "zero-state out")
    assert_close(to_f64_numpy(fin), f_ref, "zero-state state")


def test_no_final_state_leaves_state_untouched():
    inp = make_inputs(custom([1] * 4, 2, True, seed=540), DEV)
    s0 = inp["initial_state"].clone()
    out, fin = K.kda_decode(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                            initial_state=inp["initial_state"], output_final_state=False)
    torch.cuda.synchronize()
    assert fin is None and torch.equal(inp["initial_state"], s0)
    assert torch.isfinite(out.float()).all()


def oracle_stored_bf16(orc, inp, s0, B, T):
    """The recurrence over B dense sequences of T tokens with the state stored in bf16
    after every token (round to nearest even), as a bf16 state cache holds it between
    decode steps; returns (out [B*T, H, 128], final state)."""
    H = inp["workload"].num_heads
    x = {n: to_f64_numpy(inp[n]).reshape((B, T) + tuple(inp[n].shape[1:]))
         for n in ("q", "k", "v", "g", "beta")}
    st = to_f64_numpy(s0)
    cu = np.arange(B + 1, dtype=np.int64)
    outs = []
    for t in range(T):
        o, f = orc.recurrent(*(x[n][:, t] for n in ("q", "k", "v", "g", "beta")), inp["scale"],
                             s0=st, cu_seqlens=cu)
        outs.append(o)
        st = to_f64_numpy(torch.from_numpy(f).to(torch.bfloat16))
    return np.stack(outs, axis=1).reshape(B * T, H, 128), st


def test_stress_slow_decay_many_steps(orc):
    """64 slow-decay steps updating the cache in place.  fp32 storage: against the plain
    fp64 recurrence.  bf16 storage: against the recurrence that stores the state in bf16
    after each token, the same rounding the cache applies (against the unrounded
    recurrence the compounded storage rounding is a few 1e-2 here, which is what bf16
    storage costs, not an arithmetic error)."""
    B, T, H = 4, 64, 4
    inp = make_inputs(custom([T] * B, H, True, seed=550), DEV, stress=True)
    q, k, v, g, beta = dense_view(inp, B, T)
    s0 = inp["initial_state"]
    for dt in (torch.float32, torch.bfloat16):
        st = s0.to(dt, copy=True)  # the cache is updated in place; s0 stays the oracle's
        outs = []
        for t in range(T):
            o, _ = K.kda_decode(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                                g[:, t].contiguous(), beta[:, t].contiguous(), inp["scale"],
                                initial_state=st, final_state=st)
            outs.append(o)
        torch.cuda.synchronize()
        if dt == torch.float32:
            o_ref, f_ref = oracle(orc, inp, s0)
        else:
            o_ref, f_ref = oracle_stored_bf16(orc, inp, s0.to(dt), B, T)
        assert_close(to_f64_numpy(torch.stack(outs, 1).reshape(B * T, H, 128)), o_ref,
                     f"stress out {dt}")
        assert_close(to_f64_numpy(st), f_ref, f"stress state {dt}")


def test_full_size_decode_sampled_heads(orc):
    """The decode workload (256 sequences x 64 heads, one token, fp32 and bf16 state)
    at full size; the oracle checks three heads of every sequence."""
    w = WORKLOADS["decode_b256_h64"]
    inp = make_inputs(w, DEV)
    heads = [0, 37, 63]
    for dt in (torch.float32, torch.bfloat16):
        s0 = inp["initial_state"].to(dt)
        out, fin = K.kda_decode(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                inp["scale"], initial_state=s0)
        torch.cuda.synchronize()
        o_ref, f_ref = oracle(orc, inp, s0, heads)
        assert_close(to_f64_numpy(out[:, heads]), o_ref, f"full decode out {dt}")
        assert_close(to_f64_numpy(fin[:, heads]), f_ref, f"full decode state {dt}")


def test_decode_deterministic_and_graph_capturable():
    inp = make_inputs(custom([1] * 16, 12, True, seed=560), DEV)
    x = [inp[n] for n in ("q", "k", "v", "g", "beta")]
    o1, f1 = K.kda_decode(*x, inp["scale"], initial_state=inp["initial_state"])
    out = torch.empty_like(o1)
    st = inp["initial_state"].clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        K.kda_decode(*x, inp["scale"], initial_state=st, final_state=st, out=out, stream=s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            K.kda_decode(*x, inp["scale"], initial_state=st, final_state=st, out=out, stream=s)
    st.copy_(inp["initial_state"])
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, o1) and torch.equal(st, f1)
