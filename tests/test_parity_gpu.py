"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| on the bf16 output and the fp32
final state (the pages' tolerance, flashinfer PR #4351 "Correctness").
Small cases compare every element; the full-size workloads compare every
token of sampled heads (heads are independent, so the oracle computes them
one by one).  Edge cases follow the pages' list: T = 32 and 33 (a full chunk
plus a tail), packed [32, 3], H = 12, in-place state, graph replay after beta
changes (flashinfer PR #4351), every (initial?, final?) combination (cuLA PR
#103 commit notes).
"""
import numpy as np
import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.inputs import WORKLOADS, custom, make_inputs, to_f64_numpy

from kda_testutil import assert_close, gpu_out_heads, gpu_state_heads, oracle_on_heads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    K.load_library()


def run_gpu(inp, with_final=True, **kw):
    w = inp["workload"]
    q, k, v, g, beta = inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"]
    cu = None
    if w.dense:
        B, T = w.num_seqs, w.seq_lens[0]
        q, k, v, g = (x.view(B, T, w.num_heads, 128) for x in (q, k, v, g))
        beta = beta.view(B, T, w.num_heads)
    else:
        cu = inp["cu_seqlens"]
    out, fin = K.kda_prefill(q, k, v, g, beta, inp["scale"], initial_state=inp["initial_state"],
                             cu_seqlens=cu, output_final_state=with_final, **kw)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    return out.reshape(-1, w.num_heads, 128), fin


def check_heads(orc, inp, heads, out, fin, what):
    o_ref, f_ref = oracle_on_heads(orc, inp, heads)
    assert_close(gpu_out_heads(out, heads), o_ref, f"{what} out")
    if fin is not None:
        assert_close(gpu_state_heads(fin, heads), f_ref, f"{what} final_state")


# --- small cases, every element ----------------------------------------------------------

def test_tiny_workload(orc):
    inp = make_inputs(WORKLOADS["tiny_t64_h4"], DEV)
    out, fin = run_gpu(inp)
    check_heads(orc, inp, range(4), out, fin, "tiny_t64_h4")


@pytest.mark.parametrize("T", [1, 3, 15, 16, 17, 32, 33, 100])
@pytest.mark.parametrize("H", [1, 12])
def test_edge_lengths(orc, T, H):
    inp = make_inputs(custom([T], H, True, seed=1000 + T * 7 + H), DEV)
    out, fin = run_gpu(inp)
    check_heads(orc, inp, range(H), out, fin, f"T={T} H={H}")


@pytest.mark.parametrize("lens", [[32, 3], [32, 3, 33], [0, 5, 0, 17], [1] * 9, [47, 16, 1, 64]])
def test_varlen(orc, lens):
    inp = make_inputs(custom(lens, 12, True, seed=sum(lens), dense=False), DEV)
    out, fin = run_gpu(inp)
    check_heads(orc, inp, range(12), out, fin, f"varlen {lens}")


@pytest.mark.parametrize("with_init", [False, True])
@pytest.mark.parametrize("with_final", [False, True])
def test_state_combinations(orc, with_init, with_final):
    inp = make_inputs(custom([40, 40], 3, with_init, seed=77), DEV)
    out, fin = run_gpu(inp, with_final=with_final)
    assert (fin is not None) == with_final
    check_heads(orc, inp, range(3), out, fin, f"init={with_init} final={with_final}")


def test_in_place_state(orc):
    inp = make_inputs(custom([50], 4, True, seed=78), DEV)
    s0 = inp["initial_state"].clone()
    o_ref, f_ref = oracle_on_heads(orc, inp, range(4))
    st = inp["initial_state"]
    out, _ = K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                           initial_state=st, final_state=st)
    torch.cuda.synchronize()
    assert not torch.equal(st, s0)
    assert_close(to_f64_numpy(st), f_ref, "in-place final state")
    assert_close(to_f64_numpy(out), o_ref, "in-place out")


def test_continuation_two_calls(orc):
    inp = make_inputs(custom([70], 4, True, seed=79), DEV)
    cut = 37
    o_ref, f_ref = oracle_on_heads(orc, inp, range(4))
    a = {k: inp[k][:cut] for k in ("q", "k", "v", "g", "beta")}
    b = {k: inp[k][cut:].contiguous() for k in ("q", "k", "v", "g", "beta")}
    o1, f1 = K.kda_prefill(**a, scale=inp["scale"], initial_state=inp["initial_state"],
                           output_final_state=True)
    o2, f2 = K.kda_prefill(**b, scale=inp["scale"], initial_state=f1, output_final_state=True)
    torch.cuda.synchronize()
    assert_close(to_f64_numpy(torch.cat([o1, o2])), o_ref, "continuation out")
    assert_close(to_f64_numpy(f2), f_ref, "continuation final")


def test_slow_decay_stress(orc):
    inp = make_inputs(custom([300], 4, True, seed=80), DEV, stress=True)
    out, fin = run_gpu(inp)
    check_heads(orc, inp, range(4), out, fin, "stress")


def test_zero_total_tokens_copies_state():
    s0 = torch.randn(2, 3, 128, 128, device=DEV)
    z = torch.empty(1, 0, 3, 128, device=DEV, dtype=torch.bfloat16)
    z = torch.empty(2, 0, 3, 128, device=DEV, dtype=torch.bfloat16)
    zg = torch.empty(2, 0, 3, 128, device=DEV, dtype=torch.float32)
    zb = torch.empty(2, 0, 3, device=DEV, dtype=torch.bfloat16)
    out, fin = K.kda_prefill(z, z, z, zg, zb, 0.1, initial_state=s0, output_final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(fin, s0)
    _, fin0 = K.kda_prefill(z, z, z, zg, zb, 0.1, output_final_state=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(fin0) == 0


# --- full-size workloads, sampled heads ------------------------------------------------

FULL = {
    "single_t8192_h64": [0, 37, 63],
    "batch4_t4096_h128": [0, 101],
    "varlen_h12": [0, 5, 11],
    "long_t131072_h64": [0, 63],
}


@pytest.mark.parametrize("name", sorted(FULL))
def test_full_workload_sampled_heads(orc, name):
    inp = make_inputs(WORKLOADS[name], DEV)
    out, fin = run_gpu(inp)
    assert torch.isfinite(out.float()).all()
    check_heads(orc, inp, FULL[name], out, fin, name)


@pytest.mark.parametrize("name", ["single_t8192_h64", "long_t131072_h64"])
def test_full_workload_stress_sampled_heads(orc, name):
    w = WORKLOADS[name]
    w = custom(w.seq_lens, w.num_heads, True, seed=w.seed, name=name)
    inp = make_inputs(w, DEV, stress=True)
    out, fin = run_gpu(inp)
    check_heads(orc, inp, [3], out, fin, name + " stress")


# --- behaviour -------------------------------------------------------------------------

def test_deterministic():
    inp = make_inputs(custom([333, 17], 8, True, seed=81), DEV)
    o1, f1 = run_gpu(inp)
    for _ in range(5):
        o2, f2 = run_gpu(inp)
        assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_graph_capture_replay_after_beta_change():
    inp = make_inputs(custom([96], 12, True, seed=82), DEV)
    out = torch.empty_like(inp["q"])
    fin = torch.empty_like(inp["initial_state"])
    args = dict(scale=inp["scale"], initial_state=inp["initial_state"], out=out,
                final_state=fin)
    x = {k: inp[k] for k in ("q", "k", "v", "g", "beta")}
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        K.kda_prefill(**x, **args, stream=s)          # warm-up outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            K.kda_prefill(**x, **args, stream=s)
    inp["beta"].mul_(0.5)
    graph.replay()
    torch.cuda.synchronize()
    ref_out, ref_fin = K.kda_prefill(**x, scale=inp["scale"],
                                     initial_state=inp["initial_state"],
                                     output_final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)


def test_device_status_reports_bad_cu_seqlens():
    inp = make_inputs(custom([20, 20, 20], 2, False, seed=83, dense=False), DEV)
    bad = torch.tensor([0, 30, 25, 60], dtype=torch.int32, device=DEV)  # decreasing
    K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                  cu_seqlens=bad)
    assert K.kda_get_device_status() == 1
    assert K.kda_get_device_status() == 0  # read-and-clear


def test_host_entry_point_matches_device_path():
    inp = make_inputs(custom([45, 19], 5, False, seed=84, dense=False), DEV)
    o_dev, f_dev = run_gpu(inp)
    cpu = {k: inp[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
    o_h, f_h = K.kda_prefill_host(**cpu, scale=inp["scale"],
                                  cu_seqlens=inp["cu_seqlens"].cpu(), output_final_state=True)
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(f_h, f_dev.cpu())


def test_bounded_wait_timeout_is_reported_and_recoverable():
    """With the stall flag the kernel waits on a barrier nothing signals: its bounded
    wait must run out, KDA_ERR_DEVICE_TIMEOUT is recorded, copies and MMAs drain, the
    kernel exits, and the context stays usable for the next call."""
    inp = make_inputs(custom([2000], 8, True, seed=85), DEV)
    args = {k: inp[k] for k in ("q", "k", "v", "g", "beta")}
    K.kda_prefill(**args, scale=inp["scale"], initial_state=inp["initial_state"],
                  output_final_state=True, wait_limit=2000, debug_flags=K.kda.DEBUG_STALL_WAIT)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 7
    assert K.kda_get_device_status() == 0
    out, fin = run_gpu(inp)  # a normal call afterwards still works (and checks status 0)
    o2, f2 = run_gpu(inp)
    assert torch.equal(out, o2) and torch.equal(fin, f2)
