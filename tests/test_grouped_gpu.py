"""GPU parity of grouped (unequal) head counts against the fp64 oracle.

q has Hq heads, v, g, beta and the states H, k min(Hq, H) and the output max(Hq, H); one
count divides the other (the pages name unequal head counts, GVA, as a follow-up: cuLA
PR #103, intracard-CP planner notes).  The oracle runs every output head as a plain head
on the tensors it reads (oracle.grouped, pinned by a closed form in test_oracle.py).
Bar: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| (flashinfer PR #4351 "Correctness").
"""
import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.inputs import WORKLOADS, custom, make_inputs, to_f64_numpy

from kda_testutil import assert_close, oracle_grouped, oracle_grouped_on_heads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
PAIRS = [(2, 6), (6, 2), (1, 4), (4, 1), (12, 3), (3, 12)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    K.load_library()


def args_of(inp):
    w = inp["workload"]
    x = {n: inp[n] for n in ("q", "k", "v", "g", "beta")}
    cu = None
    if w.dense:
        B, T = w.num_seqs, w.seq_lens[0]
        for n in ("q", "k", "v", "g"):
            x[n] = x[n].view(B, T, x[n].shape[1], 128)
        x["beta"] = x["beta"].view(B, T, -1)
    else:
        cu = inp["cu_seqlens"]
    return x, cu


def run(inp, **kw):
    x, cu = args_of(inp)
    out, fin = K.kda_prefill(**x, scale=inp["scale"], initial_state=inp["initial_state"],
                             cu_seqlens=cu, output_final_state=True, **kw)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    return out.reshape(-1, out.shape[-2], 128), fin


@pytest.mark.parametrize("Hq,H", PAIRS)
@pytest.mark.parametrize("T", [33, 100])
def test_dense_every_element(orc, Hq, H, T):
    inp = make_inputs(custom([T, T], H, True, seed=600 + 13 * Hq + H + T, num_q_heads=Hq), DEV)
    out, fin = run(inp)
    assert out.shape[1] == max(Hq, H) and fin.shape[1] == H
    o_ref, f_ref = oracle_grouped(inp)
    assert_close(to_f64_numpy(out), o_ref, f"Hq={Hq} H={H} out")
    assert_close(to_f64_numpy(fin), f_ref, f"Hq={Hq} H={H} final")


@pytest.mark.parametrize("Hq,H", [(3, 12), (12, 3)])
def test_varlen_every_element(orc, Hq, H):
    inp = make_inputs(custom([32, 3, 0, 17, 47], H, False, seed=610 + Hq, dense=False,
                             num_q_heads=Hq), DEV)
    out, fin = run(inp)
    o_ref, f_ref = oracle_grouped(inp)
    assert_close(to_f64_numpy(out), o_ref, "varlen out")
    assert_close(to_f64_numpy(fin), f_ref, "varlen final")


def test_in_place_state_grouped_queries(orc):
    """Query heads sharing a state head run the same chain; the state is written once, so
    an in-place update is still exact."""
    inp = make_inputs(custom([60], 2, True, seed=620, num_q_heads=8), DEV)
    o_ref, f_ref = oracle_grouped(inp)
    st = inp["initial_state"]
    x, _ = args_of(inp)
    out, _ = K.kda_prefill(**x, scale=inp["scale"], initial_state=st, final_state=st)
    torch.cuda.synchronize()
    assert_close(to_f64_numpy(out.reshape(-1, 8, 128)), o_ref, "in-place out")
    assert_close(to_f64_numpy(st), f_ref, "in-place state")


def test_auto_mode_runs_grouped_serially(orc):
    inp = make_inputs(custom([300], 4, True, seed=630, num_q_heads=2), DEV)
    out, fin = run(inp, mode=K.MODE_AUTO)
    o_ref, f_ref = oracle_grouped(inp)
    assert_close(to_f64_numpy(out), o_ref, "auto out")
    assert_close(to_f64_numpy(fin), f_ref, "auto final")


@pytest.mark.parametrize("Hq,H", [(2, 6), (6, 2)])
def test_segment_mode_grouped_dense(orc, Hq, H):
    """Summaries and transitions run once per state head, the output pass once per output
    head; slow decay so the carries matter."""
    inp = make_inputs(custom([300, 300], H, True, seed=640 + Hq, num_q_heads=Hq), DEV,
                      stress=True)
    out, fin = run(inp, mode=K.MODE_SEGMENT, segment_len=64)
    o_ref, f_ref = oracle_grouped(inp)
    assert_close(to_f64_numpy(out), o_ref, "grouped segment out")
    assert_close(to_f64_numpy(fin), f_ref, "grouped segment final")


@pytest.mark.parametrize("Hq,H", [(3, 12), (12, 3)])
def test_segment_mode_grouped_varlen(orc, Hq, H):
    inp = make_inputs(custom([200, 3, 0, 97, 150], H, True, seed=645 + Hq, dense=False,
                             num_q_heads=Hq), DEV, stress=True)
    out, fin = run(inp, mode=K.MODE_SEGMENT, segment_len=48)
    o_ref, f_ref = oracle_grouped(inp)
    assert_close(to_f64_numpy(out), o_ref, "grouped varlen segment out")
    assert_close(to_f64_numpy(fin), f_ref, "grouped varlen segment final")


def test_segment_noalloc_grouped(orc):
    inp = make_inputs(custom([256], 2, True, seed=648, num_q_heads=8), DEV, stress=True)
    x, _ = args_of(inp)
    out = torch.empty(1, 256, 8, 128, dtype=torch.bfloat16, device=DEV)
    fin = torch.empty(1, 2, 128, 128, device=DEV)
    K.kda.kda_prefill_segment_noalloc(**x, out=out, segment_len=64, scale=inp["scale"],
                                      initial_state=inp["initial_state"], final_state=fin)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle_grouped(inp)
    assert_close(to_f64_numpy(out.reshape(-1, 8, 128)), o_ref, "noalloc grouped out")
    assert_close(to_f64_numpy(fin), f_ref, "noalloc grouped final")


def test_host_entry_point_grouped():
    inp = make_inputs(custom([40, 9], 6, True, seed=650, dense=False, num_q_heads=2), DEV)
    o_dev, f_dev = run(inp)
    cpu = {n: inp[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}
    o_h, f_h = K.kda_prefill_host(**cpu, scale=inp["scale"],
                                  initial_state=inp["initial_state"].cpu(),
                                  cu_seqlens=inp["cu_seqlens"].cpu(), output_final_state=True)
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(f_h, f_dev.cpu())


@pytest.mark.parametrize("name,heads", [("gva_t8192_q16_v64", [0, 37, 63]),
                                        ("gqa_t8192_q64_v16", [0, 5, 63])])
def test_full_size_sampled_heads(orc, name, heads):
    inp = make_inputs(WORKLOADS[name], DEV)
    out, fin = run(inp)
    o_ref, f_ref = oracle_grouped_on_heads(orc, inp, heads)
    assert_close(to_f64_numpy(out[:, heads]), o_ref, f"{name} out")
    w = inp["workload"]
    import oracle
    states = [oracle.grouped_heads(ho, w.num_heads, w.q_heads)[2] for ho in heads]
    assert_close(to_f64_numpy(fin[:, states]), f_ref, f"{name} final")


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("Hq,H", [(2, 6), (6, 2)])
def test_decode_grouped(orc, Hq, H, state_dtype):
    inp = make_inputs(custom([1] * 9, H, True, seed=660 + Hq, num_q_heads=Hq), DEV)
    s0 = inp["initial_state"].to(state_dtype)
    out, fin = K.kda_decode(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                            initial_state=s0)
    torch.cuda.synchronize()
    ref = dict(inp)
    ref["initial_state"] = s0
    o_ref, f_ref = oracle_grouped(ref)
    assert_close(to_f64_numpy(out), o_ref, "grouped decode out")
    assert_close(to_f64_numpy(fin), f_ref, "grouped decode state")
