"""bf16 state I/O of the prefill (kda_options.state_dtype = KDA_STATE_BF16) against the
fp64 oracle.

The reference facade returns a bf16 final state (flashinfer PR #4313, review of
kda_prefill.py).  The prefill keeps fp32 arithmetic: a bf16 initial state is widened
exactly, the final state is rounded to bf16 (nearest even) once at the end, and carries
between segments or host token blocks stay fp32.  So each case runs the oracle from the
bf16 initial state itself (exact in fp64) and compares the output, and the final state
after rounding the oracle's to bf16 the same way, at atol = rtol = 1e-2 (flashinfer PR
#4351 "Correctness").  Slow-decay gates keep the initial state visible to the end.
Covered: dense, packed varlen (with an empty sequence, whose final state is its initial
state bit for bit), the in-place update (final_state is initial_state), segment mode
(the merge reads the bf16 initial state) dense and varlen, and the host entry point
streamed in token blocks (fp32 carry between blocks).
"""
import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.inputs import custom, make_inputs, to_bf16_rne

from kda_testutil import assert_close, gpu_out_heads, oracle_on_heads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H = 4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    K.load_library()


def _bf16_inputs(lens, seed, dense):
    inp = make_inputs(custom(lens, H, True, seed=seed, dense=dense), DEV, stress=True)
    inp["initial_state"] = to_bf16_rne(inp["initial_state"])  # the caller's bf16 states
    return inp


def _oracle(orc, inp):
    o_ref, f_ref = oracle_on_heads(orc, inp, range(H))  # from the bf16 S0, exactly widened
    f_ref_bf16 = torch.from_numpy(f_ref).to(torch.float32).to(torch.bfloat16).double().numpy()
    return o_ref, f_ref_bf16


def _check(out, fin, o_ref, f_ref_bf16, what):
    assert fin.dtype == torch.bfloat16
    assert_close(gpu_out_heads(out.reshape(-1, H, 128), range(H)), o_ref, f"{what} out")
    assert_close(fin.double().cpu().numpy(), f_ref_bf16, f"{what} final state")


def _dense_call(inp, B, T, **kw):
    q, k, v, g = (inp[x].view(B, T, H, 128) for x in ("q", "k", "v", "g"))
    beta = inp["beta"].view(B, T, H)
    return K.kda_prefill(q, k, v, g, beta, inp["scale"], **kw)


@pytest.mark.parametrize("mode,seg", [(K.MODE_SERIAL, 0), (K.MODE_SEGMENT, 64)])
def test_bf16_state_dense(orc, mode, seg):
    B, T = 2, 200
    inp = _bf16_inputs([T] * B, 1201, True)
    out, fin = _dense_call(inp, B, T, initial_state=inp["initial_state"], output_final_state=True,
                           mode=mode, segment_len=seg)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    _check(out, fin, *_oracle(orc, inp), f"dense mode {mode}")


@pytest.mark.parametrize("mode,seg", [(K.MODE_SERIAL, 0), (K.MODE_SEGMENT, 32)])
def test_bf16_state_varlen(orc, mode, seg):
    lens = [70, 0, 33, 129]
    inp = _bf16_inputs(lens, 1202, False)
    out, fin = K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                             initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"],
                             output_final_state=True, mode=mode, segment_len=seg)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    _check(out, fin, *_oracle(orc, inp), f"varlen mode {mode}")
    assert torch.equal(fin[1], inp["initial_state"][1]), "an empty sequence keeps its state"


def test_bf16_state_in_place(orc):
    B, T = 1, 150
    inp = _bf16_inputs([T] * B, 1203, True)
    o_ref, f_ref = _oracle(orc, inp)  # before the call overwrites the initial state
    cache = inp["initial_state"].clone()
    out, fin = _dense_call(inp, B, T, initial_state=cache, final_state=cache)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    assert fin.data_ptr() == cache.data_ptr()
    _check(out, fin, o_ref, f_ref, "in place")


def test_bf16_state_host_blocks(orc):
    """One long sequence through the host entry point in 4 token blocks: the first reads
    the bf16 initial state, the blocks pass an fp32 carry, the last writes bf16."""
    T = 640
    inp = _bf16_inputs([T], 1204, True)
    h = {n: inp[n].cpu() for n in ("q", "k", "v", "g", "beta", "initial_state")}
    out, fin = K.kda_prefill_host(h["q"].view(1, T, H, 128), h["k"].view(1, T, H, 128),
                                  h["v"].view(1, T, H, 128), h["g"].view(1, T, H, 128),
                                  h["beta"].view(1, T, H), inp["scale"],
                                  initial_state=h["initial_state"], output_final_state=True,
                                  host_pieces=4)
    _check(out, fin, *_oracle(orc, inp), "host blocks")
