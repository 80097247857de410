"""The host entry point streamed in pieces (kda_prefill_host, host_pieces).

Several sequences split into ranges of whole sequences: every chain computes exactly
as in one device call, so outputs and final states must be bit-identical to it.  One
sequence splits into token blocks of whole chunks, the fp32 state carried from block
to block: checked against the fp64 oracle at the pages' tolerance (flashinfer PR #4351
"Correctness": atol = rtol = 1e-2).
"""
import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.inputs import custom, make_inputs, to_f64_numpy

from kda_testutil import assert_close, oracle_grouped, oracle_on_heads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    K.load_library()


def _views(inp, tensors):
    """Dense workloads as [B, T, heads, ...] views; packed ones as they are."""
    w = inp["workload"]
    if not w.dense:
        return tensors, inp["cu_seqlens"]
    B, T = w.num_seqs, w.seq_lens[0]
    out = {n: t.view(B, T, *t.shape[1:]) for n, t in tensors.items()}
    return out, None


def device_call(inp, **kw):
    args, cu = _views(inp, {n: inp[n] for n in ("q", "k", "v", "g", "beta")})
    out, fin = K.kda_prefill(**args, scale=inp["scale"], initial_state=inp["initial_state"],
                             cu_seqlens=cu, output_final_state=True, **kw)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    return out.cpu(), fin.cpu()


def host_call(inp, pieces, with_final=True, **kw):
    args, cu = _views(inp, {n: inp[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")})
    s0 = inp["initial_state"]
    out, fin = K.kda_prefill_host(**args, scale=inp["scale"],
                                  initial_state=None if s0 is None else s0.cpu().pin_memory(),
                                  cu_seqlens=None if cu is None else cu.cpu(),
                                  output_final_state=with_final, host_pieces=pieces, **kw)
    assert K.kda_get_device_status() == 0
    return out, fin


@pytest.mark.parametrize("pieces", [2, 3, 7, 64])
def test_sequence_ranges_bit_identical_packed(pieces):
    inp = make_inputs(custom([300, 45, 0, 700, 16, 129, 512], 3, True, seed=3101, dense=False), DEV)
    o_dev, f_dev = device_call(inp)
    o_h, f_h = host_call(inp, pieces)
    assert torch.equal(o_h, o_dev) and torch.equal(f_h, f_dev)


@pytest.mark.parametrize("H,Hq", [(4, 8), (6, 2)])
def test_sequence_ranges_bit_identical_grouped(H, Hq):
    inp = make_inputs(custom([200, 0, 333, 64, 17], H, True, seed=3108 + Hq, dense=False,
                             num_q_heads=Hq), DEV)
    o_dev, f_dev = device_call(inp)
    o_h, f_h = host_call(inp, 3)
    assert torch.equal(o_h, o_dev) and torch.equal(f_h, f_dev)


@pytest.mark.parametrize("pieces", [2, 5])
def test_sequence_ranges_bit_identical_dense(pieces):
    inp = make_inputs(custom([200] * 5, 2, True, seed=3102, dense=True), DEV)
    o_dev, f_dev = device_call(inp)
    o_h, f_h = host_call(inp, pieces)
    assert torch.equal(o_h, o_dev) and torch.equal(f_h, f_dev)


@pytest.mark.parametrize("pieces", [4, 63])
def test_token_blocks_against_oracle(orc, pieces):
    # 1000 tokens = 62 full chunks + 8; 63 pieces puts every chunk in its own block
    inp = make_inputs(custom([1000], 4, True, seed=3103 + pieces), DEV)
    o_h, f_h = host_call(inp, pieces)
    o_ref, f_ref = oracle_on_heads(orc, inp, range(4))
    assert_close(to_f64_numpy(o_h.reshape(-1, 4, 128)), o_ref, f"{pieces} blocks out")
    assert_close(to_f64_numpy(f_h), f_ref, f"{pieces} blocks final_state")


def test_token_blocks_without_states(orc):
    # no initial state and no final state: the carried state still lives in the arena
    inp = make_inputs(custom([777], 3, False, seed=3104), DEV)
    o_h, f_h = host_call(inp, 5, with_final=False)
    assert f_h is None
    o_ref, _ = oracle_on_heads(orc, inp, range(3))
    assert_close(to_f64_numpy(o_h.reshape(-1, 3, 128)), o_ref, "blocks without states")


@pytest.mark.parametrize("H,Hq", [(6, 2), (2, 4)])
def test_token_blocks_grouped_heads(H, Hq):
    inp = make_inputs(custom([600], H, True, seed=3105 + Hq, num_q_heads=Hq), DEV)
    o_h, f_h = host_call(inp, 3)
    o_ref, f_ref = oracle_grouped(inp)
    assert_close(to_f64_numpy(o_h.reshape(-1, max(H, Hq), 128)), o_ref, "grouped blocks out")
    assert_close(to_f64_numpy(f_h), f_ref, "grouped blocks final_state")


def test_segment_plan_runs_in_one_piece():
    # AUTO picks segment mode for one long sequence with two heads: the host call then
    # runs unsplit and matches the device call bit for bit
    assert K.kda_plan(1, 32768, 2, 76)[0] == K.MODE_SEGMENT
    inp = make_inputs(custom([32768], 2, False, seed=3106), DEV)
    o_dev, f_dev = device_call(inp, mode=K.MODE_AUTO)
    o_h, f_h = host_call(inp, 8, mode=K.MODE_AUTO)
    assert torch.equal(o_h, o_dev) and torch.equal(f_h, f_dev)


def test_default_pieces_on_a_large_input(orc):
    # 8192 tokens x 16 heads is 201 MB of inputs: the library streams it in 8 token blocks
    inp = make_inputs(custom([8192], 16, True, seed=3107), DEV)
    o_h, f_h = host_call(inp, 0)
    heads = [0, 7, 15]
    o_ref, f_ref = oracle_on_heads(orc, inp, heads)
    assert_close(to_f64_numpy(o_h.reshape(-1, 16, 128)[:, heads]), o_ref, "default pieces out")
    assert_close(to_f64_numpy(f_h[:, heads]), f_ref, "default pieces final_state")


def test_auto_plans_varlen_segments_from_host_offsets(orc):
    """The host entry sees packed offsets on the host: AUTO runs two long sequences of a
    packed batch as a segment plan (kda_plan_varlen's pick) and matches the oracle, every
    element, with slow-decay gates so the carries between segments matter."""
    lens, H = [20000, 3, 19984], 2
    mode, seg = K.kda_plan_varlen(lens, H, 76)
    assert mode == K.MODE_SEGMENT
    inp = make_inputs(custom(lens, H, True, seed=1401, dense=False), "cpu", stress=True)
    h = {n: inp[n].pin_memory() for n in ("q", "k", "v", "g", "beta", "initial_state")}
    out, fin = K.kda_prefill_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["scale"],
                                  initial_state=h["initial_state"], cu_seqlens=inp["cu_seqlens"],
                                  output_final_state=True, mode=K.MODE_AUTO)
    assert K.kda_get_device_status() == 0
    o_ref, f_ref = oracle_on_heads(orc, inp, range(H))
    assert_close(to_f64_numpy(out), o_ref, "host AUTO varlen out")
    assert_close(to_f64_numpy(fin), f_ref, "host AUTO varlen final state")
