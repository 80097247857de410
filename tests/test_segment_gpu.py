"""Segment-parallel prefill (pre_scan -> merge -> segment-K2) on the GPU.

The pages claim the segment pipeline is bit-identical to the serial one (cuLA PR #103
commit notes and test list: a bit-exactness test of the context-parallel path against
the serial path).  Under the
plain reading of the pipeline the carries are products of per-segment transitions and
round differently from the serial chain, so this suite requires both modes to match
the fp64 oracle within atol = rtol = 1e-2 and reports the max abs difference between
them instead of asserting equality.
"""
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


def run(inp, mode, seg_len=0, stream=None):
    w = inp["workload"]
    B, T = w.num_seqs, w.seq_lens[0]
    q, k, v, g = (inp[x].view(B, T, w.num_heads, 128) for x in ("q", "k", "v", "g"))
    beta = inp["beta"].view(B, T, w.num_heads)
    out, fin = K.kda_prefill(q, k, v, g, beta, inp["scale"], initial_state=inp["initial_state"],
                             output_final_state=True, mode=mode, segment_len=seg_len,
                             stream=stream)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    return out.reshape(-1, w.num_heads, 128), fin


@pytest.mark.parametrize("B,T,seg,with_s0", [
    (1, 200, 64, True),     # 4 segments, ragged last one (8 tokens)
    (2, 130, 32, True),     # dense batch, 5 segments, ragged last chunk inside a segment
    (1, 256, 64, False),    # segments divide T
    (3, 48, 16, True),      # one chunk per segment
    (1, 40, 64, True),      # a single segment: plain serial path
])
def test_segment_matches_oracle(orc, B, T, seg, with_s0):
    inp = make_inputs(custom([T] * B, 4, with_s0, seed=300 + T + seg), DEV)
    out, fin = run(inp, K.MODE_SEGMENT, seg)
    o_ref, f_ref = oracle_on_heads(orc, inp, range(4))
    assert_close(gpu_out_heads(out, range(4)), o_ref, "segment out")
    assert_close(gpu_state_heads(fin, range(4)), f_ref, "segment final")


def test_segment_stress_slow_decay(orc):
    """Slow decay makes a wrong carry or transition visible far downstream."""
    inp = make_inputs(custom([512], 4, True, seed=310), DEV, stress=True)
    out, fin = run(inp, K.MODE_SEGMENT, 128)
    o_ref, f_ref = oracle_on_heads(orc, inp, range(4))
    assert_close(gpu_out_heads(out, range(4)), o_ref, "segment stress out")
    assert_close(gpu_state_heads(fin, range(4)), f_ref, "segment stress final")


def test_segment_vs_serial_long_workload(orc):
    """T = 131072, H = 64, segments of 8192 tokens: both modes against the oracle on
    sampled heads, and the max abs difference between the two modes over every output."""
    inp = make_inputs(WORKLOADS["long_t131072_h64"], DEV)
    o_ser, f_ser = run(inp, K.MODE_SERIAL)
    o_seg, f_seg = run(inp, K.MODE_SEGMENT, 8192)
    heads = [0, 63]
    o_ref, f_ref = oracle_on_heads(orc, inp, heads)
    assert_close(gpu_out_heads(o_seg, heads), o_ref, "segment out (sampled heads)")
    assert_close(gpu_state_heads(f_seg, heads), f_ref, "segment final (sampled heads)")
    d_out = (o_seg.float() - o_ser.float()).abs().max().item()
    d_fin = (f_seg - f_ser).abs().max().item()
    print(f"\nsegment vs serial max |diff|: out {d_out:.3e}, final state {d_fin:.3e}")
    assert d_out < 2e-2 and d_fin < 2e-2


def test_workspace_bytes_matches_plan():
    nb = K.kda_workspace_bytes(1, 131072, 64, mode=K.MODE_SEGMENT, segment_len=8192)
    assert nb == (2 * 15 + 16) * 64 * 128 * 128 * 4
    assert K.kda_workspace_bytes(1, 8192, 64, mode=K.MODE_SEGMENT, segment_len=8192) == 0


def test_capture_without_warmup_is_refused():
    inp = make_inputs(custom([256], 2, False, seed=311), DEV)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with pytest.raises(K.KdaError) as ei:
        with torch.cuda.graph(graph, stream=s):
            K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                          mode=K.MODE_SEGMENT, segment_len=64, stream=s)
    assert ei.value.status == 6
    torch.cuda.synchronize()
    # after a warm-up call on that stream the same call captures and replays
    out = torch.empty_like(inp["q"])
    with torch.cuda.stream(s):
        K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                      out=out, mode=K.MODE_SEGMENT, segment_len=64, stream=s)
    torch.cuda.synchronize()
    ref = out.clone()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                      out=out, mode=K.MODE_SEGMENT, segment_len=64, stream=s)
    out.zero_()
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_auto_mode_plans_segments_for_few_chains(orc):
    """Two chains on a GPU that holds dozens of clusters: MODE_AUTO takes the segment
    path the planner reports, matches the oracle, and sizes its workspace the same way."""
    T, H = 32768, 2
    resident = torch.cuda.get_device_properties(0).multi_processor_count // 2
    m, seg = K.kda_plan(1, T, H, resident)
    assert m == K.MODE_SEGMENT
    assert K.kda_workspace_bytes(1, T, H, mode=K.MODE_AUTO) == \
        K.kda_workspace_bytes(1, T, H, mode=K.MODE_SEGMENT, segment_len=seg)
    inp = make_inputs(custom([T], H, True, seed=320), DEV)
    out, fin = run(inp, K.MODE_AUTO)
    o_ref, f_ref = oracle_on_heads(orc, inp, range(H))
    assert_close(gpu_out_heads(out, range(H)), o_ref, "auto out")
    assert_close(gpu_state_heads(fin, range(H)), f_ref, "auto final")
    o_ser, f_ser = run(inp, K.MODE_SERIAL)
    print(f"\nauto (segment_len {seg}) vs serial max |diff|: out "
          f"{(out.float() - o_ser.float()).abs().max().item():.3e}")


def test_auto_mode_keeps_serial_for_many_chains():
    assert K.kda_workspace_bytes(1, 8192, 64, mode=K.MODE_AUTO) == 0


def run_varlen(inp, mode, seg_len=0):
    w = inp["workload"]
    out, fin = K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                             initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"],
                             output_final_state=True, mode=mode, segment_len=seg_len)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    return out.reshape(-1, w.num_heads, 128), fin


@pytest.mark.parametrize("lens,seg", [
    ([300, 17, 0, 129, 64], 64),      # ragged tails, an empty sequence, exact multiple
    ([33, 1, 70, 256], 32),           # one-token sequence, many segments
    ([500], 128),                     # a single packed sequence
    ([16, 16, 16], 16),               # every sequence one segment
])
def test_varlen_segment_matches_oracle(orc, lens, seg):
    inp = make_inputs(custom(lens, 3, True, seed=400 + sum(lens) + seg, dense=False), DEV)
    out, fin = run_varlen(inp, K.MODE_SEGMENT, seg)
    o_ref, f_ref = oracle_on_heads(orc, inp, range(3))
    assert_close(gpu_out_heads(out, range(3)), o_ref, "varlen segment out")
    assert_close(gpu_state_heads(fin, range(3)), f_ref, "varlen segment final")


def test_varlen_segment_stress_slow_decay(orc):
    inp = make_inputs(custom([700, 45, 260], 2, True, seed=411, dense=False), DEV, stress=True)
    out, fin = run_varlen(inp, K.MODE_SEGMENT, 128)
    o_ref, f_ref = oracle_on_heads(orc, inp, range(2))
    assert_close(gpu_out_heads(out, range(2)), o_ref, "varlen segment stress out")
    assert_close(gpu_state_heads(fin, range(2)), f_ref, "varlen segment stress final")


def test_varlen_segment_workload_vs_serial(orc):
    """The packed varlen workload (H = 12) in segment mode: oracle on sampled heads and the
    max difference against serial mode."""
    inp = make_inputs(WORKLOADS["varlen_h12"], DEV)
    o_seg, f_seg = run_varlen(inp, K.MODE_SEGMENT, 1024)
    o_ser, f_ser = run_varlen(inp, K.MODE_SERIAL)
    heads = [0, 11]
    o_ref, f_ref = oracle_on_heads(orc, inp, heads)
    assert_close(gpu_out_heads(o_seg, heads), o_ref, "varlen_h12 segment out")
    assert_close(gpu_state_heads(f_seg, heads), f_ref, "varlen_h12 segment final")
    d_out = (o_seg.float() - o_ser.float()).abs().max().item()
    print(f"\nvarlen segment vs serial max |diff|: out {d_out:.3e}")
    assert d_out < 2e-2


def test_varlen_segment_bad_cu_seqlens_is_reported():
    inp = make_inputs(custom([100, 100, 100], 2, False, seed=412, dense=False), DEV)
    bad = torch.tensor([0, 150, 120, 300], dtype=torch.int32, device=DEV)  # decreasing
    K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                  cu_seqlens=bad, mode=K.MODE_SEGMENT, segment_len=32)
    assert K.kda_get_device_status() == 1
    assert K.kda_get_device_status() == 0
