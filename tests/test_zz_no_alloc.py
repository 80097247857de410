"""The no-allocation segment entry point against the allocating one.

kda_prefill_segment_noalloc serves callers that cannot call cudaMalloc (inside a
stream capture, under an allocator that owns all device memory, in a request path
that must not allocate): its segment scratch lives in a fixed device array of the
library.  This file calls it through the C ABI twice in a row, with different shapes
and inputs (the second call must not see the first call's scratch contents), and
compares each result with kda_prefill_ex in segment mode at the tolerance the other
GPU tests use.  It also checks that a shape whose scratch would not fit is refused
before any device work.  The file name sorts last so that a run stopping at the
first failure has run every other test already.
"""
import ctypes

import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.inputs import custom, make_inputs, to_f64_numpy
from chunked_kda_delta_gb300.kda import KdaShape

from kda_testutil import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    return K.load_library()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_no_alloc_matches_allocating_segment_mode(lib):
    for call, (B, T, H, seg, seed) in enumerate([(1, 1000, 8, 256, 401), (2, 700, 4, 128, 402)]):
        inp = make_inputs(custom([T] * B, H, True, seed=seed), DEV)
        q, k, v, g = (inp[x].view(B, T, H, 128) for x in ("q", "k", "v", "g"))
        beta = inp["beta"].view(B, T, H)
        ref_out, ref_fin = K.kda_prefill(q, k, v, g, beta, inp["scale"],
                                         initial_state=inp["initial_state"],
                                         output_final_state=True, mode=K.MODE_SEGMENT,
                                         segment_len=seg)
        out = torch.full_like(q, float("nan"))
        fin = torch.full_like(inp["initial_state"], float("nan"))
        shape = KdaShape(B, T, 0, H, 128)
        stream = torch.cuda.current_stream().cuda_stream
        st = lib.kda_prefill_segment_noalloc(
            ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta),
            ctypes.c_float(inp["scale"]), _p(inp["initial_state"]), _p(out), _p(fin),
            ctypes.c_int32(seg), ctypes.c_void_p(stream))
        assert st == 0, lib.kda_last_error_message().decode()
        torch.cuda.synchronize()
        assert K.kda_get_device_status() == 0
        assert_close(to_f64_numpy(out), to_f64_numpy(ref_out), f"call {call} out")
        assert_close(to_f64_numpy(fin), to_f64_numpy(ref_fin), f"call {call} final state")


def test_no_alloc_rejects_shapes_beyond_its_scratch(lib):
    # T = 131072, H = 64, segments of 8192: 64 * (3 * 16 - 2) = 2944 state slots > 512.
    shape = KdaShape(1, 131072, 0, 64, 128)
    a = ctypes.c_void_p(0x10000000)
    st = lib.kda_prefill_segment_noalloc(ctypes.byref(shape), a, a, a, a, a,
                                         ctypes.c_float(0.1), None, ctypes.c_void_p(0x8000000000),
                                         None, ctypes.c_int32(8192), None)
    assert st == 1
    assert "scratch" in lib.kda_last_error_message().decode()
