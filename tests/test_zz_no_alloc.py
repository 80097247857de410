"""The no-allocation segment entry point against the allocating one.

Some callers of a prefill cannot call cudaMalloc: applications whose caching allocator
owns all of device memory, real-time services that must not allocate (or risk the
synchronisation an allocation can imply) inside a request, plugin hosts that give a
library no allocation rights.  kda_prefill_segment_noalloc serves them: it runs segment
mode with its scratch in a fixed device array of the library instead of a workspace.

It runs the same kernels on the same plan as kda_prefill_ex in segment mode, so its
results must be bit-identical to that call's.  This file calls it through the C ABI
twice in a row, the larger shape first, so that the second call runs on scratch the
first one left dirty (a read of a stale byte would change its result), with slow-decay
gates so the carries between segments matter, and requires torch.equal with the
allocating call each time; the second call is also held to the fp64 oracle at the
tolerance of the other GPU tests.  A shape whose scratch would not fit is refused before
any device work.  The file name sorts last so that a run stopping at the first failure
has run every other test already.
"""
import ctypes

import numpy as np
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


def _no_alloc_call(lib, inp, B, T, H, seg):
    q, k, v, g = (inp[x].view(B, T, H, 128) for x in ("q", "k", "v", "g"))
    beta = inp["beta"].view(B, T, H)
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
    return out, fin


def test_no_alloc_bit_identical_to_segment_mode(lib, orc):
    # Larger shape first (B*H*(3*nseg-2) = 1*8*10 = 80 state slots), then a smaller one
    # (2*4*7 = 56) whose scratch lies inside what the first call wrote.
    for call, (B, T, H, seg, seed) in enumerate([(1, 1000, 8, 256, 401), (2, 700, 4, 256, 402)]):
        inp = make_inputs(custom([T] * B, H, True, seed=seed), DEV, stress=True)
        q, k, v, g = (inp[x].view(B, T, H, 128) for x in ("q", "k", "v", "g"))
        beta = inp["beta"].view(B, T, H)
        ref_out, ref_fin = K.kda_prefill(q, k, v, g, beta, inp["scale"],
                                         initial_state=inp["initial_state"],
                                         output_final_state=True, mode=K.MODE_SEGMENT,
                                         segment_len=seg)
        out, fin = _no_alloc_call(lib, inp, B, T, H, seg)
        assert torch.equal(out, ref_out), f"call {call}: out differs from segment mode"
        assert torch.equal(fin, ref_fin), f"call {call}: final state differs from segment mode"
        if call == 1:
            cu = inp["cu_seqlens"].cpu().numpy().astype(np.int64)
            o_ref, f_ref = orc.recurrent(
                *(to_f64_numpy(inp[n]) for n in ("q", "k", "v", "g", "beta")), inp["scale"],
                s0=to_f64_numpy(inp["initial_state"]), cu_seqlens=cu)
            assert_close(to_f64_numpy(out.reshape(-1, H, 128)), o_ref, "out vs oracle")
            assert_close(to_f64_numpy(fin), f_ref, "final state vs oracle")


def test_no_alloc_rejects_shapes_beyond_its_scratch(lib):
    # T = 131072, H = 64, segments of 8192: 64 * (3 * 16 - 2) = 2944 state slots > 512.
    shape = KdaShape(1, 131072, 0, 64, 128)
    a = ctypes.c_void_p(0x10000000)
    st = lib.kda_prefill_segment_noalloc(ctypes.byref(shape), a, a, a, a, a,
                                         ctypes.c_float(0.1), None, ctypes.c_void_p(0x8000000000),
                                         None, ctypes.c_int32(8192), None)
    assert st == 1
    assert "scratch" in lib.kda_last_error_message().decode()
