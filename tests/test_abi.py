"""Host-side tests of the C ABI: the library loads, exports every declared symbol,
and rejects invalid calls with the documented status before any device work."""
import ctypes
import os
import re

import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.kda import KdaOptions, KdaShape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return K.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    assert set(names) == set(K.kda.EXPORTED_SYMBOLS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(lib):
    for code, name in K.kda._STATUS.items():
        assert K.kda_status_string(code) == name
    assert lib.kda_version().decode().count(".") == 2


def _call(lib, shape, ptrs=None, scale=0.1, opts=None, **over):
    # Fake, suitably aligned device-looking addresses: validation never dereferences them.
    base = dict(q=0x10000000, k=0x20000000, v=0x30000000, g=0x40000000, beta=0x50000000,
                s0=None, cu=None, out=0x60000000, fin=None)
    base.update(ptrs or {})
    base.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.kda_prefill_ex(ctypes.byref(shape), P(base["q"]), P(base["k"]), P(base["v"]),
                              P(base["g"]), P(base["beta"]), ctypes.c_float(scale),
                              P(base["s0"]), P(base["cu"]), P(base["out"]), P(base["fin"]),
                              None, None if opts is None else ctypes.byref(opts))


INVALID, ALIAS = 1, 2


@pytest.mark.parametrize("shape", [
    KdaShape(1, 16, 0, 4, 64),     # head_dim != 128
    KdaShape(1, 16, 0, 0, 128),    # no heads
    KdaShape(1, -1, 0, 4, 128),    # negative length
    KdaShape(0, 16, 0, 4, 128),    # no batch
])
def test_bad_shapes_rejected(lib, shape):
    assert _call(lib, shape) == INVALID
    assert lib.kda_last_error_message().decode()


def test_null_and_misaligned_pointers(lib):
    s = KdaShape(1, 16, 0, 4, 128)
    assert _call(lib, s, q=None) == INVALID
    assert _call(lib, s, out=None) == INVALID
    assert _call(lib, s, g=0x40000004) == INVALID          # not 16-byte aligned
    assert _call(lib, s, beta=0x50000001) == INVALID       # odd
    assert _call(lib, s, s0=0x70000008) == INVALID
    assert _call(lib, s, scale=float("nan")) == INVALID
    assert _call(lib, s, scale=float("inf")) == INVALID


def test_varlen_rules(lib):
    assert _call(lib, KdaShape(2, 16, 1, 4, 128), cu=0x70000000) == INVALID  # batch != 1
    assert _call(lib, KdaShape(1, 16, 0, 4, 128), cu=0x70000000) == INVALID  # num_seqs 0
    assert _call(lib, KdaShape(1, 16, 1, 4, 128), cu=0x70000002) == INVALID  # misaligned
    opts = KdaOptions(1, 64, 0, 0, 0)  # segment mode accepts packed varlen input
    assert _call(lib, KdaShape(1, 16, 1, 4, 128), cu=0x70000000, opts=opts) not in (INVALID, ALIAS)


def test_options_rules(lib):
    s = KdaShape(1, 16, 0, 4, 128)
    assert _call(lib, s, opts=KdaOptions(9, 0, 0, 0, 0)) == INVALID
    assert _call(lib, s, opts=KdaOptions(1, 24, 0, 0, 0)) == INVALID   # not a multiple of 16
    assert _call(lib, s, opts=KdaOptions(1, -16, 0, 0, 0)) == INVALID
    assert _call(lib, s, opts=KdaOptions(0, 0, -1, 0, 0)) == INVALID
    assert _call(lib, s, opts=KdaOptions(0, 0, 0, 2, 0)) == INVALID    # unknown debug bit
    assert _call(lib, s, opts=KdaOptions(0, 0, 0, 0, -1)) == INVALID   # host_pieces < 0
    assert _call(lib, s, opts=KdaOptions(0, 0, 0, 0, 65)) == INVALID   # host_pieces > 64
    # host_pieces is a host-entry setting; the device entry points accept and ignore it
    assert _call(lib, s, opts=KdaOptions(0, 0, 0, 0, 8)) not in (INVALID, ALIAS)
    assert _call(lib, s, opts=KdaOptions(0, 0, 0, 0, 0, 2)) == INVALID  # unknown state_dtype
    assert _call(lib, s, opts=KdaOptions(0, 0, 0, 0, 0, 1)) not in (INVALID, ALIAS)


def test_state_dtype_sizes_the_aliasing_checks(lib):
    # 4 heads of one sequence: fp32 states take 4 * 64 KiB, bf16 states 4 * 32 KiB.  A final
    # state right after a bf16 initial state is clear of it, but overlaps an fp32 one.
    s = KdaShape(1, 16, 0, 4, 128)
    s0, fin = 0x70000000, 0x70000000 + 4 * 128 * 128 * 2
    bf16 = KdaOptions(0, 0, 0, 0, 0, 1)
    assert _call(lib, s, s0=s0, fin=fin, opts=bf16) not in (INVALID, ALIAS)
    assert _call(lib, s, s0=s0, fin=fin) == ALIAS
    assert _call(lib, s, s0=s0, fin=fin, opts=KdaOptions(0, 0, 0, 0, 0, 0)) == ALIAS
    # the exact alias (in-place update) stays allowed for either type
    assert _call(lib, s, s0=s0, fin=s0, opts=bf16) not in (INVALID, ALIAS)


def test_aliasing_rules(lib):
    s = KdaShape(1, 16, 0, 4, 128)
    x = 16 * 4 * 128 * 2
    # out overlapping q, or sitting inside g
    assert _call(lib, s, out=0x10000000 + 256) == ALIAS
    assert _call(lib, s, out=0x40000000 + x) == ALIAS
    st = 1 * 4 * 128 * 128 * 4
    # partial overlap of initial and final state is rejected
    assert _call(lib, s, s0=0x70000000, fin=0x70000000 + 4096) == ALIAS
    # final state inside an input
    assert _call(lib, s, fin=0x10000000) == ALIAS
    # out overlapping the final state
    assert _call(lib, s, fin=0x70000000, out=0x70000000 + st - 16) == ALIAS


def test_in_place_state_passes_validation(lib):
    s = KdaShape(1, 16, 0, 4, 128)
    rc = _call(lib, s, s0=0x70000000, fin=0x70000000)
    # validation accepts the exact alias; without a GPU the next step fails in CUDA
    assert rc not in (INVALID, ALIAS)


def test_workspace_bytes(lib):
    assert K.kda_workspace_bytes(1, 8192, 64) == 0
    with pytest.raises(K.KdaError):
        K.kda_workspace_bytes(1, 8192, 64, head_dim=64)


def test_binding_checks_dtypes():
    q = torch.zeros(16, 2, 128, dtype=torch.float32)
    with pytest.raises(ValueError):
        K.kda_prefill_host(q, q, q, q, torch.zeros(16, 2, dtype=torch.bfloat16))


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(K.KdaError):
        K.load_library(str(tmp_path / "nope.so"))


def test_planner_decisions(lib):
    """The AUTO plan (host only): segment mode only when the chains alone cannot fill the
    GPU and the sequence is long; never for varlen input or a single chunk."""
    R = 76
    assert K.kda_plan(1, 131072, 64, R) == (K.MODE_SERIAL, 0)
    assert K.kda_plan(4, 4096, 128, R) == (K.MODE_SERIAL, 0)
    assert K.kda_plan(1, 64, 4, R) == (K.MODE_SERIAL, 0)
    assert K.kda_plan(1, 131072, 4, R, varlen=True, num_seqs=3) == (K.MODE_SERIAL, 0)
    m, s = K.kda_plan(1, 131072, 4, R)
    assert m == K.MODE_SEGMENT and s > 0 and s % 16 == 0 and s < 131072
    m, s = K.kda_plan(1, 32768, 2, R)
    assert m == K.MODE_SEGMENT and s % 16 == 0


def test_planner_picks_the_measured_best_segment_length(lib):
    # T = 131072 on GB300 (L2 flushed before each call), segment mode:
    #   H = 4: 8192 / 7296 / 6912 / 6560 tokens (16 / 18 / 19 / 20 segments) took
    #          1.40 / 1.27 / 1.20 / 1.47 ms (serial 7.13 ms); 19 segments fill the 76
    #          cluster slots in every pass;
    #   H = 2: 4096 / 3456 tokens 0.740 / 0.664 ms;  H = 8: 2048 / 3456 / 6912 tokens
    #          2.52 / 2.31 / 2.21 ms.
    assert K.kda_plan(1, 131072, 4, 76) == (K.MODE_SEGMENT, 6912)
    assert K.kda_plan(1, 131072, 2, 76) == (K.MODE_SEGMENT, 3456)
    assert K.kda_plan(1, 131072, 8, 76) == (K.MODE_SEGMENT, 6912)


def test_planner_choices_are_valid_plans(lib):
    # Over a grid of dense shapes: a segment plan has a length that is a multiple of 16
    # of at least 512 tokens, two segments or more, and a workspace (three state tables
    # per segment and state head, less two) under the 4 GiB cap that kda_workspace_bytes
    # reports for that length; chains that fill the 76 cluster slots stay serial.
    import time
    R = 76
    for B in (1, 2):
        for H in (1, 2, 3, 4, 8, 12, 16, 64, 128):
            for T in (512, 1000, 4096, 32768, 131072, 1 << 20, 1 << 24):
                m, sl = K.kda_plan(B, T, H, R)
                if B * H >= R:
                    assert (m, sl) == (K.MODE_SERIAL, 0), (B, H, T)
                if m == K.MODE_SERIAL:
                    assert sl == 0
                    continue
                nseg = -(-T // sl)
                ws = (3 * nseg - 2) * B * H * 128 * 128 * 4
                assert sl % 16 == 0 and sl >= 512 and nseg >= 2 and ws <= 4 << 30, (B, H, T, sl)
                assert K.kda_workspace_bytes(B, T, H, mode=K.MODE_SEGMENT, segment_len=sl) == ws
    # the candidate search stays cheap at the largest sequence the shape check allows
    t0 = time.perf_counter()
    K.kda_plan(1, 1 << 39, 1, R)
    assert time.perf_counter() - t0 < 0.5


@pytest.mark.parametrize("chains_per_cluster", [1, 2])
@pytest.mark.parametrize("T", [16384, 131072, 1 << 20])
def test_planner_keeps_serial_when_chains_fill_the_gpu(lib, chains_per_cluster, T):
    # With at least one chain per resident cluster, every segment plan needs at least
    # 3 nseg - 2 waves of segment passes against one or more serial waves: never a win.
    R = 76
    assert K.kda_plan(1, T, R * chains_per_cluster, R)[0] == K.MODE_SERIAL


def test_planner_rejects_bad_arguments(lib):
    with pytest.raises(K.KdaError):
        K.kda_plan(1, 1000, 4, 0)
    with pytest.raises(K.KdaError):
        K.kda_plan(1, 1000, 4, 76, head_dim=64)


def test_varlen_segment_workspace_bound(lib):
    # N sequences over T tokens have at most N + T / segment_len segments; three fp32
    # 128 x 128 tables per (segment, head) plus the int32 segment table.
    N, T, H, seg = 5, 1000, 3, 64
    nb = K.kda_workspace_bytes(1, T, H, mode=K.MODE_SEGMENT, segment_len=seg, num_seqs=N)
    rows = N + T // seg
    assert nb == 256 + 3 * rows * H * 128 * 128 * 4
    # a packed batch no longer than one segment runs serially
    assert K.kda_workspace_bytes(1, 64, H, mode=K.MODE_SEGMENT, segment_len=64, num_seqs=3) == 0


def _decode(lib, shape, state_dtype=0, scale=0.1, **over):
    base = dict(q=0x10000000, k=0x20000000, v=0x30000000, g=0x40000000, beta=0x50000000,
                s0=None, fin=None, out=0x60000000)
    base.update(over)
    P = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return lib.kda_decode(ctypes.byref(shape), P(base["q"]), P(base["k"]), P(base["v"]),
                          P(base["g"]), P(base["beta"]), ctypes.c_float(scale), P(base["s0"]),
                          P(base["fin"]), int(state_dtype), P(base["out"]), None)


def test_decode_validation(lib):
    s = KdaShape(8, 1, 0, 4, 128)
    assert _decode(lib, s, state_dtype=2) == INVALID
    assert _decode(lib, s, state_dtype=-1) == INVALID
    assert _decode(lib, KdaShape(8, 1, 0, 4, 64)) == INVALID
    assert _decode(lib, s, q=None) == INVALID
    assert _decode(lib, s, s0=0x70000008) == INVALID                 # not 16-byte aligned
    assert _decode(lib, s, scale=float("nan")) == INVALID
    # out inside q; final state inside an input
    assert _decode(lib, s, out=0x10000000 + 64) == ALIAS
    assert _decode(lib, s, fin=0x20000000) == ALIAS
    # a bf16 state is half the bytes: states 32 KiB apart are disjoint in bf16 only
    st16 = 8 * 4 * 128 * 128 * 2
    assert _decode(lib, s, state_dtype=1, s0=0x70000000, fin=0x70000000 + st16) not in (INVALID, ALIAS)
    assert _decode(lib, s, state_dtype=0, s0=0x70000000, fin=0x70000000 + st16) == ALIAS
    # exact in-place alias is accepted (without a GPU the next step fails in CUDA)
    assert _decode(lib, s, state_dtype=1, s0=0x70000000, fin=0x70000000) not in (INVALID, ALIAS)


def test_decode_binding_checks_state_dtype():
    q = torch.zeros(2, 3, 128, dtype=torch.bfloat16)
    g = torch.zeros(2, 3, 128, dtype=torch.float32)
    b = torch.zeros(2, 3, dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # CPU tensors are refused before any library call
        K.kda_decode(q, q, q, g, b, initial_state=torch.zeros(2, 3, 128, 128))


def test_grouped_head_rules(lib):
    # num_q_heads must divide num_heads or be a multiple of it
    assert _call(lib, KdaShape(1, 16, 0, 6, 128, 4)) == INVALID
    assert _call(lib, KdaShape(1, 16, 0, 4, 128, -2)) == INVALID
    assert _call(lib, KdaShape(1, 16, 0, 6, 128, 3)) not in (INVALID, ALIAS)
    assert _call(lib, KdaShape(1, 16, 0, 2, 128, 8)) not in (INVALID, ALIAS)
    # segment mode takes grouped heads too
    assert _call(lib, KdaShape(1, 16, 0, 2, 128, 8), opts=KdaOptions(1, 64, 0, 0, 0)) not in (INVALID, ALIAS)
    # sizes follow the head counts: q of 8 heads is 32 KiB at T = 16
    assert _call(lib, KdaShape(1, 16, 0, 2, 128, 8), out=0x10000000 + 16 * 1024) == ALIAS
    assert _call(lib, KdaShape(1, 16, 0, 2, 128, 8), out=0x10000000 + 32 * 1024) not in (INVALID, ALIAS)
    # the output has max(Hq, H) heads
    assert _call(lib, KdaShape(1, 16, 0, 8, 128, 2), out=0x60000000,
                 v=0x60000000 + 16 * 8 * 256 - 16) == ALIAS


def test_grouped_planner(lib):
    """Summary passes run one chain per state head, the output pass one per output head:
    grouped value heads plan like their state heads; grouped query heads see cheaper
    summaries than equal heads of the same output count."""
    R = 76
    assert K.kda_plan(1, 131072, 4, R, num_q_heads=2) == K.kda_plan(1, 131072, 4, R)
    m, s = K.kda_plan(1, 131072, 2, R, num_q_heads=8)
    assert m == K.MODE_SEGMENT and s % 16 == 0
    assert K.kda_plan(1, 131072, 64, R, num_q_heads=16) == (K.MODE_SERIAL, 0)
    # workspace: three state tables per (segment, state head)
    nb = K.kda_workspace_bytes(1, 4096, 2, mode=K.MODE_SEGMENT, segment_len=1024, num_q_heads=8)
    assert nb == (3 * 4 - 2) * 2 * 128 * 128 * 4


def test_host_pieces_range_checked_before_device_work(lib):
    # the host entry validates its options before it touches a device or a buffer
    s = KdaShape(1, 16, 0, 2, 128)
    P = ctypes.c_void_p
    for bad in (-1, 65):
        st = lib.kda_prefill_host(ctypes.byref(s), P(0x1000), P(0x2000), P(0x3000), P(0x4000),
                                  P(0x5000), ctypes.c_float(0.1), None, None, P(0x6000), None,
                                  None, ctypes.byref(KdaOptions(0, 0, 0, 0, bad)))
        assert st == INVALID and b"host_pieces" in lib.kda_last_error_message()


def test_binding_refuses_short_outputs():
    # a caller-supplied output smaller than what the library writes is refused before the
    # call (the ABI sees only a pointer); here q has 2 heads and v 6, so out has 6
    q = torch.zeros(16, 2, 128, dtype=torch.bfloat16)
    v = torch.zeros(16, 6, 128, dtype=torch.bfloat16)
    g = torch.zeros(16, 6, 128, dtype=torch.float32)
    b = torch.zeros(16, 6, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        K.kda_prefill_host(q, q, v, g, b, out=torch.zeros(16, 2, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        K.kda_prefill_host(q, q, v, g, b, final_state=torch.zeros(1, 2, 128, 128))


def test_varlen_planner(lib):
    """kda_plan_varlen: equal-length batches get the dense plan; many or short sequences
    stay serial; a few long ones are split; malformed offsets are refused."""
    from chunked_kda_delta_gb300.inputs import varlen_h12_lengths
    R = 76
    for T, H in [(131072, 4), (65536, 2), (8192, 12), (32768, 3)]:
        assert K.kda_plan_varlen([T], H, R) == K.kda_plan(1, T, H, R)
    assert K.kda_plan_varlen([65536, 65536], 4, R) == K.kda_plan(2, 65536, 4, R)
    assert K.kda_plan_varlen(varlen_h12_lengths(3), 12, R) == (K.MODE_SERIAL, 0)
    assert K.kda_plan_varlen([512] * 32, 12, R) == (K.MODE_SERIAL, 0)
    assert K.kda_plan_varlen([100, 0, 37], 4, R) == (K.MODE_SERIAL, 0)
    m, s = K.kda_plan_varlen([20000, 20000], 2, R)
    assert m == K.MODE_SEGMENT and s % 16 == 0 and 512 <= s < 20000
    shape = KdaShape(1, 40, 2, 2, 128)
    mode, seg = ctypes.c_int32(0), ctypes.c_int32(0)
    for bad in ([0, 30, 20], [1, 20, 40], [0, 20, 41]):
        cu = (ctypes.c_int32 * 3)(*bad)
        assert lib.kda_plan_varlen(ctypes.byref(shape), ctypes.cast(cu, ctypes.c_void_p), R,
                                   ctypes.byref(mode), ctypes.byref(seg)) == INVALID
    assert lib.kda_plan_varlen(ctypes.byref(shape), None, R, ctypes.byref(mode), ctypes.byref(seg)) == INVALID
