"""Seeded random configurations of the prefill against the fp64 oracle.

Each case draws (from its own seed) the sequence count and lengths (empty, one-token,
ragged and multi-chunk sequences, dense or packed), the head counts (equal or grouped in
either direction), the mode (serial, segment with a random segment length, AUTO), the
initial state (none, fp32, bf16), whether a final state is written, and the gates
(configured, slow decay, or strong decay on a random set of channels).  Every element of
the output and of the final state is held to the oracle at atol = rtol = 1e-2 (flashinfer
PR #4351 "Correctness"); bf16 final states are compared after the same rounding of the
oracle's.  The draws cover combinations the targeted tests do not enumerate.
"""
import numpy as np
import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.inputs import custom, make_inputs, to_bf16_rne

from kda_testutil import assert_close, gpu_out_heads, gpu_state_heads, oracle_grouped

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    K.load_library()


def _draw(seed):
    r = np.random.Generator(np.random.PCG64(seed))
    n = int(r.integers(1, 6))
    dense = bool(r.integers(0, 2))
    if dense:
        lens = [int(r.integers(1, 160))] * n
    else:
        lens = [int(x) for x in r.choice([0, 1, 15, 16, 17, 31, 33, 64, 100, 150], size=n)]
        if sum(lens) == 0:
            lens[0] = 40
    H = int(r.choice([1, 2, 3, 4, 6]))
    g = int(r.choice([1, 1, 2, 3]))
    Hq = H if g == 1 else (H * g if r.integers(0, 2) else H)
    if Hq == H and g > 1 and H % g == 0:
        Hq = H // g
    mode = str(r.choice(["serial", "segment", "auto"]))
    seg = int(r.choice([16, 32, 48, 64, 96]))
    s0 = str(r.choice(["none", "fp32", "bf16"]))
    fin = bool(r.integers(0, 2)) or s0 != "none"
    gates = str(r.choice(["configured", "slow", "strong"]))
    return dict(lens=lens, dense=dense, H=H, Hq=Hq, mode=mode, seg=seg, s0=s0, fin=fin, gates=gates,
                strong_frac=float(r.uniform(0.05, 0.6)), seed=seed)


@pytest.mark.parametrize("seed", list(range(5000, 5016)))
def test_random_configuration_matches_oracle(seed):
    c = _draw(seed)
    w = custom(c["lens"], c["H"], c["s0"] != "none", seed=seed, dense=c["dense"], num_q_heads=c["Hq"])
    inp = make_inputs(w, DEV, stress=c["gates"] == "slow")
    if c["gates"] == "strong":
        gen = torch.Generator(device=DEV).manual_seed(seed)
        pick = torch.rand(128, generator=gen, device=DEV) < c["strong_frac"]
        inp["g"] = torch.where(pick, torch.full_like(inp["g"], -30.0), inp["g"]).contiguous()
    if c["s0"] == "bf16":
        inp["initial_state"] = to_bf16_rne(inp["initial_state"])
    mode = {"serial": K.MODE_SERIAL, "segment": K.MODE_SEGMENT, "auto": K.MODE_AUTO}[c["mode"]]
    H, Ho = c["H"], max(c["H"], c["Hq"])
    kw = dict(initial_state=inp["initial_state"], output_final_state=c["fin"], mode=mode,
              segment_len=c["seg"] if c["mode"] == "segment" else 0)
    if c["dense"]:
        B, T = len(c["lens"]), c["lens"][0]
        q = inp["q"].view(B, T, c["Hq"], 128)
        k = inp["k"].view(B, T, min(c["Hq"], H), 128)
        v, g = (inp[x].view(B, T, H, 128) for x in ("v", "g"))
        out, fin = K.kda_prefill(q, k, v, g, inp["beta"].view(B, T, H), inp["scale"], **kw)
    else:
        out, fin = K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                 cu_seqlens=inp["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0, c
    o_ref, f_ref = oracle_grouped(inp)
    assert_close(gpu_out_heads(out, range(Ho)), o_ref, f"out {c}")
    if c["fin"]:
        if c["s0"] == "bf16":
            assert fin.dtype == torch.bfloat16
            f_ref = torch.from_numpy(f_ref).to(torch.float32).to(torch.bfloat16).double().numpy()
        assert_close(gpu_state_heads(fin, range(H)), f_ref, f"final state {c}")
