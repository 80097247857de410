"""Strong decay on the GPU: gates far below the configured ones, against the fp64 oracle.

The prefill kernel forms the in-chunk decay ratios exp(gam_r - gam_s) through a
reference row of the chunk only for channels whose cumulative log-decay varies by at
most 80 over the chunk; other channels take the exact pairwise exponentials, and their
decayed operands are formed without any factor above 1.  These cases check the exact
path, the factored path at its limit and the two mixed in one Gram, every element at
atol = rtol = 1e-2 (flashinfer PR #4351 "Correctness"):

  g = -30 per token on every channel: every channel exact;
  g = -1e4: full forgetting, each token's state is beta k v^T (the invariant the
    oracle's own pins check);
  g = -30 on every third channel, the configured gates elsewhere: both paths in one
    Gram, and channel pairs split between them;
  g = -5.3 per token: a spread of 79.5 over a 16-token chunk, the strongest decay the
    factored path takes (its factors reach e^{79.5}).

T in {33, 100} gives ragged last chunks (and segments), H = 12; serial mode and
segment mode with 32-token segments (carries through the merge).
"""
import pytest
import torch

import chunked_kda_delta_gb300 as K
from chunked_kda_delta_gb300 import build as kbuild
from chunked_kda_delta_gb300.inputs import custom, make_inputs

from kda_testutil import assert_close, gpu_out_heads, gpu_state_heads, oracle_on_heads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H = 12


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    K.load_library()


def _gates(inp, kind):
    g = inp["g"]
    if kind == "all_m30":
        return torch.full_like(g, -30.0)
    if kind == "forget":
        return torch.full_like(g, -1e4)
    if kind == "mixed":
        strong = (torch.arange(128, device=g.device) % 3) == 0
        return torch.where(strong, torch.full_like(g, -30.0), g)
    if kind == "edge":
        return torch.full_like(g, -5.3)
    raise ValueError(kind)


@pytest.mark.parametrize("mode", ["serial", "segment"])
@pytest.mark.parametrize("kind", ["all_m30", "forget", "mixed", "edge"])
@pytest.mark.parametrize("T", [33, 100])
def test_strong_decay_matches_oracle(orc, T, kind, mode):
    inp = make_inputs(custom([T], H, True, seed=900 + T), DEV)
    inp["g"] = _gates(inp, kind).contiguous()
    q, k, v, g = (inp[x].view(1, T, H, 128) for x in ("q", "k", "v", "g"))
    beta = inp["beta"].view(1, T, H)
    m = K.MODE_SERIAL if mode == "serial" else K.MODE_SEGMENT
    out, fin = K.kda_prefill(q, k, v, g, beta, inp["scale"], initial_state=inp["initial_state"],
                             output_final_state=True, mode=m, segment_len=32 if mode == "segment" else 0)
    torch.cuda.synchronize()
    assert K.kda_get_device_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    o_ref, f_ref = oracle_on_heads(orc, inp, range(H))
    assert_close(gpu_out_heads(out.reshape(-1, H, 128), range(H)), o_ref, f"{kind} {mode} out")
    assert_close(gpu_state_heads(fin, range(H)), f_ref, f"{kind} {mode} final state")
