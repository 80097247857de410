"""Seeded synthetic inputs for the KDA forward prefill.

This module holds only the input recipe -- random draws, L2 normalisation,
log-sigmoid gates and bf16 rounding -- and none of the method's arithmetic.
It serves the CUDA path and the fp64 oracle alike; neither imports the other.

Recipe (per workload): q, k ~ N(0, 1) in fp32, L2-normalised per
(token, head), then rounded to bf16 (round-to-nearest-even); v ~ N(0, 1) -> bf16;
g = logsigmoid(N(0, 1)) kept in fp32 (per-token, per-channel log-decay);
beta = sigmoid(N(0, 1)) -> bf16; scale = 1/sqrt(D); initial state (where the
workload has one) = 0.1 * N(0, 1) in fp32.  Draws come from a torch generator
seeded per workload on the requested device (Philox on CUDA, MT19937 on CPU),
so big workloads are generated on the GPU in seconds.  The variable-length
workload's sequence lengths come from a numpy PCG64 generator so they are the
same on every device.

"stress" variants keep the shapes and replace the gates by slow decay
(g = -|N(0, 0.02)|), so that a wrong carry between chunks or segments, or a
mis-wired initial state, shows in the outputs and the final state.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

D_HEAD = 128
CHUNK = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    """One input configuration: sequence lengths, heads and whether S0 is given."""

    name: str
    seq_lens: tuple          # lengths of the sequences (one per sequence)
    num_heads: int
    has_initial_state: bool
    dense: bool              # True: equal lengths, passed as [B, T, H, D] without cu_seqlens
    seed: int
    head_dim: int = D_HEAD
    decode: bool = False     # True: one decode step (kda_decode) per sequence, not a prefill
    num_q_heads: int = 0     # heads of q (0: num_heads); k has min(Hq, H), out max(Hq, H)

    @property
    def q_heads(self) -> int:
        return self.num_q_heads or self.num_heads

    @property
    def k_heads(self) -> int:
        return min(self.q_heads, self.num_heads)

    @property
    def out_heads(self) -> int:
        return max(self.q_heads, self.num_heads)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_lens))

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def head_tokens(self) -> int:
        """Tokens x output heads: the units of work of a step."""
        return self.total_tokens * self.out_heads


def varlen_h12_lengths(seed: int = 3) -> tuple:
    """16 lengths uniform in [1, 4096] (PCG64, seeded), then the fixed lengths 32, 3, 33."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(1, 4097, size=16).tolist()
    return tuple(int(x) for x in lens) + (32, 3, 33)


WORKLOADS = {
    "tiny_t64_h4": Workload("tiny_t64_h4", (64,), 4, False, True, 0),
    "single_t8192_h64": Workload("single_t8192_h64", (8192,), 64, True, True, 1),
    "batch4_t4096_h128": Workload("batch4_t4096_h128", (4096,) * 4, 128, True, True, 2),
    "varlen_h12": Workload("varlen_h12", varlen_h12_lengths(3), 12, False, False, 3),
    "long_t131072_h64": Workload("long_t131072_h64", (131072,), 64, False, True, 4),
    # the long-sequence distributions with few heads: too few chains to fill the GPU
    # serially, the case the segment planner exists for
    "long_t131072_h4": Workload("long_t131072_h4", (131072,), 4, False, True, 5),
    # one decode step of a batch of 256 sequences over 64 heads (a state cache of
    # 256 x 64 states: 1 GiB in fp32, larger than L2)
    "decode_b256_h64": Workload("decode_b256_h64", (1,) * 256, 64, True, True, 6, decode=True),
    # grouped heads at the single-sequence size: 16 q/k heads shared by 64 state heads,
    # and 64 query heads sharing 16 k/v/g/beta heads
    "gva_t8192_q16_v64": Workload("gva_t8192_q16_v64", (8192,), 64, True, True, 7,
                                  num_q_heads=16),
    "gqa_t8192_q64_v16": Workload("gqa_t8192_q64_v16", (8192,), 16, True, True, 8,
                                  num_q_heads=64),
}

# The six H = 12 shapes timed on GB300 in flashinfer PR #4351 ("fix(cake_kda): support
# non-aligned recurrent prefill head counts", Performance table): packed and mixed lists
# are packed varlen batches, fixed shapes single dense sequences; no initial state, final
# state returned (the PR's correctness runs compare output and complete final state).
PAGES_H12 = {
    "h12_packed_512x32": (512,) * 32,
    "h12_packed_128x8": (128,) * 8,
    "h12_fixed_512": (512,),
    "h12_fixed_8192": (8192,),
    "h12_mixed6": (1300, 547, 2048, 963, 271, 3063),
    "h12_uniform_1024x8": (1024,) * 8,
}
for _i, (_name, _lens) in enumerate(PAGES_H12.items()):
    WORKLOADS[_name] = Workload(_name, _lens, 12, False, len(_lens) == 1, 20 + _i)


def custom(seq_lens: Sequence[int], num_heads: int, has_initial_state: bool, seed: int,
           dense: Optional[bool] = None, name: str = "custom", num_q_heads: int = 0) -> Workload:
    lens = tuple(int(x) for x in seq_lens)
    if dense is None:
        dense = len(set(lens)) == 1 and len(lens) >= 1 and lens[0] > 0
    return Workload(name, lens, int(num_heads), bool(has_initial_state), bool(dense), int(seed),
                    num_q_heads=int(num_q_heads))


def to_bf16_rne(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16 with round-to-nearest-even (torch's conversion rounds that way)."""
    return x.to(torch.float32).to(torch.bfloat16)


def make_inputs(w: Workload, device="cpu", stress: bool = False) -> dict:
    """Draw the inputs of workload ``w`` on ``device``.

    Returns a dict with q, k, v (bf16 [T, H, D]; with grouped heads q has Hq heads and
    k min(Hq, H)), g (fp32 [T, H, D]), beta (bf16 [T, H]), initial_state (fp32 [N, H, D, D]
    or None),
    cu_seqlens (int32 [N + 1] on ``device``; always present), seq_lens,
    scale (float) and the workload itself.
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(w.seed) * 1000003 + (17 if stress else 0))
    T, H, D = w.total_tokens, w.num_heads, w.head_dim
    N = w.num_seqs

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32)

    def unit(x):
        n = torch.linalg.vector_norm(x, dim=-1, keepdim=True)
        return x / torch.clamp(n, min=1e-30)

    q = to_bf16_rne(unit(randn(T, w.q_heads, D)))
    k = to_bf16_rne(unit(randn(T, w.k_heads, D)))
    v = to_bf16_rne(randn(T, H, D))
    if stress:
        g = -torch.abs(randn(T, H, D) * 0.02)
    else:
        g = torch.nn.functional.logsigmoid(randn(T, H, D))
    beta = to_bf16_rne(torch.sigmoid(randn(T, H)))
    s0 = (randn(N, H, D, D) * 0.1) if w.has_initial_state else None
    cu = torch.tensor([0] + list(np.cumsum(w.seq_lens)), dtype=torch.int32, device=dev)
    return dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta, initial_state=s0, cu_seqlens=cu,
                seq_lens=tuple(w.seq_lens), scale=1.0 / math.sqrt(D), workload=w)


def to_f64_numpy(t: Optional[torch.Tensor]):
    """Exact upcast of a bf16/fp32 tensor to a float64 numpy array (None stays None)."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
