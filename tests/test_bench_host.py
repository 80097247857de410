"""Host-side bench.py logic: algorithmic bytes, the L2-flush rule and the pages' GB300
baselines (no GPU)."""
import argparse

import pytest

import bench
from chunked_kda_delta_gb300.inputs import WORKLOADS, custom


def test_algorithmic_bytes_equal_heads():
    # T = 8192, H = 64: 1538 B per head-token + S0 read + final state written (64 KiB each)
    w = WORKLOADS["single_t8192_h64"]
    assert bench.algorithmic_bytes(w) == 1538 * 8192 * 64 + 2 * 64 * 65536
    # no initial state: only the final state is written
    w0 = WORKLOADS["long_t131072_h64"]
    assert bench.algorithmic_bytes(w0) == 1538 * 131072 * 64 + 64 * 65536


def test_algorithmic_bytes_grouped_and_bf16_state():
    # 16 q/k heads, 64 state heads: q, k 256 B per q/k head; v 256, g 512, beta 2 per state
    # head; out 256 per output head (64)
    w = WORKLOADS["gva_t8192_q16_v64"]
    per_token = 256 * 16 * 2 + 64 * (256 + 512 + 2) + 64 * 256
    assert bench.algorithmic_bytes(w) == per_token * 8192 + 2 * 64 * 65536
    w2 = WORKLOADS["gqa_t8192_q64_v16"]
    per_token2 = 256 * 64 + 256 * 16 + 16 * (256 + 512 + 2) + 64 * 256
    assert bench.algorithmic_bytes(w2) == per_token2 * 8192 + 2 * 16 * 65536
    d = WORKLOADS["decode_b256_h64"]
    assert bench.algorithmic_bytes(d, state_elem=2) == 1538 * 256 * 64 + 2 * 256 * 64 * 32768


def test_l2_flush_rule():
    assert not bench.needs_l2_flush(WORKLOADS["single_t8192_h64"])      # 815 MB
    assert not bench.needs_l2_flush(WORKLOADS["decode_b256_h64"])       # 2.2 GB
    assert bench.needs_l2_flush(WORKLOADS["h12_fixed_8192"])            # 152 MB
    assert bench.needs_l2_flush(WORKLOADS["tiny_t64_h4"])


def test_pages_baselines():
    # rates are head-tokens/s of the pages' GB300 span; only for their exact shapes
    w = WORKLOADS["h12_fixed_8192"]
    assert bench.published_head_tokens_per_s(w) == pytest.approx(8192 * 12 / 487.161e-6)
    w = WORKLOADS["h12_packed_512x32"]
    assert w.num_seqs == 32 and not w.dense and w.num_heads == 12
    assert bench.published_head_tokens_per_s(w) == pytest.approx(512 * 32 * 12 / 128.264e-6)
    assert bench.published_head_tokens_per_s(WORKLOADS["single_t8192_h64"]) is None
    assert set(bench.PAGES_GB300_US) <= set(WORKLOADS)


def test_workload_config_names_state_and_plan():
    args = argparse.Namespace(mode="serial", segment_len=0, gpus=1, state_dtype="bf16")
    cfg = bench.workload_config(WORKLOADS["decode_b256_h64"], args)
    assert cfg["state_dtype"] == "bf16" and cfg["mode"] == "decode"
    cfg = bench.workload_config(WORKLOADS["h12_mixed6"], args)
    assert cfg["pages_gb300_us"]["pr_path"] == 198.216 and "flushed" in cfg["l2"]
    cfg = bench.workload_config(custom([100], 4, True, seed=1, num_q_heads=8), args)
    assert cfg["num_q_heads"] == 8 and cfg["head_tokens_per_gpu"] == 100 * 8
