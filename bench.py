#!/usr/bin/env python
"""Benchmark of the KDA forward prefill on GB300: one JSON line on rank 0.

A step is one pass of the whole hot path (one ``kda_prefill`` call: K1 + K2 over
every chunk of every (sequence, head), output and final state) over the
workload's synthetic inputs, which are resident in HBM before timing starts.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--mode serial|segment] [--impl ours|reference]

Multi-GPU (launched by torchrun, one rank per GPU): every rank runs its own
independent copy of the workload (independent problems, no data-path
collective, weak scaling); the timed region is bracketed by a barrier and a
device synchronize, the time is the max over ranks, and ``value`` counts the
head-tokens of all ranks.  ``--impl reference`` times the fp64 CPU oracle (the
only reference there is) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill head-tokens/s (T·H/s) and % of roofline on 1 GB300"
UNIT = "head-tokens/s"
FALLBACK_HBM_GBS = 6800.0
BYTES_PER_HEAD_TOKEN = 3 * 256 + 512 + 2 + 256   # q, k, v bf16 + g fp32 + beta + out
STATE_BYTES = 128 * 128 * 4
# Tensor-core operands are bf16 (fp32 accumulation); the state, decays and the WY
# solve are fp32.
COMPUTE_DTYPE = "bf16"
_FWD_SOURCES = ["chunked_kda_delta_gb300/csrc/kda_fwd_tc.cu",
                "chunked_kda_delta_gb300/csrc/kda_ptx.cuh",
                "chunked_kda_delta_gb300/csrc/kda_internal.cuh"]
_DECODE_SOURCES = ["chunked_kda_delta_gb300/csrc/kda_decode.cu",
                   "chunked_kda_delta_gb300/csrc/kda_internal.cuh"]
KERNEL_SOURCES = {"serial": _FWD_SOURCES,
                  "segment": _FWD_SOURCES + ["chunked_kda_delta_gb300/csrc/kda_merge.cu"],
                  "auto": _FWD_SOURCES + ["chunked_kda_delta_gb300/csrc/kda_merge.cu"],
                  "decode_fp32": _DECODE_SOURCES, "decode_bf16": _DECODE_SOURCES}
KERNEL_NAMES = {"serial": "kda_fwd_tc_kernel",
                "segment": "kda_fwd_tc_kernel x3 + kda_merge_kernel (whole step)",
                "auto": "the plan the library picks (whole step)",
                "decode_fp32": "kda_decode_kernel<float>",
                "decode_bf16": "kda_decode_kernel<bf16>"}
LAUNCHES_PER_STEP = {"serial": 1, "segment": 4, "auto": 1, "decode_fp32": 1, "decode_bf16": 1}
DECODE_METRIC = "decode head-tokens/s (B·H/s) and % of roofline on 1 GB300"
L2_BYTES = 129 * 1000 * 1000
# GB300 kernel spans the pages publish for six H = 12 prefill shapes (flashinfer PR #4351
# "fix(cake_kda): support non-aligned recurrent prefill head counts", Performance table:
# the PR's path, and the official FlashKDA build; strict CUPTI span, cold L2, no CUDA
# graph), in microseconds.
PAGES_GB300_US = {
    "h12_packed_512x32": (128.264, 233.496),
    "h12_packed_128x8": (25.712, 52.904),
    "h12_fixed_512": (47.712, 82.240),
    "h12_fixed_8192": (487.161, 779.426),
    "h12_mixed6": (198.216, 340.913),
    "h12_uniform_1024x8": (78.440, 162.505),
}


def needs_l2_flush(w, state_elem: int = 4) -> bool:
    """Inputs that fit in L2 get it flushed before every timed step (as the pages time
    their H = 12 shapes: cold L2); larger inputs evict it by themselves."""
    return algorithmic_bytes(w, state_elem) < 4 * L2_BYTES


def published_head_tokens_per_s(w):
    """The pages' GB300 rate for this exact workload, head-tokens/s, or None."""
    if w.name not in PAGES_GB300_US:
        return None
    return w.head_tokens / (PAGES_GB300_US[w.name][0] * 1e-6)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="single_t8192_h64")
    ap.add_argument("--mode", choices=["serial", "segment", "auto"], default="serial")
    ap.add_argument("--segment-len", type=int, default=0)
    ap.add_argument("--state-dtype", choices=["fp32", "bf16"], default="fp32",
                    help="state storage of a decode workload")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def algorithmic_bytes(w, state_elem: int = 4) -> int:
    """Bytes a step must move: every input once, the output once, the states once each
    way.  Per token: q and k rows of their own head counts, v, g and beta per state head,
    out per output head (equal heads: BYTES_PER_HEAD_TOKEN per head)."""
    states = (1 if w.has_initial_state else 0) + 1   # read S0 (if given) + write final
    state_bytes = STATE_BYTES // 4 * state_elem
    per_token = 256 * (w.q_heads + w.k_heads + w.num_heads + w.out_heads) + 514 * w.num_heads
    return per_token * w.total_tokens + state_bytes * w.num_seqs * w.num_heads * states


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("hbm_gbs", "hbm_GBps", "hbm"):
                if key in d and d[key]:
                    return float(d[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++ source without comments, whitespace runs collapsed (the sources hold no
    comment markers inside string literals): comment edits keep the hash."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", " ", text).strip()


def source_hash(mode: str, read=None) -> str:
    """Hash of the code (not the comments) of the kernel sources a mode runs."""
    read = read or (lambda rel: open(os.path.join(ROOT, rel)).read())
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(mode, []):
        h.update(_code_only(read(rel)).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, mode: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current source."""
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(path).read()
        m_w = re.search(r"^workload:\s*(\S+)", text, re.M)
        m_k = re.search(r"^source_sha256:\s*(\S+)", text, re.M)
        m_t = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        m_m = re.search(r"^mode:\s*(\S+)", text, re.M)
        if m_w and m_k and m_t and m_w.group(1) == workload and \
                (m_m is None or m_m.group(1) == mode) and m_k.group(1) == source_hash(mode):
            return float(m_t.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.t0 = self.t1 = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        deadline = time.time() + 5
        while not self.samples and time.time() < deadline and self.proc.poll() is None:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        time.sleep(0.12)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return None
        inside = [s for t, s in self.samples if self.t0 and self.t0 - 0.06 <= t <= self.t1 + 0.06]
        rows = inside or [s for _, s in self.samples][-3:]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if len(r) > 1 and num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if len(r) > 2 and num(r[2]) is not None]
        reasons = set()
        for r in rows:
            for i, name in enumerate(self.NAMES):
                if len(r) > 5 + i and r[5 + i].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples_in_timed_region": len(inside)}


def gpu_identifier(torch, dev) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev.index or 0] if vis else str(dev.index or 0)


def device_inputs(K, w, dev):
    from chunked_kda_delta_gb300.inputs import make_inputs
    inp = make_inputs(w, dev)
    args = dict(q=inp["q"], k=inp["k"], v=inp["v"], g=inp["g"], beta=inp["beta"])
    if w.dense:
        B, T = w.num_seqs, w.seq_lens[0]
        for key in ("q", "k", "v", "g"):
            args[key] = args[key].view(B, T, args[key].shape[1], 128)
        args["beta"] = args["beta"].view(B, T, w.num_heads)
        cu = None
    else:
        cu = inp["cu_seqlens"]
    return inp, args, cu


def oracle_head_args(w, inp, out_heads, rows=None):
    """fp64 oracle inputs for the given OUTPUT heads (each run as a plain head on the q, k
    and state heads it reads), restricted to token rows `rows` if given."""
    import oracle
    from chunked_kda_delta_gb300.inputs import to_f64_numpy
    maps = [oracle.grouped_heads(ho, w.num_heads, w.q_heads) for ho in out_heads]
    pick = {"q": [m[0] for m in maps], "k": [m[1] for m in maps]}
    sx = [m[2] for m in maps]
    d = {}
    for key in ("q", "k", "v", "g", "beta"):
        t = inp[key] if rows is None else inp[key][rows]
        d[key] = to_f64_numpy(t[:, pick.get(key, sx)])
    s0 = None if inp["initial_state"] is None else to_f64_numpy(inp["initial_state"][:, sx])
    return d, s0


def cpu_baseline(w, inp, seconds: float):
    """The fp64 oracle on the host cores, over a bounded sample of the workload's heads."""
    import oracle
    lib = oracle.default()
    cores = lib.max_threads()
    cu = inp["cu_seqlens"].cpu().numpy().astype("int64")
    # Heads in groups of `cores`, cycling through the workload again when one pass is
    # short (a decode step takes well under a second), until `seconds`, or 3 s after at
    # least one full pass.
    done_heads, head_tokens, elapsed = 0, 0, 0.0
    while elapsed < seconds and (done_heads < w.out_heads or elapsed < min(3.0, seconds)):
        h0 = done_heads % w.out_heads
        hs = list(range(h0, min(w.out_heads, h0 + cores)))
        sel, s0 = oracle_head_args(w, inp, hs)
        t = time.perf_counter()
        lib.recurrent(sel["q"], sel["k"], sel["v"], sel["g"], sel["beta"], inp["scale"], s0=s0,
                      cu_seqlens=cu)
        elapsed += time.perf_counter() - t
        done_heads += len(hs)
        head_tokens += w.total_tokens * len(hs)
    what = (f"{done_heads} of {w.out_heads} heads" if done_heads <= w.out_heads else
            f"{done_heads / w.out_heads:.1f} passes over all {w.out_heads} heads")
    return {"value": head_tokens / elapsed, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{what} x all {w.total_tokens} tokens "
                      f"(fp64 token-by-token recurrence, {elapsed:.1f} s)"}


def run_reference(args, w):
    """Reference arm: the fp64 CPU oracle as it stands, on bounded samples of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from chunked_kda_delta_gb300.inputs import make_inputs
    lib = oracle.default()
    cores = lib.max_threads()
    # Inputs for a prefix of every head (the recurrence cost is the same for every token).
    budget = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    probe_tokens = min(w.seq_lens[0] if w.seq_lens[0] > 0 else 1, 256)
    inp = make_inputs(w, "cpu")
    hs = list(range(min(w.out_heads, cores)))
    def sample(tokens):
        lens = []
        left = tokens
        for L in w.seq_lens:
            take = min(L, left)
            lens.append(take)
            left -= take
        idx = np.concatenate([np.arange(c, c + t) for c, t in
                              zip(np.cumsum([0] + list(w.seq_lens[:-1])), lens)])
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        d, s0 = oracle_head_args(w, inp, hs, rows=idx)
        return d, s0, cu, sum(lens)
    d, s0, cu, nt = sample(probe_tokens)
    t = time.perf_counter()
    lib.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], s0=s0, cu_seqlens=cu)
    per_token = (time.perf_counter() - t) / max(1, nt)
    tokens = int(max(1, min(w.total_tokens, budget / max(per_token, 1e-9))))
    d, s0, cu, nt = sample(tokens)
    def step():
        lib.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], inp["scale"], s0=s0,
                      cu_seqlens=cu)
    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    total = time.perf_counter() - t
    ht = nt * len(hs)
    value = ht * args.steps / total
    desc = (f"{len(hs)} of {w.out_heads} heads x first {nt} of {w.total_tokens} tokens per step "
            f"(fp64 token-by-token recurrence)")
    print(json.dumps({
        "impl": "reference", "metric": DECODE_METRIC if w.decode else METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args, note="CPU oracle on a bounded sample per step"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings (identity without a process group)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(world: int, head_tokens_per_rank: int, steps: int, seconds: float) -> float:
    """Whole-job head-tokens/s: every rank runs its own copy of the workload (weak scaling)."""
    return world * head_tokens_per_rank * steps / seconds


def kind_of(w, args) -> str:
    """The kernel set a run times: a prefill mode, or the decode step with its state type."""
    return f"decode_{args.state_dtype}" if w.decode else args.mode


def state_elem_of(w, args) -> int:
    return 2 if (w.decode and args.state_dtype == "bf16") else 4


def workload_config(w, args, note=None):
    cfg = {"workload": w.name, "seq_lens": (list(w.seq_lens) if len(w.seq_lens) <= 4 else
                                            f"{w.num_seqs} sequences, {w.total_tokens} tokens"),
           "num_heads": w.num_heads, "num_q_heads": w.q_heads, "head_dim": 128, "chunk": 16,
           "initial_state": w.has_initial_state, "final_state": True, "mode": args.mode,
           "segment_len": ((args.segment_len or 8192) if args.mode == "segment" else
                           (getattr(args, "planned", ("serial", 0))[1] or None) if args.mode == "auto"
                           else None),
           "plan": getattr(args, "planned", [args.mode])[0],
           "precision": "bf16 tensor-core operands, fp32 accumulation, fp32 state",
           "head_tokens_per_gpu": w.head_tokens, "parallelism": f"replicas x{args.gpus}",
           "l2": ("flushed before every step (512 MB write, outside the timed kernel); value "
                  "from kernel time only" if needs_l2_flush(w, state_elem_of(w, args)) else
                  "no flush; inputs larger than L2 "
                  f"({algorithmic_bytes(w, state_elem_of(w, args)) / 1e6:.0f} MB per step vs 129 MB)")}
    if w.name in PAGES_GB300_US:
        cfg["pages_gb300_us"] = {"pr_path": PAGES_GB300_US[w.name][0],
                                 "flashkda": PAGES_GB300_US[w.name][1],
                                 "source": "flashinfer PR #4351 Performance table (GB300, cold L2)"}
    if w.decode:
        cfg.update(mode="decode", segment_len=None, plan="decode",
                   state_dtype=args.state_dtype, step="one decode token per sequence, "
                   "state cache updated in place",
                   precision=f"fp32 CUDA-core arithmetic, {args.state_dtype} state storage")
    if note:
        cfg["note"] = note
    return cfg


def main():
    args = parse_args()
    from chunked_kda_delta_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return
    import torch
    import chunked_kda_delta_gb300 as K
    from chunked_kda_delta_gb300 import build as kbuild

    rank, world, local = dist_env()
    kbuild.build()
    K.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    mode = {"serial": K.MODE_SERIAL, "segment": K.MODE_SEGMENT, "auto": K.MODE_AUTO}[args.mode]
    if args.mode == "auto" and not w.decode:
        # what the library will pick (its resident-cluster count is the occupancy query;
        # one cluster per SM pair is the same on this part)
        props = torch.cuda.get_device_properties(dev)
        pm, ps = K.kda_plan(w.num_seqs if w.dense else 1, w.seq_lens[0] if w.dense else w.total_tokens,
                            w.num_heads, max(1, props.multi_processor_count // 2),
                            varlen=not w.dense, num_seqs=0 if w.dense else w.num_seqs)
        args.planned = ("segment", ps) if pm == K.MODE_SEGMENT else ("serial", 0)
    kind = kind_of(w, args)
    inp, a, cu = device_inputs(K, w, dev)
    N = w.num_seqs
    out = torch.empty(tuple(a["q"].shape[:-2]) + (w.out_heads, 128), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((N, w.num_heads, 128, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    if w.decode:
        # a state cache resident in HBM, advanced in place by one token per sequence
        cache = inp["initial_state"].to(torch.bfloat16 if args.state_dtype == "bf16"
                                        else torch.float32)

        def step():
            K.kda_decode(**a, scale=inp["scale"], initial_state=cache, final_state=cache,
                         out=out, stream=stream)
    else:
        def step():
            K.kda_prefill(**a, scale=inp["scale"], initial_state=inp["initial_state"],
                          cu_seqlens=cu, out=out, final_state=fin, stream=stream, mode=mode,
                          segment_len=args.segment_len)

    clocks = ClockSampler(gpu_identifier(torch, dev))
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if K.kda_get_device_status() != 0:
        raise RuntimeError("device status error after warm-up")
    launches_per_step = LAUNCHES_PER_STEP.get(kind, 1)
    if args.mode == "auto" and not w.decode:
        launches_per_step = 4 if args.planned[0] == "segment" else 1
    if args.mode == "segment" and not w.decode:
        seg = args.segment_len or 8192
        if w.dense and w.seq_lens[0] <= seg:
            launches_per_step = 1  # a single segment runs the plain serial pass
    flush = (torch.empty(128 * 1024 * 1024, dtype=torch.int32, device=dev)
             if needs_l2_flush(w, state_elem_of(w, args)) else None)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    if pg:
        pg.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    kernel_ms = statistics.mean(s.elapsed_time(e) for s, e in evs)
    if K.kda_get_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    elapsed_ms, kernel_ms = max_over_ranks([elapsed_ms, kernel_ms], pg, dev)
    if flush is not None:
        # the timed work is the kernels alone; the flushes between them are not
        elapsed_ms = max_over_ranks([sum(s.elapsed_time(e) for s, e in evs)], pg, dev)[0]
    value = job_throughput(world, w.head_tokens, args.steps, elapsed_ms / 1e3)

    e2e = None
    if not args.no_e2e and w.decode:
        # the token inputs come from pinned host memory and the outputs go back every
        # step; the state cache stays resident on the device, as decoding keeps it
        host = {k: a[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def e2e_step():
            for key, x in host.items():
                a[key].copy_(x, non_blocking=True)
            K.kda_decode(**a, scale=inp["scale"], initial_state=cache, final_state=cache,
                         out=out, stream=stream)
            oh.copy_(out, non_blocking=True)
            stream.synchronize()
        e2e_step()
        if pg:
            pg.barrier()
        t = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        e2e_s = (time.perf_counter() - t) / args.e2e_steps
        e2e_s = max_over_ranks([e2e_s], pg, dev)[0]
        h2d = sum(x.numel() * x.element_size() for x in host.values())
        e2e = {"value": job_throughput(world, w.head_tokens, 1, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": oh.numel() * 2,
               "ms_per_step": e2e_s * 1e3,
               "note": "torch copies + kda_decode; the state cache stays on the device"}
    elif not args.no_e2e:
        host = {k: inp[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
        s0h = None if inp["initial_state"] is None else inp["initial_state"].cpu().pin_memory()
        cuh = None if cu is None else cu.cpu()
        if w.dense:
            B, T = w.num_seqs, w.seq_lens[0]
            for key in ("q", "k", "v", "g"):
                host[key] = host[key].view(B, T, host[key].shape[1], 128)
            host["beta"] = host["beta"].view(B, T, w.num_heads)
        oh = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
        fh = torch.empty((N, w.num_heads, 128, 128), dtype=torch.float32).pin_memory()

        def e2e_step():
            K.kda_prefill_host(**host, scale=inp["scale"], initial_state=s0h, cu_seqlens=cuh,
                               out=oh, final_state=fh, mode=mode, segment_len=args.segment_len)
        e2e_step()
        if pg:
            pg.barrier()
        t = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        e2e_s = (time.perf_counter() - t) / args.e2e_steps
        e2e_s = max_over_ranks([e2e_s], pg, dev)[0]
        h2d = sum(x.numel() * x.element_size() for x in host.values())
        h2d += 0 if s0h is None else s0h.numel() * 4
        h2d += 0 if cuh is None else cuh.numel() * 4
        d2h = oh.numel() * 2 + fh.numel() * 4
        e2e = {"value": job_throughput(world, w.head_tokens, 1, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, args.cpu_seconds)

    if rank == 0:
        peak, peak_kind = measured_peaks()
        algo = algorithmic_bytes(w, state_elem_of(w, args))
        achieved = algo / (kernel_ms / 1e3) / 1e9
        traffic = recorded_traffic(w.name, kind)
        line = {
            "metric": DECODE_METRIC if w.decode else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": (value / published_head_tokens_per_s(w)
                            if published_head_tokens_per_s(w) else None),
            "dtype": COMPUTE_DTYPE, "data": "synthetic",
            "config": workload_config(w, args),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} HBM copy bandwidth",
                         "kernel": KERNEL_NAMES.get(kind, kind),
                         "kernel_ms": kernel_ms, "algorithmic_bytes_per_launch": algo},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line))
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
