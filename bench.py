#!/usr/bin/env python3
"""Benchmark of the paged-KV GQA attention hot path on GB300.

Metric: paged decode KV GB/s (and % of HBM peak) at 4K-32K context; q=4096 prefill
TFLOP/s.  One JSON line on stdout (rank 0); its last key, "summary", repeats every leg's
headline figure in a few hundred bytes.

Headline workload (the `value`): decode, batch 1, context 32768, 24 query / 4 KV heads,
head_dim 256, BF16 N(0,1) with 5% of K rows scaled x8, block_size 832, pages drawn at
random from a 1 GiB K+V pool (315 pages).  One step = pa_decode of one sequence: the
split-context kernel (one launch) and the LSE combine (a second launch).  KV GB/s =
4096 bytes per context token (K+V of 4 KV heads x 256 dims x 2 bytes) / step time.

Timing of the decode legs: K consecutive steps are captured in ONE CUDA graph and
replayed once between two CUDA events (a serving loop captures a whole model step, so a
graph launch is not paid per attention call); ms per step = elapsed / K.  The steps
cycle over sequences whose K/V are disjoint and together several times the 129 MB L2
(for 32K, the 7 sequences a 1 GiB pool holds: 939 MB), so no step finds its K/V in L2.
The split kernel's own time: CUDA events the library records around its launch, in
eager steps each after an L2 flush.  The same step as a single-step graph replayed
after an L2 flush is reported too (config.step_alone_ms): it carries the graph's own
launch, ~5 us here.  The end-to-end figure (e2e) is the same stream of steps through
the public API with the step's inputs copied in from pinned host memory and its output
written to pinned host memory; it is timed between two timings of the device-resident
stream (A/B/A), all in this run.

Other legs, reported under "legs": the 4K/8K/16K/32K sweep (same pool), 32K in generic
16- and 64-token pages, the serving step at 8K (new token appended: slot derived in the
kernel, KV write, decode; 32 copies of a 64-page pool) with its own e2e, block_size 784
at 8K, batched decode (16 sequences, 4K-32K, appended token), the q=4096 prefill chunk
over 4096 prior tokens (chunk KV write + prefill; TFLOP/s counts the causal work
4*D*Hq*sum_i(4096+i+1) = 6.185e11), the q=1685 tail chunk over 12288 prior tokens and
the q=4096 first chunk (no prior tokens), a mixed batch of four sequences' chunks in one
varlen call, and the decode input preparation of a two-group model.  The prefill and
input-preparation legs replay a single-step graph after an L2 flush per step (a 512 MiB
read outside the events), with CUDA events around each step and around the prefill
kernel.  cpu_baseline: the fp64 oracle on the headline workload, on all host cores and
on one.  --impl reference times that oracle on the headline workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

HEADLINE_CTX = 32768
HEADLINE = ("decode batch 1, context 32768, 24 q / 4 kv heads, d=256, BF16 N(0,1) with 5% of "
            "K rows x8, block_size 832, pages drawn at random from a 1 GiB K+V pool")
KV_BYTES_PER_TOKEN = 2 * workloads.HKV * workloads.HEAD_DIM * 2   # K+V, all KV heads
L2_FLUSH_BYTES = 512 << 20
# DRAM bytes (read + write) of one split launch of the headline (32K) step in an ncu
# capture of the current split kernel (summarised under profiles/); None whenever the
# kernel changes after a capture.
SPLIT_32K_DRAM_BYTES = 134_296_576 + 3_398_144
# The same for one prefill launch of the q=4096 chunk over 4096 prior tokens.
PREFILL_Q4096_DRAM_BYTES = 86_582_528 + 18_139_904


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--legs", default="all",
                    help="comma list: sweep,small_pages,step8k,bs784,batched,prefill,"
                         "prefill_tail,prefill_first,prefill_mixed,prep or all/none; l2check "
                         "(not in all) runs the stream of 8K steps that an ncu capture of "
                         "DRAM bytes checks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="host seconds of oracle work per cpu_baseline timing (two timings)")
    ap.add_argument("--contexts", default="4096,8192,16384,32768",
                    help="contexts of the sweep leg")
    ap.add_argument("--skip-headline", action="store_true",
                    help="profiling runs only: run the selected legs without the headline")
    return ap.parse_args()


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                    source="fallback")


# ------------------------------------------------------------------------ distributed
def dist_init(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce_device():
    import torch.distributed as dist
    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def max_over_ranks(x, ws):
    """The largest x over all ranks (the slowest rank's time)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, ws):
    """The sum of x over all ranks (the work all ranks did)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 200 ms while the GPU legs run."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.proc = None
        self.path = None
        self.index = index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for ln in open(self.path):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        busy = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(busy),
                "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------------------------ timing
def time_steps(step, steps, warmup, flush):
    """Per-step device time (ms) of `step` with an L2 flush before each step."""
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_main_kernel(pa, call, steps, warmup, flush):
    """Per-launch device time (ms) of the main kernel of `call` (decode split kernel or
    prefill kernel), recorded by the library around that launch on its stream."""
    for _ in range(warmup):
        flush()
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush()
        pa.set_kernel_events(a, b)
        call()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def stream_graph(fns, steps):
    """One CUDA graph of `steps` consecutive steps, step i being fns[i % len(fns)]."""
    def run():
        for i in range(steps):
            fns[i % len(fns)]()
    return graph_of(run)


def time_stream(fns, steps, warmup, flush):
    """Device ms per step of `steps` consecutive steps replayed as ONE CUDA graph (so the
    graph's own launch is paid once, as in a serving loop that captures a whole model
    step), timed on its second replay (the first uploads the graph).  The cycled steps read disjoint inputs that together exceed L2 several times,
    so no step finds its K/V in L2.  W eager warm-up steps first, then one L2 flush: the
    decode's K/V loads are evict-first, so lines that generating the inputs left in L2 at
    normal priority would otherwise outlive the stream and be hit on every pass (an ncu
    capture saw the last-generated copy read 10-26 of its 33.5 MB from L2)."""
    for i in range(warmup):
        fns[i % len(fns)]()
    g = stream_graph(fns, steps)
    g.replay()  # the graph's first replay (uploads it) is warm-up too
    torch.cuda.synchronize()
    flush()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def graph_of(fn):
    """Capture fn (a sequence of C-ABI calls on the current stream) as a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


# ------------------------------------------------------------------------ legs
def append_step_fn(pa, case, max_seq_len=None):
    """One serving decode step of a batch: each sequence's newest token is appended (slot
    derived from the block table, KV write) and attended to, then the LSE combine."""
    msl = int(case.seq_lens.max()) if max_seq_len is None else max_seq_len
    S, hq, d = case.q.shape
    out = torch.empty_like(case.q)
    ws = torch.empty(max(256, pa.decode_workspace_size(S, hq, case.k_cache.shape[2], d,
                                                        case.block_size, msl)),
                     dtype=torch.uint8, device="cuda")
    slots = torch.empty(S, dtype=torch.int64, device="cuda")

    def step():
        pa.decode_append(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                         case.scale, msl, case.new_k, case.new_v, out=out, workspace=ws,
                         slot_mapping=slots)
    return step, out


def attn_fn(pa, case, s, max_seq_len):
    """Decode of sequence s of the case alone (batch 1), no write."""
    q, bt, sl = case.q[s:s + 1], case.block_table[s:s + 1], case.seq_lens[s:s + 1]
    out = torch.empty_like(q)
    ws = torch.empty(max(256, pa.decode_workspace_size(1, q.shape[1], case.k_cache.shape[2],
                                                        q.shape[2], case.block_size,
                                                        max_seq_len)),
                     dtype=torch.uint8, device="cuda")

    def call():
        pa.decode(q, case.k_cache, case.v_cache, bt, sl, case.scale, max_seq_len, out=out,
                  workspace=ws)
    return call


def headline_replicas(device, n=32, block_size=832, new_tokens=1):
    """n copies of the 8K workload, each its own shuffled 64-page pool (seeds 1002, 2002,
    ...): 32 x 33.5 MB of K/V read in rotation, 8x L2.  The decode prefetches each split's
    first tiles into L2 before it waits for the previous kernel; with 16 copies some of
    those lines were still in L2 when the same copy came round again (an ncu capture saw
    8% of a launch's bytes come from L2)."""
    return [workloads.paged_case(1002 + 1000 * r, [8192], block_size, 64,
                                 new_tokens=new_tokens, device=device) for r in range(n)]


def decode_leg(pa, fns, tokens, seqs, steps, warmup, flush, peaks, rotation):
    """A decode leg timed as a stream of steps (time_stream), fns cycled; each step reads
    `tokens` context tokens of `seqs` sequences.  The split kernel's time: events around
    its launch, the first copy's step run eagerly after an L2 flush."""
    step_ms = time_stream(fns, steps, warmup, flush)
    kms = time_main_kernel(pa, fns[0], steps, warmup, flush)
    nbytes = tokens * KV_BYTES_PER_TOKEN
    k_ms = statistics.mean(kms)
    r = {"context_tokens": tokens, "kv_bytes": nbytes, "ms_per_step": step_ms,
         "kv_gbs": nbytes / (step_ms * 1e-3) / 1e9,
         "split_kernel_ms": k_ms, "split_kernel_ms_min": min(kms),
         "split_kernel_ms_median": statistics.median(kms),
         "split_kernel_gbs": nbytes / (k_ms * 1e-3) / 1e9,
         "tokens_per_s": seqs / (step_ms * 1e-3), "rotation": rotation}
    r["kv_pct_of_hbm_peak"] = 100.0 * r["kv_gbs"] / peaks["hbm_gbs"]
    r["split_kernel_pct_of_hbm_peak"] = 100.0 * r["split_kernel_gbs"] / peaks["hbm_gbs"]
    return r


def causal_flops(q_len, q_start):
    """Algorithmic FLOPs of a causal chunk: QK^T and PV, 2*D each per (row, visible key)."""
    return 4.0 * workloads.HEAD_DIM * workloads.HQ * sum(q_start + i + 1 for i in range(q_len))


PREFILL_FLOPS = causal_flops(4096, 4096)


def prefill_leg(pa, steps, warmup, flush, peaks, make="prefill_chunk"):
    case = getattr(workloads, make)("cuda")
    out = torch.empty_like(case.q)
    slots = torch.empty(case.positions.numel(), dtype=torch.int64, device="cuda")
    cu = case.meta.get("cu_seqlens_q")
    hq, d, hkv, bs = case.q.shape[1], case.q.shape[2], case.k_cache.shape[2], case.block_size
    if cu is None:  # one sequence's chunk
        q_len, q_start = case.q.shape[0], case.q_start
        flops = causal_flops(q_len, q_start)
        bt0 = case.block_table[0].contiguous()
        need = pa.prefill_workspace_size(q_len, q_start, True, hq, hkv, d, bs)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

        def attn():
            pa.prefill_chunk(case.q, case.k_cache, case.v_cache, bt0, case.q_start, True,
                             case.scale, out=out, workspace=ws)
    else:  # a mixed batch of chunks
        k_lens = case.meta["seq_lens"]
        q_len = int(cu[-1])
        q_start = [L - (cu[b + 1] - cu[b]) for b, L in enumerate(k_lens)]
        flops = sum(causal_flops(cu[b + 1] - cu[b], q_start[b]) for b in range(len(k_lens)))
        need = pa.prefill_varlen_workspace_size(cu, k_lens, True, hq, hkv, d, bs)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

        def attn():
            pa.prefill_varlen(case.q, case.k_cache, case.v_cache, case.block_table, cu, k_lens,
                              True, case.scale, out=out, workspace=ws)

    def step():
        pa.slot_mapping(case.positions, case.block_table, case.block_size,
                        seq_idx=case.seq_idx, out=slots)
        pa.reshape_and_cache(case.new_k, case.new_v, case.k_cache, case.v_cache, slots)
        attn()
    g = graph_of(step)
    ms = time_steps(g.replay, steps, warmup, flush)
    kms = time_main_kernel(pa, attn, steps, warmup, flush)
    step_ms, k_ms = statistics.mean(ms), statistics.mean(kms)
    r = {"q_len": q_len, "q_start": q_start, "causal_flops": flops, "workspace_bytes": need,
         "ms_per_step": step_ms, "step_tflops": flops / (step_ms * 1e-3) / 1e12,
         "kernel_ms": k_ms, "kernel_ms_min": min(kms), "kernel_ms_median": statistics.median(kms),
         "kernel_tflops": flops / (k_ms * 1e-3) / 1e12}
    peak = peaks["bf16_tflops"]
    r["roofline"] = {"bound": "tensor", "achieved": r["kernel_tflops"], "peak": peak,
                     "unit": "TFLOP/s", "frac": r["kernel_tflops"] / peak,
                     "traffic": PREFILL_Q4096_DRAM_BYTES if make == "prefill_chunk" else None,
                     "peak_source": f"{peaks['source']} bf16 dense burst"}
    return r


def l2check_leg(pa, flush):
    """For an ncu capture of dram__bytes_read.sum per split launch (--cache-control none):
    64 consecutive 8K decode steps over 32 copies of the workload in turn (the 8K legs'
    timing), then 16 steps of one copy (L2 warm, the control).  Small pools (11 pages per
    copy) keep the device footprint under 1.5 GB."""
    reps = [workloads.paged_case(1002 + 1000 * r, [8192], 832, 11, new_tokens=1,
                                 device="cuda") for r in range(32)]
    fns = [append_step_fn(pa, c, 8192)[0] for c in reps]
    r = {"rotation_us_per_step": time_stream(fns, 64, 0, flush) * 1e3,
         "one_copy_us_per_step": time_stream(fns[:1], 16, 0, flush) * 1e3}
    del reps, fns
    torch.cuda.empty_cache()
    return r


def input_prep_leg(pa, steps, warmup, flush):
    """Decode input preparation of one sequence for a two-group model (block sizes 832 and
    16): one pa_decode_input_prep launch against one pa_slot_mapping launch per group plus
    the metadata written by torch ops (the unfused path), each replayed from a graph."""
    dev = "cuda"
    pos = torch.tensor([8191], dtype=torch.int32, device=dev)
    sampled = torch.tensor([42], dtype=torch.int32, device=dev)
    t0 = torch.arange(16, dtype=torch.int32, device=dev).reshape(1, 16)
    t1 = torch.arange(600, dtype=torch.int32, device=dev).reshape(1, 600)
    out = pa.decode_input_prep(pos, [t0, t1], [832, 16], sampled_ids=sampled)
    s0 = torch.empty(1, dtype=torch.int64, device=dev)
    s1 = torch.empty(1, dtype=torch.int64, device=dev)
    ids = torch.empty(1, dtype=torch.int32, device=dev)
    seq_lens = torch.empty(1, dtype=torch.int32, device=dev)

    def fused():
        pa.decode_input_prep(pos, [t0, t1], [832, 16], sampled_ids=sampled, out=out)

    def unfused():
        ids.copy_(sampled)
        torch.add(pos, 1, out=seq_lens)
        pa.slot_mapping(pos, t0, 832, out=s0)
        pa.slot_mapping(pos, t1, 16, out=s1)
    r = {}
    for name, fn in (("one_launch", fused), ("per_group", unfused)):
        g = graph_of(fn)
        ms = time_steps(g.replay, steps, warmup, flush)
        r[name + "_us"] = statistics.median(ms) * 1e3
    return r


def _staged_inputs(srcs):
    """Pinned host staging buffer and its device twin holding the tensors of `srcs`
    (name -> tensor) in 256-byte aligned slices; returns (host, device, device views)."""
    offs, total = {}, 0
    for k, t in srcs.items():
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(total, dtype=torch.uint8, device="cuda")

    def view(buf, k):
        t = srcs[k]
        nb = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
    for k, t in srcs.items():  # the host fills the step's inputs into the staging buffer
        view(stage_h, k).copy_(t.cpu())
    return stage_h, stage_d, {k: view(stage_d, k) for k in srcs}


def e2e_decode_fns(pa, case, max_seq_len):
    """Steps of the headline stream through the public API with host buffers: per step
    (sequence s of the rotation), one H2D copy of the step's inputs (q, block-table row
    and sequence length, packed in one pinned staging buffer, by a pa_copy kernel: a
    copy-engine node costs several microseconds more on this system), then pa_decode,
    whose combine writes the output straight into a pinned host buffer (the step's D2H
    transfer).  Returns (fns, outputs to check, H2D bytes, D2H bytes) per step."""
    fns, outs = [], []
    h2d = d2h = 0
    for s in range(case.q.shape[0]):
        srcs = {"q": case.q[s:s + 1].contiguous(),
                "block_table": case.block_table[s:s + 1].contiguous(),
                "seq_lens": case.seq_lens[s:s + 1].contiguous()}
        stage_h, stage_d, dev = _staged_inputs(srcs)
        out_h = torch.empty(srcs["q"].shape, dtype=torch.bfloat16).pin_memory()
        ws = torch.empty(max(256, pa.decode_workspace_size(1, case.q.shape[1],
                                                            case.k_cache.shape[2],
                                                            case.q.shape[2], case.block_size,
                                                            max_seq_len)),
                         dtype=torch.uint8, device="cuda")
        h2d, d2h = stage_h.numel(), out_h.numel() * out_h.element_size()

        def step(stage_h=stage_h, stage_d=stage_d, dev=dev, out_h=out_h, ws=ws):
            pa.copy(stage_d, stage_h)
            pa.decode(dev["q"], case.k_cache, case.v_cache, dev["block_table"],
                      dev["seq_lens"], case.scale, max_seq_len, out=out_h, workspace=ws)
        fns.append(step)
        outs.append((out_h, s))
    return fns, outs, h2d, d2h


def e2e_append_fns(pa, cases):
    """The 8K serving step through the public API with host buffers: per step one H2D
    copy of q, the new token's K/V, the block table and seq_lens of its replica (one
    pa_copy kernel from a pinned staging buffer), then pa_decode_append, whose combine
    writes the output into a pinned host buffer."""
    names = ("q", "new_k", "new_v", "block_table", "seq_lens")
    fns, outs = [], []
    h2d = d2h = 0
    for case in cases:
        S, hq, d = case.q.shape
        msl = int(case.seq_lens.max())
        stage_h, stage_d, dev = _staged_inputs({k: getattr(case, k).contiguous() for k in names})
        out_h = torch.empty((S, hq, d), dtype=torch.bfloat16).pin_memory()
        ws = torch.empty(max(256, pa.decode_workspace_size(S, hq, case.k_cache.shape[2], d,
                                                            case.block_size, msl)),
                         dtype=torch.uint8, device="cuda")
        slots = torch.empty(S, dtype=torch.int64, device="cuda")
        h2d, d2h = stage_h.numel(), out_h.numel() * out_h.element_size()

        def step(case=case, stage_h=stage_h, stage_d=stage_d, dev=dev, out_h=out_h, ws=ws,
                 slots=slots, msl=msl):
            pa.copy(stage_d, stage_h)
            pa.decode_append(dev["q"], case.k_cache, case.v_cache, dev["block_table"],
                             dev["seq_lens"], case.scale, msl, dev["new_k"], dev["new_v"],
                             out=out_h, workspace=ws, slot_mapping=slots)
        fns.append(step)
        outs.append((out_h, case, msl))
    return fns, outs, h2d, d2h


def step8k_leg(pa, steps, warmup, flush, peaks):
    """The serving step at 8K: each step appends its sequence's newest token (slot derived
    in the kernel, KV write) and decodes over 8192 keys; 32 copies of the workload in
    turn.  Its end-to-end form (host buffers) is timed between two device timings."""
    reps = headline_replicas("cuda")
    fns = [append_step_fn(pa, c, 8192)[0] for c in reps]
    r = decode_leg(pa, fns, 8192, 1, steps, warmup, flush, peaks,
                   f"{len(reps)} copies of the workload, each its own 64-page pool, in turn")
    r["step_alone_ms"] = statistics.mean(time_steps(graph_of(fns[0]).replay, steps, warmup,
                                                    flush))
    efns, outs, h2d, d2h = e2e_append_fns(pa, reps)
    e2e_ms = time_stream(efns, steps, warmup, flush)
    again_ms = time_stream(fns, steps, warmup, flush)
    torch.cuda.synchronize()
    for out_h, case, msl in outs[:min(len(outs), steps)]:
        ref = pa.decode(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                        case.scale, msl)
        assert torch.equal(out_h, ref.cpu()), "a step's host output differs from the decode's"
    r["e2e"] = {"ms_per_step": e2e_ms, "kv_gbs": 8192 * KV_BYTES_PER_TOKEN / (e2e_ms * 1e-3) / 1e9,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "device_ms_per_step_before_after": [r["ms_per_step"], again_ms]}
    del reps, fns, efns, outs
    torch.cuda.empty_cache()
    return r


# ------------------------------------------------------------------------ CPU oracle
def host_decode_case(case, s, kv=None):
    """Sequence s of a decode case as host arrays for the oracle (raw BF16 bits); kv: the
    caches' bits if already copied to the host."""
    from workloads import bits
    k, v = kv if kv is not None else (bits(case.k_cache), bits(case.v_cache))
    return dict(q=bits(case.q[s:s + 1]), k=k, v=v,
                block_table=case.block_table[s:s + 1].cpu().numpy(),
                seq_lens=case.seq_lens[s:s + 1].cpu().numpy(), scale=case.scale)


def oracle_decode_step(c, num_threads=None):
    import oracle

    def step():
        oracle.decode(c["q"], c["k"], c["v"], c["block_table"], c["seq_lens"], c["scale"],
                      num_threads=num_threads)
    return step


def cpu_oracle_timing(case_h, seconds, num_threads=None):
    """Mean host seconds of one oracle decode step (after one untimed step), repeated
    until `seconds` have passed."""
    step = oracle_decode_step(case_h, num_threads)
    step()  # builds / loads the oracle library, first touch of the pages
    n, t0 = 0, time.perf_counter()
    while True:
        step()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return el / n, n


def timed_host(fn, seconds):
    """Mean host seconds of fn() (after one untimed call), repeated until `seconds` pass."""
    fn()
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return el / n, n


def cpu_per_config(seconds):
    """The fp64 oracle on the host cores for the other configurations, with the same
    inputs as the GPU legs: the tiny decode (1701 keys), the 8K decode, the batched decode
    (16 sequences, 1.3 GB of K/V) and a sample of the q=4096 chunk's outputs (every 64th
    row, all 24 heads), each repeated for about `seconds`."""
    import oracle
    from workloads import bits
    nt = oracle.max_threads()
    r = {}
    for name, make, label in (("tiny_decode_1701", workloads.tiny_decode, "1701 keys"),
                              ("decode_8k", workloads.decode_8k, "8192 keys"),
                              ("batched_decode_16", workloads.batched_decode,
                               "16 sequences, 318,193 keys")):
        c = make(device="cuda")
        kv = (bits(c.k_cache), bits(c.v_cache))
        h = dict(q=bits(c.q), k=kv[0], v=kv[1], block_table=c.block_table.cpu().numpy(),
                 seq_lens=c.seq_lens.cpu().numpy(), scale=c.scale)
        nbytes = int(c.seq_lens.sum().item()) * KV_BYTES_PER_TOKEN
        del c, kv
        torch.cuda.empty_cache()
        sec, n = timed_host(oracle_decode_step(h), seconds)
        r[name] = {"value": nbytes / sec / 1e9, "unit": "GB/s", "cores": nt,
                   "ms_per_step": sec * 1e3,
                   "sample": f"{n} full decode steps ({label}), fp64, {nt} threads"}
        del h
    c = workloads.prefill_chunk("cuda")
    q, k, v = bits(c.q), bits(c.k_cache), bits(c.v_cache)
    bt = c.block_table[0].cpu().numpy()
    scale, q_start = c.scale, c.q_start
    slots = oracle.slot_mapping(c.positions.cpu().numpy(), c.block_table.cpu().numpy(),
                                c.block_size, seq_idx=c.seq_idx.cpu().numpy())
    oracle.reshape_and_cache(bits(c.new_k), bits(c.new_v), k, v, slots, c.block_size)
    del c
    torch.cuda.empty_cache()
    rows = np.repeat(np.arange(0, 4096, 64, dtype=np.int32), workloads.HQ)
    heads = np.tile(np.arange(workloads.HQ, dtype=np.int32), 64)
    flops = 4.0 * workloads.HEAD_DIM * float(np.sum(q_start + rows.astype(np.float64) + 1))
    sec, n = timed_host(lambda: oracle.prefill_rows(q, k, v, bt, q_start, True, scale, rows,
                                                    heads), seconds)
    r["prefill_q4096_over_4096"] = {
        "value": flops / sec / 1e9, "unit": "GFLOP/s", "cores": nt,
        "sample": f"{n} passes over 64 of the chunk's 4096 rows (every 64th) x 24 heads, "
                  f"fp64, {nt} threads; the whole chunk would take "
                  f"{sec * 4096 / 64:.1f} s"}
    return r


def headline_workload(device):
    """The headline: the 7 sequences of 32768 keys a 1 GiB pool holds (BS 832, 5% of K
    rows x8), on disjoint pages; one step decodes one of them."""
    return workloads.decode_sweep_rotation(HEADLINE_CTX, device)


METRIC = "paged decode KV GB/s (% of HBM peak) at 4K-32K ctx; q=4096 prefill TFLOP/s"


def headline_config(ws, extra=None):
    c = {"workload": HEADLINE, "block_size": 832, "context": HEADLINE_CTX,
         "step": "pa_decode of one sequence: split-context kernel (one launch) + LSE "
                 "combine (one launch)",
         "parallelism": f"replica per GPU x{ws}"}
    c.update(extra or {})
    return c


def run_reference(args, rank, ws):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores, over the
    headline workload: W untimed steps, then exactly K timed steps, each the exact
    attention of 24 heads over the 32768 keys of one sequence (the sequences of the
    rotation in turn), as the GPU step computes.  Under torchrun only rank 0 runs it."""
    if rank != 0:
        return
    import oracle
    from workloads import bits
    case = headline_workload("cpu")
    n = case.q.shape[0]
    kv = (bits(case.k_cache), bits(case.v_cache))
    steps = [oracle_decode_step(host_decode_case(case, s, kv)) for s in range(n)]
    for i in range(max(1, args.warmup)):
        steps[i % n]()
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        steps[i % n]()
        times.append(time.perf_counter() - t0)
    per_step = sum(times) / len(times)
    v = HEADLINE_CTX * KV_BYTES_PER_TOKEN / per_step / 1e9
    threads = oracle.max_threads()
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(1),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{args.steps} full decode steps of the headline "
                                       f"workload (fp64 attention of 24 heads over 32768 "
                                       f"keys each), {threads} threads"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def summary_of(value_frac, legs):
    """A few hundred bytes that repeat each leg's main figure (printed last)."""
    out = {"decode_32k_step_frac": value_frac}
    sw = legs.get("decode_sweep_1gib_pool_peaked", {})
    for ctx, r in sw.items():
        out[f"decode_{int(ctx) // 1024}k_frac"] = round(r["kv_pct_of_hbm_peak"] / 100, 4)
        out[f"decode_{int(ctx) // 1024}k_us"] = round(r["ms_per_step"] * 1e3, 2)
    for bs, r in legs.get("decode_32k_small_pages", {}).items():
        out[f"decode_32k_bs{bs}_frac"] = round(r["kv_pct_of_hbm_peak"] / 100, 4)
    r = legs.get("decode_8k_append_step")
    if r:
        out["step_8k_append_us"] = round(r["ms_per_step"] * 1e3, 2)
        out["step_8k_append_e2e_us"] = round(r["e2e"]["ms_per_step"] * 1e3, 2)
    r = legs.get("decode_8k_bs784")
    if r:
        out["decode_8k_bs784_frac"] = round(r["kv_pct_of_hbm_peak"] / 100, 4)
    r = legs.get("batched_decode_16_fused_write")
    if r:
        out["batched_16_frac"] = round(r["kv_pct_of_hbm_peak"] / 100, 4)
    for k, name in (("prefill_q4096_over_4096", "prefill_q4096"),
                    ("prefill_first_q4096_at_0", "prefill_first"),
                    ("prefill_tail_q1685_over_12288", "prefill_tail"),
                    ("prefill_mixed_4_chunks", "prefill_mixed")):
        if k in legs:
            out[name + "_frac"] = round(legs[k]["roofline"]["frac"], 4)
    return out


# ------------------------------------------------------------------------ main
def main():
    args = parse()
    rank, ws = dist_init(args)
    if args.impl == "reference":
        run_reference(args, rank, ws)
        return
    import paged_kv_cache_09_gb300 as pa
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    pa.load()
    peaks = load_peaks()
    # L2 flush by READING a buffer 4x the L2 size: the lines it leaves behind are clean,
    # so the timed step pays no write-back of the flush itself.
    flush_buf = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device="cuda")

    def flush():
        flush_buf.sum()

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()

    # ---- headline: timed K steps, barrier + synchronize on both sides
    value = kernel_gbs = k_ms = k_min = k_med = e2e_val = e2e_ms = alone_ms = again_ms = None
    step_ms = None
    h2d = d2h = 0
    head = None
    if not args.skip_headline:
        head = headline_workload("cuda")
        n = head.q.shape[0]
        fns = [attn_fn(pa, head, s, HEADLINE_CTX) for s in range(n)]
        # Warm-up outside the timed region: the first heavy GPU work of the process ran
        # ~4% slower than the same stream timed later in the run (clocks and power
        # settle), so a whole untimed stream of steps comes first.
        time_stream(fns, args.steps, args.warmup, flush)
        barrier(ws)
        torch.cuda.synchronize()
        step_ms = time_stream(fns, args.steps, args.warmup, flush)
        torch.cuda.synchronize()
        barrier(ws)
        total_ms = max_over_ranks(step_ms * args.steps, ws)
        nbytes_rank = HEADLINE_CTX * KV_BYTES_PER_TOKEN * args.steps
        value = sum_over_ranks(nbytes_rank, ws) / (total_ms * 1e-3) / 1e9
        kms = time_main_kernel(pa, fns[0], args.steps, args.warmup, flush)
        k_ms = statistics.mean(kms)
        k_min, k_med = min(kms), statistics.median(kms)
        kernel_gbs = HEADLINE_CTX * KV_BYTES_PER_TOKEN / (k_ms * 1e-3) / 1e9
        alone_ms = statistics.mean(time_steps(graph_of(fns[0]).replay, args.steps,
                                              args.warmup, flush))
        # End to end through the public API with host buffers, then the device-resident
        # stream again (A/B/A, back to back in this run).
        efns, outs, h2d, d2h = e2e_decode_fns(pa, head, HEADLINE_CTX)
        e2e_ms = time_stream(efns, args.steps, args.warmup, flush)
        again_ms = time_stream(fns, args.steps, args.warmup, flush)
        torch.cuda.synchronize()
        for out_h, s in outs[:min(len(outs), args.steps)]:
            ref = pa.decode(head.q[s:s + 1], head.k_cache, head.v_cache,
                            head.block_table[s:s + 1], head.seq_lens[s:s + 1], head.scale,
                            HEADLINE_CTX)
            assert torch.equal(out_h, ref.cpu()), "a step's host output differs from the decode's"
        e2e_val = HEADLINE_CTX * KV_BYTES_PER_TOKEN / (e2e_ms * 1e-3) / 1e9
        assert pa.device_errors() == 0, "device error word set during the headline leg"
        del fns, efns, outs

    legs = {}
    want = set() if args.legs == "none" else (
        {"sweep", "small_pages", "step8k", "bs784", "batched", "prefill", "prefill_tail",
         "prefill_first", "prefill_mixed", "prep"}
        if args.legs == "all" else set(args.legs.split(",")))
    if rank == 0 and "sweep" in want:
        sweep = {}
        for ctx in [int(x) for x in args.contexts.split(",") if x]:
            c = head if ctx == HEADLINE_CTX and head is not None else \
                workloads.decode_sweep_rotation(ctx, "cuda")
            n = c.q.shape[0]
            fns = [attn_fn(pa, c, s, ctx) for s in range(n)]
            sweep[str(ctx)] = decode_leg(
                pa, fns, ctx, 1, args.steps, args.warmup, flush, peaks,
                f"{n} sequences of {ctx} tokens on disjoint pages of one 1 GiB pool, decoded "
                f"one per step in turn ({n * ctx * KV_BYTES_PER_TOKEN / 2**20:.0f} MiB of K/V)")
            del c, fns
            torch.cuda.empty_cache()
        legs["decode_sweep_1gib_pool_peaked"] = sweep
    head = None
    torch.cuda.empty_cache()
    if rank == 0 and "small_pages" in want:
        small = {}
        for bs in (16, 64):
            c = workloads.decode_sweep_rotation(32768, "cuda", block_size=bs)
            n = c.q.shape[0]
            fns = [attn_fn(pa, c, s, 32768) for s in range(n)]
            small[str(bs)] = decode_leg(
                pa, fns, 32768, 1, args.steps, args.warmup, flush, peaks,
                f"{n} sequences of 32768 tokens in {bs}-token pages of one 1 GiB pool, "
                f"decoded one per step in turn")
            del c, fns
            torch.cuda.empty_cache()
        legs["decode_32k_small_pages"] = small
    if rank == 0 and "step8k" in want:
        legs["decode_8k_append_step"] = step8k_leg(pa, args.steps, args.warmup, flush, peaks)
    if rank == 0 and "bs784" in want:
        reps = headline_replicas("cuda", block_size=784, new_tokens=0)
        fns = [attn_fn(pa, c, 0, 8192) for c in reps]
        legs["decode_8k_bs784"] = decode_leg(
            pa, fns, 8192, 1, args.steps, args.warmup, flush, peaks,
            f"{len(reps)} copies of the workload, each its own 64-page pool, in turn")
        del reps, fns
        torch.cuda.empty_cache()
    if rank == 0 and "batched" in want:
        reps = [workloads.batched_decode("cuda"), workloads.batched_decode("cuda", seed=2005)]
        fns = [append_step_fn(pa, c)[0] for c in reps]
        legs["batched_decode_16_fused_write"] = decode_leg(
            pa, fns, int(reps[0].seq_lens.sum()), 16, max(5, args.steps // 2), args.warmup,
            flush, peaks, "two copies of the workload (same lengths, 2.2 GB pools each), in turn")
        del reps, fns
        torch.cuda.empty_cache()
    if rank == 0 and "l2check" in args.legs.split(","):
        legs["l2check"] = l2check_leg(pa, flush)
    if rank == 0 and "prep" in want:
        legs["decode_input_prep_2_groups"] = input_prep_leg(pa, args.steps, args.warmup, flush)
    if rank == 0 and "prefill_mixed" in want:
        legs["prefill_mixed_4_chunks"] = prefill_leg(
            pa, max(5, args.steps // 4), args.warmup, flush, peaks, "prefill_mixed")
    if rank == 0 and "prefill_tail" in want:
        legs["prefill_tail_q1685_over_12288"] = prefill_leg(
            pa, max(5, args.steps // 4), args.warmup, flush, peaks, "prefill_tail")
    if rank == 0 and "prefill_first" in want:
        legs["prefill_first_q4096_at_0"] = prefill_leg(
            pa, max(5, args.steps // 4), args.warmup, flush, peaks, "prefill_first")
    if rank == 0 and "prefill" in want:
        legs["prefill_q4096_over_4096"] = prefill_leg(pa, max(5, args.steps // 4), args.warmup,
                                                      flush, peaks)
    assert pa.device_errors() == 0, "device error word set during the legs"
    clk = clocks.stop() if clocks else None

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        c = headline_workload("cuda")
        ch = host_decode_case(c, 0)
        del c
        torch.cuda.empty_cache()
        per_all, n_all = cpu_oracle_timing(ch, args.cpu_seconds)
        per_one, n_one = cpu_oracle_timing(ch, args.cpu_seconds, num_threads=1)
        nbytes = HEADLINE_CTX * KV_BYTES_PER_TOKEN
        cpu = {"value": nbytes / per_all / 1e9, "unit": "GB/s", "cores": oracle.max_threads(),
               "kind": "oracle",
               "sample": f"{n_all} full decode steps of the headline workload (fp64 attention "
                         f"of 24 heads over 32768 keys), {per_all * 1e3:.1f} ms each on "
                         f"{oracle.max_threads()} threads",
               "single_thread": {"value": nbytes / per_one / 1e9, "unit": "GB/s", "cores": 1,
                                 "ms_per_step": per_one * 1e3,
                                 "sample": f"{n_one} steps of the same workload, one thread"},
               "per_config": cpu_per_config(max(1.0, args.cpu_seconds / 4))}

    if rank != 0:
        return
    frac = kernel_gbs / peaks["hbm_gbs"] if kernel_gbs else None
    line = {
        "metric": METRIC,
        "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(ws, {
            "timing": f"{args.steps} consecutive steps captured in one CUDA graph, one "
                      f"replay between two events (the graph's launch paid once)",
            "l2": "inputs larger than L2: the 7 sequences of 32768 keys the 1 GiB pool holds "
                  "(939 MB of K/V), decoded one per step in turn, so no step finds its K/V in "
                  "the 129 MB L2",
            "step_alone_ms": alone_ms,
            "step_alone": "the same step as a single-step graph replayed after an L2 flush "
                          "(its graph launch included)",
            "device_ms_per_step_after_e2e": again_ms,
            "kv_pct_of_hbm_peak": (100.0 * value / ws / peaks["hbm_gbs"] if value else None)}),
        "clocks": clk,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": "H2D: one pa_copy kernel from a pinned staging buffer (q, block-table "
                          "row, sequence length); D2H: the combine kernel writes the output "
                          "into a pinned host buffer; all inside the steps' CUDA graph, timed "
                          "between two timings of the device-resident stream"},
        # per step: the split-context decode and the LSE combine
        "gpu_launches": 0 if args.skip_headline else 2 * args.steps,
        "roofline": {"bound": "hbm", "achieved": kernel_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": frac,
                     "traffic": SPLIT_32K_DRAM_BYTES,
                     "traffic_unit": "bytes per launch",
                     "kernel": "decode_split_kernel",
                     "algorithmic_bytes_per_launch": HEADLINE_CTX * KV_BYTES_PER_TOKEN,
                     "kernel_ms": k_ms, "kernel_ms_min": k_min, "kernel_ms_median": k_med,
                     "peak_source": f"{peaks['source']} hbm_gbs",
                     "kernel_timing": "library events around the split launch of an eager "
                                      "step after an L2 flush, mean of K launches"},
        "cpu_baseline": cpu,
        "legs": legs,
        "summary": summary_of(round(value / ws / peaks["hbm_gbs"], 4) if value else None, legs),
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
