"""Benchmark: MLA decode over a paged latent KV cache on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the whole path over one batch: the tile scheduler
(mla_get_metadata), the split-KV kernel and the combine (mla_decode_kvcache),
on inputs already resident in HBM.  The default workload is the largest
single-GPU one, the long-context decode batch (b=64, s_q=1, h_q=128, 65536
cached tokens per sequence, page 64: 4.85 GB of KV pages).  --workload all
prints one line for every workload, in turn.

Reported figures (one JSON line from rank 0):
  value         KV-cache GB/s: bytes of the KV pages touched plus q, O and LSE,
                divided by the device time of a step (the metric's bytes)
  us_per_call   device time of a step in microseconds
  tflops        2 * h_q * (576 + 512) * visible keys, per second
  roofline      the split-KV kernel alone (CUDA events around it on its stream)
                against the measured HBM copy bandwidth
  decode_only   the same metric for the decode call alone (split-KV + combine),
                with the metadata computed once and reused, as every layer
                of a model reuses it
  e2e           the same metric through the public API with host buffers:
                pinned host -> device copies of every input, the two calls,
                device -> host copies of O and LSE, all inside the timed region
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample

The KV pages of every workload except the tiny one exceed the 129 MB L2, so
no flush is done between steps (config.l2 says so).  --impl reference times
the fp64 CPU oracle instead (this tier's reference arm).
"""
from __future__ import annotations

import argparse
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

import torch  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "MLA decode µs/call, KV-cache GB/s and TFLOPS vs GB300 roofline"


# ------------------------------------------------------------------ workload figures
def workload_label(case):
    """The workload named by what it is, with its sizes (the same string in both arms)."""
    lengths = "U" + str(case.seqlen_range) if case.seqlen_range else case.seqlens[0]
    cache = ", cache=e4m3+per-token fp32 scales" if case.fp8 else (f", sparse topk={case.topk}" if case.topk else "")
    return (f"{case.name}: b={case.batch}, s_q={case.s_q}, h_q={case.h_q}, h_kv={case.h_kv}, d={case.d}, "
            f"dv={case.dv}, page={case.page}, causal={case.causal}, seqlens={lengths}{cache}")


def workload_figures(case, seqlens):
    """Algorithmic bytes and FLOPs of one decode call."""
    from mla_decode_attention_latent_gb300 import workloads as W
    page_bytes = case.page_bytes  # bf16 rows, or e4m3 codes + fp32 scales
    if case.topk:
        # sparse: the gathered rows and the index lists are the cache-side bytes
        entries = W.valid_list_entries(case, seqlens)
        kv_bytes = entries * case.h_kv * case.d * 2 + case.batch * case.s_q * case.topk * 4
        q_bytes = case.batch * case.s_q * case.h_q * case.d * 2
        o_bytes = case.batch * case.s_q * case.h_q * case.dv * 2
        lse_bytes = case.batch * case.s_q * case.h_q * 4
        flops = 2.0 * case.h_q * (case.d + case.dv) * entries
        return {"bytes": kv_bytes + q_bytes + o_bytes + lse_bytes, "kv_bytes": kv_bytes, "flops": flops,
                "valid_token_bytes": entries * case.h_kv * case.d * 2}
    kv_bytes = W.kv_pages_touched(seqlens, case.page) * page_bytes
    q_bytes = case.batch * case.s_q * case.h_q * case.d * 2
    o_bytes = case.batch * case.s_q * case.h_q * case.dv * 2
    lse_bytes = case.batch * case.s_q * case.h_q * 4
    keys = 0
    for t in seqlens:
        for i in range(case.s_q):
            keys += max(0, (t - case.s_q + i + 1) if case.causal else t)
    flops = 2.0 * case.h_q * (case.d + case.dv) * keys
    return {"bytes": kv_bytes + q_bytes + o_bytes + lse_bytes, "kv_bytes": kv_bytes, "flops": flops,
            "valid_token_bytes": sum(seqlens) * page_bytes // case.page}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs")
            bf16 = d.get("bf16_tflops")
            bf16s = d.get("bf16_tflops_sustained")
            if hbm:
                return {"hbm_gbs": float(hbm), "bf16_tflops": float(bf16 or FALLBACK_BF16_TFLOPS),
                        "bf16_tflops_sustained": float(bf16s or bf16 or FALLBACK_BF16_TFLOPS),
                        "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def roofline(fig, kernel_ms, pk):
    """(bound, achieved, peak, unit) of one launch: the roof that binds is picked
    by the workload's FLOPs per byte against the ridge point of the two peaks
    (h_q = 128 decode sits just below it; multi-token decode far above)."""
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if fig["flops"] / fig["bytes"] > ridge:
        return "tensor", fig["flops"] / (kernel_ms * 1e-3) / 1e12, pk["bf16_tflops"], "TFLOP/s"
    return "hbm", fig["bytes"] / (kernel_ms * 1e-3) / 1e9, pk["hbm_gbs"], "GB/s"


def split_kernel_traffic(workload):
    """DRAM bytes per split-KV launch from the committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", f"split_kv_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h or h.group(1) != split_source_hash():
        return None
    return float(m.group(1))


def split_source_hash():
    """sha256 of the split kernel's sources with comments and blank space removed
    (a comment edit leaves the compiled kernel, and so its counters, unchanged)."""
    csrc = os.path.join(ROOT, "mla_decode_attention_latent_gb300", "csrc")
    hs = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.startswith("mla_split") or name.endswith((".cuh", ".h")):
            hs.update(_code_only(open(os.path.join(csrc, name)).read()).encode())
    return hs.hexdigest()


def _code_only(src):
    """C/C++ source without // and /* */ comments (string literals kept) or blank space."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":                       # a literal: copy through its closing quote
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join("".join(out).split())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ distributed
def dist_setup(n_gpus):
    if n_gpus <= 1 and "RANK" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(n_gpus)))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Slowest rank's time: the all-reduce runs on the process group's own device (NCCL: GPU, gloo: CPU)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_case(case, rank):
    """Weak scaling: every rank decodes its own full batch of the workload, drawn with its own seed."""
    import dataclasses
    return case if rank == 0 else dataclasses.replace(case, seed=case.seed + 7919 * rank)


def aggregate_gbs(bytes_per_rank, world, ms_step_slowest):
    """Whole-job KV-cache GB/s: every rank's bytes over the slowest rank's step time."""
    return bytes_per_rank * world / (ms_step_slowest * 1e-3) / 1e9


# ------------------------------------------------------------------ CPU oracle
def time_oracle(case, x_cpu, budget_s=10.0, max_seqs=None):
    """Time the fp64 oracle on whole sequences (all rows) until ~budget_s of work; scale to one call."""
    import numpy as np

    import oracle
    from mla_decode_attention_latent_gb300 import workloads as W
    R = case.s_q * case.h_q
    sl = x_cpu.cache_seqlens.numpy()
    q_bits = W.bf16_bits(x_cpu.q)
    k_data = x_cpu.kcache.numpy() if case.fp8 else W.bf16_bits(x_cpu.kcache)
    bt = x_cpu.block_table.numpy()
    if case.topk:
        idx = x_cpu.indices.numpy()

        def decode(q, k, bt_, sl_, dv, scale, causal, rows):
            return oracle.mla_decode_sparse(q, k, bt_, sl_, idx, dv, scale, rows=rows)
    else:
        decode = oracle.mla_decode_fp8 if case.fp8 else oracle.mla_decode

    def run(seqs):
        rows = np.concatenate([np.arange(b * R, (b + 1) * R, dtype=np.int64) for b in seqs])
        t0 = time.perf_counter()
        decode(q_bits, k_data, bt, sl, case.dv, case.softmax_scale, case.causal, rows=rows)
        return time.perf_counter() - t0

    t1 = run([0])
    n = max(1, min(case.batch if max_seqs is None else max_seqs, int(budget_s / max(t1, 1e-6))))
    seqs = list(range(n))
    t = run(seqs)
    work = [min(case.topk, int(s)) if case.topk else int(s) for s in sl]  # keys each sequence's rows see
    frac_keys = sum(work[b] for b in seqs) / max(1, sum(work))
    return {"seconds": t, "seqs": n, "call_seconds": t / frac_keys, "cores": oracle.max_threads()}


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long", help="a workload name, or 'all'")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    from mla_decode_attention_latent_gb300 import workloads as W
    names = ALL_WORKLOADS if args.workload == "all" else [args.workload]

    if args.impl == "reference":
        for name in names:
            reference_arm(args, W.CASES[name])
        return

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import mla_decode_attention_latent_gb300 as mla
    mla._lib.load()
    if world > 1:
        # one job across several GPUs: no TMA cluster multicast anywhere
        mla.mla_set_cluster_multicast(False)
    for name in names:
        line = run_workload(args, mla, W.CASES[name], name, rank, world, local, dev)
        if rank == 0:
            print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


L2_FLUSH_BYTES = 256 << 20  # twice the GB300's L2
HOLD_S_PER_STEP = 300e-6     # host time to enqueue one timed step (flush, events, three launches), generously

# every workload, in the order --workload all runs them
ALL_WORKLOADS = ["tiny", "uniform", "variable", "mtp", "long", "uniform_d512", "uniform_fp8", "sparse"]


def partition(mla, case, lens, num_parts=None):
    """The work partition as a caller of this workload computes it: a sparse
    workload over its list lengths with the sparse decode's costs."""
    if case.topk:
        return mla.mla_get_metadata_sparse(lens, case.num_q_rows, case.h_kv, num_parts=num_parts)
    return mla.mla_get_metadata(lens, case.num_q_rows, case.h_kv, num_parts=num_parts)


def run_workload(args, mla, case, name, rank, world, local, dev):
    """Time one workload; returns rank 0's JSON line (None on other ranks)."""
    from mla_decode_attention_latent_gb300 import workloads as W
    case = rank_case(case, rank)

    x = W.make_inputs(case, device=str(dev))
    sl_list = x.cache_seqlens.cpu().tolist()
    fig = workload_figures(case, sl_list)
    stream = torch.cuda.current_stream(dev)

    # the work partition runs on the cache lengths, or on the list lengths (sparse)
    part_lens = (torch.full((case.batch,), case.topk, dtype=torch.int32, device=dev) if case.topk
                 else x.cache_seqlens)
    md, ns = partition(mla, case, part_lens)
    num_parts = md.shape[0]
    o = torch.empty((case.batch, case.s_q, case.h_q, case.dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.batch, case.s_q, case.h_q), dtype=torch.float32, device=dev)
    ws = torch.empty((mla.mla_workspace_bytes(case.batch, case.s_q, case.h_q, case.h_kv, case.dv, num_parts),),
                     dtype=torch.uint8, device=dev)

    decode = mla.mla_decode_kvcache_fp8 if case.fp8 else mla.mla_decode_kvcache

    def step(md_k=None, ns_k=None):
        if md_k is None:
            md_k, ns_k = partition(mla, case, part_lens, num_parts)
        if case.topk:
            mla.mla_decode_kvcache_sparse(x.q, x.kcache, x.block_table, x.cache_seqlens, x.indices, case.dv, md_k,
                                          ns_k, list_lens=part_lens, softmax_scale=case.softmax_scale, out=o, lse=lse,
                                          workspace=ws)
        else:
            decode(x.q, x.kcache, x.block_table, x.cache_seqlens, case.dv, md_k, ns_k,
                   softmax_scale=case.softmax_scale, causal=case.causal, out=o, lse=lse, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert mla.mla_device_status(clear=True) == 0, "device-side error during warm-up"

    # per-step split-kernel events (recorded by the library around the split-KV launch)
    ev_split = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev_split:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()

    # a workload whose bytes fit in L2 is timed step by step, with L2 flushed
    # (a 256 MB buffer written) between steps, outside the timed intervals
    small = fig["bytes"] < L2_FLUSH_BYTES
    flush = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev) if small else None

    def hold_device():
        """Keep the stream busy (a GPU sleep) while the host enqueues the timed
        steps, so that the device-timed region holds the steps' GPU work and no
        host launch latency; the sleep itself stays before the first event."""
        torch.cuda._sleep(int(HOLD_S_PER_STEP * args.steps * 2.0e9))

    def timed(fn):
        """ms of args.steps calls of fn: back to back, or one by one with L2 flushed between them."""
        hold_device()
        if not small:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in pairs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in pairs)

    clocks = ClockSampler(local)
    clocks.start()
    # timed region 1 (value): the K steps back to back, nothing recorded
    # between their kernels, so each launch may overlap its predecessor's tail
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("steps")
    ms_total = timed(step)
    torch.cuda.nvtx.range_pop()
    barrier(world)
    assert mla.mla_device_status(clear=True) == 0, "device-side error in the timed region"
    # timed region 2 (roofline): the same K steps with CUDA events around each
    # split-KV launch on its stream; the events cost several us per step, which
    # is why they stay out of region 1
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("steps_with_split_events")
    hold_device()
    for k in range(args.steps):
        mla.mla_set_timing_events(*ev_split[k])
        step()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    mla.mla_set_timing_events(None, None)
    # timed region 3 (decode_only): the decode call alone, with the metadata
    # of the first step reused by every later one (as every layer reuses it)
    md_once, ns_once = partition(mla, case, part_lens, num_parts)
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("decode_only")
    ms_decode = timed(lambda: step(md_once, ns_once))
    torch.cuda.nvtx.range_pop()
    barrier(world)
    clk = clocks.stop()
    assert mla.mla_device_status(clear=True) == 0, "device-side error in the timed region"
    ms_decode = max_over_ranks(ms_decode, world) / args.steps

    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    split_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_split)
    value = aggregate_gbs(fig["bytes"], world, ms_step)
    tflops = fig["flops"] * world / (ms_step * 1e-3) / 1e12
    pk = peaks()
    bound, achieved, peak, unit = roofline(fig, split_ms, pk)
    traffic = split_kernel_traffic(name)

    # end-to-end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = e2e_run(mla, case, x, fig, dev, stream, steps=max(3, min(args.steps, 10)), world=world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_cpu = W.make_inputs(case, device="cpu") if case.name == "tiny" else \
            W.Inputs(case, x.q.cpu(), x.kcache.cpu(), x.block_table.cpu(), x.cache_seqlens.cpu(),
                     None if x.indices is None else x.indices.cpu())
        t = time_oracle(case, x_cpu)
        cpu = {"value": fig["bytes"] / t["call_seconds"] / 1e9, "unit": "GB/s", "cores": t["cores"],
               "kind": "oracle", "us_per_call": t["call_seconds"] * 1e6,
               "sample": f"{t['seqs']} of {case.batch} sequences (all {case.s_q * case.h_q} query rows each), "
                         f"{t['seconds']:.2f} s, scaled to one call by visible keys"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16" if case.fp8 else "bf16", "data": "synthetic",
            "us_per_call": round(ms_step * 1e3, 2), "tflops": round(tflops, 2),
            "hbm_frac_of_" + pk["source"]: round(value / pk["hbm_gbs"], 4),
            "hbm_frac_of_nominal_8tbs": round(value / 8000.0, 4),
            "tensor_frac_of_" + pk["source"]: round(tflops / pk["bf16_tflops"], 4),
            "config": {"workload": workload_label(case),
                       "batch": case.batch, "s_q": case.s_q, "h_q": case.h_q, "num_parts": num_parts,
                       "kv_bytes": fig["kv_bytes"], "bytes_per_call": fig["bytes"], "flops_per_call": fig["flops"],
                       "l2": ("flushed between steps (256 MB written), per-step events" if small else
                              "no flush: the bytes of a call exceed the 129 MB L2"),
                       "launch": "steps enqueued behind a GPU sleep before the first event, so host launch "
                                 "latency stays outside the device-timed region",
                       "parallelism": f"replicas x{world}, one batch per GPU" if world > 1 else "single GPU"},
            "roofline": {"bound": bound, "kernel": "split_kv", "achieved": round(achieved, 1),
                         "peak": peak, "unit": unit, "frac": round(achieved / peak, 4),
                         "peak_source": pk["source"], "split_kernel_ms": round(split_ms, 5),
                         "traffic": traffic},
            "decode_only": {"us_per_call": round(ms_decode * 1e3, 2),
                            "value": round(aggregate_gbs(fig["bytes"], world, ms_decode), 2), "unit": "GB/s",
                            "what": "split-KV + combine per call, metadata computed once and reused"},
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": 3 * args.steps,
            "cpu_baseline": cpu,
        }
        return line
    return None


def e2e_run(mla, case, x, fig, dev, stream, steps, world):
    """Inputs from pinned host memory, outputs back to pinned host memory, every step timed.

    Each step copies its inputs into one of two device buffer sets on a copy
    stream while the previous step decodes, as a serving loop would; the
    decode waits for its own copies, and a copy waits until the decode that
    last used its buffer set is done."""
    hq = x.q.cpu().pin_memory()
    hk = x.kcache.cpu().pin_memory()
    hbt = x.block_table.cpu().pin_memory()
    hsl = x.cache_seqlens.cpu().pin_memory()
    ho = torch.empty((case.batch, case.s_q, case.h_q, case.dv), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((case.batch, case.s_q, case.h_q), dtype=torch.float32).pin_memory()
    hidx = x.indices.cpu().pin_memory() if case.topk else None
    sets = []
    for _ in range(2):
        sets.append({"q": torch.empty_like(x.q), "k": torch.empty_like(x.kcache), "bt": torch.empty_like(x.block_table),
                     "sl": torch.empty_like(x.cache_seqlens),
                     "idx": torch.empty_like(x.indices) if case.topk else None,
                     "copied": torch.cuda.Event(), "used": torch.cuda.Event()})
    decode = mla.mla_decode_kvcache_fp8 if case.fp8 else mla.mla_decode_kvcache
    if case.topk:
        lens = torch.full((case.batch,), case.topk, dtype=torch.int32, device=dev)
    copy_stream = torch.cuda.Stream(dev)

    def one(i):
        d = sets[i % 2]
        copy_stream.wait_event(d["used"])  # the decode that last read this set is done
        with torch.cuda.stream(copy_stream):
            d["q"].copy_(hq, non_blocking=True)
            d["k"].copy_(hk, non_blocking=True)
            d["bt"].copy_(hbt, non_blocking=True)
            d["sl"].copy_(hsl, non_blocking=True)
            if case.topk:
                d["idx"].copy_(hidx, non_blocking=True)
            d["copied"].record(copy_stream)
        stream.wait_event(d["copied"])
        if case.topk:
            md, ns = partition(mla, case, lens)
            o, lse = mla.mla_decode_kvcache_sparse(d["q"], d["k"], d["bt"], d["sl"], d["idx"], case.dv, md, ns,
                                                   list_lens=lens, softmax_scale=case.softmax_scale)
        else:
            md, ns = mla.mla_get_metadata(d["sl"], case.num_q_rows, case.h_kv)
            o, lse = decode(d["q"], d["k"], d["bt"], d["sl"], case.dv, md, ns, softmax_scale=case.softmax_scale,
                            causal=case.causal)
        d["used"].record(stream)
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    a.record(stream)
    copy_stream.wait_stream(stream)  # no copy of the timed steps starts before the first event
    for i in range(steps):
        one(i)
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hbt, hsl) + ((hidx,) if case.topk else ()))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hl))
    del sets
    return {"value": round(fig["bytes"] * world / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "each step's host-to-device copies overlap the previous step's decode (two buffer sets)"}


def reference_arm(args, case):
    """This tier's reference arm: the fp64 CPU oracle, on a bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from mla_decode_attention_latent_gb300 import workloads as W
    x = W.make_inputs(case, device="cpu")
    fig = workload_figures(case, x.cache_seqlens.tolist())
    per_step = max(1.0, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        time_oracle(case, x, budget_s=min(per_step, 2.0), max_seqs=1)
    secs, call_secs, seqs, cores = [], [], 0, 1
    for _ in range(args.steps):
        t = time_oracle(case, x, budget_s=per_step)
        secs.append(t["seconds"])
        call_secs.append(t["call_seconds"])
        seqs, cores = t["seqs"], t["cores"]
    call = statistics.mean(call_secs)
    value = fig["bytes"] / call / 1e9
    line = {"metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(call * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_label(case), "batch": case.batch, "s_q": case.s_q, "h_q": case.h_q,
                       "kv_bytes": fig["kv_bytes"], "bytes_per_call": fig["bytes"], "flops_per_call": fig["flops"],
                       "parallelism": "host cores, rank 0 only"},
            "cpu_baseline": {"kind": "oracle", "cores": cores, "value": round(value, 4), "unit": "GB/s",
                             "sample": f"{seqs} of {case.batch} sequences per step, scaled to one call"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
