"""Benchmark of the blockwise ring-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0.  The headline step is one ra_blockwise_attn_fwd call
on the causal GQA prefill workload (B=1, S=32768, Hq=32, Hkv=8, D=128, bf16,
8 ring shards, 128-key blocks); `value` is its causal-adjusted attention
TFLOP/s (4*D FLOPs per unmasked query/key pair), `e2e` the same call with the
inputs copied from pinned host memory and the results read back every step.
The same line carries the other rows measured on their own workloads: the
headline workload in the zigzag and striped shard layouts, its backward pass
(contiguous, zigzag and striped), shared-prefix fan-out decode (HBM GB/s; contiguous and
over a paged KV pool), fan-out prefill (8 branches x 20 rows), per-shard
partials + LSE merge on the Llama-3-70B-shaped layer, and the million-token
stress case.

Under torchrun (--gpus N > 1) every rank runs an independent replica of the
same workload (the path needs no exchange between GPUs); the barrier and the
max over ranks are timing only.  `--impl reference` times the fp64 CPU oracle
on a bounded sample of the same workload (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s (causal-adjusted) & % bf16 peak; fan-out decode HBM GB/s"
HEADLINE = "gqa_causal_prefill_32k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) per launch of the headline kernel from an ncu
# capture, valid only while the kernel source hashes to the recorded value.
NCU_TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum on the timed 32768-token configuration
    # (bench.py --profile-case prefill_32k, third launch): 403008512 read + 237972736 written
    "b5ed574b6f1cc6fc": 640981248,
}


# ----------------------------------------------------------------------------------------------
# work accounting (algorithmic FLOPs and bytes)
# ----------------------------------------------------------------------------------------------

def ring_flops(B, S, Hq, D, causal):
    """4*D FLOPs (QK^T and PV) per unmasked (query, key) pair."""
    pairs = S * (S + 1) // 2 if causal else S * S
    return 4 * D * Hq * B * pairs


def fanout_flops(R, Hq, D, S_prefix, S_suffix):
    return 4 * D * Hq * R * (S_prefix + S_suffix)


def fanout_prefill_flops(rows, Hq, D, S_prefix, S_suffix):
    """Fan-out prefill with a causal suffix: row t of a branch with n new rows is
    suffix token S_suffix - n + t and sees the whole prefix plus suffix keys up to
    itself."""
    vis = sum(S_prefix + S_suffix - n + t + 1 for n in rows for t in range(n))
    return 4 * D * Hq * vis


def fanout_bytes(R, n_branches, Hq, Hkv, D, S_prefix, S_suffix, esz=2):
    """Prefix K+V once, every suffix K+V once, Q in, O out, lse out."""
    kv = 2 * esz * Hkv * D * (S_prefix + n_branches * S_suffix)
    return kv + 2 * esz * R * Hq * D + 4 * Hq * R


def ring_bytes(B, S, Hq, Hkv, D, esz=2):
    return esz * B * S * D * (2 * Hq + 2 * Hkv) + 4 * B * Hq * S


def merge_bytes(P, B, S, H, D, esz=2, causal=False):
    """Non-empty partial rows read once (with a causal mask, the query rows of
    shard k have k + 1 non-empty shard partials), every partial lse read, the
    merged O and lse written."""
    L = S // P
    nonempty_rows = B * H * (L * P * (P + 1) // 2 if causal else S * P)
    return nonempty_rows * D * esz + P * B * S * H * 4 + B * S * H * (D * esz + 4)


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (timing only: replicas exchange no data)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step: float, steps: int, total_ms: float, world: int) -> float:
    """Whole-job rate: the units all ranks processed over the slowest rank's time (x 1e-12, per s)."""
    return world * units_per_step * steps / (total_ms * 1e-3) / 1e12


def gpu_local_cpus(device_index: int):
    """Host CPUs on the GPU's own NUMA node (from sysfs), or None if unknown.

    Pinned host buffers are placed on the node of the CPU that first touches
    them; allocating them from these CPUs keeps host<->device copies off the
    link between host sockets."""
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(device_index), "--query-gpu=pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True, timeout=20).stdout.strip()
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{(dom[-4:] + ':' + rest).lower()}"
        cpus = set()
        for part in open(os.path.join(path, "local_cpulist")).read().strip().split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        node = int(open(os.path.join(path, "numa_node")).read().strip())
        return (cpus or None), node
    except Exception:
        return None, None


def pinned_on_gpu_node(device_index: int, make):
    """Runs make() (which allocates and fills pinned host tensors) on the GPU's
    NUMA-local CPUs, then restores the thread's CPU affinity."""
    cpus, node = gpu_local_cpus(device_index)
    old = os.sched_getaffinity(0)
    if cpus:
        os.sched_setaffinity(0, cpus)
    try:
        return make(), node, len(cpus) if cpus else None
    finally:
        os.sched_setaffinity(0, old)


def peaks():
    p = dict(FALLBACK_PEAKS)
    src = "fallback"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            m = json.load(open(path))
            for k in p:
                if k in m:
                    p[k] = float(m[k])
            src = "measured"
        except Exception:
            pass
    p["source"] = src
    return p


def kernel_hash():
    h = hashlib.sha256()
    for f in ("attn_tc.cu", "ra_device.cuh", "ra_walk.h"):
        h.update(open(os.path.join(ROOT, "ring_context_parallelism_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        busy = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------------------------
# timing helpers
# ----------------------------------------------------------------------------------------------

def timed_steps(fn, steps, warmup, flush=None):
    """W untimed calls, then K calls each bracketed by CUDA events on the current
    stream (L2 flushed before each call, outside the events).  Returns per-step ms."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in ev:
        if flush is not None:
            flush()
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in ev]


def make_flush(nbytes=512 << 20):
    """L2 flush between timed steps: write a buffer larger than L2, then read
    another one, so that the write-backs of the flush's dirty lines happen
    before the timed region and L2 holds only clean, unrelated lines."""
    import torch

    buf = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    rd = torch.ones(nbytes // 8, dtype=torch.float32, device="cuda")

    def flush():
        buf.fill_(1.0)
        rd.sum()

    return flush


# ----------------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------------

def run_ours(args, rank, world):
    import torch

    import ring_context_parallelism_gb300 as ra
    from ring_context_parallelism_gb300.build import build
    from ring_context_parallelism_gb300.inputs import WORKLOADS, attention_inputs, fanout_inputs

    if rank == 0 or not os.path.exists(os.path.join(ROOT, "ring_context_parallelism_gb300", "libra.so")):
        build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ra.load()
    pk = peaks()
    flush = make_flush()
    w = WORKLOADS[HEADLINE]
    q, k, v = attention_inputs(w, "cuda")
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.S, device="cuda", dtype=torch.float32)
    flops = ring_flops(w.B, w.S, w.Hq, w.D, w.causal)

    def step():
        ra.attn(q, k, v, w.n_shards, w.block, w.causal, out=out, lse=lse)

    result = {}
    with ClockSampler(torch.cuda.current_device()) as clk:
        # headline: K timed steps between barriers + syncs
        for _ in range(args.warmup):
            step()
        ra.device_status()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        ms = timed_steps(step, args.steps, 0, flush)
        ra.device_status()
        total_ms = max_over_ranks(sum(ms), world, "cuda")
        ms_step = total_ms / args.steps
        value = job_throughput(flops, args.steps, total_ms, world)

        # the same workload stored in the zigzag and striped shard layouts (same FLOPs)
        for lay in ("zigzag", "striped"):
            lms = timed_steps(lambda: ra.attn(q, k, v, w.n_shards, w.block, w.causal, out=out, lse=lse, layout=lay),
                              min(args.steps, 10), 3, flush)
            ra.device_status()
            t = statistics.median(lms) * 1e-3
            result.setdefault("layouts", {})[lay] = {
                "ms": t * 1e3, "TFLOP_per_s": flops / t / 1e12, "frac_bf16_peak": flops / t / 1e12 / pk["bf16_tflops"]}

        # backward pass on the same workload: dQ, dK, dV for a seeded upstream gradient
        gb = torch.Generator(device="cuda")
        gb.manual_seed(w.seed + 4242)
        from ring_context_parallelism_gb300.inputs import randn
        dO = randn(tuple(q.shape), gb, q.dtype, "cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = torch.empty(ra.load().ra_blockwise_attn_bwd_workspace_size(w.B, w.S, w.Hq, w.D, 1), dtype=torch.uint8,
                          device="cuda")
        bms = timed_steps(lambda: ra.attn_bwd(q, k, v, out, lse, dO, w.n_shards, w.block, w.causal, dq, dk, dv, bws),
                          min(args.steps, 10), 3, flush)
        ra.device_status()
        tb = statistics.median(bms) * 1e-3
        bflops = 2.5 * flops  # 5 GEMMs of the algorithm (QK^T, dO V^T, P^T dO, dS^T Q, dS K) vs 2 forward
        result["backward"] = {"ms": tb * 1e3, "TFLOP_per_s": bflops / tb / 1e12,
                              "frac_bf16_peak": bflops / tb / 1e12 / pk["bf16_tflops"], "flops": bflops,
                              "flop_convention": "2.5x the forward's causal-adjusted FLOPs (5 GEMMs); the kernels "
                                                 "execute 7 (dQ recomputes S and dP)",
                              "launches_per_call": 3}
        # the backward over the zigzag and striped layouts (same data in storage order, causal on positions)
        for lay in ("zigzag", "striped"):
            ra.attn(q, k, v, w.n_shards, w.block, w.causal, out=out, lse=lse, layout=lay)
            zms = timed_steps(lambda: ra.attn_bwd(q, k, v, out, lse, dO, w.n_shards, w.block, w.causal, dq, dk, dv,
                                                  bws, layout=lay), min(args.steps, 10), 3, flush)
            ra.device_status()
            tz = statistics.median(zms) * 1e-3
            result["backward"][lay] = {"ms": tz * 1e3, "TFLOP_per_s": bflops / tz / 1e12,
                                       "frac_bf16_peak": bflops / tz / 1e12 / pk["bf16_tflops"]}
        del dO, dq, dk, dv, bws

        # e2e through the public API with host buffers.  Every step copies its inputs from pinned
        # host memory and reads its O and lse back; steps are pipelined over three streams (the
        # next step's inputs in, this step's kernel, the previous step's results out) with two
        # device buffer sets, as a serving loop would.  Timed from the first copy to the last read.
        dev_index = torch.cuda.current_device()

        def host_buffers():
            hin = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (q, k, v)]
            for h, t in zip(hin, (q, k, v)):
                h.copy_(t)                                      # first touch on the GPU's node
            hout = [dict(oh=torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
                         lh=torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)) for _ in range(2)]
            for ho in hout:
                ho["oh"].zero_()
                ho["lh"].zero_()
            return hin, hout

        (hin, hout), numa_node, numa_cpus = pinned_on_gpu_node(dev_index, host_buffers)
        qh, kh, vh = hin
        slots = []
        for i in range(2):
            slots.append(dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                              o=torch.empty_like(out), l=torch.empty_like(lse), oh=hout[i]["oh"], lh=hout[i]["lh"],
                              in_done=torch.cuda.Event(), run_done=torch.cuda.Event(), out_done=torch.cuda.Event()))
        s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

        def e2e_steps(n):
            for i in range(n):
                sl = slots[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(sl["run_done"])        # step i-2's kernel has read this slot
                    sl["q"].copy_(qh, non_blocking=True)
                    sl["k"].copy_(kh, non_blocking=True)
                    sl["v"].copy_(vh, non_blocking=True)
                    sl["in_done"].record(s_in)
                with torch.cuda.stream(s_run):
                    s_run.wait_event(sl["in_done"])
                    if i >= 2:
                        s_run.wait_event(sl["out_done"])       # step i-2's results have left this slot
                    ra.attn(sl["q"], sl["k"], sl["v"], w.n_shards, w.block, w.causal, out=sl["o"], lse=sl["l"])
                    sl["run_done"].record(s_run)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(sl["run_done"])
                    sl["oh"].copy_(sl["o"], non_blocking=True)
                    sl["lh"].copy_(sl["l"], non_blocking=True)
                    sl["out_done"].record(s_out)

        h2d_bytes = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        d2h_bytes = slots[0]["oh"].numel() * slots[0]["oh"].element_size() + \
            slots[0]["lh"].numel() * slots[0]["lh"].element_size()

        def leg_gbs(copy, nbytes, reps=5):
            """One copy leg alone (host wall clock over reps copies): its own bandwidth."""
            copy()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(reps):
                copy()
            torch.cuda.synchronize()
            return nbytes * reps / (time.perf_counter() - t0) / 1e9

        sl0 = slots[0]
        h2d_gbs = leg_gbs(lambda: [d.copy_(h, non_blocking=True) for d, h in ((sl0["q"], qh), (sl0["k"], kh),
                                                                              (sl0["v"], vh))], h2d_bytes)
        d2h_gbs = leg_gbs(lambda: [h.copy_(d, non_blocking=True) for h, d in ((sl0["oh"], sl0["o"]),
                                                                              (sl0["lh"], sl0["l"]))], d2h_bytes)
        n_e2e = max(30, args.steps)
        e2e_steps(3)                                           # warm-up
        torch.cuda.synchronize()
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_steps(n_e2e)
        torch.cuda.synchronize()
        e2e_total_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, "cuda")
        ra.device_status()
        assert torch.equal(slots[0]["oh"], slots[1]["oh"])    # every step read back the same result
        e2e_ms = e2e_total_ms / n_e2e
        copy_ms = max(h2d_bytes / (h2d_gbs * 1e9), d2h_bytes / (d2h_gbs * 1e9)) * 1e3
        e2e = {"value": job_throughput(flops, n_e2e, e2e_total_ms, world), "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "steps": n_e2e,
               "pipelining": "3 streams (h2d, kernel, d2h), 2 device buffer sets; wall clock over all steps",
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "h2d_GB_per_s_alone": h2d_gbs, "d2h_GB_per_s_alone": d2h_gbs,
               "bound": "copies" if copy_ms > ms_step else "kernel",
               # the step against what bounds it: 1.0 when the copies hide fully behind the kernel
               # (or the kernel behind the copies)
               "pipeline_efficiency": max(copy_ms, ms_step) / e2e_ms,
               "host_numa_node": numa_node, "pinned_alloc_cpus": numa_cpus}
        del qh, kh, vh, slots, hin, hout

        # fan-out decode (config 4) and its R=16 sub-case
        for name in ("fanout_decode", "fanout_decode1"):
            fw = WORKLOADS[name]
            x = fanout_inputs(fw, "cuda")
            R = x["R"]
            fo = torch.empty_like(x["q_rows"])
            fl = torch.empty(fw.Hq, R, device="cuda", dtype=torch.float32)
            ws = torch.empty(ra.fanout_workspace_size(R, fw.n_branches, fw.S_prefix, fw.S_suffix, fw.Hq, fw.Hkv,
                                                      fw.D), dtype=torch.uint8, device="cuda")

            def fstep():
                ra.fanout(x["q_rows"], x["offsets"], x["k_prefix"], x["v_prefix"], x["k_suffix"], x["v_suffix"],
                          out=fo, lse=fl, workspace=ws)

            # direct calls, then the same call replayed from a captured CUDA graph
            # (a decode loop's form: no host work between steps)
            direct = statistics.median(timed_steps(fstep, 20, 5, flush)) * 1e-3
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                fstep()
            fms = timed_steps(graph.replay, 20, 5, flush)
            ra.device_status()
            t = statistics.median(fms) * 1e-3
            by = fanout_bytes(R, fw.n_branches, fw.Hq, fw.Hkv, fw.D, fw.S_prefix, fw.S_suffix)
            fl_ = fanout_flops(R, fw.Hq, fw.D, fw.S_prefix, fw.S_suffix)
            bound_t = max(by / (pk["hbm_gbs"] * 1e9), fl_ / (pk["bf16_tflops"] * 1e12))
            result[name] = {"R": R, "rows_per_branch": x["rows"], "us": t * 1e6, "timing": "CUDA graph replay",
                            "us_direct_call": direct * 1e6, "GB_per_s": by / t / 1e9,
                            "frac_hbm": by / t / 1e9 / pk["hbm_gbs"], "TFLOP_per_s": fl_ / t / 1e12,
                            "frac_binding_roofline": bound_t / t, "algorithmic_bytes": by, "flops": fl_,
                            "workspace_bytes": ws.numel(), "launches_per_call": 2}
            del x, fo, fl, ws, graph

        # the R = 16 decode mix over a paged KV cache (16-token pages, shuffled pool)
        fw = WORKLOADS["fanout_decode1"]
        x = fanout_inputs(fw, "cuda")
        R, P = x["R"], 16
        gp = torch.Generator(device="cpu").manual_seed(fw.seed + 99)
        npp, nsp = fw.S_prefix // P, fw.S_suffix // P
        n_pages = npp + fw.n_branches * nsp
        order = torch.randperm(n_pages, generator=gp).to(torch.int32).cuda()
        pp, sp = order[:npp].contiguous(), order[npp:].reshape(fw.n_branches, nsp).contiguous()
        kpool = torch.empty(n_pages, P, fw.Hkv, fw.D, dtype=x["k_prefix"].dtype, device="cuda")
        vpool = torch.empty_like(kpool)
        kpool[pp.long()] = x["k_prefix"].reshape(npp, P, fw.Hkv, fw.D)
        vpool[pp.long()] = x["v_prefix"].reshape(npp, P, fw.Hkv, fw.D)
        kpool[sp.long().reshape(-1)] = x["k_suffix"].reshape(-1, P, fw.Hkv, fw.D)
        vpool[sp.long().reshape(-1)] = x["v_suffix"].reshape(-1, P, fw.Hkv, fw.D)
        fo = torch.empty_like(x["q_rows"])
        fl = torch.empty(fw.Hq, R, device="cuda", dtype=torch.float32)
        ws = torch.empty(ra.fanout_workspace_size(R, fw.n_branches, fw.S_prefix, fw.S_suffix, fw.Hq, fw.Hkv, fw.D),
                         dtype=torch.uint8, device="cuda")
        gms = timed_steps(lambda: ra.fanout_paged(x["q_rows"], x["offsets"], kpool, vpool, pp, fw.S_prefix, sp,
                                                  fw.S_suffix, out=fo, lse=fl, workspace=ws), 20, 5, flush)
        ra.device_status()
        t = statistics.median(gms) * 1e-3
        by = fanout_bytes(R, fw.n_branches, fw.Hq, fw.Hkv, fw.D, fw.S_prefix, fw.S_suffix)
        result["fanout_decode1_paged16"] = {"R": R, "page_size": P, "us": t * 1e6, "GB_per_s": by / t / 1e9,
                                            "frac_hbm": by / t / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": by,
                                            "launches_per_call": 2}
        del x, kpool, vpool, fo, fl, ws

        # fan-out prefill: 8 branches x 20 new rows, causal inside each 512-token private suffix
        fw = WORKLOADS["fanout_prefill_8x20"]
        x = fanout_inputs(fw, "cuda")
        R = x["R"]
        fo = torch.empty_like(x["q_rows"])
        fl = torch.empty(fw.Hq, R, device="cuda", dtype=torch.float32)
        ws = torch.empty(ra.fanout_workspace_size(R, fw.n_branches, fw.S_prefix, fw.S_suffix, fw.Hq, fw.Hkv, fw.D),
                         dtype=torch.uint8, device="cuda")
        pms = timed_steps(lambda: ra.fanout(x["q_rows"], x["offsets"], x["k_prefix"], x["v_prefix"], x["k_suffix"],
                                            x["v_suffix"], out=fo, lse=fl, workspace=ws, prefill=True), 20, 5, flush)
        ra.device_status()
        t = statistics.median(pms) * 1e-3
        n_b = x["rows"][0]
        pf = fanout_prefill_flops(x["rows"], fw.Hq, fw.D, fw.S_prefix, fw.S_suffix)
        by = fanout_bytes(R, fw.n_branches, fw.Hq, fw.Hkv, fw.D, fw.S_prefix, fw.S_suffix)
        result["fanout_prefill_8x20"] = {"R": R, "rows_per_branch": n_b, "us": t * 1e6, "TFLOP_per_s": pf / t / 1e12,
                                         "frac_bf16_peak": pf / t / 1e12 / pk["bf16_tflops"],
                                         "GB_per_s": by / t / 1e9, "flops": pf, "algorithmic_bytes": by,
                                         "launches_per_call": 2}
        del x, fo, fl, ws

        # per-shard partials + LSE merge on the Llama-3-70B-shaped layer
        pw = WORKLOADS["llama70b_layer_128k_partials"]
        del q, k, v, out, lse
        torch.cuda.empty_cache()
        pq, pkk, pv = attention_inputs(pw, "cuda")
        pO = torch.empty((pw.n_shards, pw.B, pw.S, pw.Hq, pw.D), device="cuda", dtype=pq.dtype)
        pL = torch.empty((pw.n_shards, pw.B, pw.Hq, pw.S), device="cuda", dtype=torch.float32)
        mO = torch.empty_like(pq)
        mL = torch.empty(pw.B, pw.Hq, pw.S, device="cuda", dtype=torch.float32)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        times = []
        for it in range(3):
            flush()
            ev[0].record()
            ra.ring_partials(pq, pkk, pv, pw.n_shards, pw.block, pw.causal, partials_O=pO, partials_lse=pL)
            ev[1].record()
            ra.lse_merge(pO, pL, out=mO, out_lse=mL)
            ev[2].record()
            torch.cuda.synchronize()
            if it > 0:
                times.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
        ra.device_status()
        pf = ring_flops(pw.B, pw.S, pw.Hq, pw.D, pw.causal)
        tp = statistics.mean(t[0] for t in times) * 1e-3
        tm = statistics.mean(t[1] for t in times) * 1e-3
        mb = merge_bytes(pw.n_shards, pw.B, pw.S, pw.Hq, pw.D, causal=pw.causal)
        result["llama70b_layer_128k_partials"] = {
            "partials_ms": tp * 1e3, "partials_TFLOP_per_s": pf / tp / 1e12,
            "merge_ms": tm * 1e3, "merge_GB_per_s": mb / tm / 1e9, "merge_frac_hbm": mb / tm / 1e9 / pk["hbm_gbs"],
            "pipeline_ms": (tp + tm) * 1e3, "pipeline_TFLOP_per_s": pf / (tp + tm) / 1e12, "flops": pf,
            "partials_bytes": pO.numel() * 2 + pL.numel() * 4}
        # the same layer in one fused pass (ra_blockwise_attn_fwd, no partials)
        fms = timed_steps(lambda: ra.attn(pq, pkk, pv, pw.n_shards, pw.block, pw.causal, out=mO, lse=mL), 2, 1, flush)
        ra.device_status()
        tf = statistics.mean(fms) * 1e-3
        result["llama70b_layer_128k_partials"].update(
            {"fused_ms": tf * 1e3, "fused_TFLOP_per_s": pf / tf / 1e12, "fused_frac_bf16_peak": pf / tf / 1e12 / pk["bf16_tflops"]})
        del pq, pkk, pv, pO, pL, mO, mL
        torch.cuda.empty_cache()

        # the tiny exact workload (fp32 inputs, fp32 CUDA-core path; latency-bound, time only)
        tw = WORKLOADS["tiny_exact_f32"]
        tq, tk, tv = attention_inputs(tw, "cuda")
        tms = timed_steps(lambda: ra.attn(tq, tk, tv, tw.n_shards, tw.block, tw.causal), 20, 5)
        ra.device_status()
        result["tiny_exact_f32"] = {"ms": statistics.median(tms),
                                    "TFLOP_per_s": ring_flops(tw.B, tw.S, tw.Hq, tw.D, tw.causal) /
                                                   (statistics.median(tms) * 1e-3) / 1e12}
        del tq, tk, tv

        # the million-token stress workload (1% of keys x8): one untimed call, then two timed ones
        if not args.no_stress:
            sw = WORKLOADS["million_token_stress"]
            sq, sk, sv = attention_inputs(sw, "cuda")
            so = torch.empty_like(sq)
            sl = torch.empty(sw.B, sw.Hq, sw.S, device="cuda", dtype=torch.float32)
            sms = timed_steps(lambda: ra.attn(sq, sk, sv, sw.n_shards, sw.block, True, out=so, lse=sl), 2, 1)
            ra.device_status()
            sf = ring_flops(sw.B, sw.S, sw.Hq, sw.D, True)
            ts = statistics.mean(sms) * 1e-3
            result["million_token_stress"] = {"s": ts, "s_per_call": sms, "TFLOP_per_s": sf / ts / 1e12,
                                              "frac_bf16_peak": sf / ts / 1e12 / pk["bf16_tflops"],
                                              "frac_of_sustained": sf / ts / 1e12 / pk["bf16_tflops_sustained"],
                                              "flops": sf, "S": sw.S, "n_shards": sw.n_shards}
            del sq, sk, sv, so, sl
            torch.cuda.empty_cache()

    clocks = clk.summary()
    achieved = flops / (ms_step * 1e-3) / 1e12
    kh = kernel_hash()
    traffic = NCU_TRAFFIC.get(kh)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic: seeded N(0,1) bf16 inputs",
        "config": {"workload": HEADLINE, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "n_shards": w.n_shards, "block": w.block, "causal": w.causal, "flops_per_step": flops,
                   "l2": "flushed before every step (512 MB write, then a 256 MB read); inputs 402 MB > L2",
                   "parallelism": f"replicas x{world}"},
        "pct_bf16_peak": 100.0 * achieved / pk["bf16_tflops"],
        "roofline": {"kernel": "attn_tc_kernel<128>", "bound": "tensor", "achieved": achieved,
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                     "peak_source": pk["source"] + " (burst)",
                     "frac_of_sustained": achieved / pk["bf16_tflops_sustained"],
                     "traffic": traffic, "algorithmic_bytes": ring_bytes(w.B, w.S, w.Hq, w.Hkv, w.D),
                     "kernel_hash": kh},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    line.update(result)
    return line


# ----------------------------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ----------------------------------------------------------------------------------------------

def oracle_sample_rate(target_s=10.0, max_queries=1 << 16, seed=0):
    """Times the fp64 oracle on seeded query samples of the headline workload
    until about target_s seconds of CPU work; returns (TFLOP/s, seconds,
    queries, cores)."""
    import numpy as np
    import torch

    import oracle
    from ring_context_parallelism_gb300.inputs import WORKLOADS, attention_inputs

    w = WORKLOADS[HEADLINE]
    # the headline workload's shapes and seed, drawn on the host
    q, k, v = attention_inputs(w, "cpu")
    qs = q.view(torch.int16).numpy().view(np.uint16)
    ks = k.view(torch.int16).numpy().view(np.uint16)
    vs = v.view(torch.int16).numpy().view(np.uint16)
    cores = oracle.max_threads()
    n = 256
    done_q, done_flops, spent = 0, 0, 0.0
    rng = np.random.default_rng(seed)
    while spent < target_s and done_q < max_queries:
        ids = np.sort(rng.choice(w.B * w.S * w.Hq, size=n, replace=False)).astype(np.int64)
        rows = (ids // w.Hq) % w.S
        t0 = time.perf_counter()
        oracle.attention(qs, ks, vs, dtype="bf16", causal=w.causal, sel=ids)
        dt = time.perf_counter() - t0
        spent += dt
        done_q += n
        done_flops += int(4 * w.D * (rows + 1).sum())
        if dt < target_s / 8:
            n *= 2
    return done_flops / spent / 1e12, spent, done_q, cores


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle, timed per step on a bounded
    sample of the headline workload's queries."""
    per_step = []
    cores = None
    queries = 0
    for i in range(args.warmup + args.steps):
        rate, spent, nq, cores = oracle_sample_rate(target_s=2.0, max_queries=4096, seed=i)
        if i >= args.warmup:
            per_step.append((rate, spent, nq))
            queries += nq
    value = statistics.mean(r for r, _, _ in per_step)
    ms = statistics.mean(s for _, s, _ in per_step) * 1e3
    sample = (f"{queries} seeded (row, head) queries of {HEADLINE} over {args.steps} steps "
              f"(about 2 s of CPU work per step); FLOPs counted as 4*D per visible key")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic: seeded N(0,1) bf16 inputs",
            "config": {"workload": HEADLINE}, "gpu_launches": 0,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


PROFILE_CASES = ("prefill_32k", "prefill_16k", "fanout_decode", "fanout_decode1", "merge_16k", "bwd_16k",
                 "prefill_32k_zigzag", "prefill_32k_striped", "fanout_prefill_8x20", "fanout_decode1_paged16",
                 "bwd_16k_zigzag")


def run_profile_case(case):
    """Three calls of one kernel family on a case sized for an ncu capture
    (inputs larger than L2, a few GB on the device at most)."""
    import torch

    import ring_context_parallelism_gb300 as ra
    from ring_context_parallelism_gb300.build import build
    from ring_context_parallelism_gb300.inputs import WORKLOADS, attention_inputs, fanout_inputs, small

    build()
    ra.load()
    if case in ("prefill_32k", "prefill_16k"):
        # prefill_32k is the timed headline configuration itself (0.6 GB on the device, ~7 ms a launch)
        w = WORKLOADS[HEADLINE] if case == "prefill_32k" else small(WORKLOADS[HEADLINE], S=16384)
        q, k, v = attention_inputs(w, "cuda")
        o = torch.empty_like(q)
        l = torch.empty(w.B, w.Hq, w.S, device="cuda")
        for _ in range(3):
            ra.attn(q, k, v, w.n_shards, w.block, True, out=o, lse=l)
    elif case in ("prefill_32k_zigzag", "prefill_32k_striped"):
        # the headline configuration stored in a zigzag or striped shard layout (same data, same FLOPs)
        w = WORKLOADS[HEADLINE]
        q, k, v = attention_inputs(w, "cuda")
        o = torch.empty_like(q)
        l = torch.empty(w.B, w.Hq, w.S, device="cuda")
        for _ in range(3):
            ra.attn(q, k, v, w.n_shards, w.block, True, out=o, lse=l, layout=case.rsplit("_", 1)[1])
    elif case == "fanout_prefill_8x20":
        w = WORKLOADS[case]
        x = fanout_inputs(w, "cuda")
        for _ in range(3):
            ra.fanout(x["q_rows"], x["offsets"], x["k_prefix"], x["v_prefix"], x["k_suffix"], x["v_suffix"],
                      prefill=True)
    elif case == "fanout_decode1_paged16":
        # the R = 16 decode mix with its KV scattered over a shuffled pool of 16-token pages
        w = WORKLOADS["fanout_decode1"]
        x = fanout_inputs(w, "cuda")
        P = 16
        npp, nsp = w.S_prefix // P, w.S_suffix // P
        n_pages = npp + w.n_branches * nsp
        order = torch.randperm(n_pages, generator=torch.Generator().manual_seed(w.seed + 99)).to(torch.int32).cuda()
        pp, sp = order[:npp].contiguous(), order[npp:].reshape(w.n_branches, nsp).contiguous()
        kpool = torch.empty(n_pages, P, w.Hkv, w.D, dtype=x["k_prefix"].dtype, device="cuda")
        vpool = torch.empty_like(kpool)
        kpool[pp.long()] = x["k_prefix"].reshape(npp, P, w.Hkv, w.D)
        vpool[pp.long()] = x["v_prefix"].reshape(npp, P, w.Hkv, w.D)
        kpool[sp.long().reshape(-1)] = x["k_suffix"].reshape(-1, P, w.Hkv, w.D)
        vpool[sp.long().reshape(-1)] = x["v_suffix"].reshape(-1, P, w.Hkv, w.D)
        for _ in range(3):
            ra.fanout_paged(x["q_rows"], x["offsets"], kpool, vpool, pp, w.S_prefix, sp, w.S_suffix)
    elif case in ("fanout_decode", "fanout_decode1"):
        w = WORKLOADS[case]
        x = fanout_inputs(w, "cuda")
        ws = torch.empty(ra.fanout_workspace_size(x["R"], w.n_branches, w.S_prefix, w.S_suffix, w.Hq, w.Hkv, w.D),
                         dtype=torch.uint8, device="cuda")
        for _ in range(3):
            ra.fanout(x["q_rows"], x["offsets"], x["k_prefix"], x["v_prefix"], x["k_suffix"], x["v_suffix"],
                      workspace=ws)
    elif case in ("bwd_16k", "bwd_16k_zigzag"):
        # backward of the causal GQA workload at 16384 tokens (Hq 32, Hkv 8, D 128), contiguous
        # or with the rows in the zigzag layout: 3 calls
        from ring_context_parallelism_gb300.inputs import randn
        lay = "zigzag" if case.endswith("zigzag") else "contiguous"
        w = small(WORKLOADS[HEADLINE], S=16384)
        q, k, v = attention_inputs(w, "cuda")
        o, l = ra.attn(q, k, v, w.n_shards, w.block, True, layout=lay)
        g = torch.Generator(device="cuda")
        g.manual_seed(w.seed + 4242)
        dO = randn(tuple(q.shape), g, q.dtype, "cuda")
        for _ in range(3):
            ra.attn_bwd(q, k, v, o, l, dO, w.n_shards, w.block, True, layout=lay)
    elif case == "merge_16k":
        # per-shard partials of a 16384-token, 64-head causal layer (16 shards), then 3 merges
        w = small(WORKLOADS["llama70b_layer_128k_partials"], S=16384)
        q, k, v = attention_inputs(w, "cuda")
        pO, pL = ra.ring_partials(q, k, v, w.n_shards, w.block, True)
        for _ in range(3):
            ra.lse_merge(pO, pL)
    torch.cuda.synchronize()
    ra.device_status()
    print(json.dumps({"profile_case": case, "ok": True}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stress", action="store_true",
                    help="skip the million-token stress workload (e.g. for a launch-list capture under ncu)")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="run three calls of one kernel family on a small case (for ncu captures) and exit")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    import torch

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_ours(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, spent, nq, cores = oracle_sample_rate()
        line["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": f"{nq} seeded (row, head) queries of {HEADLINE}, {spent:.1f} s of "
                                          f"CPU work; FLOPs counted as 4*D per visible key"}
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
