"""Benchmark of the kernelised linear attention library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one causal forward (phi feature map,
intra-chunk masked products, inter-chunk state read-out, state carry, final
state written out) over the training-shaped workload B=16, H=8, N=3072,
D=M=64, bf16 inputs N(0,1)/sqrt(64): `value` is tokens/s (B*N per step) with
inputs resident in HBM.  No step finds its inputs in L2: each workload's
per-step data rotates over enough copies to exceed 2.5 x L2 (steps back to
back, no flush), and the JSON says how many.  The same
line carries the other legs of the metric as separate objects: decode
steps/s with the state's HBM GB/s (B=256, H=16, D=M=64 after a 1024-token
prefill), the non-causal forward (B=8, H=8, N=4096) and the long causal
forward (B=1, H=16, N=65536, D=M=128).

--impl reference times the fp64 CPU oracle (the only reference there is) on
a bounded sample of the same workload.  Under torchrun each rank runs the
same per-GPU workload on its own GPU (independent heads: weak scaling, no
collective in the data path); timings are reduced with MAX over ranks.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MAIN = "causal_b16h8n3072d64"
METRIC = "causal linear-attn fwd tokens/s & % tensor roofline; decode steps/s & HBM GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if self.t0 is None or (self.t0 - 0.05 <= t <= (self.t1 or t) + 0.05)]
        if not rows:
            rows = [l for (_, l) in self.lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in rows:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
            except ValueError:
                continue
            for n, val in zip(names, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers

# Source files each captured kernel is built from: a capture's traffic figure
# stands only while these hash to what they were when it was taken.
TC_SOURCES = ("la_tc.cu", "tc_kernels.cuh", "tc_ptx.cuh", "tc_host.h", "la_common.cuh", "la_internal.h")
KERNEL_SOURCES = {
    "causal_causal_b16h8n3072d64": TC_SOURCES,
    "causal_causal_b1h16n65536d128": TC_SOURCES,
    "noncausal_noncausal_b8h8n4096d64": TC_SOURCES,
    "causal_variant_dpfp_b16h8n3072d64": TC_SOURCES,
    "decode_decode_b256h16d64": ("la_simt.cu", "la_common.cuh", "la_internal.h"),
    "causal_variant_delta_b16h8n3072d64": ("la_tc_delta.cu", "tc_kernels.cuh", "tc_ptx.cuh", "tc_host.h",
                                           "la_common.cuh", "la_internal.h"),
    "backward_causal_b16h8n3072d64": ("la_tc_bwd.cu", "tc_kernels.cuh", "tc_ptx.cuh", "tc_host.h", "la_common.cuh",
                                      "la_internal.h"),
    # key sums (la_tc.cu), then the query and key passes
    "backward_nc_causal_b16h8n3072d64": ("la_tc_bwd_nc.cu", "tc_bwd_common.cuh", "la_tc.cu", "tc_kernels.cuh",
                                         "tc_ptx.cuh", "tc_host.h", "la_common.cuh", "la_internal.h"),
    # per-chunk key sums (la_tc.cu), two scans, the query and key passes
    "backward_causal_b1h16n65536d128": ("la_tc_bwd_chunk.cu", "tc_bwd_common.cuh", "la_tc.cu", "tc_kernels.cuh",
                                        "tc_ptx.cuh", "tc_host.h", "la_common.cuh", "la_internal.h"),
}


def _kernel_source_hash(kernel_key):
    """sha256 (first 16 hex digits) of the kernel's source files, in the listed order."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES.get(kernel_key, ()):
        with open(os.path.join(ROOT, "weight_recurrence_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel_key):
    """ncu DRAM bytes per launch recorded in profiles/traffic.json, if taken on this source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(kernel_key)
        if e and kernel_key in KERNEL_SOURCES and e.get("source_sha") == _kernel_source_hash(kernel_key):
            return e.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


class Rotation:
    """Keeps timed steps reading their inputs from HBM with no flush: a
    workload's per-step data (inputs, outputs, and a state the step rewrites)
    is replicated into n copies totalling more than 2.5 x L2, and step i uses
    copy i % n, steps back to back.  A copy was last touched n - 1 steps
    earlier, so its lines have left L2; each step also pays for the write-back
    of earlier steps' outputs, as in a steady stream of calls."""

    def __init__(self, torch, device):
        l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20) or (128 << 20)
        self.l2 = int(l2)

    def copies(self, nbytes):
        return max(1, int(math.ceil(2.5 * self.l2 / max(1, nbytes))))

    def describe(self, nbytes):
        n = self.copies(nbytes)
        if n == 1:
            return ("no flush: inputs %.0f MB exceed 2.5 x the %.0f MB L2; steps run back to back"
                    % (nbytes / 1e6, self.l2 / 1e6))
        return ("no flush: inputs rotate over %d copies (%d x %.0f MB > 2.5 x the %.0f MB L2), steps back to back"
                % (n, n, nbytes / 1e6, self.l2 / 1e6))


def _rotating(torch, tensors, n):
    """n sets of `tensors`: the originals, then n - 1 copies (None stays None)."""
    sets = [list(tensors)]
    for _ in range(n - 1):
        sets.append([None if t is None else t.clone() for t in tensors])
    return sets


def _timed_steps(torch, fn, steps, warmup, stream):
    """Mean time per step (ms): one CUDA-event pair on `stream` around `steps`
    steps issued back to back (an event between two launches would hold the
    second until the first has drained, hiding nothing of its set-up)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def _alg_bytes_fwd(w):
    """Algorithmic bytes of one forward: read Q, K, V once, write O once."""
    el = 2 if str(w.dtype).endswith("bfloat16") else 4
    return w.B * w.H * w.N * (2 * w.D + 2 * w.M) * el


def _alg_flops_fwd(w):
    """4*D*M flops per head-token: state update (2DM) + read-out (2DM)."""
    return 4.0 * w.D * w.M * w.B * w.H * w.N


def _exec_flops_causal(w, chunk):
    """Flops the chunked kernel executes: intra-chunk 2C(D+M) + inter 2DM + update 2DM per head-token."""
    return (2.0 * chunk * (w.D + w.M) + 4.0 * w.D * w.M) * w.B * w.H * w.N


# -------------------------------------------------------------- our arm

def main_config(w, world, l2):
    """The `config` object of the main line (both arms)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "M": w.M, "chunk": w.chunk,
            "chunk_note": "passed as chunk=64; the library takes it as a hint and its tcgen05 path groups "
                          "128 rows (one M=128 tile): the same sums in exact arithmetic",
            "global_batch": w.B * world, "seq_len": w.N,
            "parallelism": "dp%d (independent heads per rank)" % world, "l2": l2}


def run_ours(args, rank, world, dist):
    import torch

    from weight_recurrence_gb300 import build as labuild
    from weight_recurrence_gb300 import inputs, la, ranks

    labuild.build()
    local = _env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    pk = peaks()
    rot = Rotation(torch, dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    def max_over_ranks(x):
        return ranks.reduce_max(x, dist, dev)

    if args.only:
        # one workload alone, for profiler captures: no clocks, e2e or CPU legs
        if args.only.startswith("backward_nc_"):
            leg = _leg_backward(torch, la, inputs, args.only[len("backward_nc_"):], dev, stream, rot, pk,
                                args.steps, max_over_ranks, world, rank, warmup=args.warmup, noncausal=True)
            return {"only": args.only, "leg": leg, "gpu_launches_total": la.la_launch_count()}
        if args.only.startswith("backward_"):
            leg = _leg_backward(torch, la, inputs, args.only[len("backward_"):], dev, stream, rot, pk,
                                args.steps, max_over_ranks, world, rank, warmup=args.warmup)
            return {"only": args.only, "leg": leg, "gpu_launches_total": la.la_launch_count()}
        w = inputs.WORKLOADS[args.only]
        if w.op == "causal_variant":
            leg = _leg_variant(torch, la, inputs, args.only, dev, stream, rot, pk, args.steps, max_over_ranks,
                               world, rank, warmup=args.warmup)
        elif w.op == "decode":
            leg = _leg_decode(torch, la, inputs, dev, stream, rot, pk, args, max_over_ranks, world, rank)
        else:
            leg = _leg_fwd(torch, la, inputs, args.only, dev, stream, rot, pk, args.steps, max_over_ranks,
                           world, rank, warmup=args.warmup)
        return {"only": args.only, "leg": leg, "gpu_launches_total": la.la_launch_count()}

    # ---------------------------------------------------- main: causal cfg
    w = inputs.WORKLOADS[MAIN]
    q, k, v = [t.to(dev) for t in inputs.workload_inputs(w, rank)]
    S = torch.zeros(w.B, w.H, w.D, w.M, device=dev)
    z = torch.zeros(w.B, w.H, w.D, device=dev)
    out = torch.empty(w.B, w.H, w.N, w.M, dtype=w.dtype, device=dev)
    in_bytes = 3 * q.numel() * q.element_size()
    sets = _rotating(torch, (q, k, v, out), rot.copies(in_bytes))
    it = [0]

    # Each step continues from the state the previous one left (S, z in/out),
    # exactly as consecutive segments of one long sequence would.
    def step():
        q_, k_, v_, o_ = sets[it[0] % len(sets)]
        it[0] += 1
        la.la_forward_causal(q_, k_, v_, out=o_, chunk=w.chunk, S=S, z=z, stream=stream)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    l0 = la.la_launch_count()
    sampler.mark(True)
    t_wall0 = time.perf_counter()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    sampler.mark(False)
    barrier()
    torch.cuda.synchronize()
    launches = la.la_launch_count() - l0
    assert la.la_get_last_error() == la.LA_OK
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms = max_over_ranks(ms_local)
    clocks = sampler.stop()
    tokens_per_step = w.B * w.N
    value = ranks.whole_job_rate(tokens_per_step, world, ms / 1e3)
    launches_per_call = launches / max(1, args.steps)
    bytes_step = _alg_bytes_fwd(w)
    achieved_gbs = bytes_step / (ms / 1e3) / 1e9
    chunk_exec = 128   # the tensor-core path's row grouping, whatever chunk hint is passed
    roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved_gbs / pk["hbm_gbs"], 4), "traffic": _traffic("causal_" + MAIN),
                "peak_source": pk["source"], "alg_bytes_per_launch": bytes_step,
                "launches_per_step": launches_per_call}
    tensor = {"alg_tflops": round(_alg_flops_fwd(w) / (ms / 1e3) / 1e12, 2),
              "exec_tflops": round(_exec_flops_causal(w, chunk_exec) / (ms / 1e3) / 1e12, 2),
              "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
              "frac_alg": round(_alg_flops_fwd(w) / (ms / 1e3) / 1e12 / pk["bf16_tflops"], 4),
              "frac_exec": round(_exec_flops_causal(w, chunk_exec) / (ms / 1e3) / 1e12 / pk["bf16_tflops"], 4),
              "note": "at D=M=64 the causal forward is HBM-bound (32 flop/B algorithmic vs ~287 flop/B "
                      "machine balance); the HBM fraction is the governing roofline"}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)/sqrt(D) bf16; no dataset)",
        "config": main_config(w, world, rot.describe(in_bytes)),
        "roofline": roofline, "tensor": tensor, "clocks": clocks, "gpu_launches": launches,
        "wall_s_timed_region": round(t_wall1 - t_wall0, 4),
    }

    # ---------------------------------------------- e2e: host buffers
    if not args.no_e2e:
        qh = q.cpu().pin_memory()
        kh = k.cpu().pin_memory()
        vh = v.cpu().pin_memory()
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        qd, kd, vd = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        # The batch goes through in slices of sequences, pipelined over three
        # streams: slice i's inputs copy in while slice i-1 computes and slice
        # i-2's output copies out (each slice is one la_forward_causal call
        # on its own sequences and their state).
        n_slices = 4 if w.B % 4 == 0 else 1
        bs = w.B // n_slices
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_step():
            start = torch.cuda.Event()
            start.record(stream)
            s_in.wait_event(start)
            s_out.wait_event(start)
            done_out = None
            for i in range(n_slices):
                b0, b1 = i * bs, (i + 1) * bs
                ev_in, ev_c = torch.cuda.Event(), torch.cuda.Event()
                with torch.cuda.stream(s_in):
                    qd[b0:b1].copy_(qh[b0:b1], non_blocking=True)
                    kd[b0:b1].copy_(kh[b0:b1], non_blocking=True)
                    vd[b0:b1].copy_(vh[b0:b1], non_blocking=True)
                    ev_in.record(s_in)
                stream.wait_event(ev_in)
                la.la_forward_causal(qd[b0:b1], kd[b0:b1], vd[b0:b1], out=out[b0:b1], chunk=w.chunk,
                                     S=S[b0:b1], z=z[b0:b1], stream=stream)
                ev_c.record(stream)
                s_out.wait_event(ev_c)
                with torch.cuda.stream(s_out):
                    oh[b0:b1].copy_(out[b0:b1], non_blocking=True)
                    done_out = torch.cuda.Event()
                    done_out.record(s_out)
            stream.wait_event(done_out)

        n_e2e = max(3, min(args.steps, 20))
        et = _timed_steps(torch, e2e_step, n_e2e, 2, stream)
        e_ms = max_over_ranks(et)
        nb = q.numel() * q.element_size()
        result["e2e"] = {"value": round(world * tokens_per_step / (e_ms / 1e3), 1), "unit": "tokens/s",
                         "h2d_bytes_per_step": 3 * nb, "d2h_bytes_per_step": out.numel() * out.element_size(),
                         "ms_per_step": round(e_ms, 4), "steps": n_e2e,
                         "path": "pinned host -> device copies, la_forward_causal, device -> pinned host; "
                                 "%d batch slices pipelined over copy-in, compute and copy-out streams" % n_slices}
    del q, k, v, out, sets

    # ------------------------------------------------- secondary legs
    if not args.main_only:
        result["legs"] = {}
        result["legs"]["noncausal"] = _leg_fwd(torch, la, inputs, "noncausal_b8h8n4096d64", dev, stream,
                                               rot, pk, 30, max_over_ranks, world, rank)
        result["legs"]["long_causal"] = _leg_fwd(torch, la, inputs, "causal_b1h16n65536d128", dev, stream,
                                                 rot, pk, 5, max_over_ranks, world, rank)
        result["legs"]["decode"] = _leg_decode(torch, la, inputs, dev, stream, rot, pk, args,
                                               max_over_ranks, world, rank)
        result["legs"]["backward"] = _leg_backward(torch, la, inputs, MAIN, dev, stream, rot, pk, 5,
                                                   max_over_ranks, world, rank)
        result["legs"]["backward_noncausal"] = _leg_backward(torch, la, inputs, MAIN, dev, stream, rot, pk, 5,
                                                             max_over_ranks, world, rank, noncausal=True)
        result["legs"]["backward_long"] = _leg_backward(torch, la, inputs, "causal_b1h16n65536d128", dev, stream,
                                                        rot, pk, 5, max_over_ranks, world, rank)
        for name in ("delta_b16h8n3072d64", "dpfp_b16h8n3072d64"):
            result["legs"][name.split("_")[0]] = _leg_variant(torch, la, inputs, name, dev, stream, rot, pk, 5,
                                                              max_over_ranks, world, rank)

    # ------------------------------------------------- CPU baselines (rank 0)
    if rank == 0 and not args.no_cpu:
        cs = args.cpu_seconds
        result["cpu_baseline"] = cpu_baseline(w, budget_s=cs)
        legs = result.get("legs", {})
        if "noncausal" in legs:
            legs["noncausal"]["cpu_baseline"] = cpu_baseline(inputs.WORKLOADS["noncausal_b8h8n4096d64"], budget_s=cs)
        if "long_causal" in legs:
            # all 16 heads over their first 8192 tokens (the recurrence costs the same per token)
            legs["long_causal"]["cpu_baseline"] = cpu_baseline(inputs.WORKLOADS["causal_b1h16n65536d128"],
                                                               budget_s=cs, heads=16, rows=8192)
        if "decode" in legs:
            legs["decode"]["cpu_baseline"] = cpu_baseline_decode(inputs.WORKLOADS["decode_b256h16d64"], budget_s=cs)
        if "backward" in legs:
            legs["backward"]["cpu_baseline"] = cpu_baseline_backward(w, budget_s=cs)
        if "backward_noncausal" in legs:
            legs["backward_noncausal"]["cpu_baseline"] = cpu_baseline_backward(w, budget_s=cs, noncausal=True)
        if "backward_long" in legs:
            # all 16 heads over their first 4096 tokens (the recurrence costs the same per token)
            legs["backward_long"]["cpu_baseline"] = cpu_baseline_backward(inputs.WORKLOADS["causal_b1h16n65536d128"],
                                                                          budget_s=cs, rows=4096)
        for name in ("delta_b16h8n3072d64", "dpfp_b16h8n3072d64"):
            key = name.split("_")[0]
            if key in legs:
                legs[key]["cpu_baseline"] = cpu_baseline_variant(inputs.WORKLOADS[name], budget_s=cs)
    return result


def _leg_fwd(torch, la, inputs, name, dev, stream, rot, pk, steps, max_over_ranks, world, rank, warmup=3):
    w = inputs.WORKLOADS[name]
    q, k, v = [t.to(dev) for t in inputs.workload_inputs(w, rank)]
    out = torch.empty(w.B, w.H, w.N, w.M, dtype=w.dtype, device=dev)
    in_bytes = 3 * q.numel() * q.element_size()
    sets = _rotating(torch, (q, k, v, out), rot.copies(in_bytes))
    it = [0]

    def fn():
        q_, k_, v_, o_ = sets[it[0] % len(sets)]
        it[0] += 1
        if w.op == "causal":
            la.la_forward_causal(q_, k_, v_, out=o_, chunk=w.chunk, stream=stream)
        else:
            la.la_forward_noncausal(q_, k_, v_, out=o_, stream=stream)

    l0 = la.la_launch_count()
    t = _timed_steps(torch, fn, steps, warmup, stream)
    launches = (la.la_launch_count() - l0) // (steps + warmup)
    ms = max_over_ranks(t)
    gbs = _alg_bytes_fwd(w) / (ms / 1e3) / 1e9
    leg = {"workload": name, "op": w.op, "value": round(world * w.B * w.N / (ms / 1e3), 1), "unit": "tokens/s",
           "ms_per_step": round(ms, 5), "steps": steps, "launches_per_step": launches,
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": round(gbs / pk["hbm_gbs"], 4), "traffic": _traffic(w.op + "_" + name)},
           "alg_tflops": round(_alg_flops_fwd(w) / (ms / 1e3) / 1e12, 2), "l2": rot.describe(in_bytes)}
    del q, k, v, out, sets
    torch.cuda.empty_cache()
    return leg


def _leg_backward(torch, la, inputs, name, dev, stream, rot, pk, steps, max_over_ranks, world, rank, warmup=3,
                  noncausal=False):
    """Causal (or non-causal) backward, dQ, dK, dV from dL/dV', on a forward workload's shape."""
    w = inputs.WORKLOADS[name]
    q, k, v = [t.to(dev) for t in inputs.workload_inputs(w, rank)]
    g = torch.Generator(device=dev).manual_seed(inputs.rank_seed(w.seed + 2000, rank))
    G = torch.randn(v.shape, generator=g, device=dev).to(w.dtype)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    in_bytes = 4 * q.numel() * q.element_size()
    sets = _rotating(torch, (q, k, v, G, dq, dk, dv), rot.copies(in_bytes))
    it = [0]

    def fn():
        q_, k_, v_, G_, dq_, dk_, dv_ = sets[it[0] % len(sets)]
        it[0] += 1
        if noncausal:
            la.la_backward_noncausal(q_, k_, v_, G_, dq=dq_, dk=dk_, dv=dv_, stream=stream)
        else:
            la.la_backward_causal(q_, k_, v_, G_, dq=dq_, dk=dk_, dv=dv_, stream=stream)

    l0 = la.la_launch_count()
    t = _timed_steps(torch, fn, steps, warmup, stream)
    launches = (la.la_launch_count() - l0) // (steps + warmup)
    ms = max_over_ranks(t)
    el = q.element_size()
    alg = w.B * w.H * w.N * (4 * w.D + 3 * w.M) * el      # read Q, K, V, dO; write dQ, dK, dV
    gbs = alg / (ms / 1e3) / 1e9
    leg = {"workload": name, "op": "noncausal_backward" if noncausal else "causal_backward",
           "value": round(world * w.B * w.N / (ms / 1e3), 1),
           "unit": "tokens/s", "ms_per_step": round(ms, 5), "steps": steps, "launches_per_step": launches,
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": round(gbs / pk["hbm_gbs"], 4),
                        "traffic": _traffic(("backward_nc_" if noncausal else "backward_") + name),
                        "alg_bytes_per_launch": alg},
           "l2": rot.describe(in_bytes),
           "note": ("tcgen05 kernels: key sums [S | z], a query pass (dQ and partial sums of phi(Q)^T [g | e]), "
                    "a key pass (dK, dV); K and V are read twice, so traffic is 9 tensors against 7 algorithmic"
                    if noncausal else
                    "tcgen05 kernels (bf16 D = M = 64): a forward sweep (dQ, keeps g and e) and a reverse "
                    "sweep (dK, dV), one CTA per head each" if w.D == 64 and w.M == 64 else
                    "tcgen05 kernels, segmented (bf16 D, M in {64, 128}): segment key sums, an exclusive scan "
                    "into each segment's entering state, a query pass (dQ, g, e; S in TMEM along the segment), the "
                    "reverse scan, a key pass (dK, dV; R in TMEM), one CTA per segment of consecutive chunks (about "
                    "one per SM); K and V are read a second time by the segment key sums")}
    del q, k, v, G, dq, dk, dv, sets
    torch.cuda.empty_cache()
    return leg


# fp32 CUDA-core peak of a GB300: 152 SMs x 128 FP32 lanes x 2 flop (FMA) x 2070 MHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def _leg_variant(torch, la, inputs, name, dev, stream, rot, pk, steps, max_over_ranks, world, rank, warmup=3):
    """Causal variant forward (feature map / sum normalisation / delta rule) on CUDA cores."""
    w = inputs.WORKLOADS[name]
    fm, nu, norm, update = w.variant
    var = la.variant(fm, nu, norm, update)
    F = la.la_feature_dim(var, w.D)
    q, k, v = [t.to(dev) for t in inputs.workload_inputs(w, rank)]
    beta = inputs.workload_betas(w, rank).to(dev) if update == "delta" else None
    out = torch.empty(w.B, w.H, w.N, w.M, dtype=w.dtype, device=dev)
    el = q.element_size()
    in_bytes = (2 * q.numel() + v.numel() + (beta.numel() if beta is not None else 0)) * el
    sets = _rotating(torch, (q, k, v, beta, out), rot.copies(in_bytes))
    it = [0]

    def fn():
        q_, k_, v_, b_, o_ = sets[it[0] % len(sets)]
        it[0] += 1
        la.la_forward_causal_variant(q_, k_, v_, var, beta=b_, out=o_, stream=stream)

    l0 = la.la_launch_count()
    t = _timed_steps(torch, fn, steps, warmup, stream)
    launches = (la.la_launch_count() - l0) // (steps + warmup)
    ms = max_over_ranks(t)
    alg = in_bytes + out.numel() * el                          # read Q, K, V (beta) once, write O once
    gbs = alg / (ms / 1e3) / 1e9
    # per head-token: state update 2FM (+ retrieval 2FM for the delta rule) and read-out 2FM
    flops = w.B * w.H * w.N * (6 if update == "delta" else 4) * F * w.M
    tf = flops / (ms / 1e3) / 1e12
    # the library's routing rule: bf16 sum-update variants with F, M in
    # {64, 128} (elu + 1 or DPFP) run the chunked tcgen05 kernel
    tc = (w.dtype == torch.bfloat16 and update == "sum" and F in (64, 128) and w.M in (64, 128)
          and fm in ("elu1", "dpfp"))
    # ... and bf16 delta-rule variants with sum-normalised features of width 64, M = 64
    tc_delta = (w.dtype == torch.bfloat16 and update == "delta" and norm == "sum" and F == 64 and w.M == 64
                and (fm == "elu1" or (fm == "dpfp" and (w.D, nu) in ((32, 1), (16, 2)))))
    hbm = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
           "frac": round(gbs / pk["hbm_gbs"], 4), "alg_bytes_per_launch": alg,
           "traffic": _traffic("causal_variant_" + name)}
    alu = {"bound": "alu", "achieved": round(tf, 2), "peak": round(FP32_ALU_TFLOPS, 1), "unit": "TFLOP/s",
           "frac": round(tf / FP32_ALU_TFLOPS, 4), "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x 2070 MHz",
           "alg_flops_per_launch": flops, "traffic": _traffic("causal_variant_" + name)}
    leg = {"workload": name, "op": "causal_variant", "variant": {"feature_map": fm, "nu": nu, "norm": norm,
                                                                 "update": update, "F": F},
           "value": round(world * w.B * w.N / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
           "steps": steps, "launches_per_step": launches,
           "roofline": hbm if tc else alu,
           "l2": rot.describe(in_bytes)}
    if tc:
        leg["tensor"] = {"alg_tflops": round(tf, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac_alg": round(tf / pk["bf16_tflops"], 4)}
        leg["note"] = ("chunked tcgen05 causal kernel, the feature map applied row by row in shared memory "
                       "between TMA and MMA")
    elif tc_delta:
        leg["hbm"] = hbm
        leg["note"] = ("chunked delta rule: K K^T, Q K^T, K S, Q S + tril(Q K^T) U and K^T U on tcgen05, the "
                       "triangular solve for the pseudo-values U (C^2 M / 2 fp32 FMAs per chunk of C = 128) on "
                       "CUDA cores; alu = the recurrence's 6 F M flops per head-token against the fp32 peak")
    else:
        leg["hbm"] = hbm
        leg["note"] = ("CUDA-core recurrence: one CTA per (head, 16 state columns), each warp walking the tokens "
                       "of a chunk on its own columns")
    del q, k, v, beta, out, sets
    torch.cuda.empty_cache()
    return leg


def _leg_decode(torch, la, inputs, dev, stream, rot, pk, args, max_over_ranks, world, rank):
    w = inputs.WORKLOADS["decode_b256h16d64"]
    B, H, D, M = w.B, w.H, w.D, w.M
    # prefill the state with 1024 random tokens through the causal forward
    qp, kp, vp = [t.to(dev) for t in inputs.workload_inputs(w, rank)]
    S = torch.zeros(B, H, D, M, device=dev)
    z = torch.zeros(B, H, D, device=dev)
    la.la_forward_causal(qp, kp, vp, S=S, z=z, want_out=False, stream=stream)
    del qp, kp, vp
    steps = w.steps
    qs, ks, vs = inputs.decode_tokens(steps, B, H, D, M, w.dtype, seed=inputs.rank_seed(w.seed + 1000, rank),
                                      device=dev)
    y = torch.empty(B, H, M, dtype=w.dtype, device=dev)
    n_flush = min(args.decode_steps, steps)
    t_idx = [0]
    # the state a step rewrites rotates over copies (each a sequence of its
    # own, all prefilled alike), so every step reads its state from HBM
    state_bytes = (S.numel() + z.numel()) * 4
    states = _rotating(torch, (S, z, y), rot.copies(state_bytes))

    def one():
        i = t_idx[0] % steps
        S_, z_, y_ = states[t_idx[0] % len(states)]
        la.la_decode_step(qs[i], ks[i], vs[i], S_, z_, y=y_, stream=stream)
        t_idx[0] += 1

    times = _timed_steps(torch, one, n_flush, args.warmup if args.only else 3, stream)
    ms = max_over_ranks(times)
    bytes_step = B * H * (2 * D * M * 4 + 2 * D * 4 + (2 * D + 2 * M) * 2)
    gbs = bytes_step / (ms / 1e3) / 1e9
    leg = {"workload": "decode_b256h16d64", "value": round(world / (ms / 1e3), 1), "unit": "steps/s",
           "ms_per_step": round(ms, 5), "steps": n_flush, "prefill_tokens": w.N,
           "hbm_gbs": round(gbs, 1),
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": round(gbs / pk["hbm_gbs"], 4), "traffic": _traffic("decode_decode_b256h16d64"),
                        "alg_bytes_per_launch": bytes_step},
           "l2": rot.describe(state_bytes) + "; state rewritten in place each step"}
    # all 4096 sequential steps captured in a CUDA graph, no flush: the 65 MiB state stays in L2
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            s2 = torch.cuda.Stream(dev)
            s2.wait_stream(stream)
            with torch.cuda.stream(s2):
                la.la_decode_step(qs[0], ks[0], vs[0], S, z, y=y, stream=s2)
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=s2):
                    for i in range(steps):
                        la.la_decode_step(qs[i], ks[i], vs[i], S, z, y=y, stream=s2)
            stream.wait_stream(s2)
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            gms = max_over_ranks(a.elapsed_time(b))
            leg["graph_4096"] = {"steps_per_s": round(world * steps / (gms / 1e3), 1),
                                 "ms_total": round(gms, 3), "effective_gbs": round(bytes_step * steps / (gms / 1e3) / 1e9, 1),
                                 "l2": "not flushed: the state is L2-resident between steps; not an HBM figure"}
            del g
        except Exception as e:  # report, do not hide
            leg["graph_4096"] = {"error": repr(e)}
    # all 4096 steps in one launch (la_decode_steps): the state stays on chip
    # across the steps, so they cost their q, k, v, y traffic only
    Sf, zf = S.clone(), z.clone()
    yf = torch.empty((steps, B, H, M), dtype=w.dtype, device=dev)
    fused = lambda: la.la_decode_steps(qs, ks, vs, Sf, zf, y=yf, stream=stream)  # noqa: E731
    ft = _timed_steps(torch, fused, 3, 1, stream)
    fms = max_over_ranks(ft)
    fbytes = 2 * B * H * (D * M + D) * 4 + steps * B * H * (2 * D + 2 * M) * 2
    leg["fused_4096"] = {"steps_per_s": round(world * steps / (fms / 1e3), 1), "ms_total": round(fms, 3),
                         "launches": 1, "hbm_gbs": round(fbytes / (fms / 1e3) / 1e9, 1),
                         "roofline": {"bound": "hbm", "achieved": round(fbytes / (fms / 1e3) / 1e9, 1),
                                      "peak": pk["hbm_gbs"], "unit": "GB/s",
                                      "frac": round(fbytes / (fms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
                                      "alg_bytes_per_launch": fbytes},
                         "note": "la_decode_steps: for steps whose inputs are known together; "
                                 "state read and written once, tokens streamed"}
    del Sf, zf, yf, states
    del qs, ks, vs, S, z, y
    torch.cuda.empty_cache()
    return leg


# ------------------------------------------------------------ CPU oracle

def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or 'unknown'."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _cpu_timed(fn, budget_s):
    """Seconds per call of fn, repeating it for at least budget_s (and once at least)."""
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn()
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return (time.perf_counter() - t0) / reps, reps


def _cpu_entry(value, unit, nthreads, sample):
    return {"value": round(value, 1), "unit": unit, "cores": nthreads,
            "omp_num_threads": os.environ.get("OMP_NUM_THREADS"), "cpu_model": cpu_model(),
            "kind": "oracle", "sample": sample}


def cpu_baseline(w, budget_s=4.0, heads=None, rows=None):
    """The fp64 recurrence oracle (eqs. (10)-(12)) on the host cores, on a
    bounded sample of heads (and of their rows); tokens/s = head-tokens/s / H."""
    import oracle
    from weight_recurrence_gb300 import inputs

    oracle.build()
    nthreads = oracle.max_threads()
    heads = max(1, min(w.B * w.H, heads or 2 * nthreads))
    n = min(w.N, rows or w.N)
    # the sample's own seeded draw, with the workload's shape per head and distribution
    qs, ks, vs = inputs.qkv(1, heads, n, w.D, w.M, w.dtype, w.scale, seed=w.seed)
    fn = oracle.noncausal if w.op == "noncausal" else oracle.causal
    dt, reps = _cpu_timed(lambda: fn(qs, ks, vs, nthreads=nthreads), budget_s)
    return _cpu_entry(heads * n / dt / w.H, "tokens/s", nthreads,
                      "%d heads x %d rows of the %d-head, N=%d workload (fp64 %s oracle), %d reps; tokens/s = "
                      "head-tokens/s / H" % (heads, n, w.B * w.H, w.N,
                                             "non-causal" if w.op == "noncausal" else "recurrence", reps))


def cpu_baseline_decode(w, budget_s=4.0):
    """The fp64 recurrence over all T decode steps (eqs. (16)-(20), one token at
    a time from the prefilled state) on a sample of heads, scaled to the whole
    batch: steps/s = 1 / (time for T steps x (B*H / heads) / T)."""
    import oracle
    from weight_recurrence_gb300 import inputs

    oracle.build()
    nthreads = oracle.max_threads()
    heads = max(1, min(w.B * w.H, 8 * nthreads))
    # the sampled heads' own draws (same distributions; the whole batch's
    # 4096 steps would be 13 GB on the host)
    qp, kp, vp = inputs.qkv(1, heads, w.N, w.D, w.M, w.dtype, w.scale, seed=w.seed)
    _, S0, z0 = oracle.causal(qp, kp, vp, want_out=False, nthreads=nthreads)   # the 1024-token prefill
    qs, ks, vs = inputs.decode_tokens(w.steps, 1, heads, w.D, w.M, w.dtype, seed=w.seed + 1000)
    # step-major [T, 1, heads, .] -> [1, heads, T, .]: the steps of each head in order
    per_head = [x.transpose(0, 2).contiguous() for x in (qs, ks, vs)]
    dt, reps = _cpu_timed(lambda: oracle.causal(*per_head, S0=S0, z0=z0, nthreads=nthreads), budget_s)
    t_step_all = dt / w.steps * (w.B * w.H) / heads
    return _cpu_entry(1.0 / t_step_all, "steps/s", nthreads,
                      "%d of %d heads x all %d steps after the %d-token prefill (fp64 recurrence, one token "
                      "at a time from the state), %d reps; scaled to all heads"
                      % (heads, w.B * w.H, w.steps, w.N, reps))


def cpu_baseline_backward(w, budget_s=4.0, noncausal=False, rows=None):
    """The fp64 causal (or non-causal) backward oracle on a sample of heads (and
    of their first `rows` tokens, if given); tokens/s as the forward."""
    import oracle
    import torch
    from weight_recurrence_gb300 import inputs

    oracle.build()
    nthreads = oracle.max_threads()
    heads = max(1, min(w.B * w.H, 2 * nthreads))
    n = min(w.N, rows) if rows else w.N
    q, k, v = inputs.qkv(1, heads, n, w.D, w.M, w.dtype, w.scale, seed=w.seed)
    g = torch.Generator().manual_seed(w.seed + 2000)
    G = torch.randn(v.shape, generator=g).to(w.dtype)
    fn = oracle.noncausal_backward if noncausal else oracle.causal_backward
    dt, reps = _cpu_timed(lambda: fn(q, k, v, G, nthreads=nthreads), budget_s)
    return _cpu_entry(heads * n / dt / w.H, "tokens/s", nthreads,
                      "%d of %d heads x N=%d%s (fp64 %s backward oracle), %d reps; tokens/s = head-tokens/s / H"
                      % (heads, w.B * w.H, n, " (first rows of N=%d)" % w.N if n < w.N else "",
                         "non-causal" if noncausal else "causal", reps))


def cpu_baseline_variant(w, budget_s=4.0):
    """The fp64 variant recurrence oracle on a sample of heads."""
    import oracle
    from weight_recurrence_gb300 import inputs

    oracle.build()
    nthreads = oracle.max_threads()
    heads = max(1, min(w.B * w.H, 2 * nthreads))
    fm, nu, norm, update = w.variant
    q, k, v = inputs.qkv(1, heads, w.N, w.D, w.M, w.dtype, w.scale, seed=w.seed)
    beta = inputs.betas(1, heads, w.N, w.dtype, seed=w.seed + 1000000) if update == "delta" else None
    dt, reps = _cpu_timed(lambda: oracle.variant_causal(q, k, v, fm=fm, nu=nu, norm=norm, update=update,
                                                        beta=beta, nthreads=nthreads), budget_s)
    return _cpu_entry(heads * w.N / dt / w.H, "tokens/s", nthreads,
                      "%d of %d heads x N=%d (fp64 %s/%s variant recurrence), %d reps; tokens/s = "
                      "head-tokens/s / H" % (heads, w.B * w.H, w.N, fm, update, reps))


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle on host cores, one bounded sample per step."""
    import oracle
    from weight_recurrence_gb300 import inputs

    oracle.build()
    w = inputs.WORKLOADS[MAIN]
    nthreads = oracle.max_threads()
    heads = max(1, min(w.B * w.H, nthreads))
    q, k, v = inputs.workload_inputs(w)
    qs = q.reshape(-1, w.N, w.D)[:heads].contiguous()
    ks = k.reshape(-1, w.N, w.D)[:heads].contiguous()
    vs = v.reshape(-1, w.N, w.M)[:heads].contiguous()
    for _ in range(args.warmup):
        oracle.causal(qs, ks, vs, nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.causal(qs, ks, vs, nthreads=nthreads)
    dt = (time.perf_counter() - t0) / args.steps
    value = heads * w.N / dt / w.H
    sample = "%d of %d heads x N=%d per step (fp64 recurrence oracle); tokens/s = head-tokens/s / H" % (
        heads, w.B * w.H, w.N)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1)/sqrt(D) bf16 widened to f64)",
            "config": main_config(w, world, "host cores: no GPU cache involved (CPU oracle)"),
            "cpu_baseline": _cpu_entry(value, "tokens/s", nthreads, sample),
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=256, help="flushed decode steps to time")
    ap.add_argument("--cpu-seconds", type=float, default=3.0, help="time budget of each CPU-baseline leg")
    ap.add_argument("--main-only", action="store_true", help="skip the non-causal, long and decode legs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--only", default=None,
                    choices=["causal_b16h8n3072d64", "noncausal_b8h8n4096d64", "causal_b1h16n65536d128",
                             "decode_b256h16d64", "backward_causal_b16h8n3072d64",
                             "backward_nc_causal_b16h8n3072d64", "backward_causal_b1h16n65536d128",
                             "delta_b16h8n3072d64", "dpfp_b16h8n3072d64"],
                    help="time this one workload alone (--steps/--warmup; decode: --decode-steps) and print "
                         "its leg object; for profiler captures, not a bench line")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        tdist.init_process_group("nccl")
        dist = tdist
    res = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
