"""Benchmark: exact causal (packed) attention, forward + backward, on B300.

One step = the whole hot path over one batch of the workload: metadata pre-pass,
forward kernel, row-dot pre-pass, dK/dV kernel and dQ kernel (forward only for the
1M-token workload), all through the library's C ABI. Reported value: credited
attention TFLOP/s, counting only visible (unmasked) query-key pairs: 4*D*H per pair
forward, 14*D*H per pair forward + backward.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]

For N > 1 (one process per GPU under torch.distributed.run) every rank runs its own
copy of the workload (independent problems, no collective on the data path); the
timed region is bracketed by barriers and the slowest rank's time is used.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal attn TFLOP/s (fwd, fwd+bwd) at S=32K–1M on 1 B300; % of BF16 dense peak"
# NVIDIA's published HGX B300 figure is 36 PFLOP/s FP16/BF16 for 8 GPUs with 2:4 sparsity:
# 4.5 PFLOP/s sparse, 2.25 PFLOP/s dense per GPU.
DATASHEET_BF16_TFLOPS = 2250.0


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"bf16": p["bf16_tflops"], "bf16_sustained": p.get("bf16_tflops_sustained"),
                "hbm": p["hbm_gbs"], "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16": 1800.0, "bf16_sustained": 1400.0, "hbm": 6400.0, "source": "fallback"}


def load_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu record, or
    None when there is none or the kernel's source has changed since it was taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f).get(kernel)
        if not rec:
            return None
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha1(f.read()).hexdigest() != rec["sha1"]:
                return None
        return rec["bytes_per_launch"].get(workload)
    except (OSError, ValueError, KeyError):
        return None


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        rank = dist.get_rank()
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
        return rank, world
    return 0, 1


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """Largest value of x over all ranks (x on every rank)."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(S_sample, heads, seed=0):
    """Times the float64 oracle (forward + backward, as it stands) on the first S_sample
    tokens of `heads` heads of a single causal document. Returns (seconds, credited
    flops, threads)."""
    import oracle
    cpus = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        threads = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except ImportError:
        # numpy's bundled OpenBLAS starts one thread per available CPU unless told otherwise
        env = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
        threads = int(env) if env and env.isdigit() else cpus
    threads = min(threads, cpus)
    g = torch.Generator().manual_seed(seed)
    q, k, v, do = (torch.randn((1, S_sample, heads, 128), generator=g).to(torch.bfloat16).float().numpy()
                   for _ in range(4))
    t0 = time.perf_counter()
    oracle.attention_forward(q, k, v, None)
    oracle.attention_backward(q, k, v, do, None)
    dt = time.perf_counter() - t0
    pairs = S_sample * (S_sample + 1) // 2
    return dt, 14.0 * 128 * heads * pairs, threads


def run_reference(args, rank):
    """--impl reference: the float64 oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return
    w = workload_of(args)
    S_sample = 8192
    for _ in range(args.warmup):
        oracle_sample(S_sample, 1)
    times, flops, threads = [], 0.0, 1
    for _ in range(args.steps):
        dt, flops, threads = oracle_sample(S_sample, 1)
        times.append(dt)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    sample = (f"float64 oracle forward+backward of head 0, first {S_sample} tokens of one causal document "
              f"(D=128), per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {**w.describe(), "inputs": "host memory"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def workload_of(args):
    from blockwise_ringattention_causal_b300 import inputs as I
    if args.seq > 0:
        return I.custom(args.batch, args.seq, args.heads, 128, None, seed=0,
                        name=f"causal-S{args.seq}-H{args.heads}-B{args.batch}")
    return I.workload(args.config)


# ----------------------------------------------------------------------------- GPU leg
def run_ours(args, rank, world):
    import blockwise_ringattention_causal_b300 as lwm
    from blockwise_ringattention_causal_b300 import inputs as I

    dev = torch.device("cuda", torch.cuda.current_device())
    w = workload_of(args)
    B, S, H, D = w.B, w.S, w.H, w.D
    x = I.make_inputs(w, dev, with_dout=w.backward)
    q, k, v, seg, pos = x["q"], x["k"], x["v"], x["seg"], x["pos"]
    dout = x.get("dout")
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    if w.backward:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = lwm.new_workspace(B, S, H, D, dev, forward_only=not w.backward)
    stream = torch.cuda.current_stream()
    pairs = I.pairs_per_head(w)
    flops_fwd = 4.0 * D * H * pairs
    flops_step = (14.0 if w.backward else 4.0) * D * H * pairs

    # kernel name -> (events before, after) inside each timed step
    fused = args.bwd == "fused"
    bwd_names = ["delta", "dkdvq"] if fused else ["delta", "dkdv", "dq"]
    names = ["meta", "fwd"] + (bwd_names if w.backward else [])

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        lwm.lwm_attn_prepare(seg, pos, B, S, H, D, w.kv_chunks, ws, stream)
        mark(1)
        lwm.lwm_attn_fwd_prepared(q, k, v, out, lse, ws, stream)
        mark(2)
        if w.backward:
            lwm.lwm_attn_bwd_stages(None, None, None, out, dout, lse, None, None, None, lwm.LWM_BWD_DELTA, ws, stream)
            mark(3)
            if fused:
                # memset of the dQ accumulator, the single backward kernel, dq conversion
                lwm.lwm_attn_bwd_stages(q, k, v, None, dout, None, dq, dk, dv, lwm.LWM_BWD_FUSED, ws, stream)
                mark(4)
            else:
                lwm.lwm_attn_bwd_stages(q, k, v, None, dout, None, None, dk, dv, lwm.LWM_BWD_DKDV, ws, stream)
                mark(4)
                lwm.lwm_attn_bwd_stages(q, k, v, None, dout, None, dq, None, None, lwm.LWM_BWD_DQ, ws, stream)
                mark(5)

    # meta (3 kernels), fwd, then delta + (dK/dV/dQ kernel + dq conversion | dK/dV + dQ)
    launches_per_step = 3 + 1 + (3 if w.backward else 0)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = lwm.lwm_attn_check(ws)
    if status != 0:
        raise RuntimeError(f"device error during warm-up: {lwm.lwm_status_string(status)}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or
                                                                                           torch.cuda.current_device()))
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        step(evs[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    status = lwm.lwm_attn_check(ws)
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {lwm.lwm_status_string(status)}")
    ms_local = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_local, world, dev)
    per_kernel = {n: statistics.mean(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(args.steps))
                  for i, n in enumerate(names)}

    ms_step = ms_total / args.steps
    value = world * flops_step / (ms_step * 1e-3) / 1e12
    fwd_tflops = flops_fwd / (per_kernel["fwd"] * 1e-3) / 1e12

    # roofline of the dominant kernel (largest share of the step)
    alg = {"fwd": 4.0 * D * H * pairs, "dkdv": 8.0 * D * H * pairs, "dq": 6.0 * D * H * pairs,
           "dkdvq": 10.0 * D * H * pairs}
    dom = max((n for n in alg if n in per_kernel), key=lambda n: per_kernel[n])
    peaks = load_peaks()
    achieved = alg[dom] / (per_kernel[dom] * 1e-3) / 1e12
    traffic = load_traffic(f"{dom}_kernel", w.name)
    roofline = {"bound": "tensor", "kernel": f"{dom}_kernel", "achieved": achieved, "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16"], "traffic": traffic,
                "peak_source": f"{peaks['source']} bf16 burst", "peak_sustained": peaks["bf16_sustained"],
                "frac_of_sustained": achieved / peaks["bf16_sustained"] if peaks["bf16_sustained"] else None,
                "kernel_ms": {n: round(t, 4) for n, t in per_kernel.items()}}
    if w.backward:
        # read out, dout, lse; write delta, lse2 and the two 16-byte offset rows of the dK/dV kernel
        delta_bytes = B * S * H * D * 2 * 2 + B * H * S * 4 * 3 + B * H * S * 32
        roofline["delta_prepass_gbs"] = delta_bytes / (per_kernel["delta"] * 1e-3) / 1e9
        roofline["delta_prepass_frac_hbm"] = roofline["delta_prepass_gbs"] / peaks["hbm"]

    # End to end through the public API: pinned host inputs in, results back to the host,
    # every step. Steps are double-buffered the way a caller streaming batches would run
    # them: step i's inputs upload on one copy stream while step i - 1 computes, and its
    # results download on another copy stream while step i + 1 computes (H2D and D2H use
    # separate copy engines). The timed region runs from the first upload to the last
    # download, so the pipeline's fill and drain are inside it.
    e2e = None
    if not args.no_e2e:
        host = {n: t.to("cpu").pin_memory() for n, t in x.items() if t is not None}
        host_out = {"out": torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                    "lse": torch.empty(lse.shape, dtype=lse.dtype).pin_memory()}
        if w.backward:
            for n in ("dq", "dk", "dv"):
                host_out[n] = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        dev_in = [{n: torch.empty_like(t, device=dev) for n, t in host.items()} for _ in range(2)]
        # compute on a stream of its own (not the legacy default stream, which would
        # serialise with the copy streams); outputs are allocated on it
        comp, up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_free = [None, None]   # compute done with input set i % 2 (event), per set

        def e2e_step(i):
            bi = i % 2
            if in_free[bi] is not None:
                up.wait_event(in_free[bi])
            with torch.cuda.stream(up):
                for n, t in host.items():
                    dev_in[bi][n].copy_(t, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(up)
            comp.wait_event(ready)
            d = dev_in[bi]
            with torch.cuda.stream(comp):
                o, l, _ = lwm.forward(d["q"], d["k"], d["v"], d["seg"], d["pos"], kv_chunks=w.kv_chunks,
                                      workspace=ws, stream=comp)
                fwd_done = torch.cuda.Event()
                fwd_done.record(comp)
                g = ()
                if w.backward:
                    g = lwm.backward(d["q"], d["k"], d["v"], o, d["dout"], l, d["seg"], d["pos"], workspace=ws,
                                     stream=comp)
                done = torch.cuda.Event()
                done.record(comp)
            in_free[bi] = done
            down.wait_event(fwd_done)
            with torch.cuda.stream(down):
                host_out["out"].copy_(o, non_blocking=True)
                host_out["lse"].copy_(l, non_blocking=True)
            down.wait_event(done)
            with torch.cuda.stream(down):
                for n, t in zip(("dq", "dk", "dv"), g):
                    host_out[n].copy_(t, non_blocking=True)
            # the caching allocator must not hand these out again before the downloads end
            for t in (o, l, *g):
                t.record_stream(down)

        e2e_step(0)
        torch.cuda.synchronize()
        n_e2e = max(1, min(args.steps, 10))
        barrier(world)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(up)
        for i in range(n_e2e):
            e2e_step(i + 1)
        a1.record(down)
        torch.cuda.synchronize()
        barrier(world)
        ms_e2e = max_over_ranks(a0.elapsed_time(a1), world, dev) / n_e2e
        e2e = {"value": world * flops_step / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
               "steps": n_e2e, "overlap": "double-buffered: uploads, compute and downloads of "
                                          "neighbouring steps on three streams"}
        del dev_in

    extras = {}
    if not args.no_extras:
        del x, q, k, v, dout, out, lse
        if w.backward:
            del dq, dk, dv
        del ws
        torch.cuda.empty_cache()
        extras = run_extras(args, dev, stream, peaks, value if w.name == "causal-S32K-H32-D128" else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        S_sample, heads = 8192, 8
        dt, fl, threads = oracle_sample(S_sample, heads)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"float64 oracle forward+backward of {heads} heads x first {S_sample} tokens of one "
                         f"causal document (D=128), {dt:.1f} s; BLAS threads {threads} of "
                         f"{len(os.sched_getaffinity(0))} host CPUs"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**w.describe(), "parallelism": f"independent replicas x{world}" if world > 1 else "none",
                       "l2": "inputs larger than L2 (126 MB)" if B * S * H * D * 2 > 126e6 else "inputs fit in L2",
                       "credited_pairs_per_head": pairs, "credited_flops_per_step": flops_step},
            "fwd_tflops": fwd_tflops,
            "pct_of_peak": {"measured_burst": 100 * value / peaks["bf16"],
                            "measured_sustained": 100 * value / peaks["bf16_sustained"],
                            "datasheet_dense": 100 * value / DATASHEET_BF16_TFLOPS},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
            **extras,
        }
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- further kernels
def _time(fn, steps, warmup, stream):
    """Mean ms per call of fn() over `steps` calls after `warmup`, CUDA events on `stream`."""
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


def run_extras(args, dev, stream, peaks, value_32k):
    """The packed mixed-modality workload's fwd+bwd, and the memory-bound kernels of the
    path (RoPE, decoding against a 1M-token cache, the re-weighted packed loss), each
    timed alone on its own inputs (not inside the headline's timed region)."""
    import blockwise_ringattention_causal_b300 as lwm
    from blockwise_ringattention_causal_b300 import inputs as I
    out = {}
    steps, warmup = max(3, min(args.steps, 10)), 3
    hbm = peaks["hbm"]

    # packed mixed modality: B = 2 rows of 64K tokens, 19 + 25 documents
    w = I.workload(3)
    x = I.make_inputs(w, dev)
    B, S, H, D = w.B, w.S, w.H, w.D
    o = torch.empty_like(x["q"])
    l = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    ws = lwm.new_workspace(B, S, H, D, dev, forward_only=True)
    evs = []

    def packed_step(record=False):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(6)] if record else None
        if e: e[0].record(stream)
        lwm.lwm_attn_prepare(x["seg"], x["pos"], B, S, H, D, 1, ws, stream)
        if e: e[1].record(stream)
        lwm.lwm_attn_fwd_prepared(x["q"], x["k"], x["v"], o, l, ws, stream)
        if e: e[2].record(stream)
        lwm.lwm_attn_bwd_stages(None, None, None, o, x["dout"], l, None, None, None, lwm.LWM_BWD_DELTA, ws, stream)
        if e: e[3].record(stream)
        lwm.lwm_attn_bwd_stages(x["q"], x["k"], x["v"], None, x["dout"], None, None, dk, dv, lwm.LWM_BWD_DKDV, ws,
                                stream)
        if e: e[4].record(stream)
        lwm.lwm_attn_bwd_stages(x["q"], x["k"], x["v"], None, x["dout"], None, dq, None, None, lwm.LWM_BWD_DQ, ws,
                                stream)
        if e:
            e[5].record(stream)
            evs.append(e)

    ms = _time(lambda: packed_step(True), steps, warmup, stream)
    evs[:] = evs[warmup:]
    if lwm.lwm_attn_check(ws) != 0:
        raise RuntimeError("device error in the packed workload")
    pairs = I.pairs_per_head(w)
    names = ["meta", "fwd", "delta", "dkdv", "dq"]
    kms = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i, n in enumerate(names)}
    pv = 14.0 * D * H * pairs / (ms * 1e-3) / 1e12
    out["packed"] = {"workload": w.name, "value": pv, "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
                     "credited_pairs_per_head": pairs, "fwd_tflops": 4.0 * D * H * pairs / (kms["fwd"] * 1e-3) / 1e12,
                     "kernel_ms": {n: round(t, 4) for n, t in kms.items()},
                     "ratio_to_causal_32k": (pv / value_32k) if value_32k else None}

    # RoPE on q and k of the 32K workload (theta = 1e6, LWM's 32K stage): read q, k and
    # pos, write the rotated q, k
    w2 = I.workload(2)
    B, S, H = w2.B, w2.S, w2.H
    del x, o, l, dq, dk, dv, ws
    torch.cuda.empty_cache()
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    q = torch.randn((B, S, H, D), generator=g, device=dev, dtype=torch.bfloat16)
    k = torch.randn((B, S, H, D), generator=g, device=dev, dtype=torch.bfloat16)
    pos = torch.arange(S, dtype=torch.int32, device=dev).repeat(B, 1).contiguous()
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    ms = _time(lambda: lwm.lwm_attn_rope(q, k, pos, 1e6, qr, kr, False, stream), steps, warmup, stream)
    nbytes = 4 * B * S * H * D * 2 + B * S * 4
    out["rope"] = {"shape": [B, S, H, D], "theta": 1e6, "ms": ms, "bytes": nbytes,
                   "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                                "frac": nbytes / (ms * 1e-3) / 1e9 / hbm}}
    del q, k, qr, kr, pos
    torch.cuda.empty_cache()

    # decoding: T new tokens of one row against a 2^20-token cache, 32 heads
    Sd = 1 << 18 if args.extras_small else 1 << 20
    kc = torch.randn((1, Sd, H, D), generator=g, device=dev, dtype=torch.bfloat16)
    vc = torch.randn((1, Sd, H, D), generator=g, device=dev, dtype=torch.bfloat16)
    dec = {}
    for T in (1, 4):
        qd = torch.randn((1, T, H, D), generator=g, device=dev, dtype=torch.bfloat16)
        od = torch.empty_like(qd)
        ld = torch.empty((1, H, T), dtype=torch.float32, device=dev)
        wsd = torch.zeros(lwm.lwm_attn_decode_workspace_size(1, T, Sd, H, D), dtype=torch.uint8, device=dev)
        ms = _time(lambda: lwm.lwm_attn_decode(qd, kc, vc, None, od, ld, wsd, stream), steps, warmup, stream)
        if lwm.lwm_attn_check(wsd) != 0:
            raise RuntimeError("device error in decoding")
        nbytes = 2 * Sd * H * D * 2 + 2 * T * H * D * 2
        dec[f"T{T}"] = {"ms": ms, "bytes": nbytes,
                        "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm,
                                     "unit": "GB/s", "frac": nbytes / (ms * 1e-3) / 1e9 / hbm}}
    out["decode"] = {"cache_tokens": Sd, "heads": H, **dec}
    del kc, vc
    torch.cuda.empty_cache()

    # the re-weighted packed loss over the packed workload's rows, vocabulary 32768
    if args.extras_small:
        w = I.custom(1, 16384, 1, 128, [[4000, 258, 9000, 258, 2868]], name="packed-16K")
    Bl, Sl, V = w.B, w.S, 32768
    seg_np, _ = I.segments(w)
    seg = torch.from_numpy(seg_np).to(dev)
    logits = (torch.randn((Bl, Sl, V), generator=g, device=dev) * 2).to(torch.bfloat16)
    targets = torch.randint(0, V, (Bl, Sl), generator=g, device=dev, dtype=torch.int32)
    wt = torch.ones((Bl, Sl), dtype=torch.float32, device=dev)
    for b, lens in enumerate(w.lengths):
        ends = torch.tensor([sum(lens[:i + 1]) - 1 for i in range(len(lens))], device=dev)
        wt[b, ends] = 0.0
    loss = torch.empty(1, dtype=torch.float64, device=dev)
    dlog = torch.empty_like(logits)
    wsl = torch.zeros(lwm.lwm_packed_loss_workspace_size(Bl, Sl), dtype=torch.uint8, device=dev)
    ms = _time(lambda: lwm.lwm_packed_loss(logits, targets, wt, seg, loss, dlog, wsl, stream), steps, warmup, stream)
    if lwm.lwm_attn_check(wsl) != 0:
        raise RuntimeError("device error in the packed loss")
    nbytes = 2 * Bl * Sl * V * 2
    out["packed_loss"] = {"shape": [Bl, Sl, V], "documents": sum(len(r) for r in w.lengths), "ms": ms,
                          "bytes": nbytes,
                          "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm,
                                       "unit": "GB/s", "frac": nbytes / (ms * 1e-3) / 1e9 / hbm}}
    del logits, dlog, targets, wt, wsl
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=2, help="1..5 (2 = S=32K, H=32, D=128 causal)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seq", type=int, default=0, help="custom workload: sequence length (one document)")
    ap.add_argument("--heads", type=int, default=32, help="custom workload: heads")
    ap.add_argument("--batch", type=int, default=1, help="custom workload: batch rows")
    ap.add_argument("--bwd", choices=["separate", "fused"], default="separate",
                    help="backward path: dK/dV and dQ kernels (default) or one dK/dV/dQ kernel")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the packed workload and the RoPE / decode / packed-loss measurements")
    ap.add_argument("--extras-only", action="store_true",
                    help="run only the packed workload and the RoPE / decode / packed-loss measurements")
    ap.add_argument("--extras-small", action="store_true",
                    help="smaller extras (a 256K-token decode cache, a 16K-token packed-loss batch) for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank)
    elif args.extras_only:
        dev = torch.device("cuda", torch.cuda.current_device())
        extras = run_extras(args, dev, torch.cuda.current_stream(), load_peaks(), None)
        if rank == 0:
            print(json.dumps(extras), flush=True)
    else:
        run_ours(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
