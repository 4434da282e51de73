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
DATASHEET_BF16_TFLOPS = 2250.0   # dense bf16 per GPU (NVIDIA's figures halved for 2:4 sparsity)


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
        delta_bytes = B * S * H * D * 2 * 2 + B * H * S * 4 * 3   # read out, dout, lse; write delta, lse2
        roofline["delta_prepass_gbs"] = delta_bytes / (per_kernel["delta"] * 1e-3) / 1e9
        roofline["delta_prepass_frac_hbm"] = roofline["delta_prepass_gbs"] / peaks["hbm"]

    # end to end through the public API: pinned host inputs in, results back to the host
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
        dev_in = {n: torch.empty_like(t, device=dev) for n, t in host.items()}

        def e2e_step():
            for n, t in host.items():
                dev_in[n].copy_(t, non_blocking=True)
            o, l, _ = lwm.forward(dev_in["q"], dev_in["k"], dev_in["v"], dev_in["seg"], dev_in["pos"],
                                  kv_chunks=w.kv_chunks, workspace=ws, stream=stream)
            host_out["out"].copy_(o, non_blocking=True)
            host_out["lse"].copy_(l, non_blocking=True)
            if w.backward:
                g = lwm.backward(dev_in["q"], dev_in["k"], dev_in["v"], o, dev_in["dout"], l, dev_in["seg"],
                                 dev_in["pos"], workspace=ws, stream=stream)
                for n, t in zip(("dq", "dk", "dv"), g):
                    host_out[n].copy_(t, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(1, min(args.steps, 5))
        barrier(world)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms_e2e = max_over_ranks(a0.elapsed_time(a1), world, dev) / n_e2e
        e2e = {"value": world * flops_step / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e}
        del dev_in

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
        }
        print(json.dumps(line), flush=True)


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
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        run_ours(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
